// Backward attention on 5th-generation tensor cores (tcgen05, TMEM, TMA) for sm_103a.
//
// Operation (see include/nc_attn.h): gradients of sum(O * dO) for exact causal
// sliding-window softmax attention ("nanochat GPT-2 speedrun" post, page 2,
// FlashAttention-3 window_size paragraph).  With P the softmax weights
// recomputed from the forward's log-sum-exp and Delta_i = rowsum(dO_i * O_i):
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - Delta),  dK = scale dS^T Q,  dQ = scale dS K.
//
// Three launches on the caller's stream:
//   bwd_pre   Delta = rowsum(dO * O) (fp32) and zeroing of the fp32 dQ accumulator
//   bwd_main  persistent CTAs (one per SM) take work items, each a 128-key block of one
//             (batch, head), from a counter; an item walks the query blocks whose window
//             reaches its keys; dK and dV accumulate in TMEM and each block's dQ
//             contribution is added to the fp32 accumulator
//   bwd_post  dq = bf16(scale * dQ accumulator)
// (The deterministic backward runs bwd_main without its dQ product and a separate dQ pass,
// bwd_dq_sm103.cu, instead of the accumulator.)
//
// bwd_main warp roles:
//   warp 0      TMA producer: each item's K and V, then Q and dO blocks (128-byte swizzle).  The
//               two K/V tiles swap roles from item to item, so an item's K loads as soon as the
//               previous item's last dP^T has read that item's V, a block before its last dQ
//               frees its K (the tile the V then goes to)
//   warp 1      MMA issuer (one lane) and TMEM owner (512 columns)
//   warps 4-7   one thread per key row, query columns [0, 64): P^T and dS^T from S^T and
//               dP^T; then the dK epilogue (staged in the dS tile)
//   warps 8-11  the same for query columns [64, 128); then the dV epilogue (staged in the
//               dO stage for D = 128, in the second half of the dS tile for D = 64)
//   warps 12-15 the block's dQ partial from TMEM into the fp32 accumulator by TMA reduce-adds
//               from a shared-memory staging tile: for D = 128 the product is dQ^T (one thread
//               per dQ column, staged a 64-row half at a time); for D = 64 it is dQ (one thread
//               per query row, the whole block in the 128-byte swizzle of two 32-column boxes)
// TMEM: ST [0,128) holds S^T, then P^T (bf16, two per column) in columns
//       [0,32) for queries 0-63 and [64,96) for queries 64-127, so each
//       warpgroup overwrites only columns it has already read.  DPT [128,256)
//       holds dP^T, then dS^T packed the same way, then the block's dQ.
//       DV [256,256+D); DK [256+D,256+2D).  dS also goes to a shared-memory
//       tile [key][query], the MN-major operand of the dQ product.
// Products per query block m:
//   dP^T = V dO_m^T, S^T = K Q_m^T            (both operands K-major in smem)
//   dV += P^T dO_m, dK += dS^T Q_m              (A from TMEM, B MN-major in smem)
//   dQ_m^T = K^T dS^T (D = 128) or dQ_m = dS K (D = 64), both operands MN-major in smem
#include <cstdint>
#include <cuda_bf16.h>

#include "nc_attn.h"
#include "nc_kernels.h"
#include "nc_ptx.cuh"
#include "nc_sched.cuh"
#include "nc_tma.h"

namespace nc {
namespace {

constexpr int kBK = 128;       // keys per CTA
constexpr int kBQ = 128;       // queries per block
constexpr int kQStages = 2;
constexpr int kThreads = 512;
// warps that read each work-item slot: the MMA warp, the 8 P/dS warps and the 4 dQ warps
constexpr int kItemReaders = 13;
constexpr float kLog2e = 1.4426950408889634f;

// D = 128: dQ partials leave through a TMA reduce-add from a 64-row fp32 staging tile,
// which takes the place of the second dO stage.  D = 64: two dO stages and a 128-row staging
// tile (two swizzled 32-column boxes).
template <int D>
struct BwdSmem {
    static constexpr bool kTmaReduce = (D == 128);
    // D = 64: the block's dQ (thread = query row) leaves through a 128-row fp32 staging tile in the 128-byte
    // swizzle of two 32-column TMA boxes, added by TMA reduce-adds
    static constexpr bool kStagedRows = (D == 64);
    static constexpr int kDOStages = kTmaReduce ? 1 : 2;
    static constexpr int kStageRows = 64;                 // dQ rows per reduce-add (D = 128)
    static constexpr int kTile = kBQ * D * 2;            // 128 rows x D bf16
    static constexpr int kK = 0;
    static constexpr int kV = kK + kTile;
    static constexpr int kQ = kV + kTile;                 // kQStages tiles
    static constexpr int kDO = kQ + kQStages * kTile;     // kDOStages tiles
    static constexpr int kDS = kDO + kDOStages * kTile;   // dS [key][query], 128 x 128 bf16
    static constexpr int kDSBytes = kBK * kBQ * 2;
    static constexpr int kStage = kDS + kDSBytes;         // fp32 [kStageRows][D] (D = 128 only)
    static constexpr int kStageBytes = kTmaReduce ? kStageRows * D * 4 : (kStagedRows ? kBQ * D * 4 : 0);
    static constexpr int kLse = kStage + kStageBytes;     // [2][128] fp32 (log2 units)
    static constexpr int kDelta = kLse + 2 * kBQ * 4;     // [2][128] fp32
    static constexpr int kBars = kDelta + 2 * kBQ * 4;
    static constexpr int kBytes = kBars + 256;
};

struct BwdBarriers {
    // K/V slots: tile s (s = 0 at kK, 1 at kV) holds K of the items of parity s and V of the others, so
    // the next item's K goes into the tile whose V was freed by the item's last dP^T, a block before
    // the item's K is freed by its last dQ.  Each slot is filled once per item.
    uint64_t kv_full[2];
    uint64_t kv_empty[2];  // the slot's K (last S^T and dQ) or V (last dP^T) reader is done
    uint64_t q_full[kQStages];
    uint64_t q_empty[kQStages];
    uint64_t do_full[2];
    uint64_t do_empty[2];
    uint64_t s_full;
    uint64_t dp_full;
    uint64_t p_full;
    uint64_t ds_full;
    uint64_t dq_full;
    uint64_t dq_empty;
    uint64_t final_;
    uint64_t drain;
    uint64_t epi_done;    // dK / dV epilogue tiles in the dS region have been read by their TMA stores
    uint64_t dv_final;    // the item's last dV product has landed (D = 128 with dQ: dV leaves through the dO stage)
    uint64_t do_epi_free; // the dV epilogue's TMA stores have read the dO stage (the next item's first dO may load)
    uint64_t item_full[kItemSlots];
    uint64_t item_empty[kItemSlots];
    int item[kItemSlots];
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(BwdBarriers) <= 256, "barrier block outgrew its shared-memory slot");

struct BwdParams {
    const float* lse;      // [B, H, T]
    const float* delta;    // [B, H, T]
    float* dq_acc;         // [B, T, H, D]
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int B, T, H, W;        // W effective, 1 <= W <= T
    float scale, scale_log2;
    int n_kb, n_qb;
    int group;             // (batch, head) pairs per scheduling group
    int* work;             // work-item counter, zero on entry
    // Document-masked backward over packed rows (B = 1, T = total): document d is rows
    // cu[d] .. cu[d+1]-1; n_kb then counts the key blocks of the longest document.  nullptr otherwise.
    const int* cu;
    int n_docs;
    int* err;
};

// One work item: a 128-key block n of one (batch, head), walked over query blocks
// m_lo .. m_lo + n_it - 1 (the blocks whose causal window reaches its keys).
//
// Items are handed out in index order by an atomic counter.  The (batch, head) pairs are cut
// into groups of p.group (about one wave of CTAs' worth of items); inside a group the index
// runs over n outermost, so the longest causal walks (small n) go first, while the CTAs that
// run at the same time share the Q and dO blocks of a few heads in L2.
// Varlen: the pairs are (document, head), positions count from the document's start, and items past a
// document's last key block are empty (the producer skips them).
struct BwdItem {
    int n, h, b, j0, m_lo, n_it;
    int base;   // first packed row of the document (varlen), else 0
    int len;    // rows of the sequence or document
    bool bad;   // the document's bounds are out of range
    bool empty;
};

template <bool kVarlen>
__device__ __forceinline__ BwdItem bwd_item(int w, const BwdParams& p) {
    BwdItem it;
    const int n_pairs = kVarlen ? p.n_docs * p.H : p.B * p.H;
    const int per_group = p.n_kb * p.group;
    const int grp = w / per_group, r = w - grp * per_group;
    const int in_grp = min(p.group, n_pairs - grp * p.group);  // the last group may be short
    const int bh = grp * p.group + r % in_grp;
    it.n = r / in_grp;
    it.h = bh % p.H;
    it.b = kVarlen ? 0 : bh / p.H;
    it.j0 = it.n * kBK;
    it.m_lo = it.n;  // kBQ == kBK: query block n holds the first queries at or after key j0
    it.base = 0;
    it.len = p.T;
    it.bad = false;
    it.empty = false;
    int n_qb = p.n_qb;
    if (kVarlen) {
        const int d = bh / p.H;
        const int a = p.cu[d], e = p.cu[d + 1];
        it.bad = a < 0 || e < a || e > p.T || e - a > p.n_kb * kBK;
        it.base = it.bad ? 0 : a;
        it.len = it.bad ? 0 : e - a;
        n_qb = (it.len + kBQ - 1) / kBQ;
        it.empty = it.bad || it.j0 >= it.len;
    }
    const int m_hi = min(n_qb - 1, (it.j0 + kBK - 1 + p.W - 1) / kBQ);
    it.n_it = m_hi - it.m_lo + 1;
    return it;
}

__device__ __forceinline__ bool aborted(const BwdBarriers* bars) {
    return *reinterpret_cast<const volatile int*>(&bars->abort) != 0;
}

__device__ __forceinline__ int publish_item(BwdBarriers* bars, int k, int n_items, int* work) {
    return ring_publish_item(bars->item_full, bars->item_empty, bars->item, k, n_items, work);
}

// Like publish_item, but takes further indices while they name empty items.
template <bool kVarlen>
__device__ __forceinline__ int publish_item_skipping(BwdBarriers* bars, int k, int n_items, const BwdParams& p) {
    const int slot = k % kItemSlots;
    if (!mbar_wait_warp(&bars->item_empty[slot], ((k / kItemSlots) & 1) ^ 1)) return -2;
    int w = 0;
    if (lane_id() == 0) {
        for (;;) {
            w = atomicAdd(p.work, 1);
            if (w >= n_items) {
                w = -1;
                break;
            }
            const BwdItem it = bwd_item<kVarlen>(w, p);
            if (it.bad) set_device_error(p.err, NC_ERR_BAD_SEQLENS);
            if (!it.empty) break;
        }
        bars->item[slot] = w;
        mbar_arrive(&bars->item_full[slot]);
    }
    return __shfl_sync(0xffffffffu, w, 0);
}

__device__ __forceinline__ int read_item(BwdBarriers* bars, int k) {
    return ring_read_item(bars->item_full, bars->item_empty, bars->item, k);
}

__device__ __forceinline__ void record_timeout(BwdBarriers* bars, int* err) {
    set_device_error(err, NC_ERR_DEVICE_TIMEOUT);
    atomicExch(&bars->abort, 1);
}

// kNoDq: dK and dV only (the deterministic backward computes dQ in a separate pass).
template <int D, bool kVarlen, bool kNoDq = false>
__global__ void __launch_bounds__(kThreads, 1)
bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
    using L = BwdSmem<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    BwdBarriers* bars = reinterpret_cast<BwdBarriers*>(smem + L::kBars);
    float* s_lse = reinterpret_cast<float*>(smem + L::kLse);
    float* s_delta = reinterpret_cast<float*>(smem + L::kDelta);

    const int warp = warp_id(), lane = lane_id();
    const int n_items = p.n_kb * p.H * (kVarlen ? p.n_docs : p.B);

    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) set_device_error(p.err, NC_ERR_CUDA);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->kv_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&bars->q_full[s], 1);
            mbar_init(&bars->q_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->do_full[s], 1);
            mbar_init(&bars->do_empty[s], 1);
        }
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->dp_full, 1);
        mbar_init(&bars->p_full, 2 * kBK);
        mbar_init(&bars->ds_full, 2 * kBK);
        mbar_init(&bars->dq_full, 1);
        mbar_init(&bars->dq_empty, kBQ);
        mbar_init(&bars->final_, 1);
        mbar_init(&bars->drain, 1);
        mbar_init(&bars->epi_done, L::kTmaReduce ? 1 : 2);
        mbar_init(&bars->dv_final, 1);
        mbar_init(&bars->do_epi_free, 1);
        for (int s = 0; s < kItemSlots; ++s) {
            mbar_init(&bars->item_full[s], 1);
            mbar_init(&bars->item_empty[s], kItemReaders);
        }
        bars->abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    constexpr uint32_t kColST = 0, kColDPT = 128, kColDV = 256, kColDK = 256 + D;

    // registers: 512 x 128 at launch = 65536; producer/MMA warpgroup drops to 56, the two
    // P/dS warpgroups rise to 152 and the dQ warpgroup to 152 (65536 in all), which lets
    // the dQ warpgroup hold a whole 128 x 128 fp32 dQ block and release TMEM at once
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // the whole warp runs this loop converged; lane 0 issues each copy
        regs_decrease<56>();
        {
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                tma_prefetch_desc(&tm_do);
            }
            __syncwarp();
            int gq = 0, gd = 0;  // Q and dO blocks loaded over all items (ring positions)
            int fills[2] = {0, 0};  // loads issued into each K/V slot
            bool ok = true;
            for (int ii = 0; ok; ++ii) {
                // varlen: pass over items past a document's end (and report bad document bounds)
                // before publishing, so the other roles only ever see items with work
                const int w = kVarlen ? publish_item_skipping<kVarlen>(bars, ii, n_items, p)
                                      : publish_item(bars, ii, n_items, p.work);
                if (w == -2 || aborted(bars)) {
                    ok = false;
                    break;
                }
                if (w < 0) break;
                const BwdItem item = bwd_item<kVarlen>(w, p);
                const int sk = ii & 1, sv = sk ^ 1;
                // K into the slot whose V the previous item's last dP^T has read (a block before that item
                // ends); V, after the first Q block, into the slot its last dQ frees
                if (!mbar_wait_warp(&bars->kv_empty[sk], (ii & 1) ^ 1) || aborted(bars)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_w(&bars->kv_full[sk], L::kTile);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d_w(smem + (sk ? L::kV : L::kK) + c * kBK * 128, &tm_k, &bars->kv_full[sk], c * 64,
                                  item.h, item.base + item.j0, item.b);
                ++fills[sk];
                for (int it = 0; it < item.n_it; ++it) {
                    const int st = gq % kQStages, so = gd % L::kDOStages;
                    const int i0 = (item.m_lo + it) * kBQ;
                    if (!mbar_wait_warp(&bars->q_empty[st], ((gq / kQStages) & 1) ^ 1) || aborted(bars)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_w(&bars->q_full[st], L::kTile);
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_4d_w(smem + L::kQ + st * L::kTile + c * kBQ * 128, &tm_q, &bars->q_full[st], c * 64,
                                      item.h, item.base + i0, item.b);
                    ++gq;
                    if (it == 0) {
                        if (!mbar_wait_warp(&bars->kv_empty[sv], (ii & 1) ^ 1) || aborted(bars)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx_w(&bars->kv_full[sv], L::kTile);
                        for (int c = 0; c < D / 64; ++c)
                            tma_load_4d_w(smem + (sv ? L::kV : L::kK) + c * kBK * 128, &tm_v, &bars->kv_full[sv],
                                          c * 64, item.h, item.base + item.j0, item.b);
                        ++fills[sv];
                    }
                    // D = 128 with dQ: the previous item's dV epilogue stages its tile in the dO stage
                    if (L::kTmaReduce && !kNoDq && it == 0 && ii > 0 &&
                        (!mbar_wait_warp(&bars->do_epi_free, (ii - 1) & 1) || aborted(bars))) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait_warp(&bars->do_empty[so], ((gd / L::kDOStages) & 1) ^ 1) || aborted(bars)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx_w(&bars->do_full[so], L::kTile);
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_4d_w(smem + L::kDO + so * L::kTile + c * kBQ * 128, &tm_do, &bars->do_full[so],
                                      c * 64, item.h, item.base + i0, item.b);
                    ++gd;
                }
            }
            if (!ok) record_timeout(bars, p.err);
            // never leave while a copy into this CTA's shared memory may still land: the last
            // use of each stage is the only one whose completion can still be outstanding
            for (int x = gq - kQStages < 0 ? 0 : gq - kQStages; x < gq; ++x)
                mbar_wait_warp(&bars->q_full[x % kQStages], (x / kQStages) & 1);
            for (int x = gd - L::kDOStages < 0 ? 0 : gd - L::kDOStages; x < gd; ++x)
                mbar_wait_warp(&bars->do_full[x % L::kDOStages], (x / L::kDOStages) & 1);
            for (int s = 0; s < 2; ++s)
                if (fills[s] > 0) mbar_wait_warp(&bars->kv_full[s], (fills[s] - 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs this loop converged; lane 0 issues each product
        regs_decrease<56>();
        {
            constexpr uint32_t id_kq = idesc_bf16(kBK, kBQ, false, false);  // S^T, dP^T
            constexpr uint32_t id_kd = idesc_bf16(kBK, D, false, true);     // dV, dK (B MN-major)
            constexpr uint32_t id_qd = idesc_bf16(kBQ, D, true, true);      // dQ (A and B MN-major)
            constexpr uint32_t id_dqt = idesc_bf16(D, kBQ, true, true);     // dQ^T (A and B MN-major)
            const uint32_t s_slot[2] = {smem_u32(smem + L::kK), smem_u32(smem + L::kV)};
            const uint32_t sQ = smem_u32(smem + L::kQ), sDO = smem_u32(smem + L::kDO);
            const uint32_t sDS = smem_u32(smem + L::kDS);
            // Descriptors are built once; each product adds a constant (bytes / 16) to the start field.
            uint64_t k_kmaj = sdesc(s_slot[0], 16, 1024), v_kmaj = sdesc(s_slot[1], 16, 1024);
            const uint64_t q_kmaj = sdesc(sQ, 16, 1024), do_kmaj = sdesc(sDO, 16, 1024);
            const uint64_t q_mn = sdesc(sQ, kBQ * 128, 1024), do_mn = sdesc(sDO, kBQ * 128, 1024);
            const uint64_t ds_mn = sdesc(sDS, kBQ * 128, 1024);
            uint64_t k_mn = sdesc(s_slot[0], kBK * 128, 1024);
            constexpr uint64_t kTileStep = L::kTile >> 4;
            constexpr uint64_t kChunk = (kBQ * 128) >> 4;
            auto issue_s = [&](int st) {  // S^T = K Q^T into ST
                const uint64_t q_k = q_kmaj + st * kTileStep;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (kk / 4) * kChunk + (kk % 4) * 2;
                    mma_ss_w(tmem + kColST, k_kmaj + off, q_k + off, id_kq, kk > 0 ? 1u : 0u);
                }
                mma_commit_w(&bars->s_full);
            };
            auto issue_dp = [&](int so) {  // dP^T = V dO^T into DPT
                const uint64_t do_k = do_kmaj + so * kTileStep;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (kk / 4) * kChunk + (kk % 4) * 2;
                    mma_ss_w(tmem + kColDPT, v_kmaj + off, do_k + off, id_kq, kk > 0 ? 1u : 0u);
                }
                mma_commit_w(&bars->dp_full);
            };
            bool ok = true;
            int gi = 0;  // query blocks processed over all items: the phase of every per-block barrier
            for (int ii = 0; ok; ++ii) {
                const int w = read_item(bars, ii);
                if (w == -2) {
                    ok = false;
                    break;
                }
                if (w < 0) break;
                const BwdItem item = bwd_item<kVarlen>(w, p);
                const int sk = ii & 1, sv = sk ^ 1;
                k_kmaj = sdesc(s_slot[sk], 16, 1024);
                v_kmaj = sdesc(s_slot[sv], 16, 1024);
                k_mn = sdesc(s_slot[sk], kBK * 128, 1024);
                ok = mbar_wait_warp(&bars->kv_full[sk], ii & 1) && !aborted(bars);
                if (!ok) break;
                {
                    // first block of the item: S^T, then dP^T once the previous block's dQ has left DPT
                    const int st = gi % kQStages, so = gi % L::kDOStages;
                    ok = mbar_wait_warp(&bars->q_full[st], (gi / kQStages) & 1) && !aborted(bars);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(st);
                    ok = (kNoDq || gi == 0 || mbar_wait_warp(&bars->dq_empty, (gi - 1) & 1)) &&
                         mbar_wait_warp(&bars->kv_full[sv], ii & 1) &&
                         mbar_wait_warp(&bars->do_full[so], (gi / L::kDOStages) & 1) && !aborted(bars);
                    if (!ok) break;
                    tc_fence_after();
                    issue_dp(so);
                    if (item.n_it == 1) mma_commit_w(&bars->kv_empty[sv]);  // the item's last dP^T is issued
                }
                for (int it = 0; it < item.n_it; ++it, ++gi) {
                    const int st = gi % kQStages, so = gi % L::kDOStages;
                    const uint64_t q_m = q_mn + st * kTileStep, do_m = do_mn + so * kTileStep;
                    // dV += P^T dO  (A = P^T packed in ST, K = 128 queries, 16 per product)
                    ok = mbar_wait_warp(&bars->p_full, gi & 1) && !aborted(bars);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBQ / 16; ++kk) {
                        const uint32_t pc = (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8;  // packed P^T / dS^T columns
                        mma_ts_w(tmem + kColDV, tmem + kColST + pc, do_m + kk * (2048 >> 4), id_kd,
                                 (it > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit_w(&bars->do_empty[so]);  // dO of this block: dP^T and dV were its readers
                    if (L::kTmaReduce && !kNoDq && it + 1 == item.n_it) mma_commit_w(&bars->dv_final);
                    if (kNoDq && it + 1 < item.n_it) {
                        // without the dQ product nothing else waits on this block's DPT, so the next
                        // block's S^T goes into ST right away (dV above was the last reader of P^T) and
                        // the P/dS warps find it ready when they finish this block's dS.  (With dQ, the
                        // next dP^T waits for dQ to leave DPT, and issuing S^T early only moves the wait.)
                        const int st1 = (gi + 1) % kQStages;
                        ok = mbar_wait_warp(&bars->q_full[st1], ((gi + 1) / kQStages) & 1) && !aborted(bars);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(st1);
                    }
                    // dK += dS^T Q  (A = dS^T packed in DPT: reading A from TMEM halves this
                    // product's shared-memory traffic, and shared-memory bandwidth is what the
                    // products of this kernel compete for)
                    ok = mbar_wait_warp(&bars->ds_full, gi & 1) && !aborted(bars);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBQ / 16; ++kk) {
                        const uint32_t pc = (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8;
                        mma_ts_w(tmem + kColDK, tmem + kColDPT + pc, q_m + kk * (2048 >> 4), id_kd,
                                 (it > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit_w(&bars->q_empty[st]);  // Q of this block: S^T and dK were its readers
                    // dQ of this block into DPT (issued after dK, which read dS^T from DPT)
                    if constexpr (kNoDq) {
                    } else if constexpr (D == 128) {
                        // dQ_m^T = K^T dS^T  (M = D lanes, N = queries, K = keys)
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            mma_ss_w(tmem + kColDPT, k_mn + kk * (2048 >> 4), ds_mn + kk * (2048 >> 4), id_dqt,
                                     kk > 0 ? 1u : 0u);
                    } else {
                        // dQ_m = dS K  (M = queries, K = keys, N = D)
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            mma_ss_w(tmem + kColDPT, ds_mn + kk * (2048 >> 4), k_mn + kk * (2048 >> 4), id_qd,
                                     kk > 0 ? 1u : 0u);
                    }
                    if (!kNoDq) mma_commit_w(&bars->dq_full);
                    if (it + 1 < item.n_it) {
                        // next block: S^T into ST right away (dV above was the last reader of P^T);
                        // dP^T into DPT once this block's dQ has been read out
                        const int st1 = (gi + 1) % kQStages, so1 = (gi + 1) % L::kDOStages;
                        if (!kNoDq) {
                            ok = mbar_wait_warp(&bars->q_full[st1], ((gi + 1) / kQStages) & 1) && !aborted(bars);
                            if (!ok) break;
                            tc_fence_after();
                            issue_s(st1);
                        }
                        ok = (kNoDq || mbar_wait_warp(&bars->dq_empty, gi & 1)) &&
                             mbar_wait_warp(&bars->do_full[so1], ((gi + 1) / L::kDOStages) & 1) && !aborted(bars);
                        if (!ok) break;
                        tc_fence_after();
                        issue_dp(so1);
                        if (it + 2 == item.n_it) mma_commit_w(&bars->kv_empty[sv]);  // the item's last dP^T is issued
                    }
                }
                if (!ok) break;
                mma_commit_w(&bars->kv_empty[sk]);  // every product that reads this item's K is issued
                mma_commit_w(&bars->final_);    // DK and DV of this item are complete once these land
            }
            if (!ok) record_timeout(bars, p.err);
            mma_commit_w(&bars->drain);
            mbar_wait_warp(&bars->drain, 0);
        }
    } else if (warp < 4) {
        regs_decrease<56>();
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------ P^T / dS^T (thread = key row)
        regs_increase<152>();
        const int g = (warp - 4) / 4;            // query columns [64 g, 64 g + 64)
        const int tid = threadIdx.x - 128 * (g + 1);
        const int lane_base = 32 * (warp % 4);
        const uint32_t st_addr = tmem + (static_cast<uint32_t>(lane_base) << 16) + kColST;
        const uint32_t dpt_addr = tmem + (static_cast<uint32_t>(lane_base) << 16) + kColDPT;
        uint8_t* ds_row = smem + L::kDS + g * (kBK * 128) + tid * 128;
        const float sl2 = p.scale_log2;
        // row statistics of this warpgroup's 64 queries, loaded one block ahead (across item
        // boundaries too): threads 0-63 fetch lse, threads 64-127 fetch Delta
        const bool fetch_lse = tid < 64;
        const int qoff = 64 * g + (tid & 63);
        auto stat = [&](const BwdItem& item, int i) {  // i: row within the sequence / document
            if (i >= item.len) return fetch_lse ? INFINITY : 0.f;  // past the end: P = 0
            const size_t rowvec = (static_cast<size_t>(item.b) * p.H + item.h) * p.T + item.base;
            return fetch_lse ? p.lse[rowvec + i] * kLog2e : p.delta[rowvec + i];
        };
        bool ok = true;
        bool epi_owed = false;  // thread 0: an epilogue whose store wait and epi_done arrival are still due
        int gi = 0;  // query blocks processed over all items: the phase of every per-block barrier
        for (int ii = 0;; ++ii) {
            const int w = read_item(bars, ii);
            // every warp read the same slot; leave together if any of them timed out
            if (!named_bar_and(1 + g, 128, ok && w != -2)) {
                ok = false;
                record_timeout(bars, p.err);
                break;
            }
            if (w < 0) break;
            const BwdItem item = bwd_item<kVarlen>(w, p);
            const int n = item.n, h = item.h, b = item.b, j0 = item.j0;
            const int j = j0 + tid;
            float nx = stat(item, item.m_lo * kBQ + qoff);
            for (int it = 0; it < item.n_it; ++it, ++gi) {
                const int m = item.m_lo + it;
                const int i0 = m * kBQ;
                (fetch_lse ? s_lse : s_delta)[(gi & 1) * kBQ + qoff] = nx;
                if (it + 1 < item.n_it) nx = stat(item, i0 + kBQ + qoff);
                // the warpgroup leaves together if any of its warps saw a wait run out
                if (!named_bar_and(1 + g, 128, ok)) break;
                const float* lb = s_lse + (gi & 1) * kBQ;
                const float* db = s_delta + (gi & 1) * kBQ;
                const bool full = (n < m) && (i0 + kBQ - 1 - j0 < p.W);
                // phase 1: P^T = exp2(S^T scale log2e - lse log2e) on this warpgroup's 64 queries.
                // The row statistics of the first 32 queries are read before the wait so that their
                // shared-memory latency hides behind it; the second 32 are read while the first are used.
                float4 L4[8];
#pragma unroll
                for (int x4 = 0; x4 < 8; ++x4) L4[x4] = *reinterpret_cast<const float4*>(lb + 64 * g + 4 * x4);
                ok = mbar_wait_warp(&bars->s_full, gi & 1) && !aborted(bars);
                if (!ok) continue;
                tc_fence_after();
                // P^T in bf16, two per word: the same values feed the dV product (through TMEM)
                // and dS below, so both use one rounding of P
                uint32_t pp[32];
                {
                    uint32_t sr[64];
                    {
                        uint32_t a[32], b2[32];
                        tmem_ld32x2(st_addr + 64 * g, st_addr + 64 * g + 32, a, b2);  // one wait for both chunks
#pragma unroll
                        for (int x = 0; x < 32; ++x) {
                            sr[x] = a[x];
                            sr[32 + x] = b2[x];
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int q0 = 64 * g + 32 * c;
#pragma unroll
                        for (int x4 = 0; x4 < 8; ++x4) {
                            const float4 Lq = L4[x4];
                            if (c == 0) L4[x4] = *reinterpret_cast<const float4*>(lb + q0 + 32 + 4 * x4);
                            float e[4];
                            fma_f32x2(e[0], e[1], __uint_as_float(sr[32 * c + 4 * x4]),
                                      __uint_as_float(sr[32 * c + 4 * x4 + 1]), sl2, sl2, -Lq.x, -Lq.y);
                            fma_f32x2(e[2], e[3], __uint_as_float(sr[32 * c + 4 * x4 + 2]),
                                      __uint_as_float(sr[32 * c + 4 * x4 + 3]), sl2, sl2, -Lq.z, -Lq.w);
                            float pr[4];
#pragma unroll
                            for (int y = 0; y < 4; ++y) {
                                pr[y] = ex2_approx(e[y]);
                                if (!full) {
                                    const int i = i0 + q0 + 4 * x4 + y;
                                    if (j > i || i - j >= p.W) pr[y] = 0.f;
                                }
                            }
                            pp[16 * c + 2 * x4] = pack_bf16x2(pr[0], pr[1]);
                            pp[16 * c + 2 * x4 + 1] = pack_bf16x2(pr[2], pr[3]);
                        }
                        // packed into the first half of this warpgroup's own (already read) columns
                        uint32_t pk[16];
#pragma unroll
                        for (int x = 0; x < 16; ++x) pk[x] = pp[16 * c + x];
                        tmem_st16(st_addr + 64 * g + 16 * c, pk);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars->p_full);
                // phase 2: dS^T = P^T (dP^T - Delta), packed into DPT (A operand of dK) and into the
                // shared-memory tile [key][query] (MN-major operand of dQ)
#pragma unroll
                for (int x4 = 0; x4 < 8; ++x4) L4[x4] = *reinterpret_cast<const float4*>(db + 64 * g + 4 * x4);
                ok = mbar_wait_warp(&bars->dp_full, gi & 1) && !aborted(bars);
                // the first dS of an item goes where the previous item's dK (and for D = 64 dV)
                // tile was staged: wait until those TMA stores have read it
                // (without the dQ product the dS tile is not written, and the epilogues alone use it)
                if (!kNoDq && it == 0 && tid == 0 && epi_owed) {
                    // the previous item's dK (and for D = 64 dV) stores have read the dS tile: waited for
                    // only now, so the warpgroup went on to this item's P^T meanwhile
                    bulk_wait_read();
                    mbar_arrive(&bars->epi_done);
                    epi_owed = false;
                }
                if (!kNoDq && ok && it == 0 && ii > 0)
                    ok = mbar_wait_warp(&bars->epi_done, (ii - 1) & 1) && !aborted(bars);
                if (!ok) continue;
                tc_fence_after();
                uint32_t drr[64];
                {
                    uint32_t a[32], b2[32];
                    tmem_ld32x2(dpt_addr + 64 * g, dpt_addr + 64 * g + 32, a, b2);  // one wait for both chunks
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        drr[x] = a[x];
                        drr[32 + x] = b2[x];
                    }
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int q0 = 64 * g + 32 * c;
                    const uint32_t* dr = drr + 32 * c;
                    uint32_t dk[16];
#pragma unroll
                    for (int x4 = 0; x4 < 8; ++x4) {
                        const float4 Dq = L4[x4];
                        if (c == 0) L4[x4] = *reinterpret_cast<const float4*>(db + q0 + 32 + 4 * x4);
                        const uint32_t w0 = pp[16 * c + 2 * x4], w1 = pp[16 * c + 2 * x4 + 1];
                        float t[4], ds[4];
                        add_f32x2(t[0], t[1], __uint_as_float(dr[4 * x4]), __uint_as_float(dr[4 * x4 + 1]), -Dq.x, -Dq.y);
                        add_f32x2(t[2], t[3], __uint_as_float(dr[4 * x4 + 2]), __uint_as_float(dr[4 * x4 + 3]), -Dq.z,
                                  -Dq.w);
                        mul_f32x2(ds[0], ds[1], __uint_as_float(w0 << 16), __uint_as_float(w0 & 0xffff0000u), t[0], t[1]);
                        mul_f32x2(ds[2], ds[3], __uint_as_float(w1 << 16), __uint_as_float(w1 & 0xffff0000u), t[2], t[3]);
                        dk[2 * x4] = pack_bf16x2(ds[0], ds[1]);
                        dk[2 * x4 + 1] = pack_bf16x2(ds[2], ds[3]);
                    }
                    // dS^T (bf16) over this warpgroup's already-read DPT columns, for dK
                    tmem_st16(dpt_addr + 64 * g + 16 * c, dk);
                    // dS row into the [key][query] tile: query chunk g, 16-byte units 4c .. 4c+3
#pragma unroll
                    for (int u = 0; u < (kNoDq ? 0 : 4); ++u) {
                        const int unit = 4 * c + u;
                        uint4 v;
                        v.x = dk[4 * u + 0];
                        v.y = dk[4 * u + 1];
                        v.z = dk[4 * u + 2];
                        v.w = dk[4 * u + 3];
                        *reinterpret_cast<uint4*>(ds_row + ((unit ^ (tid & 7)) << 4)) = v;
                    }
                }
                tmem_wait_st();
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(&bars->ds_full);
            }
            // epilogue: warpgroup 0 writes dK = scale * DK, warpgroup 1 writes dV = DV, each as a
            // 128 x D bf16 tile in shared memory (the 128-byte swizzled layout of the TMA maps)
            // sent out by TMA stores, so the global writes leave as whole lines.  The next
            // item's first dV / dK products overwrite the accumulators only after this
            // warpgroup's next P^T / dS^T arrivals, which come after the reads below.
            // Warpgroup 0 stages dK in the dS tile, free once final_ has landed (dQ and dK were its last
            // readers).  Warpgroup 1 stages dV: for D = 128 with dQ in the dO stage, free once the
            // item's last dV has landed (dv_final, well before final_; the producer loads the next dO
            // after these stores have read it); without dQ in the dQ staging tile; for D = 64 in the
            // second half of the dS tile.
            const bool dv_via_do = L::kTmaReduce && !kNoDq && g == 1;
            if (ok) ok = mbar_wait_warp(dv_via_do ? &bars->dv_final : &bars->final_, ii & 1) && !aborted(bars);
            if (!named_bar_and(1 + g, 128, ok)) {  // leave together
                ok = false;
                record_timeout(bars, p.err);
                break;
            }
            {
                tc_fence_after();
                const uint32_t a = tmem + (static_cast<uint32_t>(lane_base) << 16) + (g ? kColDV : kColDK);
                const float mul = g ? 1.f : p.scale;
                uint8_t* tile = g == 0 ? smem + L::kDS
                                       : (dv_via_do ? smem + L::kDO
                                                    : (L::kTmaReduce ? smem + L::kStage : smem + L::kDS + kBK * 128));
                // a varlen key block that runs past its document's end is written row by row, so the
                // next document's rows are left alone
                const bool partial = kVarlen && j0 + kBK > item.len;
                __nv_bfloat16* grow = (g ? p.dv : p.dk) +
                                      ((static_cast<size_t>(b) * p.T + item.base + j) * p.H + h) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(a + c * 32, r);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint4 pkt;
                        pkt.x = pack_bf16x2(__uint_as_float(r[8 * v4 + 0]) * mul, __uint_as_float(r[8 * v4 + 1]) * mul);
                        pkt.y = pack_bf16x2(__uint_as_float(r[8 * v4 + 2]) * mul, __uint_as_float(r[8 * v4 + 3]) * mul);
                        pkt.z = pack_bf16x2(__uint_as_float(r[8 * v4 + 4]) * mul, __uint_as_float(r[8 * v4 + 5]) * mul);
                        pkt.w = pack_bf16x2(__uint_as_float(r[8 * v4 + 6]) * mul, __uint_as_float(r[8 * v4 + 7]) * mul);
                        // columns 32c + 8 v4 .. +7: 16-byte unit 4 (c % 2) + v4 of the row's 64-column chunk c / 2
                        const int unit = 4 * (c % 2) + v4;
                        if (partial) {
                            if (j < item.len) reinterpret_cast<uint4*>(grow + c * 32)[v4] = pkt;
                        } else {
                            *reinterpret_cast<uint4*>(tile + (c / 2) * (kBK * 128) + tid * 128 + ((unit ^ (tid & 7)) << 4)) =
                                pkt;
                        }
                    }
                }
                fence_async_smem();
                named_bar_sync(1 + g, 128);
                if (tid == 0) {
                    if (!partial) {
                        for (int c = 0; c < D / 64; ++c)
                            tma_store_4d(g ? &tm_dv : &tm_dk, tile + c * (kBK * 128), c * 64, h, item.base + j0, b);
                        bulk_commit();
                    }
                    if (dv_via_do) {
                        bulk_wait_read();
                        mbar_arrive(&bars->do_epi_free);
                    } else if (kNoDq) {
                        bulk_wait_read();
                        // the tile may be written again (the next epilogue) once this is set
                        if (g == 0 || !L::kTmaReduce) mbar_arrive(&bars->epi_done);
                    } else {
                        // the wait for these stores and the epi_done arrival come just before this
                        // warpgroup's next dS, the next write of the dS tile
                        epi_owed = true;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ dQ partials into the fp32 accumulator
        regs_increase<152>();
        if constexpr (kNoDq) {
            // no dQ product: these warps only keep reading the item ring so that its slots are released
            for (int ii = 0;; ++ii) {
                const int w = read_item(bars, ii);
                if (w == -2) record_timeout(bars, p.err);
                if (w < 0) break;
            }
        } else {
        const int tid = threadIdx.x - 384;
        const int lane_base = 32 * (warp % 4);
        const uint32_t st_addr = tmem + (static_cast<uint32_t>(lane_base) << 16) + kColDPT;  // dQ lives in DPT
        bool ok = true;
        int gi = 0;  // query blocks processed over all items
        for (int ii = 0; ok; ++ii) {
            const int w = read_item(bars, ii);
            if (!named_bar_and(3, 128, w != -2)) {  // leave together
                record_timeout(bars, p.err);
                ok = false;
                break;
            }
            if (w < 0) break;
            const BwdItem item = bwd_item<kVarlen>(w, p);
            const int h = item.h, b = item.b, base = item.base;
            for (int it = 0; it < item.n_it; ++it, ++gi) {
                const int i0 = (item.m_lo + it) * kBQ;
                const bool got = mbar_wait_warp(&bars->dq_full, gi & 1) && !aborted(bars);
                if (!named_bar_and(3, 128, got)) {  // leave together
                    record_timeout(bars, p.err);
                    ok = false;
                    break;
                }
                tc_fence_after();
                if constexpr (L::kTmaReduce) {
                    // thread = dQ column d, TMEM columns = the block's 128 query rows.  The whole
                    // block is read into registers first, so the TMEM columns go back to the MMA
                    // warp (for the next dP^T) before any of the staging work.  Each half (64 rows)
                    // then goes to the fp32 staging tile [row][d] and is added to the accumulator by
                    // one TMA reduce-add, which keeps the SM's load/store path free.
                    float* stage = reinterpret_cast<float*>(smem + L::kStage);
                    uint32_t r0[64], r1[64];
                    tmem_ld64_nowait(st_addr, r0);
                    tmem_ld64_nowait(st_addr + 64, r1);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(&bars->dq_empty);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        if (tid == 0) bulk_wait_read();  // the previous reduce-add has read the staging tile
                        named_bar_sync(3, 128);
#pragma unroll
                        for (int x = 0; x < 64; ++x) stage[x * D + tid] = __uint_as_float(half ? r1[x] : r0[x]);
                        fence_async_smem();
                        named_bar_sync(3, 128);
                        if (tid == 0) {
                            // rows past a varlen document's end carry exact zeros (P = 0 there)
                            tma_reduce_add_4d(&tm_dq, stage, 0, h, base + i0 + 64 * half, b);
                            bulk_commit();
                        }
                    }
                } else {
                    // thread = query row, TMEM columns = the D dQ columns
                    uint32_t r[64];
                    {
                        uint32_t a[32], c2[32];
                        tmem_ld32x2(st_addr, st_addr + 32, a, c2);
#pragma unroll
                        for (int x = 0; x < 32; ++x) {
                            r[x] = a[x];
                            r[32 + x] = c2[x];
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(&bars->dq_empty);
                    // the block's 128 rows into the staging tile (box c: columns 32c .. 32c+31, 128 bytes a row, its
                    // 16-byte units in the 128-byte swizzle), then one reduce-add per box.  Rows past a varlen
                    // document's end carry exact zeros (P = 0 there); rows past the tensor are clipped by the copy.
                    uint8_t* stage = smem + L::kStage;
                    if (tid == 0) bulk_wait_read();  // the previous reduce-adds have read the staging tile
                    named_bar_sync(3, 128);
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            *reinterpret_cast<uint4*>(stage + c * (kBQ * 128) + tid * 128 + ((u ^ (tid & 7)) << 4)) =
                                make_uint4(r[32 * c + 4 * u], r[32 * c + 4 * u + 1], r[32 * c + 4 * u + 2],
                                           r[32 * c + 4 * u + 3]);
                    fence_async_smem();
                    named_bar_sync(3, 128);
                    if (tid == 0) {
                        for (int c = 0; c < 2; ++c) tma_reduce_add_4d(&tm_dq, stage + c * (kBQ * 128), 32 * c, h, base + i0, b);
                        bulk_commit();
                    }
                }
            }
        }
        if constexpr (L::kTmaReduce || L::kStagedRows) {
            if (tid == 0) bulk_wait_all();  // every reduce-add has landed before the CTA exits
        }
        }
    }
    if (warp >= 4 && warp < 12 && (threadIdx.x & 127) == 0) bulk_wait_all();  // epilogue stores have landed
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Delta = rowsum(dO * O) per (b, h, i), a zeroed dQ accumulator (unless dq_acc is null) and zeroed
// work-item counters (work[0] for the main kernel, work[1] for the deterministic dQ pass).  Packed documents
// with the deterministic dQ pass (cu != nullptr): dq rows outside [cu[0], cu[n_docs]) are zeroed here, since
// that pass writes only the documents' rows.
// D / 8 lanes per row, each with one 16-byte load of O and of dO.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dO,
                                                      float* __restrict__ delta, float* __restrict__ dq_acc,
                                                      int* __restrict__ work, int B, int T, int H,
                                                      __nv_bfloat16* __restrict__ dq, const int* __restrict__ cu,
                                                      int n_docs) {
    constexpr int G = D / 8;          // lanes per row
    constexpr int RPW = 32 / G;       // rows per warp
    const long tid_g = (long)blockIdx.x * blockDim.x + threadIdx.x;
    const long row = (tid_g >> 5) * RPW + ((threadIdx.x & 31) / G);
    const int c = threadIdx.x % G;
    const long rows = (long)B * T * H;
    if (tid_g == 0) {
        work[0] = 0;
        work[1] = 0;
    }
    float acc = 0.f;
    if (row < rows) {
        const uint4 a = reinterpret_cast<const uint4*>(o + (size_t)row * D)[c];
        const uint4 g = reinterpret_cast<const uint4*>(dO + (size_t)row * D)[c];
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(a2[e]), y = __bfloat1622float2(g2[e]);
            acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
        }
        if (dq_acc != nullptr) {
            float4* z = reinterpret_cast<float4*>(dq_acc + (size_t)row * D + c * 8);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    if (cu != nullptr && row < rows) {
        const long i = row / H;  // B = 1
        if (i < __ldg(cu) || i >= __ldg(cu + n_docs))
            reinterpret_cast<uint4*>(dq + (size_t)row * D)[c] = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && c == 0) {
        const int h = row % H;
        const int i = (row / H) % T;
        const int b = row / ((long)H * T);
        delta[((size_t)b * H + h) * T + i] = acc;
    }
}

// dq = bf16(scale * dQ accumulator), 8 elements per thread.
__global__ void __launch_bounds__(256) bwd_post_kernel(const float* __restrict__ dq_acc,
                                                       __nv_bfloat16* __restrict__ dq, size_t n8, float scale) {
    const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n8) return;
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * t];
    const float4 c = reinterpret_cast<const float4*>(dq_acc)[2 * t + 1];
    uint4 pkt;
    pkt.x = pack_bf16x2(a.x * scale, a.y * scale);
    pkt.y = pack_bf16x2(a.z * scale, a.w * scale);
    pkt.z = pack_bf16x2(c.x * scale, c.y * scale);
    pkt.w = pack_bf16x2(c.z * scale, c.w * scale);
    reinterpret_cast<uint4*>(dq)[t] = pkt;
}

// Rotary variant of the conversion pass.  The main kernel ran on the turned rows qr, kr, so its dQ
// accumulator and dk hold gradients with respect to the turned q and k; both are turned back here by the
// transpose of row t's rotation (x1 = y1 c + y2 s, x2 = y2 c - y1 s, with the turn's explicit roundings):
// dq = bf16(scale * turned-back accumulator), dk turned back in place.  One thread per (row, 8 pairs):
// dimensions 8u .. 8u+7 and their partners 8u + D/2 ..; the table entries are read once for both.
template <int D>
__global__ void __launch_bounds__(256) bwd_post_rope_kernel(const float* __restrict__ dq_acc,
                                                            __nv_bfloat16* __restrict__ dq, __nv_bfloat16* dk,
                                                            const float* __restrict__ rcos,
                                                            const float* __restrict__ rsin, size_t n_units, int T,
                                                            int H, float scale) {
    constexpr int kUnits = D / 16;
    const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n_units) return;
    const size_t row = t / kUnits;
    const int u = static_cast<int>(t - row * kUnits);
    const int pos = static_cast<int>((row / H) % T);
    const size_t e1 = row * D + 8 * u, e2 = e1 + D / 2;  // first element of the unit and of its partners
    const float4 a0 = *reinterpret_cast<const float4*>(dq_acc + e1);
    const float4 a1 = *reinterpret_cast<const float4*>(dq_acc + e1 + 4);
    const float4 b0 = *reinterpret_cast<const float4*>(dq_acc + e2);
    const float4 b1 = *reinterpret_cast<const float4*>(dq_acc + e2 + 4);
    const uint4 k1 = *reinterpret_cast<const uint4*>(dk + e1);
    const uint4 k2 = *reinterpret_cast<const uint4*>(dk + e2);
    const float4 c0 = __ldg(reinterpret_cast<const float4*>(rcos + (size_t)pos * (D / 2) + 8 * u));
    const float4 c1 = __ldg(reinterpret_cast<const float4*>(rcos + (size_t)pos * (D / 2) + 8 * u) + 1);
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(rsin + (size_t)pos * (D / 2) + 8 * u));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(rsin + (size_t)pos * (D / 2) + 8 * u) + 1);
    const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const float q1[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float q2[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const uint32_t kw1[4] = {k1.x, k1.y, k1.z, k1.w}, kw2[4] = {k2.x, k2.y, k2.z, k2.w};
    uint32_t oq1[4], oq2[4], ok1[4], ok2[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float r1[2], r2[2], t1[2], t2[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int e = 2 * w + h2;
            r1[h2] = __fmaf_rn(q1[e], cv[e], __fmul_rn(q2[e], sv[e])) * scale;
            r2[h2] = __fmaf_rn(q2[e], cv[e], -__fmul_rn(q1[e], sv[e])) * scale;
            const float y1 = __uint_as_float(h2 ? (kw1[w] & 0xffff0000u) : (kw1[w] << 16));
            const float y2 = __uint_as_float(h2 ? (kw2[w] & 0xffff0000u) : (kw2[w] << 16));
            t1[h2] = __fmaf_rn(y1, cv[e], __fmul_rn(y2, sv[e]));
            t2[h2] = __fmaf_rn(y2, cv[e], -__fmul_rn(y1, sv[e]));
        }
        oq1[w] = pack_bf16x2(r1[0], r1[1]);
        oq2[w] = pack_bf16x2(r2[0], r2[1]);
        ok1[w] = pack_bf16x2(t1[0], t1[1]);
        ok2[w] = pack_bf16x2(t2[0], t2[1]);
    }
    *reinterpret_cast<uint4*>(dq + e1) = make_uint4(oq1[0], oq1[1], oq1[2], oq1[3]);
    *reinterpret_cast<uint4*>(dq + e2) = make_uint4(oq2[0], oq2[1], oq2[2], oq2[3]);
    *reinterpret_cast<uint4*>(dk + e1) = make_uint4(ok1[0], ok1[1], ok1[2], ok1[3]);
    *reinterpret_cast<uint4*>(dk + e2) = make_uint4(ok2[0], ok2[1], ok2[2], ok2[3]);
}

// cu != nullptr: document-masked packed rows (B = 1, T = total), n_docs documents of at most max_len rows.
// deterministic: dK and dV from the main kernel, dQ from the query-stationary pass (no dQ accumulator).
template <int D>
cudaError_t launch_bwd_tc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                          const float* lse, void* dq, void* dk, void* dv, int B, int T, int H, int window,
                          float scale, float* dq_acc, float* delta, int* work, const int* cu, int n_docs,
                          int max_len, int* err, cudaStream_t st, bool deterministic = false,
                          const float* rcos = nullptr, const float* rsin = nullptr) {
    CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
    if (!make_tmap_bthd(&tq, q, B, T, H, D, 64, kBQ) || !make_tmap_bthd(&tk, k, B, T, H, D, 64, kBK) ||
        !make_tmap_bthd(&tv, v, B, T, H, D, 64, kBK) || !make_tmap_bthd(&tdo, dO, B, T, H, D, 64, kBQ) ||
        !make_tmap_bthd(&tdk, dk, B, T, H, D, 64, kBK) || !make_tmap_bthd(&tdv, dv, B, T, H, D, 64, kBK) ||
        !(D == 128 ? make_tmap_bthd_f32(&tdq, dq_acc, B, T, H, D, D, BwdSmem<D>::kStageRows)
                   : make_tmap_bthd_f32(&tdq, dq_acc, B, T, H, D, 32, kBQ, true)))
        return cudaErrorInvalidValue;
    const long rows = (long)B * T * H;
    const long pre_threads = ((rows * (D / 8) + 31) / 32) * 32;
    bwd_pre_kernel<D><<<(unsigned)((pre_threads + 255) / 256), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), delta,
        deterministic ? nullptr : dq_acc, work, B, T, H, static_cast<__nv_bfloat16*>(dq),
        deterministic ? cu : nullptr, n_docs);
    BwdParams p;
    p.lse = lse;
    p.delta = delta;
    p.dq_acc = dq_acc;
    p.dk = static_cast<__nv_bfloat16*>(dk);
    p.dv = static_cast<__nv_bfloat16*>(dv);
    p.B = B;
    p.T = T;
    p.H = H;
    p.W = (window <= 0 || window >= T) ? T : window;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.n_kb = ((cu != nullptr ? max_len : T) + kBK - 1) / kBK;
    p.n_qb = (T + kBQ - 1) / kBQ;
    p.work = work;
    p.cu = cu;
    p.n_docs = n_docs;
    p.err = err;
    const int smem = BwdSmem<D>::kBytes;
    // the shared-memory limit is raised once per device and variant (atomic flags), the SM count
    // is looked up on every call
    static std::atomic<bool> attr_done[4][kAttrDevices];
    const int variant = deterministic ? (cu != nullptr ? 3 : 2) : (cu != nullptr ? 1 : 0);
    auto kern = variant == 3   ? bwd_main_kernel<D, true, true>
                : variant == 2 ? bwd_main_kernel<D, false, true>
                               : (variant == 1 ? bwd_main_kernel<D, true> : bwd_main_kernel<D, false>);
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem, attr_done[variant]);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM (its shared memory and TMEM allow one), looping over the items
    int n_sm = 0;
    e = multiprocessor_count(&n_sm);
    if (e != cudaSuccess) return e;
    const int n_pairs = (cu != nullptr ? n_docs : B) * H;
    const long n_items = (long)p.n_kb * n_pairs;
    const int grid = (int)(n_items < n_sm ? n_items : n_sm);
    // a scheduling group holds about one wave of items
    p.group = (n_sm + p.n_kb - 1) / p.n_kb;
    if (p.group > n_pairs) p.group = n_pairs;
    kern<<<grid, kThreads, smem, st>>>(tq, tk, tv, tdo, tdq, tdk, tdv, p);
    if (deterministic) {
        count_launches(2);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return launch_bwd_dq(q, k, v, dO, lse, delta, dq, B, T, H, D, window, scale, work + 1, err, st, cu, n_docs,
                             max_len);
    }
    if (rcos != nullptr) {
        const size_t nu = (size_t)rows * (D / 16);
        bwd_post_rope_kernel<D><<<(unsigned)((nu + 255) / 256), 256, 0, st>>>(
            dq_acc, static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk), rcos, rsin, nu, T, H, scale);
        count_launches(3);
        return cudaGetLastError();
    }
    const size_t n8 = (size_t)rows * D / 8;
    bwd_post_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, st>>>(dq_acc, static_cast<__nv_bfloat16*>(dq), n8,
                                                                 scale);
    count_launches(3);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                       void* dq, void* dk, void* dv, int B, int T, int H, int D, int window, float scale,
                       float* dq_acc, float* delta, int* work, int* err, cudaStream_t st) {
    return D == 128 ? launch_bwd_tc<128>(q, k, v, o, dO, lse, dq, dk, dv, B, T, H, window, scale, dq_acc, delta, work,
                                         nullptr, 0, 0, err, st)
                    : launch_bwd_tc<64>(q, k, v, o, dO, lse, dq, dk, dv, B, T, H, window, scale, dq_acc, delta, work,
                                        nullptr, 0, 0, err, st);
}

cudaError_t launch_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, const int* cu, int n_docs, int max_len, void* dq, void* dk, void* dv,
                              int total, int H, int D, int window, float scale, float* dq_acc, float* delta, int* work,
                              int* err, cudaStream_t st, bool deterministic) {
    return D == 128 ? launch_bwd_tc<128>(q, k, v, o, dO, lse, dq, dk, dv, 1, total, H, window, scale, dq_acc, delta,
                                         work, cu, n_docs, max_len, err, st, deterministic)
                    : launch_bwd_tc<64>(q, k, v, o, dO, lse, dq, dk, dv, 1, total, H, window, scale, dq_acc, delta,
                                        work, cu, n_docs, max_len, err, st, deterministic);
}

cudaError_t launch_bwd_rotary(const void* qr, const void* kr, const void* v, const float* rcos, const float* rsin,
                              const void* o, const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                              int T, int H, int D, int window, float scale, float* dq_acc, float* delta, int* work,
                              int* err, cudaStream_t st) {
    return D == 128 ? launch_bwd_tc<128>(qr, kr, v, o, dO, lse, dq, dk, dv, B, T, H, window, scale, dq_acc, delta,
                                         work, nullptr, 0, 0, err, st, false, rcos, rsin)
                    : launch_bwd_tc<64>(qr, kr, v, o, dO, lse, dq, dk, dv, B, T, H, window, scale, dq_acc, delta,
                                        work, nullptr, 0, 0, err, st, false, rcos, rsin);
}

cudaError_t launch_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                     const float* lse, void* dq, void* dk, void* dv, int B, int T, int H, int D,
                                     int window, float scale, float* dq_acc, float* delta, int* work, int* err,
                                     cudaStream_t st) {
    return D == 128 ? launch_bwd_tc<128>(q, k, v, o, dO, lse, dq, dk, dv, B, T, H, window, scale, dq_acc, delta, work,
                                         nullptr, 0, 0, err, st, true)
                    : launch_bwd_tc<64>(q, k, v, o, dO, lse, dq, dk, dv, B, T, H, window, scale, dq_acc, delta, work,
                                        nullptr, 0, 0, err, st, true);
}

}  // namespace nc
