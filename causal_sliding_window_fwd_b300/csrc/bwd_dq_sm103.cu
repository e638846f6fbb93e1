// Deterministic dQ pass of the backward on 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Operation (see include/nc_attn.h, nc_attn_bwd_deterministic): the same gradient as the main
// backward, dQ_i = scale * sum_j dS_ij k_j with dS = P * (dP - Delta), but every 128-row query
// block is owned by one CTA that walks its key blocks in a fixed order and accumulates dQ in TMEM.
// The result therefore does not depend on which CTA runs when (the main backward adds the
// partials of different key blocks with reduce-adds in whatever order they arrive).  The pass
// recomputes S = Q K^T and dP = dO V^T for every visible (query block, key block) pair: two
// products more per pair than the main pass, which in this mode computes only dK and dV.
//
// Persistent CTAs (one per SM, 384 threads).  A work item is one query block m of one
// (batch, head); the producer warp takes item indices from a global counter and publishes them
// in a shared-memory ring.  Packed documents (kVarlen): the pairs are (document, head), positions
// count from the document's first row, and the producer passes over items past a document's end.  Indices run over groups of about one wave of items; inside a group
// m runs outermost from the last block down (the longest causal walks first), so the CTAs that
// run at the same time read the K and V of a few heads and share them in L2.  Warp roles:
//   warp 0      TMA producer: Q and dO of the item once, then K blocks through a 3-slot ring and V
//               blocks through a 2-slot ring (V is free once dP has read it, K only after dQ)
//   warp 1      MMA issuer (one lane) and TMEM owner
//   warps 4-7   one thread per query row, key columns [0, 64): P, dS; then dQ columns [0, D/2)
//   warps 8-11  the same for key columns [64, 128); then dQ columns [D/2, D)
// TMEM: ST [0,128) holds S; DP0 [128,256) and DP1 [384,512) hold dP of alternate key blocks,
// then dS packed as bf16 over the columns each warpgroup has already read (the A operand of
// dQ += dS K); DQ [256,256+D) accumulates dQ.
// Products for key block j: once the P/dS warps have read S(j) out of TMEM, S(j+1) into ST and
// dP(j+1) into the other DP region (they run while the warps compute P(j) and dS(j)); once dS(j)
// is in TMEM, dQ += dS(j) K(j).  An item's dQ is written out after the next item's first dS.
#include <cstdint>
#include <cuda_bf16.h>

#include "nc_attn.h"
#include "nc_kernels.h"
#include "nc_ptx.cuh"
#include "nc_sched.cuh"
#include "nc_tma.h"

namespace nc {
namespace {

constexpr int kBQ = 128;        // query rows per block
constexpr int kBK = 128;        // keys per block
constexpr int kKStages = 3;     // K ring slots
constexpr int kVStages = 2;     // V ring slots
constexpr int kThreads = 384;
constexpr int kItemReaders = 9; // warps that read each work-item slot: the MMA warp and 8 P/dS warps
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DqSmem {
    static constexpr int kTile = kBQ * D * 2;  // one 128-row bf16 tile
    static constexpr int kQ = 0;
    static constexpr int kDO = kQ + kTile;
    static constexpr int kK = kDO + kTile;     // kKStages tiles
    static constexpr int kV = kK + kKStages * kTile;  // kVStages tiles
    static constexpr int kBytes = kV + kVStages * kTile;
};

struct DqBarriers {
    uint64_t k_full[kKStages];
    uint64_t k_empty[kKStages];
    uint64_t v_full[kVStages];
    uint64_t v_empty[kVStages];
    uint64_t q_full;
    uint64_t q_empty;
    uint64_t s_full;
    uint64_t s_free;
    // one per DP region (block parity): dP(j+1) lands before the P/dS warps wait for dP(j), so a
    // single barrier could complete two phases ahead of its waiter
    uint64_t dp_full[2];
    uint64_t ds_full[2];
    uint64_t dq_final;
    uint64_t dq_free;   // the P/dS warps have read DQ out (the next item's first dQ product may overwrite it)
    uint64_t drain;
    uint64_t item_full[kItemSlots];
    uint64_t item_empty[kItemSlots];
    int item[kItemSlots];
    uint32_t tmem_base;
    int abort;
};

struct DqParams {
    const float* lse;    // [B, H, T]
    const float* delta;  // [B, H, T]
    __nv_bfloat16* dq;   // [B, T, H, D]
    int B, T, H, W;      // W effective, 1 <= W <= T
    float scale, scale_log2;
    int n_qb;
    int group;           // (batch, head) pairs per scheduling group
    bool dq32;           // dq is 32-byte aligned: the epilogue writes whole 32-byte sectors
    int* work;           // work-item counter, zero on entry
    int* err;
    // packed documents (B = 1, T = total): document d is rows cu[d] .. cu[d+1]-1; n_qb counts the query
    // blocks of the longest document.  nullptr otherwise.
    const int* cu;
    int n_docs;
};

// One item: query block m of one (batch, head) -- or (document, head) -- and the key blocks n_lo .. m
// that its window reaches.
struct DqItem {
    int m, h, b, n_lo;
    int base;    // first packed row of the document, else 0
    int len;     // rows of the sequence or document
    bool bad;    // the document's bounds are out of range
    bool empty;  // the block lies past the document's end (or the document is bad)
};

template <bool kVarlen>
__device__ __forceinline__ DqItem dq_item(int w, const DqParams& p) {
    DqItem it;
    const int n_pairs = (kVarlen ? p.n_docs : p.B) * p.H;
    const int per_group = p.n_qb * p.group;
    const int grp = w / per_group, r = w - grp * per_group;
    const int in_grp = min(p.group, n_pairs - grp * p.group);  // the last group may be short
    const int bh = grp * p.group + r % in_grp;
    it.m = p.n_qb - 1 - r / in_grp;
    it.h = bh % p.H;
    it.b = kVarlen ? 0 : bh / p.H;
    it.base = 0;
    it.len = p.T;
    it.bad = false;
    it.empty = false;
    if (kVarlen) {
        const int d = bh / p.H;
        const int a = p.cu[d], e = p.cu[d + 1];
        it.bad = a < 0 || e < a || e > p.T || e - a > p.n_qb * kBQ;
        it.base = it.bad ? 0 : a;
        it.len = it.bad ? 0 : e - a;
        it.empty = it.bad || it.m * kBQ >= it.len;
    }
    // the earliest key any row of the block sees is m*128 - W + 1; key block n holds one of
    // those keys iff n*128 + 127 >= m*128 - W + 1
    const int x = it.m * kBQ - p.W - (kBK - 2);
    it.n_lo = x <= 0 ? 0 : (x + kBK - 1) / kBK;
    return it;
}

__device__ __forceinline__ bool aborted(const DqBarriers& bars) {
    return *reinterpret_cast<const volatile int*>(&bars.abort) != 0;
}

__device__ __forceinline__ void record_timeout(DqBarriers& bars, int* err) {
    set_device_error(err, NC_ERR_DEVICE_TIMEOUT);
    atomicExch(&bars.abort, 1);
}

// Producer (converged warp): the next item index into ring slot k; with packed documents, indices of empty
// items are passed over (and bad document bounds reported) so the other roles only see items with work.
// -1 once every item is taken, -2 if the wait for the slot ran out.
template <bool kVarlen>
__device__ __forceinline__ int publish_dq_item(DqBarriers& bars, int k, int n_items, const DqParams& p) {
    if (!kVarlen) return ring_publish_item(bars.item_full, bars.item_empty, bars.item, k, n_items, p.work);
    const int slot = k % kItemSlots;
    if (!mbar_wait_warp(&bars.item_empty[slot], ((k / kItemSlots) & 1) ^ 1)) return -2;
    int w = 0;
    if (lane_id() == 0) {
        for (;;) {
            w = atomicAdd(p.work, 1);
            if (w >= n_items) {
                w = -1;
                break;
            }
            const DqItem it = dq_item<kVarlen>(w, p);
            if (it.bad) set_device_error(p.err, NC_ERR_BAD_SEQLENS);
            if (!it.empty) break;
        }
        bars.item[slot] = w;
        mbar_arrive(&bars.item_full[slot]);
    }
    return __shfl_sync(0xffffffffu, w, 0);
}

template <int D, bool kVarlen>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do, const DqParams p) {
    using L = DqSmem<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ DqBarriers bars;
    const int warp = warp_id(), lane = lane_id();
    const int n_items = p.n_qb * p.H * (kVarlen ? p.n_docs : p.B);

    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) set_device_error(p.err, NC_ERR_CUDA);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.v_empty[s], 1);
        }
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        mbar_init(&bars.s_full, 1);
        mbar_init(&bars.s_free, 2 * kBQ);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.dp_full[s], 1);
            mbar_init(&bars.ds_full[s], 2 * kBQ);
        }
        mbar_init(&bars.dq_final, 1);
        mbar_init(&bars.dq_free, 2 * kBQ);
        mbar_init(&bars.drain, 1);
        for (int s = 0; s < kItemSlots; ++s) {
            mbar_init(&bars.item_full[s], 1);
            mbar_init(&bars.item_empty[s], kItemReaders);
        }
        bars.abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    constexpr uint32_t kColST = 0, kColDQ = 256;
    auto col_dp = [](int gj) -> uint32_t { return (gj & 1) ? 384u : 128u; };

    // registers: 384 threads x 168 at launch = 128 x 72 (producer / MMA warpgroup) + 256 x 216 (P/dS)
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // the whole warp runs this loop converged; lane 0 issues each copy
        regs_decrease<72>();
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_do);
        }
        __syncwarp();
        int seq = 0, q_loads = 0, k_loads = 0, v_loads = 0;
        bool ok = true;
        for (int ii = 0; ok; ++ii) {
            const int w = publish_dq_item<kVarlen>(bars, ii, n_items, p);
            if (w == -2 || aborted(bars)) {
                ok = false;
                break;
            }
            if (w < 0) break;
            const DqItem it = dq_item<kVarlen>(w, p);
            // Q and dO of this item once the previous item's S and dP products have read theirs
            if (!mbar_wait_warp(&bars.q_empty, (ii & 1) ^ 1) || aborted(bars)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx_w(&bars.q_full, 2 * L::kTile);
            for (int c = 0; c < D / 64; ++c) {
                tma_load_4d_w(smem + L::kQ + c * kBQ * 128, &tm_q, &bars.q_full, c * 64, it.h,
                              it.base + it.m * kBQ, it.b);
                tma_load_4d_w(smem + L::kDO + c * kBQ * 128, &tm_do, &bars.q_full, c * 64, it.h,
                              it.base + it.m * kBQ, it.b);
            }
            ++q_loads;
            for (int n = it.n_lo; n <= it.m; ++n, ++seq) {
                const int ks = seq % kKStages, vs = seq % kVStages;
                if (!mbar_wait_warp(&bars.k_empty[ks], ((seq / kKStages) & 1) ^ 1) || aborted(bars)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_w(&bars.k_full[ks], L::kTile);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d_w(smem + L::kK + ks * L::kTile + c * kBK * 128, &tm_k, &bars.k_full[ks], c * 64, it.h,
                                  it.base + n * kBK, it.b);
                ++k_loads;
                if (!mbar_wait_warp(&bars.v_empty[vs], ((seq / kVStages) & 1) ^ 1) || aborted(bars)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_w(&bars.v_full[vs], L::kTile);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d_w(smem + L::kV + vs * L::kTile + c * kBK * 128, &tm_v, &bars.v_full[vs], c * 64, it.h,
                                  it.base + n * kBK, it.b);
                ++v_loads;
            }
        }
        if (!ok) record_timeout(bars, p.err);
        // never leave while a copy into this CTA's shared memory may still land: the last use of
        // each slot is the only one whose completion can still be outstanding
        for (int x = k_loads - kKStages < 0 ? 0 : k_loads - kKStages; x < k_loads; ++x)
            mbar_wait_warp(&bars.k_full[x % kKStages], (x / kKStages) & 1);
        for (int x = v_loads - kVStages < 0 ? 0 : v_loads - kVStages; x < v_loads; ++x)
            mbar_wait_warp(&bars.v_full[x % kVStages], (x / kVStages) & 1);
        if (q_loads > 0) mbar_wait_warp(&bars.q_full, (q_loads - 1) & 1);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs this loop converged; lane 0 issues each product
        regs_decrease<72>();
        constexpr uint32_t id_qk = idesc_bf16(kBQ, kBK, false, false);  // S, dP (both operands K-major)
        constexpr uint32_t id_dq = idesc_bf16(kBQ, D, false, true);     // dQ (A from TMEM, B MN-major)
        const uint32_t sQ = smem_u32(smem + L::kQ), sDO = smem_u32(smem + L::kDO);
        const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
        // descriptors are built once; each product adds a constant (bytes / 16) to the start field
        const uint64_t q_kmaj = sdesc(sQ, 16, 1024), do_kmaj = sdesc(sDO, 16, 1024);
        const uint64_t k_kmaj = sdesc(sK, 16, 1024), v_kmaj = sdesc(sV, 16, 1024);
        const uint64_t k_mn = sdesc(sK, kBK * 128, 1024);
        constexpr uint64_t kTileStep = L::kTile >> 4;
        constexpr uint64_t kChunk = (kBQ * 128) >> 4;
        // S = Q K^T into ST, then dP = dO V^T into the DP region of block gb (ring position sq)
        auto issue_s_dp = [&](int sq, int gb) -> bool {
            const uint32_t dp_col = col_dp(gb);
            const int ks = sq % kKStages, vs = sq % kVStages;
            if (!mbar_wait_warp(&bars.k_full[ks], (sq / kKStages) & 1) || aborted(bars)) return false;
            tc_fence_after();
            const uint64_t kd = k_kmaj + ks * kTileStep;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = (kk / 4) * kChunk + (kk % 4) * 2;
                mma_ss_w(tmem + kColST, q_kmaj + off, kd + off, id_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&bars.s_full);
            if (!mbar_wait_warp(&bars.v_full[vs], (sq / kVStages) & 1) || aborted(bars)) return false;
            tc_fence_after();
            const uint64_t vd = v_kmaj + vs * kTileStep;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = (kk / 4) * kChunk + (kk % 4) * 2;
                mma_ss_w(tmem + dp_col, do_kmaj + off, vd + off, id_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&bars.dp_full[gb & 1]);
            mma_commit_w(&bars.v_empty[vs]);  // dP was the only reader of this V block
            return true;
        };
        bool ok = true;
        int seq = 0, gj = 0;  // K/V ring position; key blocks processed over all items (barrier phases)
        for (int ii = 0; ok; ++ii) {
            const int w = ring_read_item(bars.item_full, bars.item_empty, bars.item, ii);
            if (w == -2) {
                ok = false;
                break;
            }
            if (w < 0) break;
            const DqItem it = dq_item<kVarlen>(w, p);
            ok = mbar_wait_warp(&bars.q_full, ii & 1) && issue_s_dp(seq, gj);
            if (!ok) break;
            if (it.n_lo == it.m) mma_commit_w(&bars.q_empty);  // every S and dP of this item is issued
            for (int n = it.n_lo; n <= it.m; ++n, ++seq, ++gj) {
                const int ks = seq % kKStages;
                if (n < it.m) {
                    // S(j) has been read out of ST.  (The wait is skipped for an item's last block;
                    // its phase is then passed over, never overtaken: the next arrival needs the
                    // next item's first S, issued after this block's dS.)
                    ok = mbar_wait_warp(&bars.s_free, gj & 1) && !aborted(bars);
                    if (!ok) break;
                    tc_fence_after();
                    ok = issue_s_dp(seq + 1, gj + 1);
                    if (!ok) break;
                    if (n + 1 == it.m) mma_commit_w(&bars.q_empty);
                }
                // dS(j) is in TMEM, and dP(j) has been read
                ok = mbar_wait_warp(&bars.ds_full[gj & 1], (gj >> 1) & 1) && !aborted(bars);
                if (!ok) break;
                tc_fence_after();
                if (n == it.n_lo && ii > 0) {
                    // the first product of an item overwrites DQ: the P/dS warps have read the previous
                    // item's dQ out (they do so after this item's first dS)
                    ok = mbar_wait_warp(&bars.dq_free, (ii - 1) & 1) && !aborted(bars);
                    if (!ok) break;
                    tc_fence_after();
                }
                // dQ += dS K(j)  (A = dS packed in DP: keys 0-63 in columns [0,32), 64-127 in [64,96))
                const uint64_t kmn = k_mn + ks * kTileStep;
                const uint32_t a = tmem + col_dp(gj);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint32_t pc = (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8;
                    mma_ts_w(tmem + kColDQ, a + pc, kmn + kk * (2048 >> 4), id_dq, (n > it.n_lo || kk > 0) ? 1u : 0u);
                }
                mma_commit_w(&bars.k_empty[ks]);  // K(j): S and dQ were its readers
            }
            if (!ok) break;
            mma_commit_w(&bars.dq_final);
        }
        if (!ok) record_timeout(bars, p.err);
        mma_commit_w(&bars.drain);
        mbar_wait_warp(&bars.drain, 0);
    } else if (warp < 4) {
        regs_decrease<72>();
    } else {
        // ------------------------------------------------------------ P and dS (thread = query row)
        regs_increase<216>();
        const int g = (warp - 4) / 4;  // key columns [64 g, 64 g + 64)
        const int tid = threadIdx.x - 128 * (g + 1);
        const uint32_t lanes = static_cast<uint32_t>(32 * (warp % 4)) << 16;
        const float sl2 = p.scale_log2;
        // epilogue of an item: dq = bf16(scale * DQ); warpgroup g writes dQ columns [g D/2, (g+1) D/2) of its
        // row.  It runs after the next item's first dS, so the MMA warp has that block's S and dP products to
        // run meanwhile; dq_free then lets the next item's first dQ product overwrite DQ.
        auto epilogue = [&](const DqItem& item, int ie) -> bool {
            const int i = item.m * kBQ + tid;  // row within the sequence or document
            const bool row_ok = i < item.len;  // (a document's last block: the next document's rows are left alone)
            if (!(mbar_wait_warp(&bars.dq_final, ie & 1) && !aborted(bars))) return false;
            tc_fence_after();
            __nv_bfloat16* drow =
                p.dq + ((static_cast<size_t>(item.b) * p.T + item.base + (row_ok ? i : 0)) * p.H + item.h) * D +
                g * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lanes + kColDQ + g * (D / 2) + c * 32, r);
                uint32_t w[16];
#pragma unroll
                for (int x = 0; x < 16; ++x)
                    w[x] = pack_bf16x2(__uint_as_float(r[2 * x]) * p.scale, __uint_as_float(r[2 * x + 1]) * p.scale);
                if (row_ok) {
                    if (p.dq32) {
                        st_global_v8(drow + c * 32, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                        st_global_v8(drow + c * 32 + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
                    } else {
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            reinterpret_cast<uint4*>(drow + c * 32)[v4] =
                                make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bars.dq_free);
            return true;
        };
        bool ok = true;
        int gj = 0;
        bool have_prev = false;  // an item whose dQ still waits in TMEM
        DqItem prev{};
        int prev_ii = 0;
        for (int ii = 0; ok; ++ii) {
            const int w = ring_read_item(bars.item_full, bars.item_empty, bars.item, ii);
            if (w == -2) {
                ok = false;
                break;
            }
            if (w < 0) break;
            const DqItem item = dq_item<kVarlen>(w, p);
            const int i = item.m * kBQ + tid;  // this thread's query row (within the sequence or document)
            const bool row_ok = i < item.len;
            const size_t rowvec = (static_cast<size_t>(item.b) * p.H + item.h) * p.T + item.base;
            // past the last row: lse = inf, so P = 0 and dS = 0
            const float lse_l2 = row_ok ? p.lse[rowvec + i] * kLog2e : INFINITY;
            const float dlt = row_ok ? p.delta[rowvec + i] : 0.f;
            for (int n = item.n_lo; n <= item.m; ++n, ++gj) {
                ok = mbar_wait_warp(&bars.s_full, gj & 1) && !aborted(bars);
                if (!ok) break;
                tc_fence_after();
                float pf[64];  // P of this thread's row over the warpgroup's 64 keys
                {
                    uint32_t a[32], b2[32];
                    tmem_ld32x2(tmem + lanes + kColST + 64 * g, tmem + lanes + kColST + 64 * g + 32, a, b2);
                    // S is in registers: the MMA warp may write the next S into ST
                    tc_fence_before();
                    mbar_arrive(&bars.s_free);
                    const int j0 = n * kBK + 64 * g;
                    const bool full = (n < item.m) && (item.m * kBQ + kBQ - 1 - n * kBK < p.W);
#pragma unroll
                    for (int x = 0; x < 64; x += 2) {
                        const float s0 = __uint_as_float(x < 32 ? a[x] : b2[x - 32]);
                        const float s1 = __uint_as_float(x < 32 ? a[x + 1] : b2[x - 31]);
                        float e0, e1;
                        fma_f32x2(e0, e1, s0, s1, sl2, sl2, -lse_l2, -lse_l2);
                        float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
                        if (!full) {
                            const int j = j0 + x;
                            if (j > i || i - j >= p.W) p0 = 0.f;
                            if (j + 1 > i || i - (j + 1) >= p.W) p1 = 0.f;
                        }
                        pf[x] = p0;
                        pf[x + 1] = p1;
                    }
                }
                ok = mbar_wait_warp(&bars.dp_full[gj & 1], (gj >> 1) & 1) && !aborted(bars);
                if (!ok) break;
                tc_fence_after();
                const uint32_t dp_addr = tmem + lanes + col_dp(gj) + 64 * g;
                {
                    uint32_t a[32], b2[32];
                    tmem_ld32x2(dp_addr, dp_addr + 32, a, b2);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int x = 0; x < 32; x += 2) {
                            float t0, t1, d0, d1;
                            add_f32x2(t0, t1, __uint_as_float(c ? b2[x] : a[x]),
                                      __uint_as_float(c ? b2[x + 1] : a[x + 1]), -dlt, -dlt);
                            mul_f32x2(d0, d1, pf[32 * c + x], pf[32 * c + x + 1], t0, t1);
                            pk[x / 2] = pack_bf16x2(d0, d1);
                        }
                        // dS (bf16) over this warpgroup's already-read DP columns
                        tmem_st16(dp_addr + 16 * c, pk);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars.ds_full[gj & 1]);
                if (have_prev) {
                    have_prev = false;
                    ok = epilogue(prev, prev_ii);
                    if (!ok) break;
                }
            }
            if (!ok) break;
            have_prev = true;
            prev = item;
            prev_ii = ii;
        }
        if (ok && have_prev) ok = epilogue(prev, prev_ii);
        if (!ok) record_timeout(bars, p.err);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool kVarlen>
cudaError_t launch_dq_tc(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                         const float* delta, void* dq, int B, int T, int H, int window, float scale, int* work,
                         const int* cu, int n_docs, int max_len, int* err, cudaStream_t st) {
    CUtensorMap tq, tk, tv, tdo;
    if (!make_tmap_bthd(&tq, q, B, T, H, D, 64, kBQ) || !make_tmap_bthd(&tk, k, B, T, H, D, 64, kBK) ||
        !make_tmap_bthd(&tv, v, B, T, H, D, 64, kBK) || !make_tmap_bthd(&tdo, dO, B, T, H, D, 64, kBQ))
        return cudaErrorInvalidValue;
    DqParams p;
    p.lse = lse;
    p.delta = delta;
    p.dq = static_cast<__nv_bfloat16*>(dq);
    p.B = B;
    p.T = T;
    p.H = H;
    p.W = (window <= 0 || window >= T) ? T : window;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.n_qb = ((kVarlen ? max_len : T) + kBQ - 1) / kBQ;
    p.work = work;
    p.err = err;
    p.cu = cu;
    p.n_docs = n_docs;
    p.dq32 = (reinterpret_cast<uintptr_t>(dq) & 31u) == 0;
    const int smem = DqSmem<D>::kBytes;
    // the shared-memory limit is raised once per device (atomic flags), the SM count is looked up
    // on every call
    static std::atomic<bool> attr_done[kAttrDevices];
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(bwd_dq_kernel<D, kVarlen>), smem, attr_done);
    if (e != cudaSuccess) return e;
    int n_sm = 0;
    e = multiprocessor_count(&n_sm);
    if (e != cudaSuccess) return e;
    const int n_pairs = (kVarlen ? n_docs : B) * H;
    const long n_items = (long)p.n_qb * n_pairs;
    const int grid = (int)(n_items < n_sm ? n_items : n_sm);
    // a scheduling group holds about one wave of items
    p.group = (n_sm + p.n_qb - 1) / p.n_qb;
    if (p.group > n_pairs) p.group = n_pairs;
    bwd_dq_kernel<D, kVarlen><<<grid, kThreads, smem, st>>>(tq, tk, tv, tdo, p);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                          const float* delta, void* dq, int B, int T, int H, int D, int window, float scale, int* work,
                          int* err, cudaStream_t st, const int* cu, int n_docs, int max_len) {
    if (cu != nullptr)
        return D == 128 ? launch_dq_tc<128, true>(q, k, v, dO, lse, delta, dq, B, T, H, window, scale, work, cu,
                                                  n_docs, max_len, err, st)
                        : launch_dq_tc<64, true>(q, k, v, dO, lse, delta, dq, B, T, H, window, scale, work, cu,
                                                 n_docs, max_len, err, st);
    return D == 128 ? launch_dq_tc<128, false>(q, k, v, dO, lse, delta, dq, B, T, H, window, scale, work, nullptr, 0,
                                               0, err, st)
                    : launch_dq_tc<64, false>(q, k, v, dO, lse, delta, dq, B, T, H, window, scale, work, nullptr, 0,
                                              0, err, st);
}

}  // namespace nc
