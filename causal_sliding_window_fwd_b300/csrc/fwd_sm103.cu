// Forward attention on 5th-generation tensor cores (tcgen05, TMEM, TMA) for sm_103a.
//
// Operation (see include/nc_attn.h): exact causal softmax attention restricted
// to a sliding window of W keys, with the per-row log-sum-exp, as the
// "nanochat GPT-2 speedrun" post (page 2, biggest-improvements paragraph)
// uses through FlashAttention-3's window_size argument.  The computation is
// the textbook definition evaluated block by block with an online softmax.
//
// Persistent CTAs (one per SM) loop over work items.  An item is two 128-row query
// tiles of one (batch, head); the CTA walks the 128-key blocks that the causal window
// makes visible to either tile, and blocks wholly outside the window are never loaded
// (tile skipping).  Warp roles:
//   warp 0       TMA producer: Q tiles once, then K and V blocks through a
//                4-slot shared-memory ring (128-byte swizzle)
//   warp 1       MMA issuer (one lane) and TMEM owner (512 columns)
//   warps 4-7    softmax of query tile 0 (one thread per row)
//   warps 8-11   softmax of query tile 1
//   warps 12-15  epilogue of both tiles: O / l out of TMEM (handed back at once), then
//                staged in shared memory and sent with TMA stores, and the log-sum-exp;
//                it runs while the softmax warpgroups already work on the next item
// TMEM: S0 cols [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
// P (bf16, two per column) overwrites the first 64 columns of its S tile and
// feeds the P*V product straight from TMEM.  The MMA issue order
//   S0(j+1) after PV0(j), S1(j+1) after PV1(j)
// lets one tile's softmax overlap the other tile's products.  The running
// maximum is only raised (and O rescaled in TMEM) when it grows by more
// than 2^8, which keeps every exponent bounded and the sum exact; a row that
// has seen no visible key yet simply takes the next block's maximum.
#include <atomic>
#include <cstdint>
#include <cuda_bf16.h>

#include "nc_attn.h"
#include "nc_kernels.h"
#include "nc_ptx.cuh"
#include "nc_sched.cuh"
#include "nc_tma.h"

namespace nc {
namespace {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per block
constexpr int kStages = 4;        // K/V ring slots
constexpr int kThreads = 512;     // 16 warps
constexpr int kItemReaders = 13;  // warps that read each work-item slot: the MMA warp, 8 softmax warps, 4 epilogue warps

// Varlen work-item counters: one {next item, CTAs finished} pair per call, taken round-robin
// from this ring.  They are zero at load, and the last CTA of each launch zeroes its pair
// again, so a pair is zero whenever a launch starts with it; calls in flight at the same time
// (on different streams) use different pairs as long as fewer than kWorkSlots overlap.
constexpr int kWorkSlots = 4096;
__device__ int g_fwd_work[kWorkSlots][2];
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdSmem {
    static constexpr int kTileBytes = kBM * D * 2;     // one Q tile or one K/V block
    static constexpr int kQOff = 0;                    // Q0, Q1
    static constexpr int kKVOff = 2 * kTileBytes;      // ring
    static constexpr int kStageOff = kKVOff + kStages * kTileBytes;  // O epilogue: one 64-column x 128-row slice
    static constexpr int kStageBytes = kBM * 128;
    static constexpr int kStatsOff = kStageOff + kStageBytes;        // row statistics, see FwdStats
    static constexpr int kBarsOff = kStatsOff + 2 * 2 * kBM * 8;
    static constexpr int kBytes = kBarsOff + 512;
};

struct FwdBarriers {
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t q_full;
    uint64_t q_empty;
    uint64_t s_full[2];
    uint64_t p_full[2];
    // row statistics (m, l) handed from a tile's softmax warpgroup to the epilogue, in two slots
    // (item parity) per tile, each with a full and an empty barrier, so neither side can run a
    // whole phase ahead of the other on one barrier
    uint64_t stats_full[2][2];   // [slot][tile]
    uint64_t stats_empty[2][2];
    uint64_t o_final;
    uint64_t o_free[2];       // the epilogue has read a tile's O out of TMEM
    uint64_t drain;
    uint64_t item_full[kItemSlots];   // varlen: work-item ring (see nc_sched.cuh)
    uint64_t item_empty[kItemSlots];
    int item[kItemSlots];
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(FwdBarriers) <= 512, "barrier block outgrew its shared-memory slot");

struct FwdParams {
    __nv_bfloat16* o;     // [B, Tq, H, D]
    float* lse;           // [B, H, Tq]
    int B, H, W;          // W: effective window, 1 <= W <= Tk
    int Tq;               // query rows per sequence (q, o, lse)
    int Tk;               // rows of the K/V tensors per sequence
    // Plain forward: nullptr, the queries are positions 0 .. Tq-1 of K/V (Tq == Tk).
    // Prefill over a cache: per-sequence lengths L_b that count the Tq new tokens; query t
    // of sequence b is position L_b - Tq + t.  A length outside [Tq, Tk] gives NaN rows and
    // NC_ERR_BAD_CACHE_LEN.
    const int* lens;
    // Document-masked (varlen) forward: q, k, v, o are packed [1, Tq, H, D] rows (Tq = Tk = total)
    // and document d is rows cu[d] .. cu[d+1]-1, attending only within itself; nullptr otherwise.
    const int* cu;
    int n_docs;
    int* work;            // varlen: {next item, CTAs finished}, zero on entry and left zero on exit
    float scale_log2;
    int n_pairs;          // query-tile pairs per (b, h), or per (document, h): the longest document's
    // Plain / prefill: items split0 .. n_items-1 are single query tiles, two per pair item split0 + (w -
    // split0) / 2, so that a last round that would have kept fewer than half the CTAs busy runs half-length
    // items on twice as many (split0 = n_items = pair items otherwise)
    int split0;
    int n_items;
    int* err;
};

// Forward variants: plain, prefill over a KV cache, document-masked packed rows.
enum FwdMode { kModePlain = 0, kModeCache = 1, kModeVarlen = 2 };

// Key blocks [lo, hi] that intersect the window of some query of the tile whose first query sits at
// position pos0; the last query of the sequence sits at position last.  Key block kb holds the keys at
// positions kb * kBN - kpad .. kb * kBN - kpad + kBN - 1 (kpad > 0 shifts the blocks so that their edges
// line up with the query tiles' when the queries start at a position that is not a multiple of kBN).
__device__ __forceinline__ void tile_blocks(int pos0, int last, int W, int kpad, int& lo, int& hi) {
    const int first_key = pos0 - W + 1;
    lo = ((first_key <= 0 ? 0 : first_key) + kpad) / kBN;
    hi = (min(pos0 + kBM - 1, last) + kpad) / kBN;
}

__device__ __forceinline__ bool aborted(const FwdBarriers& bars) {
    return *reinterpret_cast<const volatile int*>(&bars.abort) != 0;
}

__device__ __forceinline__ void record_timeout(FwdBarriers& bars, int* err) {
    set_device_error(err, NC_ERR_DEVICE_TIMEOUT);
    atomicExch(&bars.abort, 1);
}

// Geometry of one work item: a pair of 128-row query tiles of one (batch, head).
struct FwdItem {
    int b, h;
    int off;            // position of query row 0 among the keys (prefill); 0 otherwise
    int kpad;           // key block kb starts at key position kb * kBN - kpad: (-off) mod kBN, so the key
                        // blocks line up with the query tiles (prefill items whose window starts past
                        // position 0); 0 otherwise
    int base;           // first packed row of the document (varlen); 0 otherwise
    int len;            // query rows of this sequence or document
    bool bad;           // the sequence's cache length (or the document's bounds) is out of range
    bool empty;         // nothing to do (a varlen pair past its document's end, or a bad document)
    int r0[2];
    int lo[2], hi[2];   // key blocks each tile visits (empty range for an inactive tile 1)
    int kb_lo, kb_hi;   // union of the two ranges
    bool active1;
};

// Items are numbered heaviest first (query-tile pair descending, then (h, b)), so the
// static zigzag assignment over persistent CTAs (nc_sched.cuh) hands out the long causal tiles first.
template <int kMode>
__device__ __forceinline__ FwdItem fwd_item(int w, const FwdParams& p) {
    FwdItem it;
    int tile_only = -1;  // a single-tile item: which tile of its pair
    if (kMode != kModeVarlen && w >= p.split0) {
        tile_only = (w - p.split0) & 1;
        w = p.split0 + ((w - p.split0) >> 1);
    }
    const int per_pair = kMode == kModeVarlen ? p.H * p.n_docs : p.B * p.H;
    const int bh = w % per_pair;
    const int pair = p.n_pairs - 1 - w / per_pair;
    it.h = bh % p.H;
    it.b = kMode == kModeVarlen ? 0 : bh / p.H;
    it.r0[0] = pair * 2 * kBM + (tile_only > 0 ? kBM : 0);
    it.r0[1] = it.r0[0] + kBM;
    it.off = 0;
    it.base = 0;
    it.len = p.Tq;
    it.bad = false;
    it.empty = false;
    if (kMode == kModeCache) {
        // a bad length still runs (clamped into range) so every role keeps the same schedule;
        // the epilogue then writes NaN rows instead
        const int L = p.lens[it.b];
        it.bad = L < p.Tq || L > p.Tk;
        it.off = min(max(L, p.Tq), p.Tk) - p.Tq;
    }
    if (kMode == kModeVarlen) {
        const int d = bh / p.H;
        const int a = p.cu[d], e = p.cu[d + 1];
        it.bad = a < 0 || e < a || e > p.Tq || e - a > p.n_pairs * 2 * kBM;
        it.base = it.bad ? 0 : a;
        it.len = it.bad ? 0 : e - a;
        it.empty = it.bad || it.r0[0] >= it.len;
        if (it.empty) it.len = 1;  // keeps the block arithmetic below in range; nothing is done
    }
    // shifted blocks save the half-empty block at the window's far edge; an item whose window reaches back
    // to position 0 keeps the unshifted blocks (a shift would only move the partial block to position 0)
    it.kpad = (kMode == kModeCache && it.off + it.r0[0] - p.W + 1 > 0) ? (kBN - it.off % kBN) % kBN : 0;
    if (tile_only >= 0 && it.r0[0] >= it.len) it.empty = true;  // the pair's second tile lies past the end
    const int last = it.off + it.len - 1;
    it.active1 = tile_only < 0 && it.r0[1] < it.len;
    tile_blocks(it.off + it.r0[0], last, p.W, it.kpad, it.lo[0], it.hi[0]);
    tile_blocks(it.off + it.r0[1], last, p.W, it.kpad, it.lo[1], it.hi[1]);
    if (!it.active1) {
        it.lo[1] = it.hi[0] + 1;
        it.hi[1] = it.hi[0];
    }
    it.kb_lo = it.lo[0];
    it.kb_hi = it.active1 ? it.hi[1] : it.hi[0];
    return it;
}

// Varlen producer warp (converged): take item indices from the counter until one has work (reporting
// bad document bounds on the way) and publish it in slot k % kItemSlots; -1 once all are taken,
// -2 if the wait for the slot ran out.
__device__ __forceinline__ int publish_fwd_item(FwdBarriers& bars, int k, int n_items, const FwdParams& p) {
    const int slot = k % kItemSlots;
    if (!mbar_wait_warp(&bars.item_empty[slot], ((k / kItemSlots) & 1) ^ 1)) return -2;
    int w = 0;
    if (lane_id() == 0) {
        for (;;) {
            w = atomicAdd(&p.work[0], 1);
            if (w >= n_items) {
                w = -1;
                break;
            }
            const FwdItem it = fwd_item<kModeVarlen>(w, p);
            if (it.bad) set_device_error(p.err, NC_ERR_BAD_SEQLENS);
            if (!it.empty) break;
        }
        bars.item[slot] = w;
        mbar_arrive(&bars.item_full[slot]);
    }
    return __shfl_sync(0xffffffffu, w, 0);
}

// Next work item of a role: from the static schedule (plain / prefill), or from the item ring that
// the producer fills (varlen).  -1: no more items; -2: a wait ran out.
template <int kMode>
__device__ __forceinline__ int next_item(FwdBarriers& bars, int ii, int my_items) {
    if (kMode == kModeVarlen) return ring_read_item(bars.item_full, bars.item_empty, bars.item, ii);
    return ii < my_items ? sched_item_index(ii) : -1;
}

// kMode: the plain forward, prefill over a KV cache (per-sequence query offsets from p.lens), or
// document-masked packed rows (per-document row bases from p.cu).  Varlen work items past a
// document's end are skipped by every role alike; `ip` counts the items a role really ran and
// gives the phases of the per-item barriers.
template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
    using L = FwdSmem<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    FwdBarriers& bars = *reinterpret_cast<FwdBarriers*>(smem + L::kBarsOff);
    // row statistics handed from the softmax warpgroups to the epilogue: [item parity][tile][row] (m, l)
    float2* stats = reinterpret_cast<float2*>(smem + L::kStatsOff);

    const int warp = warp_id(), lane = lane_id();
    const int n_items = kMode == kModeVarlen ? p.n_pairs * p.H * p.n_docs : p.n_items;

    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) set_device_error(p.err, NC_ERR_CUDA);
        return;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bars.kv_full[i], 1);
            mbar_init(&bars.kv_empty[i], 1);
        }
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars.s_full[t], 1);
            mbar_init(&bars.p_full[t], kBM);
            for (int sl = 0; sl < 2; ++sl) {
                mbar_init(&bars.stats_full[sl][t], kBM);
                mbar_init(&bars.stats_empty[sl][t], kBM);
            }
        }
        mbar_init(&bars.o_final, 1);
        mbar_init(&bars.o_free[0], kBM);
        mbar_init(&bars.o_free[1], kBM);
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
    // 512 threads x 128 registers at launch; the producer/MMA warpgroup drops to 56, the softmax
    // warpgroups rise to 176 and the epilogue drops to 96 (128 x 56 + 256 x 176 + 128 x 96 <= 65536)
    const uint32_t col_s[2] = {0u, 128u};
    const uint32_t col_o[2] = {256u, 256u + D};
    const int my_items = kMode == kModeVarlen ? 0 : sched_items_of_cta(n_items);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // the whole warp runs this loop converged; lane 0 issues each copy
        regs_decrease<56>();
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        __syncwarp();
        int seq = 0;          // K/V loads issued over all items (ring position)
        int q_loads = 0;
        bool ok = true;
        for (int ii = 0; ok; ++ii) {
            // plain / prefill: the static zigzag schedule; varlen: items with work, from the counter
            int w;
            if (kMode == kModeVarlen) {
                w = publish_fwd_item(bars, ii, n_items, p);
                if (w == -2 || aborted(bars)) {
                    ok = false;
                    break;
                }
                if (w < 0) break;
            } else {
                if (ii >= my_items) break;
                w = sched_item_index(ii);
            }
            const FwdItem it = fwd_item<kMode>(w, p);
            if (it.empty) {
                if (kMode == kModeVarlen && it.bad && lane == 0) set_device_error(p.err, NC_ERR_BAD_SEQLENS);
                continue;
            }
            // Q of this item once the previous item's S products have read theirs
            if (!mbar_wait_warp(&bars.q_empty, (q_loads & 1) ^ 1) || aborted(bars)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx_w(&bars.q_full, 2 * L::kTileBytes);
            for (int t = 0; t < 2; ++t)
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d_w(smem + L::kQOff + t * L::kTileBytes + c * kBM * 128, &tm_q, &bars.q_full, c * 64,
                                  it.h, it.base + it.r0[t], it.b);
            ++q_loads;
            const int n_loads = 2 * (it.kb_hi - it.kb_lo + 1);
            for (int x = 0; x < n_loads; ++x, ++seq) {
                const int slot = seq % kStages;
                if (!mbar_wait_warp(&bars.kv_empty[slot], ((seq / kStages) & 1) ^ 1) || aborted(bars)) {
                    ok = false;
                    break;
                }
                const int kb = it.kb_lo + x / 2;
                const CUtensorMap* tm = (x & 1) ? &tm_v : &tm_k;
                uint8_t* dst = smem + L::kKVOff + slot * L::kTileBytes;
                mbar_arrive_expect_tx_w(&bars.kv_full[slot], L::kTileBytes);
                for (int c = 0; c < D / 64; ++c)
                    // (a prefill block shifted by kpad may start before row 0: those rows read as zeros)
                    tma_load_4d_w(dst + c * kBN * 128, tm, &bars.kv_full[slot], c * 64, it.h,
                                  it.base + kb * kBN - it.kpad, it.b);
            }
        }
        if (!ok) record_timeout(bars, p.err);
        if (kMode == kModeVarlen && lane == 0) {
            // this CTA takes no more items: the last CTA to get here zeroes the counter pair
            __threadfence();
            if (atomicAdd(&p.work[1], 1) == static_cast<int>(gridDim.x) - 1) {
                p.work[0] = 0;
                p.work[1] = 0;
                __threadfence();
            }
        }
        __syncwarp();
        // never leave while a copy into this CTA's shared memory may still land: only the
        // last use of each slot (and of Q) can still be outstanding
        for (int x = seq - kStages < 0 ? 0 : seq - kStages; x < seq; ++x)
            mbar_wait_warp(&bars.kv_full[x % kStages], (x / kStages) & 1);
        if (q_loads > 0) mbar_wait_warp(&bars.q_full, (q_loads - 1) & 1);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs this loop converged; lane 0 issues each product
        regs_decrease<56>();
        constexpr uint32_t idesc_qk = idesc_bf16(kBM, kBN, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16(kBM, D, false, true);
        const uint32_t q_base = smem_u32(smem + L::kQOff);
        const uint32_t kv_base = smem_u32(smem + L::kKVOff);
        // Descriptors are built once; every product then only adds a constant
        // (byte offset / 16) to the start-address field, which keeps the issue loop short.
        const uint64_t q_desc = sdesc(q_base, 16, 1024);                // K-major, SW128
        const uint64_t k_desc = sdesc(kv_base, 16, 1024);               // K-major, SW128
        const uint64_t v_desc = sdesc(kv_base, kBN * 128, 1024);        // MN-major, SW128
        constexpr uint64_t kTileStep = L::kTileBytes >> 4;
        auto issue_s = [&](int t, int slot) {
            const uint64_t qd = q_desc + t * kTileStep;
            const uint64_t kd = k_desc + slot * kTileStep;
            const uint32_t d = tmem + (t ? col_s[1] : col_s[0]);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                constexpr int kChunk = (kBM * 128) >> 4;
                const uint64_t off = (kk / 4) * kChunk + (kk % 4) * 2;
                mma_ss_w(d, qd + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit_w(&bars.s_full[t]);
        };
        auto issue_pv = [&](int t, int slot, bool accumulate) {
            const uint64_t vd = v_desc + slot * kTileStep;
            const uint32_t d = tmem + (t ? col_o[1] : col_o[0]);
            const uint32_t a = tmem + (t ? col_s[1] : col_s[0]);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
                mma_ts_w(d, a + kk * 8, vd + kk * (2048 >> 4), idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
        };
        bool ok = true;
        int seq = 0;                 // K/V ring position over all items
        int n_pv0 = 0, n_pv1 = 0;    // P tiles consumed per query tile over all items
        int ip = 0;                  // items run
        for (int ii = 0; ok; ++ii) {
            const int w = next_item<kMode>(bars, ii, my_items);
            if (w == -2) {
                ok = false;
                break;
            }
            if (w < 0) break;
            const FwdItem it = fwd_item<kMode>(w, p);
            if (it.empty) continue;
            auto act = [&](int t, int kb) {
                return t ? (kb >= it.lo[1] && kb <= it.hi[1]) : (kb >= it.lo[0] && kb <= it.hi[0]);
            };
            ok = mbar_wait_warp(&bars.q_full, ip & 1);
            if (!ok) break;
            {
                const int slot_k = seq % kStages;
                ok = mbar_wait_warp(&bars.kv_full[slot_k], (seq / kStages) & 1);
                if (!ok) break;
                tc_fence_after();
                for (int t = 0; t < 2; ++t)
                    if (act(t, it.kb_lo)) issue_s(t, slot_k);
                mma_commit_w(&bars.kv_empty[slot_k]);
                ++seq;
                if (it.kb_lo == it.kb_hi) mma_commit_w(&bars.q_empty);  // every S of this item is issued
            }
            bool first_pv0 = true, first_pv1 = true;
            for (int kb = it.kb_lo; ok && kb <= it.kb_hi; ++kb) {
                const int slot_v = seq % kStages;
                ok = mbar_wait_warp(&bars.kv_full[slot_v], (seq / kStages) & 1);
                if (!ok) break;
                ++seq;
                if (kMode == kModeCache && kb == it.kb_hi) {
                    // the last block of a prefill item may hold cache rows at or past the sequence's
                    // length; their weights are 0, but 0 x NaN is NaN inside the product, so those
                    // value rows are zeroed in shared memory first (whatever the cache holds there)
                    const int r0 = it.off + it.len - (kb * kBN - it.kpad);  // first row past the last query position
                    if (r0 < kBN) {
                        uint8_t* vt = smem + L::kKVOff + slot_v * L::kTileBytes;
                        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                        for (int u = r0 * 8 + lane; u < kBN * 8; u += 32)  // 16-byte units of 128-byte rows
                            for (int c = 0; c < D / 64; ++c)
                                *reinterpret_cast<uint4*>(vt + c * kBN * 128 + u * 16) = z;
                        fence_async_smem();
                        __syncwarp();
                    }
                }
                const bool next = kb + 1 <= it.kb_hi;
                const int slot_k = seq % kStages;
                bool k_ready = false;
                for (int t = 0; t < 2 && ok; ++t) {
                    if (act(t, kb)) {
                        if ((t ? first_pv1 : first_pv0) && ip > 0) {
                            // the epilogue has read this tile's O of the previous item
                            ok = mbar_wait_warp(&bars.o_free[t], (ip - 1) & 1) && !aborted(bars);
                            if (!ok) break;
                        }
                        if (t) first_pv1 = false; else first_pv0 = false;
                        ok = mbar_wait_warp(&bars.p_full[t], (t ? n_pv1 : n_pv0) & 1) && !aborted(bars);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(t, slot_v, kb > (t ? it.lo[1] : it.lo[0]));
                        if (t) ++n_pv1; else ++n_pv0;
                    }
                    if (next && act(t, kb + 1)) {
                        if (!k_ready) {
                            ok = mbar_wait_warp(&bars.kv_full[slot_k], (seq / kStages) & 1);
                            if (!ok) break;
                            tc_fence_after();
                            k_ready = true;
                        }
                        issue_s(t, slot_k);
                    }
                }
                if (!ok) break;
                mma_commit_w(&bars.kv_empty[slot_v]);
                if (next) {
                    mma_commit_w(&bars.kv_empty[slot_k]);
                    ++seq;
                    if (kb + 1 == it.kb_hi) mma_commit_w(&bars.q_empty);  // every S of this item is issued
                }
            }
            if (ok) mma_commit_w(&bars.o_final);
            ++ip;
        }
        if (!ok) record_timeout(bars, p.err);
        // all products must have landed before TMEM is released
        mma_commit_w(&bars.drain);
        mbar_wait_warp(&bars.drain, 0);
    } else if (warp < 4) {
        regs_decrease<56>();
    } else if (warp < 12) {
        // ------------------------------------------------------------ softmax of one query tile
        // one thread per query row: the whole 128-key row of S is read from TMEM with one wait,
        // masked on straddling blocks, its maximum taken, and P written back at the end (reading the
        // row in separately waited chunks between the P stores measured 1.4-2x slower).
        regs_increase<176>();
        const int t = (warp - 4) / 4;
        const int row_in_tile = threadIdx.x - 128 * (t + 1);  // 0..127 == TMEM lane
        const int lane_base = 32 * (warp % 4);
        const uint32_t s_addr = tmem + (static_cast<uint32_t>(lane_base) << 16) + (t ? col_s[1] : col_s[0]);
        const uint32_t o_addr = tmem + (static_cast<uint32_t>(lane_base) << 16) + (t ? col_o[1] : col_o[0]);
        const float sl2 = p.scale_log2;
        bool ok = true;
        int n_s = 0;  // S tiles of this query tile consumed over all items
        int ip = 0;   // items run
        for (int ii = 0; ok; ++ii) {
            const int w = next_item<kMode>(bars, ii, my_items);
            // the warps of this warpgroup leave together if any wait ran out
            if (!named_bar_and(1 + t, 128, w != -2)) {
                ok = false;
                break;
            }
            if (w < 0) break;
            const FwdItem item = fwd_item<kMode>(w, p);
            if (item.empty) continue;
            const int tr0 = t ? item.r0[1] : item.r0[0];
            const int t_lo = t ? item.lo[1] : item.lo[0];
            const int t_hi = t ? item.hi[1] : item.hi[0];
            const int pos = item.off + tr0 + row_in_tile;  // this row's position among the keys
            const int tpos0 = item.off + tr0;
            const int key_lo = max(pos - p.W + 1, 0);  // this row's first visible key (none before position 0)
            const bool tile_on = (t == 0) || item.active1;
            float m_run = -INFINITY, l_run = 0.f;
            if (tile_on) {
                for (int kb = t_lo; kb <= t_hi; ++kb, ++n_s) {
                    ok = mbar_wait_warp(&bars.s_full[t], n_s & 1) && !aborted(bars);  // warp-uniform
                    if (!ok) break;
                    tc_fence_after();
                    // elementwise mask only on blocks that straddle the causal diagonal or the window edge
                    const int k0 = kb * kBN - item.kpad;  // position of the block's first key
                    // (a prefill block that starts before position 0 is masked too: those keys do not exist)
                    const bool masked = !((k0 + kBN - 1 <= tpos0) && (k0 >= tpos0 + kBM - p.W) && k0 >= 0);
                    const bool first = kb == t_lo;
                    float sv[kBN];
                    {
                        uint32_t r0[64], r1[64];
                        tmem_ld64_nowait(s_addr, r0);
                        tmem_ld64_nowait(s_addr + 64, r1);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 64; ++i) {
                            sv[i] = __uint_as_float(r0[i]);
                            sv[64 + i] = __uint_as_float(r1[i]);
                        }
                    }
                    if (masked) {
                        // visible columns of this row: [lo, hi] within the block; one 32-bit mask per group
                        const int lo = key_lo - k0, hi = pos - k0;
#pragma unroll
                        for (int g32 = 0; g32 < kBN / 32; ++g32) {
                            const int a = min(max(lo - 32 * g32, 0), 32), e = min(max(hi - 32 * g32 + 1, 0), 32);
                            const uint32_t upto = e >= 32 ? 0xffffffffu : ((1u << e) - 1u);
                            const uint32_t from = a >= 32 ? 0u : (0xffffffffu << a);
                            const uint32_t vis = upto & from;
#pragma unroll
                            for (int x = 0; x < 32; ++x)
                                if (!((vis >> x) & 1u)) sv[32 * g32 + x] = -INFINITY;
                        }
                    }
                    float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
#pragma unroll
                    for (int j = 4; j + 8 <= kBN; j += 8) {
                        mx0 = max3f(mx0, sv[j], sv[j + 1]);
                        mx1 = max3f(mx1, sv[j + 2], sv[j + 3]);
                        mx2 = max3f(mx2, sv[j + 4], sv[j + 5]);
                        mx3 = max3f(mx3, sv[j + 6], sv[j + 7]);
                    }
                    mx0 = max3f(mx0, sv[kBN - 4], sv[kBN - 3]);
                    mx1 = max3f(mx1, sv[kBN - 2], sv[kBN - 1]);
                    const float m_cand = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
                    // a row that has seen no visible key yet (its window starts past the first block) still
                    // has l = 0 and an exactly zero O row: it takes this block's maximum as is, like a
                    // first block, rather than asking for a rescale of O
                    const bool fresh = first || m_run == -INFINITY;
                    const bool grow = !fresh && m_cand > m_run + kRescaleThreshold;
                    if (fresh) m_run = m_cand;
                    if (__any_sync(0xffffffffu, grow)) {
                        const float m_new = fmaxf(m_run, m_cand);
                        const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(m_run - m_new);
                        m_run = m_new;
                        l_run *= alpha;
#pragma unroll 1
                        for (int d = 0; d < D / 32; ++d) {
                            uint32_t r[32];
                            tmem_ld32(o_addr + d * 32, r);
#pragma unroll
                            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                            tmem_st32(o_addr + d * 32, r);
                        }
                    }
                    const float m_use = m_run == -INFINITY ? 0.f : m_run;
                    float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
#pragma unroll
                    for (int c = 0; c < kBN / 64; ++c) {
                        uint32_t pk[32];
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            float x0, x1, x2, x3;
                            const int j = c * 64 + 2 * i;
                            fma_f32x2(x0, x1, sv[j], sv[j + 1], sl2, sl2, -m_use, -m_use);
                            fma_f32x2(x2, x3, sv[j + 2], sv[j + 3], sl2, sl2, -m_use, -m_use);
                            const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
                            const float e2 = ex2_approx(x2), e3 = ex2_approx(x3);
                            add_f32x2(sum0, sum1, sum0, sum1, e0, e1);
                            add_f32x2(sum2, sum3, sum2, sum3, e2, e3);
                            pk[i] = pack_bf16x2(e0, e1);
                            pk[i + 1] = pack_bf16x2(e2, e3);
                        }
                        tmem_st32(s_addr + c * 32, pk);
                    }
                    l_run += (sum0 + sum1) + (sum2 + sum3);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&bars.p_full[t]);
                }
            }
            // hand the row's statistics to the epilogue: slot ip % 2, once the epilogue has read what
            // this slot held two items ago
            const int slot = ip & 1, use = ip >> 1;
            if (ok) ok = mbar_wait_warp(&bars.stats_empty[slot][t], (use & 1) ^ 1) && !aborted(bars);
            if (!ok) break;
            stats[(slot * 2 + t) * kBM + row_in_tile] = make_float2(m_run, l_run);
            mbar_arrive(&bars.stats_full[slot][t]);
            ++ip;
        }
        if (!ok) record_timeout(bars, p.err);
    } else {
        // ------------------------------------------------------------ epilogue of both query tiles
        // thread = row of both tiles.  Tile by tile, O is read out of TMEM, scaled by 1/l and packed to
        // bf16 in registers, and the tile's TMEM is handed back (o_free) before any of its store work,
        // so the next item's first products wait only for these reads.  The rows then leave through
        // TMA stores of 64-column slices staged in shared memory (128-byte swizzle, the layout of the
        // TMA map): whole-line global writes.
        regs_decrease<96>();
        const int row_in_tile = threadIdx.x - 384;  // 0..127 == TMEM lane
        const int lane_base = 32 * (warp % 4);
        uint8_t* stage = smem + L::kStageOff;
        bool ok = true;
        int ip = 0;
        for (int ii = 0; ok; ++ii) {
            const int w = next_item<kMode>(bars, ii, my_items);
            if (!named_bar_and(3, 128, w != -2)) {
                ok = false;
                break;
            }
            if (w < 0) break;
            const FwdItem item = fwd_item<kMode>(w, p);
            if (item.empty) continue;
            const int slot = ip & 1, use = ip >> 1;
            ok = mbar_wait_warp(&bars.o_final, ip & 1) && mbar_wait_warp(&bars.stats_full[slot][0], use & 1) &&
                 mbar_wait_warp(&bars.stats_full[slot][1], use & 1) && !aborted(bars);
            ok = named_bar_and(3, 128, ok);  // leave together: the stores below synchronise the warpgroup
            if (!ok) break;
            tc_fence_after();
            const float2 st0 = stats[(slot * 2 + 0) * kBM + row_in_tile];
            const float2 st1 = stats[(slot * 2 + 1) * kBM + row_in_tile];
            mbar_arrive(&bars.stats_empty[slot][0]);
            mbar_arrive(&bars.stats_empty[slot][1]);
            if (item.bad && row_in_tile == 0) set_device_error(p.err, NC_ERR_BAD_CACHE_LEN);
#pragma unroll 1
            for (int t = 0; t < 2; ++t) {
                const bool tile_on = (t == 0) || item.active1;
                const float2 st = t ? st1 : st0;
                uint32_t po[D / 2];  // this row of the tile's O, scaled and packed
                if (tile_on) {
                    const float inv_l = item.bad ? __int_as_float(0x7fc00000) : 1.f / st.y;  // NaN rows for a bad length
                    const uint32_t o_addr = tmem + (static_cast<uint32_t>(lane_base) << 16) + (t ? col_o[1] : col_o[0]);
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(o_addr + c * 32, r);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            po[c * 16 + i] =
                                pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars.o_free[t]);
                if (!tile_on) continue;
                const int tr0 = t ? item.r0[1] : item.r0[0];
                const int row = tr0 + row_in_tile;
                const bool in_range = row < item.len;
                // a varlen tile that runs past its document is written row by row, so the next
                // document's rows are left alone; otherwise the TMA store clips rows past the tensor
                const bool whole = (kMode != kModeVarlen) || (tr0 + kBM <= item.len);
                if (whole) {
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        if (row_in_tile == 0) bulk_wait_read();  // the previous store has read the slice
                        named_bar_sync(3, 128);
#pragma unroll
                        for (int u = 0; u < 8; ++u) {  // 16-byte unit u of the row's 128-byte slice
                            const uint4 pkt = make_uint4(po[c * 32 + 4 * u], po[c * 32 + 4 * u + 1],
                                                         po[c * 32 + 4 * u + 2], po[c * 32 + 4 * u + 3]);
                            *reinterpret_cast<uint4*>(stage + row_in_tile * 128 + ((u ^ (row_in_tile & 7)) << 4)) = pkt;
                        }
                        fence_async_smem();
                        named_bar_sync(3, 128);
                        if (row_in_tile == 0) {
                            tma_store_4d(&tm_o, stage, c * 64, item.h, item.base + tr0, item.b);
                            bulk_commit();
                        }
                    }
                } else if (in_range) {
                    __nv_bfloat16* orow =
                        p.o + ((static_cast<size_t>(item.b) * p.Tq + item.base + row) * p.H + item.h) * D;
#pragma unroll
                    for (int u = 0; u < D / 8; ++u)
                        reinterpret_cast<uint4*>(orow)[u] = make_uint4(po[4 * u], po[4 * u + 1], po[4 * u + 2], po[4 * u + 3]);
                }
                if (in_range)
                    p.lse[(static_cast<size_t>(item.b) * p.H + item.h) * p.Tq + item.base + row] =
                        item.bad ? __int_as_float(0x7fc00000) : (st.x + __log2f(st.y)) * kLn2;
            }
            ++ip;
        }
        if (!ok) record_timeout(bars, p.err);
        if (row_in_tile == 0) bulk_wait_all();  // the O stores have landed
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Tq query rows per sequence against Tk key/value rows; lens == nullptr for the plain forward
// (Tq == Tk), else the per-sequence cache lengths of a prefill.
// cu != nullptr: document-masked packed rows (B = 1, Tq = Tk = total), n_docs documents, the longest
// at most max_len rows.
template <int D>
cudaError_t launch_fwd_tc(const void* q, const void* k, const void* v, const int* lens, const int* cu, int n_docs,
                          int max_len, void* o, float* lse, int B, int Tq, int Tk, int H, int window, float scale,
                          int* err, cudaStream_t st) {
    CUtensorMap tq, tk, tv, to;
    if (!make_tmap_bthd(&tq, q, B, Tq, H, D, 64, kBM) || !make_tmap_bthd(&tk, k, B, Tk, H, D, 64, kBN) ||
        !make_tmap_bthd(&tv, v, B, Tk, H, D, 64, kBN) || !make_tmap_bthd(&to, o, B, Tq, H, D, 64, kBM))
        return cudaErrorInvalidValue;
    FwdParams p;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.B = B;
    p.Tq = Tq;
    p.Tk = Tk;
    p.lens = lens;
    p.cu = cu;
    p.n_docs = n_docs;
    p.work = nullptr;
    p.H = H;
    p.W = (window <= 0 || window >= Tk) ? Tk : window;
    p.scale_log2 = scale * kLog2e;
    p.n_pairs = ((cu != nullptr ? max_len : Tq) + 2 * kBM - 1) / (2 * kBM);
    p.err = err;
    const int smem = FwdSmem<D>::kBytes;
    // The SM count and the counter ring's address are looked up on every call, the shared-memory
    // limit is raised once per device and variant (atomic flags): nothing that concurrent first calls
    // from several host threads could race on.
    static std::atomic<bool> attr_done[3][kAttrDevices];
    const int variant = cu != nullptr ? 2 : (lens != nullptr ? 1 : 0);
    auto kern = variant == 2 ? fwd_tc_kernel<D, kModeVarlen>
                             : (variant == 1 ? fwd_tc_kernel<D, kModeCache> : fwd_tc_kernel<D, kModePlain>);
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem, attr_done[variant]);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM (shared memory and TMEM allow one), looping over the items
    int n_sm = 0;
    e = multiprocessor_count(&n_sm);
    if (e != cudaSuccess) return e;
    const long n_pair_items = (long)p.n_pairs * H * (cu != nullptr ? n_docs : B);
    long n_items = n_pair_items;
    p.split0 = static_cast<int>(n_pair_items);
    if (cu == nullptr) {
        // a last round that would keep fewer than half the CTAs busy runs its pair items as single tiles
        const long full = n_pair_items / n_sm, left = n_pair_items - full * n_sm;
        if (full >= 1 && left > 0 && 2 * left <= n_sm) {
            p.split0 = static_cast<int>(full * n_sm);
            n_items = p.split0 + 2 * left;
        }
    }
    p.n_items = static_cast<int>(n_items);
    const int grid = (int)(n_items < n_sm ? n_items : n_sm);
    if (cu != nullptr) {
        static std::atomic<unsigned> work_seq{0};
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_fwd_work);
        if (e != cudaSuccess) return e;
        p.work = static_cast<int*>(ptr) + 2 * (work_seq.fetch_add(1u) % kWorkSlots);
    }
    kern<<<grid, kThreads, smem, st>>>(tq, tk, tv, to, p);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T, int H, int D,
                       int window, float scale, int* err, cudaStream_t st) {
    return D == 128 ? launch_fwd_tc<128>(q, k, v, nullptr, nullptr, 0, 0, o, lse, B, T, T, H, window, scale, err, st)
                    : launch_fwd_tc<64>(q, k, v, nullptr, nullptr, 0, 0, o, lse, B, T, T, H, window, scale, err, st);
}

cudaError_t launch_prefill(const void* q, const void* kcache, const void* vcache, const int* lens, void* o,
                           float* lse, int N, int Tq, int Tmax, int H, int D, int window, float scale, int* err,
                           cudaStream_t st) {
    return D == 128 ? launch_fwd_tc<128>(q, kcache, vcache, lens, nullptr, 0, 0, o, lse, N, Tq, Tmax, H, window, scale,
                                         err, st)
                    : launch_fwd_tc<64>(q, kcache, vcache, lens, nullptr, 0, 0, o, lse, N, Tq, Tmax, H, window, scale,
                                        err, st);
}

cudaError_t launch_fwd_varlen(const void* q, const void* k, const void* v, const int* cu, int n_docs, int max_len,
                              void* o, float* lse, int total, int H, int D, int window, float scale, int* err,
                              cudaStream_t st) {
    return D == 128 ? launch_fwd_tc<128>(q, k, v, nullptr, cu, n_docs, max_len, o, lse, 1, total, total, H, window,
                                         scale, err, st)
                    : launch_fwd_tc<64>(q, k, v, nullptr, cu, n_docs, max_len, o, lse, 1, total, total, H, window,
                                        scale, err, st);
}

}  // namespace nc
