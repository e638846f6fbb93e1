// Single-token decode over a padded KV cache: split-K partial softmax over
// chunks of visible cache rows, then a per-(sequence, head) combine.
//
// Operation: the "nanochat" walkthrough (page 4, close of the pretraining
// section; page 1 launch post) runs inference through an Engine with a KV
// cache and a prefill/decode split; decode is one query token attending over
// the cached keys/values, restricted to the layer's sliding window
// ("nanochat GPT-2 speedrun" post, page 2, FlashAttention-3 window_size).
//
// This path is bound by HBM bandwidth (about one flop per byte), so it runs
// on CUDA cores: a cache row of one token holds all H heads contiguously
// (H * D bf16), each warp streams one head's 256-byte (D = 128) slice of
// consecutive rows with 16-byte vector loads, and a CTA covers every head of
// a chunk of rows, so the CTA reads whole contiguous rows.
#include <cstdint>
#include <cuda_bf16.h>

#include "nc_attn.h"
#include "nc_decode.h"
#include "nc_kernels.h"
#include "nc_ptx.cuh"

namespace nc {

namespace {

// Up to 10 warps (one per head for the depth-20 shape); two CTAs fit per SM.
constexpr int kDecodeMaxThreads = 320;
// The balanced split serves up to this many sequences (its CTAs scan their visible-row counts in
// shared memory) and cuts ranges of at least kMinRowsPerCta rows.
constexpr int kBalancedMaxSeqs = 1024;
constexpr int kMinRowsPerCta = 16;
constexpr int kCombineFast = 8;
// Bulk-copy split: a ring of kBulkStages stages of kBulkHalfStage bytes of K and as many of V, heads <= 16.
constexpr int kBulkStages = 4;
constexpr int kBulkHalfStage = 24 * 1024;
constexpr int kBulkMaxHeads = 16;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Visible cache rows of a sequence of length L: [L - W', L) with W' = min(W, L).
__device__ __forceinline__ int visible_lo(int L, int window) {
    return (window <= 0 || window >= L) ? 0 : L - window;
}

__device__ __forceinline__ float fast_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Lane layout of one warp streaming one head: lanes are grouped G = D / 8 per token row (each lane holds 8
// columns), and a step covers TPS = 32 / G tokens.
template <int D>
struct RowLanes {
    static constexpr int G = D / 8;
    static constexpr int TPS = 32 / G;
};

// The query row of (n, h) as this lane's 8 columns, scaled into log2 units.
template <int D>
__device__ __forceinline__ void load_query(const __nv_bfloat16* __restrict__ q, int n, int h, int H, float (&qf)[8]) {
    const int c = (threadIdx.x & 31) % RowLanes<D>::G;
    bf16x8_to_f32(reinterpret_cast<const uint4*>(q + ((size_t)n * H + h) * D)[c], qf);
}

// U steps of the online softmax: kr[u], vr[u] are this lane's 8 columns of the key / value of token slot u,
// `valid` says whether the slot holds a visible token.  Updates the lane's running max m (log2 units), sum l
// and unnormalised output acc.
template <int D, int U>
__device__ __forceinline__ void softmax_steps(const uint4 (&kr)[U], const uint4 (&vr)[U], const bool (&valid)[U],
                                              const float (&qf)[8], float& m, float& l, float (&acc)[8]) {
    constexpr int G = RowLanes<D>::G;
    // scores of the U tokens (log2 units), reduced across the G lanes of a token
    float sc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        float kf[8];
        bf16x8_to_f32(kr[u], kf);
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) dot = fmaf(qf[i], kf[i], dot);
        sc[u] = dot;
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1)
#pragma unroll
        for (int u = 0; u < U; ++u) sc[u] += __shfl_xor_sync(0xffffffffu, sc[u], off);
    float mc = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (!valid[u]) sc[u] = -INFINITY;
        mc = fmaxf(mc, sc[u]);
    }
    const float m_new = fmaxf(m, mc);
    if (m_new == -INFINITY) return;  // no visible token in this lane's slots yet
    const float alpha = fast_ex2(m - m_new);
    l *= alpha;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] *= alpha;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const float p = fast_ex2(sc[u] - m_new);
        float vf[8];
        bf16x8_to_f32(vr[u], vf);
        l += p;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vf[i], acc[i]);
    }
    m = m_new;
}

// Merge the TPS token slots of the warp (lanes with equal column group) and write the partial (running max
// in log2 units, sum, unnormalised output) to part_ml[pidx], part_o[pidx].
template <int D>
__device__ __forceinline__ void merge_and_store(float m, float l, float (&acc)[8], size_t pidx,
                                                float* __restrict__ part_ml, float* __restrict__ part_o) {
    constexpr int G = RowLanes<D>::G;
    const int lane = threadIdx.x & 31, c = lane % G;
#pragma unroll
    for (int off = G; off < 32; off <<= 1) {
        const float m_o = __shfl_xor_sync(0xffffffffu, m, off);
        const float l_o = __shfl_xor_sync(0xffffffffu, l, off);
        const float m_new = fmaxf(m, m_o);
        const float a_s = (m == -INFINITY) ? 0.f : fast_ex2(m - m_new);
        const float a_o = (m_o == -INFINITY) ? 0.f : fast_ex2(m_o - m_new);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float o_o = __shfl_xor_sync(0xffffffffu, acc[i], off);
            acc[i] = acc[i] * a_s + o_o * a_o;
        }
        l = l * a_s + l_o * a_o;
        m = m_new;
    }
    if (lane < G) {
        float4* po = reinterpret_cast<float4*>(part_o + pidx * D + c * 8);
        po[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        po[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    if (lane == 0) {
        part_ml[pidx * 2 + 0] = m;
        part_ml[pidx * 2 + 1] = l;
    }
}

// Online softmax of one head's query over cache rows [t_begin, t_end) of sequence n, by one warp reading
// global memory: U steps of K and V loads are in flight before any arithmetic on them.
template <int D>
__device__ __forceinline__ void decode_rows(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                                            const __nv_bfloat16* __restrict__ vc, int n, int h, int H, int Tmax,
                                            int t_begin, int t_end, float scale_log2, size_t pidx,
                                            float* __restrict__ part_ml, float* __restrict__ part_o) {
    constexpr int G = RowLanes<D>::G, TPS = RowLanes<D>::TPS;
    constexpr int U = 4;              // steps in flight per iteration
    const int lane = threadIdx.x & 31;
    const int g = lane / G;           // token slot within a step
    const int c = lane % G;           // 8-element column group
    const size_t row_stride = (size_t)H * D;  // elements between consecutive tokens
    float qf[8];
    load_query<D>(q, n, h, H, qf);
#pragma unroll
    for (int i = 0; i < 8; ++i) qf[i] *= scale_log2;
    float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    const __nv_bfloat16* kbase = kc + (size_t)n * Tmax * row_stride + (size_t)h * D + c * 8;
    const __nv_bfloat16* vbase = vc + (size_t)n * Tmax * row_stride + (size_t)h * D + c * 8;
    for (int t0 = t_begin; t0 < t_end; t0 += TPS * U) {
        uint4 kr[U], vr[U];
        bool valid[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = t0 + u * TPS + g;
            valid[u] = t < t_end;
            kr[u] = make_uint4(0, 0, 0, 0);
            vr[u] = make_uint4(0, 0, 0, 0);
            if (valid[u]) {
                kr[u] = ldg_stream(reinterpret_cast<const uint4*>(kbase + (size_t)t * row_stride));
                vr[u] = ldg_stream(reinterpret_cast<const uint4*>(vbase + (size_t)t * row_stride));
            }
        }
        softmax_steps<D, U>(kr, vr, valid, qf, m, l, acc);
    }
    merge_and_store<D>(m, l, acc, pidx, part_ml, part_o);
}

// Chunked split (many sequences): one CTA per (split s, sequence n) work item; item = s + n_splits * n.
// Warp w handles heads w, w + nwarps, ...
template <int D>
__global__ void __launch_bounds__(kDecodeMaxThreads, 2)
decode_split_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                    const __nv_bfloat16* __restrict__ vc, const int* __restrict__ lens,
                    float* __restrict__ part_ml, float* __restrict__ part_o, int N, int Tmax, int H,
                    int window, float scale_log2, int n_splits, int chunk) {
    const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int n_items = n_splits * N;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int s = item % n_splits, n = item / n_splits;
        const int L = lens[n];
        if (L < 1 || L > Tmax) continue;  // reported by the combine kernel
        const int lo = visible_lo(L, window);
        const int t_begin = lo + s * chunk;
        const int t_end = min(L, t_begin + chunk);
        if (t_begin >= t_end) continue;  // this split lies past the sequence's visible rows
        for (int h = warp; h < H; h += nwarps)
            decode_rows<D>(q, kc, vc, n, h, H, Tmax, t_begin, t_end, scale_log2, ((size_t)n * n_splits + s) * H + h,
                           part_ml, part_o);
    }
    // this CTA's partials are written: once every CTA is here the combine kernel may be scheduled
    // (it still waits for this grid's completion before reading them)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Balanced split (up to kBalancedMaxSeqs sequences): the visible rows of all sequences, laid end to end
// (sequence n's at offsets P_n .. P_n + V_n - 1, P the exclusive prefix sum of the visible counts V),
// are cut into gridDim.x equal ranges of `per` rows, one per CTA, so every CTA streams the same number
// of bytes and the grid ends together (no partial last wave).  CTA c's piece of sequence n writes its
// partial to slot n + c: slots increase with (c, n), so they are distinct and below N + gridDim.x.
// Every CTA computes the prefix sums itself; CTA 0 also stores them (and `per`) in meta for the combine.
struct BalancedRange {
    int per, r0, r1;  // rows per CTA and this CTA's range [r0, r1) of the laid-out rows
    int first_seq;    // the first sequence whose rows reach past r0 (valid when r0 < r1)
};

// V_n in s_vis, P_n in s_pre (s_pre[N] = the total), this CTA's range; CTA 0 writes meta.  Called by every
// thread of the CTA (it synchronises the CTA).
__device__ __forceinline__ BalancedRange balanced_range(const int* __restrict__ lens, int* __restrict__ meta, int N,
                                                        int Tmax, int window, int* s_vis, int* s_pre) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int n = tid; n < N; n += blockDim.x) {
        const int L = lens[n];
        s_vis[n] = (L < 1 || L > Tmax) ? 0 : L - visible_lo(L, window);  // bad lengths: no rows
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scan by one warp: lane i sums a run of consecutive sequences, then the runs are scanned
        const int run = (N + 31) / 32;
        const int a = min(N, lane * run), b = min(N, a + run);
        int sum = 0;
        for (int n = a; n < b; ++n) sum += s_vis[n];
        int incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        int p = incl - sum;
        for (int n = a; n < b; ++n) {
            s_pre[n] = p;
            p += s_vis[n];
        }
        if (lane == 31) s_pre[N] = incl;
    }
    __syncthreads();
    BalancedRange r;
    const int R = s_pre[N];
    r.per = max((R + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x), kMinRowsPerCta);
    if (blockIdx.x == 0) {
        for (int n = tid; n <= N; n += blockDim.x) meta[n] = s_pre[n];
        if (tid == 0) meta[N + 1] = r.per;
    }
    r.r0 = static_cast<int>(blockIdx.x) * r.per;
    r.r1 = min(R, r.r0 + r.per);
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_pre[mid + 1] > r.r0) hi = mid;
        else lo = mid + 1;
    }
    r.first_seq = lo;
    return r;
}

// Sequence n's piece of a CTA's range: cache rows [t_begin, t_end).  False for a sequence without rows.
__device__ __forceinline__ bool balanced_piece(const BalancedRange& r, const int* __restrict__ lens, int window,
                                               const int* s_vis, const int* s_pre, int n, int& t_begin, int& t_end) {
    const int P = s_pre[n], V = s_vis[n];
    if (V == 0) return false;
    const int first = visible_lo(lens[n], window);
    t_begin = first + max(r.r0, P) - P;
    t_end = first + min(r.r1, P + V) - P;
    return true;
}

// Balanced split with plain loads: warps over heads, each streaming its head's slice of the rows.
template <int D>
__global__ void __launch_bounds__(kDecodeMaxThreads, 2)
decode_balanced_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                       const __nv_bfloat16* __restrict__ vc, const int* __restrict__ lens,
                       float* __restrict__ part_ml, float* __restrict__ part_o, int* __restrict__ meta, int N,
                       int Tmax, int H, int window, float scale_log2) {
    __shared__ int s_vis[kBalancedMaxSeqs];
    __shared__ int s_pre[kBalancedMaxSeqs + 1];
    const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const BalancedRange r = balanced_range(lens, meta, N, Tmax, window, s_vis, s_pre);
    if (r.r0 < r.r1) {
        for (int n = r.first_seq; n < N && s_pre[n] < r.r1; ++n) {
            int t_begin, t_end;
            if (!balanced_piece(r, lens, window, s_vis, s_pre, n, t_begin, t_end)) continue;
            const size_t slot = (size_t)n + blockIdx.x;
            for (int h = warp; h < H; h += nwarps)
                decode_rows<D>(q, kc, vc, n, h, H, Tmax, t_begin, t_end, scale_log2, slot * H + h, part_ml, part_o);
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Balanced split with bulk copies (up to kBulkMaxHeads heads): the same ranges, but one producer thread
// streams whole cache rows (all heads, contiguous in memory) into a ring of shared-memory stages with 1-D
// bulk copies (`cp.async.bulk`, completion counted on the stage's mbarrier), so up to kBulkStages x 2 x
// kBulkHalfStage bytes per SM are in flight without holding registers.  Consumer warp h runs the online
// softmax of head h over each stage from shared memory and releases it.  One CTA per SM.
struct BulkSmem {
    uint8_t stage[kBulkStages][2][kBulkHalfStage];  // [stage][K, V][rows x H x D bf16]
    uint64_t full[kBulkStages];
    uint64_t empty[kBulkStages];
    int s_vis[kBalancedMaxSeqs];
    int s_pre[kBalancedMaxSeqs + 1];
};

__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

template <int D>
__global__ void __launch_bounds__(32 * (kBulkMaxHeads + 1), 1)
decode_bulk_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                   const __nv_bfloat16* __restrict__ vc, const int* __restrict__ lens, float* __restrict__ part_ml,
                   float* __restrict__ part_o, int* __restrict__ meta, int N, int Tmax, int H, int window,
                   float scale_log2, int chunk_rows, int* err) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    BulkSmem& sm = *reinterpret_cast<BulkSmem*>(smem_raw);
    constexpr int G = RowLanes<D>::G, TPS = RowLanes<D>::TPS;
    constexpr int U = 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int st = 0; st < kBulkStages; ++st) {
            mbar_init(&sm.full[st], 1);
            mbar_init(&sm.empty[st], H);  // one arrival per consumer warp
        }
        fence_barrier_init();
    }
    const BalancedRange r = balanced_range(lens, meta, N, Tmax, window, sm.s_vis, sm.s_pre);  // syncs the CTA
    const size_t row_elems = (size_t)H * D;
    const uint32_t row_bytes = static_cast<uint32_t>(row_elems * 2);
    if (r.r0 < r.r1) {
        if (warp == H) {
            // ---------------------------------------------------------------- producer (one thread)
            if (lane == 0) {
                int ci = 0;  // chunks issued
                bool ok = true;
                for (int n = r.first_seq; ok && n < N && sm.s_pre[n] < r.r1; ++n) {
                    int tb, te;
                    if (!balanced_piece(r, lens, window, sm.s_vis, sm.s_pre, n, tb, te)) continue;
                    for (int t = tb; t < te; t += chunk_rows, ++ci) {
                        const int st = ci % kBulkStages;
                        if (!mbar_wait(&sm.empty[st], ((ci / kBulkStages) & 1) ^ 1)) {
                            set_device_error(err, NC_ERR_DEVICE_TIMEOUT);
                            ok = false;
                            break;
                        }
                        const uint32_t bytes = static_cast<uint32_t>(min(chunk_rows, te - t)) * row_bytes;
                        const size_t off = ((size_t)n * Tmax + t) * row_elems;
                        mbar_arrive_expect_tx(&sm.full[st], 2 * bytes);
                        bulk_load_1d(sm.stage[st][0], kc + off, bytes, &sm.full[st]);
                        bulk_load_1d(sm.stage[st][1], vc + off, bytes, &sm.full[st]);
                    }
                }
                // never leave while a copy into this CTA's shared memory may still land
                for (int x = ci - kBulkStages < 0 ? 0 : ci - kBulkStages; x < ci; ++x)
                    mbar_wait(&sm.full[x % kBulkStages], (x / kBulkStages) & 1);
            }
        } else if (warp < H) {
            // ---------------------------------------------------------------- consumer: head h = warp
            const int h = warp, g = lane / G, c = lane % G;
            int ci = 0;  // chunks consumed
            bool ok = true;
            for (int n = r.first_seq; ok && n < N && sm.s_pre[n] < r.r1; ++n) {
                int tb, te;
                if (!balanced_piece(r, lens, window, sm.s_vis, sm.s_pre, n, tb, te)) continue;
                float qf[8];
                load_query<D>(q, n, h, H, qf);
#pragma unroll
                for (int i = 0; i < 8; ++i) qf[i] *= scale_log2;
                float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.f;
                for (int t = tb; t < te; t += chunk_rows, ++ci) {
                    const int st = ci % kBulkStages;
                    if (!mbar_wait_warp(&sm.full[st], (ci / kBulkStages) & 1)) {
                        if (lane == 0) set_device_error(err, NC_ERR_DEVICE_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const int rows = min(chunk_rows, te - t);
                    const uint8_t* kst = sm.stage[st][0] + (size_t)h * D * 2 + c * 16;
                    const uint8_t* vst = sm.stage[st][1] + (size_t)h * D * 2 + c * 16;
                    for (int j0 = 0; j0 < rows; j0 += TPS * U) {
                        uint4 kr[U], vr[U];
                        bool valid[U];
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const int j = j0 + u * TPS + g;
                            valid[u] = j < rows;
                            kr[u] = make_uint4(0, 0, 0, 0);
                            vr[u] = make_uint4(0, 0, 0, 0);
                            if (valid[u]) {
                                kr[u] = *reinterpret_cast<const uint4*>(kst + (size_t)j * row_bytes);
                                vr[u] = *reinterpret_cast<const uint4*>(vst + (size_t)j * row_bytes);
                            }
                        }
                        softmax_steps<D, U>(kr, vr, valid, qf, m, l, acc);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.empty[st]);
                }
                if (!ok) break;
                merge_and_store<D>(m, l, acc, ((size_t)n + blockIdx.x) * H + h, part_ml, part_o);
            }
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Balanced combine, one warp per (sequence, head): the CTAs c0 .. c1 whose ranges hold sequence n's rows
// left partials in slots n + c0 .. n + c1.  Up to kCombineFast partials are read in one round of loads;
// more take three dependent rounds (the maxima, the sums with their weights, then the outputs, four
// partials at a time) per 32 partials.
template <int D>
__global__ void __launch_bounds__(256)
decode_balanced_combine_kernel(const float* __restrict__ part_ml, const float* __restrict__ part_o,
                               const int* __restrict__ meta, const int* __restrict__ lens,
                               __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int N, int Tmax, int H,
                               int* err) {
    constexpr int E = D / 32;  // elements per lane
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (gw >= N * H) return;
    const int n = gw / H, h = gw % H;
    const int L = lens[n];
    __nv_bfloat16* orow = o + (size_t)gw * D;
    if (L < 1 || L > Tmax) {
        if (lane == 0) set_device_error(err, NC_ERR_BAD_CACHE_LEN);
#pragma unroll
        for (int i = 0; i < E; ++i) orow[lane * E + i] = __float2bfloat16(NAN);
        if (lse != nullptr && lane == 0) lse[gw] = NAN;
        return;
    }
    const int P = meta[n], V = meta[n + 1] - P, per = meta[N + 1];
    const int c0 = P / per, k = (P + V - 1) / per - c0 + 1;
    const size_t base = ((size_t)n + c0) * H + h;  // partial s at base + s * H
    float M = -INFINITY, lsum = 0.f, acc[E];
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = 0.f;
    if (k <= kCombineFast) {
        // one round of loads: every lane reads all (max, sum) pairs (the same addresses across the warp) and
        // its E columns of every partial, then merges them with no further memory round trip
        float mv[kCombineFast], lv[kCombineFast], ov[kCombineFast][E];
#pragma unroll
        for (int s = 0; s < kCombineFast; ++s) {
            mv[s] = -INFINITY;
            lv[s] = 0.f;
#pragma unroll
            for (int i = 0; i < E; ++i) ov[s][i] = 0.f;
            if (s < k) {
                const size_t pidx = base + (size_t)s * H;
                mv[s] = part_ml[pidx * 2];
                lv[s] = part_ml[pidx * 2 + 1];
                const float* po = part_o + pidx * D + lane * E;
#pragma unroll
                for (int i = 0; i < E; ++i) ov[s][i] = po[i];
            }
        }
#pragma unroll
        for (int s = 0; s < kCombineFast; ++s) M = fmaxf(M, mv[s]);
#pragma unroll
        for (int s = 0; s < kCombineFast; ++s) {
            const float w = s < k ? exp2f(mv[s] - M) : 0.f;
            lsum = fmaf(lv[s], w, lsum);
#pragma unroll
            for (int i = 0; i < E; ++i) acc[i] = fmaf(ov[s][i], w, acc[i]);
        }
    } else {
        for (int s = lane; s < k; s += 32) M = fmaxf(M, part_ml[(base + (size_t)s * H) * 2]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        for (int s0 = 0; s0 < k; s0 += 32) {
            const int cnt = min(32, k - s0);
            float w = 0.f, lw = 0.f;
            if (lane < cnt) {
                const float* ml = part_ml + (base + (size_t)(s0 + lane) * H) * 2;
                w = exp2f(ml[0] - M);
                lw = ml[1] * w;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
            lsum += lw;
            int j = 0;
            for (; j + 4 <= cnt; j += 4) {
                float ov[4][E];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float* po = part_o + (base + (size_t)(s0 + j + u) * H) * D + lane * E;
#pragma unroll
                    for (int i = 0; i < E; ++i) ov[u][i] = po[i];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float wu = __shfl_sync(0xffffffffu, w, j + u);
#pragma unroll
                    for (int i = 0; i < E; ++i) acc[i] = fmaf(ov[u][i], wu, acc[i]);
                }
            }
            for (; j < cnt; ++j) {
                const float wj = __shfl_sync(0xffffffffu, w, j);
                const float* po = part_o + (base + (size_t)(s0 + j) * H) * D + lane * E;
#pragma unroll
                for (int i = 0; i < E; ++i) acc[i] = fmaf(po[i], wj, acc[i]);
            }
        }
    }
    const float inv = 1.f / lsum;
#pragma unroll
    for (int i = 0; i < E; ++i) orow[lane * E + i] = __float2bfloat16_rn(acc[i] * inv);
    if (lse != nullptr && lane == 0) lse[gw] = (M + log2f(lsum)) * kLn2;
}

// One warp per (sequence, head): merge the partials of the splits that saw rows.
template <int D>
__global__ void __launch_bounds__(256)
decode_combine_kernel(const float* __restrict__ part_ml, const float* __restrict__ part_o,
                      const int* __restrict__ lens, __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                      int N, int Tmax, int H, int window, int n_splits, int chunk, int* err) {
    constexpr int E = D / 32;  // elements per lane
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    // launched as a programmatic dependent of the split kernel: wait for its partials
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (gw >= N * H) return;
    const int n = gw / H, h = gw % H;
    const int L = lens[n];
    __nv_bfloat16* orow = o + (size_t)gw * D;
    if (L < 1 || L > Tmax) {
        if (lane == 0) set_device_error(err, NC_ERR_BAD_CACHE_LEN);
#pragma unroll
        for (int i = 0; i < E; ++i) orow[lane * E + i] = __float2bfloat16(NAN);
        if (lse != nullptr && lane == 0) lse[gw] = NAN;
        return;
    }
    const int lo = visible_lo(L, window);
    const int used = (L - lo + chunk - 1) / chunk;
    const float* ml = part_ml + ((size_t)n * n_splits * H + h) * 2;  // split s at ml[s * H * 2]
    // running maximum over the splits, lanes striding over them
    float M = -INFINITY;
    for (int s = lane; s < used; s += 32) M = fmaxf(M, ml[(size_t)s * H * 2]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float lsum = 0.f, acc[E];
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = 0.f;
    int s = 0;
    for (; s + 4 <= used; s += 4) {  // four splits' loads in flight
        float w[4], lp[4], ov[4][E];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t pidx = ((size_t)n * n_splits + s + u) * H + h;
            w[u] = part_ml[pidx * 2];
            lp[u] = part_ml[pidx * 2 + 1];
#pragma unroll
            for (int i = 0; i < E; ++i) ov[u][i] = part_o[pidx * D + lane * E + i];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float wu = exp2f(w[u] - M);
            lsum = fmaf(lp[u], wu, lsum);
#pragma unroll
            for (int i = 0; i < E; ++i) acc[i] = fmaf(ov[u][i], wu, acc[i]);
        }
    }
    for (; s < used; ++s) {
        const size_t pidx = ((size_t)n * n_splits + s) * H + h;
        const float w = exp2f(part_ml[pidx * 2] - M);
        lsum = fmaf(part_ml[pidx * 2 + 1], w, lsum);
        const float* po = part_o + pidx * D + lane * E;
#pragma unroll
        for (int i = 0; i < E; ++i) acc[i] = fmaf(po[i], w, acc[i]);
    }
    const float inv = 1.f / lsum;
#pragma unroll
    for (int i = 0; i < E; ++i) orow[lane * E + i] = __float2bfloat16_rn(acc[i] * inv);
    if (lse != nullptr && lane == 0) lse[gw] = (M + log2f(lsum)) * kLn2;
}

}  // namespace

// Launch the combine as a programmatic dependent of the split kernel on the same stream, so its
// launch overlaps the split kernel's tail (it waits for the split results on the device).
template <typename... KArgs, typename... Args>
static void launch_combine(void (*kern)(KArgs...), int blocks, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kern, args...);
}

int decode_chunk_rows(int D) { return D == 64 ? 128 : 64; }

bool decode_balanced(int N, int Tmax) {
    return N <= kBalancedMaxSeqs && (int64_t)N * Tmax < (int64_t(1) << 30);  // row offsets stay far from overflow
}

namespace {
size_t round_up256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

DecodeLayout decode_layout(int N, int Tmax, int H, int D, int window) {
    DecodeLayout d;
    size_t parts;
    if (decode_balanced(N, Tmax)) {
        parts = ((size_t)N + kDecodeMaxGrid) * H;
    } else {
        const int chunk = decode_chunk_rows(D);
        const int w_eff = (window <= 0 || window >= Tmax) ? Tmax : window;
        parts = (size_t)N * ((w_eff + chunk - 1) / chunk) * H;
    }
    d.off_ml = 0;
    d.off_o = round_up256(parts * 2 * 4);
    d.off_meta = d.off_o + round_up256(parts * D * 4);
    d.bytes = d.off_meta + round_up256(((size_t)N + 2) * 4);
    return d;
}

cudaError_t launch_decode(const void* q, const void* kcache, const void* vcache, const int* lens, void* o,
                          float* lse, int N, int Tmax, int H, int D, int window, float scale, void* workspace,
                          int* err, cudaStream_t stream) {
    const DecodeLayout lay = decode_layout(N, Tmax, H, D, window);
    char* ws = static_cast<char*>(workspace);
    float* part_ml = reinterpret_cast<float*>(ws + lay.off_ml);
    float* part_o = reinterpret_cast<float*>(ws + lay.off_o);
    int* meta = reinterpret_cast<int*>(ws + lay.off_meta);
    const float scale_log2 = scale * kLog2e;
    const int threads = 32 * (H < kDecodeMaxThreads / 32 ? H : kDecodeMaxThreads / 32);
    const int cblocks = (N * H * 32 + 255) / 256;
    auto bq = static_cast<const __nv_bfloat16*>(q);
    auto bk = static_cast<const __nv_bfloat16*>(kcache);
    auto bv = static_cast<const __nv_bfloat16*>(vcache);
    auto bo = static_cast<__nv_bfloat16*>(o);
    if (decode_balanced(N, Tmax) && H <= kBulkMaxHeads) {
        // one CTA per SM (its stage ring takes most of the shared memory), H consumer warps + a producer warp
        auto split = D == 128 ? decode_bulk_kernel<128> : decode_bulk_kernel<64>;
        static std::atomic<bool> attr_done[2][kAttrDevices];
        const int smem = static_cast<int>(sizeof(BulkSmem));
        cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(split), smem, attr_done[D == 128 ? 1 : 0]);
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = multiprocessor_count(&sms);
        if (e != cudaSuccess) return e;
        const int grid = sms < kDecodeMaxGrid ? sms : kDecodeMaxGrid;
        const int fit = kBulkHalfStage / (H * D * 2), batch = D == 128 ? 8 : 16;  // rows of one U-step batch
        const int chunk_rows = fit >= batch ? fit / batch * batch : fit;
        split<<<grid, 32 * (H + 1), smem, stream>>>(bq, bk, bv, lens, part_ml, part_o, meta, N, Tmax, H, window,
                                                     scale_log2, chunk_rows, err);
        if (D == 128)
            launch_combine(decode_balanced_combine_kernel<128>, cblocks, stream, (const float*)part_ml,
                           (const float*)part_o, (const int*)meta, lens, bo, lse, N, Tmax, H, err);
        else
            launch_combine(decode_balanced_combine_kernel<64>, cblocks, stream, (const float*)part_ml,
                           (const float*)part_o, (const int*)meta, lens, bo, lse, N, Tmax, H, err);
    } else if (decode_balanced(N, Tmax)) {
        // as many CTAs as fit on the GPU at once (looked up per call), at most kDecodeMaxGrid
        auto split = D == 128 ? decode_balanced_kernel<128> : decode_balanced_kernel<64>;
        int sms = 0, per_sm = 0;
        cudaError_t e = multiprocessor_count(&sms);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, split, threads, 0);
        if (e != cudaSuccess) return e;
        const long want = (long)sms * (per_sm > 0 ? per_sm : 1);
        const int grid = static_cast<int>(want < kDecodeMaxGrid ? want : kDecodeMaxGrid);
        split<<<grid, threads, 0, stream>>>(bq, bk, bv, lens, part_ml, part_o, meta, N, Tmax, H, window, scale_log2);
        if (D == 128)
            launch_combine(decode_balanced_combine_kernel<128>, cblocks, stream, (const float*)part_ml,
                           (const float*)part_o, (const int*)meta, lens, bo, lse, N, Tmax, H, err);
        else
            launch_combine(decode_balanced_combine_kernel<64>, cblocks, stream, (const float*)part_ml,
                           (const float*)part_o, (const int*)meta, lens, bo, lse, N, Tmax, H, err);
    } else {
        const int chunk = decode_chunk_rows(D);
        const int w_eff = (window <= 0 || window >= Tmax) ? Tmax : window;
        const int n_splits = (w_eff + chunk - 1) / chunk;  // splits any sequence can need
        const int grid = n_splits * N;
        if (D == 128) {
            decode_split_kernel<128><<<grid, threads, 0, stream>>>(bq, bk, bv, lens, part_ml, part_o, N, Tmax, H,
                                                                   window, scale_log2, n_splits, chunk);
            launch_combine(decode_combine_kernel<128>, cblocks, stream, (const float*)part_ml, (const float*)part_o,
                           lens, bo, lse, N, Tmax, H, window, n_splits, chunk, err);
        } else {
            decode_split_kernel<64><<<grid, threads, 0, stream>>>(bq, bk, bv, lens, part_ml, part_o, N, Tmax, H,
                                                                  window, scale_log2, n_splits, chunk);
            launch_combine(decode_combine_kernel<64>, cblocks, stream, (const float*)part_ml, (const float*)part_o,
                           lens, bo, lse, N, Tmax, H, window, n_splits, chunk, err);
        }
    }
    count_launches(2);
    return cudaGetLastError();
}

}  // namespace nc
