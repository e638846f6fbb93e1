// Warp-per-row CUDA-core attention backward.
//
// One warp owns one query row (dQ) or one key row (dK/dV) and walks the
// keys/queries that the causal window makes visible, recomputing the softmax
// weights from the stored log-sum-exp in fp32 (see the C ABI header for the
// operation and its sources).  This is the plain first CUDA path of the
// backward; the tensor-core kernel replaces it on the hot path.
#include <cstdint>
#include <cuda_bf16.h>

#include "nc_attn.h"
#include "nc_kernels.h"

namespace nc {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int E>
__device__ __forceinline__ void load_row(const __nv_bfloat16* p, float (&f)[E]) {
#pragma unroll
    for (int i = 0; i < E; i += 2) {
        float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p + i));
        f[i] = t.x;
        f[i + 1] = t.y;
    }
}

template <int E>
__device__ __forceinline__ float warp_dot(const float (&a)[E], const float (&b)[E]) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) s = fmaf(a[i], b[i], s);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    return s;
}

template <int E>
__device__ __forceinline__ void store_row(__nv_bfloat16* p, const float (&f)[E], float mul) {
#pragma unroll
    for (int i = 0; i < E; i += 2)
        *reinterpret_cast<__nv_bfloat162*>(p + i) = __floats2bfloat162_rn(f[i] * mul, f[i + 1] * mul);
}

__device__ __forceinline__ int eff_window(int window, int T) { return (window <= 0 || window >= T) ? T : window; }

// Delta_i = sum_d dO_id * O_id for every row.
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_rowwarp(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         float* __restrict__ delta, int B, int T, int H) {
    constexpr int E = D / 32;
    const long gw = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= (long)B * T * H) return;
    const int h = gw % H;
    const int i = (gw / H) % T;
    const int b = gw / ((long)H * T);
    const size_t off = (((size_t)b * T + i) * H + h) * D + lane * E;
    float a[E], c[E];
    load_row<E>(o + off, a);
    load_row<E>(dO + off, c);
    const float d = warp_dot<E>(a, c);
    if (lane == 0) delta[((size_t)b * H + h) * T + i] = d;
}

// dQ_i = scale * sum_j p_ij (dp_ij - Delta_i) k_j
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_rowwarp(const __nv_bfloat16* __restrict__ q,
                                                      const __nv_bfloat16* __restrict__ k,
                                                      const __nv_bfloat16* __restrict__ v,
                                                      const __nv_bfloat16* __restrict__ dO,
                                                      const float* __restrict__ lse, const float* __restrict__ delta,
                                                      __nv_bfloat16* __restrict__ dq, int B, int T, int H, int window,
                                                      float scale) {
    constexpr int E = D / 32;
    const long gw = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= (long)B * T * H) return;
    const int h = gw % H;
    const int i = (gw / H) % T;
    const int b = gw / ((long)H * T);
    const int W = eff_window(window, T);
    const int lo = i - W + 1 < 0 ? 0 : i - W + 1;
    const size_t rs = (size_t)H * D;
    const size_t base = (size_t)b * T * rs + (size_t)h * D + lane * E;
    const size_t ridx = ((size_t)b * H + h) * T + i;
    const float lse2 = lse[ridx] * kLog2e, dlt = delta[ridx], sl2 = scale * kLog2e;
    float qf[E], gf[E], acc[E];
    load_row<E>(q + base + (size_t)i * rs, qf);
    load_row<E>(dO + base + (size_t)i * rs, gf);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int j = lo; j <= i; ++j) {
        float kf[E], vf[E];
        load_row<E>(k + base + (size_t)j * rs, kf);
        load_row<E>(v + base + (size_t)j * rs, vf);
        const float p = exp2f(warp_dot<E>(qf, kf) * sl2 - lse2);
        const float ds = p * (warp_dot<E>(gf, vf) - dlt);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(ds, kf[e], acc[e]);
    }
    store_row<E>(dq + base + (size_t)i * rs, acc, scale);
}

// dK_j = scale * sum_i ds_ij q_i and dV_j = sum_i p_ij dO_i over the queries that see key j.
template <int D>
__global__ void __launch_bounds__(256) bwd_dkdv_rowwarp(const __nv_bfloat16* __restrict__ q,
                                                        const __nv_bfloat16* __restrict__ k,
                                                        const __nv_bfloat16* __restrict__ v,
                                                        const __nv_bfloat16* __restrict__ dO,
                                                        const float* __restrict__ lse,
                                                        const float* __restrict__ delta, __nv_bfloat16* __restrict__ dk,
                                                        __nv_bfloat16* __restrict__ dv, int B, int T, int H,
                                                        int window, float scale) {
    constexpr int E = D / 32;
    const long gw = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= (long)B * T * H) return;
    const int h = gw % H;
    const int j = (gw / H) % T;
    const int b = gw / ((long)H * T);
    const int W = eff_window(window, T);
    const int hi = j + W - 1 < T - 1 ? j + W - 1 : T - 1;
    const size_t rs = (size_t)H * D;
    const size_t base = (size_t)b * T * rs + (size_t)h * D + lane * E;
    const float sl2 = scale * kLog2e;
    float kf[E], vf[E], ak[E], av[E];
    load_row<E>(k + base + (size_t)j * rs, kf);
    load_row<E>(v + base + (size_t)j * rs, vf);
#pragma unroll
    for (int e = 0; e < E; ++e) ak[e] = av[e] = 0.f;
    for (int i = j; i <= hi; ++i) {
        float qf[E], gf[E];
        load_row<E>(q + base + (size_t)i * rs, qf);
        load_row<E>(dO + base + (size_t)i * rs, gf);
        const size_t ridx = ((size_t)b * H + h) * T + i;
        const float p = exp2f(warp_dot<E>(qf, kf) * sl2 - lse[ridx] * kLog2e);
        const float ds = p * (warp_dot<E>(gf, vf) - delta[ridx]);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            av[e] = fmaf(p, gf[e], av[e]);
            ak[e] = fmaf(ds, qf[e], ak[e]);
        }
    }
    store_row<E>(dk + base + (size_t)j * rs, ak, scale);
    store_row<E>(dv + base + (size_t)j * rs, av, 1.f);
}

template <int D>
cudaError_t bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                     void* dq, void* dk, void* dv, int B, int T, int H, int window, float scale, float* delta,
                     cudaStream_t st) {
    const long rows = (long)B * T * H;
    const unsigned blocks = (unsigned)((rows * 32 + 255) / 256);
    auto bq = (const __nv_bfloat16*)q;
    auto bk = (const __nv_bfloat16*)k;
    auto bv = (const __nv_bfloat16*)v;
    auto bg = (const __nv_bfloat16*)dO;
    bwd_delta_rowwarp<D><<<blocks, 256, 0, st>>>((const __nv_bfloat16*)o, bg, delta, B, T, H);
    bwd_dq_rowwarp<D><<<blocks, 256, 0, st>>>(bq, bk, bv, bg, lse, delta, (__nv_bfloat16*)dq, B, T, H, window,
                                              scale);
    bwd_dkdv_rowwarp<D><<<blocks, 256, 0, st>>>(bq, bk, bv, bg, lse, delta, (__nv_bfloat16*)dk,
                                                (__nv_bfloat16*)dv, B, T, H, window, scale);
    count_launches(3);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                       void* dq, void* dk, void* dv, int B, int T, int H, int D, int window, float scale,
                       float* dq_acc, float* delta, int* err, cudaStream_t st) {
    (void)dq_acc;
    (void)err;
    return D == 128 ? bwd_impl<128>(q, k, v, o, dO, lse, dq, dk, dv, B, T, H, window, scale, delta, st)
                    : bwd_impl<64>(q, k, v, o, dO, lse, dq, dk, dv, B, T, H, window, scale, delta, st);
}

}  // namespace nc
