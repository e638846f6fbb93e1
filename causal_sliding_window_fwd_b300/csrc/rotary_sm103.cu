// Rotary position embedding of [B, T, H, D] bf16 tensors ("nanochat" walkthrough, page 4, comment thread:
// a Llama-like model, whose rotate-half pairing is the reading taken).  Row t of the caller's fp32 tables
// [T, D/2] holds the cosine and sine for position t; pair (x_i, x_{i+D/2}) becomes
//   y_i = x_i c - x_{i+D/2} s,   y_{i+D/2} = x_i s + x_{i+D/2} c,
// evaluated in float32 as y_i = fma(x_i, c, -fl(x_{i+D/2} s)), y_{i+D/2} = fma(x_i, s, fl(x_{i+D/2} c)) and
// rounded to bf16 (nearest, ties to even); with `inverse` the transpose (the turn back, which takes
// gradients with respect to the turned tensor to gradients with respect to the input).
//
// Elementwise and bound by HBM: one thread per (row, 8 pairs) reads 2 x 16 bytes of the row and
// 2 x 32 bytes of the tables (T x D/2 x 8 bytes in all, which stay in L2), and writes 2 x 16 bytes.  One
// launch can turn two tensors of the same shape (q and k): blockIdx.y picks the tensor.  x and y may be
// the same tensor (in place): each thread reads its two vectors before writing them.
#include <cstdint>
#include <cuda_bf16.h>

#include "nc_kernels.h"
#include "nc_ptx.cuh"

namespace nc {

namespace {

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ void load8(const float* __restrict__ t, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(t));
    const float4 b = __ldg(reinterpret_cast<const float4*>(t) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

template <int D, bool kInverse>
__global__ void __launch_bounds__(256) rotary_kernel(const uint4* x0, uint4* y0, const uint4* x1, uint4* y1,
                                                     const float* __restrict__ rcos, const float* __restrict__ rsin,
                                                     size_t n_units, int T, int H) {
    constexpr int kUnits = D / 16;  // 8-pair units per row
    constexpr int kRowVec = D / 8;  // 16-byte vectors per row
    const uint4* x = blockIdx.y ? x1 : x0;
    uint4* y = blockIdx.y ? y1 : y0;
    for (size_t w = (size_t)blockIdx.x * blockDim.x + threadIdx.x; w < n_units; w += (size_t)gridDim.x * blockDim.x) {
        const size_t row = w / kUnits;  // a shift
        const int u = static_cast<int>(w - row * kUnits);
        // B * T * H < 2^31 (checked by every entry point), so the position comes from 32-bit divisions
        const uint32_t row32 = static_cast<uint32_t>(row);
        const int pos = static_cast<int>((row32 / static_cast<uint32_t>(H)) % static_cast<uint32_t>(T));
        const size_t i1 = row * kRowVec + u, i2 = i1 + kUnits;  // dimensions 8u .. 8u+7 and their partners
        float a[8], b[8], c[8], s[8];
        unpack_bf16x8(x[i1], a);
        unpack_bf16x8(x[i2], b);
        load8(rcos + (size_t)pos * (D / 2) + 8 * u, c);
        load8(rsin + (size_t)pos * (D / 2) + 8 * u, s);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float sn = kInverse ? -s[e] : s[e];
            // one product and one fused multiply-add per output, each rounded once
            const float ya = __fmaf_rn(a[e], c[e], -__fmul_rn(b[e], sn));
            const float yb = __fmaf_rn(a[e], sn, __fmul_rn(b[e], c[e]));
            a[e] = ya;
            b[e] = yb;
        }
        y[i1] = pack8(a);
        y[i2] = pack8(b);
    }
}

}  // namespace

cudaError_t launch_rotary(const void* x0, void* y0, const void* x1, void* y1, const float* rcos, const float* rsin,
                          int B, int T, int H, int D, bool inverse, cudaStream_t st) {
    const size_t n_units = (size_t)B * T * H * (D / 16);
    int sms = 0;
    cudaError_t e = multiprocessor_count(&sms);
    if (e != cudaSuccess) return e;
    // grid-stride over the units: 8 resident 256-thread CTAs per SM per tensor, fewer for small tensors
    const size_t want = (n_units + 255) / 256, cap = (size_t)sms * (x1 ? 4 : 8);
    const dim3 grid(static_cast<unsigned>(want < cap ? want : cap), x1 ? 2u : 1u);
    auto a0 = static_cast<const uint4*>(x0);
    auto b0 = static_cast<uint4*>(y0);
    auto a1 = static_cast<const uint4*>(x1);
    auto b1 = static_cast<uint4*>(y1);
    if (D == 128)
        inverse ? rotary_kernel<128, true><<<grid, 256, 0, st>>>(a0, b0, a1, b1, rcos, rsin, n_units, T, H)
                : rotary_kernel<128, false><<<grid, 256, 0, st>>>(a0, b0, a1, b1, rcos, rsin, n_units, T, H);
    else
        inverse ? rotary_kernel<64, true><<<grid, 256, 0, st>>>(a0, b0, a1, b1, rcos, rsin, n_units, T, H)
                : rotary_kernel<64, false><<<grid, 256, 0, st>>>(a0, b0, a1, b1, rcos, rsin, n_units, T, H);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace nc
