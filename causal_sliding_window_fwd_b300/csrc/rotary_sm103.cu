// Standalone rotary position embedding of a [B, T, H, D] bf16 tensor: the unfused form of the turn the
// rotary attention kernels apply while q and k sit in shared memory ("nanochat" walkthrough, page 4,
// comment thread: a Llama-like model, whose rotate-half pairing is the reading taken).  Row t of the
// caller's fp32 tables [T, D/2] holds the cosine and sine for position t; pair (x_i, x_{i+D/2}) becomes
//   y_i = x_i c - x_{i+D/2} s,   y_{i+D/2} = x_i s + x_{i+D/2} c,
// and with `inverse` the transpose (the turn back, which takes gradients with respect to the rotated
// tensor to gradients with respect to the input).
//
// x and y may be the same tensor (in place): each thread reads its two vectors before writing them.
// Elementwise and bound by HBM: one thread per (row, 8 pairs) reads 2 x 16 bytes of the row and
// 2 x 32 bytes of the tables (T x D/2 x 8 bytes in all, which stay in L2), and writes 2 x 16 bytes.
#include <cstdint>
#include <cuda_bf16.h>

#include "nc_kernels.h"
#include "nc_ptx.cuh"
#include "nc_rotary.cuh"

namespace nc {

template <int D, bool kInverse>
__global__ void __launch_bounds__(256) rotary_kernel(const uint4* x, const float* __restrict__ rcos,
                                                     const float* __restrict__ rsin, uint4* y,
                                                     size_t n_units, int T, int H) {
    constexpr int kUnits = D / 16;  // 8-pair units per row
    constexpr int kRowVec = D / 8;  // 16-byte vectors per row
    for (size_t w = (size_t)blockIdx.x * blockDim.x + threadIdx.x; w < n_units; w += (size_t)gridDim.x * blockDim.x) {
        const size_t row = w / kUnits;
        const int u = static_cast<int>(w - row * kUnits);
        const int pos = static_cast<int>((row / H) % T);
        const size_t i1 = row * kRowVec + u, i2 = i1 + kUnits;  // dimensions 8u .. 8u+7 and their partners
        float x1[8], x2[8], c[8], s[8];
        unpack_bf16x8(x[i1], x1);
        unpack_bf16x8(x[i2], x2);
        load_cs8(rcos + (size_t)pos * (D / 2) + 8 * u, c);
        load_cs8(rsin + (size_t)pos * (D / 2) + 8 * u, s);
        turn8<kInverse>(x1, x2, c, s);
        y[i1] = make_uint4(pack_bf16x2(x1[0], x1[1]), pack_bf16x2(x1[2], x1[3]), pack_bf16x2(x1[4], x1[5]),
                           pack_bf16x2(x1[6], x1[7]));
        y[i2] = make_uint4(pack_bf16x2(x2[0], x2[1]), pack_bf16x2(x2[2], x2[3]), pack_bf16x2(x2[4], x2[5]),
                           pack_bf16x2(x2[6], x2[7]));
    }
}

cudaError_t launch_rotary(const void* x, const float* rcos, const float* rsin, void* y, int B, int T, int H, int D,
                          bool inverse, cudaStream_t st) {
    const size_t n_units = (size_t)B * T * H * (D / 16);
    int sms = 0;
    cudaError_t e = multiprocessor_count(&sms);
    if (e != cudaSuccess) return e;
    // grid-stride over the units: 8 resident 256-thread CTAs per SM, fewer when the tensor is small
    const size_t want = (n_units + 255) / 256, cap = (size_t)sms * 8;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    auto xs = static_cast<const uint4*>(x);
    auto ys = static_cast<uint4*>(y);
    if (D == 128)
        inverse ? rotary_kernel<128, true><<<grid, 256, 0, st>>>(xs, rcos, rsin, ys, n_units, T, H)
                : rotary_kernel<128, false><<<grid, 256, 0, st>>>(xs, rcos, rsin, ys, n_units, T, H);
    else
        inverse ? rotary_kernel<64, true><<<grid, 256, 0, st>>>(xs, rcos, rsin, ys, n_units, T, H)
                : rotary_kernel<64, false><<<grid, 256, 0, st>>>(xs, rcos, rsin, ys, n_units, T, H);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace nc
