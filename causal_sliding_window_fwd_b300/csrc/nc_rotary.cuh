// Rotary position embedding applied in place to a 128-row bf16 tile in shared memory, between the
// TMA landing and the tensor-core products that read it ("nanochat" walkthrough, page 4, comment
// thread: the model is Llama-like; the rotate-half pairing of Llama is the reading taken).
//
// The tile has the TMA layout of the attention kernels: D / 64 chunks of [128 rows][64 columns] bf16,
// 128-byte swizzle (16-byte unit u of row r at byte ((u ^ (r & 7)) << 4) of the row).  Row r holds
// position pos0 + r.  Each pair (x_i, x_{i+D/2}) of a row is turned by the angle whose cosine and sine
// the caller's fp32 tables hold at (position, i):
//   y_i = x_i c - x_{i+D/2} s,   y_{i+D/2} = x_i s + x_{i+D/2} c.
// With kInverse the transpose is applied instead (the turn back).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "nc_ptx.cuh"

namespace nc {

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Turn the pairs (x1[e], x2[e]) of eight consecutive dimensions with cosines c[e] and sines s[e].
template <bool kInverse>
__device__ __forceinline__ void turn8(float (&x1)[8], float (&x2)[8], const float (&c)[8], const float (&s)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float sn = kInverse ? -s[e] : s[e];
        // explicit roundings (one product, then one fused multiply-add) so that every kernel that turns a
        // row gets the same bits
        const float y1 = __fmaf_rn(x1[e], c[e], -__fmul_rn(x2[e], sn));
        const float y2 = __fmaf_rn(x1[e], sn, __fmul_rn(x2[e], c[e]));
        x1[e] = y1;
        x2[e] = y2;
    }
}

__device__ __forceinline__ void load_cs8(const float* __restrict__ t, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(t));
    const float4 b = __ldg(reinterpret_cast<const float4*>(t) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Rotate rows [0, 128) of `tile` whose position pos0 + r is below pos_end (rows past the sequence are
// left as they are: their scores are masked).  The work is split over `nthr` threads, thread `tid`
// taking 8-pair units in turn.  The caller fences (generic -> async proxy) and signals afterwards.
template <int D>
__device__ __forceinline__ void rotate_tile(uint8_t* tile, int pos0, int pos_end, const float* __restrict__ rcos,
                                            const float* __restrict__ rsin, int tid, int nthr) {
    constexpr int kUnits = D / 16;  // 8-pair units of a row: pairs i = 8u .. 8u + 7
    constexpr int kHalf = D / 2;
    for (int w = tid; w < 128 * kUnits; w += nthr) {
        const int r = w / kUnits, u = w - (w / kUnits) * kUnits;
        const int pos = pos0 + r;
        if (pos >= pos_end) continue;
        uint8_t* row = tile + r * 128;
        // dimension 8u + e and its partner 8u + e + D/2: for D = 128 the same unit of the second
        // 64-column chunk, for D = 64 unit u + 4 of the same chunk
        uint4* p1 = reinterpret_cast<uint4*>(row + ((u ^ (r & 7)) << 4));
        uint4* p2 = D == 128 ? reinterpret_cast<uint4*>(row + 128 * 128 + ((u ^ (r & 7)) << 4))
                             : reinterpret_cast<uint4*>(row + (((u + 4) ^ (r & 7)) << 4));
        float x1[8], x2[8], c[8], s[8];
        unpack_bf16x8(*p1, x1);
        unpack_bf16x8(*p2, x2);
        load_cs8(rcos + static_cast<size_t>(pos) * kHalf + 8 * u, c);
        load_cs8(rsin + static_cast<size_t>(pos) * kHalf + 8 * u, s);
        turn8<false>(x1, x2, c, s);
        *p1 = make_uint4(pack_bf16x2(x1[0], x1[1]), pack_bf16x2(x1[2], x1[3]), pack_bf16x2(x1[4], x1[5]),
                         pack_bf16x2(x1[6], x1[7]));
        *p2 = make_uint4(pack_bf16x2(x2[0], x2[1]), pack_bf16x2(x2[2], x2[3]), pack_bf16x2(x2[4], x2[5]),
                         pack_bf16x2(x2[6], x2[7]));
    }
}

}  // namespace nc
