// Append of new tokens' keys and values to a padded KV cache ("nanochat" walkthrough, page 4: the Engine's
// KV cache, which prefill fills and every decode step extends).  The cache length of sequence n, L_n, already
// counts its Tq new tokens (the convention of prefill and decode), so new row t goes to cache position
// L_n - Tq + t:
//   kcache[n, L_n - Tq + t] = k_new[n, t],   vcache[n, L_n - Tq + t] = v_new[n, t].
//
// A plain copy, bound by HBM: a cache row [H, D] is contiguous in both tensors, so one warp copies one
// (sequence, token) row of k and of v, lanes striding over its 16-byte units (the row's destination is worked
// out once per row).  A length outside [Tq, Tmax] sets NC_ERR_BAD_CACHE_LEN and leaves that sequence's cache
// untouched.
#include <cstdint>

#include "nc_attn.h"
#include "nc_kernels.h"
#include "nc_ptx.cuh"

namespace nc {

namespace {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new, uint4* __restrict__ kcache,
                                                        uint4* __restrict__ vcache, const int* __restrict__ lens, int Tq,
                                                        int Tmax, int units_per_row, int rows, int* err) {
    const int lane = threadIdx.x & 31;
    const int warps = static_cast<int>(gridDim.x * (blockDim.x / 32));
    for (int row = static_cast<int>(blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32); row < rows; row += warps) {
        const int n = row / Tq, t = row - n * Tq;
        const int L = __ldg(lens + n);
        if (L < Tq || L > Tmax) {
            if (t == 0 && lane == 0) set_device_error(err, NC_ERR_BAD_CACHE_LEN);
            continue;
        }
        const uint4* ks = k_new + static_cast<size_t>(row) * units_per_row;
        const uint4* vs = v_new + static_cast<size_t>(row) * units_per_row;
        const size_t dst = (static_cast<size_t>(n) * Tmax + (L - Tq + t)) * units_per_row;
        uint4* kd = kcache + dst;
        uint4* vd = vcache + dst;
        // four units of k and of v in flight per lane before their stores (the caches overlap no input)
        constexpr int U = 4;
        for (int c0 = lane; c0 < units_per_row; c0 += 32 * U) {
            uint4 a[U], b[U];
#pragma unroll
            for (int i = 0; i < U; ++i) {
                const int c = c0 + 32 * i;
                if (c < units_per_row) {
                    a[i] = ks[c];
                    b[i] = vs[c];
                }
            }
#pragma unroll
            for (int i = 0; i < U; ++i) {
                const int c = c0 + 32 * i;
                if (c < units_per_row) {
                    kd[c] = a[i];
                    vd[c] = b[i];
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* kcache, void* vcache, const int* lens, int N,
                             int Tq, int Tmax, int H, int D, int* err, cudaStream_t st) {
    const int units_per_row = H * D / 8;  // N * Tmax * H < 2^31 (checked by the caller), so these fit in int
    const int rows = N * Tq;
    int sms = 0;
    cudaError_t e = multiprocessor_count(&sms);
    if (e != cudaSuccess) return e;
    // 8 rows (warps) per 256-thread CTA, up to 8 CTAs per SM, grid-stride over the rest
    const long want = (rows + 7) / 8, cap = (long)sms * 8;
    kv_append_kernel<<<static_cast<unsigned>(want < cap ? want : cap), 256, 0, st>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), static_cast<uint4*>(kcache),
        static_cast<uint4*>(vcache), lens, Tq, Tmax, units_per_row, rows, err);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace nc
