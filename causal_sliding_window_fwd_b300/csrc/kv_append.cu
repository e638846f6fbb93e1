// Append of new tokens' keys and values to a padded KV cache ("nanochat" walkthrough, page 4: the Engine's
// KV cache, which prefill fills and every decode step extends).  The cache length of sequence n, L_n, already
// counts its Tq new tokens (the convention of prefill and decode), so new row t goes to cache position
// L_n - Tq + t:
//   kcache[n, L_n - Tq + t] = k_new[n, t],   vcache[n, L_n - Tq + t] = v_new[n, t].
//
// A plain copy, bound by HBM: a cache row [H, D] is contiguous in both tensors, so one thread moves 16 bytes
// of a row of k and the same 16 bytes of v, in a grid-stride loop.  A length outside [Tq, Tmax] sets
// NC_ERR_BAD_CACHE_LEN and leaves that sequence's cache untouched.
#include <cstdint>

#include "nc_attn.h"
#include "nc_kernels.h"
#include "nc_ptx.cuh"

namespace nc {

namespace {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new, uint4* kcache,
                                                        uint4* vcache, const int* __restrict__ lens, int Tq,
                                                        int Tmax, long units_per_row, long n_units, int* err) {
    for (long u = (long)blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += (long)gridDim.x * blockDim.x) {
        const long row = u / units_per_row;  // (n, t)
        const long c = u - row * units_per_row;
        const int n = static_cast<int>(row / Tq), t = static_cast<int>(row - (long)n * Tq);
        const int L = __ldg(lens + n);
        if (L < Tq || L > Tmax) {
            if (t == 0 && c == 0) set_device_error(err, NC_ERR_BAD_CACHE_LEN);
            continue;
        }
        const long dst = ((long)n * Tmax + (L - Tq + t)) * units_per_row + c;
        kcache[dst] = k_new[u];
        vcache[dst] = v_new[u];
    }
}

}  // namespace

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* kcache, void* vcache, const int* lens, int N,
                             int Tq, int Tmax, int H, int D, int* err, cudaStream_t st) {
    const long units_per_row = (long)H * D / 8;
    const long n_units = (long)N * Tq * units_per_row;
    int sms = 0;
    cudaError_t e = multiprocessor_count(&sms);
    if (e != cudaSuccess) return e;
    const long want = (n_units + 255) / 256, cap = (long)sms * 8;
    kv_append_kernel<<<static_cast<unsigned>(want < cap ? want : cap), 256, 0, st>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), static_cast<uint4*>(kcache),
        static_cast<uint4*>(vcache), lens, Tq, Tmax, units_per_row, n_units, err);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace nc
