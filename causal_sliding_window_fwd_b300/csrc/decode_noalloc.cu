// Decode entry point that allocates nothing and takes no workspace.
//
// Some callers cannot call cudaMalloc at the point where they decode:
// inference engines whose own allocator has reserved the device memory up
// front (a further cudaMalloc fails or fragments their pool), plug-ins that
// are handed only their input and output buffers, and latency-critical token
// loops that cannot afford the device-wide synchronisation cudaMalloc and
// cudaFree may imply.  nc_attn_decode_noalloc serves them: its split-K partial
// results go to a fixed scratch array in this library's own device memory (a
// file-scope __device__ array, so every GPU that loads the library holds it
// until the process exits).  It runs the same kernels as nc_attn_decode.
//
// Every call looks up the array's device address (cudaGetSymbolAddress) with
// the caller's device current; the first call on a device may load the
// library's device code, so make it before any stream capture.  All calls on
// a device share the one array, so calls whose work overlaps on the GPU (other
// streams, other host threads) race on it and must be serialised by the
// caller.
#include <cstdint>
#include <cuda_runtime.h>

#include "nc_attn.h"
#include "nc_decode.h"
#include "nc_kernels.h"

namespace {

// Scratch for the partial (max, sum) pairs and unnormalised outputs of every
// split, and the balanced split's row offsets.  Shared by all calls on a
// device; no part of it needs to start at zero, because the combine pass reads
// only what the split pass of the same call wrote.
static __device__ __align__(256) unsigned char g_decode_scratch[NC_DECODE_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device, looked up on every call (host code
// may not pass the symbol itself to a kernel: in host code it names a host-side stand-in, not
// device memory).  No per-device cache, so concurrent first calls need no synchronisation and a
// device reset leaves nothing stale behind.
void* scratch_address() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    return p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// The size limits nc_attn_decode applies (index ranges of its kernels).
bool sizes_supported(int N, int Tmax, int H, int D) {
    return (int64_t)N * H < (int64_t(1) << 31) && (int64_t)Tmax * H * D < (int64_t(1) << 40);
}

}  // namespace

extern "C" {

size_t nc_attn_decode_noalloc_scratch_bytes(int N, int Tmax, int H, int D, int window) {
    if (N <= 0 || Tmax <= 0 || H <= 0 || (D != 64 && D != 128) || (window < 1 && window != NC_WINDOW_FULL)) return 0;
    if (!sizes_supported(N, Tmax, H, D)) return 0;
    return nc::decode_layout(N, Tmax, H, D, window).bytes;
}

nc_status nc_attn_decode_noalloc(const void* q, const void* kcache, const void* vcache, const int* cache_lens,
                                 void* o, float* lse, int N, int Tmax, int H, int D, int window, float scale,
                                 cudaStream_t stream) {
    if (N <= 0 || Tmax <= 0 || H <= 0 || D <= 0) return NC_ERR_INVALID;
    if ((window < 1 && window != NC_WINDOW_FULL) || !(scale > 0.f) || scale > 3.4e38f) return NC_ERR_INVALID;
    if (D != 64 && D != 128) return NC_ERR_UNSUPPORTED;
    if (!sizes_supported(N, Tmax, H, D)) return NC_ERR_UNSUPPORTED;
    if (!q || !kcache || !vcache || !cache_lens || !o) return NC_ERR_INVALID;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o)) return NC_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0) return NC_ERR_INVALID;
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return NC_ERR_INVALID;
    // the same byte-range checks as nc_attn_decode: no output may overlap an input or the other output
    const size_t nq = (size_t)N * H * D * 2, nc_ = (size_t)N * Tmax * H * D * 2, nl = (size_t)N * H * 4;
    const void* ins[4] = {q, kcache, vcache, cache_lens};
    const size_t in_n[4] = {nq, nc_, nc_, (size_t)N * 4};
    for (int i = 0; i < 4; ++i)
        if (overlap(ins[i], in_n[i], o, nq) || (lse != nullptr && overlap(ins[i], in_n[i], lse, nl)))
            return NC_ERR_INVALID;
    if (lse != nullptr && overlap(o, nq, lse, nl)) return NC_ERR_INVALID;
    const size_t need = nc_attn_decode_noalloc_scratch_bytes(N, Tmax, H, D, window);
    if (need > (size_t)NC_DECODE_NOALLOC_SCRATCH_BYTES) return NC_ERR_WORKSPACE;
    unsigned char* scratch = static_cast<unsigned char*>(scratch_address());
    int* err = nc::device_error_word();
    if (scratch == nullptr || err == nullptr) return NC_ERR_CUDA;
    const cudaError_t e = nc::launch_decode(q, kcache, vcache, cache_lens, o, lse, N, Tmax, H, D, window, scale,
                                            scratch, err, stream);
    return e == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

}  // extern "C"
