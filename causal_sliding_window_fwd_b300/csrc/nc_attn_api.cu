// C ABI of the attention library: argument validation, workspace sizing,
// dispatch to the kernels and the sticky device error word.  The operation
// and its sources are documented in include/nc_attn.h.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "nc_attn.h"
#include "nc_decode.h"
#include "nc_kernels.h"

namespace {

__device__ int g_nc_error_word;

// Device address of the error word on the current device.  Looked up on every call (a cheap
// runtime query) instead of being cached per device, so concurrent first calls from several host
// threads need no synchronisation and a device reset leaves nothing stale behind.
int* error_word() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_nc_error_word) != cudaSuccess) return nullptr;
    return static_cast<int*>(p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool window_ok(int window) { return window >= 1 || window == NC_WINDOW_FULL; }

bool scale_ok(float scale) { return std::isfinite(scale) && scale > 0.f; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Checks shared by the forward and backward calls.
nc_status check_shape(int B, int T, int H, int D, int window, float scale) {
    if (B <= 0 || T <= 0 || H <= 0 || D <= 0) return NC_ERR_INVALID;
    if (!window_ok(window) || !scale_ok(scale)) return NC_ERR_INVALID;
    if (D != 64 && D != 128) return NC_ERR_UNSUPPORTED;
    if ((int64_t)B * T * H >= (int64_t(1) << 31)) return NC_ERR_UNSUPPORTED;
    return NC_OK;
}

}  // namespace

extern "C" {

const char* nc_status_string(nc_status s) {
    switch (s) {
        case NC_OK: return "NC_OK";
        case NC_ERR_INVALID: return "NC_ERR_INVALID";
        case NC_ERR_UNSUPPORTED: return "NC_ERR_UNSUPPORTED";
        case NC_ERR_WORKSPACE: return "NC_ERR_WORKSPACE";
        case NC_ERR_CUDA: return "NC_ERR_CUDA";
        case NC_ERR_DEVICE_TIMEOUT: return "NC_ERR_DEVICE_TIMEOUT";
        case NC_ERR_BAD_CACHE_LEN: return "NC_ERR_BAD_CACHE_LEN";
        case NC_ERR_BAD_SEQLENS: return "NC_ERR_BAD_SEQLENS";
    }
    return "NC_ERR_UNKNOWN";
}

nc_status nc_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T, int H, int D,
                      int window, float scale, cudaStream_t stream) {
    nc_status st = check_shape(B, T, H, D, window, scale);
    if (st != NC_OK) return st;
    if (!q || !k || !v || !o || !lse) return NC_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return NC_ERR_INVALID;
    const size_t nb = (size_t)B * T * H * D * 2, nl = (size_t)B * H * T * 4;
    const void* ins[3] = {q, k, v};
    for (const void* in : ins)
        if (overlap(in, nb, o, nb) || overlap(in, nb, lse, nl)) return NC_ERR_INVALID;
    if (overlap(o, nb, lse, nl)) return NC_ERR_INVALID;
    int* err = error_word();
    if (err == nullptr) return NC_ERR_CUDA;
    const cudaError_t e = nc::launch_fwd(q, k, v, o, lse, B, T, H, D, window, scale, err, stream);
    return e == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status nc_attn_fwd_rotary(const void* q, const void* k, const void* v, const float* rope_cos, const float* rope_sin,
                             void* qr, void* kr, void* o, float* lse, int B, int T, int H, int D, int window,
                             float scale, cudaStream_t stream) {
    nc_status st = check_shape(B, T, H, D, window, scale);
    if (st != NC_OK) return st;
    if (!q || !k || !v || !rope_cos || !rope_sin || !qr || !kr || !o || !lse) return NC_ERR_INVALID;
    const void* all[9] = {q, k, v, rope_cos, rope_sin, qr, kr, o, lse};
    for (const void* ptr : all)
        if (!aligned16(ptr)) return NC_ERR_INVALID;
    const size_t nb = (size_t)B * T * H * D * 2, nl = (size_t)B * H * T * 4, nt = (size_t)T * (D / 2) * 4;
    const void* ins[5] = {q, k, v, rope_cos, rope_sin};
    const size_t in_n[5] = {nb, nb, nb, nt, nt};
    const void* outs[4] = {qr, kr, o, lse};
    const size_t out_n[4] = {nb, nb, nb, nl};
    for (int a = 0; a < 4; ++a) {
        for (int i = 0; i < 5; ++i)
            if (overlap(ins[i], in_n[i], outs[a], out_n[a])) return NC_ERR_INVALID;
        for (int b = a + 1; b < 4; ++b)
            if (overlap(outs[a], out_n[a], outs[b], out_n[b])) return NC_ERR_INVALID;
    }
    int* err = error_word();
    if (err == nullptr) return NC_ERR_CUDA;
    cudaError_t e = nc::launch_rotary(q, qr, k, kr, rope_cos, rope_sin, B, T, H, D, false, stream);
    if (e != cudaSuccess) return NC_ERR_CUDA;
    e = nc::launch_fwd(qr, kr, v, o, lse, B, T, H, D, window, scale, err, stream);
    return e == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status nc_rotary(const void* x, const float* rope_cos, const float* rope_sin, void* y, int B, int T, int H,
                    int D, int inverse, cudaStream_t stream) {
    if (B < 1 || T < 1 || H < 1) return NC_ERR_INVALID;
    if (D != 64 && D != 128) return NC_ERR_UNSUPPORTED;
    if ((int64_t)B * T * H >= (int64_t(1) << 31)) return NC_ERR_UNSUPPORTED;
    if (!x || !rope_cos || !rope_sin || !y) return NC_ERR_INVALID;
    if (!aligned16(x) || !aligned16(rope_cos) || !aligned16(rope_sin) || !aligned16(y)) return NC_ERR_INVALID;
    const size_t nb = (size_t)B * T * H * D * 2, nt = (size_t)T * (D / 2) * 4;
    if (x != y && overlap(x, nb, y, nb)) return NC_ERR_INVALID;
    if (overlap(rope_cos, nt, y, nb) || overlap(rope_sin, nt, y, nb)) return NC_ERR_INVALID;
    const cudaError_t e = nc::launch_rotary(x, y, nullptr, nullptr, rope_cos, rope_sin, B, T, H, D, inverse != 0, stream);
    return e == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status nc_attn_fwd_varlen(const void* q, const void* k, const void* v, const int* cu_seqlens, void* o, float* lse,
                             int n_docs, int total, int max_seqlen, int H, int D, int window, float scale,
                             cudaStream_t stream) {
    nc_status st = check_shape(1, total, H, D, window, scale);
    if (st != NC_OK) return st;
    if (n_docs <= 0 || max_seqlen <= 0 || max_seqlen > total) return NC_ERR_INVALID;
    if ((int64_t)n_docs * H >= (int64_t(1) << 31)) return NC_ERR_UNSUPPORTED;
    if (!q || !k || !v || !cu_seqlens || !o || !lse) return NC_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return NC_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return NC_ERR_INVALID;
    const size_t nb = (size_t)total * H * D * 2, nl = (size_t)H * total * 4, nc_ = (size_t)(n_docs + 1) * 4;
    const void* ins[4] = {q, k, v, cu_seqlens};
    const size_t in_n[4] = {nb, nb, nb, nc_};
    for (int i = 0; i < 4; ++i)
        if (overlap(ins[i], in_n[i], o, nb) || overlap(ins[i], in_n[i], lse, nl)) return NC_ERR_INVALID;
    if (overlap(o, nb, lse, nl)) return NC_ERR_INVALID;
    int* err = error_word();
    if (err == nullptr) return NC_ERR_CUDA;
    const cudaError_t e = nc::launch_fwd_varlen(q, k, v, cu_seqlens, n_docs, max_seqlen, o, lse, total, H, D, window,
                                                scale, err, stream);
    return e == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

static nc_status attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                 const float* lse, const int* cu_seqlens, void* dq, void* dk, void* dv, int n_docs,
                                 int total, int max_seqlen, int H, int D, int window, float scale, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream, bool deterministic) {
    nc_status st = check_shape(1, total, H, D, window, scale);
    if (st != NC_OK) return st;
    if (n_docs <= 0 || max_seqlen <= 0 || max_seqlen > total) return NC_ERR_INVALID;
    if ((int64_t)n_docs * H >= (int64_t(1) << 31)) return NC_ERR_UNSUPPORTED;
    if (!q || !k || !v || !o || !dO || !lse || !cu_seqlens || !dq || !dk || !dv) return NC_ERR_INVALID;
    const void* all[9] = {q, k, v, o, dO, lse, dq, dk, dv};
    for (const void* p : all)
        if (!aligned16(p)) return NC_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return NC_ERR_INVALID;
    const size_t need = nc_attn_bwd_workspace_bytes(1, total, H, D);
    if (workspace == nullptr || workspace_bytes < need) return NC_ERR_WORKSPACE;
    if (!aligned16(workspace)) return NC_ERR_INVALID;
    const size_t nb = (size_t)total * H * D * 2, nl = (size_t)H * total * 4, nc_ = (size_t)(n_docs + 1) * 4;
    const void* ins[7] = {q, k, v, o, dO, lse, cu_seqlens};
    const size_t in_n[7] = {nb, nb, nb, nb, nb, nl, nc_};
    void* outs[4] = {dq, dk, dv, workspace};
    const size_t out_n[4] = {nb, nb, nb, need};
    for (int a = 0; a < 4; ++a) {
        for (int i = 0; i < 7; ++i)
            if (overlap(ins[i], in_n[i], outs[a], out_n[a])) return NC_ERR_INVALID;
        for (int b = a + 1; b < 4; ++b)
            if (overlap(outs[a], out_n[a], outs[b], out_n[b])) return NC_ERR_INVALID;
    }
    int* err = error_word();
    if (err == nullptr) return NC_ERR_CUDA;
    char* ws = static_cast<char*>(workspace);
    float* dq_acc = reinterpret_cast<float*>(ws);
    ws += round_up((size_t)total * H * D * 4, 256);
    float* delta = reinterpret_cast<float*>(ws);
    ws += round_up((size_t)H * total * 4, 256);
    int* work = reinterpret_cast<int*>(ws);
    const cudaError_t e = nc::launch_bwd_varlen(q, k, v, o, dO, lse, cu_seqlens, n_docs, max_seqlen, dq, dk, dv,
                                                total, H, D, window, scale, dq_acc, delta, work, err, stream,
                                                deterministic);
    return e == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status nc_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                             const float* lse, const int* cu_seqlens, void* dq, void* dk, void* dv, int n_docs,
                             int total, int max_seqlen, int H, int D, int window, float scale, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
    return attn_bwd_varlen(q, k, v, o, dO, lse, cu_seqlens, dq, dk, dv, n_docs, total, max_seqlen, H, D, window, scale,
                           workspace, workspace_bytes, stream, false);
}

nc_status nc_attn_bwd_varlen_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                           const float* lse, const int* cu_seqlens, void* dq, void* dk, void* dv,
                                           int n_docs, int total, int max_seqlen, int H, int D, int window,
                                           float scale, void* workspace, size_t workspace_bytes,
                                           cudaStream_t stream) {
    return attn_bwd_varlen(q, k, v, o, dO, lse, cu_seqlens, dq, dk, dv, n_docs, total, max_seqlen, H, D, window, scale,
                           workspace, workspace_bytes, stream, true);
}

nc_status nc_attn_prefill(const void* q, const void* kcache, const void* vcache, const int* cache_lens, void* o,
                          float* lse, int N, int Tq, int Tmax, int H, int D, int window, float scale,
                          cudaStream_t stream) {
    nc_status st = check_shape(N, Tmax, H, D, window, scale);
    if (st != NC_OK) return st;
    if (Tq <= 0 || Tq > Tmax) return NC_ERR_INVALID;
    if (!q || !kcache || !vcache || !cache_lens || !o || !lse) return NC_ERR_INVALID;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) || !aligned16(lse))
        return NC_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0) return NC_ERR_INVALID;
    const size_t nq = (size_t)N * Tq * H * D * 2, nc_ = (size_t)N * Tmax * H * D * 2, nl = (size_t)N * H * Tq * 4;
    const void* ins[4] = {q, kcache, vcache, cache_lens};
    const size_t in_n[4] = {nq, nc_, nc_, (size_t)N * 4};
    for (int i = 0; i < 4; ++i)
        if (overlap(ins[i], in_n[i], o, nq) || overlap(ins[i], in_n[i], lse, nl)) return NC_ERR_INVALID;
    if (overlap(o, nq, lse, nl)) return NC_ERR_INVALID;
    int* err = error_word();
    if (err == nullptr) return NC_ERR_CUDA;
    const cudaError_t e =
        nc::launch_prefill(q, kcache, vcache, cache_lens, o, lse, N, Tq, Tmax, H, D, window, scale, err, stream);
    return e == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status nc_kv_append(const void* k_new, const void* v_new, void* kcache, void* vcache, const int* cache_lens,
                       int N, int Tq, int Tmax, int H, int D, cudaStream_t stream) {
    nc_status st = check_shape(N, Tmax, H, D, NC_WINDOW_FULL, 1.f);
    if (st != NC_OK) return st;
    if (Tq <= 0 || Tq > Tmax) return NC_ERR_INVALID;
    if (!k_new || !v_new || !kcache || !vcache || !cache_lens) return NC_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kcache) || !aligned16(vcache)) return NC_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0) return NC_ERR_INVALID;
    const size_t nn = (size_t)N * Tq * H * D * 2, nc_ = (size_t)N * Tmax * H * D * 2;
    // the caches are written: neither may overlap an input or the other cache
    const void* ins[3] = {k_new, v_new, cache_lens};
    const size_t in_n[3] = {nn, nn, (size_t)N * 4};
    for (int i = 0; i < 3; ++i)
        if (overlap(ins[i], in_n[i], kcache, nc_) || overlap(ins[i], in_n[i], vcache, nc_)) return NC_ERR_INVALID;
    if (overlap(kcache, nc_, vcache, nc_)) return NC_ERR_INVALID;
    int* err = error_word();
    if (err == nullptr) return NC_ERR_CUDA;
    const cudaError_t e = nc::launch_kv_append(k_new, v_new, kcache, vcache, cache_lens, N, Tq, Tmax, H, D, err, stream);
    return e == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

size_t nc_attn_bwd_workspace_bytes(int B, int T, int H, int D) {
    if (B <= 0 || T <= 0 || H <= 0 || D <= 0) return 0;
    return round_up((size_t)B * T * H * D * 4, 256) + round_up((size_t)B * H * T * 4, 256) + 256;
}

static nc_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                          const float* lse, void* dq, void* dk, void* dv, int B, int T, int H, int D, int window,
                          float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                          bool deterministic) {
    nc_status st = check_shape(B, T, H, D, window, scale);
    if (st != NC_OK) return st;
    if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return NC_ERR_INVALID;
    const void* all[9] = {q, k, v, o, dO, lse, dq, dk, dv};
    for (const void* p : all)
        if (!aligned16(p)) return NC_ERR_INVALID;
    const size_t need = nc_attn_bwd_workspace_bytes(B, T, H, D);
    if (workspace == nullptr || workspace_bytes < need) return NC_ERR_WORKSPACE;
    if (!aligned16(workspace)) return NC_ERR_INVALID;
    const size_t nb = (size_t)B * T * H * D * 2, nl = (size_t)B * H * T * 4;
    const void* ins[6] = {q, k, v, o, dO, lse};
    const size_t in_n[6] = {nb, nb, nb, nb, nb, nl};
    void* outs[4] = {dq, dk, dv, workspace};
    const size_t out_n[4] = {nb, nb, nb, need};
    for (int a = 0; a < 4; ++a) {
        for (int i = 0; i < 6; ++i)
            if (overlap(ins[i], in_n[i], outs[a], out_n[a])) return NC_ERR_INVALID;
        for (int b = a + 1; b < 4; ++b)
            if (overlap(outs[a], out_n[a], outs[b], out_n[b])) return NC_ERR_INVALID;
    }
    int* err = error_word();
    if (err == nullptr) return NC_ERR_CUDA;
    char* ws = static_cast<char*>(workspace);
    float* dq_acc = reinterpret_cast<float*>(ws);
    ws += round_up((size_t)B * T * H * D * 4, 256);
    float* delta = reinterpret_cast<float*>(ws);
    ws += round_up((size_t)B * H * T * 4, 256);
    int* work = reinterpret_cast<int*>(ws);
    const cudaError_t e =
        deterministic ? nc::launch_bwd_deterministic(q, k, v, o, dO, lse, dq, dk, dv, B, T, H, D, window, scale, dq_acc,
                                                     delta, work, err, stream)
                      : nc::launch_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, T, H, D, window, scale, dq_acc, delta,
                                       work, err, stream);
    return e == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status nc_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                      void* dq, void* dk, void* dv, int B, int T, int H, int D, int window, float scale,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, T, H, D, window, scale, workspace, workspace_bytes, stream,
                    false);
}

nc_status nc_attn_bwd_rotary(const void* qr, const void* kr, const void* v, const float* rope_cos,
                             const float* rope_sin, const void* o, const void* dO, const float* lse, void* dq, void* dk,
                             void* dv, int B, int T, int H, int D, int window, float scale, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
    nc_status st = check_shape(B, T, H, D, window, scale);
    if (st != NC_OK) return st;
    if (!qr || !kr || !v || !rope_cos || !rope_sin || !o || !dO || !lse || !dq || !dk || !dv) return NC_ERR_INVALID;
    const void* all[11] = {qr, kr, v, rope_cos, rope_sin, o, dO, lse, dq, dk, dv};
    for (const void* p : all)
        if (!aligned16(p)) return NC_ERR_INVALID;
    const size_t need = nc_attn_bwd_workspace_bytes(B, T, H, D);
    if (workspace == nullptr || workspace_bytes < need) return NC_ERR_WORKSPACE;
    if (!aligned16(workspace)) return NC_ERR_INVALID;
    const size_t nb = (size_t)B * T * H * D * 2, nl = (size_t)B * H * T * 4, nt = (size_t)T * (D / 2) * 4;
    const void* ins[8] = {qr, kr, v, rope_cos, rope_sin, o, dO, lse};
    const size_t in_n[8] = {nb, nb, nb, nt, nt, nb, nb, nl};
    void* outs[4] = {dq, dk, dv, workspace};
    const size_t out_n[4] = {nb, nb, nb, need};
    for (int a = 0; a < 4; ++a) {
        for (int i = 0; i < 8; ++i)
            if (overlap(ins[i], in_n[i], outs[a], out_n[a])) return NC_ERR_INVALID;
        for (int b = a + 1; b < 4; ++b)
            if (overlap(outs[a], out_n[a], outs[b], out_n[b])) return NC_ERR_INVALID;
    }
    int* err = error_word();
    if (err == nullptr) return NC_ERR_CUDA;
    char* ws = static_cast<char*>(workspace);
    float* dq_acc = reinterpret_cast<float*>(ws);
    ws += round_up((size_t)B * T * H * D * 4, 256);
    float* delta = reinterpret_cast<float*>(ws);
    ws += round_up((size_t)B * H * T * 4, 256);
    int* work = reinterpret_cast<int*>(ws);
    const cudaError_t e = nc::launch_bwd_rotary(qr, kr, v, rope_cos, rope_sin, o, dO, lse, dq, dk, dv, B, T, H, D,
                                                window, scale, dq_acc, delta, work, err, stream);
    return e == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

nc_status nc_attn_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int T, int H, int D,
                                    int window, float scale, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
    return attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, T, H, D, window, scale, workspace, workspace_bytes, stream,
                    true);
}

size_t nc_attn_decode_workspace_bytes(int N, int Tmax, int H, int D) {
    if (N <= 0 || Tmax <= 0 || H <= 0 || (D != 64 && D != 128)) return 0;
    return nc::decode_layout(N, Tmax, H, D, NC_WINDOW_FULL).bytes;  // the largest over windows
}

nc_status nc_attn_decode(const void* q, const void* kcache, const void* vcache, const int* cache_lens, void* o,
                         float* lse, int N, int Tmax, int H, int D, int window, float scale, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
    if (N <= 0 || Tmax <= 0 || H <= 0 || D <= 0) return NC_ERR_INVALID;
    if (!window_ok(window) || !scale_ok(scale)) return NC_ERR_INVALID;
    if (D != 64 && D != 128) return NC_ERR_UNSUPPORTED;
    if ((int64_t)N * H >= (int64_t(1) << 31) || (int64_t)Tmax * H * D >= (int64_t(1) << 40)) return NC_ERR_UNSUPPORTED;
    if (!q || !kcache || !vcache || !cache_lens || !o) return NC_ERR_INVALID;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o)) return NC_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0) return NC_ERR_INVALID;
    if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return NC_ERR_INVALID;
    const size_t need = nc_attn_decode_workspace_bytes(N, Tmax, H, D);
    if (workspace == nullptr || workspace_bytes < need) return NC_ERR_WORKSPACE;
    if (!aligned16(workspace)) return NC_ERR_INVALID;
    const size_t nq = (size_t)N * H * D * 2, nc_ = (size_t)N * Tmax * H * D * 2, nl = (size_t)N * H * 4;
    const void* ins[4] = {q, kcache, vcache, cache_lens};
    const size_t in_n[4] = {nq, nc_, nc_, (size_t)N * 4};
    void* outs[3] = {o, lse, workspace};
    const size_t out_n[3] = {nq, lse ? nl : 0, need};
    for (int a = 0; a < 3; ++a) {
        if (outs[a] == nullptr) continue;
        for (int i = 0; i < 4; ++i)
            if (overlap(ins[i], in_n[i], outs[a], out_n[a])) return NC_ERR_INVALID;
        for (int b = a + 1; b < 3; ++b)
            if (outs[b] != nullptr && overlap(outs[a], out_n[a], outs[b], out_n[b])) return NC_ERR_INVALID;
    }
    int* err = error_word();
    if (err == nullptr) return NC_ERR_CUDA;
    const cudaError_t e = nc::launch_decode(q, kcache, vcache, cache_lens, o, lse, N, Tmax, H, D, window, scale,
                                            workspace, err, stream);
    return e == cudaSuccess ? NC_OK : NC_ERR_CUDA;
}

unsigned long long nc_launch_count(void) { return nc::launch_count(); }

nc_status nc_get_device_error(int* code, cudaStream_t stream) {
    if (code == nullptr) return NC_ERR_INVALID;
    *code = NC_OK;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return NC_ERR_CUDA;
    int* err = error_word();
    if (err == nullptr) return NC_ERR_CUDA;
    int value = 0;
    if (cudaMemcpy(&value, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return NC_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return NC_ERR_CUDA;
    *code = value;
    return NC_OK;
}

}  // extern "C"

namespace nc {
namespace {
std::atomic<unsigned long long> g_launches{0};
}
int* device_error_word() { return error_word(); }
cudaError_t ensure_smem_attr(const void* kern, int bytes, std::atomic<bool>* done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kAttrDevices && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < kAttrDevices) done[dev].store(true, std::memory_order_release);
    return e;
}
cudaError_t multiprocessor_count(int* n) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
}
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
unsigned long long launch_count() { return g_launches.load(std::memory_order_relaxed); }
}  // namespace nc
