// Internal launch interface of the forward / backward attention kernels.
#pragma once
#include <atomic>
#include <cuda_runtime_api.h>

namespace nc {

// Host-side count of kernels enqueued by the library (see nc_launch_count).
void count_launches(unsigned n);
unsigned long long launch_count();

// Device address of the library's sticky error word on the current device (nullptr on failure).
// Looked up on every call: the library keeps no per-device host-side cache.
int* device_error_word();

// Number of SMs of the current device.
cudaError_t multiprocessor_count(int* n);

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device, once per device and
// kernel (`done` is that kernel's per-device flag array of kAttrDevices entries, zero at load).  Host
// threads racing on a first call may both set it, which is harmless; the flag is atomic.  A stale flag
// (after a device reset) can only make the launch fail with an error, never touch memory.
constexpr int kAttrDevices = 64;
cudaError_t ensure_smem_attr(const void* kern, int bytes, std::atomic<bool>* done);

// Forward: o [B,T,H,D] bf16, lse [B,H,T] fp32.  `err` is the device error word.
cudaError_t launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T, int H, int D,
                       int window, float scale, int* err, cudaStream_t st);

// Rotary turn of x0 into y0 and, if x1 is not null, of x1 into y1 in the same launch: [B,T,H,D] bf16,
// tables rcos, rsin fp32 [T, D/2]; `inverse` applies the transpose.  y may equal x (in place).
cudaError_t launch_rotary(const void* x0, void* y0, const void* x1, void* y1, const float* rcos, const float* rsin,
                          int B, int T, int H, int D, bool inverse, cudaStream_t st);

// Document-masked forward over packed rows: q/k/v/o [total,H,D] bf16, lse [H,total] fp32, cu device int32 [n_docs+1].
cudaError_t launch_fwd_varlen(const void* q, const void* k, const void* v, const int* cu, int n_docs, int max_len,
                              void* o, float* lse, int total, int H, int D, int window, float scale, int* err,
                              cudaStream_t st);

// Document-masked backward over packed rows; workspace as for launch_bwd with B = 1, T = total.
// deterministic: dK and dV from the main kernel without its dQ product, dq from the query-stationary pass.
cudaError_t launch_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, const int* cu, int n_docs, int max_len, void* dq, void* dk, void* dv,
                              int total, int H, int D, int window, float scale, float* dq_acc, float* delta, int* work,
                              int* err, cudaStream_t st, bool deterministic = false);

// Prefill over a KV cache: q/o [N,Tq,H,D] bf16, lse [N,H,Tq] fp32, caches [N,Tmax,H,D], lens device int32 [N].
cudaError_t launch_prefill(const void* q, const void* kcache, const void* vcache, const int* lens, void* o,
                           float* lse, int N, int Tq, int Tmax, int H, int D, int window, float scale, int* err,
                           cudaStream_t st);

// KV-cache append: kcache/vcache [N,Tmax,H,D] rows L_n - Tq .. L_n - 1 from k_new/v_new [N,Tq,H,D] bf16,
// lens device int32 [N] (each counting the new rows).
cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* kcache, void* vcache, const int* lens, int N,
                             int Tq, int Tmax, int H, int D, int* err, cudaStream_t st);

// Backward: dq_acc fp32 [B,T,H,D], delta fp32 [B,H,T] and the work-item counter are workspace.
cudaError_t launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                       void* dq, void* dk, void* dv, int B, int T, int H, int D, int window, float scale,
                       float* dq_acc, float* delta, int* work, int* err, cudaStream_t st);

// Backward of attention over turned rows qr, kr: dq and dk with respect to the unturned q and k (both turned
// back in the conversion pass, dk in place).  Workspace as for launch_bwd.
cudaError_t launch_bwd_rotary(const void* qr, const void* kr, const void* v, const float* rcos, const float* rsin,
                              const void* o, const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                              int T, int H, int D, int window, float scale, float* dq_acc, float* delta, int* work,
                              int* err, cudaStream_t st);

// Deterministic backward: dK and dV from the main kernel without its dQ product, then dq from the
// query-stationary pass (launch_bwd_dq).  Workspace as for launch_bwd (dq_acc is not touched).
cudaError_t launch_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                     const float* lse, void* dq, void* dk, void* dv, int B, int T, int H, int D,
                                     int window, float scale, float* dq_acc, float* delta, int* work, int* err,
                                     cudaStream_t st);

// Query-stationary dQ pass: dq [B,T,H,D] bf16 from q, k, v, dO, lse and delta [B,H,T] fp32.
// `work` is a work-item counter that must be zero when the kernel starts.  cu != nullptr: packed documents
// (B = 1, T = total, cu device int32 [n_docs+1], max_len the longest document).
cudaError_t launch_bwd_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                          const float* delta, void* dq, int B, int T, int H, int D, int window, float scale, int* work,
                          int* err, cudaStream_t st, const int* cu = nullptr, int n_docs = 0, int max_len = 0);

}  // namespace nc
