/*
 * nc_attn — exact causal sliding-window softmax attention for NVIDIA B300 (sm_103a).
 *
 * C ABI.  Every entry point takes plain device pointers, sizes and a CUDA
 * stream; none allocates, none synchronises (except nc_get_device_error), and
 * all work is enqueued on `stream`.  The caller owns every buffer, including
 * the workspaces.
 *
 * The operation (what the calls compute):
 *   "nanochat GPT-2 speedrun" post (page 2, repeated on page 5), paragraph on
 *   the biggest improvements: attention runs through FlashAttention-3 kernels
 *   whose `window_size` argument gives per-layer alternating local/global
 *   (sliding-window / full causal) attention.  "nanochat" walkthrough (page 4,
 *   close of the pretraining section; page 1 launch post): inference runs an
 *   Engine with a KV cache and a prefill/decode split.  The pages give no
 *   formula, so the calls compute the textbook definition:
 *
 *     visible(i, j)  <=>  j <= i  and  i - j < W        (W keys including i)
 *     s_ij  = scale * <q_i, k_j>
 *     lse_i = ln sum_{j visible} exp(s_ij)
 *     o_i   = sum_{j visible} exp(s_ij - lse_i) v_j
 *
 *   per batch b and head h independently.  `window` <= 0 is rejected except
 *   NC_WINDOW_FULL (-1); a window >= T is full causal attention.
 *
 * Layout (all contiguous, row-major):
 *   q, k, v, o, dO, dq, dk, dv : bf16 [B, T, H, D]
 *   lse                        : fp32 [B, H, T]   (natural log, of the scaled scores)
 *   decode q, o                : bf16 [N, H, D]
 *   decode kcache, vcache      : bf16 [N, Tmax, H, D]  (padded per sequence)
 *   decode cache_lens          : int32 [N] in device memory
 *   decode lse                 : fp32 [N, H] or NULL
 *
 * Supported sizes: D in {64, 128}; B, T, H, N >= 1; B*H and T small enough
 * that every tensor has fewer than 2^31 rows of D elements.  All pointers
 * must be 16-byte aligned (the kernels move data with TMA and 16-byte
 * vectors).  Outputs must not alias inputs or each other.
 *
 * Threads: every entry point may be called from any host thread, including
 * several threads making their first calls at the same time.  Each call looks
 * up the device addresses of the library's own __device__ variables and the SM
 * count with the caller's device current; the only shared host state is an
 * atomic launch counter and atomic per-device flags recording that a kernel's
 * shared-memory limit has been raised.
 *
 * Errors: host-side argument checks return a status synchronously and launch
 * nothing.  Conditions only the device can see (a decode cache length
 * outside [1, Tmax], a pipeline wait that exceeded its time limit) set a
 * sticky device error word, write NaN into the affected output rows and let
 * the kernel finish; nc_get_device_error() reads and clears that word.
 */
#ifndef NC_ATTN_H_
#define NC_ATTN_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NC_OK = 0,
    NC_ERR_INVALID = 1,        /* null pointer, non-positive size, bad window/scale, misalignment, aliasing */
    NC_ERR_UNSUPPORTED = 2,    /* head dimension other than 64 or 128, sizes beyond the index range */
    NC_ERR_WORKSPACE = 3,      /* workspace pointer null or smaller than the *_workspace_bytes() figure */
    NC_ERR_CUDA = 4,           /* a CUDA runtime call or kernel launch failed */
    NC_ERR_DEVICE_TIMEOUT = 5, /* device: a pipeline wait ran out of time; outputs are not valid */
    NC_ERR_BAD_CACHE_LEN = 6,  /* device: a decode/prefill cache length was out of range; its rows are NaN */
    NC_ERR_BAD_SEQLENS = 7     /* device: document bounds (cu_seqlens) out of order, out of range, or a
                                  document longer than max_seqlen; its rows are not written */
} nc_status;

#define NC_WINDOW_FULL (-1)

/* Human-readable name of a status code (static string). */
const char* nc_status_string(nc_status s);

/*
 * Forward.  o = attention(q, k, v) and lse = per-row log-sum-exp of the
 * scaled scores over the visible keys.
 *   q, k, v : const bf16 [B, T, H, D] device
 *   o       : bf16 [B, T, H, D] device, written
 *   lse     : fp32 [B, H, T] device, written (needed by nc_attn_bwd)
 *   window  : keys visible per query including itself (>= 1), or NC_WINDOW_FULL
 *   scale   : score multiplier, finite and > 0 (usually 1/sqrt(D))
 * Returns NC_OK once the work is enqueued on `stream`.
 */
nc_status nc_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int T, int H, int D, int window, float scale, cudaStream_t stream);

/* Bytes of device workspace nc_attn_bwd needs: an fp32 dQ accumulator
 * [B, T, H, D], the fp32 row term Delta = rowsum(dO * O) [B, H, T] and a
 * work-item counter for the main kernel's scheduler. */
size_t nc_attn_bwd_workspace_bytes(int B, int T, int H, int D);

/*
 * Backward.  Gradients of sum(o * dO) with respect to q, k and v, for the
 * o and lse that nc_attn_fwd produced with the same arguments.
 *   q, k, v, o, dO : const bf16 [B, T, H, D] device
 *   lse            : const fp32 [B, H, T] device
 *   dq, dk, dv     : bf16 [B, T, H, D] device, written
 *   workspace      : device, >= nc_attn_bwd_workspace_bytes(B, T, H, D),
 *                    16-byte aligned; its contents on entry do not matter
 * The dQ accumulation uses fp32 atomics, so dq may differ in the last bits
 * from run to run.
 */
nc_status nc_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                      const float* lse, void* dq, void* dk, void* dv,
                      int B, int T, int H, int D, int window, float scale,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Deterministic backward.  The same gradients, arguments, layout, workspace
 * (nc_attn_bwd_workspace_bytes) and errors as nc_attn_bwd, but dq, dk and dv
 * are bitwise identical from run to run on the same device for the same
 * inputs: dK and dV accumulate in a fixed order in the main kernel, and dq
 * comes from a second pass in which one CTA owns each 128-row query block and
 * sums its key blocks in a fixed order, instead of adding partials with fp32
 * atomics.  The second pass recomputes S = scale q k^T and dP = dO v^T for
 * every visible block pair, so this call does about 7/5 of nc_attn_bwd's
 * tensor-core work.  The fp32 dQ accumulator part of the workspace is unused.
 */
nc_status nc_attn_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                    const float* lse, void* dq, void* dk, void* dv,
                                    int B, int T, int H, int D, int window, float scale,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Bytes of device workspace nc_attn_decode needs for its split-K partial
 * results (fp32 running max, sum and output per split) and, for up to 1024
 * sequences, the per-sequence row offsets of its balanced split.  Its
 * contents on entry do not matter. */
size_t nc_attn_decode_workspace_bytes(int N, int Tmax, int H, int D);

/*
 * Single-token decode over a KV cache (one query per sequence).  The query
 * of sequence n sits at position L = cache_lens[n] - 1, whose key and value
 * are already in the cache; it sees cache rows max(0, L + 1 - window) .. L.
 *   q          : const bf16 [N, H, D] device
 *   kcache     : const bf16 [N, Tmax, H, D] device
 *   vcache     : const bf16 [N, Tmax, H, D] device
 *   cache_lens : const int32 [N] device, each in [1, Tmax]; a value outside
 *                that range sets NC_ERR_BAD_CACHE_LEN on the device and
 *                makes that sequence's o (and lse) rows NaN
 *   o          : bf16 [N, H, D] device, written
 *   lse        : fp32 [N, H] device, written, or NULL
 *   workspace  : device, >= nc_attn_decode_workspace_bytes(N, Tmax, H, D)
 * Cache rows at or beyond a sequence's length, and rows before its window,
 * are never read.
 */
nc_status nc_attn_decode(const void* q, const void* kcache, const void* vcache, const int* cache_lens,
                         void* o, float* lse, int N, int Tmax, int H, int D, int window, float scale,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Document-masked (varlen) forward over packed rows: pretraining packs
 * several documents into a row, and each token attends only to earlier
 * tokens of its own document, inside the window (positions counted from the
 * document's start).  Document d is rows cu_seqlens[d] .. cu_seqlens[d+1]-1.
 *   q, k, v     : const bf16 [total, H, D] device
 *   cu_seqlens  : const int32 [n_docs + 1] device, 0 = cu_seqlens[0] <= ...
 *                 <= cu_seqlens[n_docs] = total, each document at most
 *                 max_seqlen rows; a document whose bounds break this sets
 *                 NC_ERR_BAD_SEQLENS on the device and its rows are not written
 *   o           : bf16 [total, H, D] device, written
 *   lse         : fp32 [H, total] device, written
 * Rows of o and lse that belong to no document (none, if cu_seqlens covers
 * [0, total)) are not written.  With one document this is nc_attn_fwd with
 * B = 1, T = total.
 */
nc_status nc_attn_fwd_varlen(const void* q, const void* k, const void* v, const int* cu_seqlens, void* o,
                             float* lse, int n_docs, int total, int max_seqlen, int H, int D, int window,
                             float scale, cudaStream_t stream);

/*
 * Backward of nc_attn_fwd_varlen, for the o and lse it produced with the same
 * arguments.  Shapes as there (dO, dq, dk, dv [total, H, D] bf16, lse
 * [H, total] fp32); workspace >= nc_attn_bwd_workspace_bytes(1, total, H, D).
 * Rows that belong to no document get dq = 0 and are not written in dk, dv.
 * Bad document bounds set NC_ERR_BAD_SEQLENS as in the forward.
 */
nc_status nc_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                             const float* lse, const int* cu_seqlens, void* dq, void* dk, void* dv, int n_docs,
                             int total, int max_seqlen, int H, int D, int window, float scale, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/*
 * Deterministic form of nc_attn_bwd_varlen: the same gradients, arguments,
 * layouts, workspace and errors, but dq, dk and dv are bitwise identical from
 * run to run (as nc_attn_bwd_deterministic for packed rows: dK and dV from the
 * main kernel, dq from a pass in which one CTA owns each 128-row query block
 * of a document and sums its key blocks in a fixed order).  Rows that belong
 * to no document get dq = 0.
 */
nc_status nc_attn_bwd_varlen_deterministic(const void* q, const void* k, const void* v, const void* o,
                                           const void* dO, const float* lse, const int* cu_seqlens, void* dq,
                                           void* dk, void* dv, int n_docs, int total, int max_seqlen, int H,
                                           int D, int window, float scale, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream);

/*
 * Prefill (append) over a KV cache: Tq new tokens per sequence attend over the
 * cache ("nanochat" walkthrough, page 4: the Engine's prefill/decode split
 * over a KV cache).  The keys and values of the new tokens are already in the
 * cache: cache_lens[n] = L counts them, and new token t is the query at
 * position L - Tq + t; it sees cache rows max(0, L - Tq + t + 1 - window) ..
 * L - Tq + t.  With Tq = 1 this is nc_attn_decode's result.
 *   q          : const bf16 [N, Tq, H, D] device
 *   kcache     : const bf16 [N, Tmax, H, D] device
 *   vcache     : const bf16 [N, Tmax, H, D] device
 *   cache_lens : const int32 [N] device, each in [Tq, Tmax]; a value outside
 *                that range sets NC_ERR_BAD_CACHE_LEN on the device and makes
 *                that sequence's o and lse rows NaN
 *   o          : bf16 [N, Tq, H, D] device, written
 *   lse        : fp32 [N, H, Tq] device, written
 * The cache is read in 128-row blocks; rows from L up to the end of the
 * block that holds row L - 1 (fewer than 128) are loaded and masked out
 * (their value rows are zeroed on chip before use), so they may hold
 * anything, NaN included.  Rows beyond that block are never read.  Blocks
 * start at multiples of 128 or, where the window does not reach back to row
 * 0, at rows congruent to L - Tq modulo 128 (in line with the query tiles;
 * none past L - 1 is then loaded when Tq is a multiple of 128).  Needs no
 * workspace; Tq <= Tmax.
 */
nc_status nc_attn_prefill(const void* q, const void* kcache, const void* vcache, const int* cache_lens,
                          void* o, float* lse, int N, int Tq, int Tmax, int H, int D, int window, float scale,
                          cudaStream_t stream);

/*
 * Append of new tokens' keys and values to the KV cache ("nanochat"
 * walkthrough, page 4: the Engine's KV cache, filled by prefill and extended
 * by every decode step).  cache_lens[n] = L already counts the Tq new tokens,
 * as nc_attn_prefill and nc_attn_decode take it, so new row t is written to
 * cache position L - Tq + t:
 *   kcache[n, L - Tq + t] = k_new[n, t],  vcache[n, L - Tq + t] = v_new[n, t].
 * Run it before nc_attn_prefill (or nc_attn_decode, Tq = 1) with the same
 * lengths.  Other cache rows are not touched.
 *   k_new, v_new : const bf16 [N, Tq, H, D] device, 16-byte aligned
 *   kcache       : bf16 [N, Tmax, H, D] device, written (rows L - Tq .. L - 1)
 *   vcache       : bf16 [N, Tmax, H, D] device, written likewise
 *   cache_lens   : const int32 [N] device, each in [Tq, Tmax]; a value
 *                  outside that range sets NC_ERR_BAD_CACHE_LEN on the device
 *                  and leaves that sequence's rows unwritten
 * NC_ERR_INVALID for null or misaligned pointers, Tq outside [1, Tmax], or
 * caches overlapping each other or an input; NC_ERR_UNSUPPORTED for D other
 * than 64 or 128.  One launch, no workspace.
 */
nc_status nc_kv_append(const void* k_new, const void* v_new, void* kcache, void* vcache, const int* cache_lens,
                       int N, int Tq, int Tmax, int H, int D, cudaStream_t stream);

/*
 * Attention over rotary-embedded q and k ("nanochat" walkthrough, page 4,
 * comment thread: the model is Llama-like; the pages give no formula, and the
 * rotate-half pairing of Llama is the reading taken).  Each query and key row
 * of position t (0 .. T-1) has every pair (x_i, x_{i+D/2}), i < D/2, turned by
 * the angle whose cosine and sine the tables hold at (t, i):
 *   x_i' = x_i c - x_{i+D/2} s,   x_{i+D/2}' = x_i s + x_{i+D/2} c,
 * evaluated in float32 (one product and one fused multiply-add per output)
 * and rounded to bf16.  One launch writes the turned q and k to qr and kr,
 * which the backward takes; then o, lse are those of nc_attn_fwd on (qr, kr,
 * v).  Two launches.
 *   rope_cos, rope_sin : const fp32 [T, D/2] device, 16-byte aligned (row t,
 *                        column i; e.g. cos / sin of t * base^(-2i/D))
 *   qr, kr             : bf16 [B, T, H, D] device, written (the turned q, k)
 * Other arguments, layouts and errors as nc_attn_fwd; no output may overlap
 * an input or another output.
 */
nc_status nc_attn_fwd_rotary(const void* q, const void* k, const void* v, const float* rope_cos,
                             const float* rope_sin, void* qr, void* kr, void* o, float* lse, int B, int T,
                             int H, int D, int window, float scale, cudaStream_t stream);

/*
 * Backward of nc_attn_fwd_rotary.  Takes the turned rows qr, kr that
 * nc_attn_fwd_rotary wrote (not q and k) and the same tables; dq and dk are
 * the gradients with respect to the unturned q and k: the gradients with
 * respect to the turned rows, turned back by the transpose of each row's
 * rotation (dK in the main kernel's epilogue, dQ in the pass that converts
 * its fp32 accumulator), so the backward costs what nc_attn_bwd costs.  dv as
 * nc_attn_bwd.  The workspace is sized by nc_attn_bwd_workspace_bytes.  Other
 * arguments, layouts and errors as nc_attn_bwd.
 */
nc_status nc_attn_bwd_rotary(const void* qr, const void* kr, const void* v, const float* rope_cos,
                             const float* rope_sin, const void* o, const void* dO, const float* lse,
                             void* dq, void* dk, void* dv, int B, int T, int H, int D, int window,
                             float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The rotary turn on its own: y = the turn of x, row t of each sequence by
 * the tables' row t, as nc_attn_fwd_rotary defines it (for example to turn new
 * tokens' keys before they enter a KV cache); with inverse != 0 the transpose
 * (the turn back, which maps gradients with respect to the turned tensor to
 * gradients with respect to x).  For positions that do not start at 0 pass
 * tables offset to the first position.
 *   x                  : const bf16 [B, T, H, D] device, 16-byte aligned
 *   rope_cos, rope_sin : const fp32 [T, D/2] device, 16-byte aligned
 *   y                  : bf16 [B, T, H, D] device, written; either x itself
 *                        (in place) or a range that does not overlap x
 * D is 64 or 128.  Errors: NC_ERR_INVALID for a null or unaligned pointer, a
 * partial overlap, or B, T, H < 1; NC_ERR_UNSUPPORTED for another D or for
 * B * T * H >= 2^31; NC_ERR_CUDA if the launch fails.  One kernel launch,
 * asynchronous.
 */
nc_status nc_rotary(const void* x, const float* rope_cos, const float* rope_sin, void* y, int B, int T,
                    int H, int D, int inverse, cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device error word that
 * the kernels set (NC_OK if nothing went wrong since the last call).
 * Returns NC_ERR_CUDA if the synchronisation itself failed.
 */
nc_status nc_get_device_error(int* code, cudaStream_t stream);

/*
 * Failure-detection self-test (not part of the attention path).  Launches one
 * CTA whose thread waits on an mbarrier that nothing completes, through the
 * bounded wait all of the library's pipelines use, limited to `limit_cycles`
 * SM clock cycles (1 .. 2^31).  The wait runs out, the kernel records
 * NC_ERR_DEVICE_TIMEOUT in the device error word and returns; the context
 * stays usable.  Read the result with nc_get_device_error().
 */
nc_status nc_debug_watchdog_selftest(unsigned long long limit_cycles, cudaStream_t stream);

/*
 * Decode without a caller-provided workspace and without allocating.  The
 * pages describe nothing of the kind: this entry point exists for callers
 * that cannot allocate device memory when they decode (engines whose own
 * allocator owns the device memory, plug-ins handed only their input and
 * output buffers, token loops that cannot pay for the synchronisation that
 * cudaMalloc/cudaFree may imply).
 *
 * Same arguments, layout and results as nc_attn_decode, minus the workspace.
 * The split-K partials go to a fixed scratch array of
 * NC_DECODE_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits.  Calls needing more
 * scratch than that (see nc_attn_decode_noalloc_scratch_bytes) return
 * NC_ERR_WORKSPACE and launch nothing.  The call never allocates.
 *
 * Every call looks up the scratch array's device address with the caller's
 * device current; the first call on a device may load the library's device
 * code, so make it before any stream capture.  All calls on a device share the
 * array (it keeps the last call's contents; nothing in it needs to start at
 * zero), so calls whose GPU work overlaps race on it: the caller must order
 * them, e.g. on one stream.  The outputs may not overlap any input or each
 * other (byte ranges, as for nc_attn_decode).
 */
#define NC_DECODE_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* Scratch bytes nc_attn_decode_noalloc would use for these sizes; 0 for sizes or a window that it
 * rejects (non-positive sizes, D not 64 or 128, a bad window, or N*H >= 2^31 or Tmax*H*D >= 2^40). */
size_t nc_attn_decode_noalloc_scratch_bytes(int N, int Tmax, int H, int D, int window);

nc_status nc_attn_decode_noalloc(const void* q, const void* kcache, const void* vcache, const int* cache_lens,
                                 void* o, float* lse, int N, int Tmax, int H, int D, int window, float scale,
                                 cudaStream_t stream);

/*
 * Number of CUDA kernels this library has enqueued (all devices, all
 * streams) since it was loaded.  Host-side counter, for launch accounting in
 * benchmarks; it does not synchronise and never fails.
 */
unsigned long long nc_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* NC_ATTN_H_ */
