// Internal launch interface of the decode kernels (not part of the C ABI).
#pragma once
#include <cstddef>
#include <cuda_runtime_api.h>

namespace nc {

// Upper bound on the CTAs of the balanced split (and so on its partial slots beyond N).
constexpr int kDecodeMaxGrid = 1024;

// Cache rows per split-K chunk for head dimension D (chunked path).
int decode_chunk_rows(int D);
// Whether a decode of N sequences over a cache of Tmax rows takes the balanced split (few sequences:
// the visible rows of all of them cut into one equal range per CTA) rather than fixed chunks.
bool decode_balanced(int N, int Tmax);

// Workspace layout of one decode call, in bytes from the workspace's start (each part 256-aligned):
// partial (running max in log2 units, sum) pairs fp32 [slots][H][2] at off_ml, unnormalised partial
// outputs fp32 [slots][H][D] at off_o, and (balanced split) the sequences' visible-row offsets
// int32 [N + 1] and the rows per CTA at off_meta.  slots = N + kDecodeMaxGrid (balanced) or
// N * ceil(min(window, Tmax) / chunk) (chunked); bytes is the total.  The full window gives the
// largest layout.
struct DecodeLayout {
    size_t off_ml, off_o, off_meta, bytes;
};
DecodeLayout decode_layout(int N, int Tmax, int H, int D, int window);

cudaError_t launch_decode(const void* q, const void* kcache, const void* vcache, const int* lens, void* o,
                          float* lse, int N, int Tmax, int H, int D, int window, float scale, void* workspace,
                          int* err, cudaStream_t stream);

}  // namespace nc
