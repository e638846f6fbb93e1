// Internal launch interface of the decode kernels (not part of the C ABI).
#pragma once
#include <cuda_runtime_api.h>

namespace nc {

// Cache rows per split-K chunk for head dimension D.
int decode_chunk_rows(int D);
// Upper bound on the splits of one sequence (independent of the window).
int decode_max_splits(int Tmax, int D);

// Partials: part_ml [N][splits][H][2] (running max in log2 units, sum) and
// part_o [N][splits][H][D] (unnormalised output), fp32.
cudaError_t launch_decode(const void* q, const void* kcache, const void* vcache, const int* lens, void* o,
                          float* lse, int N, int Tmax, int H, int D, int window, float scale, float* part_ml,
                          float* part_o, int* err, cudaStream_t stream);

}  // namespace nc
