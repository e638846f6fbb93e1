// Static assignment of work items to persistent CTAs (one CTA per SM).
//
// The kernels number their items heaviest first.  Round r hands out items r*G .. r*G+G-1
// (G = gridDim.x); CTA c takes slot c on even rounds and slot G-1-c on odd ones.  With items
// sorted by decreasing cost this zigzag evens out the total work per CTA far better than plain
// round-robin, and, unlike a work-stealing counter, every role of a CTA can compute its next
// item on its own without exchanging it through shared memory.
#pragma once

namespace nc {

// Global index of this CTA's ii-th item.
__device__ __forceinline__ int sched_item_index(int ii) {
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    return ii * G + ((ii & 1) ? G - 1 - c : c);
}

// Number of items this CTA runs: every full round, plus the last partial round if its slot is in it.
__device__ __forceinline__ int sched_items_of_cta(int n_items) {
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    const int full = n_items / G, rem = n_items % G;
    const int slot = (full & 1) ? G - 1 - c : c;
    return full + (slot < rem ? 1 : 0);
}

}  // namespace nc
