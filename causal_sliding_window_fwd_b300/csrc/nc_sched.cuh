// Assignment of work items to persistent CTAs (one CTA per SM).
//
// Static: the kernel numbers its items heaviest first.  Round r hands out items r*G .. r*G+G-1
// (G = gridDim.x); CTA c takes slot c on even rounds and slot G-1-c on odd ones.  With items
// sorted by decreasing cost this zigzag evens out the total work per CTA far better than plain
// round-robin, and every role of a CTA computes its next item on its own.
//
// Dynamic: the producer warp of a CTA takes the next item index from a global counter and
// publishes it in a small ring in shared memory; every other warp that needs the item reads it
// from the ring.  Each ring slot has a "full" mbarrier (one arrival: the producer) and an
// "empty" mbarrier (one arrival per reading warp).  All waits are bounded.
#pragma once

#include "nc_ptx.cuh"

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

constexpr int kItemSlots = 2;

// Producer warp (converged): take the next item index from `*work` and publish it in slot
// k % kItemSlots; -1 once all `n_items` are taken.  Returns what it published, or -2 if the
// wait for the slot ran out.
__device__ __forceinline__ int ring_publish_item(uint64_t* full, uint64_t* empty, int* slots, int k,
                                                 int n_items, int* work) {
    const int slot = k % kItemSlots;
    if (!mbar_wait_warp(&empty[slot], ((k / kItemSlots) & 1) ^ 1)) return -2;
    int w = 0;
    if (lane_id() == 0) {
        w = atomicAdd(work, 1);
        if (w >= n_items) w = -1;
        slots[slot] = w;
        mbar_arrive(&full[slot]);  // release: the index is visible to whoever sees the phase
    }
    return __shfl_sync(0xffffffffu, w, 0);
}

// Any other warp (converged): the index in slot k % kItemSlots, or -2 if the wait ran out.
__device__ __forceinline__ int ring_read_item(uint64_t* full, uint64_t* empty, const int* slots, int k) {
    const int slot = k % kItemSlots;
    if (!mbar_wait_warp(&full[slot], (k / kItemSlots) & 1)) return -2;
    const int w = *reinterpret_cast<const volatile int*>(&slots[slot]);
    __syncwarp();
    if (lane_id() == 0) mbar_arrive(&empty[slot]);
    return w;
}

}  // namespace nc
