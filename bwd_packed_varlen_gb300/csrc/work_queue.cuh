// Dynamic work distribution inside a persistent block.
//
// The producer warp's lane 0 takes work-item indices from a per-kernel global
// counter (zeroed by the scheduler kernel at the start of every call) and hands
// them to the block's other roles through a two-slot ring in shared memory. Which
// block computes an item therefore varies from call to call, but each item is
// computed entirely by one block with the same arithmetic, so results do not.
#pragma once

#include <stdint.h>

#include "sm103_ptx.cuh"

namespace teattn {

struct WorkRing {
  int item[2];
  int aux[2];  // optional per-item value the producer hands over with the item
  uint64_t full[2];
  uint64_t empty[2];
};

// One thread, before the block-wide barrier that publishes barrier inits.
__device__ __forceinline__ void ring_init(WorkRing& r, uint32_t consumers) {
  for (int i = 0; i < 2; ++i) {
    mbar_init(&r.full[i], 1);
    mbar_init(&r.empty[i], consumers);
  }
}

// Producer (one thread): publish hand-over number k (item < 0 means "no more work").
__device__ __forceinline__ bool ring_put(WorkRing& r, int k, int item, int* status, int aux = 0) {
  const int s = k & 1;
  if (k >= 2 && !mbar_wait(&r.empty[s], ((k >> 1) - 1) & 1, status)) return false;
  *reinterpret_cast<volatile int*>(&r.item[s]) = item;
  *reinterpret_cast<volatile int*>(&r.aux[s]) = aux;
  mbar_arrive(&r.full[s]);
  return true;
}

// Consumer (a single thread): item of hand-over k; *ok = false on a timed-out wait.
__device__ __forceinline__ int ring_get(WorkRing& r, int k, int* status, bool* ok, int* aux = nullptr) {
  const int s = k & 1;
  if (!mbar_wait(&r.full[s], (k >> 1) & 1, status)) {
    *ok = false;
    return -1;
  }
  const int item = *reinterpret_cast<volatile int*>(&r.item[s]);
  if (aux) *aux = *reinterpret_cast<volatile int*>(&r.aux[s]);
  mbar_arrive(&r.empty[s]);
  return item;
}

// Consumer (a whole warp, every lane counted in `consumers`): warp-uniform result.
__device__ __forceinline__ int ring_get_warp(WorkRing& r, int k, int* status, bool* ok) {
  const int s = k & 1;
  if (!__all_sync(0xffffffffu, mbar_wait(&r.full[s], (k >> 1) & 1, status))) {
    *ok = false;
    return -1;
  }
  const int item = *reinterpret_cast<volatile int*>(&r.item[s]);
  mbar_arrive(&r.empty[s]);
  return item;
}

// Consumer (a whole warp, counted once in `consumers`): every lane waits and reads
// the warp-uniform item; lane 0 alone arrives on the slot's empty barrier.
__device__ __forceinline__ int ring_get_warp_once(WorkRing& r, int k, int* status, bool* ok,
                                                  int* aux) {
  const int s = k & 1;
  if (!__all_sync(0xffffffffu, mbar_wait(&r.full[s], (k >> 1) & 1, status))) {
    *ok = false;
    return -1;
  }
  const int item = *reinterpret_cast<volatile int*>(&r.item[s]);
  *aux = *reinterpret_cast<volatile int*>(&r.aux[s]);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&r.empty[s]);
  __syncwarp();
  return item;
}

// Producer: index of the block's next work item (the first is blockIdx.x).
__device__ __forceinline__ int next_item(int* counter) {
  return static_cast<int>(gridDim.x) + atomicAdd(counter, 1);
}

}  // namespace teattn
