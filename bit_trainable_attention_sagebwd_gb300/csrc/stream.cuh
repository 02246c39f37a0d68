// Persistent streaming over a list of work items for the HBM-bound passes.
//
// Each CTA claims items from a global ticket (one atomicAdd per item), so items are
// claimed in increasing order across the grid, and keeps the inputs of its next NS-1
// claimed items in flight in a ring of shared-memory stages: while its threads work on
// one item, the bulk copies of the following ones are under way.  A few CTAs per SM
// then hold well over 100 KB of reads in flight, and compute overlaps the copies.
//
// Items are independent: no CTA waits on another, and no co-residency of the grid is
// assumed.
#pragma once

#include <atomic>

#include "ptx.cuh"

namespace sage {

// Wait for an mbarrier phase without looking at any abort flag (draining copies in flight).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t budget_ns = SAGE_WAIT_NS) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > budget_ns) return false;
  return true;
}

template <int NS>
struct StreamCtl {
  static_assert(NS >= 2, "the ring needs two stages or more");
  uint64_t full[NS];
  int item[NS];  // item held by each stage (>= nitems: none)
  int abort;
};

// Runs body(item, stage) on every item this CTA claims, with all threads of the CTA.
// issue(item, stage, bar) runs on thread 0: it starts the copies of the item's inputs
// into `stage` and arms `bar` with their byte count (mbar_arrive_expect_tx, also when the
// count is 0).  A stage is reused only after every thread has left the body of its item.
// A body that writes a stage with generic stores before it is reused must fence them
// (fence.proxy.async) before returning.  Returns false when a wait ran out, after waiting
// (bounded) for the copies still in flight; the status word is then set.
template <int NS, class Issue, class Body>
__device__ __forceinline__ bool stream_items(StreamCtl<NS>& c, uint8_t* stages, uint32_t stage_bytes, int* ticket,
                                             int nitems, int* status, Issue&& issue, Body&& body) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&c.full[s], 1);
    c.abort = 0;
    fence_mbar_init();
    for (int s = 0; s < NS; ++s) {
      const int it = atomicAdd(ticket, 1);
      c.item[s] = it;
      if (it < nitems) issue(it, stages + (size_t)s * stage_bytes, &c.full[s]);
    }
  }
  __syncthreads();
  int k = 0;
  bool ok = true;
  for (;; ++k) {
    const int s = k % NS;
    const int it = c.item[s];  // written by thread 0 at least one CTA barrier ago
    if (it >= nitems) break;
    // the item that refills this stage is claimed now: the atomic's round trip overlaps
    // the wait and the body instead of delaying the next copy
    int nx = 0;
    if (tid == 0) nx = atomicAdd(ticket, 1);
    const bool got = mbar_wait(&c.full[s], (uint32_t)(k / NS) & 1u, &c.abort);
    if (__syncthreads_or(!got)) {
      ok = false;
      break;
    }
    body(it, stages + (size_t)s * stage_bytes);
    __syncthreads();
    if (tid == 0) {
      c.item[s] = nx;
      if (nx < nitems) issue(nx, stages + (size_t)s * stage_bytes, &c.full[s]);
    }
  }
  if (!ok && tid == 0) {
    // the copies of stages k .. k+NS-1 that were started may still land: wait for them
    // (the item claimed for stage k is dropped; no copy was started for it)
    for (int j = k; j < k + NS; ++j)
      if (c.item[j % NS] < nitems) mbar_wait_drain(&c.full[j % NS], (uint32_t)(j / NS) & 1u);
    atomicExch(status, kDevTimeout);
  }
  return ok;
}

// number of SMs of the current device (looked up once per device)
inline int sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// persistent grid: SMs x resident CTAs per SM, never more CTAs than items
template <class K>
inline int persistent_grid(K kernel, int threads, size_t smem, int nitems) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int g = sm_count() * per_sm;
  return g < nitems ? g : (nitems > 0 ? nitems : 1);
}

}  // namespace sage
