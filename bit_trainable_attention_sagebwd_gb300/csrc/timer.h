// Optional per-kernel timing: when enabled, launches are bracketed by CUDA events
// recorded on the launching stream; totals are read (and cleared) on demand.
#pragma once

#include <cuda_runtime.h>

namespace sage {

bool timer_enabled();
// enabled, and `name` passes the filter (timer_only)
bool timer_enabled_for(const char* name);
void timer_set(bool on);
// record only the launch group `name` (nullptr: every group)
void timer_only(const char* name);
// record the start event of a timed launch group; returns a handle for timer_stop
int timer_start(const char* name, cudaStream_t st);
void timer_stop(int handle, cudaStream_t st);
// synchronize the recorded events of `name`, return their summed milliseconds and
// count, and forget them
int timer_read(const char* name, double* total_ms, int* launches);

struct ScopedTimer {
  int h;
  cudaStream_t st;
  ScopedTimer(const char* name, cudaStream_t s) : h(timer_enabled_for(name) ? timer_start(name, s) : -1), st(s) {}
  ~ScopedTimer() {
    if (h >= 0) timer_stop(h, st);
  }
};

}  // namespace sage
