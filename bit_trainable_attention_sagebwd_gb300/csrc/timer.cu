// Per-kernel event timing (host code); see timer.h.
#include <mutex>
#include <string>
#include <vector>

#include "timer.h"

namespace sage {

namespace {

struct Rec {
  std::string name;
  cudaEvent_t a, b;
  bool done;
};

std::mutex g_mu;
bool g_on = false;
std::string g_only;  // empty: every group
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

bool timer_enabled() {
  std::lock_guard<std::mutex> g(g_mu);
  return g_on;
}

bool timer_enabled_for(const char* name) {
  std::lock_guard<std::mutex> g(g_mu);
  return g_on && (g_only.empty() || g_only == name);
}

void timer_only(const char* name) {
  std::lock_guard<std::mutex> g(g_mu);
  g_only = name ? name : "";
}

void timer_set(bool on) {
  std::lock_guard<std::mutex> g(g_mu);
  g_on = on;
}

int timer_start(const char* name, cudaStream_t st) {
  std::lock_guard<std::mutex> g(g_mu);
  cudaEvent_t a = take_event(), b = take_event();
  if (!a || !b) return -1;
  if (cudaEventRecord(a, st) != cudaSuccess) return -1;
  g_recs.push_back({name, a, b, false});
  return (int)g_recs.size() - 1;
}

void timer_stop(int h, cudaStream_t st) {
  std::lock_guard<std::mutex> g(g_mu);
  if (h < 0 || h >= (int)g_recs.size()) return;
  if (cudaEventRecord(g_recs[h].b, st) == cudaSuccess) g_recs[h].done = true;
}

int timer_read(const char* name, double* total_ms, int* launches) {
  std::lock_guard<std::mutex> g(g_mu);
  double tot = 0.0;
  int n = 0;
  std::vector<Rec> keep;
  for (auto& r : g_recs) {
    if (r.name != name) {
      keep.push_back(r);
      continue;
    }
    if (r.done && cudaEventSynchronize(r.b) == cudaSuccess) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
        tot += ms;
        ++n;
      }
    }
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.swap(keep);
  if (total_ms) *total_ms = tot;
  if (launches) *launches = n;
  return 0;
}

}  // namespace sage
