// One attention training step on host-resident tensors with the host<->device copies
// overlapped with the computation (C ABI: sage_attn_step_host_bytes, sage_attn_step_host).
//
// Heads are independent in every pass of the scheme, so the B*H heads are split into
// contiguous ranges.  The inputs of every range are copied in on one copy stream, each
// range is quantized, run forward and backward on the caller's stream once its inputs
// have landed, and its outputs are copied out on a second copy stream while the next
// range computes.  Host-to-device and device-to-host copies use separate copy engines.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "../../include/sage_attn.h"
#include "args.h"
#include "kernels.h"
#include "layout.h"

namespace sage {
namespace {

constexpr int kMaxGroups = 64;

struct StepHostLayout {
  size_t ws, bwd_ws, q, k, v, dO, o, dq, dk, dv, lse, total;
  int groups, hg;              // head ranges and the largest range
  int start[kMaxGroups + 1];   // range g holds heads [start[g], start[g+1])
};

int auto_groups(int bh) { return bh < 5 ? bh : 5; }

// Range sizes: with three ranges or more the first and the last take half the share of
// the others, so the computation starts early and the last copies out are short.
void split_heads(int bh, int g, int* start) {
  const double total = g >= 3 ? g - 1.0 : (double)g;
  double acc = 0.0;
  start[0] = 0;
  for (int i = 0; i < g; ++i) {
    acc += (g >= 3 && (i == 0 || i == g - 1)) ? 0.5 : 1.0;
    int e = (int)(acc / total * bh + 0.5);
    if (e < start[i] + 1) e = start[i] + 1;          // every range holds a head
    if (e > bh - (g - 1 - i)) e = bh - (g - 1 - i);  // ... and leaves one for each later range
    start[i + 1] = e;
  }
  start[g] = bh;
}

StepHostLayout step_host_layout(int B, int H, int N, int D, int groups) {
  StepHostLayout L{};
  const int bh = B * H;
  int g = groups > 0 ? groups : auto_groups(bh);
  if (g > bh) g = bh;
  if (g > kMaxGroups) g = kMaxGroups;
  L.groups = g;
  split_heads(bh, g, L.start);
  L.hg = 0;
  for (int i = 0; i < g; ++i)
    if (L.start[i + 1] - L.start[i] > L.hg) L.hg = L.start[i + 1] - L.start[i];
  const size_t t = (size_t)bh * N * D * 2;  // one bf16 [B, H, N, D] tensor
  size_t o = 0;
  L.ws = o;     o = align256(o + quant_ws_layout(1, L.hg, N, D).total);  // first: its status word
  L.bwd_ws = o; o = align256(o + bwd_ws_layout(1, L.hg, N, D).total);
  L.q = o;      o = align256(o + t);
  L.k = o;      o = align256(o + t);
  L.v = o;      o = align256(o + t);
  L.dO = o;     o = align256(o + t);
  L.o = o;      o = align256(o + t);
  L.dq = o;     o = align256(o + t);
  L.dk = o;     o = align256(o + t);
  L.dv = o;     o = align256(o + t);
  L.lse = o;    o = align256(o + (size_t)bh * N * 4);
  L.total = o;
  return L;
}

// Copy streams and events of the current device, created on first use.
struct CopyEngines {
  int device = -1;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  std::vector<cudaEvent_t> ev;  // [0] start, [1] end, then inputs in / forward done / backward done per range
};

// One set per device, created on the first step on that device and kept until exit; the
// mutex guards creation only (a set in use is never replaced).
constexpr int kMaxDevices = 64;
std::mutex g_engines_mu;
CopyEngines g_engines[kMaxDevices];

CopyEngines* copy_engines() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_engines_mu);
  CopyEngines& e = g_engines[dev];
  if (e.device != dev) {
    if (cudaStreamCreateWithFlags(&e.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&e.d2h, cudaStreamNonBlocking) != cudaSuccess)
      return nullptr;
    e.ev.resize(2 + 3 * kMaxGroups);
    for (auto& x : e.ev)
      if (cudaEventCreateWithFlags(&x, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    e.device = dev;
  }
  return &e;
}

int launch_step_host(const void* Q, const void* K, const void* V, const void* dO, void* O, float* LSE, void* dQ,
                     void* dK, void* dV, void* dev, int B, int H, int N, int D, int causal, int qk_norm,
                     int k_smooth, float sm_scale, int groups, cudaStream_t st) {
  const StepHostLayout L = step_host_layout(B, H, N, D, groups);
  CopyEngines* E = copy_engines();
  if (E == nullptr) return 3;
  uint8_t* d = static_cast<uint8_t*>(dev);
  const size_t head = (size_t)N * D * 2, head_lse = (size_t)N * 4;
  const uint8_t* hin[4] = {static_cast<const uint8_t*>(Q), static_cast<const uint8_t*>(K),
                           static_cast<const uint8_t*>(V), static_cast<const uint8_t*>(dO)};
  uint8_t* din[4] = {d + L.q, d + L.k, d + L.v, d + L.dO};
  uint8_t* hout[4] = {static_cast<uint8_t*>(O), static_cast<uint8_t*>(dQ), static_cast<uint8_t*>(dK),
                      static_cast<uint8_t*>(dV)};
  uint8_t* dout[4] = {d + L.o, d + L.dq, d + L.dk, d + L.dv};
  cudaEvent_t ev_start = E->ev[0], ev_end = E->ev[1];
  // work already on the caller's stream (a previous step using the same buffers) first
  if (cudaEventRecord(ev_start, st) != cudaSuccess || cudaStreamWaitEvent(E->h2d, ev_start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(E->d2h, ev_start, 0) != cudaSuccess)
    return 3;
  for (int g = 0; g < L.groups; ++g) {
    const int h0 = L.start[g], n = L.start[g + 1] - h0;
    for (int t = 0; t < 4; ++t)
      if (cudaMemcpyAsync(din[t] + h0 * head, hin[t] + h0 * head, n * head, cudaMemcpyHostToDevice, E->h2d) !=
          cudaSuccess)
        return 3;
    if (cudaEventRecord(E->ev[2 + 3 * g], E->h2d) != cudaSuccess) return 3;
  }
  for (int g = 0; g < L.groups; ++g) {
    const int h0 = L.start[g], n = L.start[g + 1] - h0;
    const size_t off = h0 * head;
    float* lse = reinterpret_cast<float*>(d + L.lse) + (size_t)h0 * N;
    if (cudaStreamWaitEvent(st, E->ev[2 + 3 * g], 0) != cudaSuccess) return 3;
    // one workspace serves every range in turn; its status word collects their errors
    if (int rc = launch_quantize(din[0] + off, din[1] + off, din[2] + off, 1, n, N, D, qk_norm, k_smooth, d + L.ws,
                                 st, g == 0))
      return rc;
    if (int rc = launch_fwd(d + L.ws, dout[0] + off, lse, nullptr, 1, n, N, D, causal, sm_scale, st)) return rc;
    // O and LSE go out while the range's backward runs
    if (cudaEventRecord(E->ev[3 + 3 * g], st) != cudaSuccess ||
        cudaStreamWaitEvent(E->d2h, E->ev[3 + 3 * g], 0) != cudaSuccess ||
        cudaMemcpyAsync(hout[0] + off, dout[0] + off, n * head, cudaMemcpyDeviceToHost, E->d2h) != cudaSuccess ||
        cudaMemcpyAsync(reinterpret_cast<uint8_t*>(LSE) + h0 * head_lse, lse, n * head_lse, cudaMemcpyDeviceToHost,
                        E->d2h) != cudaSuccess)
      return 3;
    if (int rc = launch_bwd(din[0] + off, din[1] + off, din[2] + off, dout[0] + off, lse, din[3] + off,
                            dout[1] + off, dout[2] + off, dout[3] + off, d + L.ws, d + L.bwd_ws, 1, n, N, D, causal,
                            qk_norm, k_smooth, sm_scale, st))
      return rc;
    if (cudaEventRecord(E->ev[4 + 3 * g], st) != cudaSuccess ||
        cudaStreamWaitEvent(E->d2h, E->ev[4 + 3 * g], 0) != cudaSuccess)
      return 3;
    for (int t = 1; t < 4; ++t)
      if (cudaMemcpyAsync(hout[t] + off, dout[t] + off, n * head, cudaMemcpyDeviceToHost, E->d2h) != cudaSuccess)
        return 3;
  }
  // the caller's stream completes once the outputs are in host memory
  if (cudaEventRecord(ev_end, E->d2h) != cudaSuccess || cudaStreamWaitEvent(st, ev_end, 0) != cudaSuccess) return 3;
  return 0;
}

bool shape_ok(int B, int H, int N, int D) {
  return B >= 1 && H >= 1 && N >= 1 && (D == 64 || D == 128) && (long long)B * H <= 65535 &&
         N <= (1 << 24);
}

}  // namespace
}  // namespace sage

extern "C" {

size_t sage_attn_step_host_bytes(int B, int H, int N, int D, int groups) {
  if (!sage::shape_ok(B, H, N, D)) return 0;
  return sage::step_host_layout(B, H, N, D, groups).total;
}

int sage_attn_step_host(const void* Q, const void* K, const void* V, const void* dO, void* O, float* LSE, void* dQ,
                        void* dK, void* dV, void* dev, size_t dev_bytes, int B, int H, int N, int D, int causal,
                        int qk_norm, int k_smooth, float sm_scale, int groups, void* stream) {
  if (!Q || !K || !V || !dO || !O || !LSE || !dQ || !dK || !dV || !dev || ((uintptr_t)dev & 255u))
    return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  if (!sage::shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  if (dev_bytes < sage::step_host_layout(B, H, N, D, groups).total) return SAGE_ERR_INVALID_ARG;
  return sage::launch_step_host(Q, K, V, dO, O, LSE, dQ, dK, dV, dev, B, H, N, D, causal != 0, qk_norm != 0,
                                k_smooth != 0, sage::resolve_scale(sm_scale, D), groups,
                                static_cast<cudaStream_t>(stream));
}

}  // extern "C"
