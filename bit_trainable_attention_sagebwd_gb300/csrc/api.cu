// C ABI entry points (declared in include/sage_attn.h): argument checks,
// workspace carving and launches on the caller's stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/sage_attn.h"
#include "args.h"
#include "kernels.h"
#include "layout.h"
#include "ptx.cuh"
#include "timer.h"

namespace {

bool shape_ok(int B, int H, int N, int D) {
  return B >= 1 && H >= 1 && N >= 1 && (D == 64 || D == 128) && (long long)B * H <= 65535 &&
         N <= (1 << 24);
}
bool aligned16(const void* p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }
// grouped-query attention: Hkv key/value heads, each shared by H / Hkv query heads
bool groups_ok(int H, int Hkv) { return Hkv >= 1 && Hkv <= H && H % Hkv == 0; }

// One CTA waits on a barrier that nothing arrives at; the bounded wait gives up
// after budget_ns and the kernel records the timeout in the status word.
__global__ void selftest_wait_kernel(int* status, unsigned long long budget_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    sage::mbar_init(&bar, 1);
    abort = 0;
    sage::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!sage::mbar_wait(&bar, 0, &abort, budget_ns)) atomicExch(status, sage::kDevTimeout);
  }
}

}  // namespace

namespace sage {
int launch_selftest_wait(void* ws, unsigned long long budget_ns, cudaStream_t st) {
  int* status = reinterpret_cast<int*>(static_cast<uint8_t*>(ws));
  selftest_wait_kernel<<<1, 32, 0, st>>>(status, budget_ns);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
}  // namespace sage

namespace {
// the device pointers of a quantize workspace's sections (qmean, dsb: Q-smoothing layouts only)
void fill_views(uint8_t* w, const sage::QuantWs& L, bool qs, sage_ws_views* v) {
  v->qc = w + L.qc;
  v->kc = w + L.kc;
  v->v8t = w + L.v8t;
  v->sq = reinterpret_cast<float*>(w + L.sq);
  v->sk = reinterpret_cast<float*>(w + L.sk);
  v->sv = reinterpret_cast<float*>(w + L.sv);
  v->kmean = reinterpret_cast<float*>(w + L.kmean);
  v->qr = reinterpret_cast<float*>(w + L.qr);
  v->kr = reinterpret_cast<float*>(w + L.kr);
  v->status = reinterpret_cast<int*>(w + L.status);
  v->n_pad = L.np;
  v->qmean = qs ? reinterpret_cast<float*>(w + L.qmean) : nullptr;
  v->dsb = qs ? reinterpret_cast<float*>(w + L.dsb) : nullptr;
  const bool fp4 = L.v4sf > L.v4;
  v->vg = fp4 ? reinterpret_cast<float*>(w + L.vg) : nullptr;
  v->v4 = fp4 ? w + L.v4 : nullptr;
  v->v4sf = fp4 ? w + L.v4sf : nullptr;
}
}  // namespace

extern "C" {

size_t sage_attn_ws_bytes(int B, int H, int N, int D) {
  if (!shape_ok(B, H, N, D)) return 0;
  return sage::quant_ws_layout(B, H, N, D).total;
}

size_t sage_attn_bwd_ws_bytes(int B, int H, int N, int D) {
  if (!shape_ok(B, H, N, D)) return 0;
  return sage::bwd_ws_layout(B, H, N, D).total;
}

int sage_attn_quantize(const void* Q, const void* K, const void* V, int B, int H, int N, int D, int qk_norm,
                       int k_smooth, void* ws, size_t ws_bytes, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(ws)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  if (ws_bytes < sage::quant_ws_layout(B, H, N, D).total) return SAGE_ERR_INVALID_ARG;
  return sage::launch_quantize(Q, K, V, B, H, N, D, qk_norm != 0, k_smooth != 0, ws,
                               static_cast<cudaStream_t>(stream));
}

int sage_attn_fwd(const void* ws, void* O, float* LSE, float* O32, int B, int H, int N, int D, int causal,
                  float sm_scale, void* stream) {
  if (!aligned16(ws) || !aligned16(O) || LSE == nullptr || ((uintptr_t)LSE & 3u)) return SAGE_ERR_INVALID_ARG;
  if (O32 != nullptr && !aligned16(O32)) return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  return sage::launch_fwd(ws, O, LSE, O32, B, H, N, D, causal != 0, sage::resolve_scale(sm_scale, D),
                          static_cast<cudaStream_t>(stream));
}

int sage_attn_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
                  void* dQ, void* dK, void* dV, const void* ws, void* bwd_ws, size_t bwd_ws_bytes, int B, int H,
                  int N, int D, int causal, int qk_norm, int k_smooth, float sm_scale, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
      !aligned16(dK) || !aligned16(dV) || !aligned16(ws) || !aligned16(bwd_ws) || LSE == nullptr ||
      ((uintptr_t)LSE & 3u))
    return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  if (bwd_ws_bytes < sage::bwd_ws_layout(B, H, N, D).total) return SAGE_ERR_INVALID_ARG;
  return sage::launch_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, B, H, N, D, causal != 0, qk_norm != 0,
                          k_smooth != 0, sage::resolve_scale(sm_scale, D), static_cast<cudaStream_t>(stream));
}

int sage_attn_bwd_o32(const void* Q, const void* K, const void* V, const float* O32, const float* LSE,
                      const void* dO, void* dQ, void* dK, void* dV, const void* ws, void* bwd_ws, size_t bwd_ws_bytes,
                      int B, int H, int N, int D, int causal, int qk_norm, int k_smooth, float sm_scale,
                      void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O32) || !aligned16(dO) || !aligned16(dQ) ||
      !aligned16(dK) || !aligned16(dV) || !aligned16(ws) || !aligned16(bwd_ws) || LSE == nullptr ||
      ((uintptr_t)LSE & 3u))
    return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  if (bwd_ws_bytes < sage::bwd_ws_layout(B, H, N, D).total) return SAGE_ERR_INVALID_ARG;
  return sage::launch_bwd(Q, K, V, nullptr, LSE, dO, dQ, dK, dV, ws, bwd_ws, B, H, N, D, causal != 0,
                          qk_norm != 0, k_smooth != 0, sage::resolve_scale(sm_scale, D), static_cast<cudaStream_t>(stream),
                          O32);
}

size_t sage_attn_gqa_ws_bytes(int B, int H, int Hkv, int N, int D) {
  if (!shape_ok(B, H, N, D) || !groups_ok(H, Hkv)) return 0;
  return sage::quant_ws_layout(B, H, N, D, Hkv).total;
}

size_t sage_attn_gqa_bwd_ws_bytes(int B, int H, int Hkv, int N, int D) {
  if (!shape_ok(B, H, N, D) || !groups_ok(H, Hkv)) return 0;
  return sage::bwd_ws_layout(B, H, N, D, Hkv).total;
}

int sage_attn_gqa_quantize(const void* Q, const void* K, const void* V, int B, int H, int Hkv, int N, int D,
                           int qk_norm, int k_smooth, void* ws, size_t ws_bytes, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(ws)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D) || !groups_ok(H, Hkv)) return SAGE_ERR_UNSUPPORTED;
  if (ws_bytes < sage::quant_ws_layout(B, H, N, D, Hkv).total) return SAGE_ERR_INVALID_ARG;
  return sage::launch_quantize(Q, K, V, B, H, N, D, qk_norm != 0, k_smooth != 0, ws,
                               static_cast<cudaStream_t>(stream), true, Hkv);
}

int sage_attn_gqa_fwd(const void* ws, void* O, float* LSE, float* O32, int B, int H, int Hkv, int N, int D,
                      int causal, float sm_scale, void* stream) {
  if (!aligned16(ws) || !aligned16(O) || LSE == nullptr || ((uintptr_t)LSE & 3u)) return SAGE_ERR_INVALID_ARG;
  if (O32 != nullptr && !aligned16(O32)) return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D) || !groups_ok(H, Hkv)) return SAGE_ERR_UNSUPPORTED;
  return sage::launch_fwd(ws, O, LSE, O32, B, H, N, D, causal != 0, sage::resolve_scale(sm_scale, D),
                          static_cast<cudaStream_t>(stream), Hkv);
}

int sage_attn_gqa_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
                      void* dQ, void* dK, void* dV, const void* ws, void* bwd_ws, size_t bwd_ws_bytes, int B, int H,
                      int Hkv, int N, int D, int causal, int qk_norm, int k_smooth, float sm_scale, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
      !aligned16(dK) || !aligned16(dV) || !aligned16(ws) || !aligned16(bwd_ws) || LSE == nullptr ||
      ((uintptr_t)LSE & 3u))
    return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D) || !groups_ok(H, Hkv)) return SAGE_ERR_UNSUPPORTED;
  if (bwd_ws_bytes < sage::bwd_ws_layout(B, H, N, D, Hkv).total) return SAGE_ERR_INVALID_ARG;
  return sage::launch_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, B, H, N, D, causal != 0, qk_norm != 0,
                          k_smooth != 0, sage::resolve_scale(sm_scale, D), static_cast<cudaStream_t>(stream), nullptr,
                          Hkv);
}

size_t sage_attn_qs_ws_bytes(int B, int H, int Hkv, int N, int D) {
  if (!shape_ok(B, H, N, D) || !groups_ok(H, Hkv)) return 0;
  return sage::quant_ws_layout(B, H, N, D, Hkv, true).total;
}

int sage_attn_qs_quantize(const void* Q, const void* K, const void* V, int B, int H, int Hkv, int N, int D,
                          int qk_norm, int k_smooth, void* ws, size_t ws_bytes, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(ws)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D) || !groups_ok(H, Hkv)) return SAGE_ERR_UNSUPPORTED;
  if (ws_bytes < sage::quant_ws_layout(B, H, N, D, Hkv, true).total) return SAGE_ERR_INVALID_ARG;
  return sage::launch_quantize(Q, K, V, B, H, N, D, qk_norm != 0, k_smooth != 0, ws,
                               static_cast<cudaStream_t>(stream), true, Hkv, true);
}

int sage_attn_qs_fwd(const void* ws, void* O, float* LSE, float* O32, int B, int H, int Hkv, int N, int D,
                     int causal, float sm_scale, void* stream) {
  if (!aligned16(ws) || !aligned16(O) || LSE == nullptr || ((uintptr_t)LSE & 3u)) return SAGE_ERR_INVALID_ARG;
  if (O32 != nullptr && !aligned16(O32)) return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D) || !groups_ok(H, Hkv)) return SAGE_ERR_UNSUPPORTED;
  return sage::launch_fwd(ws, O, LSE, O32, B, H, N, D, causal != 0, sage::resolve_scale(sm_scale, D),
                          static_cast<cudaStream_t>(stream), Hkv, true);
}

int sage_attn_qs_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
                     void* dQ, void* dK, void* dV, const void* ws, void* bwd_ws, size_t bwd_ws_bytes, int B, int H,
                     int Hkv, int N, int D, int causal, int qk_norm, int k_smooth, float sm_scale, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
      !aligned16(dK) || !aligned16(dV) || !aligned16(ws) || !aligned16(bwd_ws) || LSE == nullptr ||
      ((uintptr_t)LSE & 3u))
    return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D) || !groups_ok(H, Hkv)) return SAGE_ERR_UNSUPPORTED;
  if (bwd_ws_bytes < sage::bwd_ws_layout(B, H, N, D, Hkv).total) return SAGE_ERR_INVALID_ARG;
  return sage::launch_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, B, H, N, D, causal != 0, qk_norm != 0,
                          k_smooth != 0, sage::resolve_scale(sm_scale, D), static_cast<cudaStream_t>(stream), nullptr,
                          Hkv, true);
}

int sage_attn_qs_ws_views(void* ws, int B, int H, int Hkv, int N, int D, sage_ws_views* v) {
  if (ws == nullptr || v == nullptr) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D) || !groups_ok(H, Hkv)) return SAGE_ERR_UNSUPPORTED;
  fill_views(static_cast<uint8_t*>(ws), sage::quant_ws_layout(B, H, N, D, Hkv, true), true, v);
  return SAGE_OK;
}

int sage_attn_gqa_ws_views(void* ws, int B, int H, int Hkv, int N, int D, sage_ws_views* v) {
  if (ws == nullptr || v == nullptr) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D) || !groups_ok(H, Hkv)) return SAGE_ERR_UNSUPPORTED;
  fill_views(static_cast<uint8_t*>(ws), sage::quant_ws_layout(B, H, N, D, Hkv), false, v);
  return SAGE_OK;
}

size_t sage_attn_fp4_ws_bytes(int B, int H, int N, int D) {
  if (!shape_ok(B, H, N, D)) return 0;
  return sage::quant_ws_layout(B, H, N, D, 0, false, true).total;
}

int sage_attn_fp4_quantize(const void* Q, const void* K, const void* V, int B, int H, int N, int D, int qk_norm,
                           int k_smooth, void* ws, size_t ws_bytes, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(ws)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  if (ws_bytes < sage::quant_ws_layout(B, H, N, D, 0, false, true).total) return SAGE_ERR_INVALID_ARG;
  return sage::launch_quantize(Q, K, V, B, H, N, D, qk_norm != 0, k_smooth != 0, ws,
                               static_cast<cudaStream_t>(stream), true, 0, false, true);
}

int sage_attn_fp4_fwd(const void* ws, void* O, float* LSE, float* O32, int B, int H, int N, int D, int causal,
                      float sm_scale, void* stream) {
  if (!aligned16(ws) || !aligned16(O) || LSE == nullptr || ((uintptr_t)LSE & 3u)) return SAGE_ERR_INVALID_ARG;
  if (O32 != nullptr && !aligned16(O32)) return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  return sage::launch_fwd(ws, O, LSE, O32, B, H, N, D, causal != 0, sage::resolve_scale(sm_scale, D),
                          static_cast<cudaStream_t>(stream), 0, false, nullptr, true);
}

size_t sage_attn_fp4_bwd_ws_bytes(int B, int H, int N, int D) {
  if (!shape_ok(B, H, N, D)) return 0;
  return sage::bwd_ws_layout(B, H, N, D, 0, true).total;
}

int sage_attn_fp4_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
                      void* dQ, void* dK, void* dV, const void* ws, void* bwd_ws, size_t bwd_ws_bytes, int B, int H,
                      int N, int D, int causal, int qk_norm, int k_smooth, float sm_scale, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
      !aligned16(dK) || !aligned16(dV) || !aligned16(ws) || !aligned16(bwd_ws) || LSE == nullptr ||
      ((uintptr_t)LSE & 3u))
    return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  if (bwd_ws_bytes < sage::bwd_ws_layout(B, H, N, D, 0, true).total) return SAGE_ERR_INVALID_ARG;
  return sage::launch_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, ws, bwd_ws, B, H, N, D, causal != 0, qk_norm != 0,
                          k_smooth != 0, sage::resolve_scale(sm_scale, D), static_cast<cudaStream_t>(stream), nullptr,
                          0, false, true);
}

int sage_attn_fp4_ws_views(void* ws, int B, int H, int N, int D, sage_ws_views* v) {
  if (ws == nullptr || v == nullptr) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  fill_views(static_cast<uint8_t*>(ws), sage::quant_ws_layout(B, H, N, D, 0, false, true), false, v);
  return SAGE_OK;
}

size_t sage_attn_thrift_ws_bytes(int B, int H, int N, int D) {
  if (!shape_ok(B, H, N, D)) return 0;
  return sage::thrift_ws_layout(B, H, N, D).total;
}

int sage_attn_thrift_quantize(const void* Q, const void* K, const void* V, int B, int H, int N, int D, int qk_norm,
                              int k_smooth, int causal, double budget, void* ws, size_t ws_bytes, void* tws,
                              size_t tws_bytes, void* stream) {
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(ws) || !aligned16(tws))
    return SAGE_ERR_INVALID_ARG;
  if (!(budget >= 0.0 && budget <= 1.0)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  if (ws_bytes < sage::quant_ws_layout(B, H, N, D).total || tws_bytes < sage::thrift_ws_layout(B, H, N, D).total)
    return SAGE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (int rc = sage::launch_quantize(Q, K, V, B, H, N, D, qk_norm != 0, k_smooth != 0, ws, st)) return rc;
  return sage::launch_thrift_prepare(Q, K, V, B, H, N, D, qk_norm != 0, causal != 0, budget, ws, tws, st);
}

int sage_attn_thrift_fwd(const void* ws, const void* tws, void* O, float* LSE, float* O32, int B, int H, int N,
                         int D, int causal, float sm_scale, void* stream) {
  if (!aligned16(ws) || !aligned16(tws) || !aligned16(O) || LSE == nullptr || ((uintptr_t)LSE & 3u))
    return SAGE_ERR_INVALID_ARG;
  if (O32 != nullptr && !aligned16(O32)) return SAGE_ERR_INVALID_ARG;
  if (!sage::scale_ok(sm_scale)) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float scale = sage::resolve_scale(sm_scale, D);
  if (int rc = sage::launch_fwd(ws, O, LSE, O32, B, H, N, D, causal != 0, scale, st, 0, false,
                                const_cast<void*>(tws)))
    return rc;
  return sage::launch_thrift_hp(ws, tws, O, LSE, O32, B, H, N, D, causal != 0, scale, st);
}

uint8_t* sage_attn_thrift_sel(void* tws, int B, int H, int N, int D) {
  if (tws == nullptr || !shape_ok(B, H, N, D)) return nullptr;
  return static_cast<uint8_t*>(tws) + sage::thrift_ws_layout(B, H, N, D).sel;
}

int sage_attn_ws_views(void* ws, int B, int H, int N, int D, sage_ws_views* v) {
  if (ws == nullptr || v == nullptr) return SAGE_ERR_INVALID_ARG;
  if (!shape_ok(B, H, N, D)) return SAGE_ERR_UNSUPPORTED;
  fill_views(static_cast<uint8_t*>(ws), sage::quant_ws_layout(B, H, N, D), false, v);
  return SAGE_OK;
}

int sage_attn_get_status(void* ws, void* stream) {
  if (ws == nullptr) return SAGE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int h = 0;
  int* dev = static_cast<int*>(ws);
  if (cudaMemcpyAsync(&h, dev, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return SAGE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SAGE_ERR_CUDA;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpyAsync(dev, &zero, sizeof(int), cudaMemcpyHostToDevice, st) != cudaSuccess) return SAGE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SAGE_ERR_CUDA;
  }
  return h == 0 ? SAGE_OK : (h == sage::kDevTimeout ? SAGE_ERR_TIMEOUT : SAGE_ERR_CUDA);
}

int sage_attn_selftest_wait(void* ws, unsigned long long budget_ns, void* stream) {
  if (!aligned16(ws)) return SAGE_ERR_INVALID_ARG;
  if (budget_ns > 1000000000ull) budget_ns = 1000000000ull;
  return sage::launch_selftest_wait(ws, budget_ns, static_cast<cudaStream_t>(stream));
}

int sage_attn_timer_enable(int on) {
  sage::timer_set(on != 0);
  return SAGE_OK;
}

int sage_attn_timer_only(const char* kernel) {
  sage::timer_only(kernel);
  return SAGE_OK;
}

int sage_attn_timer_read(const char* kernel, double* total_ms, int* launches) {
  if (kernel == nullptr) return SAGE_ERR_INVALID_ARG;
  return sage::timer_read(kernel, total_ms, launches) == 0 ? SAGE_OK : SAGE_ERR_CUDA;
}

const char* sage_attn_status_str(int s) {
  switch (s) {
    case SAGE_OK: return "ok";
    case SAGE_ERR_INVALID_ARG: return "invalid argument";
    case SAGE_ERR_UNSUPPORTED: return "unsupported shape";
    case SAGE_ERR_CUDA: return "CUDA runtime error";
    case SAGE_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
