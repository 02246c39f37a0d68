// Internal launchers (host side); each returns 0 or a sage_status code.
#pragma once

#include <cuda_runtime.h>

namespace sage {

// Grouped-query attention: Hkv key/value heads per batch entry, Hkv divides H (0: Hkv = H);
// query head h reads key/value head h / (H / Hkv).
// clear_status = false keeps the workspace status word (errors of earlier launches).
// q_smooth: Q-smoothing (the query blocks' channel means leave the INT8 codes and come back as
// a logit term); the workspace then has the layout quant_ws_layout(..., qs = true), and the
// forward and backward on it take q_smooth too.
// fp4: also V's NVFP4 codes and block scales (quant_ws_layout(..., fp4 = true))
int launch_quantize(const void* Q, const void* K, const void* V, int B, int H, int N, int D, int qk_norm,
                    int k_smooth, void* ws, cudaStream_t st, bool clear_status = true, int Hkv = 0,
                    bool q_smooth = false, bool fp4 = false);
struct QuantWs;
int launch_vfp4(const void* V, int BHk, int N, int D, void* ws, const QuantWs& L, cudaStream_t st);
// tws (ThriftAttention scratch, thrift_ws_layout): skip the promoted pairs and hand the rows of
// query tiles that have any to launch_thrift_hp (plain heads only)
// fp4: NVFP4 PV on a workspace quantized with fp4 (plain heads only)
int launch_fwd(const void* ws, void* O, float* LSE, float* O32, int B, int H, int N, int D, int causal,
               float sm_scale, cudaStream_t st, int Hkv = 0, bool q_smooth = false, void* tws = nullptr,
               bool fp4 = false);
// ThriftAttention: block means, pair scores and the promoted pairs of ceil(budget x visible
// pairs) per head, and the fp16 operands of the high-precision path (after launch_quantize)
int launch_thrift_prepare(const void* Q, const void* K, const void* V, int B, int H, int N, int D, int qk_norm,
                          int causal, double budget, const void* ws, void* tws, cudaStream_t st);
// ThriftAttention: the promoted tiles of every query tile that has any, after launch_fwd(..., tws)
int launch_thrift_hp(const void* ws, const void* tws, void* O, float* LSE, float* O32, int B, int H, int N, int D,
                     int causal, float sm_scale, cudaStream_t st);
// O32 (optional, fp32 [B,H,N,D]) replaces O in the row terms D_i = sum_d dO O
int launch_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
               void* dQ, void* dK, void* dV, const void* ws, void* bwd_ws, int B, int H, int N, int D,
               int causal, int qk_norm, int k_smooth, float sm_scale, cudaStream_t st, const float* O32 = nullptr,
               int Hkv = 0, bool q_smooth = false, bool fp4 = false);
// dQ epilogue of the backward (the work ticket in the backward workspace must be zero)
int launch_bwd_dq(const void* Q, const float* qr, void* bwd_ws, void* dQ, int B, int H, int N, int D, int qk_norm,
                  float sm_scale, int* status, cudaStream_t st, int Hkv = 0);
int launch_selftest_wait(void* ws, unsigned long long budget_ns, cudaStream_t st);

}  // namespace sage
