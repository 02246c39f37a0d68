// dQ epilogue of the backward of SageBwd-style attention: dQ = sm_scale * acc, through the
// QK-norm Jacobian, to bf16 rows.
//
// "SageBwd: A Trainable Low-bit Attention" (euno.news summary), Methodology 4: with QK-norm
// the gradient of q = x / ||x|| is passed back as r (g - q (q . g)), r = 1 / ||x||.
//
// HBM-bound: the fp32 accumulator [BH][D][Np] (feature-major) is read once and dQ written
// once.  One persistent launch walks 64-query chunk items (stream.cuh); each chunk
// [D x 64 queries] arrives in shared memory by one TMA tile copy, several items ahead.
#include <cuda_bf16.h>

#include "kernels.h"
#include "launch.h"
#include "layout.h"
#include "ptx.cuh"
#include "stream.cuh"
#include "timer.h"
#include "tmap.h"

namespace sage {

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 64;  // queries per item

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

struct DqParams {
  const __nv_bfloat16* Q;
  const float* qr;
  int N, np, nc, BH, qk_norm;
  float sm_scale;
  __nv_bfloat16* dQ;
  int* ticket;
  int* status;
};

// One item: 64 queries of one head.  Warp w takes the queries 32 (w & 1) + lane and the
// features [F (w >> 1), F (w >> 1) + F), F = D / 4; the accumulator chunk is [D][64] fp32
// in shared memory, so a warp reads 32 consecutive floats per feature.
template <int D>
__global__ void __launch_bounds__(kThreads, 2) bwd_dq_kernel(const __grid_constant__ CUtensorMap tacc,
                                                             const DqParams p) {
  constexpr int NS = D == 128 ? 3 : 4;
  constexpr int F = D / 4;
  constexpr uint32_t kStage = kChunk * D * 4;
  extern __shared__ __align__(128) uint8_t stages[];
  __shared__ StreamCtl<NS> ctl;
  __shared__ float s_dot[4][kChunk];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tl = (warp & 1) * 32 + lane, fg = warp >> 1;
  if (tid == 0) tma_prefetch_desc(&tacc);
  pdl_wait();  // the accumulator comes from the main backward kernel
  pdl_trigger();
  auto issue = [&](int item, uint8_t* stage, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, kStage);
    tma_load_3d(stage, &tacc, (item % p.nc) * kChunk, 0, item / p.nc, bar);
  };
  auto body = [&](int item, uint8_t* stage) {
    const int bh = item / p.nc, t = (item % p.nc) * kChunk + tl;
    const bool live = t < p.N;
    const float* tile = reinterpret_cast<const float*>(stage);
    float x[F];
#pragma unroll
    for (int j = 0; j < F; ++j) x[j] = tile[(fg * F + j) * kChunk + tl] * p.sm_scale;
    const size_t row = ((size_t)bh * p.N + t) * D + fg * F;
    if (p.qk_norm) {
      // dq = r (g - qn (qn . g)) with qn = q r: the Jacobian of q -> q / ||q||
      const float rr = live ? p.qr[(size_t)bh * p.np + t] : 0.f;
      float qn[F];
#pragma unroll
      for (int u = 0; u < F / 8; ++u) {
        float v[8];
        unpack8(live ? __ldg(reinterpret_cast<const uint4*>(p.Q + row) + u) : make_uint4(0, 0, 0, 0), v);
#pragma unroll
        for (int i = 0; i < 8; ++i) qn[8 * u + i] = __fmul_rn(v[i], rr);
      }
      float dot = 0.f;
#pragma unroll
      for (int j = 0; j < F; ++j) dot = fmaf(qn[j], x[j], dot);
      s_dot[fg][tl] = dot;
      __syncthreads();
      dot = (s_dot[0][tl] + s_dot[1][tl]) + (s_dot[2][tl] + s_dot[3][tl]);
#pragma unroll
      for (int j = 0; j < F; ++j) x[j] = rr * (x[j] - qn[j] * dot);
    }
    if (live) {
#pragma unroll
      for (int u = 0; u < F / 8; ++u) {
        uint4 o;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(x[8 * u + 2 * e], x[8 * u + 2 * e + 1]);
        reinterpret_cast<uint4*>(p.dQ + row)[u] = o;
      }
    }
  };
  stream_items<NS>(ctl, stages, kStage, p.ticket, p.BH * p.nc, p.status, issue, body);
}

}  // namespace

int launch_bwd_dq(const void* Q, const float* qr, void* bwd_ws, void* dQ, int B, int H, int N, int D, int qk_norm,
                  float sm_scale, int* status, cudaStream_t st, int Hkv) {
  const BwdWs L = bwd_ws_layout(B, H, N, D, Hkv);
  uint8_t* bw = static_cast<uint8_t*>(bwd_ws);
  const int BH = B * H;
  CUtensorMap tacc;
  // the accumulator [BH][D][Np] fp32, boxes of all D features x 64 queries, unswizzled
  if (!make_tmap_3d(&tacc, bw + L.dqacc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, L.np, D, BH, kChunk, D,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
    return 3;
  DqParams p;
  p.Q = static_cast<const __nv_bfloat16*>(Q);
  p.qr = qr;
  p.N = N;
  p.np = L.np;
  p.nc = L.np / kChunk;
  p.BH = BH;
  p.qk_norm = qk_norm;
  p.sm_scale = sm_scale;
  p.dQ = static_cast<__nv_bfloat16*>(dQ);
  p.ticket = reinterpret_cast<int*>(bw + L.sync);  // zeroed by bwd_pre
  p.status = status;
  const int nitems = BH * p.nc;
  if (nitems == 0) return 0;
  auto kern = D == 128 ? bwd_dq_kernel<128> : bwd_dq_kernel<64>;
  const size_t smem = (size_t)(D == 128 ? 3 : 4) * kChunk * D * 4;
  // the attribute is per device: set on every launch, so a second GPU of the process gets it too
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 3;
  if (launch_pdl(kern, dim3(persistent_grid(kern, kThreads, smem, nitems)), dim3(kThreads), smem, st, tacc, p) !=
      cudaSuccess)
    return 3;
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace sage
