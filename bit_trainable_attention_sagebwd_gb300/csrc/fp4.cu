// NVFP4 codes of V for the FP4 variant of the forward PV.
//
// "Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (gist.science summary),
// Methodology principle 1 and Implementation: attention trained in FP4, with the backward
// recomputing P at the forward's precision and a native FP4 path on Blackwell;
// "ThriftAttention" (gist.science summary), Methodology step 2: the NVFP4 microscaling format
// of Blackwell's FP4 tensor cores.  Neither page prints the recipe; the format used is NVFP4:
// e2m1 codes (0, 0.5, 1, 1.5, 2, 3, 4, 6; nearest, ties to the even code, saturating), one
// e4m3 scale per 16 consecutive values along the contracted axis, one fp32 scale per tensor.
//
// V (contracted over keys in PV), per head: g = RN(max|V| / (448 * 6)) (written by kstats);
// per channel d and 16-token block, s = e4m3(RN(amax / RN(6 g))), code = e2m1(RN(v / RN(s g))).
// The tensor core multiplies code by s; g comes back in the forward's epilogue.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "launch.h"
#include "layout.h"
#include "ptx.cuh"
#include "stage.cuh"

namespace sage {

namespace {

constexpr int kThreadsV4 = 256;

// e2m1 codes of two values, the first in the low nibble
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(lo, hi), __NV_E2M1, cudaRoundNearest);
}

// One CTA per (128-token block, key/value head): the block is staged in shared memory; a
// thread takes (channel, 16-token block) pairs, channel fastest, so a warp reads 64
// contiguous bytes of a token row.
template <int D>
__global__ void __launch_bounds__(kThreadsV4) vfp4_kernel(const __nv_bfloat16* __restrict__ V, int N, int np,
                                                         const float* __restrict__ vg, uint8_t* __restrict__ v4,
                                                         uint8_t* __restrict__ v4sf, int* __restrict__ status) {
  const int blk = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int rows = min(128, N - blk * 128);
  extern __shared__ __align__(128) uint8_t stage_buf[];
  __shared__ BlockStage st;
  if (!stage_block(st, stage_buf, V + ((size_t)bh * N + (size_t)blk * 128) * D, (uint32_t)rows * D * 2, status))
    return;
  pdl_wait();  // g comes from kstats (two kernels back)
  pdl_trigger();
  const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(stage_buf);
  const float g = vg[bh];
  const float g6 = __fmul_rn(6.0f, g);
#pragma unroll
  for (int i = 0; i < D * 8 / kThreadsV4; ++i) {
    const int pr = tid + kThreadsV4 * i, d = pr % D, b16 = pr / D;
    float v[16];
    float a = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int t = b16 * 16 + r;
      v[r] = t < rows ? __bfloat162float(x[t * D + d]) : 0.f;
      a = fmaxf(a, fabsf(v[r]));
    }
    float s = 0.f;
    uint32_t sbyte = 0;
    if (a > 0.f && g6 > 0.f) {
      sbyte = (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(a, g6), __NV_SATFINITE, __NV_E4M3);
      s = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sbyte, __NV_E4M3)));
    }
    const float sg = __fmul_rn(s, g);
    uint32_t w[2] = {0u, 0u};
    if (sg > 0.f) {
#pragma unroll
      for (int r = 0; r < 16; r += 2)
        w[r >> 3] |= e2m1x2(__fdiv_rn(v[r], sg), __fdiv_rn(v[r + 1], sg)) << (4 * (r & 7));
    }
    *reinterpret_cast<uint2*>(v4 + ((size_t)bh * D + d) * (np / 2) + blk * 64 + b16 * 8) = make_uint2(w[0], w[1]);
    v4sf[((size_t)bh * (np / 64) + blk * 2 + (b16 >> 2)) * 512 + (d & 31) * 16 + (d >> 5) * 4 + (b16 & 3)] =
        (uint8_t)sbyte;
  }
}

}  // namespace

int launch_vfp4(const void* V, int BHk, int N, int D, void* ws, const QuantWs& L, cudaStream_t st) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t stage = (size_t)128 * D * 2;
  auto kern = D == 128 ? vfp4_kernel<128> : vfp4_kernel<64>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)stage) != cudaSuccess) return 3;
  if (launch_pdl(kern, dim3(L.np / 128, BHk), dim3(kThreadsV4), stage, st, static_cast<const __nv_bfloat16*>(V), N,
                 L.np, reinterpret_cast<const float*>(w + L.vg), w + L.v4, w + L.v4sf,
                 reinterpret_cast<int*>(w + L.status)) != cudaSuccess)
    return 3;
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace sage
