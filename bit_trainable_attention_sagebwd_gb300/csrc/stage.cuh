// Block staging for the HBM-bound passes, and the channel-scaled e4m3 codes of a staged
// block written channel-major (V in the quantize pass, dO in the backward).
//
// "SageBwd: A Trainable Low-bit Attention" (euno.news summary), Methodology 1 and 2: V and
// dO are FP8 (e4m3) operands with one scale per channel, the scale s = max|x| / 448 of
// the channel over the head's tokens; a code is e4m3(RN(x / s)), round to nearest even,
// saturating at +-448.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "codes.cuh"
#include "ptx.cuh"

namespace sage {
namespace {  // internal linkage: each translation unit keeps its own copy

// the two bf16 of a word as fp32 (exact)
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// fp32 pair of the two bf16 of a word
__device__ __forceinline__ uint64_t bf2f2(uint32_t w) { return f2(bf_lo(w), bf_hi(w)); }
__device__ __forceinline__ float f2lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }


// A 128-token block of one head is contiguous in memory ([token][channel] bf16 rows).
// Each CTA stages its block in shared memory with one bulk copy (issued by thread 0,
// completion on an mbarrier) and computes from there: no data stays in registers across
// the block reductions, so several CTAs per SM keep well over 100 KB in flight.
struct BlockStage {
  uint64_t bar;
  int abort;
};

// Copy `bytes` (a multiple of 16) from src to dst and wait; false for every thread of the
// CTA when the wait ran out (then the workspace status is set).
__device__ __forceinline__ bool stage_block(BlockStage& st, void* dst, const void* src, uint32_t bytes,
                                            int* status) {
  if (threadIdx.x == 0) {
    mbar_init(&st.bar, 1);
    st.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&st.bar, bytes);
    bulk_load(dst, src, bytes, &st.bar);
  }
  mbar_wait(&st.bar, 0, &st.abort);
  __syncthreads();  // every thread sees the same outcome
  if (st.abort) {
    if (threadIdx.x == 0) atomicExch(status, kDevTimeout);
    return false;
  }
  return true;
}

// row `row` (token) of a staged block, channels [8g, 8g+8); zero past the sequence end
template <int D>
__device__ __forceinline__ uint4 staged(const uint8_t* buf, int row, int rows, int g) {
  return row < rows ? reinterpret_cast<const uint4*>(buf + (size_t)row * D * 2)[g] : make_uint4(0, 0, 0, 0);
}


// e4m3 codes of a 128-token block with the channel scales sc[D], written channel-major:
// row d of dst (stride `np` bytes) gets the block's 128 codes of channel d.  load(t, g)
// returns channels [8g, 8g+8) of token t as bf16 (zero past the sequence end).  s8 is
// D x 128 bytes of shared memory.  All NT threads of the CTA take part.
//
// A thread takes 4 consecutive tokens of 8 channels at a time, so the 4 codes of each of
// its channels make one 32-bit word of the transposed block.  q = RN(x inv) with
// inv = RN(1 / s) is within 2 ulps of x / s; its code is that of RN(x / s) unless q lies
// within 8 ulps of an e4m3 midpoint or in e4m3's subnormal range (0 < |q| < 2^-6).  Those
// tokens (a few in a million) take the division.
template <int D, int NT, class Load>
__device__ __forceinline__ void e4m3_block_codes(Load&& load, const float* sc, uint8_t* s8, uint8_t* dst, int np) {
  constexpr int TPR = D / 8, RPP = NT / TPR;
  const int tid = threadIdx.x, g = tid % TPR, ro = tid / TPR;
  float svv[8], inv[8];
  bool force = false;  // a reciprocal that is not finite: that thread's codes all divide
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    svv[i] = sc[g * 8 + i];
    inv[i] = svv[i] > 0.f ? __frcp_rn(svv[i]) : 0.f;
    force |= !(inv[i] < INFINITY);
  }
  uint64_t inv2[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) inv2[w] = f2(inv[2 * w], inv[2 * w + 1]);
  // the word of channel d, tokens 4j..4j+3, sits at byte (4j) ^ f(d) of row d, so that
  // the stores of a warp fall in distinct banks
  constexpr int kFs = D == 128 ? 3 : 4;
#pragma unroll 1
  for (int jj = 0; jj < 32 / RPP; ++jj) {
    const int j = ro + jj * RPP;
    uint32_t c2[4][4];  // [token][channel pair]: two e4m3 codes in the low 16 bits
    uint32_t kmin = ~0u, smin = ~0u;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint4 u = load(4 * j + r, g);
      const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint64_t q = fmul2(bf2f2(wv[w]), inv2[w]);
        const uint32_t b0 = __float_as_uint(f2lo(q)), b1 = __float_as_uint(f2hi(q));
        // a normal e4m3 midpoint has fp32 mantissa bit 19 set and bits 18..0 clear: the key
        // is at most 16 << 12 exactly when q is within 8 ulps of one
        kmin = min(kmin, min(b0 * 4096u + ((8u - 0x80000u) << 12), b1 * 4096u + ((8u - 0x80000u) << 12)));
        // 2 |q|bits - 2 < 2 * 0x3c800000 - 2 exactly when 0 < |q| < 2^-6
        smin = min(smin, min(b0 * 2u - 2u, b1 * 2u - 2u));
        c2[r][w] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(f2lo(q), f2hi(q)), __NV_SATFINITE, __NV_E4M3);
      }
    }
    if (kmin <= (16u << 12) || smin < 0x78fffffeu || force) {
      // rare: the division decides the 32 codes of these 4 tokens
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint4 u = load(4 * j + r, g);
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 x = make_float2(__fdiv_rn(bf_lo(wv[w]), svv[2 * w]), __fdiv_rn(bf_hi(wv[w]), svv[2 * w + 1]));
          c2[r][w] = (uint32_t)__nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
        }
      }
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t x = __byte_perm(c2[0][w], c2[1][w], 0x5410);  // channels 2w, 2w+1 of tokens 0, 1
      const uint32_t y = __byte_perm(c2[2][w], c2[3][w], 0x5410);  // ... of tokens 2, 3
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int d = g * 8 + 2 * w + e;
        *reinterpret_cast<uint32_t*>(s8 + d * 128 + ((4 * j) ^ (((d >> 3) & 15) << kFs))) =
            __byte_perm(x, y, e ? 0x7531 : 0x6420);
      }
    }
  }
  __syncthreads();
  // D rows of 128 bytes: 16 bytes per thread per step
  for (int idx = tid; idx < D * 8; idx += NT) {
    const int d = idx >> 3, c = idx & 7, f = ((d >> 3) & 15) << kFs;
    const uint8_t* row = s8 + d * 128;
    uint4 val;
    val.x = *reinterpret_cast<const uint32_t*>(row + ((c * 16 + 0) ^ f));
    val.y = *reinterpret_cast<const uint32_t*>(row + ((c * 16 + 4) ^ f));
    val.z = *reinterpret_cast<const uint32_t*>(row + ((c * 16 + 8) ^ f));
    val.w = *reinterpret_cast<const uint32_t*>(row + ((c * 16 + 12) ^ f));
    reinterpret_cast<uint4*>(dst + (size_t)d * np)[c] = val;
  }
}

}  // namespace
}  // namespace sage
