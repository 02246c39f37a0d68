// Quantize pass of the SageBwd scheme ("SageBwd: A Trainable Low-bit Attention",
// Methodology 1 and 4): QK-norm, K-smoothing, per-block INT8 codes of Q (128
// tokens) and K (64 tokens), per-channel FP8 e4m3 codes of V (stored
// channel-major for the PV matmul).
//
// HBM-bound, two launches: kstats (V channel maxima, column sums of k'; the last block
// of a head combines them into the V scales and the smoothing mean), then quantize (the
// codes).  Each CTA stages one 128-token block in shared memory with a bulk copy.
// Without QK-norm the maxima run on packed bf16 pairs and the codes on fp32 pairs.
//
// Bit-exactness rules: every operation the scheme states in fp32 is a single
// correctly rounded intrinsic (__fmul_rn, __fdiv_rn, ...), so no FMA contraction
// changes a code; sums that feed codes (sum of squares per token, sum over tokens
// per channel) are carried in double-float and rounded once.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "codes.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "launch.h"
#include "layout.h"
#include "stage.cuh"
#include "timer.h"

namespace sage {

namespace {

constexpr int kThreads = 256;

// Knuth's two-sum: s + e == a + b exactly, s = fl(a + b)
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF df_add(DF x, float y) {
  float s, e;
  two_sum(x.hi, y, s, e);
  return {s, __fadd_rn(x.lo, e)};
}
__device__ __forceinline__ DF df_add(DF x, DF y) {
  float s, e;
  two_sum(x.hi, y.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(x.lo, y.lo));
  float h, l;
  two_sum(s, e, h, l);
  return {h, l};
}
__device__ __forceinline__ DF df_shfl_xor(DF x, int m) {
  return {__shfl_xor_sync(0xffffffffu, x.hi, m), __shfl_xor_sync(0xffffffffu, x.lo, m)};
}
// fp32 rounding of the (exact) value hi + lo
__device__ __forceinline__ float df_round(DF x) { return (float)((double)x.hi + (double)x.lo); }

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 pack8_bf16(const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// 1/||x|| of the token whose 8-channel slices are spread over `tpr` adjacent
// lanes; sigma = fp32 rounding of the exact sum of squares (squares of bf16
// values are exact in fp32), r = RN(1 / RN(sqrt(sigma))), 0 for a zero token.
template <int TPR>
__device__ __forceinline__ float inv_norm(const float (&x)[8]) {
  DF s{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 8; ++i) s = df_add(s, __fmul_rn(x[i], x[i]));
#pragma unroll
  for (int m = TPR / 2; m >= 1; m >>= 1) s = df_add(s, df_shfl_xor(s, m));
  const float sig = df_round(s);
  return sig > 0.f ? __fdiv_rn(1.0f, __fsqrt_rn(sig)) : 0.f;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

// ---- packed pairs: two bf16 in a 32-bit word, or two fp32 in a 64-bit register

// max of two pairs of non-negative bf16 bit patterns (ordered like unsigned integers)
__device__ __forceinline__ uint32_t umax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// largest |x| of the bf16 of a staged row slice (4 words), folded into m (bit patterns)
__device__ __forceinline__ uint32_t absmax_bits(uint32_t m, const uint4& u) {
  m = umax2(m, u.x & 0x7fff7fffu);
  m = umax2(m, u.y & 0x7fff7fffu);
  m = umax2(m, u.z & 0x7fff7fffu);
  return umax2(m, u.w & 0x7fff7fffu);
}

// Knuth's two-sum on fp32 pairs: s + e == a + b exactly in each lane
__device__ __forceinline__ void two_sum2(uint64_t a, uint64_t b, uint64_t& s, uint64_t& e) {
  s = fadd2(a, b);
  const uint64_t bb = fsub2(s, a);
  e = fadd2(fsub2(a, fsub2(s, bb)), fsub2(b, bb));
}

// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// kstats: per (head, 128-token block): partial fp64 column sums of k' (with smoothing only:
// blockIdx.z = 0) and partial channel maxima of |V| (the last z).  The last block
// of a head to finish (a counter per head and tensor, zeroed before the launch) combines
// the partials: the V channel scales max|V| / 448, and the smoothing mean as the fp32
// rounding of (sum over the head's tokens) / N (0 without smoothing).
template <int D, bool QKN>
__global__ void __launch_bounds__(kThreads) kstats_kernel(const __nv_bfloat16* __restrict__ K,
                                                           const __nv_bfloat16* __restrict__ V, int N,
                                                           int k_smooth, double* __restrict__ kpart,
                                                           float* __restrict__ vpart, int* __restrict__ cnt,
                                                           float* __restrict__ kmean, float* __restrict__ sv,
                                                           int* __restrict__ status, float* __restrict__ vg) {
  constexpr int TPR = D / 8, RPP = kThreads / TPR, PASSES = 128 / RPP;
  constexpr int J = kThreads / D;  // threads per channel in the combine
  const int blk = blockIdx.x, bh = blockIdx.y, nb = gridDim.x;
  const bool isk = gridDim.z == 2 && blockIdx.z == 0;  // keys first (with smoothing), then values
  const int tid = threadIdx.x, g = tid % TPR, ro = tid / TPR;
  const int rows = min(128, N - blk * 128);
  extern __shared__ __align__(128) uint8_t stage_buf[];
  __shared__ BlockStage st;
  __shared__ int s_last;
  const __nv_bfloat16* src = (isk ? K : V) + (size_t)bh * N * D + (size_t)blk * 128 * D;
  if (!stage_block(st, stage_buf, src, (uint32_t)rows * D * 2, status)) return;
  pdl_wait();  // the input block is staged; the partials and counters come after the predecessor
  pdl_trigger();
  if (isk) {
    DF cs[8];  // this thread's column sums of its channels (double-float)
    if constexpr (!QKN) {
      // k' = k: the double-float sums run on channel pairs straight from the bf16 words
      uint64_t hi[4], lo[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) hi[w] = lo[w] = 0;
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        const uint4 u = staged<D>(stage_buf, p * RPP + ro, rows, g);
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint64_t sum, err;
          two_sum2(hi[w], bf2f2(wv[w]), sum, err);
          hi[w] = sum;
          lo[w] = fadd2(lo[w], err);
        }
      }
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        cs[2 * w] = {f2lo(hi[w]), f2lo(lo[w])};
        cs[2 * w + 1] = {f2hi(hi[w]), f2hi(lo[w])};
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) cs[i] = {0.f, 0.f};
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        float k[8];
        unpack8(staged<D>(stage_buf, p * RPP + ro, rows, g), k);
        const float r = inv_norm<TPR>(k);
#pragma unroll
        for (int i = 0; i < 8; ++i) k[i] = __fmul_rn(k[i], r);
#pragma unroll
        for (int i = 0; i < 8; ++i) cs[i] = df_add(cs[i], k[i]);
      }
    }
    // combine the rows per channel: the lanes of a warp that hold the same channels (in
    // double-float), then the warps in fp64 in a fixed order.  The per-warp sums go where the
    // staged block was, once every warp is done with it: the block's shared memory is then
    // the staged block alone, and more blocks fit on an SM (the pass is bound by the bytes in
    // flight)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int m = TPR; m < 32; m <<= 1) cs[i] = df_add(cs[i], df_shfl_xor(cs[i], m));
    __syncthreads();
    double(*s_sum)[D] = reinterpret_cast<double(*)[D]>(stage_buf);  // [kThreads / 32][D]
    if ((tid & 31) < TPR) {
#pragma unroll
      for (int i = 0; i < 8; ++i) s_sum[tid >> 5][g * 8 + i] = (double)cs[i].hi + (double)cs[i].lo;
    }
    __syncthreads();
    if (tid < D) {
      double s = 0.0;
      for (int r = 0; r < kThreads / 32; ++r) s += s_sum[r][tid];
      kpart[((size_t)bh * nb + blk) * D + tid] = s;
    }
  } else {
    // |v| maxima on the bf16 bit patterns, two channels per word
    uint32_t vb[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const uint4 u = staged<D>(stage_buf, p * RPP + ro, rows, g);
      vb[0] = umax2(vb[0], u.x & 0x7fff7fffu);
      vb[1] = umax2(vb[1], u.y & 0x7fff7fffu);
      vb[2] = umax2(vb[2], u.z & 0x7fff7fffu);
      vb[3] = umax2(vb[3], u.w & 0x7fff7fffu);
    }
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
      for (int m = TPR; m < 32; m <<= 1) vb[w] = umax2(vb[w], __shfl_xor_sync(0xffffffffu, vb[w], m));
    __syncthreads();  // the staged block is consumed: its space takes the per-warp maxima
    float(*s_max)[D] = reinterpret_cast<float(*)[D]>(stage_buf);  // [kThreads / 32][D]
    if ((tid & 31) < TPR) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        s_max[tid >> 5][g * 8 + 2 * w] = bf_lo(vb[w]);
        s_max[tid >> 5][g * 8 + 2 * w + 1] = bf_hi(vb[w]);
      }
    }
    __syncthreads();
    if (tid < D) {
      float m = 0.f;
      for (int r = 0; r < kThreads / 32; ++r) m = fmaxf(m, s_max[r][tid]);
      vpart[((size_t)bh * nb + blk) * D + tid] = m;
    }
  }
  // count this block; the head's last block combines.  The barrier orders the partial's
  // stores before thread 0's fence, which releases them to the other blocks with the count.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(cnt + (isk ? gridDim.y : 0) + bh, 1) == nb - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // channel tid % D over the blocks j, j + J, ... (j = tid / D), eight loads in flight,
  // then the J results of a channel in a fixed order
  const int d = tid % D, j = tid / D;
  if (isk) {
    double(*s_comb)[D] = reinterpret_cast<double(*)[D]>(stage_buf);  // [J][D], staged block consumed
    const double* part = kpart + (size_t)bh * nb * D + d;
    double s = 0.0;
    int b = j;
    for (; b + 7 * J < nb; b += 8 * J) {
      double v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(part + (size_t)(b + u * J) * D);
#pragma unroll
      for (int u = 0; u < 8; ++u) s += v[u];
    }
    for (; b < nb; b += J) s += __ldcg(part + (size_t)b * D);
    s_comb[j][d] = s;
    __syncthreads();
    if (tid < D) {
      double t = 0.0;
#pragma unroll
      for (int u = 0; u < J; ++u) t += s_comb[u][tid];
      kmean[(size_t)bh * D + tid] = (float)(t / (double)N);
    }
  } else {
    float(*f_comb)[D] = reinterpret_cast<float(*)[D]>(stage_buf);  // [J][D], staged block consumed
    const float* part = vpart + (size_t)bh * nb * D + d;
    float m = 0.f;
    int b = j;
    for (; b + 7 * J < nb; b += 8 * J) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(part + (size_t)(b + u * J) * D);
#pragma unroll
      for (int u = 0; u < 8; ++u) m = fmaxf(m, v[u]);
    }
    for (; b < nb; b += J) m = fmaxf(m, __ldcg(part + (size_t)b * D));
    f_comb[j][d] = m;
    __syncthreads();
    if (tid < D) {
#pragma unroll
      for (int u = 0; u < J; ++u) m = fmaxf(m, f_comb[u][tid]);
      sv[(size_t)bh * D + tid] = m > 0.f ? __fdiv_rn(m, 448.0f) : 0.f;
      if (!k_smooth) kmean[(size_t)bh * D + tid] = 0.f;
    }
    if (vg != nullptr) {
      // NVFP4's tensor scale of V: the head's largest |V| / (448 * 6); every thread's m is at
      // most its channel's maximum, and the threads below D hold the channel maxima
      __syncthreads();  // f_comb is read: its space takes the per-warp maxima
      float* s_hm = reinterpret_cast<float*>(stage_buf);
      float hm = m;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, o));
      if ((tid & 31) == 0) s_hm[tid >> 5] = hm;
      __syncthreads();
      if (tid == 0) {
        float a = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) a = fmaxf(a, s_hm[w]);
        vg[bh] = a > 0.f ? __fdiv_rn(a, 2688.0f) : 0.f;
      }
    }
  }
}

// quantize: per (head, 128-token block, tensor): which = 0 for Q, 1 for K, 2 for V.
template <int D, bool QKN>
__global__ void __launch_bounds__(kThreads) quantize_kernel(
    const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
    const __nv_bfloat16* __restrict__ V, int N, int k_smooth, const float* __restrict__ kmean,
    const float* __restrict__ sv, __nv_bfloat16* __restrict__ qc, __nv_bfloat16* __restrict__ kc,
    uint8_t* __restrict__ v8t, float* __restrict__ sq, float* __restrict__ sk, float* __restrict__ qr,
    float* __restrict__ kr, int* __restrict__ status, int bhk) {
  constexpr int TPR = D / 8, RPP = kThreads / TPR, PASSES = 128 / RPP;
  // grid z runs V, K, then Q: kstats reads K first, then V, so the values it read last are
  // re-read first, then the keys, while they are still in L2
  const int which = blockIdx.z == 2 ? 0 : 2 - (int)blockIdx.z;
  const int blk = blockIdx.x, bh = blockIdx.y, nb = gridDim.x, np = nb * 128;
  const int tid = threadIdx.x, g = tid % TPR, ro = tid / TPR, warp = tid >> 5, lane = tid & 31;
  const size_t phead = (size_t)bh * np * D;
  const int rows = min(128, N - blk * 128);
  extern __shared__ __align__(128) uint8_t stage_buf[];
  __shared__ BlockStage st;
  __shared__ float s_red[2][kThreads / 32];
  // V codes transposed: row d holds the block's 128 tokens; 4-byte groups are
  // permuted by (d / 8) so the byte stores of one warp fall in distinct banks
  __shared__ __align__(16) uint8_t s_v8[D][128];

  // grid y spans the query heads; key/value blocks of heads past bhk (grouped-query
  // attention: fewer key/value heads) have nothing to do
  if (which != 0 && bh >= bhk) return;
  const __nv_bfloat16* src = (which == 0 ? Q : (which == 1 ? K : V)) + (size_t)bh * N * D + (size_t)blk * 128 * D;
  if (!stage_block(st, stage_buf, src, (uint32_t)rows * D * 2, status)) return;
  pdl_wait();  // the scales and the mean come from kstats
  pdl_trigger();

  if (which == 2) {
    // ---- V: e4m3 codes with channel scales, channel-major
    e4m3_block_codes<D, kThreads>([&](int t, int gg) { return staged<D>(stage_buf, t, rows, gg); },
                                  sv + (size_t)bh * D, &s_v8[0][0], v8t + (size_t)bh * D * np + blk * 128, np);
    return;
  }

  // ---- Q (which == 0): optional norm, one 128-token block max;
  //      K (which == 1): optional norm, minus the channel mean, two 64-token block maxima.
  // The staged block is read twice: for the maxima, then for the codes.  Without QK-norm
  // both passes run on bf16 pairs (packed maxima, fp32-pair arithmetic); with it, or for a
  // smoothed key block shorter than 128 tokens, the maxima take the general path.
  const bool isk = which == 1;
  const bool smooth = isk && k_smooth;
  float km[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) km[i] = smooth ? kmean[(size_t)bh * D + g * 8 + i] : 0.f;
  float* rout = isk ? kr : qr;
  float rn[PASSES];
  // x' = x r - m for keys inside the sequence (x r for queries), 0 past its end
  auto prep = [&](int p, float r, float (&x)[8]) {
    const int row = p * RPP + ro;
    unpack8(staged<D>(stage_buf, row, rows, g), x);
    if constexpr (QKN) {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(x[i], r);
    }
    if (isk) {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = (row < rows) ? (k_smooth ? __fsub_rn(x[i], km[i]) : x[i]) : 0.f;
    }
  };
  // rows [0, 64) of the block are passes [0, PASSES / 2): the key half of a pass is uniform
  float am[2] = {0.f, 0.f};
  if (!QKN && !smooth) {
    // x' = x (zero past the end): largest |x| on the bf16 bit patterns
    uint32_t mb[2] = {0u, 0u};
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      // the key half of a pass is uniform: isk selects between two registers
      const uint4 u = staged<D>(stage_buf, p * RPP + ro, rows, g);
      if (isk && p >= PASSES / 2)
        mb[1] = absmax_bits(mb[1], u);
      else
        mb[0] = absmax_bits(mb[0], u);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) am[h] = fmaxf(bf_lo(mb[h]), bf_hi(mb[h]));
  } else if (!QKN && rows == 128) {
    // x' = RN(k - m): |x'| is largest at a channel's largest or smallest k, and rounding
    // is monotonic, so max |x'| = max over channels of RN(kmax - m), RN(m - kmin)
    uint32_t mx[2][4], mn[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        mx[h][w] = 0xff80ff80u;  // -inf, -inf
        mn[h][w] = 0x7f807f80u;  // +inf, +inf
      }
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int h = p >= PASSES / 2;
      const uint4 u = staged<D>(stage_buf, p * RPP + ro, rows, g);
      const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        mx[h][w] = bmax2(mx[h][w], wv[w]);
        mn[h][w] = bmin2(mn[h][w], wv[w]);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        am[h] = max3(am[h], __fsub_rn(bf_lo(mx[h][w]), km[2 * w]), __fsub_rn(km[2 * w], bf_lo(mn[h][w])));
        am[h] = max3(am[h], __fsub_rn(bf_hi(mx[h][w]), km[2 * w + 1]), __fsub_rn(km[2 * w + 1], bf_hi(mn[h][w])));
      }
  }
  if constexpr (!QKN) {
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      rn[p] = 1.f;
      if (g == 0) rout[(size_t)bh * np + blk * 128 + p * RPP + ro] = 1.f;
    }
  }
  if (QKN || (smooth && rows < 128)) {
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int row = p * RPP + ro;
      float x[8];
      if constexpr (QKN) {
        unpack8(staged<D>(stage_buf, row, rows, g), x);
        rn[p] = inv_norm<TPR>(x);
        if (g == 0) rout[(size_t)bh * np + blk * 128 + row] = rn[p];
      }
      prep(p, rn[p], x);
      float a = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(x[i]));
      if (isk && row >= 64)
        am[1] = fmaxf(am[1], a);
      else
        am[0] = fmaxf(am[0], a);
    }
  }
  am[0] = warp_max(am[0]);
  am[1] = warp_max(am[1]);
  if (lane == 0) {
    s_red[0][warp] = am[0];
    s_red[1][warp] = am[1];
  }
  __syncthreads();
  float sc[2], inv[2];
  bool exact[2];  // a scale whose reciprocal is not a finite number: every code divides
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) a = fmaxf(a, s_red[h][w]);
    sc[h] = a > 0.f ? __fdiv_rn(a, 127.0f) : 0.f;
    inv[h] = sc[h] > 0.f ? __frcp_rn(sc[h]) : 0.f;
    exact[h] = !(sc[h] < INFINITY && inv[h] < INFINITY);
  }
  if (!isk) {
    if (tid == 0) sq[(size_t)bh * nb + blk] = sc[0];
  } else if (tid < 2) {
    sk[(size_t)bh * nb * 2 + blk * 2 + tid] = tid ? sc[1] : sc[0];
  }
  __nv_bfloat16* dst = isk ? kc : qc;
  if constexpr (QKN) {
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int row = p * RPP + ro;
      const bool hs = isk && row >= 64;
      float x[8], c[8];
      prep(p, rn[p], x);
      int_codes8(x, hs ? sc[1] : sc[0], hs ? inv[1] : inv[0], c);
      reinterpret_cast<uint4*>(dst + phead + (size_t)(blk * 128 + row) * D)[g] = pack8_bf16(c);
    }
  } else {
    // codes on fp32 pairs: q = RN(x' inv), code = rint(q); q is within 2 ulps of x' / s, so
    // the code is that of the division unless q is within 2^-14 of a half-integer.  With a
    // finite reciprocal |q| <= RN(a inv) < 127.5: no clamp is needed.
    uint64_t km2[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) km2[w] = f2(km[2 * w], km[2 * w + 1]);
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int row = p * RPP + ro;
      const bool hs = isk && p >= PASSES / 2;
      const float sch = hs ? sc[1] : sc[0], invh = hs ? inv[1] : inv[0];
      const bool exacth = hs ? exact[1] : exact[0];
      uint4 out = make_uint4(0u, 0u, 0u, 0u);  // past the end: zero codes
      if (row < rows) {
        const uint4 u = staged<D>(stage_buf, row, rows, g);
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
        uint32_t ow[4];
        const uint64_t inv2 = f2(invh, invh);
        float dm = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint64_t x = bf2f2(wv[w]);
          if (smooth) x = fsub2(x, km2[w]);
          const uint64_t q = fmul2(x, inv2);
          const float r0 = rintf(f2lo(q)), r1 = rintf(f2hi(q));
          const uint64_t d = fsub2(q, f2(r0, r1));
          dm = max3(dm, fabsf(f2lo(d)), fabsf(f2hi(d)));
          __nv_bfloat162 h = __floats2bfloat162_rn(r0, r1);
          ow[w] = *reinterpret_cast<uint32_t*>(&h);
        }
        if (dm > 0.49993896484375f || exacth) {
          // rare: the division decides (and clamps, for non-finite scales)
          float x[8], c[8];
          unpack8(u, x);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (smooth) x[i] = __fsub_rn(x[i], km[i]);
            c[i] = fminf(fmaxf(rintf(__fdiv_rn(x[i], sch)), -127.f), 127.f);
          }
          out = pack8_bf16(c);
        } else {
          out = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
      }
      reinterpret_cast<uint4*>(dst + phead + (size_t)(blk * 128 + row) * D)[g] = out;
    }
  }
}

// ---------------------------------------------------------------------------
// Q-smoothing ("SageBwd: A Trainable Low-bit Attention", Methodology 4 names it beside
// K-smoothing): a 128-token query block loses its channel mean before the INT8 quantizer,
//   qmean_d = RN(sum over the block's tokens of q'_d / tokens),   qs = RN(q' - qmean),
// and the codes and the block scale are those of qs.  The sums are carried in double-float
// and combined in fp64, so the mean is the fp32 rounding of the exact one (as the smoothing
// mean of K in kstats).
template <int D, bool QKN>
__global__ void __launch_bounds__(kThreads) qsmooth_q_kernel(const __nv_bfloat16* __restrict__ Q, int N,
                                                              __nv_bfloat16* __restrict__ qc, float* __restrict__ sq,
                                                              float* __restrict__ qr, float* __restrict__ qmean,
                                                              int* __restrict__ status) {
  constexpr int TPR = D / 8, RPP = kThreads / TPR, PASSES = 128 / RPP;
  const int blk = blockIdx.x, bh = blockIdx.y, nb = gridDim.x, np = nb * 128;
  const int tid = threadIdx.x, g = tid % TPR, ro = tid / TPR, warp = tid >> 5, lane = tid & 31;
  const int rows = min(128, N - blk * 128);
  extern __shared__ __align__(128) uint8_t stage_buf[];
  __shared__ BlockStage st;
  __shared__ double s_sum[kThreads / 32][D];
  __shared__ float s_mean[D];
  __shared__ float s_red[kThreads / 32];
  const __nv_bfloat16* src = Q + (size_t)bh * N * D + (size_t)blk * 128 * D;
  if (!stage_block(st, stage_buf, src, (uint32_t)rows * D * 2, status)) return;
  pdl_wait();
  pdl_trigger();
  // q' of pass p (zero past the end of the sequence)
  float rn[PASSES];
  auto load = [&](int p, float (&x)[8]) {
    unpack8(staged<D>(stage_buf, p * RPP + ro, rows, g), x);
    if constexpr (QKN) {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(x[i], rn[p]);
    }
  };
  DF cs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) cs[i] = {0.f, 0.f};
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int row = p * RPP + ro;
    float x[8];
    if constexpr (QKN) {
      unpack8(staged<D>(stage_buf, row, rows, g), x);
      rn[p] = inv_norm<TPR>(x);
    } else {
      rn[p] = 1.f;
    }
    if (g == 0) qr[(size_t)bh * np + blk * 128 + row] = rn[p];
    load(p, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) cs[i] = df_add(cs[i], x[i]);  // zero past the end
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int m = TPR; m < 32; m <<= 1) cs[i] = df_add(cs[i], df_shfl_xor(cs[i], m));
  if (lane < TPR) {
#pragma unroll
    for (int i = 0; i < 8; ++i) s_sum[warp][g * 8 + i] = (double)cs[i].hi + (double)cs[i].lo;
  }
  __syncthreads();
  if (tid < D) {
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) t += s_sum[w][tid];
    const float m = (float)(t / (double)rows);
    s_mean[tid] = m;
    qmean[((size_t)bh * nb + blk) * D + tid] = m;
  }
  __syncthreads();
  float qm[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) qm[i] = s_mean[g * 8 + i];
  // qs = RN(q' - qmean) for tokens of the sequence, 0 past its end
  auto smoothed = [&](int p, float (&x)[8]) {
    load(p, x);
    const bool live = p * RPP + ro < rows;
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = live ? __fsub_rn(x[i], qm[i]) : 0.f;
  };
  float am = 0.f;
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    float x[8];
    smoothed(p, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(x[i]));
  }
  am = warp_max(am);
  if (lane == 0) s_red[warp] = am;
  __syncthreads();
  float a = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) a = fmaxf(a, s_red[w]);
  const float sc = a > 0.f ? __fdiv_rn(a, 127.0f) : 0.f;
  const float inv = sc > 0.f ? __frcp_rn(sc) : 0.f;
  const bool exact = !(sc < INFINITY && inv < INFINITY);  // every code divides
  if (tid == 0) sq[(size_t)bh * nb + blk] = sc;
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int row = p * RPP + ro;
    float x[8], c[8];
    smoothed(p, x);
    if (exact) {
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = sc > 0.f ? fminf(fmaxf(rintf(__fdiv_rn(x[i], sc)), -127.f), 127.f) : 0.f;
    } else {
      int_codes8(x, sc, inv, c);
    }
    reinterpret_cast<uint4*>(qc + (size_t)bh * np * D + (size_t)(blk * 128 + row) * D)[g] = pack8_bf16(c);
  }
}

// The logit term of Q-smoothing, dsb[qh][I][j] = sum_d qmean[qh][I][d] k''[kvh][j][d] (fp32
// products and sums, d ascending), for the 128 keys j of block kb and every query block I.
// k'' is recomputed as K's quantizer forms it: RN(k r) with QK-norm, minus the smoothing mean.
// One CTA per (key block, query head); a warp takes 8 query blocks at a time, a lane 4 keys:
// 32 FMAs per 16-byte shared load of keys (the query means are a broadcast), which keeps the
// FMA pipe ahead of shared-memory bandwidth (with 4 query blocks it ran at half the FMA rate).
template <int D, bool QKN>
__global__ void __launch_bounds__(kThreads) qs_bias_kernel(const __nv_bfloat16* __restrict__ K, int N,
                                                            int k_smooth, const float* __restrict__ kmean,
                                                            const float* __restrict__ kr,
                                                            const float* __restrict__ qmean, float* __restrict__ dsb,
                                                            int group) {
  constexpr int IC = 64;  // query blocks per chunk: 8 warps x 8
  const int kb = blockIdx.x, qh = blockIdx.y, nb = gridDim.x, np = nb * 128;
  const int kvh = qh / group;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  extern __shared__ __align__(16) float ks[];  // [D][128]: k'' transposed
  __shared__ __align__(16) float qt[D][IC + 4];  // qmean of a chunk of query blocks, transposed
  pdl_wait();  // kmean, the key norms and the query means come from the quantize passes
  pdl_trigger();
  {
    // thread: key t of the block, channels [h D/2, h D/2 + D/2)
    const int t = tid & 127, h = tid >> 7;
    const int key = kb * 128 + t;
    const bool live = key < N;
    const float r = (QKN && live) ? kr[(size_t)kvh * np + key] : 1.f;
    const uint4* row = reinterpret_cast<const uint4*>(K + ((size_t)kvh * N + (live ? key : 0)) * D + h * (D / 2));
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      float x[8];
      unpack8(live ? __ldg(row + c) : make_uint4(0u, 0u, 0u, 0u), x);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int d = h * (D / 2) + c * 8 + i;
        float v = QKN ? __fmul_rn(x[i], r) : x[i];
        if (k_smooth) v = __fsub_rn(v, kmean[(size_t)kvh * D + d]);
        ks[d * 128 + t] = live ? v : 0.f;
      }
    }
  }
  for (int I0 = 0; I0 < nb; I0 += IC) {
    __syncthreads();  // ks is written; the previous chunk's qt is read
    for (int idx = tid; idx < IC * D; idx += kThreads) {
      const int i = idx / D, d = idx % D;
      qt[d][i] = I0 + i < nb ? qmean[((size_t)qh * nb + I0 + i) * D + d] : 0.f;
    }
    __syncthreads();
    float acc[8][4];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; ++d) {
      const float4 kv = *reinterpret_cast<const float4*>(&ks[d * 128 + 4 * lane]);
      const float4 qv0 = *reinterpret_cast<const float4*>(&qt[d][8 * warp]);
      const float4 qv1 = *reinterpret_cast<const float4*>(&qt[d][8 * warp + 4]);
      const float kk[4] = {kv.x, kv.y, kv.z, kv.w};
      const float qq[8] = {qv0.x, qv0.y, qv0.z, qv0.w, qv1.x, qv1.y, qv1.z, qv1.w};
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(qq[a], kk[b], acc[a][b]);
    }
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      const int I = I0 + 8 * warp + a;
      if (I < nb)
        *reinterpret_cast<float4*>(dsb + ((size_t)qh * nb + I) * np + kb * 128 + 4 * lane) =
            make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    }
  }
}

}  // namespace

int launch_quantize(const void* Q, const void* K, const void* V, int B, int H, int N, int D, int qk_norm,
                    int k_smooth, void* ws, cudaStream_t st, bool clear_status, int Hkv, bool q_smooth, bool fp4) {
  const QuantWs L = quant_ws_layout(B, H, N, D, Hkv, q_smooth, fp4);
  const int BHk = B * (Hkv > 0 ? Hkv : H);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int nb = L.np / 128;
  // grid z: V, K, then Q (with Q-smoothing the query blocks take their own kernel)
  const dim3 qgrid(nb, B * H, q_smooth ? 2 : 3);
  auto* q = static_cast<const __nv_bfloat16*>(Q);
  auto* k = static_cast<const __nv_bfloat16*>(K);
  auto* v = static_cast<const __nv_bfloat16*>(V);
  double* kpart = reinterpret_cast<double*>(w + L.kpart);
  float* vpart = reinterpret_cast<float*>(w + L.vpart);
  float* kmean = reinterpret_cast<float*>(w + L.kmean);
  float* sv = reinterpret_cast<float*>(w + L.sv);
  int* status = reinterpret_cast<int*>(w + L.status);
  const size_t stage = (size_t)128 * D * 2;  // one staged token block
  ScopedTimer timer("quantize", st);
  // the per-head counters (and normally the status word) are cleared before the kernels
  const size_t clear_from = clear_status ? L.status : L.sync;
  if (cudaMemsetAsync(w + clear_from, 0, L.qc - clear_from, st) != cudaSuccess) return 3;
  auto stats = D == 128 ? (qk_norm ? kstats_kernel<128, true> : kstats_kernel<128, false>)
                        : (qk_norm ? kstats_kernel<64, true> : kstats_kernel<64, false>);
  auto quant = D == 128 ? (qk_norm ? quantize_kernel<128, true> : quantize_kernel<128, false>)
                        : (qk_norm ? quantize_kernel<64, true> : quantize_kernel<64, false>);
  if (cudaFuncSetAttribute(stats, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)stage) != cudaSuccess ||
      cudaFuncSetAttribute(quant, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)stage) != cudaSuccess)
    return 3;
  int* cnt = reinterpret_cast<int*>(w + L.sync);
  if (launch_pdl(stats, dim3(nb, BHk, k_smooth ? 2 : 1), dim3(kThreads), stage, st, k, v, N, k_smooth, kpart, vpart,
                 cnt, kmean, sv, status, fp4 ? reinterpret_cast<float*>(w + L.vg) : nullptr) != cudaSuccess)
    return 3;
  if (launch_pdl(quant, qgrid, dim3(kThreads), stage, st, q, k, v, N, k_smooth, (const float*)kmean, (const float*)sv,
                 reinterpret_cast<__nv_bfloat16*>(w + L.qc), reinterpret_cast<__nv_bfloat16*>(w + L.kc), w + L.v8t,
                 reinterpret_cast<float*>(w + L.sq), reinterpret_cast<float*>(w + L.sk),
                 reinterpret_cast<float*>(w + L.qr), reinterpret_cast<float*>(w + L.kr), status, BHk) != cudaSuccess)
    return 3;
  // NVFP4 V codes after the quantize pass (its tensor scale comes from kstats)
  if (fp4)
    if (int rc = launch_vfp4(V, BHk, N, D, ws, L, st)) return rc;
  if (q_smooth) {
    auto qsq = D == 128 ? (qk_norm ? qsmooth_q_kernel<128, true> : qsmooth_q_kernel<128, false>)
                        : (qk_norm ? qsmooth_q_kernel<64, true> : qsmooth_q_kernel<64, false>);
    auto bias = D == 128 ? (qk_norm ? qs_bias_kernel<128, true> : qs_bias_kernel<128, false>)
                         : (qk_norm ? qs_bias_kernel<64, true> : qs_bias_kernel<64, false>);
    const size_t ks_bytes = (size_t)D * 128 * 4;
    if (cudaFuncSetAttribute(qsq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)stage) != cudaSuccess ||
        cudaFuncSetAttribute(bias, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ks_bytes) != cudaSuccess)
      return 3;
    float* qmean = reinterpret_cast<float*>(w + L.qmean);
    if (launch_pdl(qsq, dim3(nb, B * H), dim3(kThreads), stage, st, q, N,
                   reinterpret_cast<__nv_bfloat16*>(w + L.qc), reinterpret_cast<float*>(w + L.sq),
                   reinterpret_cast<float*>(w + L.qr), qmean, status) != cudaSuccess)
      return 3;
    // after the Q blocks (their means) and, through them, the K blocks (their norms)
    if (launch_pdl(bias, dim3(nb, B * H), dim3(kThreads), ks_bytes, st, k, N, k_smooth, (const float*)kmean,
                   reinterpret_cast<const float*>(w + L.kr), (const float*)qmean, reinterpret_cast<float*>(w + L.dsb),
                   H / (Hkv > 0 ? Hkv : H)) != cudaSuccess)
      return 3;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace sage
