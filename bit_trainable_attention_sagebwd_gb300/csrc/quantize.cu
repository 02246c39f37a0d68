// Quantize pass of the SageBwd scheme ("SageBwd: A Trainable Low-bit Attention",
// Methodology 1 and 4): QK-norm, K-smoothing, per-block INT8 codes of Q (128
// tokens) and K (64 tokens), per-channel FP8 e4m3 codes of V (stored
// channel-major for the PV matmul).  HBM-bound: 128-bit loads and stores, one CTA
// per (head, 128-token block), values held in registers between the block
// maximum and the code computation.
//
// Bit-exactness rules: every operation the scheme states in fp32 is a single
// correctly rounded intrinsic (__fmul_rn, __fdiv_rn, ...), so no FMA contraction
// changes a code; sums that feed codes (sum of squares per token, sum over tokens
// per channel) are carried in double-float and rounded once.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "codes.cuh"
#include "kernels.h"
#include "layout.h"
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

// ---------------------------------------------------------------------------
// kstats: per (head, 128-token block): partial fp64 column sums of k' and the
// partial channel maxima of |V|.
template <int D>
__global__ void __launch_bounds__(kThreads) kstats_kernel(const __nv_bfloat16* __restrict__ K,
                                                           const __nv_bfloat16* __restrict__ V, int N,
                                                           int qk_norm, double* __restrict__ kpart,
                                                           float* __restrict__ vpart) {
  constexpr int TPR = D / 8, RPP = kThreads / TPR, PASSES = 128 / RPP;
  const int blk = blockIdx.x, bh = blockIdx.y, nb = gridDim.x;
  const int tid = threadIdx.x, g = tid % TPR, ro = tid / TPR;
  const size_t head = (size_t)bh * N * D;
  DF cs[8];
  float vm[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    cs[i] = {0.f, 0.f};
    vm[i] = 0.f;
  }
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int t = blk * 128 + p * RPP + ro;
    float k[8], v[8];
    uint4 uk = make_uint4(0, 0, 0, 0), uv = make_uint4(0, 0, 0, 0);
    if (t < N) {
      uk = __ldg(reinterpret_cast<const uint4*>(K + head + (size_t)t * D) + g);
      uv = __ldg(reinterpret_cast<const uint4*>(V + head + (size_t)t * D) + g);
    }
    unpack8(uk, k);
    unpack8(uv, v);
    if (qk_norm) {
      const float r = inv_norm<TPR>(k);
#pragma unroll
      for (int i = 0; i < 8; ++i) k[i] = __fmul_rn(k[i], r);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      cs[i] = df_add(cs[i], k[i]);
      vm[i] = fmaxf(vm[i], fabsf(v[i]));
    }
  }
  // combine the RPP row groups per channel in fp64, fixed order
  __shared__ double s_sum[RPP][D];
  __shared__ float s_max[RPP][D];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    s_sum[ro][g * 8 + i] = (double)cs[i].hi + (double)cs[i].lo;
    s_max[ro][g * 8 + i] = vm[i];
  }
  __syncthreads();
  if (tid < D) {
    double s = 0.0;
    float m = 0.f;
    for (int r = 0; r < RPP; ++r) {
      s += s_sum[r][tid];
      m = fmaxf(m, s_max[r][tid]);
    }
    kpart[((size_t)bh * nb + blk) * D + tid] = s;
    vpart[((size_t)bh * nb + blk) * D + tid] = m;
  }
}

// kcombine: per head: channel mean of k' (fp32 rounding of the fp64 sum / N) and
// the V channel scales max|V|/448.
__global__ void kcombine_kernel(const double* __restrict__ kpart, const float* __restrict__ vpart, int N,
                                int D, int nb, int k_smooth, float* __restrict__ kmean,
                                float* __restrict__ sv) {
  const int bh = blockIdx.x, d = threadIdx.x;
  if (d >= D) return;
  double s = 0.0;
  float m = 0.f;
  for (int b = 0; b < nb; ++b) {
    s += kpart[((size_t)bh * nb + b) * D + d];
    m = fmaxf(m, vpart[((size_t)bh * nb + b) * D + d]);
  }
  kmean[(size_t)bh * D + d] = k_smooth ? (float)(s / (double)N) : 0.f;
  sv[(size_t)bh * D + d] = m > 0.f ? __fdiv_rn(m, 448.0f) : 0.f;
}

// quantize: per (head, 128-token block, tensor): blockIdx.z = 0 for Q, 1 for K, 2 for V.
// Each thread issues all of its 128-bit loads before any arithmetic (values stay
// packed bf16 until used) so that a CTA keeps a whole 32 KB block in flight.
template <int D>
__global__ void __launch_bounds__(kThreads) quantize_kernel(
    const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
    const __nv_bfloat16* __restrict__ V, int N, int qk_norm, int k_smooth, const float* __restrict__ kmean,
    const float* __restrict__ sv, __nv_bfloat16* __restrict__ qc, __nv_bfloat16* __restrict__ kc,
    uint8_t* __restrict__ v8t, float* __restrict__ sq, float* __restrict__ sk, float* __restrict__ qr,
    float* __restrict__ kr, int* __restrict__ status) {
  constexpr int TPR = D / 8, RPP = kThreads / TPR, PASSES = 128 / RPP;
  const int blk = blockIdx.x, bh = blockIdx.y, which = blockIdx.z, nb = gridDim.x, np = nb * 128;
  const int tid = threadIdx.x, g = tid % TPR, ro = tid / TPR, warp = tid >> 5, lane = tid & 31;
  const size_t head = (size_t)bh * N * D;
  const size_t phead = (size_t)bh * np * D;
  __shared__ float s_red[2][kThreads / 32];
  // V codes transposed: row d holds the block's 128 tokens; 4-byte groups are
  // permuted by (d / 8) so the byte stores of one warp fall in distinct banks
  __shared__ __align__(16) uint8_t s_v8[D][128];
  if (blk == 0 && bh == 0 && which == 0 && tid == 0) *status = 0;

  const __nv_bfloat16* src = which == 0 ? Q : (which == 1 ? K : V);
  uint4 raw[PASSES];
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int t = blk * 128 + p * RPP + ro;
    raw[p] = t < N ? __ldg(reinterpret_cast<const uint4*>(src + head + (size_t)t * D) + g) : make_uint4(0, 0, 0, 0);
  }

  if (which == 2) {
    // ---- V: e4m3 codes with channel scales, transposed through shared memory
    float svv[8], inv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      svv[i] = sv[(size_t)bh * D + g * 8 + i];
      inv[i] = svv[i] > 0.f ? __frcp_rn(svv[i]) : 0.f;
    }
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      const int row = p * RPP + ro;
      float v[8];
      unpack8(raw[p], v);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int d = g * 8 + i;
        // e4m3(RN(v / s_v)): round to nearest even, saturating to +-448
        s_v8[d][row ^ (((d >> 3) & 15) << 2)] = (uint8_t)e4m3_code(v[i], svv[i], inv[i]);
      }
    }
    __syncthreads();
    // D rows of 128 bytes: 16 bytes per thread per step
    for (int idx = tid; idx < D * 8; idx += kThreads) {
      const int d = idx >> 3, c = idx & 7, f = ((d >> 3) & 15) << 2;
      uint4 val;
      val.x = *reinterpret_cast<const uint32_t*>(&s_v8[d][(c * 16 + 0) ^ f]);
      val.y = *reinterpret_cast<const uint32_t*>(&s_v8[d][(c * 16 + 4) ^ f]);
      val.z = *reinterpret_cast<const uint32_t*>(&s_v8[d][(c * 16 + 8) ^ f]);
      val.w = *reinterpret_cast<const uint32_t*>(&s_v8[d][(c * 16 + 12) ^ f]);
      reinterpret_cast<uint4*>(v8t + ((size_t)bh * D + d) * np + blk * 128)[c] = val;
    }
    return;
  }

  // ---- Q (which == 0): optional norm, one 128-token block max;
  //      K (which == 1): optional norm, minus the channel mean, two 64-token block maxima
  const bool isk = which == 1;
  float km[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) km[i] = (isk && k_smooth) ? kmean[(size_t)bh * D + g * 8 + i] : 0.f;
  float* rout = isk ? kr : qr;
  float x[PASSES][8];
  float am[2] = {0.f, 0.f};
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int t = blk * 128 + p * RPP + ro;
    unpack8(raw[p], x[p]);
    float r = 1.f;
    if (qk_norm) {
      r = inv_norm<TPR>(x[p]);
#pragma unroll
      for (int i = 0; i < 8; ++i) x[p][i] = __fmul_rn(x[p][i], r);
    }
    if (g == 0) rout[(size_t)bh * np + blk * 128 + p * RPP + ro] = r;
    const int hsel = isk && (p * RPP + ro) >= 64;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (isk) x[p][i] = (t < N) ? (k_smooth ? __fsub_rn(x[p][i], km[i]) : x[p][i]) : 0.f;
      am[hsel] = fmaxf(am[hsel], fabsf(x[p][i]));
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
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) a = fmaxf(a, s_red[h][w]);
    sc[h] = a > 0.f ? __fdiv_rn(a, 127.0f) : 0.f;
    inv[h] = sc[h] > 0.f ? __frcp_rn(sc[h]) : 0.f;
  }
  if (!isk) {
    if (tid == 0) sq[(size_t)bh * nb + blk] = sc[0];
  } else if (tid < 2) {
    sk[(size_t)bh * nb * 2 + blk * 2 + tid] = sc[tid];
  }
  __nv_bfloat16* dst = isk ? kc : qc;
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int hs = isk && (p * RPP + ro) >= 64;
    const float s = sc[hs], si = inv[hs];
    float c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = int_code(x[p][i], s, si);
    reinterpret_cast<uint4*>(dst + phead + (size_t)(blk * 128 + p * RPP + ro) * D)[g] = pack8_bf16(c);
  }
}

}  // namespace

int launch_quantize(const void* Q, const void* K, const void* V, int B, int H, int N, int D, int qk_norm,
                    int k_smooth, void* ws, cudaStream_t st) {
  const QuantWs L = quant_ws_layout(B, H, N, D);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int nb = L.np / 128;
  const dim3 grid(nb, B * H);
  const dim3 qgrid(nb, B * H, 3);
  auto* q = static_cast<const __nv_bfloat16*>(Q);
  auto* k = static_cast<const __nv_bfloat16*>(K);
  auto* v = static_cast<const __nv_bfloat16*>(V);
  double* kpart = reinterpret_cast<double*>(w + L.kpart);
  float* vpart = reinterpret_cast<float*>(w + L.vpart);
  float* kmean = reinterpret_cast<float*>(w + L.kmean);
  float* sv = reinterpret_cast<float*>(w + L.sv);
  ScopedTimer timer("quantize", st);
  if (D == 128)
    kstats_kernel<128><<<grid, kThreads, 0, st>>>(k, v, N, qk_norm, kpart, vpart);
  else
    kstats_kernel<64><<<grid, kThreads, 0, st>>>(k, v, N, qk_norm, kpart, vpart);
  kcombine_kernel<<<B * H, 128, 0, st>>>(kpart, vpart, N, D, nb, k_smooth, kmean, sv);
  auto args = [&](auto kern) {
    kern<<<qgrid, kThreads, 0, st>>>(q, k, v, N, qk_norm, k_smooth, kmean, sv,
                                    reinterpret_cast<__nv_bfloat16*>(w + L.qc),
                                    reinterpret_cast<__nv_bfloat16*>(w + L.kc), w + L.v8t,
                                    reinterpret_cast<float*>(w + L.sq), reinterpret_cast<float*>(w + L.sk),
                                    reinterpret_cast<float*>(w + L.qr), reinterpret_cast<float*>(w + L.kr),
                                    reinterpret_cast<int*>(w + L.status));
  };
  if (D == 128)
    args(quantize_kernel<128>);
  else
    args(quantize_kernel<64>);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace sage
