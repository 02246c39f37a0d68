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
#include "ptx.cuh"
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

// ---------------------------------------------------------------------------
// kstats: per (head, 128-token block): blockIdx.z = 0: partial fp64 column sums of k';
// blockIdx.z = 1: partial channel maxima of |V|.
template <int D>
__global__ void __launch_bounds__(kThreads) kstats_kernel(const __nv_bfloat16* __restrict__ K,
                                                           const __nv_bfloat16* __restrict__ V, int N,
                                                           int qk_norm, double* __restrict__ kpart,
                                                           float* __restrict__ vpart, int* __restrict__ status) {
  constexpr int TPR = D / 8, RPP = kThreads / TPR, PASSES = 128 / RPP;
  const int blk = blockIdx.x, bh = blockIdx.y, nb = gridDim.x;
  const int tid = threadIdx.x, g = tid % TPR, ro = tid / TPR;
  const int rows = min(128, N - blk * 128);
  extern __shared__ __align__(128) uint8_t stage_buf[];
  __shared__ BlockStage st;
  const __nv_bfloat16* src = (blockIdx.z == 0 ? K : V) + (size_t)bh * N * D + (size_t)blk * 128 * D;
  if (!stage_block(st, stage_buf, src, (uint32_t)rows * D * 2, status)) return;
  if (blockIdx.z == 0) {
    DF cs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cs[i] = {0.f, 0.f};
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      float k[8];
      unpack8(staged<D>(stage_buf, p * RPP + ro, rows, g), k);
      if (qk_norm) {
        const float r = inv_norm<TPR>(k);
#pragma unroll
        for (int i = 0; i < 8; ++i) k[i] = __fmul_rn(k[i], r);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) cs[i] = df_add(cs[i], k[i]);
    }
    // combine the RPP row groups per channel in fp64, fixed order
    __shared__ double s_sum[RPP][D];
#pragma unroll
    for (int i = 0; i < 8; ++i) s_sum[ro][g * 8 + i] = (double)cs[i].hi + (double)cs[i].lo;
    __syncthreads();
    if (tid < D) {
      double s = 0.0;
      for (int r = 0; r < RPP; ++r) s += s_sum[r][tid];
      kpart[((size_t)bh * nb + blk) * D + tid] = s;
    }
  } else {
    float vm[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) vm[i] = 0.f;
#pragma unroll
    for (int p = 0; p < PASSES; ++p) {
      float v[8];
      unpack8(staged<D>(stage_buf, p * RPP + ro, rows, g), v);
#pragma unroll
      for (int i = 0; i < 8; ++i) vm[i] = fmaxf(vm[i], fabsf(v[i]));
    }
    __shared__ float s_max[RPP][D];
#pragma unroll
    for (int i = 0; i < 8; ++i) s_max[ro][g * 8 + i] = vm[i];
    __syncthreads();
    if (tid < D) {
      float m = 0.f;
      for (int r = 0; r < RPP; ++r) m = fmaxf(m, s_max[r][tid]);
      vpart[((size_t)bh * nb + blk) * D + tid] = m;
    }
  }
}

// kcombine: per head: channel mean of k' (fp32 rounding of the fp64 sum / N) and
// the V channel scales max|V|/448.
__global__ void kcombine_kernel(const double* __restrict__ kpart, const float* __restrict__ vpart, int N,
                                int D, int nb, int k_smooth, float* __restrict__ kmean,
                                float* __restrict__ sv) {
  const int bh = blockIdx.x, d = threadIdx.x;
  if (d >= D) return;
  // partials summed in block order; their loads are issued 8 at a time
  double s = 0.0;
  float m = 0.f;
  const size_t base = (size_t)bh * nb * D + d;
  int b = 0;
  for (; b + 8 <= nb; b += 8) {
    double ks[8];
    float vs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ks[i] = kpart[base + (size_t)(b + i) * D];
      vs[i] = vpart[base + (size_t)(b + i) * D];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s += ks[i];
      m = fmaxf(m, vs[i]);
    }
  }
  for (; b < nb; ++b) {
    s += kpart[base + (size_t)b * D];
    m = fmaxf(m, vpart[base + (size_t)b * D]);
  }
  kmean[(size_t)bh * D + d] = k_smooth ? (float)(s / (double)N) : 0.f;
  sv[(size_t)bh * D + d] = m > 0.f ? __fdiv_rn(m, 448.0f) : 0.f;
}

// quantize: per (head, 128-token block, tensor): blockIdx.z = 0 for Q, 1 for K, 2 for V.
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
  const size_t phead = (size_t)bh * np * D;
  const int rows = min(128, N - blk * 128);
  extern __shared__ __align__(128) uint8_t stage_buf[];
  __shared__ BlockStage st;
  __shared__ float s_red[2][kThreads / 32];
  // V codes transposed: row d holds the block's 128 tokens; 4-byte groups are
  // permuted by (d / 8) so the byte stores of one warp fall in distinct banks
  __shared__ __align__(16) uint8_t s_v8[D][128];

  const __nv_bfloat16* src = (which == 0 ? Q : (which == 1 ? K : V)) + (size_t)bh * N * D + (size_t)blk * 128 * D;
  if (!stage_block(st, stage_buf, src, (uint32_t)rows * D * 2, status)) return;

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
      uint32_t c8[8];
      unpack8(staged<D>(stage_buf, row, rows, g), v);
      // e4m3(RN(v / s_v)): round to nearest even, saturating to +-448
      e4m3_codes8(v, svv, inv, c8);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int d = g * 8 + i;
        s_v8[d][row ^ (((d >> 3) & 15) << 2)] = (uint8_t)c8[i];
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
  //      K (which == 1): optional norm, minus the channel mean, two 64-token block maxima.
  // The staged block is read twice: for the maxima, then for the codes.
  const bool isk = which == 1;
  float km[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) km[i] = (isk && k_smooth) ? kmean[(size_t)bh * D + g * 8 + i] : 0.f;
  float* rout = isk ? kr : qr;
  float rn[PASSES];
  // x' = x r - m for keys inside the sequence (x r for queries), 0 past its end
  auto prep = [&](int p, float (&x)[8]) {
    const int row = p * RPP + ro;
    unpack8(staged<D>(stage_buf, row, rows, g), x);
    if (qk_norm) {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(x[i], rn[p]);
    }
    if (isk) {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = (row < rows) ? (k_smooth ? __fsub_rn(x[i], km[i]) : x[i]) : 0.f;
    }
  };
  float am[2] = {0.f, 0.f};
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int row = p * RPP + ro;
    float x[8];
    if (qk_norm) {
      unpack8(staged<D>(stage_buf, row, rows, g), x);
      rn[p] = inv_norm<TPR>(x);
    } else {
      rn[p] = 1.f;
    }
    if (g == 0) rout[(size_t)bh * np + blk * 128 + row] = rn[p];
    prep(p, x);
    const int hsel = isk && row >= 64;
#pragma unroll
    for (int i = 0; i < 8; ++i) am[hsel] = fmaxf(am[hsel], fabsf(x[i]));
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
    const int row = p * RPP + ro;
    const int hs = isk && row >= 64;
    float x[8], c[8];
    prep(p, x);
    int_codes8(x, sc[hs], inv[hs], c);
    reinterpret_cast<uint4*>(dst + phead + (size_t)(blk * 128 + row) * D)[g] = pack8_bf16(c);
  }
}

}  // namespace

int launch_quantize(const void* Q, const void* K, const void* V, int B, int H, int N, int D, int qk_norm,
                    int k_smooth, void* ws, cudaStream_t st) {
  const QuantWs L = quant_ws_layout(B, H, N, D);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int nb = L.np / 128;
  const dim3 qgrid(nb, B * H, 3);
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
  // the status word is cleared before the kernels that may set it
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return 3;
  auto stats = D == 128 ? kstats_kernel<128> : kstats_kernel<64>;
  auto quant = D == 128 ? quantize_kernel<128> : quantize_kernel<64>;
  if (cudaFuncSetAttribute(stats, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)stage) != cudaSuccess ||
      cudaFuncSetAttribute(quant, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)stage) != cudaSuccess)
    return 3;
  stats<<<dim3(nb, B * H, 2), kThreads, stage, st>>>(k, v, N, qk_norm, kpart, vpart, status);
  kcombine_kernel<<<B * H, 128, 0, st>>>(kpart, vpart, N, D, nb, k_smooth, kmean, sv);
  quant<<<qgrid, kThreads, stage, st>>>(q, k, v, N, qk_norm, k_smooth, kmean, sv,
                                        reinterpret_cast<__nv_bfloat16*>(w + L.qc),
                                        reinterpret_cast<__nv_bfloat16*>(w + L.kc), w + L.v8t,
                                        reinterpret_cast<float*>(w + L.sq), reinterpret_cast<float*>(w + L.sk),
                                        reinterpret_cast<float*>(w + L.qr), reinterpret_cast<float*>(w + L.kr), status);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace sage
