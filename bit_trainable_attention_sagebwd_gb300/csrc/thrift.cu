// ThriftAttention's selective mixed precision on tcgen05 tensor cores (forward only).
//
// "ThriftAttention" (gist.science summary), Methodology:
//   step 1: the importance of a (query block, key block) pair is the dot product of the
//           blocks' token means, qbar_I . kbar_J; the top-k pairs are promoted;
//   step 2: promoted pairs run in FP16, the others on the low-precision path, and both merge
//           in one FlashAttention-2 online softmax;
//   implementation: the kernel runs the non-selected blocks on the low-precision path first,
//           then the promoted ones in a separate high-precision routine that loads FP16 query
//           tiles only where needed; warps without promoted blocks skip it.
//
// Blocks are this library's 128-query blocks and 128-key tiles.  The low-precision path is
// the INT8 QK^T / e4m3 PV forward of fwd.cu, which skips the promoted tiles and hands the
// rows of query tiles that have any to the kernel here (unnormalised fp32 output, running
// maximum, row sum).  Kernels:
//   thrift_means_kernel   per (128-token block, head, tensor): fp64 channel means of the raw
//                         Q or K block, tokens added in order
//   thrift_score_kernel   per (query block, head): scores qbar_I . kbar_J in fp64, channels
//                         added in order, as order-preserving 64-bit keys
//   thrift_select_kernel  per head: the n largest keys of the visible pairs, ties in index order
//   thrift_prep_kernel    fp16 copies of q', k'' and V for the high-precision path
//   fwd_hp_kernel         per (head, 128-query tile with a promoted pair): S16 = Q16 K16^T and
//                         O += P16 V16 (kind::f16 with fp16 operands) over the promoted tiles,
//                         then O / l and LSE
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "launch.h"
#include "layout.h"
#include "ptx.cuh"
#include "timer.h"
#include "tmap.h"

namespace sage {

namespace {

constexpr float kLog2_448 = 8.807354922057604f;

// ------------------------------------------------------------------ selection
// channel means of one 128-token block of the raw input (tokens [0, cnt) of the block): the
// fp64 sum of the tokens in order, divided by cnt.  That sum is exact whenever every partial
// sum is representable, which holds when the nonzero values' exponents span at most 38: a bf16
// value is m 2^(e - 134) with an 8-bit m (e >= 1), so each partial sum is an integer multiple
// of 2^(emin - 134) below 128 * 2^8 * 2^38 = 2^53 of them.  Then the sum is accumulated exactly
// in a 64-bit integer (fp64 runs at 1/64 of the fp32 rate on this part); otherwise, or with an
// infinity or NaN in the block, the fp64 sum is taken in order.
template <int D>
__global__ void __launch_bounds__(D) thrift_means_kernel(const __nv_bfloat16* __restrict__ Q,
                                                        const __nv_bfloat16* __restrict__ K, int N,
                                                        double* __restrict__ qbar, double* __restrict__ kbar) {
  const int blk = blockIdx.x, bh = blockIdx.y, d = threadIdx.x, nb = gridDim.x;
  const uint16_t* x = reinterpret_cast<const uint16_t*>(blockIdx.z == 0 ? Q : K) +
                      ((size_t)bh * N + (size_t)blk * 128) * D + d;
  double* out = blockIdx.z == 0 ? qbar : kbar;
  pdl_wait();
  pdl_trigger();
  const int cnt = min(128, N - blk * 128);
  int emin = 255, emax = 0;
  bool special = false;
  for (int t = 0; t < cnt; ++t) {
    const uint32_t u = x[(size_t)t * D];
    const int e = (int)((u >> 7) & 0xFFu);
    if (e == 0xFF) special = true;
    if ((u & 0x7FFFu) != 0u) {
      const int ee = e > 0 ? e : 1;
      emin = min(emin, ee);
      emax = max(emax, ee);
    }
  }
  double s;
  if (!special && emax - emin <= 38) {
    long long acc = 0;
    for (int t = 0; t < cnt; ++t) {
      const uint32_t u = x[(size_t)t * D];
      const uint32_t e = (u >> 7) & 0xFFu, f = u & 0x7Fu;
      if ((u & 0x7FFFu) == 0u) continue;
      const long long v = (long long)(e ? (f | 0x80u) : f) << ((e ? (int)e : 1) - emin);
      acc += (u & 0x8000u) ? -v : v;
    }
    s = ldexp((double)acc, emin - 134);  // |acc| < 2^53: exact
  } else {
    s = 0.0;
    for (int t = 0; t < cnt; ++t) s = __dadd_rn(s, (double)__bfloat162float(__ushort_as_bfloat16(x[(size_t)t * D])));
  }
  out[((size_t)bh * nb + blk) * D + d] = __ddiv_rn(s, (double)cnt);
}

// descending order of the score <-> descending unsigned order of the key; -0 counts as +0
__device__ __forceinline__ unsigned long long score_key(double s) {
  s = __dadd_rn(s, 0.0);  // -0 + 0 = +0
  const unsigned long long u = (unsigned long long)__double_as_longlong(s);
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// one query block's scores against every key block it may see; the key blocks' means pass
// through shared memory 32 at a time (row stride D + 1 doubles against bank conflicts)
template <int D>
__global__ void __launch_bounds__(256) thrift_score_kernel(const double* __restrict__ qbar,
                                                          const double* __restrict__ kbar, int causal,
                                                          unsigned long long* __restrict__ keys) {
  constexpr int R = 32;
  __shared__ double sq[D];
  __shared__ double sk[R][D + 1];
  const int I = blockIdx.x, bh = blockIdx.y, nb = gridDim.x, tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  for (int d = tid; d < D; d += 256) sq[d] = qbar[((size_t)bh * nb + I) * D + d];
  const int nJ = causal ? I + 1 : nb;
  unsigned long long* out = keys + ((size_t)bh * nb + I) * nb;
  for (int J0 = 0; J0 < nJ; J0 += R) {
    const int rows = min(R, nJ - J0);
    __syncthreads();
    for (int e = tid; e < rows * D; e += 256) {
      const int r = e / D, d = e - r * D;
      sk[r][d] = kbar[((size_t)bh * nb + J0 + r) * D + d];
    }
    __syncthreads();
    if (tid < rows) {
      double s = 0.0;
#pragma unroll 8
      for (int d = 0; d < D; ++d) s = __dadd_rn(s, __dmul_rn(sq[d], sk[tid][d]));
      out[J0 + tid] = score_key(s);
    }
  }
}

// Per head: promote the n pairs of largest key among the visible ones (causal: J <= I), the
// pairs of the n-th largest key in index order (I nb + J).  The n-th largest key is found by
// radix selection, eight bits at a time from the top.
__global__ void __launch_bounds__(1024) thrift_select_kernel(const unsigned long long* __restrict__ keys, int nb,
                                                            int causal, int n, uint8_t* __restrict__ sel) {
  __shared__ unsigned int hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ int s_remaining;
  __shared__ int s_warp[32];
  __shared__ int s_base;
  const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t npairs = (size_t)nb * nb;
  const unsigned long long* kh = keys + (size_t)bh * npairs;
  uint8_t* sh = sel + (size_t)bh * npairs;
  pdl_wait();
  pdl_trigger();
  auto visible = [&](size_t p) { return !causal || (int)(p % nb) <= (int)(p / nb); };
  if (n <= 0) {
    for (size_t p = tid; p < npairs; p += 1024) sh[p] = 0;
    return;
  }
  if (tid == 0) {
    s_prefix = 0ull;
    s_remaining = n;
  }
  unsigned long long mask = 0ull;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += 1024) hist[b] = 0u;
    __syncthreads();
    const unsigned long long prefix = s_prefix;
    for (size_t p = tid; p < npairs; p += 1024) {
      if (!visible(p)) continue;
      const unsigned long long k = kh[p];
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      int rem = s_remaining, b = 255;
      for (; b > 0; --b) {
        if ((int)hist[b] >= rem) break;
        rem -= (int)hist[b];
      }
      s_prefix = prefix | ((unsigned long long)b << shift);
      s_remaining = rem;
    }
    mask |= 255ull << shift;
    __syncthreads();
  }
  // s_prefix is the n-th largest key T; s_remaining of the pairs equal to T are taken
  const unsigned long long T = s_prefix;
  const int take = s_remaining;
  if (tid == 0) s_base = 0;
  __syncthreads();
  for (size_t p0 = 0; p0 < npairs; p0 += 1024) {
    const size_t p = p0 + tid;
    int eq = 0;
    uint8_t v = 0;
    if (p < npairs && visible(p)) {
      const unsigned long long k = kh[p];
      v = k > T;
      eq = k == T;
    }
    // exclusive prefix count of the equal keys in index order
    const unsigned int ballot = __ballot_sync(0xffffffffu, eq);
    const int in_warp = __popc(ballot & ((1u << lane) - 1u));
    if (lane == 0) s_warp[warp] = __popc(ballot);
    __syncthreads();
    int before = s_base;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    if (eq && before + in_warp < take) v = 1;
    if (p < npairs) sh[p] = v;
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int w = 0; w < 32; ++w) tot += s_warp[w];
      s_base += tot;
    }
    __syncthreads();
  }
}

// fp16 copies of the high-precision path's operands: q' (QK-norm), k'' = RN(k' - kmean), V;
// rows past N are zero.  grid (Np / 128, BH, 3): z = q, k, v
template <int D>
__global__ void __launch_bounds__(256) thrift_prep_kernel(const __nv_bfloat16* __restrict__ Q,
                                                         const __nv_bfloat16* __restrict__ K,
                                                         const __nv_bfloat16* __restrict__ V, int N, int np,
                                                         int qk_norm, const float* __restrict__ qr,
                                                         const float* __restrict__ kr,
                                                         const float* __restrict__ kmean, __half* __restrict__ q16,
                                                         __half* __restrict__ k16, __half* __restrict__ v16) {
  const int blk = blockIdx.x, bh = blockIdx.y, which = blockIdx.z;
  const __nv_bfloat16* src = which == 0 ? Q : (which == 1 ? K : V);
  __half* dst = which == 0 ? q16 : (which == 1 ? k16 : v16);
  const float* rr = which == 0 ? qr : kr;
  pdl_wait();  // the norms and the key mean come from the quantize pass
  pdl_trigger();
  for (int e = threadIdx.x; e < 128 * D / 2; e += 256) {
    const int t = blk * 128 + (2 * e) / D, d = (2 * e) % D;
    __half2 h = __floats2half2_rn(0.f, 0.f);
    if (t < N) {
      const __nv_bfloat162 x2 = *reinterpret_cast<const __nv_bfloat162*>(src + ((size_t)bh * N + t) * D + d);
      float a = __low2float(x2), b = __high2float(x2);
      if (which < 2 && qk_norm) {
        const float r = rr[(size_t)bh * np + t];
        a = __fmul_rn(a, r);
        b = __fmul_rn(b, r);
      }
      if (which == 1) {
        a = __fsub_rn(a, kmean[(size_t)bh * D + d]);
        b = __fsub_rn(b, kmean[(size_t)bh * D + d + 1]);
      }
      h = __floats2half2_rn(a, b);
    }
    *reinterpret_cast<__half2*>(dst + ((size_t)bh * np + t) * D + d) = h;
  }
}

// ------------------------------------------------------- high-precision tiles
template <int D>
struct HpSmem {
  uint8_t q[128 * D * 2];     // Q16 tile (fp16 q'), 128B-swizzled K-major, 64-channel atoms
  uint8_t k[2][128 * D * 2];  // K16 tiles
  uint8_t v[2][128 * D * 2];  // V16 tiles, [64-channel atom][128 keys][128 B] (MN-major B)
  uint8_t p[128 * 128 * 2];   // P16 (fp16), [64-key atom][128 rows][128 B] (K-major A)
  uint64_t bar_q, bar_kv_full[2], bar_kv_empty[2], bar_s[2], bar_p, bar_o;
  uint32_t tmem_base;
  int abort;
};

struct HpParams {
  int N, np, nb, causal;
  float alpha;
  const uint8_t* sel;   // [BH][nb][nb]
  const float* oacc;    // [BH][np][D] unnormalised O (true units) of tiles with promoted pairs
  const float* ml;      // [BH][np][2] running maximum (log2 units) and 448 x row sum
  __nv_bfloat16* O;
  float* O32;
  float* LSE;
  int* status;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// instruction descriptor of kind::f16 with fp16 A and B, fp32 accumulator
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// One CTA per (128-query tile, head): warps 0-3 own the tile's rows (thread t = row t = TMEM
// lane t, all 128 keys of a tile), warp 4 loads tiles with TMA, warp 5 allocates TMEM and
// issues the MMAs in the order S(0) | S(i+1) PV(i) ...: S is double-buffered, so the next
// promoted tile's S runs while the softmax works on this one.  TMEM: S of tile i at
// [128 (i % 2), 128 (i % 2) + 128), O [256, 256 + D).
template <int D>
__global__ void __launch_bounds__(192, 1)
    fwd_hp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const HpParams prm) {
  extern __shared__ uint8_t smem_raw[];
  HpSmem<D>& sm = *reinterpret_cast<HpSmem<D>*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int qb = blockIdx.x, bh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint8_t* srow = prm.sel + ((size_t)bh * prm.nb + qb) * prm.nb;
  const int nJ = prm.causal ? qb + 1 : prm.nb;
  pdl_wait();  // the selection, the fp16 copies and the low-bit pass's rows
  int nhp = 0;
  for (int j = 0; j < nJ; ++j) nhp += srow[j] != 0;
  if (nhp == 0) return;  // the low-bit pass has finished this tile's rows
  constexpr uint32_t kCols = 512, cO = 256;
  if (tid == 0) {
    mbar_init(&sm.bar_q, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.bar_kv_full[s], 1);
      mbar_init(&sm.bar_kv_empty[s], 1);
      mbar_init(&sm.bar_s[s], 1);  // one phase per use of S buffer s
    }
    mbar_init(&sm.bar_p, 128);
    mbar_init(&sm.bar_o, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&sm.tmem_base, kCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  // Dependents launch only once this CTA holds its TMEM (or has exited): a later forward
  // allocates all 512 columns before it waits on its predecessors, so it must not reach
  // this SM while this CTA still waits for columns.
  pdl_trigger();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  constexpr uint32_t kTile = 128 * D * 2;
  if (warp == 4) {
    if (lane == 0) {
      // ---------------- producer: Q16 once, then K16 and V16 of each promoted tile
      mbar_arrive_expect_tx(&sm.bar_q, kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_3d(sm.q + c * 16384, &tm_q, c * 64, qb * 128, bh, &sm.bar_q);
      int i = 0;
      for (int j = 0; j < nJ; ++j) {
        if (!srow[j]) continue;
        const int s = i & 1;
        if (i >= 2 && !mbar_wait(&sm.bar_kv_empty[s], ((i >> 1) - 1) & 1, abort)) break;
        mbar_arrive_expect_tx(&sm.bar_kv_full[s], 2 * kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(sm.k[s] + c * 16384, &tm_k, c * 64, j * 128, bh, &sm.bar_kv_full[s]);
          tma_load_3d(sm.v[s] + c * 16384, &tm_v, c * 64, j * 128, bh, &sm.bar_kv_full[s]);
        }
        ++i;
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ---------------- MMA issuer: S16 of tile i + 1 as soon as its K16 is in (its S buffer
      // was freed when the softmax handed over P16 of tile i - 1, waited for below before PV16
      // of tile i - 1), then PV16 of tile i once P16 is in
      constexpr uint32_t id_s = idesc_f16(128, 128, false, false);
      constexpr uint32_t id_o = idesc_f16(128, D, false, true);
      const uint32_t a_q = smem_u32(sm.q), a_p = smem_u32(sm.p);
      auto issue_s = [&](int i) {
        const uint32_t a_k = smem_u32(sm.k[i & 1]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_bf16(tmem + (uint32_t)((i & 1) * 128), sdesc_sw128(a_q + off, 16, 1024),
                    sdesc_sw128(a_k + off, 16, 1024), id_s, kk > 0);
        }
        umma_commit(&sm.bar_s[i & 1]);
      };
      bool ok = mbar_wait(&sm.bar_q, 0, abort) && mbar_wait(&sm.bar_kv_full[0], 0, abort);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int i = 0; ok && i < nhp; ++i) {
        if (i + 1 < nhp) {
          if (!mbar_wait(&sm.bar_kv_full[(i + 1) & 1], ((i + 1) >> 1) & 1, abort)) break;
          tc_fence_after();
          issue_s(i + 1);
        }
        if (!mbar_wait(&sm.bar_p, i & 1, abort)) break;
        tc_fence_after();
        const uint32_t a_v = smem_u32(sm.v[i & 1]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + cO, sdesc_sw128(a_p + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                    sdesc_sw128(a_v + kk * 2048, 16384, 1024), id_o, 1);
        umma_commit(&sm.bar_o);
        umma_commit(&sm.bar_kv_empty[i & 1]);
      }
    }
  } else {
    // ---------------- softmax: thread t owns row t
    const int t = tid;
    const int row = qb * 128 + t;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t o_col = tmem + lane_base + cO;
    uint8_t* prow = sm.p + (t >> 3) * 1024 + (t & 7) * 128;
    const float* ml = prm.ml + ((size_t)bh * prm.np + row) * 2;
    float m = ml[0], l = ml[1];
    // the low-bit pass's unnormalised output of this row into the O columns
    {
      const float* src = prm.oacc + ((size_t)bh * prm.np + row) * D;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 f = *reinterpret_cast<const float4*>(src + c + i);
          o[i] = __float_as_uint(f.x), o[i + 1] = __float_as_uint(f.y), o[i + 2] = __float_as_uint(f.z),
          o[i + 3] = __float_as_uint(f.w);
        }
        tmem_st32(o_col + c, o);
      }
      tmem_st_wait();
    }
    tc_fence_before();
    bool ok = true;
    int i = 0;
    for (int j = 0; j < nJ; ++j) {
      if (!srow[j]) continue;
      ok = ok && mbar_wait(&sm.bar_s[i & 1], (i >> 1) & 1, abort);
      tc_fence_after();
      const uint32_t s_col = tmem + lane_base + (uint32_t)((i & 1) * 128);
      // keys [0, lim) of the tile are valid; the others become -inf (2^-inf = 0 below), on the
      // tiles that have any
      int lim = min(128, prm.N - j * 128);
      if (prm.causal && j == qb) lim = min(lim, t + 1);
      uint32_t sv[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_col + 32 * c, sv[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence32(sv[c]);
      if (__any_sync(0xffffffffu, lim < 128)) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * c + e >= lim) sv[c][e] = 0xff800000u;
      }
      // the maximum of RN(s alpha) is RN(max(s) alpha): alpha > 0 and rounding is monotone
      float a[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) a[c] = max3(a[c], __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
      const float amax = fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
      const float mx = amax == -INFINITY ? -INFINITY : __fmul_rn(amax, prm.alpha);
      const float m_new = fmaxf(m, mx);
      const float corr = (m == -INFINITY) ? 0.f : ex2f(m - m_new);
      // the previous tile's PV must be done before O is rescaled (and P16 rewritten)
      if (i > 0) {
        ok = ok && mbar_wait(&sm.bar_o, (i - 1) & 1, abort);
        tc_fence_after();
      }
      const uint64_t al2 = f2(prm.alpha, prm.alpha), nm2 = f2(-m_new, -m_new);
      uint64_t ls2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};  // two independent chains
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float t0, t1;
          f2split(ffma2(f2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), al2, nm2), t0, t1);
          const float p0 = ex2f(t0), p1 = ex2f(t1);
          ls2[(e >> 1) & 1] = fadd2(ls2[(e >> 1) & 1], f2(p0, p1));
          const __half2 h = __floats2half2_rn(p0, p1);
          w[e >> 1] = *reinterpret_cast<const uint32_t*>(&h);
        }
        // 32 keys = 64 bytes: units 4(c & 1) .. 4(c & 1) + 3 of 64-key atom c >> 1
        uint8_t* base = prow + (c >> 1) * 16384;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = 4 * (c & 1) + u;
          *reinterpret_cast<uint4*>(base + ((unit ^ (t & 7)) << 4)) =
              make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
      float la, lb;
      f2split(fadd2(ls2[0], ls2[1]), la, lb);
      l = fmaf(l, corr, 448.f * (la + lb));
      // O rescale when the maximum of any row of the warp moved (TMEM access is warp-wide)
      if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(o_col + c, o);
          tmem_wait32(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
          tmem_st32(o_col + c, o);
        }
        tmem_st_wait();
      }
      m = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.bar_p);
      ++i;
    }
    ok = ok && mbar_wait(&sm.bar_o, (nhp - 1) & 1, abort);
    tc_fence_after();
    // every lane takes part in the TMEM loads (warp-collective); rows past N store nothing
    const bool live = ok && row < prm.N;
    const float scale = 448.0f / l;
    const size_t obase = ((size_t)bh * prm.N + row) * D;
#pragma unroll 1
    for (int c = 0; c < D; c += 32) {
      uint32_t o[32];
      tmem_ld32(o_col + c, o);
      tmem_wait32(o);
      if (live) {
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(o[e]) * scale;
        uint4* dst = reinterpret_cast<uint4*>(prm.O + obase + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 u;
          __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
          for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(f[8 * q + 2 * e], f[8 * q + 2 * e + 1]);
          dst[q] = u;
        }
        if (prm.O32) {
          float4* d32 = reinterpret_cast<float4*>(prm.O32 + obase + c);
#pragma unroll
          for (int q = 0; q < 8; ++q) d32[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
        }
      }
    }
    if (live) prm.LSE[(size_t)bh * prm.N + row] = (m + (log2f(l) - kLog2_448)) * 0.69314718055994531f;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem, kCols);
  if (tid == 0 && sm.abort) atomicExch(prm.status, kDevTimeout);
}

}  // namespace

int launch_thrift_prepare(const void* Q, const void* K, const void* V, int B, int H, int N, int D, int qk_norm,
                          int causal, double budget, const void* ws, void* tws, cudaStream_t st) {
  const QuantWs QL = quant_ws_layout(B, H, N, D);
  const ThriftWs TL = thrift_ws_layout(B, H, N, D);
  const uint8_t* w = static_cast<const uint8_t*>(ws);
  uint8_t* t = static_cast<uint8_t*>(tws);
  const int BH = B * H, nb = QL.np / 128;
  auto* q = static_cast<const __nv_bfloat16*>(Q);
  auto* k = static_cast<const __nv_bfloat16*>(K);
  auto* v = static_cast<const __nv_bfloat16*>(V);
  double* qbar = reinterpret_cast<double*>(t + TL.qbar);
  double* kbar = reinterpret_cast<double*>(t + TL.kbar);
  auto* keys = reinterpret_cast<unsigned long long*>(t + TL.keys);
  uint8_t* sel = t + TL.sel;
  // the number of promoted pairs: ceil(budget x visible pairs), as a double expression
  const double vis = causal ? (double)nb * (nb + 1) / 2.0 : (double)nb * nb;
  double want = ceil(budget * vis - 1e-12);
  if (want < 0.0) want = 0.0;
  if (want > vis) want = vis;
  const int n = (int)want;
  ScopedTimer timer("thrift_prepare", st);
  if (launch_pdl(D == 128 ? thrift_means_kernel<128> : thrift_means_kernel<64>, dim3(nb, BH, 2), dim3(D), 0, st, q,
                 k, N, qbar, kbar) != cudaSuccess ||
      launch_pdl(D == 128 ? thrift_score_kernel<128> : thrift_score_kernel<64>, dim3(nb, BH), dim3(256), 0, st,
                 (const double*)qbar, (const double*)kbar, causal, keys) != cudaSuccess ||
      launch_pdl(thrift_select_kernel, dim3(BH), dim3(1024), 0, st, (const unsigned long long*)keys, nb, causal, n,
                 sel) != cudaSuccess ||
      launch_pdl(D == 128 ? thrift_prep_kernel<128> : thrift_prep_kernel<64>, dim3(nb, BH, 3), dim3(256), 0, st, q,
                 k, v, N, QL.np, qk_norm, reinterpret_cast<const float*>(w + QL.qr),
                 reinterpret_cast<const float*>(w + QL.kr), reinterpret_cast<const float*>(w + QL.kmean),
                 reinterpret_cast<__half*>(t + TL.q16), reinterpret_cast<__half*>(t + TL.k16),
                 reinterpret_cast<__half*>(t + TL.v16)) != cudaSuccess)
    return 3;
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

int launch_thrift_hp(const void* ws, const void* tws, void* O, float* LSE, float* O32, int B, int H, int N, int D,
                     int causal, float sm_scale, cudaStream_t st) {
  const QuantWs QL = quant_ws_layout(B, H, N, D);
  const ThriftWs TL = thrift_ws_layout(B, H, N, D);
  const uint8_t* t = static_cast<const uint8_t*>(tws);
  const int BH = B * H, np = QL.np, nb = np / 128;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_3d(&tq, t + TL.q16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, D, np, BH, 64, 128) ||
      !make_tmap_3d(&tk, t + TL.k16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, D, np, BH, 64, 128) ||
      !make_tmap_3d(&tv, t + TL.v16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, D, np, BH, 64, 128))
    return 3;
  HpParams p;
  p.N = N;
  p.np = np;
  p.nb = nb;
  p.causal = causal;
  p.alpha = (float)((double)sm_scale * 1.4426950408889634074);
  p.sel = t + TL.sel;
  p.oacc = reinterpret_cast<const float*>(t + TL.oacc);
  p.ml = reinterpret_cast<const float*>(t + TL.ml);
  p.O = static_cast<__nv_bfloat16*>(O);
  p.O32 = O32;
  p.LSE = LSE;
  p.status = reinterpret_cast<int*>(const_cast<uint8_t*>(static_cast<const uint8_t*>(ws)) + QL.status);
  const size_t smem = sizeof(HpSmem<128>) + 1024;
  auto kern = D == 128 ? fwd_hp_kernel<128> : fwd_hp_kernel<64>;
  const size_t sm_d = D == 128 ? smem : sizeof(HpSmem<64>) + 1024;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_d) != cudaSuccess) return 3;
  ScopedTimer timer("thrift_hp", st);
  if (launch_pdl(kern, dim3(nb, BH), dim3(192), sm_d, st, tq, tk, tv, p) != cudaSuccess) return 3;
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace sage
