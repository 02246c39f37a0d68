// Forward of SageBwd-style low-bit attention on tcgen05 tensor cores.
//
// "SageBwd: A Trainable Low-bit Attention" (euno.news summary), Methodology 1:
// QK^T and PV run quantized.  "ThriftAttention" (gist.science summary),
// Methodology step 2: FlashAttention-2 online softmax over key tiles.
//
// One CTA per (head, pair of 128-query tiles A and B); keys in 128-token tiles.
//   warps 0..15   : softmax, four warpgroups.  Warpgroup 2X + hh serves query tile X and the
//                   64-key half hh of every key tile; thread t owns query row t (TMEM lane t).
//   warp 16 lane 0: TMA producer for Q, the K tiles (bf16 containers of INT8 codes) and the
//                   V tiles (e4m3, channel-major)
//   warp 17       : TMEM allocator; lane 0 issues the UMMAs
//       S_j = Q8 K8_j^T   kind::f16 on bf16-held integers -> exact int sums in fp32
//       O  += P8_j V8_j   kind::f8f6f4 e4m3 x e4m3 -> fp32
// TMEM: S_A, S_B (128 columns each) + O_A, O_B (D columns each).  The tensor core works on one
// tile while the softmax of the other runs.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "launch.h"
#include "layout.h"
#include "ptx.cuh"
#include "timer.h"
#include "tmap.h"

namespace sage {

namespace {

constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr float kLog2_448 = 8.807354922057604f;  // log2(448)
constexpr float kLog2_2688 = 11.392317422778761f;  // log2(448 * 6)

template <int D>
struct FwdSmem {
  uint8_t q[2][128 * D * 2];        // query tiles A and B (bf16 containers of INT8 codes)
  uint8_t k[kKStages][128 * D * 2];  // key tiles
  uint8_t v[kVStages][D * 128];      // value tiles (e4m3, channel-major)
  uint8_t p[2][128 * 128];           // P of tiles A and B (e4m3, 128B-swizzled K-major)
  float xmax[2][2][128];             // per tile and key half: row maxima of the current key tile
  float xsum[2][2][128];             // per tile and key half: row sums, exchanged at the end
  // Q-smoothing: the logit terms of tiles A and B for the keys of each value stage
  __align__(16) float dsb[kVStages][2][128];
  // NVFP4: the block scales of P (per tile, one 512-byte atom per 64-key half, as the tensor
  // core reads them) and of each value stage's V tile (two atoms)
  __align__(128) uint8_t sfa[2][2][512];
  __align__(128) uint8_t sfb[kVStages][1024];
  uint64_t bar_q;
  uint64_t bar_k_full[kKStages], bar_k_empty[kKStages];
  uint64_t bar_v_full[kVStages], bar_v_empty[kVStages];
  uint64_t bar_s_full[2], bar_s_free[2], bar_p_full[2], bar_o_done[2];
  uint32_t tmem_base;
  int abort;
};

struct FwdParams {
  int N, np, nqb, npairs;
  int BH, hgroup;  // heads, and heads per CTA-order group (tile_head_order)
  int group;       // query heads per key/value head (grouped-query attention; 1 otherwise)
  float alpha;  // RN(sm_scale * log2 e)
  // 4096, passed at run time so that the band key stays one integer multiply-add (FMA pipe)
  // instead of a shift and an add on the busier ALU pipe
  uint32_t band_mult;
  const float* sq;
  const float* sk;
  const float* sv;
  const float* dsb;  // Q-smoothing: [BH][nqb][np] logit terms (nullptr without)
  // ThriftAttention: the promoted (query block, key tile) pairs [BH][nqb][nqb], skipped here;
  // query tiles with any hand their unnormalised output (true units, [BH][np][D]) and per row
  // the running maximum and 448 x the row sum ([BH][np][2]) to the high-precision pass
  const uint8_t* sel;
  float* oacc;
  float* ml;
  const float* vg;  // NVFP4: V's tensor scale per key/value head
  const uint8_t* v4sf;  // NVFP4: V's block-scale atoms [BHk][np/64][512]
  __nv_bfloat16* O;
  float* O32;
  float* LSE;
  int* status;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// The e4m3 code of x = RN(448 * RN(2^t)) flips where x crosses a rounding
// midpoint of e4m3: fp32 mantissa bit 19 set and bits 18..0 clear.  The fast
// value 448 * ex2.approx(t) is within 2 ulps of x (measured over 2^26 values of
// t in [-16, 0]), so a code is trusted unless the fast value lies within
// kBandUlps (twice that error) of such a midpoint; those few are recomputed from
// an accurate 2^t.  band_key(x) <= kBandMax marks them.  (Below 2^-6, e4m3 is
// subnormal and its midpoints are coarser; a flip there moves P by 2^-9 / 448 at most.)
constexpr uint32_t kBandUlps = 4;
constexpr uint32_t kBandC = (kBandUlps - 0x80000u) << 12;
constexpr uint32_t kBandMax = (2u * kBandUlps) << 12;
__device__ __forceinline__ uint32_t band_key(float x, uint32_t mult4096) {
  return __float_as_uint(x) * mult4096 + kBandC;
}

// Pairs of fp32 (hi + lo) as extended precision: error-free transformations of
// Knuth (two-sum) and Dekker (fast two-sum, two-product via FMA).
struct F2x {
  float h, l;
};
__device__ __forceinline__ F2x fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ F2x two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ F2x f2x_mul(F2x a, F2x b) {
  const float p = __fmul_rn(a.h, b.h);
  const float e = fmaf(a.h, b.h, -p) + fmaf(a.h, b.l, __fmul_rn(a.l, b.h));
  return fast_two_sum(p, e);
}
__device__ __forceinline__ F2x f2x_add(F2x a, F2x b) {
  const F2x s = two_sum(a.h, b.h);
  return fast_two_sum(s.h, __fadd_rn(s.l, __fadd_rn(a.l, b.l)));
}

// RN(2^t), and the e4m3 code of RN(448 * RN(2^t)).  t = n + f with n = rint(t) and |f| <= 1/2 (exact);
// 2^f = e^y, y = f ln 2, from the Taylor series of e^y to degree 12 (truncation below
// 2^-50 for |y| < 0.35): degrees 7..12 in fp32, 0..6 in fp32 pairs, so 2^f carries about
// 2^-45 relative error and its leading fp32 is RN(2^f) except within that distance of
// an fp32 midpoint.  Scaling by 2^n is exact in the normal range.
__device__ __forceinline__ float exact_pt(float t) {
  if (!(t >= -125.f)) return 0.f;  // far below anything a code can hold
  const float n = rintf(t);
  const float f = __fsub_rn(t, n);
  const float kLn2Hi = 0x1.62e430p-1f, kLn2Lo = -0x1.05c610p-29f;
  const float yh0 = __fmul_rn(f, kLn2Hi);
  const F2x y = fast_two_sum(yh0, fmaf(f, kLn2Hi, -yh0) + __fmul_rn(f, kLn2Lo));
  // 1/k! for k = 7..12 (fp32) and k = 0..6 (hi, lo)
  const float c12 = 2.0876755879584152e-09f, c11 = 2.5052107943679403e-08f, c10 = 2.755731998149713e-07f,
              c9 = 2.7557318844628753e-06f, c8 = 2.4801587642286904e-05f, c7 = 0.00019841270113829523f;
  float q = c12;
  q = fmaf(q, y.h, c11);
  q = fmaf(q, y.h, c10);
  q = fmaf(q, y.h, c9);
  q = fmaf(q, y.h, c8);
  q = fmaf(q, y.h, c7);
  const F2x c[7] = {{1.0f, 0.0f},
                    {1.0f, 0.0f},
                    {0.5f, 0.0f},
                    {0.1666666716337204f, -4.967053879312289e-09f},
                    {0.0416666679084301f, -1.2417634698280722e-09f},
                    {0.008333333767950535f, -4.34617203337595e-10f},
                    {0.0013888889225199819f, -3.3631094437103215e-11f}};
  F2x r = {q, 0.0f};
#pragma unroll
  for (int k = 6; k >= 0; --k) r = f2x_add(f2x_mul(r, y), c[k]);
  return __fmul_rn(r.h, __int_as_float(((int)n + 127) << 23));
}
__device__ __forceinline__ uint32_t exact_p_code(float t) {
  return (uint32_t)__nv_cvt_float_to_fp8(__fmul_rn(448.0f, exact_pt(t)), __NV_SATFINITE, __NV_E4M3);
}

// a[e] for a run-time e, by a tree of selects (a stays in registers)
__device__ __forceinline__ uint32_t pick32(const uint32_t (&a)[32], int e) {
  uint32_t b[16], c[8], d[4], f[2];
#pragma unroll
  for (int i = 0; i < 16; ++i) b[i] = (e & 16) ? a[i + 16] : a[i];
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = (e & 8) ? b[i + 8] : b[i];
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = (e & 4) ? c[i + 4] : c[i];
#pragma unroll
  for (int i = 0; i < 2; ++i) f[i] = (e & 2) ? d[i + 2] : d[i];
  return (e & 1) ? f[1] : f[0];
}

// Masked keys of a tile (padding, or after the query on the causal diagonal): their S values
// become -inf right after the TMEM load, so the max and exp passes need no per-element test
// (2^-inf = 0).  Columns [0, valid) of the 64 held in s stay.
__device__ __forceinline__ void mask_half(uint32_t (&s)[2][32], int valid) {
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (q * 32 + e >= valid) s[q][e] = 0xff800000u;
}

// the same for one 32-column chunk: columns [0, valid) stay
__device__ __forceinline__ void mask_chunk(uint32_t (&s)[32], int valid) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (e >= valid) s[e] = 0xff800000u;
}

// A zero logit scale (an all-zero Q or K block, so every unmasked S there is 0) becomes the
// smallest subnormal: -inf * scale stays -inf, and 0 * scale - m is still exactly -m.
__device__ __forceinline__ float logit_scale(float c) { return c > 0.f ? c : __uint_as_float(1u); }

// named barrier 1 + X over the two warpgroups of tile X
__device__ __forceinline__ void named_bar_tile(int X) { asm volatile("bar.sync %0, 256;" ::"r"(1 + X) : "memory"); }

// e2m1 codes of two values, the first in the low nibble
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(lo, hi), __NV_E2M1, cudaRoundNearest);
}

__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Softmax of one 128-query tile (tile X of the CTA) by two warpgroups: thread t of half hh
// owns query row t (TMEM lane t) and the 64 keys [64 hh, 64 hh + 64) of every key tile, which
// is exactly one K scale block.  The two halves exchange their row maxima once per tile and
// their row sums at the end; each rescales and writes half of the O columns.
// QS (Q-smoothing): the logit first takes back the query block mean's term in natural units,
// u = RN(acc RN(s_q s_k) + dsb_j), and u alpha stands where acc c stands otherwise.
// TH (ThriftAttention): the promoted key tiles of this query tile are skipped (the barriers
// count processed tiles), and a tile with any promoted pair ends with its unnormalised output.
// F4 (NVFP4 PV): P takes e2m1 codes with an e4m3 scale per 16 keys: y = RN(2688 p~),
// s = e4m3(RN(max y / 6)), code = e2m1(RN(y / s)); codes and scales near a rounding boundary
// are redone from an accurate 2^t, so they equal the exact definition.  l sums y (2688 units).
template <int D, bool CAUSAL, bool QS, bool TH, bool F4>
__device__ __forceinline__ void softmax_tile_loop(FwdSmem<D>& sm, const FwdParams& prm, int X, int hh, int qb,
                                                  int bh, uint32_t tmem, volatile int* abort) {
  constexpr int DH = D / 2;  // O columns of this half
  const int t = threadIdx.x & 127;
  const int warp_in_wg = t >> 5;
  const int row = qb * 128 + t;
  const uint32_t lane_base = (uint32_t)(warp_in_wg * 32) << 16;
  const uint32_t s_col = tmem + lane_base + (uint32_t)(X * 128 + hh * 64);
  const uint32_t o_col = tmem + lane_base + 256u + (uint32_t)(X * D + hh * DH);
  const int n_tiles = CAUSAL ? qb + 1 : prm.nqb;
  const float s_q = prm.sq[(size_t)bh * prm.nqb + qb];
  const int kvh = bh / prm.group;  // the key/value head of this query head
  const float* skh = prm.sk + (size_t)kvh * prm.nqb * 2 + hh;  // this half's K block scale
  uint8_t* prow = sm.p[X] + (t >> 3) * 1024 + (t & 7) * 128;
  float m = -INFINITY, l = 0.f;  // l: this half's share of the row sum
  // a wait that runs out raises the abort flag; from then on this thread skips its waits but
  // still runs every tile, so neither half is left behind at a named barrier
  bool ok = true;
  const uint8_t* srow = TH ? prm.sel + ((size_t)bh * prm.nqb + qb) * prm.nqb : nullptr;
  int cnt = 0;  // tiles processed (with TH the promoted ones are not)
  bool hp_any = false;
  // the K-block scale of a tile is fetched one tile early (global latency off the path)
  float sk_next = skh[0];
  for (int j = 0; j < n_tiles; ++j) {
    if constexpr (TH) {
      if (srow[j]) {
        hp_any = true;
        continue;
      }
      sk_next = skh[2 * j];
    }
    const float skj = sk_next;
    if (!TH && j + 1 < n_tiles) sk_next = skh[2 * (j + 1)];
    ok = ok && mbar_wait(&sm.bar_s_full[X], cnt & 1, abort);
    tc_fence_after();
    // with Q-smoothing the tile's logit terms travel with its value tile
    const float* brow = &sm.dsb[j % kVStages][X][hh * 64];
    if constexpr (QS) ok = ok && mbar_wait(&sm.bar_v_full[j % kVStages], (j / kVStages) & 1, abort);
    const float cc = QS ? logit_scale(__fmul_rn(s_q, skj)) : logit_scale(__fmul_rn(__fmul_rn(s_q, skj), prm.alpha));
    const int kbase = j * 128;
    const bool masked_tile = (kbase + 128 > prm.N) || (CAUSAL && j == qb);
    int lim = prm.N - kbase;  // keys [0, lim) of the tile are valid
    if (CAUSAL && j == qb) lim = min(lim, t + 1);
    // ---- max pass over this half's 64 S values (two 32-column loads)
    float mx;
    {
      uint32_t sh[2][32];
      tmem_ld32(s_col, sh[0]);
      tmem_ld32(s_col + 32, sh[1]);
      tmem_ld_wait();
      reg_fence32(sh[0]);
      reg_fence32(sh[1]);
      if (masked_tile) mask_half(sh, lim - hh * 64);
      float a[2] = {-INFINITY, -INFINITY};  // one running maximum per load: two chains
      if constexpr (QS) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 b = *reinterpret_cast<const float4*>(brow + 32 * q + e);
            const float u0 = fmaf(__uint_as_float(sh[q][e]), cc, b.x), u1 = fmaf(__uint_as_float(sh[q][e + 1]), cc, b.y);
            const float u2 = fmaf(__uint_as_float(sh[q][e + 2]), cc, b.z), u3 = fmaf(__uint_as_float(sh[q][e + 3]), cc, b.w);
            a[q] = max3(a[q], u0, u1);
            a[q] = max3(a[q], u2, u3);
          }
      } else {
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int e = 0; e < 32; e += 2) a[q] = max3(a[q], __uint_as_float(sh[q][e]), __uint_as_float(sh[q][e + 1]));
      }
      mx = fmaxf(a[0], a[1]);
    }
    // the log2-domain logit is acc * c with c > 0, so its maximum is max(acc) * c (with
    // Q-smoothing: u * alpha, alpha > 0)
    const float mt = mx == -INFINITY ? -INFINITY : __fmul_rn(mx, QS ? prm.alpha : cc);
    sm.xmax[X][hh][t] = mt;
    named_bar_tile(X);
    const float m_new = max3(m, sm.xmax[X][0][t], sm.xmax[X][1][t]);
    const float corr = (m == -INFINITY) ? 0.f : ex2(m - m_new);
    // ---- PV of the previous tile must be complete before P is overwritten and O rescaled
    // (the tensor core took it right after this tile's S, so it has normally finished by now)
    if (cnt > 0) {
      ok = ok && mbar_wait(&sm.bar_o_done[X], (cnt - 1) & 1, abort);
      tc_fence_after();
    }
    // ---- t = RN(acc*c - m_new) (one FMA), x = 448 * 2^t, e4m3 codes -> shared memory; one
    // 32-column chunk at a time (reloaded from TMEM), so few registers stay live
    if constexpr (F4) {
      // NVFP4: per 16-key block y = RN(2688 p~), s = e4m3(RN(max y / 6)), codes e2m1(RN(y / s)).
      // A scale or code whose decision a few ulps could change (checked by rounding the value
      // moved 2^-18 up and down) is redone from an accurate 2^t and a correctly rounded division.
      const uint64_t neg_m2 = f2(-m_new, -m_new), cc2 = f2(cc, cc), k2688 = f2(2688.f, 2688.f);
      constexpr float kUp = 1.0f + 0x1p-18f, kDn = 1.0f - 0x1p-18f;
      uint64_t lsum2 = f2(0.f, 0.f);
      uint32_t sfw = 0;  // this half's four block scales (e4m3), block 0 in the low byte
      // row t of the P tile: 64 bytes (128 keys), 64-byte swizzle: 16-byte unit c at c ^ ((t & 7) >> 1)
      uint8_t* prow4 = sm.p[X] + (t >> 3) * 512 + (t & 7) * 64;
#pragma unroll 1
      for (int q = 0; q < 2; ++q) {
        uint32_t sv[32];
        tmem_ld32(s_col + 32 * q, sv);
        tmem_wait32(sv);
        if (q == 1) {
          tc_fence_before();
          mbar_arrive(&sm.bar_s_free[X]);
        }
        if (masked_tile) mask_chunk(sv, lim - hh * 64 - 32 * q);
        uint32_t cw[4];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float y[16];
          float ym = 0.f;
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float t0, t1;
            f2split(ffma2(f2(__uint_as_float(sv[16 * b + e]), __uint_as_float(sv[16 * b + e + 1])), cc2, neg_m2), t0, t1);
            const uint64_t y2 = fmul2(f2(ex2(t0), ex2(t1)), k2688);
            lsum2 = fadd2(lsum2, y2);
            f2split(y2, y[e], y[e + 1]);
            ym = max3(ym, y[e], y[e + 1]);
          }
          // the fast values are within a few ulps of RN(max y / 6) and RN(y / s); the 2^-18 band
          // (32 ulps) covers the product with a rounded 1/6 and an approximate reciprocal
          float qs = ym * (1.0f / 6.0f);
          uint32_t sb = (uint32_t)__nv_cvt_float_to_fp8(qs, __NV_SATFINITE, __NV_E4M3);
          bool redo = sb != (uint32_t)__nv_cvt_float_to_fp8(qs * kUp, __NV_SATFINITE, __NV_E4M3) ||
                      sb != (uint32_t)__nv_cvt_float_to_fp8(qs * kDn, __NV_SATFINITE, __NV_E4M3);
          uint32_t w0 = 0, w1 = 0;
          float sval = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sb, __NV_E4M3)));
          if (sval > 0.f) {
            const float inv = __fdividef(1.0f, sval);
            const uint64_t inv2 = f2(inv, inv), up2 = f2(kUp, kUp), dn2 = f2(kDn, kDn);
            uint32_t diff = 0;
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const uint64_t q2 = fmul2(f2(y[e], y[e + 1]), inv2);
              float q0, q1, u0, u1, d0, d1;
              f2split(q2, q0, q1);
              f2split(fmul2(q2, up2), u0, u1);
              f2split(fmul2(q2, dn2), d0, d1);
              const uint32_t c = e2m1x2(q0, q1);
              diff |= (c ^ e2m1x2(u0, u1)) | (c ^ e2m1x2(d0, d1));
              if (e < 8) w0 |= c << (4 * e);
              else w1 |= c << (4 * (e - 8));
            }
            redo = redo || diff != 0;
          }
          if (redo) {
            // the definition itself: RN(2^t) accurately, then the correctly rounded steps
            ym = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              y[e] = __fmul_rn(2688.0f, exact_pt(fmaf(__uint_as_float(sv[16 * b + e]), cc, -m_new)));
              ym = fmaxf(ym, y[e]);
            }
            qs = __fdiv_rn(ym, 6.0f);
            sb = (uint32_t)__nv_cvt_float_to_fp8(qs, __NV_SATFINITE, __NV_E4M3);
            sval = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sb, __NV_E4M3)));
            w0 = w1 = 0;
            if (sval > 0.f) {
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                const uint32_t c = e2m1x2(__fdiv_rn(y[e], sval), __fdiv_rn(y[e + 1], sval));
                if (e < 8) w0 |= c << (4 * e);
                else w1 |= c << (4 * (e - 8));
              }
            }
          }
          cw[2 * b] = w0;
          cw[2 * b + 1] = w1;
          sfw |= sb << (8 * (2 * q + b));
        }
        const int unit = 2 * hh + q;  // 32 keys = 16 bytes
        *reinterpret_cast<uint4*>(prow4 + ((unit ^ ((t & 7) >> 1)) << 4)) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      }
      // this half's scales into its atom: row t at byte (t % 32) * 16 + (t / 32) * 4
      *reinterpret_cast<uint32_t*>(sm.sfa[X][hh] + (t & 31) * 16 + (t >> 5) * 4) = sfw;
      float la, lb;
      f2split(lsum2, la, lb);
      l = fmaf(l, corr, la + lb);
    } else {
      const uint64_t neg_m2 = f2(-m_new, -m_new);
      const uint64_t k448 = f2(448.f, 448.f);
      const uint64_t cc2 = f2(cc, cc), al2 = f2(prm.alpha, prm.alpha);
      const uint32_t bm = prm.band_mult;
      // t = RN(acc c - m) (one FMA), or RN(u alpha - m) with u = RN(acc c + dsb_e)
      auto targ = [&](uint32_t s0, uint32_t s1, int e) -> uint64_t {
        const uint64_t a2 = f2(__uint_as_float(s0), __uint_as_float(s1));
        if constexpr (QS) {
          const float2 b = *reinterpret_cast<const float2*>(brow + e);
          return ffma2(ffma2(a2, cc2, f2(b.x, b.y)), al2, neg_m2);
        } else {
          return ffma2(a2, cc2, neg_m2);
        }
      };
      uint64_t lsum[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};  // two independent chains
#pragma unroll 1
      for (int q = 0; q < 2; ++q) {
        uint32_t sv[32];
        tmem_ld32(s_col + 32 * q, sv);
        tmem_wait32(sv);
        if (masked_tile) mask_chunk(sv, lim - hh * 64 - 32 * q);
        uint32_t band[2] = {~0u, ~0u};  // smallest band keys of the chunk's codes
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float x[4];
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            float t0, t1;
            f2split(targ(sv[e + u], sv[e + u + 1], 32 * q + e + u), t0, t1);
            f2split(fmul2(f2(ex2(t0), ex2(t1)), k448), x[u], x[u + 1]);
            lsum[u >> 1] = fadd2(lsum[u >> 1], f2(x[u], x[u + 1]));
            band[u >> 1] = min(band[u >> 1], min(band_key(x[u], bm), band_key(x[u + 1], bm)));
          }
          w[e >> 2] = pack4_e4m3(x[0], x[1], x[2], x[3]);
        }
        const int c = 2 * hh + q;  // 32-key chunk of the row: 16-byte units 2c, 2c+1
        *reinterpret_cast<uint4*>(prow + (((2 * c) ^ (t & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(prow + (((2 * c + 1) ^ (t & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
        // rare: codes whose fast value is near an e4m3 midpoint are redone exactly and
        // patched in shared memory.  S stays in TMEM until this tile's P is handed over, so the
        // chunk is loaded again here and the loop above keeps no S value alive for this path
        // (the load is warp-collective: the whole warp enters when any lane needs it)
        if (__any_sync(0xffffffffu, min(band[0], band[1]) <= kBandMax)) {
          tmem_ld32(s_col + 32 * q, sv);
          tmem_wait32(sv);
          if (masked_tile) mask_chunk(sv, lim - hh * 64 - 32 * q);
          uint32_t flags = 0;
          // the fast values are recomputed with the very instruction sequence of the loop above
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float t0, t1, x0, x1;
            f2split(targ(sv[e], sv[e + 1], 32 * q + e), t0, t1);
            f2split(fmul2(f2(ex2(t0), ex2(t1)), k448), x0, x1);
            if (band_key(x0, bm) <= kBandMax) flags |= 1u << e;
            if (band_key(x1, bm) <= kBandMax) flags |= 1u << (e + 1);
          }
          while (flags) {
            const int e = __ffs(flags) - 1;
            flags &= flags - 1;
            const int byte = 32 * c + e;  // key column in the row
            const float acc = __uint_as_float(pick32(sv, e));
            const float targ1 = QS ? fmaf(fmaf(acc, cc, brow[32 * q + e]), prm.alpha, -m_new) : fmaf(acc, cc, -m_new);
            prow[((((byte >> 4) ^ (t & 7)) << 4)) | (byte & 15)] = (uint8_t)exact_p_code(targ1);
          }
        }
      }
      float la, lb;
      f2split(fadd2(lsum[0], lsum[1]), la, lb);
      l = fmaf(l, corr, la + lb);
    }
    // ---- this half's O columns are rescaled when the row maximum moved (any lane of the warp)
    if (cnt > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
      for (int c = 0; c < DH; c += 32) {
        uint32_t o[32];
        tmem_ld32(o_col + c, o);
        tmem_wait32(o);
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          f2split(fmul2(f2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), f2(corr, corr)),
                  *reinterpret_cast<float*>(&o[i]), *reinterpret_cast<float*>(&o[i + 1]));
        tmem_st32(o_col + c, o);
      }
      tmem_st_wait();
    }
    m = m_new;
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(&sm.bar_p_full[X]);
    ++cnt;
  }
  // ---- epilogue: O = A * sv / l (l sums 448 p~ over both halves), LSE = ln2 (m + log2(l / 448))
  if (cnt > 0) ok = ok && mbar_wait(&sm.bar_o_done[X], (cnt - 1) & 1, abort);
  tc_fence_after();
  sm.xsum[X][hh][t] = l;
  named_bar_tile(X);
  l = sm.xsum[X][0][t] + sm.xsum[X][1][t];  // the same order in both halves
  if (TH && hp_any) {
    // the high-precision pass finishes this tile: A sv / 448 (true units) and (m, l) of every row
    float* dst = prm.oacc + ((size_t)bh * prm.np + row) * D + hh * DH;
    const float* svh = prm.sv + (size_t)kvh * D + hh * DH;
#pragma unroll 1
    for (int c = 0; c < DH; c += 32) {
      float f[32];
      if (cnt > 0) {
        uint32_t o[32];
        tmem_ld32(o_col + c, o);
        tmem_wait32(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(o[i]) * (svh[c + i] * (1.0f / 448.0f));
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = 0.f;
      }
      float4* d4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
      for (int i = 0; i < 8; ++i) d4[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
    }
    if (hh == 0) *reinterpret_cast<float2*>(prm.ml + ((size_t)bh * prm.np + row) * 2) = make_float2(m, l);
  } else if (ok) {
    const float inv_l = 1.0f / l;
    const bool live = row < prm.N;
    const size_t obase = ((size_t)bh * prm.N + row) * D + hh * DH;
    const float* svh = prm.sv + (size_t)kvh * D + hh * DH;
    // NVFP4: the accumulator holds sum (2688 P^)(V^ / g) and l sums 2688 p~, so O = acc g / l
    const float g_l = F4 ? prm.vg[kvh] * inv_l : 0.f;
#pragma unroll 1
    for (int c = 0; c < DH; c += 32) {
      uint32_t o[32];
      tmem_ld32(o_col + c, o);
      tmem_wait32(o);
      float f[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(o[i]) * (F4 ? g_l : svh[c + i] * inv_l);
      if (live) {
        uint4* dst = reinterpret_cast<uint4*>(prm.O + obase + c);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 u;
          __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
          for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(f[8 * i + 2 * e], f[8 * i + 2 * e + 1]);
          dst[i] = u;
        }
        if (prm.O32) {
          float4* d32 = reinterpret_cast<float4*>(prm.O32 + obase + c);
#pragma unroll
          for (int i = 0; i < 8; ++i) d32[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
        }
      }
    }
    if (live && hh == 0)
      prm.LSE[(size_t)bh * prm.N + row] = (m + (log2f(l) - (F4 ? kLog2_2688 : kLog2_448))) * 0.69314718055994531f;
  }
}

// One CTA per (head, pair of 128-query blocks A = 2c, B = 2c + 1).  Warpgroups 0-1 run
// the softmax of tile A (keys [0,64) and [64,128) of each key tile), 2-3 that of tile B;
// warp 16 loads K and V tiles with TMA; warp 17 allocates TMEM and issues the UMMAs in
// the order
//   S_A(0) S_B(0) | S_A(j+1) PV_A(j) S_B(j+1) PV_B(j) ...
// (a tile's pair once its softmax has handed over P(j), and with it S(j)), so the tensor core
// works on one tile's pair while the other tile's softmax runs.  The tile's next softmax waits
// for its S; the PV behind it finishes during the max pass (o_done, waited before P is
// rewritten).  A tile's softmax keeps nothing of S for the rare exact-code path (it reloads S
// from TMEM).  Issuing S(j+1) earlier, as soon as S(j) is in registers, measured slower on
// long_32k (7.80 ms against 7.09 ms): the softmax then had to hold the S values for that path.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,256+D), O_B [256+D,256+2D).
// F4 (NVFP4 PV): PV runs as two kind::mxf4nvf4 MMAs (K = 64 keys each) on packed e2m1
// operands with a 64-byte swizzle; the scale factors of P and V go to the last 16 TMEM columns
// of the tile's S, which its softmax has finished reading, and the tile's next S waits until
// that PV has completed.
template <int D, bool CAUSAL, bool QS, bool TH, bool F4>
__global__ void __launch_bounds__(640, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams prm) {
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<D>& sm = *reinterpret_cast<FwdSmem<D>*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int px, bh;  // one CTA per (pair of query blocks, head); causal: the longest pairs first
  tile_head_order((int)blockIdx.x, prm.npairs, prm.BH, prm.hgroup, px, bh);
  const int pc = CAUSAL ? (prm.npairs - 1 - px) : px;
  const int qbA = 2 * pc, qbB = 2 * pc + 1;
  const bool hasB = qbB < prm.nqb;
  // KV tiles: tile A needs [0, lastA], tile B [0, lastB]
  const int lastA = CAUSAL ? qbA : prm.nqb - 1;
  const int lastB = hasB ? (CAUSAL ? qbB : prm.nqb - 1) : -1;
  const int n_kv = (lastB > lastA ? lastB : lastA) + 1;
  constexpr uint32_t kTmemCols = 512;

  if (tid == 0) {
    mbar_init(&sm.bar_q, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&sm.bar_k_full[s], 1);
      mbar_init(&sm.bar_k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&sm.bar_v_full[s], 1);
      mbar_init(&sm.bar_v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sm.bar_s_full[x], 1);
      mbar_init(&sm.bar_s_free[x], 256);
      mbar_init(&sm.bar_p_full[x], 256);
      mbar_init(&sm.bar_o_done[x], 1);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 17) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  pdl_wait();  // the codes and scales come from the quantize pass
  pdl_trigger();

  // the producer/MMA warpgroup needs few registers: hand them to the softmax groups
  // (launch: 96 x 640; after: 56 x 128 + 104 x 512)
  constexpr uint32_t kRegsIssue = 56, kRegsSoftmax = 104;
  static_assert(kRegsIssue * 128 + kRegsSoftmax * 512 <= 96 * 640, "register split exceeds the launch budget");
  if (warp >= 16) {
    regs_decrease<kRegsIssue>();
    if (warp == 16 && lane == 0) {
      // ---------------- producer: Q tiles once, then K and V tiles
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&sm.bar_q, (hasB ? 2 : 1) * 128 * D * 2);
  #pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sm.q[0] + c * 16384, &tm_q, c * 64, qbA * 128, bh, &sm.bar_q);
        if (hasB) tma_load_3d(sm.q[1] + c * 16384, &tm_q, c * 64, qbB * 128, bh, &sm.bar_q);
      }
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % kKStages;
        if (j >= kKStages && !mbar_wait(&sm.bar_k_empty[s], ((j / kKStages) - 1) & 1, abort)) break;
        mbar_arrive_expect_tx(&sm.bar_k_full[s], 128 * D * 2);
  #pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sm.k[s] + c * 16384, &tm_k, c * 64, j * 128, bh / prm.group, &sm.bar_k_full[s]);
        const int vs = j % kVStages;
        if (j >= kVStages && !mbar_wait(&sm.bar_v_empty[vs], ((j / kVStages) - 1) & 1, abort)) break;
        if constexpr (F4) {
          // packed e2m1 codes of V ([D][64 bytes], 64-byte swizzle) and their two scale atoms
          const int kvh = bh / prm.group;
          mbar_arrive_expect_tx(&sm.bar_v_full[vs], D * 64 + 1024);
          tma_load_3d(sm.v[vs], &tm_v, j * 64, 0, kvh, &sm.bar_v_full[vs]);
          bulk_load(sm.sfb[vs], prm.v4sf + ((size_t)kvh * (prm.np / 64) + 2 * j) * 512, 1024, &sm.bar_v_full[vs]);
        } else {
          mbar_arrive_expect_tx(&sm.bar_v_full[vs], D * 128 + (QS ? (hasB ? 1024 : 512) : 0));
          tma_load_3d(sm.v[vs], &tm_v, j * 128, 0, bh / prm.group, &sm.bar_v_full[vs]);
        }
        if constexpr (QS) {
          // the logit terms of both query tiles for this key tile
          const float* b = prm.dsb + ((size_t)bh * prm.nqb + qbA) * prm.np + j * 128;
          bulk_load(sm.dsb[vs][0], b, 512, &sm.bar_v_full[vs]);
          if (hasB) bulk_load(sm.dsb[vs][1], b + prm.np, 512, &sm.bar_v_full[vs]);
        }
      }
    } else if (warp == 17 && lane == 0) {
      // ---------------- UMMA issuer
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_e4m3(128, D);
      auto issue_s = [&](int X, int j) {
        // per 64-channel atom (16 KB) four K = 16 steps of 32 bytes
        const uint64_t a = sdesc_sw128(smem_u32(sm.q[X]), 16, 1024);
        const uint64_t b = sdesc_sw128(smem_u32(sm.k[j % kKStages]), 16, 1024);
  #pragma unroll
        for (int h = 0; h < D / 64; ++h)
          umma_bf16_x4<2, 2>(tmem + (uint32_t)(X * 128), a + 1024 * h, b + 1024 * h, idesc_s, h > 0);
        umma_commit(&sm.bar_s_full[X]);
      };
      auto issue_pv = [&](int X, int j, int first) {
        const uint32_t p_addr = smem_u32(sm.p[X]);
        const uint32_t v_addr = smem_u32(sm.v[j % kVStages]);
        if constexpr (F4) {
          // scale factors to the last 16 columns of the tile's S (P's two atoms, then V's), then
          // two K = 64 MMAs
          constexpr uint32_t idesc_f4 = idesc_nvf4(128, D);
          const uint32_t sf = tmem + (uint32_t)(X * 128) + 112u;
  #pragma unroll
          for (int h = 0; h < 2; ++h) {
            tmem_cp_32x128b_x4(sf + 4 * h, sdesc_none(smem_u32(sm.sfa[X][h]), 128, 128));
            tmem_cp_32x128b_x4(sf + 8 + 4 * h, sdesc_none(smem_u32(sm.sfb[j % kVStages] + 512 * h), 128, 128));
          }
  #pragma unroll
          for (int h = 0; h < 2; ++h)
            umma_nvf4(tmem + 256u + (uint32_t)(X * D), sdesc_sw64(p_addr + 32 * h, 16, 512),
                      sdesc_sw64(v_addr + 32 * h, 16, 512), idesc_f4, sf + 4 * h, sf + 8 + 4 * h, (!first || h > 0));
        } else {
          // four K = 32 steps of 32 bytes
          umma_f8_x4<2, 2>(tmem + 256u + (uint32_t)(X * D), sdesc_sw128(p_addr, 16, 1024), sdesc_sw128(v_addr, 16, 1024),
                           idesc_o, !first);
        }
        umma_commit(&sm.bar_o_done[X]);
      };
      // tile X takes key tile j (ThriftAttention: unless the pair is promoted); ns, np count
      // the S and PV issued per tile, which the barrier phases follow
      const uint8_t* selA = TH ? prm.sel + ((size_t)bh * prm.nqb + qbA) * prm.nqb : nullptr;
      auto use = [&](int X, int j) -> bool {
        const int last = X == 0 ? lastA : lastB;
        if (j > last) return false;
        if constexpr (TH) return selA[X * prm.nqb + j] == 0;  // tile B's row follows tile A's
        return true;
      };
      int ns[2] = {0, 0}, npv[2] = {0, 0};
      bool ok = mbar_wait(&sm.bar_q, 0, abort) && mbar_wait(&sm.bar_k_full[0], 0, abort);
      if (ok) {
        tc_fence_after();
        for (int X = 0; X < 2; ++X)
          if (use(X, 0)) {
            issue_s(X, 0);
            ++ns[X];
          }
        umma_commit(&sm.bar_k_empty[0]);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const bool nextk = j + 1 < n_kv;
        if (nextk && !mbar_wait(&sm.bar_k_full[(j + 1) % kKStages], ((j + 1) / kKStages) & 1, abort)) break;
        if (!mbar_wait(&sm.bar_v_full[j % kVStages], (j / kVStages) & 1, abort)) break;
        if constexpr (F4) {
          // per tile: its PV once the codes are in shared memory, then its next S once that PV
          // has completed (the PV reads scale factors from the S columns)
          for (int X = 0; X < 2; ++X) {
            if (!use(X, j)) continue;
            if (!mbar_wait(&sm.bar_p_full[X], npv[X] & 1, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(X, j, npv[X] == 0);
            ++npv[X];
            if (!use(X, j + 1)) continue;
            if (!mbar_wait(&sm.bar_o_done[X], (npv[X] - 1) & 1, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(X, j + 1);
            ++ns[X];
          }
        } else {
          // per tile, once its softmax has handed over P (and so is done with S): its next S,
          // then its PV behind it.  The tile's next softmax waits only for the S; the PV finishes
          // during its max pass.  The tensor core works on one tile's pair while the other tile's
          // softmax runs.
          for (int X = 0; X < 2; ++X) {
            const bool pv = use(X, j);
            if (pv) {
              if (!mbar_wait(&sm.bar_p_full[X], npv[X] & 1, abort)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (use(X, j + 1)) {
              issue_s(X, j + 1);
              ++ns[X];
            }
            if (pv) {
              issue_pv(X, j, npv[X] == 0);
              ++npv[X];
            }
          }
        }
        if (!ok) break;
        umma_commit(&sm.bar_v_empty[j % kVStages]);
        if (nextk) umma_commit(&sm.bar_k_empty[(j + 1) % kKStages]);
      }
    }
  } else {
    regs_increase<kRegsSoftmax>();
    // one call site, so the four warpgroups run (and share instruction-cache lines of) one copy
    const int X = warp >> 3, hh = (warp >> 2) & 1;
    if (X == 0 || hasB) softmax_tile_loop<D, CAUSAL, QS, TH, F4>(sm, prm, X, hh, X ? qbB : qbA, bh, tmem, abort);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 17) tmem_dealloc(tmem, kTmemCols);
  if (tid == 0 && sm.abort) atomicExch(prm.status, kDevTimeout);
}

template <int D, bool CAUSAL, bool QS, bool TH, bool F4 = false>
int launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                 int BH, cudaStream_t st) {
  // at least 120 KB so that one CTA (which takes all 512 TMEM columns) runs per SM
  const size_t smem = sizeof(FwdSmem<D>) + 1024 > 120 * 1024 ? sizeof(FwdSmem<D>) + 1024 : 120 * 1024;
  auto kern = fwd_kernel<D, CAUSAL, QS, TH, F4>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 3;
  ScopedTimer timer("fwd", st);
  if (launch_pdl(kern, dim3(p.npairs * BH), dim3(640), smem, st, tq, tk, tv, p) != cudaSuccess) return 3;
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace

int launch_fwd(const void* ws, void* O, float* LSE, float* O32, int B, int H, int N, int D, int causal,
               float sm_scale, cudaStream_t st, int Hkv, bool q_smooth, void* tws, bool fp4) {
  const QuantWs L = quant_ws_layout(B, H, N, D, Hkv, q_smooth, fp4);
  const uint8_t* w = static_cast<const uint8_t*>(ws);
  const int BH = B * H, BHk = B * (Hkv > 0 ? Hkv : H), np = L.np;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_3d(&tq, w + L.qc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, np, BH, 64, 128)) return 3;
  if (!make_tmap_3d(&tk, w + L.kc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, np, BHk, 64, 128)) return 3;
  if (!make_tmap_3d(&tv, w + L.v8t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, np, D, BHk, 128, D)) return 3;
  FwdParams p;
  p.N = N;
  p.np = np;
  p.nqb = np / 128;
  p.npairs = (p.nqb + 1) / 2;
  p.BH = BH;
  p.group = BH / BHk;
  // K codes and V codes of a head (shared by a group of query heads, which are adjacent)
  p.hgroup = l2_head_group((size_t)p.np * D * 3 / p.group, BH);
  p.alpha = (float)((double)sm_scale * 1.4426950408889634074);
  p.band_mult = 4096u;
  p.sq = reinterpret_cast<const float*>(w + L.sq);
  p.sk = reinterpret_cast<const float*>(w + L.sk);
  p.sv = reinterpret_cast<const float*>(w + L.sv);
  p.dsb = q_smooth ? reinterpret_cast<const float*>(w + L.dsb) : nullptr;
  p.O = static_cast<__nv_bfloat16*>(O);
  p.O32 = O32;
  p.LSE = LSE;
  p.status = reinterpret_cast<int*>(const_cast<uint8_t*>(w) + L.status);
  p.sel = nullptr;
  p.oacc = p.ml = nullptr;
  p.vg = reinterpret_cast<const float*>(w + L.vg);
  p.v4sf = w + L.v4sf;
  if (fp4) {
    // NVFP4 PV (plain heads); V's packed e2m1 codes [BHk][D][Np/2]
    CUtensorMap tv4;
    if (!make_tmap_3d(&tv4, w + L.v4, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, np / 2, D, BHk, 64, D,
                      CU_TENSOR_MAP_SWIZZLE_64B))
      return 3;
    if (D == 128)
      return causal ? launch_fwd_t<128, true, false, false, true>(tq, tk, tv4, p, BH, st)
                    : launch_fwd_t<128, false, false, false, true>(tq, tk, tv4, p, BH, st);
    return causal ? launch_fwd_t<64, true, false, false, true>(tq, tk, tv4, p, BH, st)
                  : launch_fwd_t<64, false, false, false, true>(tq, tk, tv4, p, BH, st);
  }
  if (tws) {
    // ThriftAttention (plain heads, no Q-smoothing): the low-bit tiles here, the promoted ones
    // in the high-precision pass that follows
    const ThriftWs T = thrift_ws_layout(B, H, N, D);
    uint8_t* t = static_cast<uint8_t*>(tws);
    p.sel = t + T.sel;
    p.oacc = reinterpret_cast<float*>(t + T.oacc);
    p.ml = reinterpret_cast<float*>(t + T.ml);
    if (D == 128)
      return causal ? launch_fwd_t<128, true, false, true>(tq, tk, tv, p, BH, st)
                    : launch_fwd_t<128, false, false, true>(tq, tk, tv, p, BH, st);
    return causal ? launch_fwd_t<64, true, false, true>(tq, tk, tv, p, BH, st)
                  : launch_fwd_t<64, false, false, true>(tq, tk, tv, p, BH, st);
  }
  if (q_smooth) {
    if (D == 128)
      return causal ? launch_fwd_t<128, true, true, false>(tq, tk, tv, p, BH, st)
                    : launch_fwd_t<128, false, true, false>(tq, tk, tv, p, BH, st);
    return causal ? launch_fwd_t<64, true, true, false>(tq, tk, tv, p, BH, st)
                  : launch_fwd_t<64, false, true, false>(tq, tk, tv, p, BH, st);
  }
  if (D == 128)
    return causal ? launch_fwd_t<128, true, false, false>(tq, tk, tv, p, BH, st)
                  : launch_fwd_t<128, false, false, false>(tq, tk, tv, p, BH, st);
  return causal ? launch_fwd_t<64, true, false, false>(tq, tk, tv, p, BH, st)
                : launch_fwd_t<64, false, false, false>(tq, tk, tv, p, BH, st);
}

}  // namespace sage
