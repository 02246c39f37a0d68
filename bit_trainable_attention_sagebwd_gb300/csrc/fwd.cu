// Forward of SageBwd-style low-bit attention on tcgen05 tensor cores.
//
// "SageBwd: A Trainable Low-bit Attention" (euno.news summary), Methodology 1:
// QK^T and PV run quantized.  "ThriftAttention" (gist.science summary),
// Methodology step 2: FlashAttention-2 online softmax over key tiles.
//
// One CTA per (head, 128-query block); keys in 128-token tiles.
//   warp 0 lane 0 : TMA producer for Q and the K tiles (bf16 containers of INT8 codes)
//   warp 2 lane 0 : TMA producer for the V tiles (e4m3, channel-major)
//   warp 1        : TMEM allocator; lane 0 issues the UMMAs
//       S_j = Q8 K8_j^T   kind::f16 on bf16-held integers -> exact int sums in fp32
//       O  += P8_j V8_j   kind::f8f6f4 e4m3 x e4m3 -> fp32
//   warps 4..7    : softmax, thread t owns query row t (TMEM lane t)
// TMEM: S double buffer (2 x 128 columns) + O (D columns).  S_{j+1} is computed
// while the softmax warps work on S_j.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "layout.h"
#include "ptx.cuh"
#include "timer.h"
#include "tmap.h"

namespace sage {

namespace {

constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr float kLog2_448 = 8.807354922057604f;  // log2(448)

template <int D>
struct FwdSmem {
  uint8_t q[128 * D * 2];
  uint8_t k[kKStages][128 * D * 2];
  uint8_t v[kVStages][D * 128];
  uint8_t p[2][128 * 128];
  uint64_t bar_q;
  uint64_t bar_k_full[kKStages], bar_k_empty[kKStages];
  uint64_t bar_v_full[kVStages], bar_v_empty[kVStages];
  uint64_t bar_s_full[2], bar_p_full[2];
  uint64_t bar_o;
  uint32_t tmem_base;
  int abort;
};

struct FwdParams {
  int N, np, nqb;
  float alpha;  // RN(sm_scale * log2 e)
  const float* sq;
  const float* sk;
  const float* sv;
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
// value 448 * ex2.approx(t) is within a few ulps of x, so a code is trusted
// unless the fast value lies within kBandUlps of such a midpoint; those few are
// recomputed with a correctly rounded exp2.  band_key(x) <= kBandMax marks them.
constexpr uint32_t kBandUlps = 16;
constexpr uint32_t kBandC = (kBandUlps - 0x80000u) << 12;
constexpr uint32_t kBandMax = (2u * kBandUlps) << 12;
__device__ __forceinline__ uint32_t band_key(float x) { return __float_as_uint(x) * 4096u + kBandC; }

// e4m3 code of RN(448 * RN(2^t)) with 2^t evaluated in fp64 and rounded once
__device__ __noinline__ uint32_t exact_p_code(float t) {
  const float pt = (float)exp2((double)t);
  return (uint32_t)__nv_cvt_float_to_fp8(__fmul_rn(448.0f, pt), __NV_SATFINITE, __NV_E4M3);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(256, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams prm) {
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<D>& sm = *reinterpret_cast<FwdSmem<D>*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.y;
  const int qb = CAUSAL ? (prm.nqb - 1 - (int)blockIdx.x) : (int)blockIdx.x;
  const int n_tiles = CAUSAL ? qb + 1 : prm.nqb;
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kOCol = 256;

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
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.bar_s_full[s], 1);
      mbar_init(&sm.bar_p_full[s], 128);
    }
    mbar_init(&sm.bar_o, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;

  if (warp == 0 && lane == 0) {
    // ---------------- producer: Q once, then K tiles
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    mbar_arrive_expect_tx(&sm.bar_q, 128 * D * 2);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) tma_load_3d(sm.q + c * 16384, &tm_q, c * 64, qb * 128, bh, &sm.bar_q);
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kKStages;
      if (j >= kKStages && !mbar_wait(&sm.bar_k_empty[s], ((j / kKStages) - 1) & 1, abort)) break;
      mbar_arrive_expect_tx(&sm.bar_k_full[s], 128 * D * 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(sm.k[s] + c * 16384, &tm_k, c * 64, j * 128, bh, &sm.bar_k_full[s]);
    }
  } else if (warp == 2 && lane == 0) {
    // ---------------- producer: V tiles
    tma_prefetch_desc(&tm_v);
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kVStages;
      if (j >= kVStages && !mbar_wait(&sm.bar_v_empty[s], ((j / kVStages) - 1) & 1, abort)) break;
      mbar_arrive_expect_tx(&sm.bar_v_full[s], D * 128);
      tma_load_3d(sm.v[s], &tm_v, j * 128, 0, bh, &sm.bar_v_full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- UMMA issuer
    constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc_o = idesc_e4m3(128, D);
    const uint32_t q_addr = smem_u32(sm.q);
    auto issue_s = [&](int j) -> bool {
      const int s = j % kKStages;
      if (!mbar_wait(&sm.bar_k_full[s], (j / kKStages) & 1, abort)) return false;
      tc_fence_after();
      const uint32_t k_addr = smem_u32(sm.k[s]);
      const uint32_t d_col = tmem + (uint32_t)((j & 1) * 128);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        umma_bf16(d_col, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024), idesc_s,
                  kk > 0);
      }
      umma_commit(&sm.bar_s_full[j & 1]);
      umma_commit(&sm.bar_k_empty[s]);
      return true;
    };
    bool ok = mbar_wait(&sm.bar_q, 0, abort) && issue_s(0);
    for (int j = 0; ok && j < n_tiles; ++j) {
      if (j + 1 < n_tiles && !issue_s(j + 1)) break;
      const int vs = j % kVStages;
      if (!mbar_wait(&sm.bar_p_full[j & 1], (j >> 1) & 1, abort)) break;
      if (!mbar_wait(&sm.bar_v_full[vs], (j / kVStages) & 1, abort)) break;
      tc_fence_after();
      const uint32_t p_addr = smem_u32(sm.p[j & 1]);
      const uint32_t v_addr = smem_u32(sm.v[vs]);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        umma_f8(tmem + kOCol, sdesc_sw128(p_addr + kk * 32, 16, 1024), sdesc_sw128(v_addr + kk * 32, 16, 1024),
                idesc_o, (j > 0 || kk > 0));
      }
      umma_commit(&sm.bar_o);
      umma_commit(&sm.bar_v_empty[vs]);
    }
  } else if (warp >= 4) {
    // ---------------- softmax: one query row per thread
    const int t = tid - 128;
    const int row = qb * 128 + t;
    const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
    const float s_q = prm.sq[(size_t)bh * prm.nqb + qb];
    const float* skh = prm.sk + (size_t)bh * prm.nqb * 2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!mbar_wait(&sm.bar_s_full[j & 1], (j >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld32(tmem + lane_base + (uint32_t)((j & 1) * 128 + c * 32),
                  *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
      tmem_ld_wait();
      const float c0 = __fmul_rn(__fmul_rn(s_q, skh[2 * j]), prm.alpha);
      const float c1 = __fmul_rn(__fmul_rn(s_q, skh[2 * j + 1]), prm.alpha);
      const int kbase = j * 128;
      // keys past the sequence end (last tile) or after the query (causal diagonal)
      const bool masked_tile = (kbase + 128 > prm.N) || (CAUSAL && j == qb);
      int lim = prm.N - kbase;  // keys [0, lim) of the tile are valid
      if (CAUSAL && j == qb) lim = min(lim, t + 1);
      float mx0 = -INFINITY, mx1 = -INFINITY;
      if (masked_tile) {
#pragma unroll
        for (int i = 0; i < 64; ++i) mx0 = fmaxf(mx0, i < lim ? s[i] : -INFINITY);
#pragma unroll
        for (int i = 64; i < 128; ++i) mx1 = fmaxf(mx1, i < lim ? s[i] : -INFINITY);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) mx0 = fmaxf(mx0, s[i]);
#pragma unroll
        for (int i = 64; i < 128; ++i) mx1 = fmaxf(mx1, s[i]);
      }
      // the log2-domain logit is acc * c with c >= 0, so its maximum is max(acc) * c
      const float mt0 = mx0 == -INFINITY ? -INFINITY : __fmul_rn(mx0, c0);
      const float mt1 = mx1 == -INFINITY ? -INFINITY : __fmul_rn(mx1, c1);
      const float m_new = fmaxf(m, fmaxf(mt0, mt1));
      const float corr = (m == -INFINITY) ? 0.f : ex2(m - m_new);
      // t = RN(acc*c - m_new) in one FMA; x = 448 * 2^t (to be rounded to e4m3)
      const float neg_m = -m_new;
      float lt = 0.f;
      uint32_t pk[32];
      uint32_t band[4] = {~0u, ~0u, ~0u, ~0u};  // per 32-key chunk: min band key
#pragma unroll
      for (int i = 0; i < 128; i += 4) {
        const float c = i < 64 ? c0 : c1;
        float p0 = ex2(fmaf(s[i], c, neg_m)) * 448.f;
        float p1 = ex2(fmaf(s[i + 1], c, neg_m)) * 448.f;
        float p2 = ex2(fmaf(s[i + 2], c, neg_m)) * 448.f;
        float p3 = ex2(fmaf(s[i + 3], c, neg_m)) * 448.f;
        if (masked_tile) {
          p0 = i < lim ? p0 : 0.f;
          p1 = i + 1 < lim ? p1 : 0.f;
          p2 = i + 2 < lim ? p2 : 0.f;
          p3 = i + 3 < lim ? p3 : 0.f;
        }
        band[i >> 5] = min(band[i >> 5], min(min(band_key(p0), band_key(p1)), min(band_key(p2), band_key(p3))));
        lt += (p0 + p1) + (p2 + p3);
        const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(p0, p1), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(p2, p3), __NV_SATFINITE, __NV_E4M3);
        pk[i >> 2] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      // rare: codes whose fast value is near an e4m3 midpoint are redone exactly
      // (S is still in TMEM: reload the flagged 32-key chunk rather than keep it live)
      if (__any_sync(0xffffffffu, min(min(band[0], band[1]), min(band[2], band[3])) <= kBandMax)) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (__any_sync(0xffffffffu, band[cc] <= kBandMax)) {
            uint32_t sr[32];
            tmem_ld32(tmem + lane_base + (uint32_t)((j & 1) * 128 + cc * 32), sr);
            tmem_ld_wait();
            if (band[cc] <= kBandMax) {
              const float c = cc < 2 ? c0 : c1;
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const int i = cc * 32 + e;
                const float tt = fmaf(__uint_as_float(sr[e]), c, neg_m);
                const float x = ex2(tt) * 448.f;
                const bool valid = !masked_tile || i < lim;
                if (valid && band_key(x) <= kBandMax) {
                  const uint32_t code = exact_p_code(tt);
                  pk[i >> 2] = (pk[i >> 2] & ~(0xffu << ((i & 3) * 8))) | (code << ((i & 3) * 8));
                }
              }
            }
          }
        }
      }
      l = fmaf(l, corr, lt);
      m = m_new;
      // P row -> shared memory, 128B-swizzled K-major layout (row t, 128 key bytes)
      uint8_t* prow = sm.p[j & 1] + (t >> 3) * 1024 + (t & 7) * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (t & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      if (j > 0) {
        // PV_{j-1} must be complete before O is rescaled (and before the P buffer
        // it read is overwritten next iteration)
        if (!mbar_wait(&sm.bar_o, (j - 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + kOCol + c, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
            tmem_st32(tmem + lane_base + kOCol + c, o);
          }
          tmem_st_wait();
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.bar_p_full[j & 1]);
    }
    // ---------------- epilogue: O = A * sv / l, LSE
    if (ok && mbar_wait(&sm.bar_o, (n_tiles - 1) & 1, abort)) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const bool live = row < prm.N;
      const size_t obase = ((size_t)bh * prm.N + row) * D;
      const float* svh = prm.sv + (size_t)bh * D;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + kOCol + c, o);
        tmem_ld_wait();
        float f[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(o[i]) * (svh[c + i] * inv_l);
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
      if (live) prm.LSE[(size_t)bh * prm.N + row] = (m + (log2f(l) - kLog2_448)) * 0.69314718055994531f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (tid == 0 && sm.abort) atomicExch(prm.status, kDevTimeout);
}

template <int D, bool CAUSAL>
int launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                 int BH, cudaStream_t st) {
  // at least 120 KB so that one CTA (which takes all 512 TMEM columns) runs per SM
  const size_t smem = sizeof(FwdSmem<D>) + 1024 > 120 * 1024 ? sizeof(FwdSmem<D>) + 1024 : 120 * 1024;
  auto kern = fwd_kernel<D, CAUSAL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 3;
  ScopedTimer timer("fwd", st);
  kern<<<dim3(p.nqb, BH), 256, smem, st>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace

int launch_fwd(const void* ws, void* O, float* LSE, float* O32, int B, int H, int N, int D, int causal,
               float sm_scale, cudaStream_t st) {
  const QuantWs L = quant_ws_layout(B, H, N, D);
  const uint8_t* w = static_cast<const uint8_t*>(ws);
  const int BH = B * H, np = L.np;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_3d(&tq, w + L.qc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, np, BH, 64, 128)) return 3;
  if (!make_tmap_3d(&tk, w + L.kc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, np, BH, 64, 128)) return 3;
  if (!make_tmap_3d(&tv, w + L.v8t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, np, D, BH, 128, D)) return 3;
  FwdParams p;
  p.N = N;
  p.np = np;
  p.nqb = np / 128;
  p.alpha = (float)((double)sm_scale * 1.4426950408889634074);
  p.sq = reinterpret_cast<const float*>(w + L.sq);
  p.sk = reinterpret_cast<const float*>(w + L.sk);
  p.sv = reinterpret_cast<const float*>(w + L.sv);
  p.O = static_cast<__nv_bfloat16*>(O);
  p.O32 = O32;
  p.LSE = LSE;
  p.status = reinterpret_cast<int*>(const_cast<uint8_t*>(w) + L.status);
  if (D == 128) return causal ? launch_fwd_t<128, true>(tq, tk, tv, p, BH, st) : launch_fwd_t<128, false>(tq, tk, tv, p, BH, st);
  return causal ? launch_fwd_t<64, true>(tq, tk, tv, p, BH, st) : launch_fwd_t<64, false>(tq, tk, tv, p, BH, st);
}

}  // namespace sage
