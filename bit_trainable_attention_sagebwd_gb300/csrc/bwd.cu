// Backward of SageBwd-style low-bit attention on tcgen05 tensor cores.
//
// "SageBwd: A Trainable Low-bit Attention" (euno.news summary), Methodology 2:
// the backward keeps the forward's quantization; only the softmax-gradient
// matmul dP = dO V^T stays in high precision (bf16 operands, fp32 accumulate).
// "Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (gist.science
// summary), Methodology, principle 1: P is recomputed from the saved LSE and
// rounded to e4m3 exactly as the forward rounds it.
//
// Kernels (all on the caller's stream):
//   bwd_pre    per (head, 128-query block): D_i = sum_d dO*O, log2(448) - LSE*log2(e)
//              (-inf on padded rows), partial channel maxima of |dO|
//   bwd_docomb per head: dO channel scales max|dO|/448
//   bwd_do8    per (head, 128-query block): e4m3 codes of dO, channel-major; zeroed dQ
//              accumulator
//   bwd_main   per (head, 128-key block), looping over query blocks:
//                S  = Q8 K8^T          kind::f16 (bf16-held INT8 codes, exact)
//                dP = dO V^T           kind::f16 (bf16)
//                P  = e4m3(448 * 2^(S2 - LSE2)) / 448;  dS = P (dP - D)
//                dV  += P8^T dO8       kind::f8f6f4, P read transposed from its query rows
//                dS  -> INT8, one scale per (128 query x 64 key) tile
//                dK_part = dS8^T Q8    kind::f16, scaled per tile, summed in registers
//                dQ_part = dS8 K8      kind::f16 per 64-key half, scaled, staged in shared
//                                      memory and added to the fp32 accumulator by TMA reduce
//              dV and dK (x sm_scale, through QK-norm) written at the end
//   bwd_dq     (bwd_dq.cu) dQ = sm_scale * acc, through QK-norm, to bf16
#include <cstddef>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "../../include/sage_attn.h"
#include "codes.cuh"
#include "kernels.h"
#include "launch.h"
#include "layout.h"
#include "ptx.cuh"
#include "stage.cuh"
#include "timer.h"
#include "tmap.h"

namespace sage {

namespace {

constexpr float kLog2_448 = 8.807354922057604f;
constexpr float kLog2_6 = 2.584962500721156f;
constexpr int kPreThreads = 256;

// e2m1 codes of two values, the first in the low nibble
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(lo, hi), __NV_E2M1, cudaRoundNearest);
}
// the eight e2m1 codes of a word (low nibble first) times the e4m3 scale sbyte
__device__ __forceinline__ void fp4_decode8(uint32_t w, uint32_t sbyte, float (&v)[8]) {
  const float s = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sbyte, __NV_E4M3)));
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((w >> (8 * b)) & 255u), __NV_E2M1);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    v[2 * b] = f.x * s;
    v[2 * b + 1] = f.y * s;
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// ------------------------------------------------------------------ bwd_pre
// O32 (fp32, the forward's output before its bf16 rounding) replaces O in D_i when it is not
// null: the high-precision auxiliary output of the Attn-QAT backward
template <int D>
__global__ void __launch_bounds__(kPreThreads) bwd_pre_kernel(const __nv_bfloat16* __restrict__ O,
                                                               const float* __restrict__ O32,
                                                               const __nv_bfloat16* __restrict__ dO,
                                                               const float* __restrict__ LSE, int N,
                                                               float* __restrict__ dvec, float* __restrict__ bias,
                                                               float* __restrict__ dopart,
                                                               float* __restrict__ dqacc, int* __restrict__ ticket) {
  constexpr int TPR = D / 8, RPP = kPreThreads / TPR, PASSES = 128 / RPP;
  const int blk = blockIdx.x, bh = blockIdx.y, nb = gridDim.x, np = nb * 128;
  const int tid = threadIdx.x, g = tid % TPR, ro = tid / TPR;
  const size_t head = (size_t)bh * N * D;
  pdl_wait();  // O and LSE come from the forward
  pdl_trigger();
  if (blk == 0 && bh == 0 && tid == 0) *ticket = 0;  // the dQ pass claims its work from it
  float am[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) am[i] = 0.f;
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int r = p * RPP + ro, t = blk * 128 + r;
    uint4 uo = make_uint4(0, 0, 0, 0), ud = make_uint4(0, 0, 0, 0);
    float4 oa = make_float4(0.f, 0.f, 0.f, 0.f), ob = oa;
    if (t < N) {
      if (O32) {
        const float4* o32 = reinterpret_cast<const float4*>(O32 + head + (size_t)t * D) + 2 * g;
        oa = __ldg(o32);
        ob = __ldg(o32 + 1);
      } else {
        uo = __ldg(reinterpret_cast<const uint4*>(O + head + (size_t)t * D) + g);
      }
      ud = __ldg(reinterpret_cast<const uint4*>(dO + head + (size_t)t * D) + g);
    }
    float o[8], d[8];
    if (O32) {
      o[0] = oa.x, o[1] = oa.y, o[2] = oa.z, o[3] = oa.w, o[4] = ob.x, o[5] = ob.y, o[6] = ob.z, o[7] = ob.w;
    } else {
      unpack8(uo, o);
    }
    unpack8(ud, d);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s = fmaf(o[i], d[i], s);
      am[i] = fmaxf(am[i], fabsf(d[i]));
    }
#pragma unroll
    for (int m = TPR / 2; m >= 1; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    if (g == 0) {
      dvec[(size_t)bh * np + t] = t < N ? s : 0.f;
      // P = 2^(S2 - LSE log2 e) is formed as 2^(S2 + bias) / 448 with bias = log2(448) - LSE log2 e;
      // padded rows get bias = -inf, hence P = 0
      bias[(size_t)bh * np + t] =
          t < N ? kLog2_448 - (float)((double)LSE[(size_t)bh * N + t] * 1.4426950408889634074) : -INFINITY;
    }
  }
  __shared__ float s_max[RPP][D];
#pragma unroll
  for (int i = 0; i < 8; ++i) s_max[ro][g * 8 + i] = am[i];
  __syncthreads();
  if (tid < D) {
    float m = 0.f;
    for (int r = 0; r < RPP; ++r) m = fmaxf(m, s_max[r][tid]);
    dopart[((size_t)bh * nb + blk) * D + tid] = m;
  }
}

// per key/value head: the channel maxima of |dO| over the blocks of its `group` query heads
// (one scale per channel for all of them: dV sums P^T dO over their tokens)
__global__ void bwd_docomb_kernel(const float* __restrict__ dopart, int D, int nb, int group,
                                  float* __restrict__ sdo) {
  const int kvh = blockIdx.x, d = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (d >= D) return;
  float m = 0.f;
  for (int b = 0; b < nb * group; ++b) m = fmaxf(m, dopart[((size_t)kvh * group * nb + b) * D + d]);
  sdo[(size_t)kvh * D + d] = m > 0.f ? __fdiv_rn(m, 448.0f) : 0.f;
}

// e4m3 codes of one 128-query block of dO with the head's channel scales, written
// channel-major [BH, D, Np]; the rows are read straight from global memory.  The block's
// columns of the dQ accumulator are zeroed here rather than in bwd_pre, whose dO reads then
// stay in L2 for this kernel.  With the query heads of a key/value head split over several
// backward CTAs (kvacc not null), the first query head of each key/value head also zeroes
// the block's rows of the dK and dV sums and the block's counter.
template <int D>
__global__ void __launch_bounds__(kPreThreads, 4) bwd_do8_kernel(const __nv_bfloat16* __restrict__ dO, int N,
                                                               const float* __restrict__ sdo, int group,
                                                               uint8_t* __restrict__ do8t, float* __restrict__ dqacc,
                                                               float* __restrict__ kvacc, int* __restrict__ kvcnt,
                                                               size_t kv_stride) {
  constexpr int TPR = D / 8;
  const int tid = threadIdx.x;
  // blocks in the reverse order of bwd_pre: the dO blocks it read last are re-read first
  const int blk = gridDim.x - 1 - blockIdx.x, bh = gridDim.y - 1 - blockIdx.y, np = gridDim.x * 128;
  const int rows = min(128, N - blk * 128);
  __shared__ __align__(16) uint8_t s8[D * 128];
  const uint4* src = reinterpret_cast<const uint4*>(dO + ((size_t)bh * N + (size_t)blk * 128) * D);
  pdl_wait();  // the channel scales come from bwd_docomb
  pdl_trigger();
  e4m3_block_codes<D, kPreThreads>(
      [&](int t, int g) { return t < rows ? __ldg(src + t * TPR + g) : make_uint4(0, 0, 0, 0); },
      sdo + (size_t)(bh / group) * D, s8, do8t + (size_t)bh * D * np + blk * 128, np);
  // zero this block's columns of the feature-major dQ accumulator [bh][d][token]
  for (int idx = tid; idx < D * 32; idx += kPreThreads) {
    const int d = idx >> 5, c = idx & 31;
    reinterpret_cast<float4*>(dqacc + ((size_t)bh * D + d) * np + blk * 128)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (kvacc != nullptr && bh % group == 0) {
    // dK sums then dV sums (kv_stride floats apart): rows [128 blk, 128 blk + 128) of the head
    const int kvh = bh / group;
    float4* a = reinterpret_cast<float4*>(kvacc + ((size_t)kvh * np + blk * 128) * D);
    float4* b = reinterpret_cast<float4*>(kvacc + kv_stride + ((size_t)kvh * np + blk * 128) * D);
    for (int idx = tid; idx < 32 * D; idx += kPreThreads) {
      a[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
      b[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid == 0) kvcnt[(size_t)kvh * (np / 128) + blk] = 0;
  }
}

// NVFP4 backward: the e4m3 codes of dO ([BH][D][Np] bytes) as bf16 values (exact), 16 per thread
__global__ void __launch_bounds__(256) do8_bf16_kernel(const uint8_t* __restrict__ do8t, size_t n16,
                                                      __nv_bfloat16* __restrict__ do16) {
  pdl_wait();  // the codes come from bwd_do8
  pdl_trigger();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 u = reinterpret_cast<const uint4*>(do8t)[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const __half2_raw h =
          __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)((w[k >> 1] >> (16 * (k & 1))) & 0xffffu), __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
      const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
      o[k] = *reinterpret_cast<const uint32_t*>(&b);
    }
    uint4* dst = reinterpret_cast<uint4*>(do16) + 2 * i;
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// ------------------------------------------------------------------ bwd_main
template <int D>
struct BwdSmem {
  uint8_t k[128 * D * 2];    // K codes of this key block (resident)
  uint8_t v[128 * D * 2];    // V bf16 of this key block (resident)
  uint8_t q[2][128 * D * 2]; // Q codes of the current and next query blocks
  // dO bf16 of the current query block; D = 64: two, by query block parity (pipelined order)
  uint8_t dob[D == 64 ? 2 : 1][128 * D * 2];
  uint8_t do8[D * 128];      // dO e4m3 codes, channel-major
  uint8_t p[128 * 128];      // P e4m3, query rows of 128 keys
  uint8_t ds[128 * 128 * 2]; // dS INT8 codes in bf16, query rows; keys [0,64) then [64,128)
  // D = 64 (pipelined order): the dQ boxes, [query block parity][group] x 16 KB, so that the dS
  // codes need not wait for the previous block's reduce to read them
  uint8_t dqst[D == 64 ? 4 * 16384 : 16];
  // Q-smoothing: bf16 ones, the B operand (16 x 16, unswizzled) of the dS column sums
  __align__(128) uint16_t ones[256];
  __align__(16) float bias[2][128];  // log2(448) - LSE_i log2(e), per Q buffer
  union {
    __align__(16) float dvec[2][128];  // D_i, per Q buffer
    __align__(16) float dsb[2][128];   // Q-smoothing: the logit terms of the block's keys (D_i then
                                       // comes from global memory)
  };
  // per query block parity and compute warp: max |448 dS| over its rows of its group's keys
  float smax[2][8];
  uint64_t bar_kv;
  uint64_t bar_q_full[2], bar_do_full[2], bar_do8_full;
  uint64_t bar_q_free[2], bar_do_free[2], bar_do8_free;
  uint64_t bar_s, bar_dp, bar_p, bar_ds[2][2], bar_dk, bar_part, bar_dk_read, bar_dq_read, bar_free_dp, bar_cs;
  uint64_t bar_dv;  // NVFP4: the dV MMA has read P^ (which shares the dS block)
  uint32_t tmem_base;
  int abort;
  int last;  // split query heads: this CTA is the last of its key block to finish
};

static_assert(sizeof(BwdSmem<128>) <= 227 * 1024, "the backward's shared memory exceeds 227 KB");
static_assert(sizeof(BwdSmem<64>) <= 227 * 1024, "the backward's shared memory exceeds 227 KB");

struct BwdParams {
  int N, np, nqb, causal, qk_norm;
  int BH, hgroup;  // key/value heads, and heads per CTA-order group (tile_head_order)
  int group;       // query heads per key/value head (grouped-query attention; 1 otherwise)
  float alpha, sm_scale;
  const float* sq;
  const float* sk;
  const float* sdo;
  const float* bias;
  const float* dvec;
  const float* dsb;    // Q-smoothing: [BH query heads][nqb][np] logit terms (nullptr without)
  const float* qmean;  // Q-smoothing: [BH query heads][nqb][D] query block means
  // grouped heads: the query heads of a key/value head are split over `split` CTAs per key
  // block, which add dK and dV into fp32 sums [BH][np][D]; the last to count finishes them
  int split;
  float* dkacc;
  float* dvacc;
  int* kvcnt;
  const __nv_bfloat16* K;
  const float* kr;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  int* status;
};

// named barrier 1 over both compute warpgroups
__device__ __forceinline__ void named_bar_compute() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// named barrier 2 + g over compute warpgroup g
__device__ __forceinline__ void named_bar_group(int g) {
  asm volatile("bar.sync %0, 128;" ::"r"(2 + g) : "memory");
}

constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23: x + M - M rounds x to an integer (ties to even)

// One CTA per (key/value head, 128-key block), looping over the query blocks that see it: of
// every query head of the group that shares the key/value head (one query head without
// grouped-query attention).
//   warps 0-7 : two compute warpgroups.  In the P and dS phases thread t of group g owns query
//               row t (TMEM lane t of S and dP) and the keys of K block g (columns [64g, 64g+64)):
//               the row's LSE and D_i are then scalars, and each group's dS tile (128 queries x
//               64 keys) is quantized with its own scale.  In the epilogues thread t reads TMEM
//               lane t of dK_part and dV (key row t) or of dQ (query row t), output columns
//               [DG*g, DG*g + DG) (DG = D/2).
//   warp 8 lane 0: TMA producer;  warp 9: TMEM allocator, lane 0 issues UMMAs.
// TMEM columns: [0,128) S, then dK_part; [128,256) dP, then dQ of keys [64,128);
// [256,256+D) dV; [384,384+D) dQ of keys [0,64).  At D = 64 (plain e4m3 path) dK_part and the
// dQ of keys [64,128) take the free columns [320,384) and [448,512) instead, so that S and dP
// of the next query block can go in while this one's parts wait for their readout: the compute
// warps then run P of block s + 1 between the dS codes of block s and its readouts (PIPE).
// dQ staging: each group writes its scaled dQ part as [32 features][128 queries] fp32
// boxes (16 KB) into shared memory the next MMAs do not read (its own dS block, then half
// of the Q buffer just consumed); one thread per group adds them to the feature-major
// accumulator with TMA reduce and, once the boxes are read, frees the Q buffer.
// QS (Q-smoothing): the logit is u = RN(acc RN(s_q s_k) + dsb_j) and P = 2^(u alpha + bias);
// the dS codes' column sums (an extra MMA against ones into TMEM columns [128,144), read
// before dQ1 overwrites them) give dK its term s_dS (sum_i dS8_ij) qmean_I.
// F4 (NVFP4): P^ is recomputed in NVFP4 per 16-key block, y = 2688 P, s = e4m3(max y / 6),
// code = e2m1(y / s); dS = P^ (dP - D) and dV = P^T dO8 use it, dV on bf16 tensor cores
// (code s and the e4m3 codes of dO are exact in bf16; P^'s scales run along the keys, which
// dV does not contract).  P^ (bf16) is written into the dS block, which the dS codes take
// over once the dV MMA has read it; dO's codes come as bf16 in the dO8 and P regions.
template <int D, bool QS, bool F4>
__global__ void __launch_bounds__(384, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_do8, const __grid_constant__ CUtensorMap tm_dq,
                    const BwdParams prm) {
  // the tile buffers need 1024-byte alignment (128-byte swizzle atoms); the layout
  // fills almost all of the 227 KB, so the base is used as is and checked
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicExch(prm.status, kDevSetup);
    return;
  }
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(smem_raw);
  constexpr int DG = D / 2;  // output columns per compute thread
  constexpr int WPROD = 8, WMMA = 9;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int kb, bh;  // one CTA per (key block, key/value head, share of its query heads)
  const int tile = (int)blockIdx.x / prm.split, sp = (int)blockIdx.x - tile * prm.split;
  tile_head_order(tile, prm.nqb, prm.BH, prm.hgroup, kb, bh);
  const int I0 = prm.causal ? kb : 0;
  // iteration it: query block I0 + it % nq of query head qh0 + it / nq (grouped-query
  // attention: every query head of the group sees this key block; this CTA takes gs of them)
  const int nq = prm.nqb - I0;
  const int gs = prm.group / prm.split;
  const int qh0 = bh * prm.group + sp * gs;
  const int n_it = gs * nq;
  // D = 64 without Q-smoothing or NVFP4: the software-pipelined order (dK, dQ and dP in TMEM
  // columns of their own)
  constexpr bool PIPE = D == 64 && !QS && !F4;
  constexpr uint32_t kCols = 512;
  // TMEM column bases
  constexpr uint32_t cS = 0, cDP = 128, cDV = 256, cDQ0 = 384;
  constexpr uint32_t cDK = PIPE ? 320 : cS, cDQ1 = PIPE ? 448 : cDP;
  static_assert(!PIPE || cDQ1 + D <= kCols, "the pipelined TMEM layout exceeds 512 columns");
  constexpr uint32_t kTile = 128 * D * 2;

  if (tid == 0) {
    mbar_init(&sm.bar_kv, 1);
    mbar_init(&sm.bar_q_full[0], 1);
    mbar_init(&sm.bar_q_full[1], 1);
    mbar_init(&sm.bar_do_full[0], 1);
    mbar_init(&sm.bar_do_full[1], 1);
    mbar_init(&sm.bar_do8_full, 1);
    // one arrival per group once its dQ boxes are read; PIPE: the dK MMA's commit (no dQ box
    // goes into a Q buffer at D = 64)
    mbar_init(&sm.bar_q_free[0], PIPE ? 1 : 2);
    mbar_init(&sm.bar_q_free[1], PIPE ? 1 : 2);
    mbar_init(&sm.bar_do_free[0], 1);
    mbar_init(&sm.bar_do_free[1], 1);
    mbar_init(&sm.bar_do8_free, 1);
    mbar_init(&sm.bar_s, 1);
    mbar_init(&sm.bar_dp, 1);
    mbar_init(&sm.bar_p, 256);
    mbar_init(&sm.bar_ds[0][0], 128);  // [query block parity][group]: the group's dS codes are in
    mbar_init(&sm.bar_ds[0][1], 128);
    mbar_init(&sm.bar_ds[1][0], 128);
    mbar_init(&sm.bar_ds[1][1], 128);
    mbar_init(&sm.bar_dk, 1);
    mbar_init(&sm.bar_part, 1);
    mbar_init(&sm.bar_dk_read, 256);
    mbar_init(&sm.bar_dq_read, 256);
    mbar_init(&sm.bar_free_dp, 256);
    mbar_init(&sm.bar_cs, 256);
    mbar_init(&sm.bar_dv, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (QS && tid < 128) {
    reinterpret_cast<uint32_t*>(sm.ones)[tid] = 0x3f803f80u;  // bf16 1.0, 1.0
    fence_proxy_async_smem();  // read by the tensor core
  }
  if (warp == WMMA) {
    tmem_alloc(&sm.tmem_base, kCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  pdl_wait();  // dO codes, scales and the zeroed accumulator come from the preparation
  pdl_trigger();
  // the producer/MMA warpgroup needs few registers: hand them to the compute groups
  // (launch: 168 x 384; after: 80 x 128 + 208 x 256)
  constexpr uint32_t kRegsIssue = 80, kRegsCompute = 208;
  static_assert(kRegsIssue + 2 * kRegsCompute <= 3 * 168, "register split exceeds the launch budget");

  if (warp >= 8) {
    regs_decrease<kRegsIssue>();
    if (warp == WPROD && lane == 0) {
      // ---------------- producer
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_do8);
      tma_prefetch_desc(&tm_dq);
      mbar_arrive_expect_tx(&sm.bar_kv, 2 * kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sm.k + c * 16384, &tm_k, c * 64, kb * 128, bh, &sm.bar_kv);
        tma_load_3d(sm.v + c * 16384, &tm_v, c * 64, kb * 128, bh, &sm.bar_kv);
      }
      auto load_do = [&](int b, int I, int qh) {
        mbar_arrive_expect_tx(&sm.bar_do_full[b], kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sm.dob[b] + c * 16384, &tm_do, c * 64, I * 128, qh, &sm.bar_do_full[b]);
      };
      auto load_do8 = [&](int I, int qh) {
        if constexpr (F4) {
          // the e4m3 codes of dO as bf16, channel-major, in two 64-query boxes
          mbar_arrive_expect_tx(&sm.bar_do8_full, D * 256);
          tma_load_3d(sm.do8, &tm_do8, I * 128, 0, qh, &sm.bar_do8_full);
          tma_load_3d(sm.do8 + D * 128, &tm_do8, I * 128 + 64, 0, qh, &sm.bar_do8_full);
        } else {
          mbar_arrive_expect_tx(&sm.bar_do8_full, D * 128);
          tma_load_3d(sm.do8, &tm_do8, I * 128, 0, qh, &sm.bar_do8_full);
        }
      };
      auto load_q = [&](int qs, int I, int qh) {
        mbar_arrive_expect_tx(&sm.bar_q_full[qs], kTile + 1024);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sm.q[qs] + c * 16384, &tm_q, c * 64, I * 128, qh, &sm.bar_q_full[qs]);
        // the query block's bias and D_i rows (with Q-smoothing: its logit terms for this key
        // block) travel with its Q tile
        bulk_load(sm.bias[qs], prm.bias + (size_t)qh * prm.np + I * 128, 512, &sm.bar_q_full[qs]);
        if constexpr (QS)
          bulk_load(sm.dsb[qs], prm.dsb + ((size_t)qh * prm.nqb + I) * prm.np + kb * 128, 512, &sm.bar_q_full[qs]);
        else
          bulk_load(sm.dvec[qs], prm.dvec + (size_t)qh * prm.np + I * 128, 512, &sm.bar_q_full[qs]);
      };
      if constexpr (PIPE) {
        // S(it + 1) goes in early in block it, so Q(it + 1) comes first: as soon as the dK MMA
        // of block it - 1 has read its buffer; then dO of block it + 1 (once dP(it - 1) has read
        // its buffer) and its codes (once dV(it) has read theirs)
        load_q(0, I0, qh0);
        load_do(0, I0, qh0);
        load_do8(I0, qh0);
        // (query block I, query head qh) of block j + 1, advanced without a division
        int I = I0, qh = qh0;
        for (int j = 0; j + 1 < n_it; ++j) {
          if (I + 1 < prm.nqb) {
            ++I;
          } else {
            I = I0;
            ++qh;
          }
          const int q = j + 1;
          if (q > 1 && !mbar_wait(&sm.bar_q_free[q & 1], ((q >> 1) - 1) & 1, abort)) break;
          load_q(q & 1, I, qh);
          if (q > 1 && !mbar_wait(&sm.bar_do_free[q & 1], ((q >> 1) - 1) & 1, abort)) break;
          load_do(q & 1, I, qh);
          if (!mbar_wait(&sm.bar_do8_free, j & 1, abort)) break;
          load_do8(I, qh);
        }
      } else {
        // (query block I, query head qh) of iteration it, advanced without a division
        for (int it = 0, I = I0, qh = qh0; it < n_it; ++it, I = I + 1 < prm.nqb ? I + 1 : I0,
                 qh = I == I0 ? qh + 1 : qh) {
          if (it > 0 && !mbar_wait(&sm.bar_do_free[0], (it - 1) & 1, abort)) break;
          load_do(0, I, qh);
          if (it > 0 && !mbar_wait(&sm.bar_do8_free, (it - 1) & 1, abort)) break;
          load_do8(I, qh);
          const int qs = it & 1;
          if (it > 1 && !mbar_wait(&sm.bar_q_free[qs], ((it >> 1) - 1) & 1, abort)) break;
          load_q(qs, I, qh);
        }
      }
    } else if (warp == WMMA && lane == 0) {
      // ---------------- UMMA issuer
      constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);  // S = Q K^T, dP = dO V^T
      constexpr uint32_t id_dv = idesc_e4m3(128, D, true);            // dV = P^T dO8: A from query rows
      constexpr uint32_t id_dk = idesc_bf16(128, D, true, true);      // dK = dS^T Q: A from query rows
      constexpr uint32_t id_dq = idesc_bf16(128, D, false, true);     // dQ = dS K: B from key rows
      constexpr uint32_t id_cs = idesc_bf16(128, 16, true, false);    // dS^T ones: column sums
      const uint32_t a_k = smem_u32(sm.k), a_v = smem_u32(sm.v);
      const uint32_t a_do8 = smem_u32(sm.do8), a_p = smem_u32(sm.p), a_ds = smem_u32(sm.ds);
      // S(it) = Q(it) K^T
      auto issue_s = [&](int it) {
        const uint32_t a_q = smem_u32(sm.q[it & 1]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_bf16(tmem + cS, sdesc_sw128(a_q + off, 16, 1024), sdesc_sw128(a_k + off, 16, 1024), id_s, kk > 0);
        }
        umma_commit(&sm.bar_s);
      };
      // dP(it) = dO(it) V^T; dO's bf16 buffer is free once it completes
      auto issue_dp = [&](int it) {
        const int b = PIPE ? it & 1 : 0;
        const uint32_t a_do = smem_u32(sm.dob[b]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_bf16(tmem + cDP, sdesc_sw128(a_do + off, 16, 1024), sdesc_sw128(a_v + off, 16, 1024), id_s,
                    kk > 0);
        }
        umma_commit(&sm.bar_dp);
        umma_commit(&sm.bar_do_free[b]);
      };
      // dV += P^T dO8; dO's codes are free once it completes
      auto issue_dv = [&](int it) {
        if constexpr (F4) {
          // dV[key, d] += sum_q (2688 P^)[q, key] dO8[q, d] on bf16: A read MN-major from the query
          // rows of the dS block, B = dO8 codes K-major in two 64-query atoms; 16 queries per step
          constexpr uint32_t id_dv16 = idesc_bf16(128, D, true, false);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16(tmem + cDV, sdesc_sw128(a_ds + kk * 2048, 16384, 1024),
                      sdesc_sw128(a_do8 + (kk >> 2) * (D * 128) + (kk & 3) * 32, 16, 1024), id_dv16,
                      (it > 0 || kk > 0));
          umma_commit(&sm.bar_dv);
        } else {
          // dV[key, d] += sum_q P[q, key] dO8[q, d]: 32 query rows per step
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f8(tmem + cDV, sdesc_sw128(a_p + kk * 4096, 16384, 1024), sdesc_sw128(a_do8 + kk * 32, 16, 1024),
                    id_dv, (it > 0 || kk > 0));
        }
        umma_commit(&sm.bar_do8_free);
      };
      // dK part, then dQ of keys [0,64) and [64,128), once both groups' dS codes are in: dK
      // first, so that its readout starts as early as possible
      auto issue_dk_dq = [&](int it) -> bool {
        const uint32_t a_q = smem_u32(sm.q[it & 1]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + cDK, sdesc_sw128(a_ds + kk * 2048, 16384, 1024), sdesc_sw128(a_q + kk * 2048, 16384, 1024),
                    id_dk, kk > 0);
        if constexpr (QS) {
          // column sums of the dS codes (exact integers) into the dP columns, which are free
          // until dQ1: 16 identical columns, every step reads the same 16 x 16 ones
          const uint64_t b1 = sdesc_none(smem_u32(sm.ones), 128, 256);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16(tmem + cDQ1, sdesc_sw128(a_ds + kk * 2048, 16384, 1024), b1, id_cs, kk > 0);
        }
        umma_commit(&sm.bar_dk);
        if constexpr (PIPE) umma_commit(&sm.bar_q_free[it & 1]);  // dK was Q(it)'s last reader
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem + cDQ0, sdesc_sw128(a_ds + kk * 32, 16, 1024), sdesc_sw128(a_k + kk * 2048, 16384, 1024),
                    id_dq, kk > 0);
        if constexpr (QS) {
          if (!mbar_wait(&sm.bar_cs, it & 1, abort)) return false;  // the column sums are read
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem + cDQ1, sdesc_sw128(a_ds + 16384 + kk * 32, 16, 1024),
                    sdesc_sw128(a_k + 8192 + kk * 2048, 16384, 1024), id_dq, kk > 0);
        umma_commit(&sm.bar_part);
        return true;
      };
      bool ok = mbar_wait(&sm.bar_kv, 0, abort);
      if constexpr (PIPE) {
        // S(it + 1) goes in once P(it) has read S(it), and dP(it + 1) once dS(it) has read dP(it),
        // both while the compute warps still work on block it.  A group is then at most one dS
        // phase ahead of the other's readout: the tile maxima and the dS barriers it reads there
        // are kept per query block parity.
        ok = ok && mbar_wait(&sm.bar_q_full[0], 0, abort) && mbar_wait(&sm.bar_do_full[0], 0, abort);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          issue_dp(0);
        }
        for (int it = 0; ok && it < n_it; ++it) {
          const uint32_t ph = it & 1;
          const bool more = it + 1 < n_it;
          if (!mbar_wait(&sm.bar_p, ph, abort) || !mbar_wait(&sm.bar_do8_full, ph, abort)) break;
          tc_fence_after();
          // dV(it) before the wait for Q(it + 1): the producer loads that only after dO's codes
          // of block it have been read
          issue_dv(it);
          if (more) {
            if (!mbar_wait(&sm.bar_q_full[(it + 1) & 1], ((it + 1) >> 1) & 1, abort)) break;
            tc_fence_after();
            issue_s(it + 1);
          }
          if (!mbar_wait(&sm.bar_ds[ph][0], (it >> 1) & 1, abort) || !mbar_wait(&sm.bar_ds[ph][1], (it >> 1) & 1, abort))
            break;
          // the parts of block it - 1 have been read out of their columns
          if (it > 0 && (!mbar_wait(&sm.bar_dk_read, (it - 1) & 1, abort) ||
                         !mbar_wait(&sm.bar_dq_read, (it - 1) & 1, abort)))
            break;
          tc_fence_after();
          if (!issue_dk_dq(it)) break;
          if (more) {
            if (!mbar_wait(&sm.bar_do_full[(it + 1) & 1], ((it + 1) >> 1) & 1, abort) ||
                !mbar_wait(&sm.bar_free_dp, ph, abort))
              break;
            tc_fence_after();
            issue_dp(it + 1);
          }
        }
      } else {
        for (int it = 0; ok && it < n_it; ++it) {
          const uint32_t ph = it & 1;
          // S(it) goes in as soon as the previous dK part has been read out of its columns,
          // dP(it) once the previous dQ halves have been read: both overlap the compute
          // warps' work on iteration it - 1
          if (!mbar_wait(&sm.bar_q_full[it & 1], (it >> 1) & 1, abort)) break;
          if (it > 0 && !mbar_wait(&sm.bar_dk_read, (it - 1) & 1, abort)) break;
          tc_fence_after();
          issue_s(it);
          if (!mbar_wait(&sm.bar_do_full[0], ph, abort)) break;
          if (it > 0 && !mbar_wait(&sm.bar_free_dp, (it - 1) & 1, abort)) break;
          tc_fence_after();
          issue_dp(it);
          if (!mbar_wait(&sm.bar_p, ph, abort) || !mbar_wait(&sm.bar_do8_full, ph, abort)) break;
          tc_fence_after();
          issue_dv(it);
          if (!mbar_wait(&sm.bar_ds[ph][0], (it >> 1) & 1, abort) || !mbar_wait(&sm.bar_ds[ph][1], (it >> 1) & 1, abort))
            break;
          tc_fence_after();
          if (!issue_dk_dq(it)) break;
        }
      }
    }
  } else {
    regs_increase<kRegsCompute>();
    // ---------------- compute: group g, thread t
    const int g = warp >> 2;
    const int t = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int key = kb * 128 + t;  // key row of the epilogues
    const bool key_ok = key < prm.N;
    const float* skh = prm.sk + (size_t)bh * prm.nqb * 2;
    const float sk0 = skh[2 * kb], sk1 = skh[2 * kb + 1];
    const float sk_mine = g ? sk1 : sk0;  // scale of this group's 64-key block
    const uint32_t kcol = (uint32_t)(64 * g);  // first key column of this group
    const uint32_t dcol = (uint32_t)(DG * g);
    // P row t: keys [64g, 64g + 64) are 16-byte units 4g .. 4g+3 of the 128-byte row
    uint8_t* prow = sm.p + (t >> 3) * 1024 + (t & 7) * 128;
    // dS row t of this group's 64-key block: 128 bytes, units 0..7
    uint8_t* dsrow = sm.ds + g * 16384 + (t >> 3) * 1024 + (t & 7) * 128;
    // keys of this block that exist: columns kc >= klim_pad are padding
    const int klim_pad = min(128, prm.N - kb * 128);
    float dk[DG];
#pragma unroll
    for (int d = 0; d < DG; ++d) dk[d] = 0.f;
    int pending_qs = -1;  // Q buffer whose dQ boxes are still being read by TMA (elected thread)
    // a wait that times out raises the abort flag; from then on this thread skips its waits
    // but still runs every iteration, so no thread is left behind at a named barrier
    bool ok = true;
    // one query block of the loop: iteration it, query block I of query head qh, the block's
    // Q scale and (with Q-smoothing) this row's D_i, both fetched an iteration early
    struct Blk {
      int it, I, qh;
      float sqI, dvec;
    };
    int cur_I = I0, cur_qh = qh0, taken = 0;
    float sq_next = prm.sq[(size_t)qh0 * prm.nqb + I0];
    float dvec_next = QS ? prm.dvec[(size_t)qh0 * prm.np + I0 * 128 + t] : 0.f;
    // the next block in loop order; (I, qh) advance without a division
    auto take = [&]() -> Blk {
      const Blk b{taken, cur_I, cur_qh, sq_next, dvec_next};
      ++taken;
      if (cur_I + 1 < prm.nqb) {
        ++cur_I;
      } else {
        cur_I = I0;
        ++cur_qh;
      }
      if (taken < n_it) {
        sq_next = prm.sq[(size_t)cur_qh * prm.nqb + cur_I];
        if (QS) dvec_next = prm.dvec[(size_t)cur_qh * prm.np + cur_I * 128 + t];
      }
      return b;
    };
    // P's codes of the block between its P and dS phases: e4m3 (pw), or NVFP4 (pf, psc)
    uint32_t pw[2][8];
    uint32_t pf[F4 ? 8 : 1];  // NVFP4: the 64 keys' e2m1 codes, key 8i + k at nibble k of pf[i]
    uint32_t psc = 0;         // NVFP4: the four 16-key blocks' e4m3 scales, block 0 low
    float ca = 0.f, cb = 0.f;  // dQ factors of keys [0,64) and [64,128), from the dK readout
    // ---- P = e4m3(448 * 2^(S2 - LSE2)) on this row's 64 keys of block b, 32 per chunk.  The
    // codes go to shared memory for the dV MMA and stay in registers for dS.
    auto p_phase = [&](const Blk& b) {
      const int qs = b.it & 1;
      ok = ok && mbar_wait(&sm.bar_q_full[qs], (b.it >> 1) & 1, abort);
      // this query row's scalars: P = 2^(S2 - LSE2) is formed as 2^(S2 + bias) / 448
      const float bias_t = sm.bias[qs][t];
      // a zero logit scale (all-zero Q or K block: every unmasked S there is 0) becomes the
      // smallest subnormal, so that a masked -inf times it stays -inf.  With Q-smoothing the
      // scale leaves alpha out: it multiplies u = acc c + dsb.
      const float cs_raw = QS ? __fmul_rn(b.sqI, sk_mine) : __fmul_rn(__fmul_rn(b.sqI, sk_mine), prm.alpha);
      const float cs = cs_raw > 0.f ? cs_raw : __uint_as_float(1u);
      // masked key columns kc >= klim: padding, and keys after this query on the diagonal block
      const int klim = (prm.causal && b.I == kb) ? min(klim_pad, t + 1) : klim_pad;
      const bool any_mask = __any_sync(0xffffffffu, klim < (int)kcol + 64);
      ok = ok && mbar_wait(&sm.bar_s, b.it & 1, abort);
      tc_fence_after();
      uint32_t buf[2][32];
      psc = 0;
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld32(tmem + lane_base + cS + kcol + 32 * c, buf[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 2; ++c) reg_fence32(buf[c]);
      if (any_mask) {
        // masked keys: S = -inf, so 2^(S2 + bias) = 0 without a test per element below
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if ((int)kcol + 32 * c + e >= klim) buf[c][e] = 0xff800000u;
      }
      {
        const uint64_t cs2 = f2(cs, cs), b2 = f2(bias_t, bias_t), al2 = f2(prm.alpha, prm.alpha);
        const float* drow = &sm.dsb[qs][kcol];  // Q-smoothing: this group's 64 keys
        // exponent of 448 P: acc cs + bias, or (acc cs + dsb) alpha + bias
        auto arg = [&](uint32_t s0, uint32_t s1, int e) -> uint64_t {
          const uint64_t a2 = f2(__uint_as_float(s0), __uint_as_float(s1));
          if constexpr (QS) {
            const float2 d = *reinterpret_cast<const float2*>(drow + e);
            return ffma2(ffma2(a2, cs2, f2(d.x, d.y)), al2, b2);
          } else {
            return ffma2(a2, cs2, b2);
          }
        };
        if constexpr (F4) {
          // NVFP4 P^ per 16-key block: y = 2688 P (the exponent takes log2 6 more), codes e2m1(y / s)
          // with s = e4m3(max y / 6); the codes and the four scales stay in registers for dS
          const uint64_t b6 = f2(kLog2_6, kLog2_6);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              float y[16];
              float ym = 0.f;
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                float z0, z1;
                f2split(fadd2(arg(buf[c][16 * b + e], buf[c][16 * b + e + 1], 32 * c + 16 * b + e), b6), z0, z1);
                y[e] = ex2(z0);
                y[e + 1] = ex2(z1);
                ym = max3(ym, y[e], y[e + 1]);
              }
              const uint32_t sb = (uint32_t)__nv_cvt_float_to_fp8(ym * (1.0f / 6.0f), __NV_SATFINITE, __NV_E4M3);
              const float sval = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sb, __NV_E4M3)));
              uint32_t w0 = 0, w1 = 0;
              if (sval > 0.f) {
                const float inv = 1.0f / sval;
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                  const uint32_t cd = e2m1x2(y[e] * inv, y[e + 1] * inv);
                  if (e < 8) w0 |= cd << (4 * e);
                  else w1 |= cd << (4 * (e - 8));
                }
              }
              pf[4 * c + 2 * b] = w0;
              pf[4 * c + 2 * b + 1] = w1;
              psc |= sb << (8 * (2 * c + b));
            }
          }
          // P^ (2688 units, bf16) into this group's dS block: the previous iteration's dQ boxes
          // there must have been read first
          if (t == 0 && pending_qs >= 0) {
            bulk_wait_read_all();
            mbar_arrive(&sm.bar_q_free[pending_qs]);
            pending_qs = -1;
          }
          named_bar_group(g);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float v[8];
              fp4_decode8(pf[4 * c + u], psc >> (8 * (2 * c + (u >> 1))) & 255u, v);
              uint32_t h[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 hv = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                h[e] = *reinterpret_cast<const uint32_t*>(&hv);
              }
              *reinterpret_cast<uint4*>(dsrow + (((4 * c + u) ^ (t & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
            }
          }
        } else {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            float p[4];
            f2split(arg(buf[c][e], buf[c][e + 1], 32 * c + e), p[0], p[1]);
            f2split(arg(buf[c][e + 2], buf[c][e + 3], 32 * c + e + 2), p[2], p[3]);
#pragma unroll
            for (int u = 0; u < 4; ++u) p[u] = ex2(p[u]);
            const __nv_fp8x2_storage_t lo =
                __nv_cvt_float2_to_fp8x2(make_float2(p[0], p[1]), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi =
                __nv_cvt_float2_to_fp8x2(make_float2(p[2], p[3]), __NV_SATFINITE, __NV_E4M3);
            pw[c][e >> 2] = (uint32_t)lo | ((uint32_t)hi << 16);
          }
          const int u0 = 4 * g + 2 * c;
          *reinterpret_cast<uint4*>(prow + ((u0 ^ (t & 7)) << 4)) =
              make_uint4(pw[c][0], pw[c][1], pw[c][2], pw[c][3]);
          *reinterpret_cast<uint4*>(prow + (((u0 + 1) ^ (t & 7)) << 4)) =
              make_uint4(pw[c][4], pw[c][5], pw[c][6], pw[c][7]);
        }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.bar_p);
    };
    // ---- 448 dS = p8 (dP - D_i) of block b, then its INT8 codes into shared memory
    auto ds_phase = [&](const Blk& b) {
      // ---- 448 dS = p8 (dP - D_i), kept in registers until the tile scale is known
      const float dvec_t = QS ? b.dvec : sm.dvec[b.it & 1][t];
      ok = ok && mbar_wait(&sm.bar_dp, b.it & 1, abort);
      tc_fence_after();
      uint32_t buf[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld32(tmem + lane_base + cDP + kcol + 32 * c, buf[c]);
      tmem_ld_wait();
      if constexpr (PIPE) {
        // dP is in registers: the next dP may go in
        tc_fence_before();
        mbar_arrive(&sm.bar_free_dp);
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) reg_fence32(buf[c]);
      float amax = 0.f;
      if constexpr (F4) {
        // 2688 dS = (2688 P^) (dP - D_i)
        const uint64_t d2 = f2(dvec_t, dvec_t);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            float pv[8];
            fp4_decode8(pf[(32 * c + e) >> 3], (psc >> (8 * ((32 * c + e) >> 4))) & 255u, pv);
#pragma unroll
            for (int u = 0; u < 8; u += 2) {
              float x0, x1;
              f2split(fmul2(f2(pv[u], pv[u + 1]),
                            fsub2(f2(__uint_as_float(buf[c][e + u]), __uint_as_float(buf[c][e + u + 1])), d2)),
                      x0, x1);
              amax = max3(amax, fabsf(x0), fabsf(x1));
              buf[c][e + u] = __float_as_uint(x0);
              buf[c][e + u + 1] = __float_as_uint(x1);
            }
          }
        }
      } else {
        const uint64_t d2 = f2(dvec_t, dvec_t);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const uint32_t w = pw[c][e >> 2];
            const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
            const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
            const float2 p01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
            const float2 p23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
            float x[4];
            f2split(fmul2(f2(p01.x, p01.y), fsub2(f2(__uint_as_float(buf[c][e]), __uint_as_float(buf[c][e + 1])), d2)),
                    x[0], x[1]);
            f2split(fmul2(f2(p23.x, p23.y),
                          fsub2(f2(__uint_as_float(buf[c][e + 2]), __uint_as_float(buf[c][e + 3])), d2)),
                    x[2], x[3]);
            amax = max3(amax, fabsf(x[0]), fabsf(x[1]));
            amax = max3(amax, fabsf(x[2]), fabsf(x[3]));
#pragma unroll
            for (int u = 0; u < 4; ++u) buf[c][e + u] = __float_as_uint(x[u]);
          }
        }
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
      if (lane == 0) sm.smax[b.it & 1][warp] = amax;
      // the previous iteration's dQ boxes (this group's dS block and Q half) must be read
      // before the block is rewritten below and before the producer refills that Q buffer
      if constexpr (PIPE) {
        // the boxes of block it - 2, whose buffer block it's staging takes, must be read
        if (t == 0) bulk_wait_read_but_last();
      } else if (t == 0 && pending_qs >= 0) {
        bulk_wait_read_all();
        mbar_arrive(&sm.bar_q_free[pending_qs]);
        pending_qs = -1;
      }
      named_bar_group(g);
      // NVFP4: the dS codes take the block over once the dV MMA has read P^ from it
      if constexpr (F4) {
        ok = ok && mbar_wait(&sm.bar_dv, b.it & 1, abort);
        tc_fence_after();
      }
      // the group's tile (128 queries x 64 keys) max; values are 448 dS
      const float* smx = sm.smax[b.it & 1] + 4 * g;
      const float amine = fmaxf(fmaxf(smx[0], smx[1]), fmaxf(smx[2], smx[3]));
      const float inv = amine > 0.f ? 127.0f / amine : 0.f;  // code = rint(448 dS * 127 / max|448 dS|)
      // ---- dS codes -> shared memory (bf16 containers, 128B-swizzled query rows).  Rounding to
      // the nearest integer (ties to even) stays in the fp32 pipe: RN(x * inv + 1.5 * 2^23) - 1.5 * 2^23;
      // |x * inv| <= 127 (plus rounding), so no clamp is needed
      {
        const uint64_t inv2 = f2(inv, inv), magic2 = f2(kRoundMagic, kRoundMagic);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t packed[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float c0, c1;
            f2split(fsub2(ffma2(f2(__uint_as_float(buf[c][e]), __uint_as_float(buf[c][e + 1])), inv2, magic2), magic2),
                    c0, c1);
            const __nv_bfloat162 hv = __floats2bfloat162_rn(c0, c1);
            packed[e >> 1] = *reinterpret_cast<const uint32_t*>(&hv);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(dsrow + (((4 * c + u) ^ (t & 7)) << 4)) =
                make_uint4(packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.bar_ds[b.it & 1][g]);
    };
    // ---- dK += RN(s_dS * s_q) * part (key row t) of block b, and the dQ factors of its parts
    auto readout = [&](const Blk& b) {
      // Q-smoothing: this query block's mean over this group's features, for the dK term
      // (loaded while the dK MMA runs)
      float qb[QS ? DG : 1];
      if constexpr (QS) {
        const float4* src = reinterpret_cast<const float4*>(prm.qmean + ((size_t)b.qh * prm.nqb + b.I) * D + dcol);
#pragma unroll
        for (int c = 0; c < DG / 4; ++c) {
          const float4 v = __ldg(src + c);
          qb[4 * c] = v.x, qb[4 * c + 1] = v.y, qb[4 * c + 2] = v.z, qb[4 * c + 3] = v.w;
        }
      }
      // ---- dK += RN(s_dS * s_q) * part (key row t);  dQ (query row t) += ca * part0 + cb * part1
      ok = ok && mbar_wait(&sm.bar_dk, b.it & 1, abort);
      tc_fence_after();
      // the other group's tile max: its codes are in (bar_dk completed after both groups' codes),
      // and the waits below make its smax writes visible here
      ok = ok && mbar_wait(&sm.bar_ds[b.it & 1][0], (b.it >> 1) & 1, abort) &&
           mbar_wait(&sm.bar_ds[b.it & 1][1], (b.it >> 1) & 1, abort);
      const float* smx = sm.smax[b.it & 1];
      const float a0 = fmaxf(fmaxf(smx[0], smx[1]), fmaxf(smx[2], smx[3]));
      const float a1 = fmaxf(fmaxf(smx[4], smx[5]), fmaxf(smx[6], smx[7]));
      // values are 448 * dS: scale s_dS = max|dS| / 127
      const float sds0 = a0 > 0.f ? __fdiv_rn(a0 * (F4 ? 1.0f / 2688.0f : 1.0f / 448.0f), 127.0f) : 0.f;
      const float sds1 = a1 > 0.f ? __fdiv_rn(a1 * (F4 ? 1.0f / 2688.0f : 1.0f / 448.0f), 127.0f) : 0.f;
      const float ck = __fmul_rn(t >> 6 ? sds1 : sds0, b.sqI);
      ca = __fmul_rn(sds0, sk0);
      cb = __fmul_rn(sds1, sk1);
      // Q-smoothing: dK row t += RN(s_dS * sum_i dS8_it) * qmean (the sum is exact in TMEM)
      float cq = 0.f;
      if constexpr (QS) {
        uint32_t csum;
        tmem_ld1(tmem + lane_base + cDQ1, csum);
        tmem_ld_wait();
        asm volatile("" : "+r"(csum));
        cq = __fmul_rn(t >> 6 ? sds1 : sds0, __uint_as_float(csum));
        tc_fence_before();
        mbar_arrive(&sm.bar_cs);  // dQ1 may overwrite the column sums
      }
      {
        uint32_t kA[16], kB[16];
        tmem_ld16(tmem + lane_base + cDK + dcol, kA);
        tmem_wait16(kA);
#pragma unroll
        for (int c = 0; c < DG; c += 32) {
          tmem_ld16(tmem + lane_base + cDK + dcol + c + 16, kB);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            dk[c + e] = fmaf(ck, __uint_as_float(kA[e]), dk[c + e]);
            if constexpr (QS) dk[c + e] = fmaf(cq, qb[c + e], dk[c + e]);
          }
          tmem_wait16(kB);
          if (c + 32 < DG) tmem_ld16(tmem + lane_base + cDK + dcol + c + 32, kA);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            dk[c + 16 + e] = fmaf(ck, __uint_as_float(kB[e]), dk[c + 16 + e]);
            if constexpr (QS) dk[c + 16 + e] = fmaf(cq, qb[c + 16 + e], dk[c + 16 + e]);
          }
          if (c + 32 < DG) tmem_wait16(kA);
        }
      }
      // the dK part is in registers: its columns are free
      tc_fence_before();
      mbar_arrive(&sm.bar_dk_read);
    };
    // ---- dQ parts of block bk: ca * part0 + cb * part1 (query row t) staged as fp32 boxes and
    // added to the accumulator by TMA reduce
    auto staging = [&](const Blk& bk) {
      const int qs = bk.it & 1;
      ok = ok && mbar_wait(&sm.bar_part, bk.it & 1, abort);
      tc_fence_after();
      {
        // staging slot of box b (features dcol + 32b ..): this group's dS block, then half g of
        // q[qs]; PIPE: this group's box of the block's parity
        auto slot = [&](int b) -> float* {
          if constexpr (PIPE) return reinterpret_cast<float*>(sm.dqst + (2 * qs + g) * 16384);
          return reinterpret_cast<float*>(b == 0 ? sm.ds + g * 16384 : sm.q[qs] + g * 16384);
        };
        uint32_t va[2][16], vb[2][16];
        tmem_ld16(tmem + lane_base + cDQ0 + dcol, va[0]);
        tmem_ld16(tmem + lane_base + cDQ1 + dcol, vb[0]);
        tmem_ld_wait();
        reg_fence16(va[0]);
        reg_fence16(vb[0]);
#pragma unroll
        for (int c = 0; c < DG; c += 16) {
          const int cur = (c >> 4) & 1;
          if (c + 16 < DG) {
            tmem_ld16(tmem + lane_base + cDQ0 + dcol + c + 16, va[cur ^ 1]);
            tmem_ld16(tmem + lane_base + cDQ1 + dcol + c + 16, vb[cur ^ 1]);
          } else {
            // every TMEM read of the block is done: the next dQ parts (and, with dQ1 in the
            // dP columns, the next dP) may go in
            tc_fence_before();
            mbar_arrive(PIPE ? &sm.bar_dq_read : &sm.bar_free_dp);
          }
          // box row = feature, column = query row t: a warp stores 128 contiguous bytes
          float* box = slot(c >> 5) + (c & 31) * 128 + t;
#pragma unroll
          for (int e = 0; e < 16; ++e)
            box[e * 128] = fmaf(ca, __uint_as_float(va[cur][e]), cb * __uint_as_float(vb[cur][e]));
          if (c + 16 < DG) {
            tmem_ld_wait();
            reg_fence16(va[cur ^ 1]);
            reg_fence16(vb[cur ^ 1]);
          }
        }
        fence_proxy_async_smem();
        named_bar_group(g);
        if (t == 0) {
#pragma unroll
          for (int bx = 0; bx < DG / 32; ++bx) tma_reduce_add_3d(&tm_dq, slot(bx), bk.I * 128, (int)dcol + 32 * bx, bk.qh);
          bulk_commit();
          pending_qs = qs;
        }
      }
    };
    // Without PIPE each query block runs P, dS, the dK readout and the dQ staging in turn.  With
    // PIPE (dK, dQ and dP in TMEM columns of their own) the order is software-pipelined: step s
    // runs P of block s, then the readouts of block s - 1 (whose dK and dQ MMAs ran meanwhile),
    // then dS of block s (whose dP went in after block s - 1's dK readout).
    Blk cur{}, prev{};
    for (int s = 0; s < n_it + (PIPE ? 1 : 0); ++s) {
      if (s < n_it) {
        cur = take();
        p_phase(cur);
      }
      if constexpr (PIPE) {
        if (s > 0) {
          readout(prev);
          staging(prev);
        }
        if (s < n_it) ds_phase(cur);
        prev = cur;
      } else {
        ds_phase(cur);
        readout(cur);
        staging(cur);
      }
    }
    // the last reductions must complete before the CTA's shared memory goes away
    if (t == 0) bulk_wait_all();
    // ---------------- epilogue: dK then dV rows of this key block, this group's columns
    // (after a timed-out wait the results are not stored, but every thread still takes part
    // in the barriers below)
    {
      tc_fence_after();
      const size_t orow = ((size_t)bh * prm.N + key) * D;
#pragma unroll
      for (int d = 0; d < DG; ++d) dk[d] *= prm.sm_scale;
      const float* sdoh = prm.sdo + (size_t)bh * D;
      // split query heads: add this CTA's dK and (scaled) dV rows to the fp32 sums; the last
      // CTA of the key block to count reads the sums back and finishes them below
      const size_t arow = ((size_t)bh * prm.np + key) * D + dcol;
      bool fin = true;
      if (prm.split > 1) {
        if (key_ok && ok) {
#pragma unroll
          for (int c = 0; c < DG; c += 4) red_add_v4(prm.dkacc + arow + c, dk[c], dk[c + 1], dk[c + 2], dk[c + 3]);
        }
#pragma unroll 1
        for (int c = 0; c < DG; c += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_base + cDV + dcol + c, v);
          tmem_wait16(v);
          if (key_ok && ok) {
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              float f[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                f[e] = __uint_as_float(v[i + e]) * (sdoh[dcol + c + i + e] * (F4 ? 1.0f / 2688.0f : 1.0f / 448.0f));
              red_add_v4(prm.dvacc + arow + c + i, f[0], f[1], f[2], f[3]);
            }
          }
        }
        __threadfence();
        named_bar_compute();
        if (tid == 0) sm.last = atomicAdd(prm.kvcnt + (size_t)bh * prm.nqb + kb, 1) == prm.split - 1;
        named_bar_compute();
        fin = sm.last != 0;
        if (fin) {
          __threadfence();
          if (key_ok) {
#pragma unroll
            for (int c = 0; c < DG; c += 4) {
              const float4 a = __ldcg(reinterpret_cast<const float4*>(prm.dkacc + arow + c));
              dk[c] = a.x, dk[c + 1] = a.y, dk[c + 2] = a.z, dk[c + 3] = a.w;
            }
          }
        }
      }
      const uint4* krow = reinterpret_cast<const uint4*>(prm.K + orow + dcol);
      if (fin && prm.qk_norm) {
        // dk = r (dk' - k' (k' . dk')), k' = RN(k r): the dot spans both groups' columns
        const float r = key_ok ? prm.kr[(size_t)bh * prm.np + key] : 0.f;
        float dot = 0.f;
        if (key_ok) {
#pragma unroll
          for (int c = 0; c < DG / 8; ++c) {
            float f[8];
            unpack8(__ldg(krow + c), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) dot = fmaf(__fmul_rn(f[e], r), dk[c * 8 + e], dot);
          }
        }
        // partial dot products through the (now idle) bias rows
        float* xch = &sm.bias[0][0];
        named_bar_compute();
        xch[g * 128 + t] = dot;
        named_bar_compute();
        dot = xch[t] + xch[128 + t];
        if (key_ok) {
#pragma unroll
          for (int c = 0; c < DG / 8; ++c) {
            float f[8];
            unpack8(__ldg(krow + c), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) dk[c * 8 + e] = r * (dk[c * 8 + e] - __fmul_rn(f[e], r) * dot);
          }
        }
      }
      if (fin && key_ok && ok) {
        uint4* dstk = reinterpret_cast<uint4*>(prm.dK + orow + dcol);
#pragma unroll
        for (int c = 0; c < DG / 8; ++c) {
          uint4 u;
          __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
          for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(dk[c * 8 + 2 * e], dk[c * 8 + 2 * e + 1]);
          dstk[c] = u;
        }
      }
#pragma unroll
      for (int c = 0; fin && c < DG; c += 16) {
        float f[16];
        if (prm.split > 1) {
          // the finished sums, already scaled
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 a = key_ok ? __ldcg(reinterpret_cast<const float4*>(prm.dvacc + arow + c + i))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            f[i] = a.x, f[i + 1] = a.y, f[i + 2] = a.z, f[i + 3] = a.w;
          }
        } else {
          uint32_t v[16];
          tmem_ld16(tmem + lane_base + cDV + dcol + c, v);
          tmem_wait16(v);
#pragma unroll
          for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(v[e]) * (sdoh[dcol + c + e] * (F4 ? 1.0f / 2688.0f : 1.0f / 448.0f));
        }
        if (key_ok && ok) {
          uint4* dstv = reinterpret_cast<uint4*>(prm.dV + orow + dcol + c);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            uint4 u;
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(f[8 * i + 2 * e], f[8 * i + 2 * e + 1]);
            dstv[i] = u;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == WMMA) tmem_dealloc(tmem, kCols);
  if (tid == 0 && sm.abort) atomicExch(prm.status, kDevTimeout);
}

template <int D, bool QS, bool F4 = false>
int launch_main_t(const CUtensorMap& tk, const CUtensorMap& tq, const CUtensorMap& tv, const CUtensorMap& tdo,
                  const CUtensorMap& tdo8, const CUtensorMap& tdq, const BwdParams& p, int BH, cudaStream_t st) {
  size_t smem = sizeof(BwdSmem<D>);
  if (smem < 120 * 1024) smem = 120 * 1024;  // one CTA per SM: it holds all 512 TMEM columns
  auto kern = bwd_main_kernel<D, QS, F4>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 3;
  ScopedTimer timer("bwd_main", st);
  if (launch_pdl(kern, dim3(p.nqb * BH * p.split), dim3(384), smem, st, tk, tq, tv, tdo, tdo8, tdq, p) != cudaSuccess)
    return 3;
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // namespace

int launch_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
               void* dQ, void* dK, void* dV, const void* ws, void* bwd_ws, int B, int H, int N, int D, int causal,
               int qk_norm, int k_smooth, float sm_scale, cudaStream_t st, const float* O32, int Hkv,
               bool q_smooth, bool fp4) {
  (void)k_smooth;  // the smoothing Jacobian is applied as the identity (dS rows sum to zero)
  const QuantWs QL = quant_ws_layout(B, H, N, D, Hkv, q_smooth, fp4);
  const BwdWs BL = bwd_ws_layout(B, H, N, D, Hkv, fp4);
  const uint8_t* w = static_cast<const uint8_t*>(ws);
  uint8_t* bw = static_cast<uint8_t*>(bwd_ws);
  // BH query heads, BHk key/value heads, `group` query heads per key/value head
  const int BH = B * H, BHk = B * (Hkv > 0 ? Hkv : H), group = BH / BHk, np = QL.np, nb = np / 128;
  float* dvec = reinterpret_cast<float*>(bw + BL.dvec);
  float* biasv = reinterpret_cast<float*>(bw + BL.bias);
  float* dopart = reinterpret_cast<float*>(bw + BL.dopart);
  float* sdo = reinterpret_cast<float*>(bw + BL.sdo);
  float* dqacc = reinterpret_cast<float*>(bw + BL.dqacc);
  uint8_t* do8t = bw + BL.do8t;
  int* ticket = reinterpret_cast<int*>(bw + BL.sync);
  auto* o = static_cast<const __nv_bfloat16*>(O);
  auto* dob = static_cast<const __nv_bfloat16*>(dO);
  const dim3 g(nb, BH);
  // Grouped heads with too few (key block, key/value head) tiles to fill the GPU twice over
  // split each tile's query heads over `split` CTAs (a divisor of the group); their dK and dV
  // meet in fp32 sums.  One query head per key/value head never splits.
  int split = 1;
  if (group > 1) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 3;
    const int want = (2 * sms) / (BHk * nb);
    for (int s = want < group ? want : group; s > 1; --s)
      if (group % s == 0) {
        split = s;
        break;
      }
  }
  float* kvacc = split > 1 ? reinterpret_cast<float*>(bw + BL.dkacc) : nullptr;
  int* kvcnt = reinterpret_cast<int*>(bw + BL.kvcnt);
  {
  ScopedTimer timer("bwd_pre", st);
  if (launch_pdl(D == 128 ? bwd_pre_kernel<128> : bwd_pre_kernel<64>, g, dim3(kPreThreads), 0, st, o, O32, dob, LSE, N,
                 dvec, biasv, dopart, dqacc, ticket) != cudaSuccess ||
      launch_pdl(bwd_docomb_kernel, dim3(BHk), dim3(128), 0, st, (const float*)dopart, D, nb, group, sdo) !=
          cudaSuccess ||
      launch_pdl(D == 128 ? bwd_do8_kernel<128> : bwd_do8_kernel<64>, g, dim3(kPreThreads), 0, st, dob, N,
                 (const float*)sdo, group, do8t, dqacc, kvacc, kvcnt, (size_t)(BL.dvacc - BL.dkacc) / 4) !=
          cudaSuccess)
    return 3;
  }
  if (cudaGetLastError() != cudaSuccess) return 3;

  CUtensorMap tk, tq, tv, tdo, tdo8;
  if (!make_tmap_3d(&tk, w + QL.kc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, np, BHk, 64, 128)) return 3;
  if (!make_tmap_3d(&tq, w + QL.qc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, np, BH, 64, 128)) return 3;
  if (!make_tmap_3d(&tv, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, N, BHk, 64, 128)) return 3;
  if (!make_tmap_3d(&tdo, dO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, N, BH, 64, 128)) return 3;
  if (fp4) {
    // the codes as bf16 for the dV MMA: converted after bwd_do8, loaded in 64-query boxes
    const size_t n16 = (size_t)BH * D * np / 16;
    __nv_bfloat16* do16 = reinterpret_cast<__nv_bfloat16*>(bw + BL.do16);
    if (launch_pdl(do8_bf16_kernel, dim3((unsigned)((n16 + 255) / 256 < 4096 ? (n16 + 255) / 256 : 4096)), dim3(256),
                   0, st, (const uint8_t*)do8t, n16, do16) != cudaSuccess)
      return 3;
    if (!make_tmap_3d(&tdo8, do16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, np, D, BH, 64, D)) return 3;
  } else if (!make_tmap_3d(&tdo8, do8t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, np, D, BH, 128, D)) {
    return 3;
  }
  // dQ accumulator [BH][D][np] fp32, boxes of 32 features x 128 queries, unswizzled
  CUtensorMap tdq;
  if (!make_tmap_3d(&tdq, dqacc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, np, D, BH, 128, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
    return 3;
  BwdParams p;
  p.N = N;
  p.np = np;
  p.nqb = nb;
  p.BH = BHk;  // one CTA per (key block, key/value head)
  p.group = group;
  // Q codes, dO (bf16 and e4m3) of the query heads of a key/value head
  p.hgroup = l2_head_group((size_t)np * D * 5 * group, BHk);
  p.causal = causal;
  p.qk_norm = qk_norm;
  p.alpha = (float)((double)sm_scale * 1.4426950408889634074);
  p.sm_scale = sm_scale;
  p.sq = reinterpret_cast<const float*>(w + QL.sq);
  p.sk = reinterpret_cast<const float*>(w + QL.sk);
  p.sdo = sdo;
  p.bias = biasv;
  p.dvec = dvec;
  p.dsb = q_smooth ? reinterpret_cast<const float*>(w + QL.dsb) : nullptr;
  p.split = split;
  p.dkacc = reinterpret_cast<float*>(bw + BL.dkacc);
  p.dvacc = reinterpret_cast<float*>(bw + BL.dvacc);
  p.kvcnt = kvcnt;
  p.qmean = q_smooth ? reinterpret_cast<const float*>(w + QL.qmean) : nullptr;
  p.K = static_cast<const __nv_bfloat16*>(K);
  p.kr = reinterpret_cast<const float*>(w + QL.kr);
  p.dK = static_cast<__nv_bfloat16*>(dK);
  p.dV = static_cast<__nv_bfloat16*>(dV);
  p.status = reinterpret_cast<int*>(const_cast<uint8_t*>(w) + QL.status);
  int rc = fp4        ? (D == 128 ? launch_main_t<128, false, true>(tk, tq, tv, tdo, tdo8, tdq, p, BHk, st)
                                 : launch_main_t<64, false, true>(tk, tq, tv, tdo, tdo8, tdq, p, BHk, st))
           : q_smooth ? (D == 128 ? launch_main_t<128, true>(tk, tq, tv, tdo, tdo8, tdq, p, BHk, st)
                                : launch_main_t<64, true>(tk, tq, tv, tdo, tdo8, tdq, p, BHk, st))
                     : (D == 128 ? launch_main_t<128, false>(tk, tq, tv, tdo, tdo8, tdq, p, BHk, st)
                                 : launch_main_t<64, false>(tk, tq, tv, tdo, tdo8, tdq, p, BHk, st));
  if (rc) return rc;
  ScopedTimer timer("bwd_dq", st);
  return launch_bwd_dq(Q, reinterpret_cast<const float*>(w + QL.qr), bwd_ws, dQ, B, H, N, D, qk_norm, sm_scale,
                       p.status, st, Hkv);
}

}  // namespace sage
