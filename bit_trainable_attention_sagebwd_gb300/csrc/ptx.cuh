// Thin inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM alloc, UMMA issue/commit, TMEM load/store) and the operand
// descriptors that UMMA reads.  Every wait is bounded by wall-clock time so a
// lost arrival turns into an error status instead of a hung GPU.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sage {

// device-side status codes (kept in the workspace header word)
enum : int { kDevOk = 0, kDevTimeout = 4, kDevSetup = 5 };

// Wall-clock budget of one wait; generous next to any single tile of work.
#ifndef SAGE_WAIT_NS
#define SAGE_WAIT_NS 2000000000ull
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// order this thread's generic-proxy shared-memory writes before later async-proxy
// (TMA / UMMA) accesses
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity to complete.  Returns false (and
// raises *abort) when the budget runs out or another thread already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t budget_ns = SAGE_WAIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > budget_ns) {
        *abort = 1;
        return false;
      }
    }
  }
}

// ------------------------------------------------------------ CTA order
// Linear CTA index -> (tile index t in [0, ntile), head bh).  Heads go in groups of
// `hgroup` whose per-head operands fit in L2 together; inside a group the tile index is
// major, so in a causal pass the longest CTAs of the group (t = 0) start first and the
// short ones fill the tail.
__device__ __forceinline__ void tile_head_order(int idx, int ntile, int BH, int hgroup, int& t, int& bh) {
  const int s = idx / (ntile * hgroup);
  const int h0 = s * hgroup;
  const int r = idx - h0 * ntile;
  const int gs = BH - h0 < hgroup ? BH - h0 : hgroup;
  t = r / gs;
  bh = h0 + r % gs;
}

// heads per group for tile_head_order: as many as keep `bytes_per_head` within ~96 MB of L2
inline int l2_head_group(size_t bytes_per_head, int BH) {
  const size_t budget = (size_t)96 << 20;
  size_t g = bytes_per_head > 0 ? budget / bytes_per_head : (size_t)BH;
  if (g < 1) g = 1;
  if (g > (size_t)BH) g = BH;
  return (int)g;
}

// ------------------------------------------------ programmatic dependent launch
// Kernels of one pass follow each other on a stream with programmatic serialization:
// the next kernel's CTAs may start while this one drains.  Each kernel waits for its
// predecessor (completion and memory) before touching anything the predecessor writes or
// reads, then lets its own successor launch.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ----------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
// plain bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// element-wise add of a shared-memory box into global memory through a tensor map
// (the TMA unit performs the fp32 additions in L2); completion is tracked per thread
// by bulk async-groups
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(map),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until every committed bulk group of this thread has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// wait until at most the most recent committed bulk group of this thread is still reading
// shared memory
__device__ __forceinline__ void bulk_wait_read_but_last() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// wait until every committed bulk group of this thread has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ------------------------------------------------------------ fp32 pairs
// max of three floats in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// two fp32 lanes in one 64-bit register: each lane is an ordinary IEEE fp32 op
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2split(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// -------------------------------------------------------- register budgets
// Per-warpgroup register limits (all four warps of a warpgroup execute these).  The
// block's registers at launch (threads x registers per thread) form the pool: the
// increases must not exceed what the decreases hand back.
template <uint32_t N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// four fp32 additions to global memory, performed in L2 (16-byte aligned address)
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// ------------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, 16-bit operands (bf16), fp32 accumulate
__device__ __forceinline__ void umma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, 8-bit float operands (e4m3), fp32 accumulate
__device__ __forceinline__ void umma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Four MMAs along K into the same accumulator, in one asm block so that they issue back to
// back: the k-th (k = 0..3) reads the descriptors a + k SA and b + k SB (steps in 16-byte units
// of the start-address field, which never carries: shared addresses are below 256 KB).  The
// first accumulates when acc != 0, the other three always.  An MMA issuer that shares its SM
// sub-partition with busy warps spends about a third of the instructions per MMA this way.
#define SAGE_UMMA_X4(KIND)                                                                          \
  asm volatile(                                                                                     \
      "{\n .reg .pred p, q;\n .reg .b64 a1, a2, a3, b1, b2, b3;\n"                                \
      " setp.ne.b32 p, %4, 0;\n setp.eq.b32 q, %4, %4;\n"                                           \
      " add.s64 a1, %1, %5;\n add.s64 a2, %1, %6;\n add.s64 a3, %1, %7;\n"                          \
      " add.s64 b1, %2, %8;\n add.s64 b2, %2, %9;\n add.s64 b3, %2, %10;\n"                         \
      " tcgen05.mma.cta_group::1.kind::" KIND " [%0], %1, %2, %3, p;\n"                            \
      " tcgen05.mma.cta_group::1.kind::" KIND " [%0], a1, b1, %3, q;\n"                            \
      " tcgen05.mma.cta_group::1.kind::" KIND " [%0], a2, b2, %3, q;\n"                            \
      " tcgen05.mma.cta_group::1.kind::" KIND " [%0], a3, b3, %3, q;\n}\n" ::"r"(d),                \
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "n"(SA), "n"(2 * SA), "n"(3 * SA), "n"(SB), "n"(2 * SB), \
      "n"(3 * SB)                                                                                   \
      : "memory")
template <int SA, int SB>
__device__ __forceinline__ void umma_bf16_x4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  SAGE_UMMA_X4("f16");
}
template <int SA, int SB>
__device__ __forceinline__ void umma_f8_x4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  SAGE_UMMA_X4("f8f6f4");
}
#undef SAGE_UMMA_X4
// D[tmem] (+)= (A * scale A)[smem] * (B * scale B)[smem]^T: packed e2m1 operands (two per byte,
// K-major), one ue4m3 scale per 16 values along K for each row of A and of B, read from TMEM
// (sfa, sfb: four columns each, the 32 x 16-byte atom that tmem_cp_32x128b_x4 writes); fp32
// accumulate; K = 64 per instruction
__device__ __forceinline__ void umma_nvf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                          uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
// copy a 32-row x 16-byte shared-memory block (descriptor, no swizzle) to TMEM lanes 0-31,
// columns [taddr, taddr + 4), and the same to lanes 32-63, 64-95 and 96-127
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// arrive once on *bar when every UMMA issued so far by this thread has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets lane
// (warp's lane quarter + t), columns [col, col + 32)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
}
// one 32-bit column: thread t of the warp gets lane (warp's lane quarter + t)
__device__ __forceinline__ void tmem_ld1(uint32_t taddr, uint32_t& r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Marks 32 registers as produced at this point, so that no use of a value loaded
// by tcgen05.ld can be scheduled above the wait that precedes this call.
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]));
}
// wait for every tcgen05.ld of this thread, then fence the loaded registers
__device__ __forceinline__ void tmem_wait32(uint32_t (&r)[32]) {
  tmem_ld_wait();
  reg_fence32(r);
}
__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
  tmem_ld_wait();
  reg_fence16(r);
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// --------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor, 128-byte swizzle.  A tile is stored as
// blocks of 8 rows x 128 bytes (1024 B, 1024-aligned) in the pattern TMA's
// SWIZZLE_128B writes: the 16-byte chunk c of row r sits at chunk (c ^ (r & 7)).
//   K-major operand: rows = M (or N) index, the 128 bytes run along K;
//     sbo = byte distance between 8-row groups; lbo unused (16).
//   MN-major operand: rows = K index, the 128 bytes run along M (or N);
//     sbo = byte distance between 8-row (K) groups, lbo = byte distance
//     between 128-byte (M/N) column blocks.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for tcgen05
  d |= 2ull << 61;  // 128-byte swizzle
  return d;
}

// Shared-memory matrix descriptor, 64-byte swizzle (K-major): blocks of 8 rows x 64 bytes
// (512 B), the 16-byte chunk c of row r at chunk c ^ ((r & 7) >> 1); sbo = 512.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for tcgen05
  d |= 4ull << 61;  // 64-byte swizzle
  return d;
}

// Shared-memory matrix descriptor without swizzle: the tile is made of core matrices of
// 8 rows x 16 bytes (128 contiguous bytes); lbo and sbo are the byte distances between
// core matrices adjacent along K and along M (or N).
__device__ __forceinline__ uint64_t sdesc_none(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for tcgen05
  return d;         // layout type 0: no swizzle
}

// Instruction descriptors (kind::f16 with bf16 inputs / kind::f8f6f4 with
// e4m3 inputs; fp32 accumulator; dense; no negation).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                             // D = F32
         | (1u << 7)                           // A = BF16
         | (1u << 10)                          // B = BF16
         | ((a_mn_major ? 1u : 0u) << 15)      // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)      // B major-ness
         | ((uint32_t)(N >> 3) << 17)          // N / 8
         | ((uint32_t)(M >> 4) << 24);         // M / 16
}
// block-scaled kind::mxf4nvf4: A = B = e2m1, ue4m3 scales (format bit 0), K-major, scale
// factor ids 0
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7)                     // A = E2M1
         | (1u << 10)                  // B = E2M1
         | ((uint32_t)(N >> 3) << 17)  // N / 8
         | ((uint32_t)(M >> 4) << 24); // M / 16
}
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool a_mn_major = false) {
  return (1u << 4)                         // D = F32
         | (0u << 7) | (0u << 10)          // A = B = E4M3
         | ((a_mn_major ? 1u : 0u) << 15)  // A major-ness
         | ((uint32_t)(N >> 3) << 17)      // N / 8
         | ((uint32_t)(M >> 4) << 24);     // M / 16
}

}  // namespace sage
