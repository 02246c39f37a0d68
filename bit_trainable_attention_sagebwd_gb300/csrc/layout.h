// Workspace layouts (device memory owned by the caller, carved by the library).
// Every section starts on a 256-byte boundary.  Np = N rounded up to 128.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace sage {

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline int pad128(int n) { return (n + 127) / 128 * 128; }

struct QuantWs {
  // byte offsets
  size_t status, sync, qc, kc, v8t, sq, sk, sv, kmean, qr, kr, kpart, vpart, qmean, dsb, vg, v4, v4sf, total;
  int np;
};

// quantize workspace: codes and scales the forward and backward read, and the
// per-128-token partial sums that the smoothing mean and the V scales come from.
// Hkv key/value heads per batch entry (Hkv divides H; 0 means Hkv = H): the Q sections hold
// B*H heads, the K and V sections B*Hkv.  With Q-smoothing (qs) two more sections per query
// head: the query blocks' channel means [nb][D] and the logit terms they carry [nb][Np].
// With NVFP4 (fp4) three more per key/value head: V's tensor scale g (fp32), its e2m1 codes
// packed two per byte [D][Np/2] (channel-major, the lower token in the low nibble) and their
// e4m3 block scales, one per (channel, 16 tokens), as the tensor core reads them: per 64-token
// chunk a 512-byte atom, byte (d % 32) * 16 + (d / 32) * 4 + (16-token block within the chunk).
inline QuantWs quant_ws_layout(int B, int H, int N, int D, int Hkv = 0, bool qs = false, bool fp4 = false) {
  QuantWs L{};
  const size_t bh = (size_t)B * H, bk = (size_t)B * (Hkv > 0 ? Hkv : H);
  const int np = pad128(N);
  const size_t nb = np / 128;
  size_t o = 0;
  L.status = o; o = align256(o + 256);
  L.sync = o;   o = align256(o + 2 * bk * 4);  // per-head counters of finished statistics blocks
  L.qc = o;     o = align256(o + bh * np * D * 2);
  L.kc = o;     o = align256(o + bk * np * D * 2);
  L.v8t = o;    o = align256(o + bk * D * np);
  L.sq = o;     o = align256(o + bh * nb * 4);
  L.sk = o;     o = align256(o + bk * nb * 2 * 4);
  L.sv = o;     o = align256(o + bk * D * 4);
  L.kmean = o;  o = align256(o + bk * D * 4);
  L.qr = o;     o = align256(o + bh * np * 4);
  L.kr = o;     o = align256(o + bk * np * 4);
  L.kpart = o;  o = align256(o + bk * nb * D * 8);  // fp64 partial column sums of k'
  L.vpart = o;  o = align256(o + bk * nb * D * 4);  // partial channel max |V|
  L.qmean = o;  o = align256(o + (qs ? bh * nb * D * 4 : 0));
  L.dsb = o;    o = align256(o + (qs ? bh * nb * np * 4 : 0));
  L.vg = o;     o = align256(o + (fp4 ? bk * 4 : 0));
  L.v4 = o;     o = align256(o + (fp4 ? bk * D * np / 2 : 0));
  L.v4sf = o;   o = align256(o + (fp4 ? bk * (np / 64) * 512 : 0));
  L.total = o;
  L.np = np;
  return L;
}

struct BwdWs {
  size_t sync, dvec, bias, do8t, sdo, dopart, dqacc, dkacc, dvacc, kvcnt, do16, total;
  int np;
};

// backward scratch: the dQ pass's work ticket, D_i, log2(448) - LSE*log2(e) (-inf on padded rows), FP8 dO codes
// (channel-major), their channel scales (one set per key/value head: the query heads that
// share it share the scale) and partial maxima, fp32 dQ accumulator (feature-major
// [BH, D, Np] so that reductions from query rows coalesce)
// fp4 (NVFP4 backward): the e4m3 codes of dO also as bf16 [BH, D, Np], the dV operand
inline BwdWs bwd_ws_layout(int B, int H, int N, int D, int Hkv = 0, bool fp4 = false) {
  BwdWs L{};
  const size_t bh = (size_t)B * H, bk = (size_t)B * (Hkv > 0 ? Hkv : H);
  const int np = pad128(N);
  const size_t nb = np / 128;
  size_t o = 0;
  L.sync = o;   o = align256(o + 16);
  L.dvec = o;   o = align256(o + bh * np * 4);
  L.bias = o;   o = align256(o + bh * np * 4);
  L.do8t = o;   o = align256(o + bh * D * np);
  L.sdo = o;    o = align256(o + bk * D * 4);
  L.dopart = o; o = align256(o + bh * nb * D * 4);
  L.dqacc = o;  o = align256(o + bh * np * D * 4);
  // grouped heads: fp32 sums of dK and dV [Bk, Np, D] for key blocks whose query heads are
  // split over several CTAs, and a counter per (key/value head, key block)
  const bool grouped = bk < bh;
  L.dkacc = o;  o = align256(o + (grouped ? bk * np * D * 4 : 0));
  L.dvacc = o;  o = align256(o + (grouped ? bk * np * D * 4 : 0));
  L.kvcnt = o;  o = align256(o + (grouped ? bk * nb * 4 : 0));
  L.do16 = o;   o = align256(o + (fp4 ? bh * D * np * 2 : 0));
  L.total = o;
  L.np = np;
  return L;
}

struct ThriftWs {
  size_t qbar, kbar, keys, sel, q16, k16, v16, oacc, ml, total;
  int np;
};

// ThriftAttention scratch: the raw blocks' channel means (fp64), the pair scores as
// order-preserving keys, the promoted pairs (uint8 [BH][nb][nb]), the high-precision path's
// fp16 copies of q', k'' and V ([BH][Np][D], rows past N zero), and what the low-bit pass
// hands over for query tiles with promoted pairs: the unnormalised output (fp32 [BH][Np][D])
// and per row the running maximum and the row sum ([BH][Np][2])
inline ThriftWs thrift_ws_layout(int B, int H, int N, int D) {
  ThriftWs L{};
  const size_t bh = (size_t)B * H;
  const int np = pad128(N);
  const size_t nb = np / 128;
  size_t o = 0;
  L.qbar = o;  o = align256(o + bh * nb * D * 8);
  L.kbar = o;  o = align256(o + bh * nb * D * 8);
  L.keys = o;  o = align256(o + bh * nb * nb * 8);
  L.sel = o;   o = align256(o + bh * nb * nb);
  L.q16 = o;   o = align256(o + bh * np * D * 2);
  L.k16 = o;   o = align256(o + bh * np * D * 2);
  L.v16 = o;   o = align256(o + bh * np * D * 2);
  L.oacc = o;  o = align256(o + bh * np * D * 4);
  L.ml = o;    o = align256(o + bh * np * 8);
  L.total = o;
  L.np = np;
  return L;
}

}  // namespace sage
