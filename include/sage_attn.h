/*
 * sage_attn.h -- C ABI of the GB300 (sm_103a) low-bit attention library:
 * the SageBwd scheme's quantize pass, forward and backward for training.
 *
 * What the calls compute
 * ----------------------
 * "SageBwd: A Trainable Low-bit Attention" (euno.news summary), Methodology 1-2:
 * six of the seven matmuls of an attention block run in low precision -- QK^T and
 * PV in the forward, the S recompute, dV, dQ and dK in the backward -- while the
 * softmax-gradient matmul dP = dO V^T stays in high precision (bf16 here).
 * Methodology 4 and Results: QK-norm (each query and key scaled to unit L2 norm
 * before the dot product) and K-smoothing (read here as subtracting the per-head
 * channel mean of K over tokens, which leaves the softmax unchanged).
 * "Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (gist.science
 * summary), Methodology, principle 1: the backward recomputes P from the saved
 * log-sum-exp in the forward's low precision.  "ThriftAttention" (gist.science
 * summary), Methodology step 2: the FlashAttention-2 online softmax over key tiles.
 *
 * Number formats (the pages give no formulas; these are the plainest reading):
 *   Q: INT8, one fp32 scale max|q'|/127 per 128-token block (all channels);
 *   K: INT8, one fp32 scale max|k''|/127 per 64-token block;
 *   V, dO: FP8 e4m3, one fp32 scale max|x|/448 per (head, channel);
 *   P: FP8 e4m3 with the static scale 1/448 (probabilities relative to the
 *      running row maximum are at most 1);
 *   dS: INT8, one scale max|dS|/127 per (128-query x 64-key) tile.
 * INT8 products accumulate exactly (the codes sit in bf16 containers and every
 * partial sum is an integer below 2^24, exact in the fp32 accumulator).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensors Q, K, V, O, dO, dQ, dK, dV: bf16, contiguous [B, H, N, D] (D fastest),
 *    device memory owned by the caller, 16-byte aligned.  LSE: fp32 [B, H, N],
 *    natural log.  O32 (optional): fp32 [B, H, N, D].
 *  - Supported shapes: B, H >= 1; N >= 1 (any value; tiles are padded internally);
 *    D in {64, 128}; queries and keys share N.  Other shapes: SAGE_ERR_UNSUPPORTED.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on that stream, allocates nothing and never synchronises,
 *    except sage_attn_get_status.
 *  - Argument errors are returned synchronously before anything is launched.
 *  - Workspaces are device memory the caller allocates with at least the size the
 *    *_ws_bytes call reports; their contents are owned by the library between
 *    sage_attn_quantize and the last forward/backward that reads them.
 *  - Every device-side wait is bounded; a wait that runs out records
 *    SAGE_ERR_TIMEOUT in the workspace status word (read with
 *    sage_attn_get_status) and the kernel returns.
 *  - The forward is deterministic.  dQ is accumulated with fp32 additions in L2
 *    (TMA reductions) across key blocks, so its last bits depend on their order.
 */
#ifndef SAGE_ATTN_H
#define SAGE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SAGE_OK = 0,
  SAGE_ERR_INVALID_ARG = 1, /* null or misaligned pointer, bad size, workspace too small */
  SAGE_ERR_UNSUPPORTED = 2, /* shape outside the supported set */
  SAGE_ERR_CUDA = 3,        /* a CUDA runtime call failed (launch, attribute, tensor map) */
  SAGE_ERR_TIMEOUT = 4      /* a device-side wait ran out of its time budget */
} sage_status;

/* Pointers into a quantize workspace (for inspection and parity tests).
 * Np = N rounded up to a multiple of 128; rows past N hold zero codes. */
typedef struct sage_ws_views {
  void *qc;      /* bf16 [B*H, Np, D]: INT8 codes of q' (bf16 containers)           */
  void *kc;      /* bf16 [B*H, Np, D]: INT8 codes of k'' (smoothed, bf16 containers) */
  void *v8t;     /* e4m3 [B*H, D, Np]: FP8 codes of V, channel-major                 */
  float *sq;     /* [B*H, Np/128] Q block scales                                     */
  float *sk;     /* [B*H, Np/64]  K block scales                                     */
  float *sv;     /* [B*H, D]      V channel scales                                   */
  float *kmean;  /* [B*H, D]      channel mean of k' (0 without K-smoothing)         */
  float *qr;     /* [B*H, Np]     1/||q|| per token (1 without QK-norm)              */
  float *kr;     /* [B*H, Np]     1/||k|| per token (1 without QK-norm)              */
  int *status;   /* device status word                                               */
  int n_pad;     /* Np                                                               */
  float *qmean;  /* Q-smoothing: [B*H, Np/128, D] query block means (else NULL)      */
  float *dsb;    /* Q-smoothing: [B*H, Np/128, Np] logit terms (else NULL)           */
  float *vg;     /* NVFP4: [B*H] V's tensor scale max|V| / 2688 (else NULL)          */
  uint8_t *v4;   /* NVFP4: [B*H, D, Np/2] V's e2m1 codes, two per byte, the lower    */
                 /*        token in the low nibble (else NULL)                       */
  uint8_t *v4sf; /* NVFP4: [B*H, Np/64, 512] V's e4m3 block scales; in atom c (tokens */
                 /*        64c ..) byte (d % 32) * 16 + (d / 32) * 4 + 16-token block */
} sage_ws_views;

/* Bytes of the quantize workspace for this shape (0 if unsupported). It holds the
 * codes and scales the forward and backward read, plus the status word. */
size_t sage_attn_ws_bytes(int B, int H, int N, int D);

/* Bytes of the backward scratch for this shape (0 if unsupported): the row terms
 * D_i = rowsum(dO * O) and LSE*log2(e), the FP8 codes of dO, and the fp32 dQ
 * accumulator. */
size_t sage_attn_bwd_ws_bytes(int B, int H, int N, int D);

/*
 * Quantize pass (SageBwd summary, Methodology 1 and 4).
 * Reads Q, K, V; optionally L2-normalises q and k per token (qk_norm != 0);
 * optionally subtracts the per-(b,h) channel mean of k over the N tokens
 * (k_smooth != 0); writes the INT8 codes and scales of q' and k'' and the FP8
 * codes and scales of V into `ws`, and clears the status word.
 * Rounding: every scale and quotient is a correctly rounded fp32 operation;
 * codes round half to even; the norms and means are the fp32 rounding of the
 * exact sums.
 */
int sage_attn_quantize(const void *Q, const void *K, const void *V, int B, int H, int N, int D,
                       int qk_norm, int k_smooth, void *ws, size_t ws_bytes, void *stream);

/*
 * Forward (SageBwd summary, Methodology 1; ThriftAttention summary, Methodology 2).
 * S = (q8 k8^T) * sq * sk * sm_scale computed exactly in integers and scaled in
 * fp32; causal (causal != 0) masks keys j > i; online softmax over 128-key tiles
 * with the running maximum; P = 2^(S*log2e - m) rounded to e4m3 after scaling by
 * 448; O = (P8 V8) * sv / (448 l).  Writes O (bf16), LSE (fp32, natural log) and,
 * if O32 is not NULL, O in fp32 before the bf16 rounding.
 * sm_scale <= 0 selects 1/sqrt(D).  `ws` comes from sage_attn_quantize with the
 * same B, H, N, D.
 */
int sage_attn_fwd(const void *ws, void *O, float *LSE, float *O32, int B, int H, int N, int D,
                  int causal, float sm_scale, void *stream);

/*
 * Backward (SageBwd summary, Methodology 2; Attn-QAT summary, principle 1).
 * D_i = sum_d dO*O; P recomputed from LSE and rounded to e4m3 exactly as in the
 * forward; dP = dO V^T in bf16 with fp32 accumulation (the one unquantized
 * matmul); dS = P (dP - D_i); dV = P8^T dO8 (FP8); dS to INT8 per 128x64 tile;
 * dQ = dS8 k8 and dK = dS8^T q8 (exact integer sums, scaled per tile); then
 * dQ, dK times sm_scale and back through QK-norm when qk_norm != 0.  K-smoothing
 * passes dK through unchanged (the exact dS rows sum to zero).
 * Q, K, V, dO are the same inputs the forward saw; O and LSE the forward's outputs;
 * `ws` the quantize workspace; `bwd_ws` scratch of sage_attn_bwd_ws_bytes.
 * Writes dQ, dK, dV (bf16).
 */
int sage_attn_bwd(const void *Q, const void *K, const void *V, const void *O, const float *LSE,
                  const void *dO, void *dQ, void *dK, void *dV, const void *ws, void *bwd_ws,
                  size_t bwd_ws_bytes, int B, int H, int N, int D, int causal, int qk_norm,
                  int k_smooth, float sm_scale, void *stream);

/*
 * Backward with the high-precision auxiliary output ("Attn-QAT: 4-Bit Attention With
 * Quantization-Aware Training" (gist.science summary), Methodology, principle 2): the same
 * as sage_attn_bwd, except that the row terms D_i = sum_d dO_id O'_id take O' = O32, the
 * forward's fp32 output before its bf16 rounding (the O32 output of sage_attn_fwd), instead
 * of the bf16 O.  O32: fp32 [B, H, N, D], device memory, 16-byte aligned.  The bf16 O is
 * not read.  Errors as for sage_attn_bwd.
 */
int sage_attn_bwd_o32(const void *Q, const void *K, const void *V, const float *O32, const float *LSE,
                      const void *dO, void *dQ, void *dK, void *dV, const void *ws, void *bwd_ws,
                      size_t bwd_ws_bytes, int B, int H, int N, int D, int causal, int qk_norm,
                      int k_smooth, float sm_scale, void *stream);

/*
 * Grouped-query attention: Hkv key/value heads per batch entry, each shared by G = H / Hkv
 * consecutive query heads (query head h reads key/value head h / G; Hkv = 1 is multi-query
 * attention).  The pages leave grouped heads unvalidated ("SageBwd: A Trainable Low-bit
 * Attention" (euno.news summary), Limitations); these calls extend the scheme as follows.
 *  - K, V, dK, dV are bf16 [B, Hkv, N, D]; Q, O, dO, dQ bf16 [B, H, N, D]; LSE [B, H, N].
 *  - Quantize: Q per query head as above; K (smoothing mean, block scales) and V (channel
 *    scales) per key/value head.
 *  - Forward: each query head against its key/value head, exactly as above.
 *  - Backward: dK and dV of a key/value head sum over its G query heads.  The e4m3 channel
 *    scale of dO spans the G query heads' tokens (one scale per key/value head and channel),
 *    so dV stays one FP8 accumulation over all of them.
 * With Hkv = H every call equals its counterpart above.  Hkv must divide H
 * (else SAGE_ERR_UNSUPPORTED).
 */
size_t sage_attn_gqa_ws_bytes(int B, int H, int Hkv, int N, int D);
size_t sage_attn_gqa_bwd_ws_bytes(int B, int H, int Hkv, int N, int D);
int sage_attn_gqa_quantize(const void *Q, const void *K, const void *V, int B, int H, int Hkv, int N, int D,
                           int qk_norm, int k_smooth, void *ws, size_t ws_bytes, void *stream);
int sage_attn_gqa_fwd(const void *ws, void *O, float *LSE, float *O32, int B, int H, int Hkv, int N, int D,
                      int causal, float sm_scale, void *stream);
int sage_attn_gqa_bwd(const void *Q, const void *K, const void *V, const void *O, const float *LSE,
                      const void *dO, void *dQ, void *dK, void *dV, const void *ws, void *bwd_ws,
                      size_t bwd_ws_bytes, int B, int H, int Hkv, int N, int D, int causal, int qk_norm,
                      int k_smooth, float sm_scale, void *stream);
/* Workspace views for the grouped layout: qc, sq, qr hold B*H heads; kc, v8t, sk, sv,
 * kmean, kr hold B*Hkv. */
int sage_attn_gqa_ws_views(void *ws, int B, int H, int Hkv, int N, int D, sage_ws_views *views);

/*
 * Q-smoothing (the optional companion of K-smoothing that "SageBwd: A Trainable Low-bit
 * Attention" (euno.news summary), Methodology 4, names without a formula), with grouped
 * heads as the sage_attn_gqa_* calls (Hkv = H: one key/value head per query head).
 *  - Quantize: each 128-token query block I loses its channel mean before the INT8
 *    quantizer: qmean_I = RN32(sum of the block's q' / its token count) (the fp32 rounding of
 *    the exact mean), qs = RN32(q' - qmean_I), codes and block scale of qs.  The logit terms
 *    dsb[I][j] = qmean_I . k''_j (fp32 products and sums, k'' the smoothed keys of the query
 *    head's key/value head) are stored for every (query block, key).  Workspace:
 *    sage_attn_qs_ws_bytes; it adds 4*B*H*Np/128*(D + Np) bytes to the grouped layout.
 *  - Forward: the logit of query i (block I) and key j is u = RN32(acc * RN32(s_q s_k) +
 *    dsb[I][j]) in natural units; u * RN32(sm_scale log2 e) enters the online softmax.
 *  - Backward (scratch: sage_attn_gqa_bwd_ws_bytes): P is recomputed with the same u, and
 *    dK of each key gets, per (query block, 64-key block) tile, s_dS (sum over the tile's
 *    queries of the dS codes) qmean_I: the mean's share of S = qs k'' + qmean k''.
 * Arguments, layouts, ownership and errors as in the sage_attn_gqa_* calls; a workspace
 * quantized with Q-smoothing is read only by sage_attn_qs_fwd and sage_attn_qs_bwd.
 */
size_t sage_attn_qs_ws_bytes(int B, int H, int Hkv, int N, int D);
int sage_attn_qs_quantize(const void *Q, const void *K, const void *V, int B, int H, int Hkv, int N, int D,
                          int qk_norm, int k_smooth, void *ws, size_t ws_bytes, void *stream);
int sage_attn_qs_fwd(const void *ws, void *O, float *LSE, float *O32, int B, int H, int Hkv, int N, int D,
                     int causal, float sm_scale, void *stream);
int sage_attn_qs_bwd(const void *Q, const void *K, const void *V, const void *O, const float *LSE,
                     const void *dO, void *dQ, void *dK, void *dV, const void *ws, void *bwd_ws,
                     size_t bwd_ws_bytes, int B, int H, int Hkv, int N, int D, int causal, int qk_norm,
                     int k_smooth, float sm_scale, void *stream);
/* Workspace views of the Q-smoothing layout, qmean and dsb included. */
int sage_attn_qs_ws_views(void *ws, int B, int H, int Hkv, int N, int D, sage_ws_views *views);

/*
 * ThriftAttention's selective mixed precision, forward only ("ThriftAttention"
 * (gist.science summary), Methodology steps 1-2 and its implementation paragraph).
 *  - Selection: the importance of the pair (128-query block I, 128-key tile J) is
 *    qbar_I . kbar_J, the dot product of the blocks' channel means over the raw Q and K
 *    (fp64: each mean sums the block's tokens in order and divides by their count; the
 *    dot product adds the channel products in order).  Of the pairs the mask lets through
 *    (causal: J <= I) the n = ceil(budget * pairs - 1e-12) largest are promoted, ties in
 *    index order I * nb + J (nb = Np / 128), per head.
 *  - Promoted pairs run in high precision: S = q16 . k16 (fp16 copies of q' and of the
 *    smoothed keys k'' = RN32(k' - kmean), fp32 accumulation), P16 = fp16(p~), O += P16 v16
 *    (v16 = fp16(V)) in fp32.  The others take the low-bit path of sage_attn_fwd.  A row
 *    runs its low-bit tiles first and its promoted tiles after them, in one online softmax
 *    (shared running maximum and row sum).
 * sage_attn_thrift_ws_bytes: size of the scratch (device memory, caller-owned) that holds
 *   the selection, the fp16 operands and the low-bit pass's hand-over; 0 for an unsupported
 *   shape.
 * sage_attn_thrift_quantize: the quantize pass of sage_attn_quantize into `ws`, then the
 *   selection and the fp16 operands into `tws`; budget in [0, 1].
 * sage_attn_thrift_fwd: the forward on `ws` and `tws` from that call; outputs, sm_scale
 *   and errors as in sage_attn_fwd.
 * sage_attn_thrift_sel: device pointer to the promoted pairs, uint8 [B*H, nb, nb] (1 =
 *   promoted), inside `tws`; NULL for an unsupported shape.
 * Q-smoothing and grouped heads are not combined with this path.
 */
size_t sage_attn_thrift_ws_bytes(int B, int H, int N, int D);
int sage_attn_thrift_quantize(const void *Q, const void *K, const void *V, int B, int H, int N, int D,
                              int qk_norm, int k_smooth, int causal, double budget, void *ws, size_t ws_bytes,
                              void *tws, size_t tws_bytes, void *stream);
int sage_attn_thrift_fwd(const void *ws, const void *tws, void *O, float *LSE, float *O32, int B, int H, int N,
                         int D, int causal, float sm_scale, void *stream);
uint8_t *sage_attn_thrift_sel(void *tws, int B, int H, int N, int D);

/*
 * NVFP4 variant of the forward PV ("Attn-QAT: 4-Bit Attention With Quantization-Aware
 * Training" (gist.science summary), Methodology principle 1 and Implementation: attention
 * trained in FP4 on Blackwell's FP4 path; "ThriftAttention" (gist.science summary),
 * Methodology step 2: the NVFP4 format).  The pages print no recipe; this is NVFP4 for P and
 * V with the rest of the scheme unchanged:
 *  - e2m1 codes (0, 0.5, 1, 1.5, 2, 3, 4, 6, signed; nearest, ties to the even code,
 *    saturating), one e4m3 scale per 16 consecutive values along the contracted axis (keys),
 *    one fp32 scale per tensor;
 *  - V, per head: g = RN32(max|V| / 2688); per channel and 16-token block
 *    s = e4m3(RN32(amax / RN32(6 g))), code = e2m1(RN32(v / RN32(s g)));
 *  - P, per row and 16-key block of the online softmax's p~ (relative to the running maximum):
 *    y = RN32(2688 p~), s = e4m3(RN32(max y / 6)), code = e2m1(RN32(y / s)); P^ = code s / 2688;
 *  - O = sum(P^ V^) / l with l the sum of the fp32 p~; QK^T stays INT8.
 * The tensor core multiplies the e2m1 codes and their block scales
 * (tcgen05.mma kind::mxf4nvf4.block_scale); the codes and scales equal the definition above
 * bit for bit.
 * sage_attn_fp4_ws_bytes: workspace size; sage_attn_fp4_quantize: the quantize pass plus V's
 * NVFP4 codes and scales; sage_attn_fp4_fwd: the forward on that workspace (outputs, sm_scale
 * and errors as in sage_attn_fwd); sage_attn_fp4_ws_views: the workspace's pointers, vg, v4
 * and v4sf included.  Plain heads (no grouped heads, no Q-smoothing).
 */
size_t sage_attn_fp4_ws_bytes(int B, int H, int N, int D);
int sage_attn_fp4_quantize(const void *Q, const void *K, const void *V, int B, int H, int N, int D, int qk_norm,
                           int k_smooth, void *ws, size_t ws_bytes, void *stream);
int sage_attn_fp4_fwd(const void *ws, void *O, float *LSE, float *O32, int B, int H, int N, int D, int causal,
                      float sm_scale, void *stream);
int sage_attn_fp4_ws_views(void *ws, int B, int H, int N, int D, sage_ws_views *views);
/* NVFP4 backward (Attn-QAT, principle 1: P recomputed at the forward's precision): P^ in
 * NVFP4 from the saved LSE with the forward's 16-key blocks, used in dS = P^ (dP - D_i) and
 * dV = P^T dO8; the rest as sage_attn_bwd.  dV runs on bf16 tensor cores with the exact
 * values code * s and dO's e4m3 codes (P^'s scales vary along the keys, which dV does not
 * contract).  Scratch: sage_attn_fp4_bwd_ws_bytes (it adds dO's codes as bf16).  `ws` comes
 * from sage_attn_fp4_quantize. */
size_t sage_attn_fp4_bwd_ws_bytes(int B, int H, int N, int D);
int sage_attn_fp4_bwd(const void *Q, const void *K, const void *V, const void *O, const float *LSE, const void *dO,
                      void *dQ, void *dK, void *dV, const void *ws, void *bwd_ws, size_t bwd_ws_bytes, int B, int H,
                      int N, int D, int causal, int qk_norm, int k_smooth, float sm_scale, void *stream);

/* Fill `views` with the device pointers inside a quantize workspace (qmean, dsb: NULL). */
int sage_attn_ws_views(void *ws, int B, int H, int N, int D, sage_ws_views *views);

/* Synchronise `stream`, read and clear the workspace status word.  Returns SAGE_OK
 * or SAGE_ERR_TIMEOUT (or SAGE_ERR_CUDA if the read itself failed). */
int sage_attn_get_status(void *ws, void *stream);

/* Self-test of the bounded wait: launches one CTA that waits on a barrier nothing
 * arrives at, with a budget of `budget_ns` nanoseconds (capped at 1 s); the kernel
 * gives up, records SAGE_ERR_TIMEOUT in the status word of `ws` and returns. */
int sage_attn_selftest_wait(void *ws, unsigned long long budget_ns, void *stream);

/* Size of the library-owned scratch array used by sage_attn_bwd_noalloc. */
#define SAGE_ATTN_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * Backward without a caller-supplied scratch buffer.  The pages have no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory: code running while a CUDA graph is being captured (where a fresh
 * allocation is not allowed), hosts whose memory pool owns every device byte and
 * forbids allocations from extensions, and real-time or embedded deployments
 * that allocate nothing after start-up.  They still pass the inputs, outputs and
 * the quantize workspace, exactly as for sage_attn_bwd, and get the same result.
 *
 * The scratch is one fixed array of SAGE_ATTN_NOALLOC_SCRATCH_BYTES inside the
 * library; every GPU that loads the library holds it until the process exits.
 * Shapes whose scratch (sage_attn_bwd_ws_bytes) exceeds it are rejected with
 * SAGE_ERR_UNSUPPORTED before anything is launched.  The call allocates nothing.
 * Its first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture.
 * Every call shares the one array and each call clears what must start at zero,
 * so calls are independent in sequence, but calls that overlap on the GPU (on
 * different streams, or from several threads) race on the array.
 */
int sage_attn_bwd_noalloc(const void *Q, const void *K, const void *V, const void *O, const float *LSE,
                          const void *dO, void *dQ, void *dK, void *dV, const void *ws, int B, int H,
                          int N, int D, int causal, int qk_norm, int k_smooth, float sm_scale,
                          void *stream);

/*
 * One training step of the attention block on HOST-resident tensors: the quantize
 * pass, the forward and the backward above, with the host<->device copies overlapped
 * with the computation.  Every pass of the scheme treats heads independently, so the
 * B*H heads are split into `groups` contiguous ranges (groups <= 0: automatic, 5 or
 * fewer; at most 64; with 3 ranges or more the first and last hold half the heads of the
 * others): the inputs of all ranges are copied in on one copy stream, range g
 * runs on `stream` once its inputs have landed, and its outputs are copied out on a
 * second copy stream while range g+1 runs.  The results equal those of the three calls
 * on device tensors.
 *  - Q, K, V, dO: host bf16 [B, H, N, D] (read).  O, dQ, dK, dV: host bf16 [B, H, N, D]
 *    and LSE: host fp32 [B, H, N] (written).  Page-locked host memory lets the copies
 *    run asynchronously; with pageable memory the call is correct but the copies do
 *    not overlap the computation.
 *  - dev: device scratch, 256-byte aligned, of sage_attn_step_host_bytes(B, H, N, D,
 *    groups) bytes (the same `groups`): device copies of the inputs and outputs and
 *    the workspaces of one head range.  It begins with a quantize workspace whose
 *    status word collects the errors of every range: read it with
 *    sage_attn_get_status(dev, stream).
 *  - Returns once everything is enqueued; the outputs are in host memory when work
 *    enqueued on `stream` before the next call completes (e.g. after
 *    cudaStreamSynchronize(stream)).  The library's two copy streams are shared by all
 *    calls of the process: calls from several host threads at once are not supported.
 */
size_t sage_attn_step_host_bytes(int B, int H, int N, int D, int groups);
int sage_attn_step_host(const void *Q, const void *K, const void *V, const void *dO, void *O, float *LSE,
                        void *dQ, void *dK, void *dV, void *dev, size_t dev_bytes, int B, int H, int N,
                        int D, int causal, int qk_norm, int k_smooth, float sm_scale, int groups,
                        void *stream);

/* Kernel timing for benchmarks.  While enabled (on != 0) the library brackets
 * each launch group with CUDA events recorded on the launching stream: "quantize"
 * (the two quantize kernels), "fwd", "bwd_pre" (D_i, LSE*log2e, dO codes),
 * "bwd_main" and "bwd_dq".  Costs two event records per group; off by default. */
int sage_attn_timer_enable(int on);

/* Restrict the timing to the launch group `kernel` (one of the names above; NULL:
 * every group).  An event recorded between two launches orders the second after the
 * first's completion, so timing every group removes the overlap of each launch with
 * its predecessor's tail; timing one group keeps it everywhere else. */
int sage_attn_timer_only(const char *kernel);

/* Synchronise the events recorded for `kernel` since the last read, store their
 * summed duration (ms) and number of launches, and forget them.  Unknown names
 * give zero. */
int sage_attn_timer_read(const char *kernel, double *total_ms, int *launches);

/* Static description of a status code. */
const char *sage_attn_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* SAGE_ATTN_H */
