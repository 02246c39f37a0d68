/*
 * CPU oracle of SageBwd-style low-bit attention (forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the bench's CPU
 * baseline leg are the only callers.  It shares no code, header, table or
 * constant with the CUDA path and never calls it.
 *
 * What it computes, and where that is defined:
 *  - "SageBwd: A Trainable Low-bit Attention" (euno.news summary, Methodology
 *    1-2): six of the seven attention matmuls run quantized (QK^T and PV in the
 *    forward; S recompute, dV, dQ, dK in the backward); the softmax-gradient
 *    matmul dP = dO V^T stays in high precision.  Methodology 4 / Results:
 *    QK-norm (unit-norm q and k per token before the dot product) and
 *    K-smoothing.  K-smoothing is read as subtracting the per-(b,h) channel mean
 *    of K over tokens, the only softmax-invariant reading of "smoothing K".
 *  - "Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (gist.science
 *    summary, Methodology, principle 1): the backward recomputes P from the
 *    saved log-sum-exp L in the same low precision as the forward.
 *  - "ThriftAttention" (gist.science summary, Methodology step 2): the
 *    FlashAttention-2 online softmax that merges key tiles into one output.
 *  - The quantization granularity (Q per 128-token block, K per 64-token block,
 *    symmetric INT8 with scale max|x|/127; FP8 e4m3 for P, V and dO) is the
 *    plainest scheme consistent with those pages; they print no formula for it.
 *
 * Precision: softmax, accumulations and the dP matmul in fp64; integer dot
 * products of the INT8 codes exact; every value the scheme stores in fp32 (the
 * scales, the normalised q/k, the smoothed k, the logits, the probabilities
 * before FP8 rounding) rounded to fp32 with round-to-nearest-even.  Build with
 * -ffp-contract=off and without -ffast-math so that each written operation is
 * one IEEE operation.
 *
 * Quantizer mask (qmask): each bit switches one quantizer on; all bits off
 * turns the same code into exact fp64 attention, which the tests compare with
 * textbook attention and finite differences.  QM_FP4 selects the NVFP4 variant
 * (P and V in block-scaled FP4 instead of e4m3; "Attn-QAT" trains attention in
 * FP4 and recomputes P in the backward in the forward's precision, principle 1).
 *
 * Parity status: every function below is pinned by the CPU tests (e4m3 rounding
 * exhaustively against a library cast; the quantizers-off path against library
 * attention and autograd and against finite differences; the quantized path on
 * inputs it must reproduce exactly; invariants).  The exact FP8/INT8 codes on
 * random inputs have no printed worked example to pin them to.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QM_QK 1   /* INT8 codes for Q and K (forward QK^T, backward S, dQ, dK) */
#define QM_V 2    /* e4m3 codes for V (forward PV) */
#define QM_P 4    /* e4m3 codes for P (forward PV, backward dV and dS) */
#define QM_DO 8   /* e4m3 codes for dO (backward dV) */
#define QM_DS 16  /* INT8 codes for dS (backward dQ, dK) */
#define QM_F32 32 /* fp32 rounding of the stored intermediate values */
#define QM_FP4 64 /* NVFP4 in place of e4m3 for V and P (the forward PV, P^ in the backward) */

#define QBLK 128  /* Q tokens per INT8 scale */
#define KBLK 64   /* K tokens per INT8 scale */
#define TILE 128  /* keys per online-softmax step */

static const double LOG2E = 1.4426950408889634074;
static const double LN2 = 0.69314718055994530942;

static inline double r32(int on, double x) { return on ? (double)(float)x : x; }

/* OCP FP8 E4M3 (bias 7, no infinities, max 448, subnormal step 2^-9):
 * round to nearest, ties to even, saturating to +-448. */
double sage_oracle_e4m3(double x)
{
    double a = fabs(x);
    if (a != a) return x;
    if (a >= 448.0) return copysign(448.0, x);
    if (a == 0.0) return x;
    int e;
    frexp(a, &e);          /* a = f * 2^e, f in [0.5, 1) */
    int E = e - 1;         /* floor(log2 a) */
    if (E < -6) E = -6;    /* subnormals share the quantum of the lowest binade */
    double quantum = ldexp(1.0, E - 3);
    double r = nearbyint(a / quantum) * quantum;
    if (r > 448.0) r = 448.0;
    return copysign(r, x);
}

/* e2m1 (FP4) rounding: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (one exponent pair of bits,
 * one mantissa bit, subnormal 0.5); round to nearest with ties to the even mantissa,
 * saturating at 6.  The spacing is 0.5 below 2, 1 in [2, 4) and 2 from 4, and the parity
 * of the count of spacings is the mantissa bit. */
double sage_oracle_e2m1(double x)
{
    double a = fabs(x);
    if (a != a) return x;
    double quantum = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    double r = nearbyint(a / quantum) * quantum;
    if (r > 6.0) r = 6.0;
    return copysign(r, x);
}

void sage_oracle_e2m1_f64(const double *x, double *y, long n)
{
    for (long i = 0; i < n; ++i) y[i] = sage_oracle_e2m1(x[i]);
}

void sage_oracle_e4m3_f32(const float *x, float *y, long n)
{
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i) y[i] = (float)sage_oracle_e4m3((double)x[i]);
}

/* fp64 -> fp32 (nearest even) -> bf16 (nearest even), returned as a double */
static double bf16_round(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) != 0x7f800000u) u += 0x7fffu + ((u >> 16) & 1u);
    u &= 0xffff0000u;
    memcpy(&f, &u, 4);
    return (double)f;
}

void sage_oracle_to_bf16(const double *x, double *y, long n)
{
    for (long i = 0; i < n; ++i) y[i] = bf16_round(x[i]);
}

/* Symmetric per-block INT8: scale = max|x| / 127 over `blk` consecutive tokens
 * (all D channels), code = round-half-even(x / scale) clamped to [-127, 127]. */
static void block_int8(const double *x, int N, int D, int blk, int on, int f32,
                       double *codes, double *scales)
{
    int nb = (N + blk - 1) / blk;
    for (int b = 0; b < nb; ++b) {
        int t0 = b * blk, t1 = t0 + blk < N ? t0 + blk : N;
        if (!on) {
            scales[b] = 1.0;
            memcpy(codes + (size_t)t0 * D, x + (size_t)t0 * D, sizeof(double) * (size_t)(t1 - t0) * D);
            continue;
        }
        double a = 0.0;
        for (size_t i = (size_t)t0 * D; i < (size_t)t1 * D; ++i) a = fmax(a, fabs(x[i]));
        double s = r32(f32, a / 127.0);
        scales[b] = a > 0.0 ? s : 0.0;
        for (size_t i = (size_t)t0 * D; i < (size_t)t1 * D; ++i) {
            if (a == 0.0) { codes[i] = 0.0; continue; }
            double c = nearbyint(r32(f32, x[i] / s));
            codes[i] = c > 127.0 ? 127.0 : (c < -127.0 ? -127.0 : c);
        }
    }
}

/* Per-channel e4m3: scale = max_t |x[t,d]| / 448, code = e4m3(x / scale). */
static void channel_e4m3(const double *x, int N, int D, int on, int f32,
                         double *codes, double *scales)
{
    for (int d = 0; d < D; ++d) {
        if (!on) {
            scales[d] = 1.0;
            for (int t = 0; t < N; ++t) codes[(size_t)t * D + d] = x[(size_t)t * D + d];
            continue;
        }
        double a = 0.0;
        for (int t = 0; t < N; ++t) a = fmax(a, fabs(x[(size_t)t * D + d]));
        double s = r32(f32, a / 448.0);
        scales[d] = a > 0.0 ? s : 0.0;
        for (int t = 0; t < N; ++t) {
            size_t i = (size_t)t * D + d;
            codes[i] = a > 0.0 ? sage_oracle_e4m3(r32(f32, x[i] / s)) : 0.0;
        }
    }
}

/* NVFP4 (the block-scaled FP4 that Blackwell's tensor cores take; "ThriftAttention"
 * (gist.science summary), Methodology step 2, names it for the low-precision path, and the
 * Attn-QAT summary trains attention in FP4): e2m1 codes, one e4m3 scale per 16 consecutive
 * values along the contraction axis, and one fp32 scale for the tensor.
 *
 * V (contracted over keys in PV): per head, g = RN32(max|V| / (448 * 6)); per channel d and
 * block of 16 tokens, s = e4m3(RN32(amax / RN32(6 g))); code = e2m1(RN32(v / RN32(s g))).
 * vx receives the values the matmul sees, code * s * g, and sv = 1 (so that the forward's
 * O = A sv / (448 l) holds with A summing 448 P^ times them). */
static void channel_nvfp4(const double *x, int N, int D, int f32, double *vx, double *sv)
{
    double amax = 0.0;
    for (size_t i = 0; i < (size_t)N * D; ++i) amax = fmax(amax, fabs(x[i]));
    double g = r32(f32, amax / 2688.0);
    double g6 = r32(f32, 6.0 * g);
    for (int d = 0; d < D; ++d) {
        sv[d] = 1.0;
        for (int t0 = 0; t0 < N; t0 += 16) {
            int t1 = t0 + 16 < N ? t0 + 16 : N;
            double a = 0.0;
            for (int t = t0; t < t1; ++t) a = fmax(a, fabs(x[(size_t)t * D + d]));
            double sb = (a > 0.0 && g6 > 0.0) ? sage_oracle_e4m3(r32(f32, a / g6)) : 0.0;
            double sg = r32(f32, sb * g);
            for (int t = t0; t < t1; ++t) {
                size_t i = (size_t)t * D + d;
                vx[i] = sg > 0.0 ? sage_oracle_e2m1(r32(f32, x[i] / sg)) * sb * g : 0.0;
            }
        }
    }
}

/* P in NVFP4 along keys: the values p[k] (k < n <= 16: one block of a row, P or the
 * forward's p~, both <= 1) take the static tensor scale 1 / (448 * 6): with
 * y = RN32(2688 p), s = e4m3(RN32(max y / 6)), code = e2m1(RN32(y / s)).  p8[k] receives
 * 448 P^ = code * s / 6, the scale the e4m3 path's codes carry. */
static void p_block_nvfp4(const double *p, int n, int f32, double *p8)
{
    double ym = 0.0;
    for (int k = 0; k < n; ++k) ym = fmax(ym, r32(f32, 2688.0 * p[k]));
    double sb = ym > 0.0 ? sage_oracle_e4m3(r32(f32, ym / 6.0)) : 0.0;
    for (int k = 0; k < n; ++k)
        p8[k] = sb > 0.0 ? sage_oracle_e2m1(r32(f32, r32(f32, 2688.0 * p[k]) / sb)) * sb / 6.0 : 0.0;
}

/* Per-token L2 normalisation: sigma = sum x^2 (fp64, exact for bf16 inputs),
 * r = 1 / sqrt(sigma) (r = 0 for an all-zero token), x' = x * r. */
static void l2_normalise(const double *x, int N, int D, int f32, double *xn, double *r)
{
    for (int t = 0; t < N; ++t) {
        const double *row = x + (size_t)t * D;
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += row[d] * row[d];
        double sig = r32(f32, s);
        double rt = sig > 0.0 ? r32(f32, 1.0 / r32(f32, sqrt(sig))) : 0.0;
        r[t] = rt;
        for (int d = 0; d < D; ++d) xn[(size_t)t * D + d] = r32(f32, row[d] * rt);
    }
}

/*
 * Quantize one head.  Inputs Q, K, V are [N, D] (row-major, token-major).
 * Outputs: qn/kn the (optionally) normalised q', k' [N, D]; qr/kr the 1/||x||
 * factors [N] (1 when QK-norm is off); kmean [D] (0 when smoothing is off);
 * qx/kx INT8 codes [N, D] with scales sq [ceil(N/128)], sk [ceil(N/64)];
 * vx e4m3 codes [N, D] with per-channel scales sv [D].
 *
 * Q-smoothing (q_smooth; "SageBwd: A Trainable Low-bit Attention", euno.news
 * summary, Methodology 4, names it as the optional companion of K-smoothing and
 * prints no formula).  Read as the query-side smoothing of the SageAttention
 * line: each 128-token query block I loses its channel mean before the INT8
 * quantizer, and the logits get back what the mean carries as a per-(block, key)
 * term kept in high precision:
 *   qmean_I,d = RN32(sum_{t in I} q'_td / |I|)      (valid tokens of the block)
 *   qs_td     = RN32(q'_td - qmean_I,d)             -> INT8 codes qx, scales sq
 *   dsb_I,j   = RN32(sum_d qmean_I,d k''_jd)        (k'' = the smoothed k' that K's
 *                                                    quantizer takes)
 * so that qs.k'' + dsb = q'.k'' exactly in exact arithmetic.  qmean is
 * [ceil(N/128), D], dsb [ceil(N/128), N].
 */
static int quantize_head(int N, int D, const double *Q, const double *K, const double *V,
                         int qk_norm, int k_smooth, int q_smooth, int qmask,
                         double *qn, double *qr, double *kn, double *kr, double *kmean,
                         double *qx, double *sq, double *kx, double *sk,
                         double *vx, double *sv, double *qmean, double *dsb);

int sage_oracle_quantize(int N, int D, const double *Q, const double *K, const double *V,
                         int qk_norm, int k_smooth, int qmask,
                         double *qn, double *qr, double *kn, double *kr, double *kmean,
                         double *qx, double *sq, double *kx, double *sk,
                         double *vx, double *sv)
{
    return quantize_head(N, D, Q, K, V, qk_norm, k_smooth, 0, qmask, qn, qr, kn, kr, kmean,
                         qx, sq, kx, sk, vx, sv, NULL, NULL);
}

int sage_oracle_quantize_qs(int N, int D, const double *Q, const double *K, const double *V,
                            int qk_norm, int k_smooth, int qmask,
                            double *qn, double *qr, double *kn, double *kr, double *kmean,
                            double *qx, double *sq, double *kx, double *sk,
                            double *vx, double *sv, double *qmean, double *dsb)
{
    if (!qmean || !dsb) return 1;
    return quantize_head(N, D, Q, K, V, qk_norm, k_smooth, 1, qmask, qn, qr, kn, kr, kmean,
                         qx, sq, kx, sk, vx, sv, qmean, dsb);
}

static int quantize_head(int N, int D, const double *Q, const double *K, const double *V,
                         int qk_norm, int k_smooth, int q_smooth, int qmask,
                         double *qn, double *qr, double *kn, double *kr, double *kmean,
                         double *qx, double *sq, double *kx, double *sk,
                         double *vx, double *sv, double *qmean, double *dsb)
{
    if (N < 0 || D <= 0) return 1;
    int f32 = (qmask & QM_F32) != 0;
    size_t E = (size_t)N * D;
    if (qk_norm) {
        l2_normalise(Q, N, D, f32, qn, qr);
        l2_normalise(K, N, D, f32, kn, kr);
    } else {
        memcpy(qn, Q, sizeof(double) * E);
        memcpy(kn, K, sizeof(double) * E);
        for (int t = 0; t < N; ++t) qr[t] = kr[t] = 1.0;
    }
    double *ks = (double *)malloc(sizeof(double) * (E ? E : 1));
    if (!ks) return 2;
    for (int d = 0; d < D; ++d) {
        double m = 0.0;
        if (k_smooth && N > 0) {
            double s = 0.0;
            for (int t = 0; t < N; ++t) s += kn[(size_t)t * D + d];
            m = r32(f32, s / N);
        }
        kmean[d] = m;
        for (int t = 0; t < N; ++t) {
            size_t i = (size_t)t * D + d;
            ks[i] = k_smooth ? r32(f32, kn[i] - m) : kn[i];
        }
    }
    if (q_smooth) {
        double *qs = (double *)malloc(sizeof(double) * (E ? E : 1));
        if (!qs) { free(ks); return 2; }
        int nI = (N + QBLK - 1) / QBLK;
        for (int I = 0; I < nI; ++I) {
            int t0 = I * QBLK, t1 = t0 + QBLK < N ? t0 + QBLK : N;
            for (int d = 0; d < D; ++d) {
                double s = 0.0;
                for (int t = t0; t < t1; ++t) s += qn[(size_t)t * D + d];
                double m = r32(f32, s / (t1 - t0));
                qmean[(size_t)I * D + d] = m;
                for (int t = t0; t < t1; ++t) qs[(size_t)t * D + d] = r32(f32, qn[(size_t)t * D + d] - m);
            }
            for (int j = 0; j < N; ++j) {
                double a = 0.0;
                for (int d = 0; d < D; ++d) a += qmean[(size_t)I * D + d] * ks[(size_t)j * D + d];
                dsb[(size_t)I * N + j] = r32(f32, a);
            }
        }
        block_int8(qs, N, D, QBLK, (qmask & QM_QK) != 0, f32, qx, sq);
        free(qs);
    } else {
        block_int8(qn, N, D, QBLK, (qmask & QM_QK) != 0, f32, qx, sq);
    }
    block_int8(ks, N, D, KBLK, (qmask & QM_QK) != 0, f32, kx, sk);
    if (qmask & QM_FP4)
        channel_nvfp4(V, N, D, f32, vx, sv);
    else
        channel_e4m3(V, N, D, (qmask & QM_V) != 0, f32, vx, sv);
    free(ks);
    return 0;
}

/* sum_d qx*kx.  With INT8 codes every product and partial sum is an integer
 * below 2^53, so this fp64 sum is the exact integer dot product. */
static inline double dot(const double *qrow, const double *krow, int D)
{
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qrow[d] * krow[d];
    return acc;
}

/* The dequantization factor of a (query block, key block) pair is
 * c = RN(RN(sq_I * sk_J) * alpha), alpha = RN(sm_scale * log2 e): the
 * log2-domain logit is acc * c. */

static inline double qk_factor(double sqI, double skJ, double alpha, int f32)
{
    return r32(f32, r32(f32, sqI * skJ) * alpha);
}

/*
 * Forward for one head: online softmax over ascending 128-key tiles.
 * Per row and tile, with acc_ij the integer dot product and c the tile's
 * dequantization factor (S2 = acc c, log2 units):
 *   m' = max(m, max_j RN32(acc_ij c));
 *   t = RN32(acc_ij c - m')  (one rounding of the exact value);
 *   p~ = RN32(2^t) (fp64 exp2);  p8 = e4m3(RN32(448 p~));
 *   l = l 2^(m - m') + sum p~;  A = A 2^(m - m') + sum p8 v8.
 * Finish: O = A sv / (448 l), LSE = ln2 (m + log2 l).
 * With Q-smoothing (dsb given, [ceil(N/128), N]) the logit of query i in block I
 * first takes back the block mean's term in natural units,
 *   u_ij = RN32(acc_ij RN32(sq_I sk_J) + dsb_Ij),
 * and u_ij alpha plays the part of acc_ij c above (alpha = RN32(sm_scale log2 e)).
 * Outputs O64 [N, D], O32 [N, D] (float), LSE64 [N].
 */
/* ThriftAttention's promoted tiles ("ThriftAttention" (gist.science summary), Methodology
 * steps 1-2): sel[I * nkt + J] != 0 computes the pair (128-query block I, 128-key tile J) in
 * the high-precision path from qh, kh, vh (the softmax's q', k'' and V rounded to fp16):
 * x = RN32(qh . kh) (fp16 products, one rounding of the sum), the log2 logit RN32(x alpha),
 * P16 = fp16(p~) times vh into an fp32 accumulator of its own; the other tiles take the
 * low-bit path; both merge in the one online softmax (shared m and l).  A row takes its
 * low-bit tiles first and its promoted tiles after them, as the page's kernel does (the
 * non-selected blocks through the low-precision path, then the promoted blocks in a
 * separate high-precision routine); since P is quantized relative to the running maximum,
 * the order is part of the result. */
struct thrift {
    const unsigned char *sel;
    int nkt;
    const double *qh, *kh, *vh;
};

static int fwd_head(int N, int D, int causal, double sm_scale, int qmask,
                    const double *qx, const double *sq, const double *kx, const double *sk,
                    const double *vx, const double *sv, const double *dsb, const struct thrift *th,
                    double *O64, float *O32, double *LSE64);

/* fp16 rounding: 11-bit significand, nearest even, subnormal below 2^-14, saturating at the
 * largest finite 65504 (inputs here stay far below it) */
static double fp16_round(double x)
{
    double a = fabs(x);
    if (a != a || a == 0.0) return x;
    if (a >= 65504.0) return copysign(65504.0, x);
    int e;
    frexp(a, &e);
    int E = e - 1;
    if (E < -14) E = -14;
    double quantum = ldexp(1.0, E - 10);
    return copysign(nearbyint(a / quantum) * quantum, x);
}

void sage_oracle_fp16_f64(const double *x, double *y, long n)
{
    for (long i = 0; i < n; ++i) y[i] = fp16_round(x[i]);
}

int sage_oracle_fwd_thrift(int N, int D, int causal, double sm_scale, int qmask,
                           const double *qx, const double *sq, const double *kx, const double *sk,
                           const double *vx, const double *sv, const unsigned char *sel,
                           const double *qh, const double *kh, const double *vh,
                           double *O64, float *O32, double *LSE64)
{
    if (!sel || !qh || !kh || !vh) return 1;
    struct thrift th = {sel, (N + TILE - 1) / TILE, qh, kh, vh};
    return fwd_head(N, D, causal, sm_scale, qmask, qx, sq, kx, sk, vx, sv, NULL, &th, O64, O32, LSE64);
}

int sage_oracle_fwd(int N, int D, int causal, double sm_scale, int qmask,
                    const double *qx, const double *sq, const double *kx, const double *sk,
                    const double *vx, const double *sv,
                    double *O64, float *O32, double *LSE64)
{
    return fwd_head(N, D, causal, sm_scale, qmask, qx, sq, kx, sk, vx, sv, NULL, NULL, O64, O32, LSE64);
}

int sage_oracle_fwd_qs(int N, int D, int causal, double sm_scale, int qmask,
                       const double *qx, const double *sq, const double *kx, const double *sk,
                       const double *vx, const double *sv, const double *dsb,
                       double *O64, float *O32, double *LSE64)
{
    if (!dsb) return 1;
    return fwd_head(N, D, causal, sm_scale, qmask, qx, sq, kx, sk, vx, sv, dsb, NULL, O64, O32, LSE64);
}

/* The log2-domain logit of query i and key j is RN32(x f) for the value x and
 * factor f this returns: x = acc, f = c without Q-smoothing; x = u, f = alpha
 * with it (see fwd_head). */
static inline double logit_parts(double acc, double sqI, double skJ, double alpha, int f32,
                                 const double *dsb_row, int j, double *f)
{
    if (!dsb_row) {
        *f = qk_factor(sqI, skJ, alpha, f32);
        return acc;
    }
    *f = alpha;
    return r32(f32, acc * r32(f32, sqI * skJ) + dsb_row[j]);
}

static int fwd_head(int N, int D, int causal, double sm_scale, int qmask,
                    const double *qx, const double *sq, const double *kx, const double *sk,
                    const double *vx, const double *sv, const double *dsb, const struct thrift *th,
                    double *O64, float *O32, double *LSE64)
{
    if (N < 0 || D <= 0) return 1;
    int f32 = (qmask & QM_F32) != 0;
    int qp = (qmask & QM_P) != 0;
    double alpha = r32(f32, sm_scale * LOG2E);
    int err = 0;
#pragma omp parallel
    {
        double *A = (double *)malloc(sizeof(double) * 2 * D);
        double *A16 = A ? A + D : NULL;  /* the high-precision tiles' accumulator (true units) */
        /* x, f per key (logit_parts); with NVFP4 also p~ and 448 P^ per key */
        double *s2 = (double *)malloc(sizeof(double) * 4 * TILE);
        if (!A || !s2) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for schedule(dynamic, 8)
        for (int i = 0; i < N; ++i) {
            if (!A || !s2) continue;
            const double *qrow = qx + (size_t)i * D;
            double m = -INFINITY, l = 0.0;
            for (int d = 0; d < D; ++d) A[d] = A16[d] = 0.0;
            /* ThriftAttention: the low-bit tiles first, then the promoted ones (pass 1), each
             * pass in ascending key order; without it one pass over every tile */
            for (int pass = 0; pass < (th ? 2 : 1); ++pass)
            for (int j0 = 0; j0 < N; j0 += TILE) {
                int j1 = j0 + TILE < N ? j0 + TILE : N;
                if (causal && j1 > i + 1) j1 = i + 1;
                if (j1 <= j0) break;
                const int hp = th && th->sel[(size_t)(i / QBLK) * th->nkt + j0 / TILE];
                if (th && hp != pass) continue;
                double mt = -INFINITY;
                double *acc = s2, *cj = s2 + TILE;
                const double *dsb_row = dsb ? dsb + (size_t)(i / QBLK) * N : NULL;
                for (int j = j0; j < j1; ++j) {
                    double c;
                    if (hp) {
                        acc[j - j0] = r32(f32, dot(th->qh + (size_t)i * D, th->kh + (size_t)j * D, D));
                        c = alpha;
                    } else {
                        acc[j - j0] = logit_parts(dot(qrow, kx + (size_t)j * D, D), sq[i / QBLK], sk[j / KBLK],
                                                  alpha, f32, dsb_row, j, &c);
                    }
                    cj[j - j0] = c;
                    mt = fmax(mt, r32(f32, acc[j - j0] * c));
                }
                double mn = fmax(m, mt);
                double corr = (m == -INFINITY) ? 0.0 : exp2(m - mn);
                l *= corr;
                for (int d = 0; d < D; ++d) {
                    A[d] *= corr;
                    A16[d] *= corr;
                }
                if (hp) {
                    for (int j = j0; j < j1; ++j) {
                        double pt = r32(f32, exp2(r32(f32, acc[j - j0] * cj[j - j0] - mn)));
                        double p16 = fp16_round(pt);
                        l += pt;
                        const double *vrow = th->vh + (size_t)j * D;
                        for (int d = 0; d < D; ++d) A16[d] += p16 * vrow[d];
                    }
                } else if (qmask & QM_FP4) {
                    /* p~ of the tile's keys, then NVFP4 per block of 16 keys (blocks start at
                     * multiples of 16; keys past the causal limit are not in any block) */
                    double *ptv = s2 + 2 * TILE, *p8v = s2 + 3 * TILE;
                    for (int j = j0; j < j1; ++j) {
                        ptv[j - j0] = r32(f32, exp2(r32(f32, acc[j - j0] * cj[j - j0] - mn)));
                        l += ptv[j - j0];
                    }
                    for (int b0 = j0; b0 < j1; b0 += 16)
                        p_block_nvfp4(ptv + (b0 - j0), (b0 + 16 < j1 ? b0 + 16 : j1) - b0, f32, p8v + (b0 - j0));
                    for (int j = j0; j < j1; ++j) {
                        const double *vrow = vx + (size_t)j * D;
                        for (int d = 0; d < D; ++d) A[d] += p8v[j - j0] * vrow[d];
                    }
                } else {
                    for (int j = j0; j < j1; ++j) {
                        double t = r32(f32, acc[j - j0] * cj[j - j0] - mn);
                        double pt = r32(f32, exp2(t));
                        double p8 = qp ? sage_oracle_e4m3(r32(f32, 448.0 * pt)) : 448.0 * pt;
                        l += pt;
                        const double *vrow = vx + (size_t)j * D;
                        for (int d = 0; d < D; ++d) A[d] += p8 * vrow[d];
                    }
                }
                m = mn;
            }
            for (int d = 0; d < D; ++d) {
                double o = (A[d] * sv[d] / 448.0 + A16[d]) / l;
                O64[(size_t)i * D + d] = o;
                O32[(size_t)i * D + d] = (float)o;
            }
            LSE64[i] = LN2 * (m + log2(l));
        }
        free(A);
        free(s2);
    }
    return err;
}

/* One (128-query block I, 64-key block J) tile of the backward.
 * P = RN32(2^RN32(acc c - RN32(LSE log2 e))), p8 = e4m3(RN32(448 P)), P^ = p8 / 448,
 * dP = dO V^T (fp64, unquantized), dS = RN32(P^ (dP - Dvec)),
 * dS8 = INT8 of dS with one scale max|dS|/127 for the tile.
 * With Q-smoothing (dsb given) the logit is formed as in the forward (logit_parts).
 * p8t/ds8t are [QBLK][KBLK]; returns the tile's dS scale. */
static double bwd_tile(int I, int J, int N, int D, int causal, double alpha, int qmask,
                       const double *qx, const double *sq, const double *kx, const double *sk,
                       const double *V, const double *dO, const double *lse2, const double *Dv,
                       const double *dsb, double *p8t, double *ds8t)
{
    int f32 = (qmask & QM_F32) != 0;
    int i0 = I * QBLK, i1 = i0 + QBLK < N ? i0 + QBLK : N;
    int j0 = J * KBLK, j1 = j0 + KBLK < N ? j0 + KBLK : N;
    double amax = 0.0;
    const double *dsb_row = dsb ? dsb + (size_t)I * N : NULL;
    for (int i = i0; i < i1; ++i) {
        /* the row's P on this key block (0 past the causal limit), then 448 P^: e4m3 codes, or
         * NVFP4 per 16 keys as in the forward */
        double Pr[KBLK], p8r[KBLK];
        for (int j = j0; j < j1; ++j) {
            if (causal && j > i) { Pr[j - j0] = 0.0; continue; }
            double c;
            double x = logit_parts(dot(qx + (size_t)i * D, kx + (size_t)j * D, D), sq[I], sk[J], alpha, f32,
                                   dsb_row, j, &c);
            Pr[j - j0] = r32(f32, exp2(r32(f32, x * c - lse2[i])));
        }
        if (qmask & QM_FP4) {
            for (int b0 = j0; b0 < j1; b0 += 16)
                p_block_nvfp4(Pr + (b0 - j0), (b0 + 16 < j1 ? b0 + 16 : j1) - b0, f32, p8r + (b0 - j0));
        } else {
            for (int j = j0; j < j1; ++j)
                p8r[j - j0] = (qmask & QM_P) ? sage_oracle_e4m3(r32(f32, 448.0 * Pr[j - j0])) : 448.0 * Pr[j - j0];
        }
        for (int j = j0; j < j1; ++j) {
            double *pp = p8t + (size_t)(i - i0) * KBLK + (j - j0);
            double *dd = ds8t + (size_t)(i - i0) * KBLK + (j - j0);
            if (causal && j > i) { *pp = 0.0; *dd = 0.0; continue; }
            double p8 = p8r[j - j0];
            double dp = 0.0;
            for (int d = 0; d < D; ++d) dp += dO[(size_t)i * D + d] * V[(size_t)j * D + d];
            double ds = r32(f32, (p8 / 448.0) * (dp - Dv[i]));
            *pp = p8;
            *dd = ds;
            amax = fmax(amax, fabs(ds));
        }
    }
    if (!(qmask & QM_DS)) return 1.0;
    double s = amax > 0.0 ? r32(f32, amax / 127.0) : 0.0;
    for (int i = i0; i < i1; ++i)
        for (int j = j0; j < j1; ++j) {
            double *dd = ds8t + (size_t)(i - i0) * KBLK + (j - j0);
            if (s == 0.0) { *dd = 0.0; continue; }
            double q = nearbyint(r32(f32, *dd / s));
            *dd = q > 127.0 ? 127.0 : (q < -127.0 ? -127.0 : q);
        }
    return s;
}

/* dx = r (dx' - x' (x' . dx')): gradient through x' = x / ||x||. */
static void l2_normalise_grad(double *g, const double *xn, const double *r, int N, int D)
{
    for (int t = 0; t < N; ++t) {
        double *gr = g + (size_t)t * D;
        const double *xr = xn + (size_t)t * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += xr[d] * gr[d];
        for (int d = 0; d < D; ++d) gr[d] = r[t] * (gr[d] - xr[d] * dot);
    }
}

/*
 * Backward for one head.  V, dO are the unquantized inputs [N, D]; O the
 * forward output used for Dvec_i = sum_d dO O; LSE the forward's natural-log
 * LSE [N].  Codes and scales as returned by sage_oracle_quantize.
 * dV_j  = (s_dO,d / 448) sum_i p8_ij dO8_id
 * dQ_i += RN32(s_dS sk_J) sum_j dS8_ij kx_jd          (per tile)
 * dK_j += RN32(s_dS sq_I) sum_i dS8_ij qx_id          (per tile)
 * then dQ, dK scaled by sm_scale, and passed back through QK-norm; the
 * K-smoothing Jacobian (I - 11^T/N) is applied as the identity: the exact dS
 * rows sum to zero, so the smoothed-K gradient already has zero token mean.
 * With Q-smoothing (dsb and qmean given) the codes qx are those of q' - qmean_I,
 * and the keys' gradient takes back the mean's share of S = (q' - qmean) k'' +
 * qmean k'', per tile:
 *   dK_j += s_dS (sum_i dS8_ij) qmean_I
 * (the dequantized dS of the tile, summed over its queries).  dQ needs no such
 * term: the mean's gradient through qmean_I and through q' - qmean_I cancel.
 * Outputs dQ, dK, dV [N, D] and Dvec [N] in fp64.
 */
static int bwd_head(int N, int D, int causal, double sm_scale, int qk_norm, int qmask,
                    const double *V, const double *dO, const double *O, const double *LSE,
                    const double *qx, const double *sq, const double *kx, const double *sk,
                    const double *qn, const double *qr, const double *kn, const double *kr,
                    const double *sdo_in, const double *dsb, const double *qmean,
                    double *dQ, double *dK, double *dV, double *Dvec);

int sage_oracle_bwd(int N, int D, int causal, double sm_scale, int qk_norm, int qmask,
                    const double *V, const double *dO, const double *O, const double *LSE,
                    const double *qx, const double *sq, const double *kx, const double *sk,
                    const double *qn, const double *qr, const double *kn, const double *kr,
                    double *dQ, double *dK, double *dV, double *Dvec)
{
    return bwd_head(N, D, causal, sm_scale, qk_norm, qmask, V, dO, O, LSE, qx, sq, kx, sk, qn, qr, kn, kr,
                    NULL, NULL, NULL, dQ, dK, dV, Dvec);
}

/*
 * The same backward with the channel scales of dO given (sdo_in[D]) instead of taken
 * from this head's dO.  Grouped-query attention: the query heads that share one
 * key/value head put their dO tokens on one axis for dV = sum_i P_ij dO_i, so its
 * e4m3 channel scale spans all of them (the caller computes it as for one head).
 */
int sage_oracle_bwd_sdo(int N, int D, int causal, double sm_scale, int qk_norm, int qmask,
                        const double *V, const double *dO, const double *O, const double *LSE,
                        const double *qx, const double *sq, const double *kx, const double *sk,
                        const double *qn, const double *qr, const double *kn, const double *kr,
                        const double *sdo_in, double *dQ, double *dK, double *dV, double *Dvec)
{
    return bwd_head(N, D, causal, sm_scale, qk_norm, qmask, V, dO, O, LSE, qx, sq, kx, sk, qn, qr, kn, kr,
                    sdo_in, NULL, NULL, dQ, dK, dV, Dvec);
}

/* The backward with Q-smoothing: dsb [ceil(N/128), N] and qmean [ceil(N/128), D] as
 * sage_oracle_quantize_qs returns them; sdo_in as in sage_oracle_bwd_sdo, or NULL. */
int sage_oracle_bwd_qs(int N, int D, int causal, double sm_scale, int qk_norm, int qmask,
                       const double *V, const double *dO, const double *O, const double *LSE,
                       const double *qx, const double *sq, const double *kx, const double *sk,
                       const double *qn, const double *qr, const double *kn, const double *kr,
                       const double *sdo_in, const double *dsb, const double *qmean,
                       double *dQ, double *dK, double *dV, double *Dvec)
{
    if (!dsb || !qmean) return 1;
    return bwd_head(N, D, causal, sm_scale, qk_norm, qmask, V, dO, O, LSE, qx, sq, kx, sk, qn, qr, kn, kr,
                    sdo_in, dsb, qmean, dQ, dK, dV, Dvec);
}

static int bwd_head(int N, int D, int causal, double sm_scale, int qk_norm, int qmask,
                    const double *V, const double *dO, const double *O, const double *LSE,
                    const double *qx, const double *sq, const double *kx, const double *sk,
                    const double *qn, const double *qr, const double *kn, const double *kr,
                    const double *sdo_in, const double *dsb, const double *qmean,
                    double *dQ, double *dK, double *dV, double *Dvec)
{
    if (N < 0 || D <= 0) return 1;
    int f32 = (qmask & QM_F32) != 0;
    double alpha = r32(f32, sm_scale * LOG2E);
    size_t E = (size_t)N * D;
    double *lse2 = (double *)malloc(sizeof(double) * (N ? N : 1));
    double *do8 = (double *)malloc(sizeof(double) * (E ? E : 1));
    double *sdo = (double *)malloc(sizeof(double) * D);
    if (!lse2 || !do8 || !sdo) { free(lse2); free(do8); free(sdo); return 2; }

    for (int i = 0; i < N; ++i) {
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += dO[(size_t)i * D + d] * O[(size_t)i * D + d];
        Dvec[i] = s;
        lse2[i] = r32(f32, LSE[i] * LOG2E);
    }
    if (sdo_in && (qmask & QM_DO)) {
        /* e4m3(x / s) with the given channel scale, as channel_e4m3 forms it */
        for (int d = 0; d < D; ++d) {
            sdo[d] = sdo_in[d];
            for (int t = 0; t < N; ++t) {
                size_t i = (size_t)t * D + d;
                do8[i] = sdo[d] > 0.0 ? sage_oracle_e4m3(r32(f32, dO[i] / sdo[d])) : 0.0;
            }
        }
    } else {
        channel_e4m3(dO, N, D, (qmask & QM_DO) != 0, f32, do8, sdo);
    }
    memset(dQ, 0, sizeof(double) * E);
    memset(dK, 0, sizeof(double) * E);
    memset(dV, 0, sizeof(double) * E);
    int nI = (N + QBLK - 1) / QBLK, nJ = (N + KBLK - 1) / KBLK;
    int err = 0;

    /* dQ: one query block per task, all key blocks in order */
#pragma omp parallel
    {
        double *p8t = (double *)malloc(sizeof(double) * QBLK * KBLK);
        double *ds8t = (double *)malloc(sizeof(double) * QBLK * KBLK);
        double *acc = (double *)malloc(sizeof(double) * 2 * D);
        double *acc2 = acc ? acc + D : NULL;
        if (!p8t || !ds8t || !acc) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int I = 0; I < nI; ++I) {
            if (!p8t || !ds8t || !acc) continue;
            int i0 = I * QBLK, i1 = i0 + QBLK < N ? i0 + QBLK : N;
            for (int J = 0; J < nJ; ++J) {
                if (causal && J * KBLK > i1 - 1) break;
                double s = bwd_tile(I, J, N, D, causal, alpha, qmask, qx, sq, kx, sk, V, dO,
                                    lse2, Dvec, dsb, p8t, ds8t);
                double c = r32(f32, s * sk[J]);
                int j0 = J * KBLK, j1 = j0 + KBLK < N ? j0 + KBLK : N;
                for (int i = i0; i < i1; ++i) {
                    /* acc_d = sum_j dS8_ij kx_jd, j ascending */
                    for (int d = 0; d < D; ++d) acc[d] = 0.0;
                    for (int j = j0; j < j1; ++j) {
                        double t = ds8t[(size_t)(i - i0) * KBLK + (j - j0)];
                        const double *kr_ = kx + (size_t)j * D;
                        for (int d = 0; d < D; ++d) acc[d] += t * kr_[d];
                    }
                    for (int d = 0; d < D; ++d) dQ[(size_t)i * D + d] += c * acc[d];
                }
            }
        }
        free(p8t);
        free(ds8t);
        free(acc);
        (void)acc2;
    }
    /* dK, dV: one key block per task, all query blocks in order */
#pragma omp parallel
    {
        double *p8t = (double *)malloc(sizeof(double) * QBLK * KBLK);
        double *ds8t = (double *)malloc(sizeof(double) * QBLK * KBLK);
        double *acc = (double *)malloc(sizeof(double) * 2 * D);
        double *acc2 = acc ? acc + D : NULL;
        if (!p8t || !ds8t || !acc) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int J = 0; J < nJ; ++J) {
            if (!p8t || !ds8t || !acc) continue;
            int j0 = J * KBLK, j1 = j0 + KBLK < N ? j0 + KBLK : N;
            for (int I = 0; I < nI; ++I) {
                int i0 = I * QBLK, i1 = i0 + QBLK < N ? i0 + QBLK : N;
                if (causal && j0 > i1 - 1) continue;
                double s = bwd_tile(I, J, N, D, causal, alpha, qmask, qx, sq, kx, sk, V, dO,
                                    lse2, Dvec, dsb, p8t, ds8t);
                double c = r32(f32, s * sq[I]);
                for (int j = j0; j < j1; ++j) {
                    /* acck_d = sum_i dS8_ij qx_id, accv_d = sum_i p8_ij dO8_id, i ascending */
                    for (int d = 0; d < D; ++d) { acc[d] = 0.0; acc2[d] = 0.0; }
                    double colsum = 0.0;
                    for (int i = i0; i < i1; ++i) {
                        size_t t = (size_t)(i - i0) * KBLK + (j - j0);
                        double a = ds8t[t], p = p8t[t];
                        const double *qrow = qx + (size_t)i * D, *orow = do8 + (size_t)i * D;
                        colsum += a;
                        for (int d = 0; d < D; ++d) {
                            acc[d] += a * qrow[d];
                            acc2[d] += p * orow[d];
                        }
                    }
                    for (int d = 0; d < D; ++d) {
                        dK[(size_t)j * D + d] += c * acc[d];
                        if (qmean) dK[(size_t)j * D + d] += s * colsum * qmean[(size_t)I * D + d];
                        dV[(size_t)j * D + d] += (sdo[d] / 448.0) * acc2[d];
                    }
                }
            }
        }
        free(p8t);
        free(ds8t);
        free(acc);
        (void)acc2;
    }
    for (size_t i = 0; i < E; ++i) {
        dQ[i] *= sm_scale;
        dK[i] *= sm_scale;
    }
    if (qk_norm) {
        l2_normalise_grad(dQ, qn, qr, N, D);
        l2_normalise_grad(dK, kn, kr, N, D);
    }
    free(lse2);
    free(do8);
    free(sdo);
    return err;
}
