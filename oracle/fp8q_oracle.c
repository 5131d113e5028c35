/*
 * fp8q oracle -- plain, slow CPU restatement of FP8 scaled quantization and
 * the scaled GEMM that consumes it.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  The
 * product (the CUDA library under fp8_scaled_quantization_quantize_gb300/)
 * never calls it, and the two share no code, header, table or constant.
 *
 * Sources (the four web pages on FP8 training):
 *   - "2025 FP8 quantized-training guide" (blog.gitcode.com), sec. 1.1: the
 *     E4M3 (1 sign / 4 exponent / 3 mantissa) and E5M2 (1/5/2) layouts and the
 *     PyTorch dtypes torch.float8_e4m3fn / torch.float8_e5m2 they map to;
 *     sec. 2.1: per-tensor delayed (amax history) and current scaling;
 *     sec. 2.2: blockwise 1x128 (inputs, gradients) and 128x128 (weights)
 *     tiles with one scale per tile; sec. 2.3: MXFP8, 1x32 blocks with an
 *     8-bit-exponent / 0-mantissa (E8M0) scale; sec. 3.1: fprop / dgrad /
 *     wgrad GEMMs take quantized inputs and produce BF16/FP32 outputs.
 *   - bjdmk.com.cn/news/5220490, sec. 2: E5M2 bias 15, max 57344;
 *     sec. 3.3: DelayedScaling(margin=0, interval=1).
 *   - "mastering FP8 LLM training 1.5x speedup" (nmedialink.com), scaling
 *     strategies 1-4: delayed, current, sub-channel block, MXFP8 with E8M0
 *     power-of-two scales over fixed 32-value blocks.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - FP8 codes follow torch.float8_e4m3fn (bias 7, max 448, subnormals to
 *     2^-9, no Inf, NaN = S.1111.111) and torch.float8_e5m2 (bias 15, max
 *     57344, subnormals to 2^-16, Inf = S.11111.00, NaN otherwise).
 *   - The cast is saturating round-to-nearest-even: round the fp32 value to
 *     the format's grid (ties to the even code), clamp finite overflow and
 *     +-Inf to +-max, NaN -> S.1111111 (sign kept).
 *   - Per-tensor: s = fmax / amax (fp32 division) multiplies x; amax = 0 -> s = 1;
 *     s = +Inf -> FLT_MAX; the GEMM dequantizes with s_inv = fp32(1 / s).
 *   - Blockwise: d = amax / fmax (fp32 division) divides x and dequantizes;
 *     amax = 0 -> d = 1; a d that underflows to 0 -> 2^-149.
 *   - MXFP8: e = floor(log2 amax) - emax_elem (8 for E4M3, 15 for E5M2),
 *     clamped to [-127, 127]; amax = 0 -> e = 0; E8M0 code = e + 127;
 *     x is multiplied by 2^-e (exact) and 2^e dequantizes.
 *   - amax covers the finite elements of the block; NaN/Inf are counted as
 *     nonfinite.  Saturated = finite x whose scaled fp32 value exceeds fmax.
 *   - Delayed: step t casts with the scale from the history of steps < t,
 *     then records amax_t, rolls the ring and sets
 *     s = fmax / max(history) * 2^-margin (amax 0 -> 1; a product below
 *     the smallest normal fp32 is raised to it, so 1 / s stays finite); a
 *     step with a nonfinite input leaves the state unchanged.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -fPIC -shared (no
 * fused multiply-add contraction, so every fp32 operation rounds on its own).
 * OpenMP only splits independent work across host threads: blocks of a
 * quantizer, elements of a per-tensor cast, output points of the GEMM.  Each
 * block, element and point is computed exactly as in a serial loop (a GEMM
 * point still sums k = 0..K-1 in order), and what is combined across threads
 * is a maximum or a count, so the results do not depend on the thread count
 * (orc_set_threads(1) gives the single-core oracle).
 */
#include <float.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_E4M3 0
#define ORC_E5M2 1

/* Largest finite magnitude, mantissa bits, exponent bias, and the exponent of
 * the largest binade of each format. */
static double orc_fmax(int fmt) { return fmt == ORC_E4M3 ? 448.0 : 57344.0; }
static int orc_mbits(int fmt) { return fmt == ORC_E4M3 ? 3 : 2; }
static int orc_bias(int fmt) { return fmt == ORC_E4M3 ? 7 : 15; }
static int orc_emax_elem(int fmt) { return fmt == ORC_E4M3 ? 8 : 15; }

/* ---------------------------------------------------------------- decode */

/* Value of an FP8 code, exactly, as a double (sec. 1.1 bit layouts). */
double orc_fp8_decode(uint8_t code, int fmt)
{
    int mbits = orc_mbits(fmt);
    int ebits = 7 - mbits;
    int bias = orc_bias(fmt);
    int sign = code >> 7;
    int e = (code >> mbits) & ((1 << ebits) - 1);
    int m = code & ((1 << mbits) - 1);
    double v;
    if (fmt == ORC_E4M3 && e == 15 && m == 7) {
        v = NAN;
    } else if (fmt == ORC_E5M2 && e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        /* subnormal: 0.m * 2^(1 - bias) */
        v = ldexp((double)m, 1 - bias - mbits);
    } else {
        /* normal: 1.m * 2^(e - bias) */
        v = ldexp((double)((1 << mbits) + m), e - bias - mbits);
    }
    return sign ? -v : v;
}

/* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits. */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ---------------------------------------------------------------- encode */

/* Saturating round-to-nearest-even cast of an fp32 value to an FP8 code. */
uint8_t orc_fp8_encode(float v, int fmt)
{
    uint32_t bits;
    memcpy(&bits, &v, 4);
    uint8_t sign = (uint8_t)((bits >> 24) & 0x80u);
    int mbits = orc_mbits(fmt);
    int bias = orc_bias(fmt);
    int emin = 1 - bias;                     /* exponent of the smallest normal */
    double fmax = orc_fmax(fmt);

    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    double a = fabs((double)v);
    if (a >= fmax) {
        /* +-Inf and everything at or above the largest finite value: the
         * rounded result is either fmax or beyond it, and beyond clamps. */
        a = fmax;
    }
    if (a == 0.0)
        return sign;

    /* Grid spacing at a's binade (the subnormal spacing below 2^emin). */
    int ex;
    (void)frexp(a, &ex);                     /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;                          /* floor(log2 a) */
    int eq = (E < emin ? emin : E) - mbits;  /* log2 of the quantum */
    double n = nearbyint(ldexp(a, -eq));     /* a / quantum, ties to even */
    double r = ldexp(n, eq);                 /* rounded magnitude */
    if (r > fmax)
        r = fmax;
    if (r == 0.0)
        return sign;

    (void)frexp(r, &ex);
    int Er = ex - 1;
    uint32_t efield, mfield;
    if (Er < emin) {
        efield = 0;
        mfield = (uint32_t)ldexp(r, -(emin - mbits));
    } else {
        efield = (uint32_t)(Er + bias);
        mfield = (uint32_t)(ldexp(r, -(Er - mbits)) - (double)(1 << mbits));
    }
    return (uint8_t)(sign | (efield << mbits) | mfield);
}

/* Encodes the fp32 values whose bit patterns are start, start+1, ... */
void orc_fp8_encode_bits_range(uint32_t start, uint64_t count, int fmt, uint8_t* out)
{
    for (uint64_t i = 0; i < count; ++i) {
        uint32_t u = (uint32_t)(start + i);
        float f;
        memcpy(&f, &u, 4);
        out[i] = orc_fp8_encode(f, fmt);
    }
}

/* Encodes n fp32 values. */
void orc_fp8_encode_array(const float* v, int64_t n, int fmt, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_fp8_encode(v[i], fmt);
}

/* ------------------------------------------------------------ scale rules */

/* Per-tensor multiplier s = fmax / amax. */
float orc_pertensor_scale(float amax, int fmt)
{
    if (!(amax > 0.0f))
        return 1.0f;
    float s = (float)orc_fmax(fmt) / amax;
    if (isinf(s))
        s = FLT_MAX;
    return s;
}

/* Blockwise divisor d = amax / fmax. */
float orc_block_scale(float amax, int fmt)
{
    if (!(amax > 0.0f))
        return 1.0f;
    float d = amax / (float)orc_fmax(fmt);
    if (d == 0.0f)
        d = FLT_TRUE_MIN;
    return d;
}

/* MXFP8 exponent e = floor(log2 amax) - emax_elem, clamped to [-127, 127]. */
int orc_mx_exponent(float amax, int fmt)
{
    if (!(amax > 0.0f))
        return 0;
    int ex;
    (void)frexp((double)amax, &ex);
    int e = (ex - 1) - orc_emax_elem(fmt);
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

/* ------------------------------------------------------------- threads */

/* Host threads the oracle's loops may use (n >= 1); returns the count now in
 * force.  Without OpenMP everything runs on one thread. */
int orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ------------------------------------------------------------- quantizers */

#define ORC_KIND_MULT 0  /* per-tensor: y = x * s,  s = fmax / amax */
#define ORC_KIND_DIV 1   /* blockwise:  y = x / d,  d = amax / fmax */
#define ORC_KIND_POW2 2  /* MXFP8:      y = x * 2^-e                */

/*
 * Quantizes x [R][C] (bf16 bits, row-major) in blocks of br x bc elements
 * (partial edge blocks take the elements present).  For block (i, j):
 *   amax[i][j]   = max |x| over its finite elements,
 *   scale[i][j]  = s (MULT), d (DIV) or 2^e (POW2) as fp32,
 *   e8m0[i][j]   = e + 127 (POW2 only; may be NULL),
 *   q[r][c]      = encode(y) for every element of the block.
 * sat / nonfinite receive the totals over the whole matrix.
 */
void orc_quant_blocks(const uint16_t* x, int64_t R, int64_t C, int64_t br, int64_t bc,
                      int kind, int fmt, uint8_t* q, float* scale, uint8_t* e8m0,
                      float* amax_out, uint64_t* sat, uint64_t* nonfinite)
{
    int64_t nbr = (R + br - 1) / br;
    int64_t nbc = (C + bc - 1) / bc;
    double fmax = orc_fmax(fmt);
    uint64_t nsat = 0, nnf = 0;
    /* one block (a per-tensor scope): its rows are split across threads;
     * several blocks: the blocks are */
    const int one = nbr * nbc == 1;
#pragma omp parallel for collapse(2) reduction(+ : nsat, nnf) schedule(dynamic, 16) if (!one)
    for (int64_t bi = 0; bi < nbr; ++bi) {
        for (int64_t bj = 0; bj < nbc; ++bj) {
            int64_t r0 = bi * br, r1 = r0 + br < R ? r0 + br : R;
            int64_t c0 = bj * bc, c1 = c0 + bc < C ? c0 + bc : C;
            float amax = 0.0f;
#pragma omp parallel for reduction(max : amax) if (one)
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = c0; c < c1; ++c) {
                    float f = orc_bf16_to_f32(x[r * C + c]);
                    if (isfinite(f) && fabsf(f) > amax)
                        amax = fabsf(f);
                }
            float sc;
            int e = 0;
            if (kind == ORC_KIND_MULT) {
                sc = orc_pertensor_scale(amax, fmt);
            } else if (kind == ORC_KIND_DIV) {
                sc = orc_block_scale(amax, fmt);
            } else {
                e = orc_mx_exponent(amax, fmt);
                sc = ldexpf(1.0f, e);
            }
            float mul = (kind == ORC_KIND_POW2) ? ldexpf(1.0f, -e) : sc;
            uint64_t bsat = 0, bnf = 0;
#pragma omp parallel for reduction(+ : bsat, bnf) if (one)
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = c0; c < c1; ++c) {
                    float f = orc_bf16_to_f32(x[r * C + c]);
                    float y = (kind == ORC_KIND_DIV) ? f / sc : f * mul;
                    if (!isfinite(f))
                        ++bnf;
                    else if (fabs((double)y) > fmax)
                        ++bsat;
                    q[r * C + c] = orc_fp8_encode(y, fmt);
                }
            nsat += bsat;
            nnf += bnf;
            if (scale)
                scale[bi * nbc + bj] = sc;
            if (e8m0)
                e8m0[bi * nbc + bj] = (uint8_t)(e + 127);
            if (amax_out)
                amax_out[bi * nbc + bj] = amax;
        }
    }
    if (sat)
        *sat = nsat;
    if (nonfinite)
        *nonfinite = nnf;
}

/* Per-tensor cast with a given multiplier s (the delayed recipe's step):
 * q = encode(x * s); also the tensor's amax over finite elements. */
void orc_cast_scaled(const uint16_t* x, int64_t n, float s, int fmt, uint8_t* q,
                     float* amax_out, uint64_t* sat, uint64_t* nonfinite)
{
    double fmax = orc_fmax(fmt);
    float amax = 0.0f;
    uint64_t nsat = 0, nnf = 0;
#pragma omp parallel for reduction(max : amax) reduction(+ : nsat, nnf) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float f = orc_bf16_to_f32(x[i]);
        float y = f * s;
        if (!isfinite(f))
            ++nnf;
        else {
            if (fabsf(f) > amax)
                amax = fabsf(f);
            if (fabs((double)y) > fmax)
                ++nsat;
        }
        q[i] = orc_fp8_encode(y, fmt);
    }
    if (amax_out)
        *amax_out = amax;
    if (sat)
        *sat = nsat;
    if (nonfinite)
        *nonfinite = nnf;
}

/* The scalars of a per-tensor cast with multiplier s without the codes:
 * amax over finite elements, saturated and nonfinite counts (same rules as
 * orc_cast_scaled). */
void orc_amax_sat(const uint16_t* x, int64_t n, float s, int fmt, float* amax_out, uint64_t* sat,
                  uint64_t* nonfinite)
{
    double fmax = orc_fmax(fmt);
    float amax = 0.0f;
    uint64_t nsat = 0, nnf = 0;
#pragma omp parallel for reduction(max : amax) reduction(+ : nsat, nnf) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float f = orc_bf16_to_f32(x[i]);
        if (!isfinite(f)) {
            ++nnf;
            continue;
        }
        if (fabsf(f) > amax)
            amax = fabsf(f);
        float y = f * s;
        if (fabs((double)y) > fmax)
            ++nsat;
    }
    *amax_out = amax;
    *sat = nsat;
    *nonfinite = nnf;
}

/* ------------------------------------------------------- delayed scaling */

#define ORC_MAX_HIST 4096

typedef struct {
    int H;
    int head;
    int fmt;
    int margin;
    float scale;
    float scale_inv;
    float hist[ORC_MAX_HIST];
} orc_delayed;

int orc_delayed_sizeof(void) { return (int)sizeof(orc_delayed); }

/* Fresh state: empty (all-zero) history, s = 1. */
int orc_delayed_init(orc_delayed* st, int H, int fmt, int margin)
{
    if (H < 1 || H > ORC_MAX_HIST)
        return -1;
    memset(st, 0, sizeof(*st));
    st->H = H;
    st->fmt = fmt;
    st->margin = margin;
    st->scale = 1.0f;
    st->scale_inv = 1.0f;
    return 0;
}

/* Records amax_t in the ring and derives the next step's scale. */
void orc_delayed_update(orc_delayed* st, float amax, uint64_t nonfinite)
{
    if (nonfinite != 0 || !isfinite(amax))
        return;
    st->hist[st->head] = amax;
    st->head = (st->head + 1) % st->H;
    float m = 0.0f;
    for (int i = 0; i < st->H; ++i)
        if (st->hist[i] > m)
            m = st->hist[i];
    float s;
    if (!(m > 0.0f)) {
        s = 1.0f;
    } else {
        s = (float)orc_fmax(st->fmt) / m;
        s = s * ldexpf(1.0f, -st->margin);
        if (isinf(s))
            s = FLT_MAX;
        /* a margin can push s below the normal range (margin 64 with a
         * history max near the bf16 maximum): raise it to the smallest
         * normal fp32, so that 1 / s stays finite */
        if (s < FLT_MIN)
            s = FLT_MIN;
    }
    st->scale = s;
    st->scale_inv = 1.0f / s;
}

/* --------------------------------------------------------- scale layouts */

/*
 * MXFP8 scale layout consumed by the block-scaled tensor-core MMA: the
 * [R][S] E8M0 matrix (S = scale columns) is cut into tiles of 128 rows x 4
 * scale columns, 512 bytes each, tiles ordered row-tile-major; inside a tile
 * row r, column c sits at byte (r % 32) * 16 + (r / 32) * 4 + c.  Rows are
 * padded to 128 and columns to 4 with code 127 (2^0).
 */
void orc_pack_mx(const uint8_t* codes, int64_t R, int64_t S, uint8_t* out)
{
    int64_t rt = (R + 127) / 128, ct = (S + 3) / 4;
    for (int64_t i = 0; i < rt * ct * 512; ++i)
        out[i] = 127;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < S; ++c) {
            int64_t tile = (r / 128) * ct + (c / 4);
            int64_t rr = r % 128, cc = c % 4;
            out[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cc] = codes[r * S + c];
        }
}

/*
 * 1x128 blockwise scale layout consumed by the GEMM: the [R][Kb] fp32
 * matrix stored K-block-major, [Kb][Rp] with Rp = R rounded up to 128 and
 * the pad rows set to 1.0.
 */
void orc_pack_block1x128(const float* d, int64_t R, int64_t Kb, float* out)
{
    int64_t Rp = (R + 127) / 128 * 128;
    for (int64_t i = 0; i < Kb * Rp; ++i)
        out[i] = 1.0f;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < Kb; ++k)
            out[k * Rp + r] = d[r * Kb + k];
}

/* ------------------------------------------------------------------ GEMM */

/*
 * Scaled FP8 GEMM, D = A . B^T with A [M][K] and B [N][K] (K contiguous,
 * sec. 3.1 fprop/dgrad/wgrad all reduce to this form).  Each element is
 * dequantized on its own, code value times its dequantization scale in
 * fp64, and the products are summed in fp64 in index order k = 0..K-1.
 * The scale of A[m][k] is sA[(m / a_bm) * a_ld + (k / a_bk)], likewise for B.
 * Only the requested output points (pm[i], pn[i]) are computed.
 */
void orc_gemm_points(const uint8_t* A, int fmtA, const float* sA, int64_t a_bm, int64_t a_bk, int64_t a_ld,
                     const uint8_t* B, int fmtB, const float* sB, int64_t b_bn, int64_t b_bk, int64_t b_ld,
                     int64_t M, int64_t N, int64_t K,
                     const int64_t* pm, const int64_t* pn, int64_t npts, double* out)
{
    (void)M;
    (void)N;
    double tabA[256], tabB[256];
    for (int c = 0; c < 256; ++c) {
        tabA[c] = orc_fp8_decode((uint8_t)c, fmtA);
        tabB[c] = orc_fp8_decode((uint8_t)c, fmtB);
    }
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t p = 0; p < npts; ++p) {
        int64_t m = pm[p], n = pn[p];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = tabA[A[m * K + k]] * (double)sA[(m / a_bm) * a_ld + (k / a_bk)];
            double b = tabB[B[n * K + k]] * (double)sB[(n / b_bn) * b_ld + (k / b_bk)];
            acc += a * b;
        }
        out[p] = acc;
    }
}

/* Round a double to bf16 (round-to-nearest-even, overflow to Inf); returns
 * the bf16 bits. */
uint16_t orc_f64_to_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int ex;
    (void)frexp(a, &ex);
    int E = ex - 1;
    int eq = (E < -126 ? -126 : E) - 7;      /* bf16: 8 significant bits */
    double r = ldexp(nearbyint(ldexp(a, -eq)), eq);
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80);
    float f = (float)r;                       /* exact: r has <= 8 bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (u >> 16));
}
