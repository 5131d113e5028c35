// Quantize kernels: per-tensor current / delayed, blockwise 1x128 / 128x128,
// MXFP8 1x32 ("2025 FP8 quantized-training guide", sec. 2.1-2.3; "mastering
// FP8 LLM training 1.5x speedup", scaling strategies 1-4), per-channel
// current and sub-channel blocks of 1 x b / b x b (the same page, scaling
// strategy 3 and Figure 1's channel-wise scaling).
//
// One tile kernel serves every recipe.  A persistent CTA of 256 threads walks
// 128x128 tiles of x; TMA loads each tile (two 64-column boxes in the 128-byte
// swizzle) into a 3-stage shared-memory ring, two tiles ahead.  Row path:
// thread t owns row t % 128 and the 64-column half t / 128, i.e. two whole
// 1x32 blocks or half of a 1x128 block, so block maxima are packed u16x2
// maxima inside the thread and each scale is computed once per 32 or 64
// elements.  Column path (1x128, MXFP8, per channel, 1 x b): thread t reads
// rows 32 (t / 64) .. +31 of columns 2 (t % 64), +1 from the same swizzled
// tile (conflict-free) and reduces the column blocks; for per-tensor, 128x128
// and b x b scales the column copy is the byte transpose of the row codes.
// Per-channel scales and 256-wide blocks span tiles: a pass over x leaves
// their maxima in the scale buffers before the tile pass.  Once the bf16 tile
// is consumed, its stage takes the two 128x128 code tiles, which TMA stores
// write out; the stage is reloaded after those stores have read it.  The
// 128-aligned tiles make every scale-layout pad entry the scale of an all-zero
// block (code 127 / 1.0).
#include <string.h>

#include <mutex>
#include <type_traits>

#include "fp8q_internal.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace fp8q {

// Device error word of the quantize kernels (bit 1: a tile-load wait timed out).
__device__ unsigned int g_quant_errors = 0;

namespace {

constexpr int kThreads = 256;
constexpr int kTile = 128;
constexpr int kStages = 3;
constexpr uint32_t kStageBytes = kTile * kTile * 2;  // one bf16 tile
constexpr uint32_t kTileSmem = kStages * kStageBytes + 1024;

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Largest finite |x| of the two bf16 in w, as bf16 magnitude bits (0 if none),
// and the number of NaN / Inf among them.
__device__ __forceinline__ uint32_t absmax_bits(uint32_t w, uint32_t& nonfinite) {
    uint32_t lo = w & 0x7FFFu, hi = (w >> 16) & 0x7FFFu;
    uint32_t flo = lo < 0x7F80u, fhi = hi < 0x7F80u;
    nonfinite += (1u - flo) + (1u - fhi);
    lo = flo ? lo : 0u;
    hi = fhi ? hi : 0u;
    return lo > hi ? lo : hi;
}

__device__ __forceinline__ uint32_t vec_absmax(const uint4& v, uint32_t& nonfinite) {
    uint32_t a = absmax_bits(v.x, nonfinite), b = absmax_bits(v.y, nonfinite);
    uint32_t c = absmax_bits(v.z, nonfinite), d = absmax_bits(v.w, nonfinite);
    a = a > b ? a : b;
    c = c > d ? c : d;
    return a > c ? a : c;
}

// The hardware conversion returns the canonical NaN 0x7F whatever the input's
// sign; a NaN keeps its sign bit here (S.1111111, as torch's float8 casts do).
// q holds the codes of the two bf16 of w in its low (x0) and next (x1) byte.
__device__ __forceinline__ uint32_t nan_sign2(uint32_t q, uint32_t w) {
    if ((w & 0x7FFFu) > 0x7F80u) q = (q & ~0xFFu) | ((w >> 8) & 0x80u) | 0x7Fu;
    if ((w & 0x7FFF0000u) > 0x7F800000u) q = (q & ~0xFF00u) | ((w >> 16) & 0x8000u) | 0x7F00u;
    return q;
}

// Scaled value of one element for the recipe's scale rule.
template <int KIND>
__device__ __forceinline__ float scaled(float x, float k) {
    if constexpr (KIND == kB1 || KIND == kB128 || KIND == kGen)
        return __fdiv_rn(x, k);  // blockwise: x / d
    else
        return __fmul_rn(x, k);  // per-tensor x * s, MXFP8 x * 2^-e (exact)
}

template <int FMT>
__device__ __forceinline__ uint32_t sat_count(float x, float y) {
    return (fabsf(x) <= 3.402823466e38f && fabsf(y) > Fmt<FMT>::fmax) ? 1u : 0u;
}

// Converts the 8 bf16 of v with factor k; returns 8 codes, counts saturation.
template <int KIND, int FMT>
__device__ __forceinline__ uint2 convert8(const uint4& v, float k, uint32_t& nsat, bool nonfinite) {
    float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                  bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        y[j] = scaled<KIND>(f[j], k);
        nsat += sat_count<FMT>(f[j], y[j]);
    }
    uint2 q = make_uint2(cvt4<FMT>(y[0], y[1], y[2], y[3]), cvt4<FMT>(y[4], y[5], y[6], y[7]));
    if (nonfinite) {
        q.x = nan_sign2(q.x & 0xFFFFu, v.x) | (nan_sign2(q.x >> 16, v.y) << 16);
        q.y = nan_sign2(q.y & 0xFFFFu, v.z) | (nan_sign2(q.y >> 16, v.w) << 16);
    }
    return q;
}


// Per-half maxima of |x| over the 8 bf16 of v, NaN / Inf included (their
// magnitude bits are >= 0x7F80, so a fold of 0x7F80 or more flags them).
__device__ __forceinline__ uint32_t vec_pmax(const uint4& v) {
    const uint32_t M = 0x7FFF7FFFu;
    return max_u16x2(max_u16x2(v.x & M, v.y & M), max_u16x2(v.z & M, v.w & M));
}
__device__ __forceinline__ uint32_t fold16(uint32_t p) { return max(p & 0xFFFFu, p >> 16); }

// Scale factor of one block: the multiplier k (per-tensor s, MX 2^-e), or for
// the blockwise recipes the divisor d = k with r = RN(1 / d).
struct Factor {
    float k, r;
    bool fast;
};

template <int KIND>
__device__ __forceinline__ Factor make_factor(float k) {
    Factor f;
    f.k = k;
    if constexpr (KIND == kB1 || KIND == kB128 || KIND == kGen) {
        f.r = k >= 0x1p-80f ? rcp_rn(k) : 0.0f;  // the reciprocal serves the shortcut only
        f.fast = k >= 0x1p-80f;  // keeps the residual below exact in fp32
    } else {
        f.r = 0.0f;
        f.fast = true;
    }
    return f;
}

// x / d correctly rounded from r = RN(1 / d): q = RN(x r) lies within one ulp
// of x / d, the residual x - d q is exactly representable and one FMA gives
// it, and RN(q + residual * r) = RN(x / d) (Markstein's theorem on division
// with a correctly rounded reciprocal).  The residual is formed negated,
// t = RN(q d - x), and added back as -t r: the same values for x != 0, and the
// sign of a zero x survives (-0: t = +0, -0 + -0 = -0), as it does for
// quotients that underflow (d > 0).  Valid for finite x, d in [2^-80, 2^128)
// and quotients in [2^-24, 2^126): near overflow x r can round to infinity,
// and for tiny x the residual can fall below the normal range; quotients under
// 2^-24 are below half the smallest subnormal of either FP8 format and encode
// to zero whatever their last bits, and quantization only divides |x| <= amax
// by RN(amax / fmax), so its quotients stay below fmax (1 + 2^-23).
__device__ __forceinline__ float div_rn_recip(float x, float d, float r) {
    const float q = __fmul_rn(x, r);
    const float t = __fmaf_rn(q, d, -x);
    return __fmaf_rn(-t, r, q);
}

// The recipe's scaled value of a finite element (FAST: the blockwise divisor
// is in the reciprocal shortcut's range; the caller branches once per block).
template <int KIND, bool FAST = true>
__device__ __forceinline__ float apply(float x, const Factor& f) {
    if constexpr (KIND == kB1 || KIND == kB128 || KIND == kGen) {
        if constexpr (FAST)
            return div_rn_recip(x, f.k, f.r);
        else
            return __fdiv_rn(x, f.k);
    } else {
        return __fmul_rn(x, f.k);
    }
}

// Two elements at a time with Blackwell's two-lane fp32 instructions (each
// lane an independent round-to-nearest operation, bit-identical to the
// scalar forms).  Factor2 holds the factors of the two lanes.
struct Factor2 {
    float2 k, nr;  // multiplier or divisor; minus the divisor's reciprocal
};
__device__ __forceinline__ Factor2 pair_factor(const Factor& a, const Factor& b) {
    Factor2 f;
    f.k = make_float2(a.k, b.k);
    f.nr = make_float2(-a.r, -b.r);
    return f;
}
__device__ __forceinline__ float2 bf16x2_f32(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }
// The blockwise recipes' lanes come out negated: with nr = -RN(1/d),
// -q = RN(x nr), e = RN(x - q d) = RN(-q d + x) (exact), -q2 = RN(e nr - q)
// = -RN(q + e r) -- Markstein's three steps with no negation at run time, and
// a zero x gives -q2 = -0 * sign(x), so the codes of -q2 with their sign bits
// flipped (kNegated) are the codes of RN(x / d) with the sign of a zero kept.
// Other recipes: the product.
template <int KIND>
constexpr bool kNegated = KIND == kB1 || KIND == kB128 || KIND == kGen;
template <int KIND>
__device__ __forceinline__ float2 apply2(float2 x, const Factor2& f) {
    if constexpr (kNegated<KIND>) {
        return div2_neg(x, f.k, f.nr);
    } else {
        return __fmul2_rn(x, f.k);
    }
}
// cvt4 of apply2's lanes, sign bits restored for the negated recipes.
template <int KIND, int FMT>
__device__ __forceinline__ uint32_t cvt4_applied(float a, float b, float c, float d) {
    const uint32_t q = cvt4<FMT>(a, b, c, d);
    return kNegated<KIND> ? q ^ 0x80808080u : q;
}
template <int FMT>
__device__ __forceinline__ uint32_t sat2(float2 y, bool cx, bool cy) {
    return (uint32_t)(cx && fabsf(y.x) > Fmt<FMT>::fmax) + (uint32_t)(cy && fabsf(y.y) > Fmt<FMT>::fmax);
}

// The 8 finite bf16 of v (one row) with one factor in both lanes of f; counts
// saturation only when the caller found that the vector's largest magnitude
// can exceed fmax once scaled (the scaled value is monotone in |x|).
template <int KIND, int FMT>
__device__ __forceinline__ uint2 convert8_packed(const uint4& v, const Factor2& f, uint32_t& nsat, bool count) {
    const float2 y0 = apply2<KIND>(bf16x2_f32(v.x), f), y1 = apply2<KIND>(bf16x2_f32(v.y), f);
    const float2 y2 = apply2<KIND>(bf16x2_f32(v.z), f), y3 = apply2<KIND>(bf16x2_f32(v.w), f);
    // blockwise scales almost never saturate (a uniform, untaken branch);
    // MXFP8 and per-tensor blocks often can: count without branching
    if (KIND != kB1 && KIND != kB128 && KIND != kGen || count)
        nsat += sat2<FMT>(y0, count, count) + sat2<FMT>(y1, count, count) + sat2<FMT>(y2, count, count) +
                sat2<FMT>(y3, count, count);
    return make_uint2(cvt4_applied<KIND, FMT>(y0.x, y0.y, y1.x, y1.y), cvt4_applied<KIND, FMT>(y2.x, y2.y, y3.x, y3.y));
}

// Converts the 8 finite bf16 of v; counts saturation only when the caller
// found that the vector's largest magnitude can exceed fmax once scaled
// (the scaled value is monotone in |x|).
template <int KIND, int FMT, bool FAST>
__device__ __forceinline__ uint2 convert8_fast(const uint4& v, const Factor& f, uint32_t& nsat, bool count) {
    float y[8] = {apply<KIND, FAST>(bf16_lo(v.x), f), apply<KIND, FAST>(bf16_hi(v.x), f),
                  apply<KIND, FAST>(bf16_lo(v.y), f), apply<KIND, FAST>(bf16_hi(v.y), f),
                  apply<KIND, FAST>(bf16_lo(v.z), f), apply<KIND, FAST>(bf16_hi(v.z), f),
                  apply<KIND, FAST>(bf16_lo(v.w), f), apply<KIND, FAST>(bf16_hi(v.w), f)};
#pragma unroll
    for (int j = 0; j < 8; ++j) nsat += (count && fabsf(y[j]) > Fmt<FMT>::fmax) ? 1u : 0u;  // predicated, no branch
    return make_uint2(cvt4<FMT>(y[0], y[1], y[2], y[3]), cvt4<FMT>(y[4], y[5], y[6], y[7]));
}

template <int KIND, int FMT>
__device__ __forceinline__ bool may_saturate(uint32_t max_bits16, const Factor& f) {
    const float m = __uint_as_float(max_bits16 << 16);
    return fabsf(f.fast ? apply<KIND, true>(m, f) : apply<KIND, false>(m, f)) > Fmt<FMT>::fmax;
}

template <int KIND, int FMT>
__device__ __forceinline__ float pertensor_factor(const QuantArgs& a) {
    if constexpr (KIND == kCur)
        return pertensor_scale<FMT>(*a.amax);
    else
        return a.st->scale;
}

// Byte offset of the 16-byte chunk `chunk` (8 bf16) of row r inside one
// 128-byte-swizzled half tile [128 rows][64 bf16], as the TMA writes it.
__device__ __forceinline__ uint32_t swz(int r, int chunk) { return (uint32_t)(r * 128 + ((chunk ^ (r & 7)) << 4)); }

// Exact largest finite |x| over vectors [j0, j1) of v, counting NaN / Inf and
// marking the vectors that hold them (the rare path behind the packed maxima).
template <int J0, int J1>
__device__ __forceinline__ uint32_t exact_max(const uint4 (&v)[8], uint32_t& nnf, uint32_t& vnf) {
    uint32_t m = 0;
#pragma unroll
    for (int j = J0; j < J1; ++j) {
        const uint32_t before = nnf;
        const uint32_t mj = vec_absmax(v[j], nnf);
        m = m > mj ? m : mj;
        if (nnf != before) vnf |= 1u << j;
    }
    return m;
}

// Two FP8 codes (low byte: column c, high byte: column c + 1) of row r of a
// 128x128 code tile in the 128-byte swizzle.
__device__ __forceinline__ uint32_t code_pair(const uint8_t* tile, int r, int c) {
    return *(const uint16_t*)(tile + swz(r, c >> 4) + (c & 15));
}
// From the code pairs of rows j .. j + 3 (h0 .. h3), the four codes of the
// low column (x) and of the high column (y), row j in the lowest byte.
__device__ __forceinline__ void transpose4(uint32_t h0, uint32_t h1, uint32_t h2, uint32_t h3, uint32_t& x,
                                           uint32_t& y) {
    const uint32_t a = __byte_perm(h0, h1, 0x5140), b = __byte_perm(h2, h3, 0x5140);  // x0 x1 y0 y1 / x2 x3 y2 y3
    x = __byte_perm(a, b, 0x5410);
    y = __byte_perm(a, b, 0x7632);
}

// Per 16-bit lane of the packed magnitudes of w (both no larger than their
// lane's m): 1 where the magnitude equals m, else 0, counted in the lane.
// c2 = (0x8000 - m_lo) | (0x8000 - m_hi) << 16: |x| + 0x8000 - m reaches bit
// 15 of its lane exactly when |x| == m, and no lane carries into the next.
__device__ __forceinline__ uint32_t lanes_at_max(uint32_t w, uint32_t c2) {
    return (((w & 0x7FFF7FFFu) + c2) >> 15) & 0x00010001u;
}
// Saturated elements of a per-tensor-current, per-channel or blockwise block whose maximum
// m can saturate.  Those scales are one correctly rounded division of fmax and
// amax (relative error <= 2^-24) and the next bf16 below m is at least 2^-8
// smaller, so only elements equal to m in magnitude can exceed fmax once
// scaled: count those, looking only inside the vectors whose packed maxima
// vp (from the analysis) hold m.  No element of v exceeds m.
template <int J0, int J1>
__device__ __forceinline__ uint32_t count_at_max(const uint4 (&v)[8], const uint32_t (&vp)[8], uint32_t m) {
    const uint32_t c2 = (0x8000u - m) * 0x00010001u;
    uint32_t acc = 0;
#pragma unroll
    for (int j = J0; j < J1; ++j)
        if (fold16(vp[j]) == m)
            acc += lanes_at_max(v[j].x, c2) + lanes_at_max(v[j].y, c2) + lanes_at_max(v[j].z, c2) +
                   lanes_at_max(v[j].w, c2);
    return (acc & 0xFFFFu) + (acc >> 16);
}

// The rare paths of a tile -- a NaN / Inf in the data, or a blockwise divisor
// below the reciprocal shortcut's range -- out of line, so that the loop's
// common path stays compact in the instruction cache.  Arrays travel by value
// in small structs: the common path never takes their address, so they stay
// in registers there.
struct Row8 {
    uint4 v[8];
};
struct RowCodes {
    uint2 q[8];
    uint32_t nsat;
};
struct MaxNf {
    uint32_t m, nnf, vnf;
};
struct Col32 {
    uint32_t w[32];
};
struct ColCodes {
    uint32_t o0[8], o1[8];
    uint32_t ns;
};

template <int J0, int J1>
__device__ __noinline__ MaxNf exact_max_rare(Row8 r) {
    MaxNf e;
    e.nnf = 0;
    e.vnf = 0;
    e.m = exact_max<J0, J1>(r.v, e.nnf, e.vnf);
    return e;
}

template <int KIND, int FMT>
__device__ __noinline__ RowCodes row_codes_rare(Row8 r, uint32_t vnf, Factor f0, Factor f1, bool s0, bool s1) {
    RowCodes out;
    out.nsat = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const Factor f = (j < 4) ? f0 : f1;
        if ((vnf >> j) & 1u)
            out.q[j] = convert8<KIND, FMT>(r.v[j], f.k, out.nsat, true);
        else
            out.q[j] = convert8_fast<KIND, FMT, false>(r.v[j], f, out.nsat, (j < 4) ? s0 : s1);
    }
    return out;
}

// Largest finite magnitudes of the two columns of c (NaN / Inf excluded).
__device__ __noinline__ uint2 col_exact_max_rare(Col32 c) {
    uint32_t m0 = 0, m1 = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint32_t lo = c.w[j] & 0x7FFFu, hi = (c.w[j] >> 16) & 0x7FFFu;
        m0 = (lo < 0x7F80u && lo > m0) ? lo : m0;
        m1 = (hi < 0x7F80u && hi > m1) ? hi : m1;
    }
    return make_uint2(m0, m1);
}

// Codes of 32 rows of two columns element by element (exact saturation
// counts, NaN signs kept).
template <int KIND, int FMT>
__device__ __noinline__ ColCodes col_codes_rare(Col32 c, float k0, float k1) {
    ColCodes out;
    out.ns = 0;
    const uint32_t* w = c.w;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        float a0 = bf16_lo(w[j]), a1 = bf16_lo(w[j + 1]), a2 = bf16_lo(w[j + 2]), a3 = bf16_lo(w[j + 3]);
        float b0 = bf16_hi(w[j]), b1 = bf16_hi(w[j + 1]), b2 = bf16_hi(w[j + 2]), b3 = bf16_hi(w[j + 3]);
        float ya0 = scaled<KIND>(a0, k0), ya1 = scaled<KIND>(a1, k0), ya2 = scaled<KIND>(a2, k0),
              ya3 = scaled<KIND>(a3, k0);
        float yb0 = scaled<KIND>(b0, k1), yb1 = scaled<KIND>(b1, k1), yb2 = scaled<KIND>(b2, k1),
              yb3 = scaled<KIND>(b3, k1);
        out.ns += sat_count<FMT>(a0, ya0) + sat_count<FMT>(a1, ya1) + sat_count<FMT>(a2, ya2) +
                  sat_count<FMT>(a3, ya3) + sat_count<FMT>(b0, yb0) + sat_count<FMT>(b1, yb1) +
                  sat_count<FMT>(b2, yb2) + sat_count<FMT>(b3, yb3);
        // rebuild the bf16 pairs of each output column to reuse nan_sign2
        const uint32_t a01 = (w[j] & 0xFFFFu) | (w[j + 1] << 16), a23 = (w[j + 2] & 0xFFFFu) | (w[j + 3] << 16);
        const uint32_t b01 = (w[j] >> 16) | (w[j + 1] & 0xFFFF0000u), b23 = (w[j + 2] >> 16) | (w[j + 3] & 0xFFFF0000u);
        const uint32_t qa = cvt4<FMT>(ya0, ya1, ya2, ya3), qb = cvt4<FMT>(yb0, yb1, yb2, yb3);
        out.o0[j / 4] = nan_sign2(qa & 0xFFFFu, a01) | (nan_sign2(qa >> 16, a23) << 16);
        out.o1[j / 4] = nan_sign2(qb & 0xFFFFu, b01) | (nan_sign2(qb >> 16, b23) << 16);
    }
    return out;
}

// Per-thread counters of a tile pass: saturated elements of the row-wise and
// of a re-quantized column-wise copy, NaN / Inf elements, and (delayed
// scaling) the largest finite magnitude seen, as bf16 bits.
struct TileCounts {
    uint32_t sat_row, sat_col, nonfinite, tmax;
};

// Generic blocks (KIND kGen): where the block maxima come from and the
// blocks' shape.  Blocks of 32 or 64 lie inside a 128 x 128 tile, so the tile
// pass finds their maxima itself (as for 1 x 128 and MXFP8); 256-wide blocks
// span tiles and take a pass over x first, whose maxima the tile pass loads.
enum { kGenNone = 0, kGenPass1D = 1, kGenPassSq = 2, kGenTile1D = 3, kGenTileSq = 4 };
template <int GEN>
constexpr bool kGenSquare = GEN == kGenPassSq || GEN == kGenTileSq;
template <int GEN>
constexpr bool kGenPass = GEN == kGenPass1D || GEN == kGenPassSq;

template <int KIND, bool COL, int GEN>
struct TileTraits {
    static constexpr bool kPerTensor = (KIND == kCur || KIND == kDel);
    // the column copy of a recipe whose scale does not depend on the copy's
    // direction is the byte transpose of the row codes
    static constexpr bool kTranspose = COL && (kPerTensor || KIND == kB128 || (KIND == kGen && kGenSquare<GEN>));
};

// Per-channel and generic blocks: the maxima that the amax pass left in the
// scale buffers for this thread's part of tile `tileid`, loaded before the
// tile's wait so that their latency overlaps it (pre_r: the row path's two
// 32-column blocks; pre_c: the column path's column pair).  Nothing for the
// other recipes.
template <int KIND, bool ROW, bool COL, int GEN>
__device__ __forceinline__ void tile_maxima(const QuantArgs& a, uint32_t tileid, uint32_t tiles_c,
                                            uint32_t (&pre_r)[2], uint32_t (&pre_c)[2]) {
    constexpr bool kTranspose = TileTraits<KIND, COL, GEN>::kTranspose;
    constexpr bool kRowCodes = ROW || kTranspose;
    const int t = threadIdx.x, rr = t & (kTile - 1), hh = t >> 7;
    const uint32_t tr = tileid / tiles_c, tc = tileid - tr * tiles_c;
    const int64_t r0g = a.row0 + (int64_t)tr * kTile, c0 = (int64_t)tc * kTile;
    (void)rr;
    (void)hh;
    (void)r0g;
    (void)c0;
    (void)kRowCodes;
    // per-channel and generic blocks: the maxima the amax pass left in the
    // scale buffers, loaded before the tile's wait so that their latency
    // overlaps it (pre_r: this thread's row path, two 32-column blocks;
    // pre_c: its column pair); rows and columns past x read 0
    if constexpr (KIND == kPC) {
        if constexpr (ROW) pre_r[0] = pre_r[1] = ((const uint32_t*)a.s_row)[r0g + rr];
        if constexpr (COL && !kTranspose) {
            const int64_t cc = c0 + 2 * (t & 63);
            pre_c[0] = ((const uint32_t*)a.s_col)[cc];
            pre_c[1] = ((const uint32_t*)a.s_col)[cc + 1];
        }
    } else if constexpr (KIND == kGen && kGenPass<GEN>) {
        const int bc = a.bc, sh = __ffs(bc) - 1;  // b is a power of two
        if constexpr (kRowCodes) {
            const int64_t rg = r0g + rr, cf = c0 + 64 * hh;  // row; first column of this half
            const int64_t nbc = (a.C + bc - 1) >> sh;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int64_t cc = cf + 32 * i;
                if (rg < a.R_total && cc < a.C && (i == 0 || bc == 32)) {
                    const int64_t bj = cc >> sh;
                    if constexpr (kGenSquare<GEN>) {
                        const int64_t nbr = (a.R_total + bc - 1) >> sh, bi = rg >> sh;
                        pre_r[i] = ROW ? ((const uint32_t*)a.s_row)[bi * nbc + bj]
                                       : ((const uint32_t*)a.s_col)[bj * nbr + bi];
                    } else {
                        pre_r[i] = ((const uint32_t*)a.s_row)[bj * (a.tiles_r_total * kTile) + rg];
                    }
                }
            }
            if (bc != 32) pre_r[1] = pre_r[0];
        }
        if constexpr (COL && !kTranspose) {
            const int64_t rq = r0g + 32 * (t >> 6), cc = c0 + 2 * (t & 63);
            if (rq < a.R_total) {
                const uint32_t* sc = (const uint32_t*)a.s_col + (rq >> sh) * (a.tiles_c * kTile) + cc;
                pre_c[0] = sc[0];
                pre_c[1] = sc[1];
            }
        }
    }
}

// One 128 x 128 tile (`tileid` of a tensor of tiles_c tile columns) whose
// bf16 values sit in `stage` as TMA loaded them (two 64-column halves,
// 128-byte swizzle): its row-wise and / or column-wise codes and scales; the
// codes replace the bf16 tile in the stage and thread 0 issues their TMA
// stores (the caller commits them).  Called by every thread of the CTA.
template <int KIND, int FMT, bool ROW, bool COL, int GEN>
__device__ __forceinline__ void tile_body(const QuantArgs& a, const CUtensorMap* tmrow, const CUtensorMap* tmcol,
                                          uint8_t* stage, uint32_t tileid, uint32_t tiles_c, float ks,
                                          const uint32_t (&pre_r)[2], const uint32_t (&pre_c)[2], uint32_t* colred,
                                          uint32_t* rowred, uint32_t* red, TileCounts& cnt) {
    constexpr bool kPerTensor = TileTraits<KIND, COL, GEN>::kPerTensor;
    constexpr bool kTranspose = TileTraits<KIND, COL, GEN>::kTranspose;
    constexpr bool kRowCodes = ROW || kTranspose;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rr = t & (kTile - 1), hh = t >> 7;  // row path: row and 64-column half of the tile
    const uint32_t tr = tileid / tiles_c, tc = tileid - tr * tiles_c;
    const int64_t r0 = (int64_t)tr * kTile, c0 = (int64_t)tc * kTile;
    // the tile's place in the whole tensor (a block of rows starts at row0)
    const int64_t trg = (int64_t)tr + a.row0 / kTile, r0g = a.row0 + r0;
    const int64_t tileg = trg * (int64_t)tiles_c + tc;
    uint32_t& nsat_row = cnt.sat_row;
    uint32_t& nsat_col = cnt.sat_col;
    uint32_t& nnf = cnt.nonfinite;
    uint32_t& tmax_all = cnt.tmax;
    (void)kPerTensor;
    (void)lane;
    (void)warp;
    (void)r0;
    (void)tileg;
    (void)ks;
    (void)pre_r;
    (void)pre_c;
    (void)tmax_all;
    (void)nsat_col;
    (void)red;
    (void)rowred;
    (void)colred;
    // ---------------- analysis: row rr, columns 64 hh .. 64 hh + 63 of the tile
    const uint8_t* half = stage + hh * (kStageBytes / 2);
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = *(const uint4*)(half + swz(rr, j));
    uint32_t vnf = 0;       // bit j: vector j holds a NaN / Inf
    uint32_t mq[2];         // MX: the two 1x32 blocks' maxima; else mq[0] = the half-row maximum
    uint32_t mh[2];         // the maxima of vectors 0-3 and 4-7 (NaN / Inf-free halves)
    uint32_t vp[8];         // each vector's packed maxima (NaN / Inf included)
    {
#pragma unroll
        for (int j = 0; j < 8; ++j) vp[j] = vec_pmax(v[j]);
        const uint32_t p0 = max_u16x2(max_u16x2(vp[0], vp[1]), max_u16x2(vp[2], vp[3]));
        const uint32_t p1 = max_u16x2(max_u16x2(vp[4], vp[5]), max_u16x2(vp[6], vp[7]));
        mh[0] = fold16(p0);
        mh[1] = fold16(p1);
        if (KIND == kMX || (KIND == kGen && a.bc == 32)) {
            mq[0] = fold16(p0);
            mq[1] = fold16(p1);
            if (mq[0] >= 0x7F80u || mq[1] >= 0x7F80u) {
                Row8 r;
#pragma unroll
                for (int j = 0; j < 8; ++j) r.v[j] = v[j];
                if (mq[0] >= 0x7F80u) {
                    const MaxNf e = exact_max_rare<0, 4>(r);
                    mq[0] = e.m;
                    nnf += e.nnf;
                    vnf |= e.vnf;
                }
                if (mq[1] >= 0x7F80u) {
                    const MaxNf e = exact_max_rare<4, 8>(r);
                    mq[1] = e.m;
                    nnf += e.nnf;
                    vnf |= e.vnf;
                }
            }
        } else {
            mq[0] = fold16(max_u16x2(p0, p1));
            if (mq[0] >= 0x7F80u) {
                Row8 r;
#pragma unroll
                for (int j = 0; j < 8; ++j) r.v[j] = v[j];
                const MaxNf e = exact_max_rare<0, 8>(r);
                mq[0] = e.m;
                nnf += e.nnf;
                vnf |= e.vnf;
            }
            mq[1] = mq[0];
        }
    }

    // ---------------- block scales
    float kq[2] = {ks, ks};
    if constexpr (KIND == kDel) {
        tmax_all = tmax_all > mq[0] ? tmax_all : mq[0];
    } else if constexpr (KIND == kB128) {
        const uint32_t m = warp_max_u32(mq[0]);
        if (lane == 0) red[warp] = m;
        __syncthreads();
        uint32_t mm = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) mm = mm > red[w] ? mm : red[w];
        kq[0] = kq[1] = block_scale<FMT>(__uint_as_float(mm << 16));
        if (t == 0) {
            if (ROW) ((float*)a.s_row)[tileg] = kq[0];
            if (COL) ((float*)a.s_col)[tc * a.tiles_r_total + trg] = kq[0];
        }
    } else if constexpr (KIND == kB1) {
        rowred[hh * kTile + rr] = mq[0];
        __syncthreads();
        const uint32_t m = max(rowred[rr], rowred[kTile + rr]);
        mq[0] = mq[1] = m;
        kq[0] = kq[1] = block_scale<FMT>(__uint_as_float(m << 16));
        if (ROW && hh == 0) ((float*)a.s_row)[tc * (a.tiles_r_total * kTile) + r0g + rr] = kq[0];
    } else if constexpr (KIND == kPC) {
        // the row's maximum over all of x (the amax pass left it in s_row as
        // bf16 magnitude bits): s = fmax / amax, the per-tensor current rule
        if constexpr (ROW) {
            const uint32_t m = pre_r[0];
            mq[0] = mq[1] = m;
            kq[0] = kq[1] = pertensor_scale<FMT>(__uint_as_float(m << 16));
        }
    } else if constexpr (KIND == kGen && kGenPass<GEN>) {
        // the blocks' maxima over all of x (the amax pass left them in the
        // scale buffers as bf16 magnitude bits); rows and columns past x read 0
        if constexpr (kRowCodes) {
            mq[0] = pre_r[0];
            mq[1] = pre_r[1];
            kq[0] = block_scale<FMT>(__uint_as_float(pre_r[0] << 16));
            kq[1] = block_scale<FMT>(__uint_as_float(pre_r[1] << 16));
        }
    } else if constexpr (KIND == kGen) {
        // blocks of b = 32 or 64 inside the tile (tiles start on multiples of
        // 128): 1 x b blocks are this half row's two 32-column pieces or all
        // of it; b x b blocks gather the half rows of one warp (b = 32: rows
        // 32 (warp % 4) ..) or of two (b = 64: warps w and w ^ 1)
        const int bc = a.bc, sh = __ffs(bc) - 1;  // b is a power of two
        if constexpr (GEN == kGenTileSq) {
            if (bc == 32) {
                mq[0] = warp_max_u32(mq[0]);
                mq[1] = warp_max_u32(mq[1]);
            } else {
                const uint32_t m = warp_max_u32(mq[0]);
                if (lane == 0) red[warp] = m;
                __syncthreads();
                mq[0] = mq[1] = max(red[warp], red[warp ^ 1]);
            }
        }
        kq[0] = block_scale<FMT>(__uint_as_float(mq[0] << 16));
        kq[1] = bc == 32 ? block_scale<FMT>(__uint_as_float(mq[1] << 16)) : kq[0];
        const int64_t nbc = (a.C + bc - 1) >> sh, bj0 = (c0 + 64 * hh) >> sh;
        if constexpr (GEN == kGenTile1D) {
            // row copy's scales [ceil(C / b)][Rp]: every row of the tile, pad rows included
            if (ROW) {
                float* sr = (float*)a.s_row + r0g + rr;
                const int64_t rp = a.tiles_r_total * kTile;
                if (bj0 < nbc) sr[bj0 * rp] = kq[0];
                if (bc == 32 && bj0 + 1 < nbc) sr[(bj0 + 1) * rp] = kq[1];
            }
        } else {
            // [ceil(R / b)][ceil(C / b)] and, for the transposed column copy,
            // [ceil(C / b)][ceil(R / b)]: one lane per block writes
            const int64_t nbr = (a.R_total + bc - 1) >> sh, bi = (r0g + rr) >> sh;
            if (lane == 0 && (bc == 32 || (warp & 1) == 0) && bi < nbr) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    if (i == 1 && bc != 32) break;
                    if (bj0 + i < nbc) {
                        if (ROW) ((float*)a.s_row)[bi * nbc + bj0 + i] = kq[i];
                        if (COL) ((float*)a.s_col)[(bj0 + i) * nbr + bi] = kq[i];
                    }
                }
            }
        }
    } else if constexpr (KIND == kMX) {
        const int e0 = mx_exponent<FMT>(mq[0] << 16), e1 = mx_exponent<FMT>(mq[1] << 16);
        kq[0] = exp2_neg(e0);
        kq[1] = exp2_neg(e1);
        if (ROW) {
            // this row's scale columns 4 tc + 2 hh + {0, 1} in the 128x4 tile (tr, tc)
            uint8_t* tileb = (uint8_t*)a.s_row + (size_t)tileg * 512;
            *(uint16_t*)(tileb + (rr & 31) * 16 + (rr >> 5) * 4 + 2 * hh) =
                (uint16_t)((uint32_t)(e0 + 127) | ((uint32_t)(e1 + 127) << 8));
        }
    }

    // ---------------- row-wise codes
    uint2 q[8];
    uint32_t nsat_rc = 0;
    if constexpr (kRowCodes) {
        const bool two = KIND == kMX || (KIND == kGen && a.bc == 32);  // two blocks in this half row
        const Factor f0 = make_factor<KIND>(kq[0]);
        const Factor f1 = two ? make_factor<KIND>(kq[1]) : f0;
        const bool s0 = may_saturate<KIND, FMT>(mq[0], f0);
        const bool s1 = two ? may_saturate<KIND, FMT>(mq[1], f1) : s0;
        if (vnf == 0 && f0.fast && f1.fast) {  // the common case: one straight-line block
            const Factor2 g0 = pair_factor(f0, f0), g1 = pair_factor(f1, f1);
            constexpr bool kAtMax = KIND == kCur || KIND == kB1 || KIND == kB128 || KIND == kPC || KIND == kGen;
            // only elements equal to the block maximum can saturate; counted
            // before the conversions, so that each vector's registers are free
            // once it is converted
            if (kAtMax) {
                if (s0 && mh[0] == mq[0]) nsat_rc += count_at_max<0, 4>(v, vp, mq[0]);
                if (s1 && mh[1] == mq[1]) nsat_rc += count_at_max<4, 8>(v, vp, mq[1]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                q[j] = convert8_packed<KIND, FMT>(v[j], (j < 4) ? g0 : g1, nsat_rc,
                                                  kAtMax ? false : ((j < 4) ? s0 : s1));
        } else {
            Row8 r;
#pragma unroll
            for (int j = 0; j < 8; ++j) r.v[j] = v[j];
            const RowCodes rc = row_codes_rare<KIND, FMT>(r, vnf, f0, f1, s0, s1);
#pragma unroll
            for (int j = 0; j < 8; ++j) q[j] = rc.q[j];
            nsat_rc += rc.nsat;
        }
        if (ROW) nsat_row += nsat_rc;  // a transposed column copy reports no count of its own
    }
    // the stage takes the codes once every thread has read its bf16 tile:
    // after the block-maximum barrier (128x128; 1x128 without a column
    // copy), after the column-block barrier (1x128), else after one more
    uint8_t* rowt = stage;                  // [128 rows][128 codes], 128-byte swizzle
    uint8_t* colt = stage + kTile * kTile;  // [128 columns][128 codes], 128-byte swizzle
    auto put_row_codes = [&]() {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            *(uint4*)(rowt + swz(rr, 4 * hh + c)) = make_uint4(q[2 * c].x, q[2 * c].y, q[2 * c + 1].x, q[2 * c + 1].y);
    };
    constexpr bool kCodesAfterBlockMax = KIND == kB128 || (KIND == kB1 && !COL);
    if constexpr (kRowCodes && kCodesAfterBlockMax) put_row_codes();

    // ---------------- column-wise codes re-quantized along the columns (1x128, MXFP8, per channel)
    const int p = t & 63, qd = t >> 6;  // column pair 2p, 2p + 1; rows 32 qd .. 32 qd + 31
    uint32_t o0[8], o1[8];
    if constexpr (COL && !kTranspose) {
        // columns 2p, 2p+1 sit in half p / 32, chunk (2p % 64) / 8, bytes (2p % 8) * 2
        const uint8_t* chalf = stage + (p >> 5) * (kStageBytes / 2) + ((2 * p) & 7) * 2;
        const int chunk = ((2 * p) & 63) >> 3;
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) w[j] = *(const uint32_t*)(chalf + swz(32 * qd + j, chunk));
        float k0, k1;
        uint32_t m0, m1, own0, own1;  // column block maxima; this thread's 32-row maxima
        bool col_nf;                   // a NaN / Inf among these 64 elements
        uint32_t pmg[4];               // packed maxima of rows 8g .. 8g + 7
        {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                uint32_t x = w[8 * g] & 0x7FFF7FFFu;
#pragma unroll
                for (int i = 1; i < 8; ++i) x = max_u16x2(x, w[8 * g + i] & 0x7FFF7FFFu);
                pmg[g] = x;
            }
            const uint32_t pm = max_u16x2(max_u16x2(pmg[0], pmg[1]), max_u16x2(pmg[2], pmg[3]));
            m0 = pm & 0xFFFFu;
            m1 = pm >> 16;
            own0 = m0;
            own1 = m1;
            col_nf = m0 >= 0x7F80u || m1 >= 0x7F80u;
            if (col_nf) {  // NaN / Inf: exact finite maxima
                Col32 cw;
#pragma unroll
                for (int j = 0; j < 32; ++j) cw.w[j] = w[j];
                const uint2 m = col_exact_max_rare(cw);
                m0 = m.x;
                m1 = m.y;
            }
            const int64_t cc = c0 + 2 * p;
            if constexpr (KIND == kMX) {
                const int e0 = mx_exponent<FMT>(m0 << 16), e1 = mx_exponent<FMT>(m1 << 16);
                k0 = exp2_neg(e0);
                k1 = exp2_neg(e1);
                // column-wise scales: logical [C][ceil(R/32)], tiles over (c/128, kb/4)
                uint8_t* tileb = (uint8_t*)a.s_col + ((size_t)tc * a.tiles_r_total + trg) * 512;
                const int cr = 2 * p;
                tileb[(cr & 31) * 16 + (cr >> 5) * 4 + qd] = (uint8_t)(e0 + 127);
                tileb[((cr + 1) & 31) * 16 + ((cr + 1) >> 5) * 4 + qd] = (uint8_t)(e1 + 127);
            } else if constexpr (KIND == kGen && kGenPass<GEN>) {
                // blocks of bc rows of one column (1 x bc blocks of x^T): their maxima
                // from the amax pass, in s_col [ceil(R/bc)][Cp]; rows past x read 0
                m0 = pre_c[0];
                m1 = pre_c[1];
                k0 = block_scale<FMT>(__uint_as_float(m0 << 16));
                k1 = block_scale<FMT>(__uint_as_float(m1 << 16));
            } else if constexpr (KIND == kGen) {
                // blocks of b = 32 rows of one column are this thread's rows; b = 64
                // joins the row quarters 2i, 2i + 1; scales [ceil(R / b)][Cp]
                const int bc = a.bc, sh = __ffs(bc) - 1;  // b is a power of two
                if (bc == 64) {
                    colred[qd * kTile + 2 * p] = m0;
                    colred[qd * kTile + 2 * p + 1] = m1;
                    __syncthreads();
                    const int q0 = qd & ~1;
                    m0 = max(colred[q0 * kTile + 2 * p], colred[(q0 + 1) * kTile + 2 * p]);
                    m1 = max(colred[q0 * kTile + 2 * p + 1], colred[(q0 + 1) * kTile + 2 * p + 1]);
                }
                k0 = block_scale<FMT>(__uint_as_float(m0 << 16));
                k1 = block_scale<FMT>(__uint_as_float(m1 << 16));
                const int64_t nbr = (a.R_total + bc - 1) >> sh, bi = (r0g + 32 * qd) >> sh;
                if ((bc == 32 || (qd & 1) == 0) && bi < nbr) {
                    float* sc = (float*)a.s_col + bi * (a.tiles_c * kTile) + cc;
                    sc[0] = k0;
                    sc[1] = k1;
                }
            } else if constexpr (KIND == kPC) {
                // the columns' maxima over all of x (from the amax pass, in s_col)
                m0 = pre_c[0];
                m1 = pre_c[1];
                k0 = pertensor_scale<FMT>(__uint_as_float(m0 << 16));
                k1 = pertensor_scale<FMT>(__uint_as_float(m1 << 16));
            } else {  // 1x128 along the rows of x: reduce the four quarters
                colred[qd * kTile + 2 * p] = m0;
                colred[qd * kTile + 2 * p + 1] = m1;
                __syncthreads();  // also: every bf16 read of the tile is done
                if constexpr (kRowCodes) put_row_codes();
                m0 = max(max(colred[2 * p], colred[kTile + 2 * p]),
                         max(colred[2 * kTile + 2 * p], colred[3 * kTile + 2 * p]));
                m1 = max(max(colred[2 * p + 1], colred[kTile + 2 * p + 1]),
                         max(colred[2 * kTile + 2 * p + 1], colred[3 * kTile + 2 * p + 1]));
                k0 = block_scale<FMT>(__uint_as_float(m0 << 16));
                k1 = block_scale<FMT>(__uint_as_float(m1 << 16));
                if (qd == 0) {
                    const int64_t Cp = a.tiles_c * kTile;
                    float* sc = (float*)a.s_col + trg * Cp + cc;
                    sc[0] = k0;
                    sc[1] = k1;
                }
            }
        }
        // convert 32 rows of columns 2p, 2p+1
        uint32_t ns = 0;
        const Factor f0 = make_factor<KIND>(k0), f1 = make_factor<KIND>(k1);
        if (!col_nf && f0.fast && f1.fast) {
            const bool c0s = may_saturate<KIND, FMT>(m0, f0), c1s = may_saturate<KIND, FMT>(m1, f1);
            const Factor2 g = pair_factor(f0, f1);  // lanes: column 2p, column 2p + 1
            if ((KIND == kB1 || KIND == kPC || KIND == kGen) && ((c0s && own0 == m0) || (c1s && own1 == m1))) {
                // only elements equal to the block maximum can saturate (as in
                // count_at_max), looked for in the 8-row groups whose maximum it
                // is, before the conversions
                const uint32_t c2 = (0x8000u - m0) | ((0x8000u - m1) << 16);
#pragma unroll
                for (int gi = 0; gi < 4; ++gi) {
                    const bool lo = c0s && (pmg[gi] & 0xFFFFu) == m0, hi = c1s && (pmg[gi] >> 16) == m1;
                    if (lo || hi) {
                        uint32_t acc = 0;
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc += lanes_at_max(w[8 * gi + i], c2);
                        ns += (lo ? (acc & 0xFFFFu) : 0u) + (hi ? (acc >> 16) : 0u);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float2 y0 = apply2<KIND>(bf16x2_f32(w[j]), g), y1 = apply2<KIND>(bf16x2_f32(w[j + 1]), g);
                const float2 y2 = apply2<KIND>(bf16x2_f32(w[j + 2]), g), y3 = apply2<KIND>(bf16x2_f32(w[j + 3]), g);
                if (KIND != kB1 && KIND != kPC && KIND != kGen)
                    ns += sat2<FMT>(y0, c0s, c1s) + sat2<FMT>(y1, c0s, c1s) + sat2<FMT>(y2, c0s, c1s) +
                          sat2<FMT>(y3, c0s, c1s);
                o0[j / 4] = cvt4_applied<KIND, FMT>(y0.x, y1.x, y2.x, y3.x);
                o1[j / 4] = cvt4_applied<KIND, FMT>(y0.y, y1.y, y2.y, y3.y);
            }
        } else {
            Col32 cw;
#pragma unroll
            for (int j = 0; j < 32; ++j) cw.w[j] = w[j];
            const ColCodes cc2 = col_codes_rare<KIND, FMT>(cw, k0, k1);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                o0[j] = cc2.o0[j];
                o1[j] = cc2.o1[j];
            }
            ns += cc2.ns;
        }
        nsat_col += ns;
    }

    // ---------------- codes into the stage (its bf16 tile is consumed), then TMA stores
    if constexpr (!kCodesAfterBlockMax && KIND != kB1) {
        __syncthreads();
        if constexpr (kRowCodes) put_row_codes();
    }
    if constexpr (kTranspose) {
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const int r = 32 * qd + j;
            transpose4(code_pair(rowt, r, 2 * p), code_pair(rowt, r + 1, 2 * p), code_pair(rowt, r + 2, 2 * p),
                       code_pair(rowt, r + 3, 2 * p), o0[j / 4], o1[j / 4]);
        }
    }
    if constexpr (COL) {
        *(uint4*)(colt + swz(2 * p, 2 * qd)) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
        *(uint4*)(colt + swz(2 * p, 2 * qd + 1)) = make_uint4(o0[4], o0[5], o0[6], o0[7]);
        *(uint4*)(colt + swz(2 * p + 1, 2 * qd)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
        *(uint4*)(colt + swz(2 * p + 1, 2 * qd + 1)) = make_uint4(o1[4], o1[5], o1[6], o1[7]);
    }
    fence_async_smem();
    __syncthreads();
    if (t == 0) {
        if (ROW) tma_store_2d(tmrow, (int)c0, (int)r0g, smem_u32(rowt));
        if (COL) tma_store_2d(tmcol, (int)r0g, (int)c0, smem_u32(colt));
    }
}

// GEN (generic blocks only): the blocks' shape and the source of their
// maxima (kGen* above); the block width b is a.bc, read at run time.
template <int KIND, int FMT, bool ROW, bool COL, int GEN = kGenNone>
__global__ void __launch_bounds__(kThreads, 2)
    quant_tile_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmrow,
                      const __grid_constant__ CUtensorMap tmcol, QuantArgs a) {
    constexpr bool kPerTensor = TileTraits<KIND, COL, GEN>::kPerTensor;
    extern __shared__ uint8_t qsmem_raw[];
    uint8_t* qsmem = (uint8_t*)(((uintptr_t)qsmem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(qsmem);
    __shared__ uint32_t colred[COL && (KIND == kB1 || (KIND == kGen && GEN == kGenTile1D)) ? 4 * kTile : 1];
    __shared__ uint32_t rowred[KIND == kB1 ? 2 * kTile : 1];
    __shared__ uint32_t red[kThreads / 32];
    __shared__ __align__(8) uint64_t bars[kStages];
    __shared__ int abort_flag;

    const int t = threadIdx.x, lane = t & 31;
    const uint32_t ntiles = (uint32_t)(a.tiles_r * a.tiles_c), tiles_c = (uint32_t)a.tiles_c;
    auto bar = [&](int s) { return smem_u32(&bars[s]); };

    // the CTA's j-th tile into stage j % kStages: two 64-column boxes, each
    // [128 rows][128 bytes] in the 128-byte swizzle
    auto issue = [&](uint32_t j) {
        const uint32_t tileid = blockIdx.x + j * gridDim.x;
        if (tileid >= ntiles || a.stall) return;  // a stalled launch (diagnostic) loads nothing
        const uint32_t s = j % kStages;
        const uint32_t tr = tileid / tiles_c, tc = tileid - tr * tiles_c;
        mbar_expect_tx(bar(s), kStageBytes);
        tma_load_2d(sbase + s * kStageBytes, &tmx, (int)(tc * kTile), (int)(tr * kTile), bar(s));
        tma_load_2d(sbase + s * kStageBytes + kStageBytes / 2, &tmx, (int)(tc * kTile + 64), (int)(tr * kTile), bar(s));
    };
    if (t == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar(s), 1);
        abort_flag = 0;
        mbar_fence_init();
        if (ntiles > 0) {
            prefetch_map(&tmx);
            if (ROW) prefetch_map(&tmrow);
            if (COL) prefetch_map(&tmcol);
        }
    }
    __syncthreads();
    // two tiles in flight; the third stage holds the previous tile's codes
    // until its stores have read them
    if (t == 0) {
        issue(0);
        issue(1);
    }

    float ks = 1.0f;
    if constexpr (kPerTensor) {
        ks = pertensor_factor<KIND, FMT>(a);
        if (blockIdx.x == 0 && t == 0) {
            *a.scale = ks;
            *a.scale_inv = (KIND == kDel) ? a.st->scale_inv : __fdiv_rn(1.0f, ks);
        }
    }

    TileCounts cnt = {0u, 0u, 0u, 0u};
    uint32_t it = 0, stg = 0, ph = 0;
    for (uint32_t tileid = blockIdx.x; tileid < ntiles; tileid += gridDim.x, ++it) {
        uint32_t pre_r[2] = {0u, 0u}, pre_c[2] = {0u, 0u};
        tile_maxima<KIND, ROW, COL, GEN>(a, tileid, tiles_c, pre_r, pre_c);
        const bool ok = mbar_wait_bounded(bar(stg), ph, &abort_flag, &g_quant_errors, 2u, a.wait_ns);
        if (__syncthreads_or(!ok)) break;  // the whole CTA leaves together
        tile_body<KIND, FMT, ROW, COL, GEN>(a, &tmrow, &tmcol, qsmem + stg * kStageBytes, tileid, tiles_c, ks, pre_r,
                                            pre_c, colred, rowred, red, cnt);
        if (t == 0) {
            bulk_commit();
            bulk_wait_read1();  // the previous tile's stores have read their stage ...
            issue(it + 2);      // ... which now takes the tile after next
        }
        if (++stg == kStages) {
            stg = 0;
            ph ^= 1u;
        }
    }
    if (t == 0) {
        bulk_wait_all();  // the codes' stores are complete before the CTA's shared memory goes away
        if (abort_flag && !a.stall) {
            // let the tile loads already issued land before the CTA exits (bounded)
            for (uint32_t j = it; j < it + 2; ++j)
                if (blockIdx.x + j * gridDim.x < ntiles)
                    mbar_drain(bar((int)(j % kStages)), (j / kStages) & 1u, a.wait_ns / 10);
        }
    }

    // ---------------- counters (and the delayed recipe's tensor amax)
    const uint32_t nsat_row = warp_sum_u32(cnt.sat_row);
    const uint32_t nsat_col = warp_sum_u32(cnt.sat_col);
    const uint32_t nnf = warp_sum_u32(cnt.nonfinite);
    if (lane == 0) {
        if (nsat_row) atomicAdd(&a.counters[0], (unsigned long long)nsat_row);
        if (nsat_col) atomicAdd(&a.counters[1], (unsigned long long)nsat_col);
        if (KIND != kCur && KIND != kPC && !(KIND == kGen && kGenPass<GEN>) && nnf)
            atomicAdd(&a.counters[2], (unsigned long long)nnf);  // else the amax pass
    }
    if constexpr (KIND == kDel) {
        const uint32_t tmax_all = warp_max_u32(cnt.tmax);
        if (lane == 0 && tmax_all) atomicMax((unsigned int*)a.amax, tmax_all << 16);
    }
}

// Per-tensor current scaling, pass 1: amax over the finite elements of x and
// the NaN / Inf count.  Four independent 16-byte loads in flight per thread.
// The common path takes the packed maxima of the magnitude bits (one AND and
// one u16x2 maximum a word); a thread whose maximum flags a NaN / Inf (>=
// 0x7F80) reads its vectors again with the exact per-element test.
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint16_t* x, int64_t nvec, float* amax,
                                                        unsigned long long* counters) {
    __shared__ uint32_t redm[kThreads / 32], redn[kThreads / 32];
    const uint4* xv = (const uint4*)x;
    uint32_t pm = 0, nf = 0;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t i0 = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    int64_t i = i0;
    for (; i + 3 * stride < nvec; i += 4 * stride) {
        const uint4 v0 = ld_nc_v4(xv + i), v1 = ld_nc_v4(xv + i + stride);
        const uint4 v2 = ld_nc_v4(xv + i + 2 * stride), v3 = ld_nc_v4(xv + i + 3 * stride);
        pm = max_u16x2(pm, max_u16x2(max_u16x2(vec_pmax(v0), vec_pmax(v1)), max_u16x2(vec_pmax(v2), vec_pmax(v3))));
    }
    for (; i < nvec; i += stride) pm = max_u16x2(pm, vec_pmax(ld_nc_v4(xv + i)));
    uint32_t m = fold16(pm);
    if (m >= 0x7F80u) {  // a NaN / Inf among this thread's elements (rare): exact finite maximum and count
        m = 0;
        for (i = i0; i < nvec; i += stride) m = max(m, vec_absmax(ld_nc_v4(xv + i), nf));
    }
    m = warp_max_u32(m);
    nf = warp_sum_u32(nf);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        redm[warp] = m;
        redn[warp] = nf;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t mm = 0, nn = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
            mm = max(mm, redm[w]);
            nn += redn[w];
        }
        if (mm) atomicMax((unsigned int*)amax, mm << 16);
        if (nn) atomicAdd(&counters[2], (unsigned long long)nn);
    }
}

// The two bf16 of w as magnitude bits, a NaN / Inf half replaced by 0.
__device__ __forceinline__ uint32_t finite_mag2(uint32_t w) {
    const uint32_t lo = w & 0x7FFFu, hi = (w >> 16) & 0x7FFFu;
    return (lo < 0x7F80u ? lo : 0u) | ((hi < 0x7F80u ? hi : 0u) << 16);
}
__device__ __forceinline__ uint32_t nonfinite2(uint32_t w) {
    return (uint32_t)((w & 0x7FFFu) >= 0x7F80u) + (uint32_t)(((w >> 16) & 0x7FFFu) >= 0x7F80u);
}

// The exact finite maxima of a thread's 8 x 8 elements of a strip (rows r0 ..
// r0 + 7, columns c .. c + 7; column pairs cm, rows rm) and its NaN / Inf
// count: the rare path of the per-channel amax pass, taken when a warp's
// packed maxima flag a NaN / Inf; it loads the elements again.
struct StripMax {
    uint32_t cm[4], rm[8], nf;
};
__device__ __noinline__ StripMax strip_exact(const uint16_t* x, int64_t R, int64_t C, int64_t r0, int64_t c) {
    StripMax e;
    e.nf = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) e.cm[k] = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = (c < C && r0 + i < R) ? ld_nc_v4(x + (r0 + i) * C + c) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t rm = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t f = finite_mag2(w[k]);
            e.nf += nonfinite2(w[k]);
            e.cm[k] = max_u16x2(e.cm[k], f);
            rm = max_u16x2(rm, f);
        }
        e.rm[i] = rm;
    }
    return e;
}

// Per-channel current scaling, pass 1: the largest finite |x| of every row
// (rowmax[r]) and of every column (colmax[c]) of x, as bf16 magnitude bits in
// uint32 words of the zeroed scale buffers (atomicMax merges the strips), and
// the NaN / Inf count.  CTA i walks the strips of 64 rows x 256 columns of
// column band i % bands, rows i / bands, + the grid's CTAs per band ...:
// warp w rows 8w .. 8w + 7, lane l columns 8l .. 8l + 7 (one 16-byte load a
// row); the column maxima stay in registers across the walk and meet in
// shared memory once at its end.  The common path takes the packed maxima of
// the magnitude bits (one AND and the u16x2 maxima a word) and leaves NaN /
// Inf to a rare exact path.
template <bool ROW, bool COL>
__global__ void __launch_bounds__(256, 4) pc_amax_kernel(const uint16_t* x, int64_t R, int64_t C, uint32_t* rowmax,
                                                         uint32_t* colmax, unsigned long long* counters) {
    __shared__ uint32_t cred[8][128];  // per warp: column-pair maxima of its rows
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // strips counted in 32 bits (the host refuses more than 2^31); the grid
    // is a multiple of the band count
    const uint32_t bands = (uint32_t)((C + 255) / 256), strips_r = (uint32_t)((R + 63) / 64);
    const uint32_t per_band = gridDim.x / bands, band = blockIdx.x % bands;
    const int64_t cs = (int64_t)band * 256, c = cs + 8 * lane;
    uint32_t nf = 0, cm[4] = {0u, 0u, 0u, 0u};
    for (uint32_t sr = blockIdx.x / bands; sr < strips_r; sr += per_band) {
        const int64_t r0 = (int64_t)sr * 64 + 8 * warp;
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)  // C % 8 == 0: a vector is wholly inside or outside
            v[i] = (c < C && r0 + i < R) ? ld_nc_v4(x + (r0 + i) * C + c) : make_uint4(0u, 0u, 0u, 0u);
        // packed maxima of the magnitude bits, NaN / Inf included (they are
        // >= 0x7F80, so the fold of all of them flags any)
        uint32_t sm[4] = {0u, 0u, 0u, 0u}, rm[8], all = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t M = 0x7FFF7FFFu;
            const uint32_t w[4] = {v[i].x & M, v[i].y & M, v[i].z & M, v[i].w & M};
#pragma unroll
            for (int k = 0; k < 4; ++k) sm[k] = max_u16x2(sm[k], w[k]);
            rm[i] = max_u16x2(max_u16x2(w[0], w[1]), max_u16x2(w[2], w[3]));
            all = max_u16x2(all, rm[i]);
        }
        if (__any_sync(0xFFFFFFFFu, fold16(all) >= 0x7F80u)) {  // NaN / Inf in the warp's rows: exact maxima
            const StripMax e = strip_exact(x, R, C, r0, c);
            nf += e.nf;
#pragma unroll
            for (int k = 0; k < 4; ++k) sm[k] = e.cm[k];
#pragma unroll
            for (int i = 0; i < 8; ++i) rm[i] = e.rm[i];
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) cm[k] = max_u16x2(cm[k], sm[k]);
        if constexpr (ROW) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, fold16(rm[i]));
                if (lane == 0 && m != 0u && r0 + i < R) atomicMax(rowmax + r0 + i, m);
            }
        }
    }
    if constexpr (COL) {
#pragma unroll
        for (int k = 0; k < 4; ++k) cred[warp][4 * lane + k] = cm[k];
        __syncthreads();
        if (threadIdx.x < 128) {
            uint32_t m = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) m = max_u16x2(m, cred[w][threadIdx.x]);
            const int64_t cc = cs + 2 * threadIdx.x;
            if (cc < C) {
                if (m & 0xFFFFu) atomicMax(colmax + cc, m & 0xFFFFu);
                if (m >> 16) atomicMax(colmax + cc + 1, m >> 16);
            }
        }
    }
    nf = warp_sum_u32(nf);
    if (lane == 0 && nf) atomicAdd(&counters[2], (unsigned long long)nf);
}

// Generic blockwise scaling (1 x b or b x b blocks, b = bc), pass 1: the
// largest finite |x| of every block, as bf16 magnitude bits in uint32 words of
// the zeroed scale buffers (atomicMax merges the strips), at the position the
// block's scale takes: 1 x b blocks in the row copy's [ceil(C/b)][Rp] and, for
// the column copy, the blocks of b rows of one column in [ceil(R/b)][Cp];
// b x b blocks in the row copy's [ceil(R/b)][ceil(C/b)], or without a row
// copy at the transposed position of the column copy's buffer.  NaN / Inf
// counted.  A CTA takes strips of 64 rows x 256 columns: warp w rows 8w ..
// 8w + 7, lane l columns 8l .. 8l + 7 (one 16-byte load a row); the bc / 8
// lanes of a block column meet by shuffles, the warps of a block of rows of
// one column through shared memory.
template <bool SQ, bool ROW, bool COL>
__global__ void __launch_bounds__(256) gen_amax_kernel(const uint16_t* x, int64_t R, int64_t C, int bc,
                                                       uint32_t* srow, uint32_t* scol,
                                                       unsigned long long* counters) {
    __shared__ uint32_t cred[8][128];  // per warp: column-pair maxima of its 8 rows
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int lg = bc / 8 < 32 ? bc / 8 : 32;  // lanes per block column
    const int64_t strips_c = (C + 255) / 256, strips = ((R + 63) / 64) * strips_c;
    const int64_t Rp = (R + 127) / 128 * 128, Cp = (C + 127) / 128 * 128;
    const int sh = __ffs(bc) - 1;  // b is a power of two
    const int64_t nbc = (C + bc - 1) >> sh, nbr = (R + bc - 1) >> sh;
    uint32_t nf = 0;
    for (int64_t sidx = blockIdx.x; sidx < strips; sidx += gridDim.x) {
        const int64_t rs = (sidx / strips_c) * 64, r0 = rs + 8 * warp, cs = (sidx % strips_c) * 256, c = cs + 8 * lane;
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)  // C % 8 == 0: a vector is wholly inside or outside
            v[i] = (c < C && r0 + i < R) ? ld_nc_v4(x + (r0 + i) * C + c) : make_uint4(0u, 0u, 0u, 0u);
        uint32_t cm[4] = {0u, 0u, 0u, 0u};
        uint32_t sq = 0;
        // packed magnitudes (one AND a word) unless a NaN / Inf is in the warp's
        // rows (a warp vote on their packed maximum): then the exact finite test
        uint32_t all = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) all = max_u16x2(all, vec_pmax(v[i]));
        const bool exact = __any_sync(0xFFFFFFFFu, fold16(all) >= 0x7F80u);
        auto rows = [&](auto exact_tag) {
            constexpr bool kExact = decltype(exact_tag)::value;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t rm = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t f = kExact ? finite_mag2(w[k]) : (w[k] & 0x7FFF7FFFu);
                    if (kExact) nf += nonfinite2(w[k]);
                    cm[k] = max_u16x2(cm[k], f);
                    rm = max_u16x2(rm, f);
                }
                uint32_t m = fold16(rm);
                if constexpr (!SQ && ROW) {
                    for (int o = 1; o < lg; o <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                    if (lane % lg == 0 && m != 0u && r0 + i < R && c < C) atomicMax(srow + (c >> sh) * Rp + r0 + i, m);
                }
                sq = max(sq, m);
            }
        };
        if (exact)
            rows(std::true_type{});
        else
            rows(std::false_type{});
        if constexpr (SQ) {  // the warp's 8 rows lie in one block row (b >= 32)
            for (int o = 1; o < lg; o <<= 1) sq = max(sq, __shfl_xor_sync(0xFFFFFFFFu, sq, o));
            if (lane % lg == 0 && sq != 0u && c < C) {
                const int64_t bi = r0 >> sh, bj = c >> sh;
                if (ROW)
                    atomicMax(srow + bi * nbc + bj, sq);
                else
                    atomicMax(scol + bj * nbr + bi, sq);
            }
        }
        if constexpr (!SQ && COL) {
#pragma unroll
            for (int k = 0; k < 4; ++k) cred[warp][4 * lane + k] = cm[k];
            __syncthreads();
            if (threadIdx.x < 128) {
                // the warps of one block of b rows: all eight (b >= 64; strips start
                // at multiples of 64) or four (b = 32)
                const int g = bc >= 64 ? 8 : 4;
                for (int g0 = 0; g0 < 8; g0 += g) {
                    uint32_t m = 0;
                    for (int w = g0; w < g0 + g; ++w) m = max_u16x2(m, cred[w][threadIdx.x]);
                    const int64_t cc = cs + 2 * threadIdx.x, rb = (rs + 8 * g0) >> sh;
                    if (cc < C && rs + 8 * g0 < R) {
                        if (m & 0xFFFFu) atomicMax(scol + rb * Cp + cc, m & 0xFFFFu);
                        if (m >> 16) atomicMax(scol + rb * Cp + cc + 1, m >> 16);
                    }
                }
            }
            __syncthreads();  // cred is rewritten by the next strip
        }
    }
    nf = warp_sum_u32(nf);
    if (lane == 0 && nf) atomicAdd(&counters[2], (unsigned long long)nf);
}

// Generic blockwise scaling, last pass: each entry of a scale buffer (a
// block's amax bits; 0 in pad entries) becomes d = RN(amax / fmax), amax 0 -> 1.
template <int FMT>
__global__ void gen_finalize_kernel(uint32_t* m, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        ((float*)m)[i] = block_scale<FMT>(__uint_as_float(m[i] << 16));
}

// Square blocks with both copies: the column copy's scales are the row copy's
// transposed, d of the amax bits [nbr][nbc] into [nbc][nbr] (run before the row
// buffer is finalized in place).
template <int FMT>
__global__ void gen_transpose_scales_kernel(const uint32_t* rowm, float* cold, int64_t nbr, int64_t nbc) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nbr * nbc;
         i += (int64_t)gridDim.x * blockDim.x)
        cold[(i % nbc) * nbr + i / nbc] = block_scale<FMT>(__uint_as_float(rowm[i] << 16));
}

// Per-channel current scaling, last pass: each entry of a scale buffer (a
// row's or column's amax bits, 0 past the copy's rows) becomes the
// dequantization factor fp32(1 / s), s = fmax / amax (amax 0 -> s = 1).
template <int FMT>
__global__ void pc_finalize_kernel(uint32_t* m, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        ((float*)m)[i] = __fdiv_rn(1.0f, pertensor_scale<FMT>(__uint_as_float(m[i] << 16)));
}

__global__ void delayed_update_kernel(DelayedDev* st, const float* amax, const unsigned long long* nonfinite) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    if (nonfinite != nullptr && *nonfinite != 0ull) return;
    const float am = *amax;
    if (!(fabsf(am) <= 3.402823466e38f)) return;
    const int H = st->H;
    st->hist[st->head] = am;
    st->head = (st->head + 1) % H;
    float m = 0.0f;
    for (int i = 0; i < H; ++i) m = fmaxf(m, st->hist[i]);
    float s;
    if (!(m > 0.0f)) {
        s = 1.0f;
    } else {
        s = __fdiv_rn(st->fmt == FP8Q_E4M3 ? 448.0f : 57344.0f, m);
        s = __fmul_rn(s, exp2_neg(st->margin));
        if (isinf(s)) s = 3.402823466e38f;
        // a large margin can push s below the normal range: the smallest
        // normal fp32 keeps 1 / s finite
        if (s < 1.175494351e-38f) s = 1.175494351e-38f;
    }
    st->scale = s;
    st->scale_inv = __fdiv_rn(1.0f, s);
}

template <int FMT>
__global__ void cast_bits_kernel(uint32_t start, uint64_t count, uint8_t* out) {
    const uint64_t i0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i0 >= count) return;
    float f[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) f[j] = __uint_as_float((uint32_t)(start + i0 + j));
    uint32_t q = cvt4<FMT>(f[0], f[1], f[2], f[3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t u = __float_as_uint(f[j]);
        if ((u & 0x7FFFFFFFu) > 0x7F800000u) q = (q & ~(0xFFu << (8 * j))) | ((((u >> 24) & 0x80u) | 0x7Fu) << (8 * j));
    }
    if (i0 + 4 <= count) {
        *(uint32_t*)(out + i0) = q;
    } else {
        for (uint64_t j = 0; i0 + j < count; ++j) out[i0 + j] = (uint8_t)(q >> (8 * j));
    }
}

// For every finite bf16 x and each divisor d[j] in the fast range whose
// quotient is below 2^126 in magnitude, compares div_rn_recip(x, d, RN(1/d))
// and the tile kernel's two-lane negated form (on x and -x) with the IEEE
// quotient: [0] counts FP8 codes that differ (all such pairs), [1] fp32
// results that differ where the IEEE quotient is at least 2^-24, plus the
// kernels' rcp_rn(d) against the IEEE reciprocal and their block_scale(x)
// against IEEE amax / fmax for every positive bf16 x.
template <int FMT>
__global__ void div_selftest_kernel(const float* d, int64_t nd, unsigned long long* mismatch) {
    const uint32_t xb = blockIdx.x * blockDim.x + threadIdx.x;  // bf16 pattern
    const float x = __uint_as_float(xb << 16);
    const bool xfin = (xb & 0x7F80u) != 0x7F80u;
    uint32_t bad_code = 0, bad_bits = 0;
    if (blockIdx.y == 0 && xfin && x > 0.0f &&  // the kernels' block divisor, every positive bf16 amax
        __float_as_uint(block_scale<FMT>(x)) != __float_as_uint(__fdiv_rn(x, Fmt<FMT>::fmax)))
        ++bad_bits;
    for (int64_t j = blockIdx.y; j < nd; j += gridDim.y) {
        const float dj = d[j];
        if (!xfin || !(dj >= 0x1p-80f) || !(dj < 0x1p+128f)) continue;
        const float exact = __fdiv_rn(x, dj);
        if (!(fabsf(exact) < 0x1p+126f)) continue;
        const float r = __frcp_rn(dj);
        if (xb == 0 && dj <= 0x1p+120f && __float_as_uint(rcp_rn(dj)) != __float_as_uint(r))
            ++bad_bits;  // the kernels' reciprocal, on its domain (a bf16 amax gives d < 2^120)
        const float fast = div_rn_recip(x, dj, r);
        // the two-lane, negated form the tile kernel runs (lane x: this pair)
        Factor f;
        f.k = dj;
        f.r = r;
        f.fast = true;
        const float2 ny = apply2<kB1>(make_float2(x, -x), pair_factor(f, f));
        const uint32_t ce = cvt2<FMT>(exact, -exact);
        const bool big = fabsf(exact) >= 0x1p-24f;
        bad_bits += big && __float_as_uint(exact) != __float_as_uint(fast);
        bad_bits += big && (__float_as_uint(exact) != __float_as_uint(-ny.x) ||
                            __float_as_uint(-exact) != __float_as_uint(-ny.y));
        bad_code += (ce & 0xFFu) != (cvt2<FMT>(fast, 0.0f) & 0xFFu);
        bad_code += ce != ((cvt2<FMT>(ny.x, ny.y) ^ 0x8080u) & 0xFFFFu);
    }
    bad_code = warp_sum_u32(bad_code);
    bad_bits = warp_sum_u32(bad_bits);
    if ((threadIdx.x & 31) == 0) {
        if (bad_code) atomicAdd(&mismatch[0], (unsigned long long)bad_code);
        if (bad_bits) atomicAdd(&mismatch[1], (unsigned long long)bad_bits);
    }
}

// SMs of the current device (at least 1, so that a grid size stays valid; a
// device that cannot be queried fails at the launch instead).
int num_sms() {
    const int n = sm_count();
    return n > 0 ? n : 1;
}

template <int KIND, int FMT, bool ROW, bool COL, int GEN = kGenNone>
fp8q_status launch_tile(const QuantArgs& args, cudaStream_t s) {
    QuantArgs a = args;
    a.stall = take_stall();
    static PerDevice<bool> attr;
    auto kern = quant_tile_kernel<KIND, FMT, ROW, COL, GEN>;
    if (!smem_opt_in(attr, kern, kTileSmem)) return FP8Q_ERR_CUDA;
    const int64_t ntiles = a.tiles_r * a.tiles_c;
    if (a.tiles_r_total * a.tiles_c >= ((int64_t)1 << 31)) return FP8Q_ERR_SHAPE;  // tiles counted in 32 bits
    CUtensorMap tm, trow, tcol;
    memset(&tm, 0, sizeof(tm));
    memset(&trow, 0, sizeof(trow));
    memset(&tcol, 0, sizeof(tcol));
    if (ntiles > 0) {
        if (!make_map_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.x, a.R, a.C, kTile / 2, kTile,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return FP8Q_ERR_CUDA;
        // code tiles [128][128] in the 128-byte swizzle: row copy [R][C], column copy [C][R]
        if (ROW && !make_map_2d(&trow, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.q_row, a.R_total, a.C, kTile, kTile,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return FP8Q_ERR_CUDA;
        if (COL && !make_map_2d(&tcol, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.q_col, a.C, a.R_total, kTile, kTile,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return FP8Q_ERR_CUDA;
    }
    int64_t grid = (int64_t)num_sms() * 2;
    if (a.grid_cap > 0 && a.grid_cap < grid) grid = a.grid_cap;
    if (ntiles < grid) grid = ntiles;
    if (grid < 1) grid = 1;
    kern<<<(unsigned)grid, kThreads, kTileSmem, s>>>(tm, trow, tcol, a);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

template <int KIND, int FMT, int GEN = kGenNone>
fp8q_status launch_tile_rc(const QuantArgs& a, bool row, bool col, cudaStream_t s) {
    if (row && col) return launch_tile<KIND, FMT, true, true, GEN>(a, s);
    if (row) return launch_tile<KIND, FMT, true, false, GEN>(a, s);
    return launch_tile<KIND, FMT, false, true, GEN>(a, s);
}

template <int KIND, int GEN = kGenNone>
fp8q_status launch_tile_fmt(const QuantArgs& a, int fmt, bool row, bool col, cudaStream_t s) {
    return fmt == FP8Q_E4M3 ? launch_tile_rc<KIND, FP8Q_E4M3, GEN>(a, row, col, s)
                            : launch_tile_rc<KIND, FP8Q_E5M2, GEN>(a, row, col, s);
}

// Generic blockwise scaling of shapes other than 1 x 128 / 128 x 128.  Blocks
// of 32 or 64: the tile pass alone (block maxima inside each tile).  Blocks
// of 256: zero the scale buffers, the block-amax pass into them, the tile
// pass (reads them), then the buffers' amax bits become d (for square blocks
// with both copies the column copy's scales are the row copy's transposed).
fp8q_status launch_generic(const QuantArgs& a, int fmt, bool row, bool col, cudaStream_t s) {
    const int64_t Rp = a.tiles_r * 128, Cp = a.tiles_c * 128;
    if (Rp == 0 || Cp == 0) return FP8Q_OK;  // empty x: nothing to write
    const int bc = a.bc;
    const bool sq = a.br == a.bc;
    if (bc <= 64)
        return sq ? launch_tile_fmt<kGen, kGenTileSq>(a, fmt, row, col, s)
                  : launch_tile_fmt<kGen, kGenTile1D>(a, fmt, row, col, s);
    const int64_t nbr = (a.R + bc - 1) / bc, nbc = (a.C + bc - 1) / bc;
    const int64_t row_n = sq ? nbr * nbc : nbc * Rp, col_n = sq ? nbr * nbc : nbr * Cp;
    uint32_t* rm = (uint32_t*)a.s_row;
    uint32_t* cm = (uint32_t*)a.s_col;
    if (row && cudaMemsetAsync(rm, 0, (size_t)row_n * 4, s) != cudaSuccess) return FP8Q_ERR_CUDA;
    if (col && cudaMemsetAsync(cm, 0, (size_t)col_n * 4, s) != cudaSuccess) return FP8Q_ERR_CUDA;
    const int64_t strips = ((a.R + 63) / 64) * ((a.C + 255) / 256);
    int64_t grid = (int64_t)num_sms() * 8;
    if (strips < grid) grid = strips;
    const unsigned g = (unsigned)grid;
    if (sq) {
        if (row)
            gen_amax_kernel<true, true, false><<<g, 256, 0, s>>>(a.x, a.R, a.C, bc, rm, cm, a.counters);
        else
            gen_amax_kernel<true, false, true><<<g, 256, 0, s>>>(a.x, a.R, a.C, bc, rm, cm, a.counters);
    } else if (row && col) {
        gen_amax_kernel<false, true, true><<<g, 256, 0, s>>>(a.x, a.R, a.C, bc, rm, cm, a.counters);
    } else if (row) {
        gen_amax_kernel<false, true, false><<<g, 256, 0, s>>>(a.x, a.R, a.C, bc, rm, cm, a.counters);
    } else {
        gen_amax_kernel<false, false, true><<<g, 256, 0, s>>>(a.x, a.R, a.C, bc, rm, cm, a.counters);
    }
    if (cudaGetLastError() != cudaSuccess) return FP8Q_ERR_CUDA;
    const fp8q_status r = sq ? launch_tile_fmt<kGen, kGenPassSq>(a, fmt, row, col, s)
                             : launch_tile_fmt<kGen, kGenPass1D>(a, fmt, row, col, s);
    if (r != FP8Q_OK) return r;
    auto blocks = [](int64_t n) { return (unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096); };
    const bool e4 = fmt == FP8Q_E4M3;
    if (sq && row && col) {
        if (e4)
            gen_transpose_scales_kernel<FP8Q_E4M3><<<blocks(row_n), 256, 0, s>>>(rm, (float*)cm, nbr, nbc);
        else
            gen_transpose_scales_kernel<FP8Q_E5M2><<<blocks(row_n), 256, 0, s>>>(rm, (float*)cm, nbr, nbc);
        if (cudaGetLastError() != cudaSuccess) return FP8Q_ERR_CUDA;
    }
    for (int w = 0; w < 2; ++w) {
        // in place: the row buffer; the column buffer unless it was filled above
        if (w == 0 ? !row : (!col || (sq && row))) continue;
        uint32_t* m = w == 0 ? rm : cm;
        const int64_t n = w == 0 ? row_n : col_n;
        if (e4)
            gen_finalize_kernel<FP8Q_E4M3><<<blocks(n), 256, 0, s>>>(m, n);
        else
            gen_finalize_kernel<FP8Q_E5M2><<<blocks(n), 256, 0, s>>>(m, n);
        if (cudaGetLastError() != cudaSuccess) return FP8Q_ERR_CUDA;
    }
    return FP8Q_OK;
}

// Per-channel current: zero the scale buffers, the amax pass into them, the
// tile pass (reads them), then the buffers' amax bits become fp32(1 / s).
fp8q_status launch_perchannel(const QuantArgs& a, int fmt, bool row, bool col, cudaStream_t s) {
    const int64_t Rp = a.tiles_r * 128, Cp = a.tiles_c * 128;
    if (Rp == 0 || Cp == 0) return FP8Q_OK;  // empty x: nothing to write
    // a block of rows (fp8q_quantize_rows) owns entries row0 .. row0 + Rp - 1
    uint32_t* rm = a.s_row ? (uint32_t*)a.s_row + a.row0 : nullptr;
    if (row && cudaMemsetAsync(rm, 0, (size_t)Rp * sizeof(float), s) != cudaSuccess) return FP8Q_ERR_CUDA;
    if (col && cudaMemsetAsync(a.s_col, 0, (size_t)Cp * sizeof(float), s) != cudaSuccess) return FP8Q_ERR_CUDA;
    const int64_t bands = (a.C + 255) / 256, strips_r = (a.R + 63) / 64;
    if (bands * strips_r >= ((int64_t)1 << 31)) return FP8Q_ERR_SHAPE;  // strips counted in 32 bits
    // CTAs per column band: about four resident CTAs per SM in all, at most
    // one per strip of the band; the grid is a multiple of the band count
    int64_t per_band = (int64_t)num_sms() * 4 / bands;
    if (per_band < 1) per_band = 1;
    if (per_band > strips_r) per_band = strips_r;
    const int64_t grid = bands * per_band;
    uint32_t* cm = (uint32_t*)a.s_col;
    if (row && col)
        pc_amax_kernel<true, true><<<(unsigned)grid, 256, 0, s>>>(a.x, a.R, a.C, rm, cm, a.counters);
    else if (row)
        pc_amax_kernel<true, false><<<(unsigned)grid, 256, 0, s>>>(a.x, a.R, a.C, rm, cm, a.counters);
    else
        pc_amax_kernel<false, true><<<(unsigned)grid, 256, 0, s>>>(a.x, a.R, a.C, rm, cm, a.counters);
    if (cudaGetLastError() != cudaSuccess) return FP8Q_ERR_CUDA;
    const fp8q_status r = launch_tile_fmt<kPC>(a, fmt, row, col, s);
    if (r != FP8Q_OK) return r;
    for (int w = 0; w < 2; ++w) {
        if (w == 0 ? !row : !col) continue;
        uint32_t* m = w == 0 ? rm : cm;
        const int64_t n = w == 0 ? Rp : Cp;
        const unsigned blocks = (unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
        if (fmt == FP8Q_E4M3)
            pc_finalize_kernel<FP8Q_E4M3><<<blocks, 256, 0, s>>>(m, n);
        else
            pc_finalize_kernel<FP8Q_E5M2><<<blocks, 256, 0, s>>>(m, n);
        if (cudaGetLastError() != cudaSuccess) return FP8Q_ERR_CUDA;
    }
    return FP8Q_OK;
}

}  // namespace

fp8q_status launch_quantize(const fp8q_recipe* rc, const QuantArgs& a, DelayedDev* st, cudaStream_t s) {
    const bool row = rc->want_rowwise != 0, col = rc->want_colwise != 0;
    if (!a.add_counters && cudaMemsetAsync(a.counters, 0, 3 * sizeof(unsigned long long), s) != cudaSuccess)
        return FP8Q_ERR_CUDA;
    switch (rc->kind) {
        case kCur: {
            if (cudaMemsetAsync(a.amax, 0, sizeof(float), s) != cudaSuccess) return FP8Q_ERR_CUDA;
            const int64_t nvec = a.R * a.C / 8;
            if (nvec > 0) {
                int64_t grid = (int64_t)num_sms() * 4;
                const int64_t need = (nvec + kThreads * 4 - 1) / (kThreads * 4);
                if (need < grid) grid = need;
                amax_kernel<<<(unsigned)grid, kThreads, 0, s>>>(a.x, nvec, a.amax, a.counters);
                if (cudaGetLastError() != cudaSuccess) return FP8Q_ERR_CUDA;
            }
            return launch_tile_fmt<kCur>(a, rc->fmt, row, col, s);
        }
        case kDel: {
            if (cudaMemsetAsync(a.amax, 0, sizeof(float), s) != cudaSuccess) return FP8Q_ERR_CUDA;
            fp8q_status r = launch_tile_fmt<kDel>(a, rc->fmt, row, col, s);
            if (r != FP8Q_OK) return r;
            return launch_delayed_update(st, a.amax, a.counters + 2, s);
        }
        case kB1:
            return launch_tile_fmt<kB1>(a, rc->fmt, row, col, s);
        case kB128:
            return launch_tile_fmt<kB128>(a, rc->fmt, row, col, s);
        case kMX:
            return launch_tile_fmt<kMX>(a, rc->fmt, row, col, s);
        case kPC:
            return launch_perchannel(a, rc->fmt, row, col, s);
        case kGen:  // 1 x 128 and 128 x 128 are the specialised kinds' kernels
            if (a.br == 1 && a.bc == 128) return launch_tile_fmt<kB1>(a, rc->fmt, row, col, s);
            if (a.br == 128 && a.bc == 128) return launch_tile_fmt<kB128>(a, rc->fmt, row, col, s);
            return launch_generic(a, rc->fmt, row, col, s);
        default:
            return FP8Q_ERR_ARG;
    }
}


// Fork / join of fp8q_quantize_multi: one library-owned stream per job
// (created once per device), the tile passes' two resident CTAs per SM
// shared out by the jobs' tile counts.
namespace {
std::mutex g_multi_mu;
struct MultiStreams {
    cudaStream_t s[FP8Q_MULTI_MAX];
    cudaEvent_t fork, join[FP8Q_MULTI_MAX];
    bool ready;
};
MultiStreams g_multi[64];
}  // namespace

fp8q_status launch_quantize_multi(int n, const fp8q_recipe* const* rcs, QuantArgs* a, DelayedDev* const* sts,
                                  cudaStream_t s) {
    if (n == 0) return FP8Q_OK;
    if (n == 1) return launch_quantize(rcs[0], a[0], sts[0], s);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8Q_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_multi_mu);
    MultiStreams& m = g_multi[dev];
    if (!m.ready) {
        for (int i = 0; i < FP8Q_MULTI_MAX; ++i) {
            if (cudaStreamCreateWithFlags(&m.s[i], cudaStreamNonBlocking) != cudaSuccess ||
                cudaEventCreateWithFlags(&m.join[i], cudaEventDisableTiming) != cudaSuccess)
                return FP8Q_ERR_CUDA;
        }
        if (cudaEventCreateWithFlags(&m.fork, cudaEventDisableTiming) != cudaSuccess) return FP8Q_ERR_CUDA;
        m.ready = true;
    }
    // each job's share of the resident CTAs follows its tiles weighted by
    // their cost: a re-quantized column copy (1 x 128 blocks, MXFP8) takes a
    // second conversion per element, the byte transposes do not (measured on
    // the Llama-3-8B up-projection's X 1 x 128 + W 128 x 128, both copies:
    // 66.5 us with equal weights, 60 us with 1.3 - 1.6 for X's tiles)
    auto weight = [&](int i) -> int64_t {
        if (!rcs[i]->want_colwise) return 100;
        if (rcs[i]->kind == kB1 || (rcs[i]->kind == kGen && rcs[i]->block_rows == 1)) return 145;
        return rcs[i]->kind == kMX ? 120 : 100;
    };
    int64_t total = 0;
    for (int i = 0; i < n; ++i) total += a[i].tiles_r * a[i].tiles_c * weight(i);
    const int64_t budget = (int64_t)num_sms() * 2;
    if (cudaEventRecord(m.fork, s) != cudaSuccess) return FP8Q_ERR_CUDA;
    fp8q_status r = FP8Q_OK;
    for (int i = 0; i < n; ++i) {
        const int64_t tiles = a[i].tiles_r * a[i].tiles_c * weight(i);
        a[i].grid_cap = total > 0 ? (budget * tiles / total > 0 ? budget * tiles / total : 1) : 0;
        if (cudaStreamWaitEvent(m.s[i], m.fork, 0) != cudaSuccess) return FP8Q_ERR_CUDA;
        const fp8q_status ri = launch_quantize(rcs[i], a[i], sts[i], m.s[i]);
        if (ri != FP8Q_OK && r == FP8Q_OK) r = ri;
        // join even after a failed launch: the caller's stream never waits on a
        // job that was not enqueued behind the fork
        if (cudaEventRecord(m.join[i], m.s[i]) != cudaSuccess || cudaStreamWaitEvent(s, m.join[i], 0) != cudaSuccess)
            return FP8Q_ERR_CUDA;
    }
    return r;
}

fp8q_status launch_div_selftest(const float* d, int64_t nd, int fmt, unsigned long long* mismatch, cudaStream_t s) {
    if (cudaMemsetAsync(mismatch, 0, 2 * sizeof(unsigned long long), s) != cudaSuccess) return FP8Q_ERR_CUDA;
    if (nd <= 0) return FP8Q_OK;
    const dim3 grid(65536 / 256, (unsigned)(nd < 4096 ? nd : 4096));
    if (fmt == FP8Q_E4M3)
        div_selftest_kernel<FP8Q_E4M3><<<grid, 256, 0, s>>>(d, nd, mismatch);
    else
        div_selftest_kernel<FP8Q_E5M2><<<grid, 256, 0, s>>>(d, nd, mismatch);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

fp8q_status read_quant_errors(unsigned int* flags) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_quant_errors, sizeof(v)) != cudaSuccess) return FP8Q_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_quant_errors, &zero, sizeof(zero)) != cudaSuccess) return FP8Q_ERR_CUDA;
    *flags |= v;
    return FP8Q_OK;
}

fp8q_status launch_delayed_update(DelayedDev* st, const float* amax, const unsigned long long* nonfinite,
                                  cudaStream_t s) {
    delayed_update_kernel<<<1, 32, 0, s>>>(st, amax, nonfinite);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

fp8q_status launch_cast_bits(uint32_t start, uint64_t count, int fmt, uint8_t* out, cudaStream_t s) {
    if (count == 0) return FP8Q_OK;
    const uint64_t threads = (count + 3) / 4;
    const uint64_t blocks = (threads + 255) / 256;
    if (fmt == FP8Q_E4M3)
        cast_bits_kernel<FP8Q_E4M3><<<(unsigned)blocks, 256, 0, s>>>(start, count, out);
    else
        cast_bits_kernel<FP8Q_E5M2><<<(unsigned)blocks, 256, 0, s>>>(start, count, out);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

}  // namespace fp8q
