// Scaled FP8 GEMM on SM pairs: tcgen05.mma.cta_group::2 (M = 256).
//
// Same arithmetic as gemm.cu ("2025 FP8 quantized-training guide", sec. 2.1-2.3
// and 3.1): D = A_q . B_q^T with per-tensor, MXFP8 (block-scaled MMA) or
// blockwise (per-128-K partials scaled in the epilogue) scales.  A cluster of
// two CTAs on two SMs computes a 256 x BN tile (BN = 256): CTA r
// loads rows 256 mp + 128 r of A and rows BN nb + (BN / 2) r of B, and the
// leader CTA (r = 0) issues each MMA for both, so every SM streams half of the
// B panel it would need alone and each shared-memory stage is a third smaller.
//
// Per CTA: warp 0 TMA producer (its halves, completing on the leader's
// barriers), warp 1 TMEM allocation (with the peer) and, in the leader, the
// single-thread MMA issuer; then the epilogue warps for the CTA's own 128
// rows (TMEM lanes 32 (w % 4) .., columns EC ((w - 2) / 4) ..), which release
// TMEM on the leader's barrier and store D by TMA: eight warps of 128
// columns (320 threads).  One more warp (352 threads) for two recipes.
// Blockwise: it loads each K block's scales into a ring of shared-memory
// slots, apart from the operand producer, whose loads would otherwise queue
// behind the ring's waits (measured: 0.626 -> 0.646 of peak at the
// Llama-3-8B up-projection).  MXFP8: in the leader it copies each stage's
// scale tiles (landed with the operands) into both CTAs' TMEM with
// tcgen05.cp and commits to a barrier the MMA issuer waits on (measured:
// 0.763 -> 0.799 at the Llama-3-8B MLP fprop against moving them with the
// epilogue warps' tcgen05.st).  Blockwise: with two K-block partial buffers
// the MMAs of K block g + 2 wait for the epilogue to release block g, which
// is what limits this recipe (measured: about 445 cycles from a partial's
// arrival to its release against about 600 cycles of MMAs per K block).
// The epilogue can also quantize D for the next layer (MXFP8 1x32 or 1x128,
// row-wise along N and optionally column-wise along M, the transposed copy a
// wgrad reads): the row blocks lie in a lane's registers; for the column
// blocks each warp transposes its rows through shared memory, 32 columns at
// a time, so that a lane holds a column's 32 rows -- a whole 32-row block,
// or a quarter of a 128-row one, whose four warps then exchange their maxima
// through shared memory on a bounded mbarrier.
// TMEM per CTA: per-tensor two 256-column accumulators; MXFP8 one accumulator
// plus 12 scale columns per stage; blockwise two 256-column partial buffers,
// so the MMAs run one K block ahead of the epilogue.
// All mbarrier waits are bounded as in gemm.cu; both CTAs always reach the
// closing cluster barrier, so neither exits while its shared memory or TMEM
// can still be used by the pair.
#include <string.h>

#include <type_traits>

#include "fp8q_internal.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace fp8q {

__device__ unsigned int g_device_errors2 = 0;

namespace {

constexpr int BM = 128, BK = 128;
// recipes: per-tensor, MXFP8, blockwise 1x128 x 128x128 / 1x128 x 1x128, per-channel
enum { REC_PT = 0, REC_MX = 1, REC_B2D = 2, REC_B1D = 3, REC_PC = 4 };

template <int REC>
struct Cfg {
    static constexpr bool BLOCKWISE = REC == REC_B2D || REC == REC_B1D;
    // pair tile columns and epilogue warps (two per TMEM lane quarter).  The
    // code also runs blockwise tiles of 192 columns with twelve warps of 64
    // columns, which measured slower (0.50 vs 0.63 of peak at the Llama-3-8B
    // up-projection)
    static constexpr int BN = 256;
    static constexpr int BH = BN / 2;  // B rows per CTA
    static constexpr int EPI_WARPS = 8;
    // blockwise: the scale ring's producer; MXFP8: the copier of each stage's
    // scale tiles into TMEM (in the leader CTA)
    static constexpr int SCALE_WARP = 2 + EPI_WARPS;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS + ((BLOCKWISE || REC == REC_MX) ? 32 : 0);
    static constexpr int STAGES = BLOCKWISE ? 4 : 5;
    static constexpr int NACC = (REC == REC_MX) ? 1 : 2;  // TMEM accumulators (blockwise: K-block partials)
    static constexpr int EPI_COLS = BN / (EPI_WARPS / 4);
    // blockwise scales ring: per K block, this CTA's 128 A-row scales (512 B)
    // and the tile's B scales (two floats for 128x128 blocks, BN for 1x128);
    // deep enough that the scale producer runs ahead of the MMAs
    static constexpr int SR = BLOCKWISE ? STAGES + NACC + 2 : 0;
    static constexpr uint32_t SLOT = 512 + 4 * BN;
    static constexpr uint32_t A_STAGE = BM * BK, B_STAGE = BH * BK;
    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_STAGE;
    static constexpr uint32_t OFF_SFB = OFF_SFA + (REC == REC_MX ? STAGES * 512 : 0);
    static constexpr uint32_t OFF_SCL = OFF_SFB + (REC == REC_MX ? STAGES * 1024 : 0);
    static constexpr uint32_t OFF_STG = OFF_SCL + SR * SLOT;
    static constexpr uint32_t STG_WARP = 4096;  // four 1 KB output boxes per epilogue warp
    static constexpr uint32_t OFF_BAR = OFF_STG + EPI_WARPS * STG_WARP;
    static constexpr int NSFB = (REC == REC_MX) ? STAGES : 0;  // MXFP8: a stage's scale tiles are in TMEM
    static constexpr uint32_t NBARS = 2 * STAGES + 2 * NACC + 1 + 2 * SR + NSFB;
    static constexpr uint32_t OFF_MISC = OFF_BAR + 8 * NBARS;
    static constexpr uint32_t SMEM = OFF_MISC + 16 + 1024;
    // the fused column-wise copy (kernels with it allocate these): the 1x128
    // exchange of column maxima ([tile parity][column half][4 warps][128
    // columns] words) and its mbarriers ([tile parity][column half][32-column
    // chunk]), then each epilogue warp's transpose area (2.25 KB)
    static constexpr uint32_t OFF_XB = OFF_MISC + 16;
    static constexpr uint32_t OFF_XBAR = OFF_XB + 2 * 2 * 4 * 128 * 4;
    static constexpr uint32_t OFF_TR = (OFF_XBAR + 16 * 8 + 15) / 16 * 16;
    static constexpr uint32_t TR_WARP = 16 * 36 * 4;  // 16 words of 32 rows, 36-word stride
    static constexpr uint32_t SMEM_COL = OFF_TR + EPI_WARPS * TR_WARP + 1024;
    static_assert(SMEM_COL <= 232448, "shared memory budget of one CTA with the column-wise copy");
    static_assert(SMEM <= 232448, "shared memory budget of one CTA");
};

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_TMEM_COL = 256;

struct Params2 {
    int64_t M, N, K;
    int64_t tiles_m2, tiles_n, nkb, tiles_m128, nbn128;
    int64_t nkbq, nbnq;              // blockwise: K blocks of the scales (KB wide), B's KB-row blocks
    const float* sa_inv;
    const float* sb_inv;
    const float* bsa;
    const float* bsb;
    int64_t Mp, Np;
    uint32_t idesc;
    // fused quantization of the bf16 output (QOut<QF> below)
    uint8_t* qscale;                 // MXFP8: packed 128x4 E8M0 tiles; 1x128: fp32 [ceil(N/128)][Mp]
    void* qscale_col;                // column copy: MXFP8 packed tiles of [N][ceil(M/32)]; 1x128 fp32 [ceil(M/128)][Np]
    unsigned long long* qcounters;   // [0] saturated (row copy), [1] saturated (column copy), [2] NaN / Inf
    int hasD;                        // also store the bf16 D
    uint64_t wait_ns;                // bounded-wait limit
    int stall;                       // 1: the producers issue no loads (diagnostic)
};

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Arrive on an mbarrier of a CTA of the cluster (default semantics: release
// at CTA scope; a cluster-scope release costs about a microsecond per arrive).
// The TMEM reads this signal covers have completed (tcgen05.wait::ld) before it.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_wait2(uint32_t a, uint32_t parity, volatile int* abort_flag, uint64_t limit_ns) {
    if (mbar_try(a, parity)) return true;
    return mbar_wait_bounded(a, parity, abort_flag, &g_device_errors2, 1u, limit_ns);
}
// TMA load into this CTA's shared memory (its shared::cta address, which is
// also its shared::cluster address) completing on an mbarrier given by a
// shared::cluster address, here always the leader CTA's.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(mbar)
        : "memory");
}
// 4-byte asynchronous copy whose completion is reported to an mbarrier by
// cp_async_arrive (which does not raise the barrier's pending count: the
// barrier's initial count includes it).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint32_t mbar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void tc2_commit_both(uint32_t mbar) {
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            mbar),
        "h"(mask)
        : "memory");
}
// 32 rows x 128 bits of shared memory into TMEM, replicated to the four lane
// quarters, in both CTAs of the pair (each from its own shared memory)
__device__ __forceinline__ void tc2_cp_32x128b(uint32_t taddr, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
__device__ __forceinline__ void tc2_commit_local(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void mma2_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma2_mx(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
            d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc));
}

// Stores this warp's 32 rows x COLS columns through its staging area of NBOX
// 1 KB boxes of 32-byte row pieces (32-byte swizzle: chunk c of row r at
// r*32 + (c ^ ((r / 4) % 2))*16); waits for the staging to be read out each
// time all NBOX boxes are in flight.
template <bool OUT_F32, int COLS, int NBOX>
__device__ __forceinline__ void store_slice2(const CUtensorMap* mapD, uint8_t* stg, uint32_t stg_s, int lane, int x0,
                                             int y0, int n_extent, int m_extent, const float* v, float scale) {
    constexpr int kPiece = OUT_F32 ? 8 : 16;  // columns per 32-byte row piece
    constexpr int kBoxes = COLS / kPiece;
    const int r = lane, sw = (r >> 2) & 1;
    bulk_wait_read();  // the previous tile's boxes have left the staging area
    __syncwarp();
#pragma unroll
    for (int bx = 0; bx < kBoxes; ++bx) {
        if (bx > 0 && bx % NBOX == 0) {
            bulk_wait_read();
            __syncwarp();
        }
        uint8_t* box = stg + (bx % NBOX) * 1024;
        const float* q = v + kPiece * bx;
        uint4 c0, c1;
        if (!OUT_F32) {
            c0 = make_uint4(pack_bf16(q[0] * scale, q[1] * scale), pack_bf16(q[2] * scale, q[3] * scale),
                            pack_bf16(q[4] * scale, q[5] * scale), pack_bf16(q[6] * scale, q[7] * scale));
            c1 = make_uint4(pack_bf16(q[8] * scale, q[9] * scale), pack_bf16(q[10] * scale, q[11] * scale),
                            pack_bf16(q[12] * scale, q[13] * scale), pack_bf16(q[14] * scale, q[15] * scale));
        } else {
            c0 = make_uint4(__float_as_uint(q[0] * scale), __float_as_uint(q[1] * scale), __float_as_uint(q[2] * scale),
                            __float_as_uint(q[3] * scale));
            c1 = make_uint4(__float_as_uint(q[4] * scale), __float_as_uint(q[5] * scale), __float_as_uint(q[6] * scale),
                            __float_as_uint(q[7] * scale));
        }
        *(uint4*)(box + r * 32 + ((0 ^ sw) << 4)) = c0;
        *(uint4*)(box + r * 32 + ((1 ^ sw) << 4)) = c1;
        fence_async_smem();
        __syncwarp();
        if (lane == 0 && x0 + kPiece * bx < n_extent && y0 < m_extent) {
            tma_store_2d(mapD, x0 + kPiece * bx, y0, stg_s + (bx % NBOX) * 1024);
            bulk_commit();
        }
    }
}

// MXFP8 (1x32 along N) quantization of this warp's 32 rows x COLS columns of
// D as stored in bf16 (RN(v scale), as store_slice2 writes it): per 32-column
// block the amax over finite |x|, e = floor(log2 amax) - emax_elem clamped to
// [-127, 127] (E8M0 e + 127), codes sat_rne(x 2^-e) with a NaN keeping its
// sign, saturated / NaN-Inf elements counted -- the quantize kernel's MXFP8
// row path ("2025 FP8 quantized-training guide", sec. 2.3) on these values.
// Codes leave through the staging boxes by TMA (uint8 32 x 32 boxes, 32-byte
// swizzle); each row's four scale bytes of a 128-column group go to the packed
// 128x4 tile layout.  Blocks past N and rows past M are not counted; scales
// are written for rows up to Mp and columns up to Np (blocks past M or N get
// code 127, the pad).
template <int QFMT, int COLS, int NBOX>
__device__ __forceinline__ void store_q(const CUtensorMap* mapQ, uint8_t* stg, uint32_t stg_s, int lane, int x0, int y0,
                                        const Params2& p, const float* v, float scale, uint32_t& nsat, uint32_t& nnf) {
    static_assert(COLS == 128 || COLS == 64, "a slice is all or half of one 128-column scale group");
    const int r = lane, sw = (r >> 2) & 1;
    const int64_t row = (int64_t)y0 + r;
    const bool row_live = row < p.M;
    uint32_t ebytes = 0;
    bulk_wait_read();  // the D boxes have left the staging area
    __syncwarp();
#pragma unroll
    for (int b = 0; b < COLS / 32; ++b) {
        uint32_t h[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) h[i] = pack_bf16(v[32 * b + 2 * i] * scale, v[32 * b + 2 * i + 1] * scale);
        const bool live = row_live && (int64_t)x0 + 32 * b < p.N;
        uint32_t pm = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) pm = max_u16x2(pm, h[i] & 0x7FFF7FFFu);
        uint32_t m = max(pm & 0xFFFFu, pm >> 16);
        const bool nf = m >= 0x7F80u;
        if (nf) {  // exact finite maximum; NaN / Inf counted
            m = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const uint32_t a = (h[i / 2] >> (16 * (i & 1))) & 0x7FFFu;
                if (a < 0x7F80u)
                    m = a > m ? a : m;
                else if (live)
                    ++nnf;
            }
        }
        if (!live) m = 0;
        const int e = mx_exponent<QFMT>(m << 16);
        const float k = exp2_neg(e);
        ebytes |= (uint32_t)(e + 127) << (8 * b);
        const float2 k2 = make_float2(k, k);
        const bool sat = live && __uint_as_float(m << 16) * k > Fmt<QFMT>::fmax;
        uint32_t c[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 y0 = __fmul2_rn(make_float2(__uint_as_float(h[2 * i] << 16), __uint_as_float(h[2 * i] & 0xFFFF0000u)), k2);
            const float2 y1 = __fmul2_rn(
                make_float2(__uint_as_float(h[2 * i + 1] << 16), __uint_as_float(h[2 * i + 1] & 0xFFFF0000u)), k2);
            c[i] = cvt4<QFMT>(y0.x, y0.y, y1.x, y1.y);
            if (sat)
                nsat += (fabsf(y0.x) <= 3.402823466e38f && fabsf(y0.x) > Fmt<QFMT>::fmax) +
                        (fabsf(y0.y) <= 3.402823466e38f && fabsf(y0.y) > Fmt<QFMT>::fmax) +
                        (fabsf(y1.x) <= 3.402823466e38f && fabsf(y1.x) > Fmt<QFMT>::fmax) +
                        (fabsf(y1.y) <= 3.402823466e38f && fabsf(y1.y) > Fmt<QFMT>::fmax);
            if (nf) {  // the hardware's NaN code is 0x7F whatever the sign
                uint32_t lo = c[i] & 0xFFFFu, hi = c[i] >> 16;
                if ((h[2 * i] & 0x7FFFu) > 0x7F80u) lo = (lo & ~0xFFu) | ((h[2 * i] >> 8) & 0x80u) | 0x7Fu;
                if ((h[2 * i] & 0x7FFF0000u) > 0x7F800000u) lo = (lo & ~0xFF00u) | ((h[2 * i] >> 16) & 0x8000u) | 0x7F00u;
                if ((h[2 * i + 1] & 0x7FFFu) > 0x7F80u) hi = (hi & ~0xFFu) | ((h[2 * i + 1] >> 8) & 0x80u) | 0x7Fu;
                if ((h[2 * i + 1] & 0x7FFF0000u) > 0x7F800000u)
                    hi = (hi & ~0xFF00u) | ((h[2 * i + 1] >> 16) & 0x8000u) | 0x7F00u;
                c[i] = lo | (hi << 16);
            }
        }
        if (b > 0 && b % NBOX == 0) {
            bulk_wait_read();
            __syncwarp();
        }
        uint8_t* box = stg + (b % NBOX) * 1024;
        *(uint4*)(box + r * 32 + ((0 ^ sw) << 4)) = make_uint4(c[0], c[1], c[2], c[3]);
        *(uint4*)(box + r * 32 + ((1 ^ sw) << 4)) = make_uint4(c[4], c[5], c[6], c[7]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0 && (int64_t)x0 + 32 * b < p.N && (int64_t)y0 < p.M) {
            tma_store_2d(mapQ, x0 + 32 * b, y0, stg_s + (b % NBOX) * 1024);
            bulk_commit();
        }
    }
    if (row < p.Mp && (int64_t)x0 < p.Np) {  // pads of the last 128-column group included (code 127)
        const int64_t tile = (row / 128) * p.nbn128 + x0 / 128;
        uint8_t* dst = p.qscale + tile * 512 + (row % 32) * 16 + ((row % 128) / 32) * 4 + (x0 % 128) / 32;
        if (COLS == 128)
            *(uint32_t*)dst = ebytes;
        else
            *(uint16_t*)dst = (uint16_t)ebytes;
    }
}

// The exact finite maximum of 128 bf16 (two to a word) and the NaN / Inf
// count among the first `live` of them: the rare path of store_q128, out of
// line so that the common path stays compact.
struct Bf16x128 {
    uint32_t w[64];
};
struct MaxCount {
    uint32_t m, n;
};
__device__ __noinline__ MaxCount exact_max128(Bf16x128 h, int live) {
    MaxCount r = {0u, 0u};
    for (int i = 0; i < 128; ++i) {
        const uint32_t a = (h.w[i / 2] >> (16 * (i & 1))) & 0x7FFFu;
        if (a < 0x7F80u)
            r.m = a > r.m ? a : r.m;
        else if (i < live)
            ++r.n;
    }
    return r;
}

// The codes of 32 bf16 values (two to a word) divided by d with IEEE division,
// a NaN keeping its sign (the hardware's NaN code is 0x7F whatever the sign):
// the rare path of the 1x128 conversions (a block holding NaN / Inf, or d
// below 2^-80), out of line so that the common path's code stays compact.
struct Bf16x32 {
    uint32_t w[16];
};
struct Codes32 {
    uint32_t c[8];
};
template <int QFMT>
__device__ __noinline__ Codes32 codes_ieee_div(Bf16x32 x, float d) {
    Codes32 r;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t w0 = x.w[2 * i], w1 = x.w[2 * i + 1];
        uint32_t c = cvt4<QFMT>(__fdiv_rn(__uint_as_float(w0 << 16), d), __fdiv_rn(__uint_as_float(w0 & 0xFFFF0000u), d),
                                __fdiv_rn(__uint_as_float(w1 << 16), d), __fdiv_rn(__uint_as_float(w1 & 0xFFFF0000u), d));
        uint32_t lo = c & 0xFFFFu, hi = c >> 16;
        if ((w0 & 0x7FFFu) > 0x7F80u) lo = (lo & ~0xFFu) | ((w0 >> 8) & 0x80u) | 0x7Fu;
        if ((w0 & 0x7FFF0000u) > 0x7F800000u) lo = (lo & ~0xFF00u) | ((w0 >> 16) & 0x8000u) | 0x7F00u;
        if ((w1 & 0x7FFFu) > 0x7F80u) hi = (hi & ~0xFFu) | ((w1 >> 8) & 0x80u) | 0x7Fu;
        if ((w1 & 0x7FFF0000u) > 0x7F800000u) hi = (hi & ~0xFF00u) | ((w1 >> 16) & 0x8000u) | 0x7F00u;
        r.c[i] = lo | (hi << 16);
    }
    return r;
}

// 1x128 (along N) quantization of this warp's 32 rows x 128 columns of D as
// stored in bf16 (h: RN(v scale) two to a word, as store_slice2 writes it): per row the amax of
// the 128 bf16 over the finite ones (NaN / Inf counted), d = RN(amax / fmax)
// (block_scale: 1 for amax 0), codes sat_rne(x / d) correctly rounded
// (Markstein's division from RN(1 / d), two lanes, negated; IEEE division for
// d below 2^-80 or a block holding NaN / Inf) with a NaN keeping its sign --
// the quantize kernel's 1x128 row path ("2025 FP8 quantized-training guide",
// sec. 2.2) on these values.  Saturation: d is one correctly rounded division
// and the next bf16 below the block maximum is at least 2^-8 smaller, so only
// elements equal to the maximum can exceed fmax; they are counted when the
// maximum does.  Codes leave through the staging boxes by TMA (uint8 32 x 32
// boxes, 32-byte swizzle); each row's d goes to the K-block-major scale array
// at (x0 / 128) Mp + row (rows past M, up to Mp, get the pad 1.0).
template <int QFMT, int NBOX>
__device__ __forceinline__ void store_q128(const CUtensorMap* mapQ, uint8_t* stg, uint32_t stg_s, int lane, int x0,
                                           int y0, const Params2& p, const uint32_t (&h)[64], uint32_t& nsat,
                                           uint32_t& nnf) {
    static_assert(NBOX >= 4, "a warp's 128 code columns fill four staging boxes");
    const int r = lane, sw = (r >> 2) & 1;
    const int64_t row = (int64_t)y0 + r;
    const bool row_live = row < p.M;
    const int live = !row_live ? 0 : ((int64_t)x0 + 128 <= p.N ? 128 : (int)(p.N - x0));  // columns inside D
    uint32_t cm[8];  // packed maxima of each 16-column chunk
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint32_t x = h[8 * c] & 0x7FFF7FFFu;
#pragma unroll
        for (int i = 1; i < 8; ++i) x = max_u16x2(x, h[8 * c + i] & 0x7FFF7FFFu);
        cm[c] = x;
    }
    const uint32_t pm = max_u16x2(max_u16x2(max_u16x2(cm[0], cm[1]), max_u16x2(cm[2], cm[3])),
                                  max_u16x2(max_u16x2(cm[4], cm[5]), max_u16x2(cm[6], cm[7])));
    uint32_t m = max(pm & 0xFFFFu, pm >> 16);
    const bool nf = m >= 0x7F80u;
    if (nf) {
        Bf16x128 hb;
#pragma unroll
        for (int i = 0; i < 64; ++i) hb.w[i] = h[i];
        const MaxCount e = exact_max128(hb, live);
        m = e.m;
        nnf += e.n;
    }
    if (!row_live) m = 0;
    const float d = block_scale<QFMT>(__uint_as_float(m << 16));
    const bool fast = !nf && d >= 0x1p-80f;
    const float rd = fast ? rcp_rn(d) : 1.0f;
    const float2 d2 = make_float2(d, d), nr2 = make_float2(-rd, -rd);
    // only elements equal to the block maximum can saturate
    const bool may_sat = row_live && fabsf(__fdiv_rn(__uint_as_float(m << 16), d)) > Fmt<QFMT>::fmax;
    if (may_sat) {  // look only inside the chunks whose maximum it is (all of them when NaN / Inf hide it)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (!nf && max(cm[c] & 0xFFFFu, cm[c] >> 16) != m) continue;
#pragma unroll
            for (int i = 8 * c; i < 8 * c + 8; ++i)
                nsat += (2 * i < live && (h[i] & 0x7FFFu) == m) + (2 * i + 1 < live && ((h[i] >> 16) & 0x7FFFu) == m);
        }
    }
    bulk_wait_read();  // the D boxes have left the staging area
    __syncwarp();
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        uint32_t c[8];
        if (fast) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t w0 = h[16 * b + 2 * i], w1 = h[16 * b + 2 * i + 1];
                const float2 a0 = make_float2(__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xFFFF0000u));
                const float2 a1 = make_float2(__uint_as_float(w1 << 16), __uint_as_float(w1 & 0xFFFF0000u));
                const float2 y0 = div2_neg(a0, d2, nr2), y1 = div2_neg(a1, d2, nr2);
                c[i] = cvt4<QFMT>(y0.x, y0.y, y1.x, y1.y) ^ 0x80808080u;
            }
        } else {
            Bf16x32 x;
#pragma unroll
            for (int i = 0; i < 16; ++i) x.w[i] = h[16 * b + i];
            const Codes32 k = codes_ieee_div<QFMT>(x, d);
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] = k.c[i];
        }
        uint8_t* box = stg + b * 1024;
        *(uint4*)(box + r * 32 + ((0 ^ sw) << 4)) = make_uint4(c[0], c[1], c[2], c[3]);
        *(uint4*)(box + r * 32 + ((1 ^ sw) << 4)) = make_uint4(c[4], c[5], c[6], c[7]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0 && (int64_t)x0 + 32 * b < p.N && (int64_t)y0 < p.M) {
            tma_store_2d(mapQ, x0 + 32 * b, y0, stg_s + b * 1024);
            bulk_commit();
        }
    }
    if (row < p.Mp && (int64_t)x0 < p.N) ((float*)p.qscale)[(int64_t)(x0 / 128) * p.Mp + row] = d;
}

// The column-wise copy of the fused output quantization (codes of D^T, blocks
// along M): shared by the MXFP8 and 1x128 column paths below.
//
// Four FP8 codes (byte k from element k) with a NaN element given its sign:
// the hardware's NaN code is 0x7F whatever the sign.  w0 holds bf16 elements
// 0, 1 and w1 elements 2, 3.
__device__ __forceinline__ uint32_t nan_signs4(uint32_t c, uint32_t w0, uint32_t w1) {
    uint32_t lo = c & 0xFFFFu, hi = c >> 16;
    if ((w0 & 0x7FFFu) > 0x7F80u) lo = (lo & ~0xFFu) | ((w0 >> 8) & 0x80u) | 0x7Fu;
    if ((w0 & 0x7FFF0000u) > 0x7F800000u) lo = (lo & ~0xFF00u) | ((w0 >> 16) & 0x8000u) | 0x7F00u;
    if ((w1 & 0x7FFFu) > 0x7F80u) hi = (hi & ~0xFFu) | ((w1 >> 8) & 0x80u) | 0x7Fu;
    if ((w1 & 0x7FFF0000u) > 0x7F800000u) hi = (hi & ~0xFF00u) | ((w1 >> 16) & 0x8000u) | 0x7F00u;
    return lo | (hi << 16);
}
// This lane's 128 values of D as stored in bf16 (RN(v scale)), two to a word:
// the column paths work on these, so the fp32 values are dead by then.
__device__ __forceinline__ void bf16_row(const float* v, float scale, uint32_t (&h)[64]) {
#pragma unroll
    for (int i = 0; i < 64; ++i) h[i] = pack_bf16(v[2 * i] * scale, v[2 * i + 1] * scale);
}
// Chunk b (columns 32 b .. 32 b + 31) of this lane's row, picked by selects so
// that a chunk loop can stay rolled and the row stay in registers.
__device__ __forceinline__ void pick_chunk(const uint32_t (&hr)[64], int b, uint32_t (&h)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t lo = (b & 1) ? hr[16 + i] : hr[i];
        const uint32_t hi = (b & 1) ? hr[48 + i] : hr[32 + i];
        h[i] = (b & 2) ? hi : lo;
    }
}
// A 32 x 32 chunk of the warp's rows (h: this lane's row, two columns to a
// word) transposed through the warp's area T (16-byte aligned, 16 x 36
// words; word w of row r at w * 36 + r): the writes of one w by the 32 lanes
// are consecutive words, and lane c reads the 32 words of its column pair as
// eight 16-byte loads at (c / 2) * 36, which the 36-word stride spreads over
// distinct banks.  Afterwards lane c holds column c of the chunk, rows 2 i
// and 2 i + 1 in the low and high halves of hv[i].
__device__ __forceinline__ void transpose32(uint32_t* T, int lane, const uint32_t (&h)[16], uint32_t (&hv)[16]) {
    __syncwarp();  // the previous chunk's reads of T are done
#pragma unroll
    for (int w = 0; w < 16; ++w) T[w * 36 + lane] = h[w];
    __syncwarp();
    const uint4* src = (const uint4*)(T + (lane >> 1) * 36);
    const uint32_t sel = (lane & 1) ? 0x7632u : 0x5410u;  // the high or the low halves
#pragma unroll
    for (int t = 0; t < 8; ++t) {  // rows 4 t .. 4 t + 3
        const uint4 v = src[t];
        hv[2 * t] = __byte_perm(v.x, v.y, sel);
        hv[2 * t + 1] = __byte_perm(v.z, v.w, sel);
    }
}
// The largest finite magnitude among a column's 32 values (two to a word) and
// whether a NaN / Inf is among them: packed maxima, the exact pass only when
// they flag a NaN / Inf.
__device__ __forceinline__ uint32_t col_max32(const uint32_t (&hv)[16], bool* nf) {
    uint32_t pm = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) pm = max_u16x2(pm, hv[i] & 0x7FFF7FFFu);
    uint32_t m = max(pm & 0xFFFFu, pm >> 16);
    *nf = m >= 0x7F80u;
    if (*nf) {
        m = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t a = (hv[i / 2] >> (16 * (i & 1))) & 0x7FFFu;
            if (a < 0x7F80u) m = a > m ? a : m;
        }
    }
    return m;
}
// A column's 32 codes (rows 4 i .. 4 i + 3 in c[i]) as row `lane` of a 32 x 32
// box of the transposed copy (32 bytes, no swizzle).
__device__ __forceinline__ void put_col_codes(uint8_t* box, int lane, const uint32_t (&c)[8]) {
    *(uint4*)(box + lane * 32) = make_uint4(c[0], c[1], c[2], c[3]);
    *(uint4*)(box + lane * 32 + 16) = make_uint4(c[4], c[5], c[6], c[7]);
}

// MXFP8 column-wise copy (1x32 blocks along M) of this warp's 32 rows x 128
// columns of D as stored in bf16: the block of column n is the warp's rows
// y0 .. y0 + 31 (y0 a multiple of 32; rows past M are zeros of the GEMM), so
// after a transpose through shared memory each lane holds one column's block
// and finds its amax, e, the codes sat_rne(x 2^-e), the NaN signs and the
// saturation count (finite |y| > fmax) alone, as the row path does for a
// row's block; the codes leave transposed ([N][M], uint8 32 x 32 boxes by
// TMA) and each column's E8M0 byte goes to the packed 128x4 tiles of the
// [N][ceil(M/32)] scale matrix -- the quantize kernel's MXFP8 column copy of
// these values.
template <int QFMT>
__device__ __forceinline__ void store_qc_mx(const CUtensorMap* mapQc, uint8_t* stg, uint32_t stg_s, uint32_t* T,
                                            int lane, int x0, int y0, const Params2& p, const uint32_t (&hr)[64],
                                            uint32_t& nsat) {
    bulk_wait_read();  // the row codes' boxes have left the staging area
    __syncwarp();
#pragma unroll 1
    for (int b = 0; b < 4; ++b) {
        uint32_t h[16], hv[16];
        pick_chunk(hr, b, h);
        transpose32(T, lane, h, hv);
        bool nf;
        const uint32_t m = col_max32(hv, &nf);
        const int64_t n = (int64_t)x0 + 32 * b + lane;  // this lane's column
        const int e = mx_exponent<QFMT>(m << 16);
        const float k = exp2_neg(e);
        if (n < p.Np && (int64_t)y0 < p.Mp) {  // pads (columns past N, blocks past M) get 127
            const int64_t tile = (n / 128) * p.tiles_m128 + y0 / 128;
            ((uint8_t*)p.qscale_col)[tile * 512 + (n % 32) * 16 + ((n % 128) / 32) * 4 + (y0 / 32) % 4] =
                (uint8_t)(e + 127);
        }
        const bool sat = __uint_as_float(m << 16) * k > Fmt<QFMT>::fmax;
        const float2 k2 = make_float2(k, k);
        uint32_t c[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w0 = hv[2 * i], w1 = hv[2 * i + 1];
            const float2 ya =
                __fmul2_rn(make_float2(__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xFFFF0000u)), k2);
            const float2 yb =
                __fmul2_rn(make_float2(__uint_as_float(w1 << 16), __uint_as_float(w1 & 0xFFFF0000u)), k2);
            c[i] = cvt4<QFMT>(ya.x, ya.y, yb.x, yb.y);
            if (sat) {  // a saturating block: count its finite elements past fmax
                const float y[4] = {ya.x, ya.y, yb.x, yb.y};
#pragma unroll
                for (int t = 0; t < 4; ++t) nsat += fabsf(y[t]) <= 3.402823466e38f && fabsf(y[t]) > Fmt<QFMT>::fmax;
            }
            if (nf) c[i] = nan_signs4(c[i], w0, w1);
        }
        uint8_t* box = stg + b * 1024;
        put_col_codes(box, lane, c);
        fence_async_smem();
        __syncwarp();
        if (lane == 0 && (int64_t)x0 + 32 * b < p.N && (int64_t)y0 < p.M) {
            tma_store_2d(mapQc, y0, x0 + 32 * b, stg_s + b * 1024);
            bulk_commit();
        }
    }
}

// 1x128 column-wise copy (blocks of 128 rows of one column) of this warp's
// 32 rows x 128 columns of D as stored in bf16, after the row path.  A CTA's
// 128 tile rows are one 128-row group, so the block of column n is the rows
// of the four warps of this column half.  Each warp transposes its chunks
// through shared memory (a lane then holds one column's 32 rows, kept in
// registers), takes each column's 32-row maximum in the lane and posts it to
// xb ([4 warps][128 columns]) with one arrival per chunk on that chunk's
// mbarrier (xbar0 + 8 chunk); then, chunk by chunk, it waits for the four
// warps' maxima (bounded, like every other wait; the first chunk's are in
// while the later ones are still being posted) and turns its column's
// maxima into d = RN(amax / fmax) and the codes sat_rne(x / d) (Markstein's
// division from RN(1 / d), or IEEE division for d below 2^-80 or a block
// holding NaN / Inf, with the NaN signs), saturation counted at the
// elements equal to a saturating block's maximum (the row path's argument);
// codes transposed by TMA, d into the [ceil(M/128)][Np] scale array by the
// first warp -- the quantize kernel's 1x128 column copy of these values.
// Returns false when an exchange wait gave up (the caller leaves its tile
// loop).
template <int QFMT>
__device__ __forceinline__ bool store_qc128(const CUtensorMap* mapQc, uint8_t* stg, uint32_t stg_s, uint32_t* T,
                                            int lane, int q, int x0, int y0, const Params2& p,
                                            const uint32_t (&hr)[64], uint32_t& nsat, uint32_t* xb, uint32_t xbar0,
                                            uint32_t xph, volatile int* abort_flag) {
    uint32_t ht[64];  // this lane's column of each chunk, two rows to a word
    auto post = [&](auto bc) {
        constexpr int b = decltype(bc)::value;
        uint32_t h[16], hv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) h[i] = hr[16 * b + i];
        transpose32(T, lane, h, hv);
#pragma unroll
        for (int i = 0; i < 16; ++i) ht[16 * b + i] = hv[i];
        bool nf;
        const uint32_t m = col_max32(hv, &nf);
        xb[q * 128 + 32 * b + lane] = m | (nf ? 0x10000u : 0u);
        __syncwarp();
        if (lane == 0) mbar_arrive(xbar0 + 8u * b);
    };
    post(std::integral_constant<int, 0>{});
    post(std::integral_constant<int, 1>{});
    post(std::integral_constant<int, 2>{});
    post(std::integral_constant<int, 3>{});
    bulk_wait_read();  // the row codes' boxes have left the staging area
    __syncwarp();
    bool ok = true;
    auto codes = [&](auto bc) {
        constexpr int b = decltype(bc)::value;
        if (!ok) return;
        if (!mbar_wait2(xbar0 + 8u * b, xph, abort_flag, p.wait_ns)) {
            ok = false;
            return;
        }
        const uint32_t* hv = ht + 16 * b;
        uint32_t m = 0, f = 0;  // this lane's column: the block maximum over the four warps
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint32_t x = xb[w * 128 + 32 * b + lane];
            m = max(m, x & 0xFFFFu);
            f |= x >> 16;
        }
        const float d = block_scale<QFMT>(__uint_as_float(m << 16));
        const bool fast = f == 0u && d >= 0x1p-80f;
        const int64_t n = (int64_t)x0 + 32 * b + lane;
        if (q == 0 && n < p.Np && (int64_t)y0 < p.Mp)  // y0: the 128-row group's first row (pads: d = 1)
            ((float*)p.qscale_col)[(int64_t)(y0 / 128) * p.Np + n] = d;
        const bool may_sat = fabsf(__fdiv_rn(__uint_as_float(m << 16), d)) > Fmt<QFMT>::fmax;
        uint32_t c[8];
        if (fast) {
            const float nrd = -rcp_rn(d);
            const float2 d2 = make_float2(d, d), nr2 = make_float2(nrd, nrd);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t w0 = hv[2 * i], w1 = hv[2 * i + 1];
                const float2 a0 = make_float2(__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xFFFF0000u));
                const float2 a1 = make_float2(__uint_as_float(w1 << 16), __uint_as_float(w1 & 0xFFFF0000u));
                const float2 ya = div2_neg(a0, d2, nr2), yb = div2_neg(a1, d2, nr2);
                c[i] = cvt4<QFMT>(ya.x, ya.y, yb.x, yb.y) ^ 0x80808080u;
            }
        } else {
            Bf16x32 x;
#pragma unroll
            for (int i = 0; i < 16; ++i) x.w[i] = hv[i];
            const Codes32 kc = codes_ieee_div<QFMT>(x, d);
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] = kc.c[i];
        }
        if (may_sat) {  // only elements equal to a saturating block's maximum exceed fmax
#pragma unroll
            for (int i = 0; i < 16; ++i) nsat += ((hv[i] & 0x7FFFu) == m) + (((hv[i] >> 16) & 0x7FFFu) == m);
        }
        uint8_t* box = stg + b * 1024;
        put_col_codes(box, lane, c);
        fence_async_smem();
        __syncwarp();
        if (lane == 0 && (int64_t)x0 + 32 * b < p.N && (int64_t)y0 < p.M) {
            tma_store_2d(mapQc, y0, x0 + 32 * b, stg_s + b * 1024);
            bulk_commit();
        }
    };
    codes(std::integral_constant<int, 0>{});
    codes(std::integral_constant<int, 1>{});
    codes(std::integral_constant<int, 2>{});
    codes(std::integral_constant<int, 3>{});
    return ok;
}

// QF, the fused quantization of the bf16 output: 0 none; 1, 2 MXFP8 1x32
// (E4M3, E5M2) and 3, 4 1x128, row-wise along N; 5, 6 and 7, 8 the same with
// the column-wise copy (blocks along M) as well.
template <int QF>
struct QOut {
    static constexpr bool mx = QF == 1 || QF == 2 || QF == 5 || QF == 6;
    static constexpr bool b128 = QF == 3 || QF == 4 || QF == 7 || QF == 8;
    static constexpr bool col = QF >= 5;
    static constexpr int fmt = (QF + 1) % 2;  // QF 1, 3, 5, 7: E4M3
};

// KB (blockwise recipes): the K block of the scales, i.e. of the partial sums
// the epilogue promotes -- 128 for the 1x128 / 128x128 recipes, 32, 64 or 256
// for the generic sub-channel blocks ("mastering FP8 LLM training 1.5x
// speedup", scaling strategy 3).  A 128-wide pipeline stage then holds
// 128 / KB partials (KB <= 128) or half of one (KB = 256).
template <int REC, bool OUT_F32, int QF, int KB = 128>
__global__ void __launch_bounds__(Cfg<REC>::THREADS, 1)
    gemm2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmSFA,
                 const __grid_constant__ CUtensorMap tmSFB, const __grid_constant__ CUtensorMap tmQ,
                 const __grid_constant__ CUtensorMap tmQc, const Params2 p) {
    using C = Cfg<REC>;
    constexpr int BN = C::BN, BH = C::BH, STAGES = C::STAGES, NACC = C::NACC, EC = C::EPI_COLS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(smem);
    auto full = [&](int s) { return sb + C::OFF_BAR + 8u * s; };
    auto empty = [&](int s) { return sb + C::OFF_BAR + 8u * (STAGES + s); };
    auto tfull = [&](int b) { return sb + C::OFF_BAR + 8u * (2 * STAGES + b); };
    auto tempty = [&](int b) { return sb + C::OFF_BAR + 8u * (2 * STAGES + NACC + b); };
    const uint32_t mma_done = sb + C::OFF_BAR + 8u * (2 * STAGES + 2 * NACC);
    auto sfull = [&](int r) { return sb + C::OFF_BAR + 8u * (2 * STAGES + 2 * NACC + 1 + r); };
    auto sempty = [&](int r) { return sb + C::OFF_BAR + 8u * (2 * STAGES + 2 * NACC + 1 + C::SR + r); };
    // MXFP8: stage s's scale tiles are in both CTAs' TMEM (the leader's
    // barrier; the copier's commit arrives once the copies are complete)
    auto sfr = [&](int st) { return sb + C::OFF_BAR + 8u * (2 * STAGES + 2 * NACC + 1 + 2 * C::SR + st); };
    uint32_t* tmem_slot = (uint32_t*)(smem + C::OFF_MISC);
    volatile int* abort_flag = (volatile int*)(smem + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t cr = cluster_rank();
    const bool leader = cr == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < NACC; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), 2 * C::EPI_WARPS);
        }
        mbar_init(mma_done, 1);
        for (int r = 0; r < C::SR; ++r) {
            mbar_init(sfull(r), REC == REC_B2D ? 2 : 1);
            mbar_init(sempty(r), C::EPI_WARPS);
        }
        for (int st = 0; st < C::NSFB; ++st) mbar_init(sfr(st), 1);
        if constexpr (QOut<QF>::col && QOut<QF>::b128)
            for (int i = 0; i < 16; ++i) mbar_init(sb + C::OFF_XBAR + 8u * i, 4);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_map(&tmA);
        prefetch_map(&tmB);
    }
    if (warp == 1) {  // collective with the peer CTA's warp 1
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    __syncwarp();
    cluster_sync();  // both CTAs' barriers exist before any remote arrive / complete_tx
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int64_t npt = p.tiles_m2 * p.tiles_n;
    const int64_t cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0 && !p.stall) {  // a stalled launch (diagnostic) loads nothing
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int64_t t = cid; t < npt && ok; t += ncl) {
                int64_t mp, nb;
                tile_coords(t, p.tiles_m2, p.tiles_n, mp, nb);
                const bool b2 = (2 * nb + 1) < p.nbn128;  // MX: second 128-row scale tile of B exists
                for (int64_t kb = 0; kb < p.nkb; ++kb) {
                    if (!mbar_wait2(empty(s), ph ^ 1u, abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fl = mapa(full(s), 0);
                    // MXFP8: each CTA's scale tiles (its A rows' tile, B's one or two)
                    // land on the leader's stage barrier with the operands
                    if (leader)
                        mbar_expect_tx(full(s), 2 * (C::A_STAGE + C::B_STAGE) +
                                                    (REC == REC_MX ? 2 * (512 + (b2 ? 1024u : 512u)) : 0u));
                    tma_load_2d_pair(sb + C::OFF_A + s * C::A_STAGE, &tmA, (int)(kb * BK), (int)(mp * 256 + BM * cr), fl);
                    tma_load_2d_pair(sb + C::OFF_B + s * C::B_STAGE, &tmB, (int)(kb * BK), (int)(nb * BN + BH * cr), fl);
                    if (REC == REC_MX) {
                        tma_load_2d_pair(sb + C::OFF_SFA + s * 512, &tmSFA, 0, (int)((2 * mp + cr) * p.nkb + kb), fl);
                        tma_load_2d_pair(sb + C::OFF_SFB + s * 1024, &tmSFB, 0, (int)((2 * nb) * p.nkb + kb), fl);
                        if (b2)
                            tma_load_2d_pair(sb + C::OFF_SFB + s * 1024 + 512, &tmSFB, 0,
                                             (int)((2 * nb + 1) * p.nkb + kb), fl);
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader only)
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t tile_i = 0, kbg = 0;
            bool ok = true;
            for (int64_t t = cid; t < npt && ok; t += ncl, ++tile_i) {
                const uint32_t abuf = tile_i % NACC;
                if (REC == REC_PT || REC == REC_PC || REC == REC_MX) {
                    if (!mbar_wait2(tempty(abuf), ((tile_i / NACC) & 1u) ^ 1u, abort_flag, p.wait_ns)) break;
                    tc_fence_after();
                }
                for (int64_t kb = 0; kb < p.nkb; ++kb) {
                    uint32_t dcol = (REC == REC_PT || REC == REC_PC) ? abuf * BN : 0;
                    if ((REC == REC_B2D || REC == REC_B1D) && KB == 128) {
                        const uint32_t buf = kbg % NACC;
                        if (!mbar_wait2(tempty(buf), ((kbg / NACC) & 1u) ^ 1u, abort_flag, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        dcol = buf * BN;
                    }
                    if (!mbar_wait2(full(s), ph, abort_flag, p.wait_ns) || (REC == REC_MX && !mbar_wait2(sfr(s), ph, abort_flag, p.wait_ns))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sb + C::OFF_A + s * C::A_STAGE, b0 = sb + C::OFF_B + s * C::B_STAGE;
                    if (REC == REC_MX) {
                        const uint32_t sft = tmem + SF_TMEM_COL + 12u * s;
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k) {
                            const uint32_t idesc = p.idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29);
                            mma2_mx(tmem, desc_sw128(a0 + 32 * k), desc_sw128(b0 + 32 * k), idesc, sft, sft + 4,
                                    (kb > 0 || k > 0) ? 1u : 0u);
                        }
                    } else if ((REC == REC_B2D || REC == REC_B1D) && KB != 128) {
                        // K blocks of KB: each partial takes a free TMEM buffer before its
                        // first MMA and is handed to the epilogue after its last
                        constexpr int MPB = KB / 32;  // MMAs of K = 32 per partial
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k) {
                            const int64_t kq = KB > 128 ? kb / 2 : (kb * BK + 32 * k) / KB;  // this MMA's partial
                            if (kq >= p.nkbq) break;
                            const bool first = KB > 128 ? ((kb & 1) == 0 && k == 0) : (k % MPB == 0);
                            const bool last = KB > 128 ? (((kb & 1) == 1 || kb + 1 == p.nkb) && k == BK / 32 - 1)
                                                       : (k % MPB == MPB - 1);
                            if (first) {
                                if (!mbar_wait2(tempty(kbg % NACC), ((kbg / NACC) & 1u) ^ 1u, abort_flag, p.wait_ns)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                            }
                            mma2_f8(tmem + (kbg % NACC) * BN, desc_sw128(a0 + 32 * k), desc_sw128(b0 + 32 * k), p.idesc,
                                    first ? 0u : 1u);
                            if (last) {
                                tc2_commit_both(tfull(kbg % NACC));
                                ++kbg;
                            }
                        }
                        if (!ok) break;
                    } else {
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k) {
                            const uint32_t acc =
                                (REC == REC_PT || REC == REC_PC) ? ((kb > 0 || k > 0) ? 1u : 0u) : (k > 0 ? 1u : 0u);
                            mma2_f8(tmem + dcol, desc_sw128(a0 + 32 * k), desc_sw128(b0 + 32 * k), p.idesc, acc);
                        }
                    }
                    tc2_commit_both(empty(s));
                    if ((REC == REC_B2D || REC == REC_B1D) && KB == 128) {
                        tc2_commit_both(tfull(kbg % NACC));
                        ++kbg;
                    }
                    const bool last = kb + 1 == p.nkb;
                    if ((REC == REC_PT || REC == REC_PC || REC == REC_MX) && last) tc2_commit_both(tfull(abuf));
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
            }
            tc2_commit_local(mma_done);
            mbar_drain(mma_done, 0, p.wait_ns);
        }
    } else if ((REC == REC_MX || C::BLOCKWISE) && warp == C::SCALE_WARP) {
        if constexpr (REC == REC_MX) {
            // ------------------------------------------------ scale-tile copier (MXFP8, leader only)
            // stage s's scale tiles from both CTAs' shared memory into their TMEM
            // (tcgen05.cp.cta_group::2, the replicated 32-row layout the
            // block-scaled MMA reads), then a commit that the MMA issuer waits on;
            // a stage's TMEM slot is rewritten only after its operands landed
            // again, i.e. after the MMAs that read it
            if (leader && lane == 0) {
                int s = 0;
                uint32_t ph = 0;
                bool ok = true, any = false;
                int last_s = 0;
                uint32_t last_ph = 0;
                for (int64_t t = cid; t < npt && ok; t += ncl) {
                    for (int64_t kb = 0; kb < p.nkb; ++kb) {
                        if (!mbar_wait2(full(s), ph, abort_flag, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sft = tmem + SF_TMEM_COL + 12u * s;
                        tc2_cp_32x128b(sft, smem_desc(sb + C::OFF_SFA + s * 512, 0, 128, 0));
                        tc2_cp_32x128b(sft + 4, smem_desc(sb + C::OFF_SFB + s * 1024, 0, 128, 0));
                        tc2_cp_32x128b(sft + 8, smem_desc(sb + C::OFF_SFB + s * 1024 + 512, 0, 128, 0));
                        tc2_commit_local(sfr(s));
                        any = true;
                        last_s = s;
                        last_ph = ph;
                        if (++s == STAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                }
                // the copies are complete before this CTA can free TMEM (bounded)
                if (any) mbar_drain(sfr(last_s), last_ph, p.wait_ns);
            }
        } else if constexpr (C::BLOCKWISE) {
            // ------------------------------------------------ scale producer (blockwise, both CTAs)
            // the scales of every K block (partial) of each tile in turn: this
            // CTA's A-row scales, and the tile's B scales, into the next ring slot
            if (lane == 0 && !p.stall) {  // a stalled launch (diagnostic) loads nothing
                uint32_t kbp = 0;
                bool ok = true;
                for (int64_t t = cid; t < npt && ok; t += ncl) {
                    int64_t mp, nb;
                    tile_coords(t, p.tiles_m2, p.tiles_n, mp, nb);
                    const int64_t rs = mp * 256 + BM * cr;  // this CTA's first row
                    const bool arow = rs < p.Mp;           // else all its rows are past M: no A scales
                    // 1 x KB B scales of the tile's columns that exist (Np is a multiple of 128)
                    const uint32_t bbytes = (p.Np - nb * BN >= BN) ? 4u * BN : 4u * (uint32_t)(p.Np - nb * BN);
                    for (int64_t kq = 0; kq < p.nkbq; ++kq, ++kbp) {
                        const uint32_t r = kbp % C::SR;
                        if (!mbar_wait2(sempty(r), ((kbp / C::SR) & 1u) ^ 1u, abort_flag, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dst = sb + C::OFF_SCL + r * C::SLOT;
                        mbar_expect_tx(sfull(r), (arow ? 512u : 0u) + (REC == REC_B1D ? bbytes : 0u));
                        if (arow) bulk_load(dst, p.bsa + kq * p.Mp + rs, 512, sfull(r));
                        if (REC == REC_B1D) bulk_load(dst + 512, p.bsb + kq * p.Np + nb * BN, bbytes, sfull(r));
                        if (REC == REC_B2D) {  // the scales of the tile's KB-row B blocks (BN / KB, at least one)
                            const int64_t b0 = (nb * BN) / KB;
    #pragma unroll
                            for (int u = 0; u < (BN >= KB ? BN / KB : 1); ++u)
                                if (b0 + u < p.nbnq) cp_async_4(dst + 512 + 4 * u, p.bsb + (b0 + u) * p.nkbq + kq);
                            cp_async_arrive(sfull(r));
                        }
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------ epilogue (both CTAs, own 128 rows)
        const int ew = warp - 2, q = warp & 3, j = ew >> 2;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint32_t tcol = (uint32_t)(EC * j);
        float sab = 1.0f;
        if (REC == REC_PT) sab = __fmul_rn(*p.sa_inv, *p.sb_inv);
        uint8_t* stg = smem + C::OFF_STG + ew * C::STG_WARP;
        const uint32_t stg_s = sb + C::OFF_STG + ew * C::STG_WARP;
        auto release = [&](int b) {  // this warp is done with TMEM buffer b: tell the leader's MMA issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(mapa(tempty(b), 0));
        };
        uint32_t q_sat = 0, q_nf = 0, q_satc = 0;  // fused output quantization's counters
        uint32_t tile_i = 0, kbg = 0;
        for (int64_t t = cid; t < npt; t += ncl, ++tile_i) {
            int64_t mp, nb;
            tile_coords(t, p.tiles_m2, p.tiles_n, mp, nb);
            const int64_t row0 = mp * 256 + BM * cr + 32 * q;  // this warp's first row
            const int64_t col0 = nb * BN + EC * j;
            if constexpr (!C::BLOCKWISE) {
                const uint32_t abuf = tile_i % NACC;
                if (!mbar_wait2(tfull(abuf), (tile_i / NACC) & 1u, abort_flag, p.wait_ns)) break;
                tc_fence_after();
                uint32_t r[EC];
#pragma unroll
                for (int c = 0; c < EC / 32; ++c) FP8Q_LD32(tmem + lane_base + abuf * BN + tcol + 32 * c, (r + 32 * c));
                tc_wait_ld();
#pragma unroll
                for (int c = 0; c < EC / 32; ++c) reg_fence32(r + 32 * c);
                release(abuf);
                float vf[EC];
#pragma unroll
                for (int i = 0; i < EC; ++i) vf[i] = __uint_as_float(r[i]);
                if constexpr (REC == REC_PC) {
                    // per channel: D = fp32(s_inv_A[m] s_inv_B[n]) x acc; the factor
                    // vectors are padded to 128 entries, and a warp's 128 columns lie
                    // wholly inside or past them
                    const int64_t m = row0 + lane;
                    const float ia = m < p.Mp ? p.bsa[m] : 0.0f;
                    if (col0 < p.Np) {
                        const float4* ib = (const float4*)(p.bsb + col0);
#pragma unroll
                        for (int i = 0; i < EC / 4; ++i) {
                            const float4 b = ib[i];
                            vf[4 * i] = __fmul_rn(vf[4 * i], __fmul_rn(ia, b.x));
                            vf[4 * i + 1] = __fmul_rn(vf[4 * i + 1], __fmul_rn(ia, b.y));
                            vf[4 * i + 2] = __fmul_rn(vf[4 * i + 2], __fmul_rn(ia, b.z));
                            vf[4 * i + 3] = __fmul_rn(vf[4 * i + 3], __fmul_rn(ia, b.w));
                        }
                    }
                }
                const float osc = (REC == REC_PC) ? 1.0f : sab;
                if (QF == 0 || p.hasD)
                    store_slice2<OUT_F32, EC, C::STG_WARP / 1024>(&tmD, stg, stg_s, lane, (int)col0, (int)row0, (int)p.N,
                                                                  (int)p.M, vf, osc);
                if constexpr (QOut<QF>::mx)
                    store_q<QOut<QF>::fmt, EC, C::STG_WARP / 1024>(&tmQ, stg, stg_s, lane, (int)col0, (int)row0, p, vf,
                                                                   osc, q_sat, q_nf);
                if constexpr (QOut<QF>::b128 || QOut<QF>::col) {
                    uint32_t hc[64];  // D as stored in bf16, two to a word: the 1x128 row path and the column paths
                    bf16_row(vf, osc, hc);
                    if constexpr (QOut<QF>::col) {
                        if (row0 + lane >= p.M) {  // rows past M take no part in a column block
#pragma unroll
                            for (int i = 0; i < 64; ++i) hc[i] = 0u;
                        }
                    }
                    // the column copy's transpose area of this warp and its 1x128 exchange
                    // slot [tile parity][column half] (buffer, and the chunks' mbarriers)
                    uint32_t* const tr = (uint32_t*)(smem + C::OFF_TR + ew * C::TR_WARP);
                    const uint32_t xs = (tile_i & 1u) * 2 + (uint32_t)j;
                    if constexpr (QOut<QF>::b128)
                        store_q128<QOut<QF>::fmt, C::STG_WARP / 1024>(&tmQ, stg, stg_s, lane, (int)col0, (int)row0, p,
                                                                      hc, q_sat, q_nf);
                    if constexpr (QOut<QF>::col && QOut<QF>::mx)
                        store_qc_mx<QOut<QF>::fmt>(&tmQc, stg, stg_s, tr, lane, (int)col0, (int)row0, p, hc, q_satc);
                    if constexpr (QOut<QF>::col && QOut<QF>::b128) {
                        if (!store_qc128<QOut<QF>::fmt>(&tmQc, stg, stg_s, tr, lane, q, (int)col0, (int)row0, p, hc,
                                                        q_satc, (uint32_t*)(smem + C::OFF_XB) + xs * 512,
                                                        sb + C::OFF_XBAR + 8u * (4 * xs), (tile_i >> 1) & 1u,
                                                        abort_flag))
                            break;
                    }
                }
            } else {
                float2 acc[EC / 2];  // packed pairs: Blackwell's two-lane FMA halves the promotion's instructions
#pragma unroll
                for (int i = 0; i < EC / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);
                bool ok = true;
                for (int64_t kb = 0; kb < p.nkbq; ++kb, ++kbg) {
                    const uint32_t r = kbg % C::SR;
                    if (!mbar_wait2(sfull(r), (kbg / C::SR) & 1u, abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const float* scl = (const float*)(smem + C::OFF_SCL + r * C::SLOT);
                    const float sa = scl[32 * q + lane];
                    // KB >= 128: this warp's EC columns lie in one KB-row B block (tiles
                    // start on 256-column boundaries); smaller KB: one per chunk, below
                    const float sc = (REC == REC_B2D && KB >= 128) ? __fmul_rn(sa, scl[128 + (EC * j) / KB]) : 0.0f;
                    const uint32_t buf = kbg % NACC;
                    if (!mbar_wait2(tfull(buf), (kbg / NACC) & 1u, abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // four 16-column chunks: partial -> registers -> promoted into acc
#pragma unroll
                    for (int c = 0; c < EC / 16; ++c) {
                        uint64_t v[8];
                        FP8Q_LD16_PAIRS(tmem + lane_base + buf * BN + tcol + 16 * c, v);
                        if (c == EC / 16 - 1) release(buf);
                        if (REC == REC_B2D) {
                            const float scc = KB >= 128 ? sc : __fmul_rn(sa, scl[128 + (EC * j + 16 * c) / KB]);
                            const float2 sc2 = make_float2(scc, scc);
#pragma unroll
                            for (int i = 0; i < 8; ++i) acc[8 * c + i] = __ffma2_rn(u64_as_float2(v[i]), sc2, acc[8 * c + i]);
                        } else {
                            const float2 sa2 = make_float2(sa, sa);
                            const float* sv = scl + 128 + EC * j + 16 * c;  // B scales of these columns
#pragma unroll
                            for (int i = 0; i < 8; i += 2) {
                                const float4 s4 = *(const float4*)(sv + 2 * i);
                                const float2 p0 = __fmul2_rn(sa2, make_float2(s4.x, s4.y));
                                const float2 p1 = __fmul2_rn(sa2, make_float2(s4.z, s4.w));
                                acc[8 * c + i] = __ffma2_rn(u64_as_float2(v[i]), p0, acc[8 * c + i]);
                                acc[8 * c + i + 1] = __ffma2_rn(u64_as_float2(v[i + 1]), p1, acc[8 * c + i + 1]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sempty(r));
                }
                if (!ok) break;
                if (QF == 0 || p.hasD)
                    store_slice2<OUT_F32, EC, C::STG_WARP / 1024>(&tmD, stg, stg_s, lane, (int)col0, (int)row0, (int)p.N,
                                                                  (int)p.M, reinterpret_cast<const float*>(acc), 1.0f);
                const float* accf = reinterpret_cast<const float*>(acc);
                if constexpr (QOut<QF>::mx)
                    store_q<QOut<QF>::fmt, EC, C::STG_WARP / 1024>(&tmQ, stg, stg_s, lane, (int)col0, (int)row0, p, accf,
                                                                   1.0f, q_sat, q_nf);
                if constexpr (QOut<QF>::b128 || QOut<QF>::col) {
                    uint32_t hc[64];  // D as stored in bf16, two to a word: the 1x128 row path and the column paths
                    bf16_row(accf, 1.0f, hc);
                    if constexpr (QOut<QF>::col) {
                        if (row0 + lane >= p.M) {  // rows past M take no part in a column block
#pragma unroll
                            for (int i = 0; i < 64; ++i) hc[i] = 0u;
                        }
                    }
                    // the column copy's transpose area of this warp and its 1x128 exchange
                    // slot [tile parity][column half] (buffer, and the chunks' mbarriers)
                    uint32_t* const tr = (uint32_t*)(smem + C::OFF_TR + ew * C::TR_WARP);
                    const uint32_t xs = (tile_i & 1u) * 2 + (uint32_t)j;
                    if constexpr (QOut<QF>::b128)
                        store_q128<QOut<QF>::fmt, C::STG_WARP / 1024>(&tmQ, stg, stg_s, lane, (int)col0, (int)row0, p,
                                                                      hc, q_sat, q_nf);
                    if constexpr (QOut<QF>::col && QOut<QF>::mx)
                        store_qc_mx<QOut<QF>::fmt>(&tmQc, stg, stg_s, tr, lane, (int)col0, (int)row0, p, hc, q_satc);
                    if constexpr (QOut<QF>::col && QOut<QF>::b128) {
                        if (!store_qc128<QOut<QF>::fmt>(&tmQc, stg, stg_s, tr, lane, q, (int)col0, (int)row0, p, hc,
                                                        q_satc, (uint32_t*)(smem + C::OFF_XB) + xs * 512,
                                                        sb + C::OFF_XBAR + 8u * (4 * xs), (tile_i >> 1) & 1u,
                                                        abort_flag))
                            break;
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        if constexpr (QF != 0) {
            q_sat = warp_sum_u32(q_sat);
            q_nf = warp_sum_u32(q_nf);
            q_satc = warp_sum_u32(q_satc);
            if (lane == 0) {
                if (q_sat) atomicAdd(&p.qcounters[0], (unsigned long long)q_sat);
                if (q_satc) atomicAdd(&p.qcounters[1], (unsigned long long)q_satc);
                if (q_nf) atomicAdd(&p.qcounters[2], (unsigned long long)q_nf);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    __syncwarp();
    cluster_sync();  // the pair's MMAs, copies and remote arrivals are over
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

template <int REC, bool F32, int QF, int KB = 128>
fp8q_status launch2_t(const CUtensorMap* maps, const Params2& p, cudaStream_t s) {
    using C = Cfg<REC>;
    auto kern = gemm2_kernel<REC, F32, QF, KB>;
    constexpr uint32_t smem = QOut<QF>::col ? C::SMEM_COL : C::SMEM;
    static PerDevice<bool> attr;
    if (!smem_opt_in(attr, kern, smem)) return FP8Q_ERR_CUDA;
    const int sms = sm_count();
    if (sms < 2) return FP8Q_ERR_CUDA;
    const int64_t npt = p.tiles_m2 * p.tiles_n;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeClusterDimension;
    la[0].val.clusterDim.x = 2;
    la[0].val.clusterDim.y = 1;
    la[0].val.clusterDim.z = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    // as many persistent pairs as can be resident at once (SM pairs must sit
    // in one GPC, so this can be below half the SM count), once per device
    static PerDevice<int> resident;
    int max_clusters = 0;
    resident.get(current_device(), max_clusters, [&](int& v) {
        cfg.gridDim = dim3((unsigned)sms, 1, 1);
        if (cudaOccupancyMaxActiveClusters(&v, kern, &cfg) != cudaSuccess || v < 1) v = sms / 2;
        return true;
    });
    if (max_clusters < 1) max_clusters = sms / 2;
    const int64_t ncl = npt < max_clusters ? npt : max_clusters;
    cfg.gridDim = dim3((unsigned)(2 * ncl), 1, 1);
    if (cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], p) !=
        cudaSuccess)
        return FP8Q_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

template <int REC>
fp8q_status launch2_rec(CUtensorMap* maps, const Params2& p, void* D, int out_dtype, int qkind, int qfmt,
                        void* qdata, void* qcol, cudaStream_t s) {
    const bool f32 = out_dtype == 1;
    if (D != nullptr && !make_map_2d(&maps[2], f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                     f32 ? 4 : 2, D, p.M, p.N, f32 ? 8 : 16, 32, CU_TENSOR_MAP_SWIZZLE_32B))
        return FP8Q_ERR_CUDA;
    if (qkind < 0) return f32 ? launch2_t<REC, true, 0>(maps, p, s) : launch2_t<REC, false, 0>(maps, p, s);
    // fused output codes: uint8 [M][N] in 32 x 32 boxes (32-byte swizzle)
    if (f32 || !make_map_2d(&maps[5], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qdata, p.M, p.N, 32, 32,
                            CU_TENSOR_MAP_SWIZZLE_32B))
        return f32 ? FP8Q_ERR_ARG : FP8Q_ERR_CUDA;
    if (qcol != nullptr) {
        // the column copy's codes: uint8 [N][M] in 32 x 32 boxes (no swizzle)
        if (!make_map_2d(&maps[6], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qcol, p.N, p.M, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
            return FP8Q_ERR_CUDA;
        if (qkind == FP8Q_BLOCK_1x128)
            return qfmt == FP8Q_E4M3 ? launch2_t<REC, false, 7 + FP8Q_E4M3>(maps, p, s)
                                     : launch2_t<REC, false, 7 + FP8Q_E5M2>(maps, p, s);
        return qfmt == FP8Q_E4M3 ? launch2_t<REC, false, 5 + FP8Q_E4M3>(maps, p, s)
                                 : launch2_t<REC, false, 5 + FP8Q_E5M2>(maps, p, s);
    }
    if (qkind == FP8Q_BLOCK_1x128)
        return qfmt == FP8Q_E4M3 ? launch2_t<REC, false, 3 + FP8Q_E4M3>(maps, p, s)
                                 : launch2_t<REC, false, 3 + FP8Q_E5M2>(maps, p, s);
    return qfmt == FP8Q_E4M3 ? launch2_t<REC, false, 1 + FP8Q_E4M3>(maps, p, s)
                             : launch2_t<REC, false, 1 + FP8Q_E5M2>(maps, p, s);
}

}  // namespace

fp8q_status read_device_errors2(unsigned int* flags) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_errors2, sizeof(v)) != cudaSuccess) return FP8Q_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_device_errors2, &zero, sizeof(zero)) != cudaSuccess) return FP8Q_ERR_CUDA;
    *flags |= v;
    return FP8Q_OK;
}

fp8q_status launch_gemm_pair(const GemmOperand& A, const GemmOperand& B, void* D, int out_dtype, int64_t M,
                             int64_t N, int64_t K, cudaStream_t s, int qkind, int qfmt, void* qdata, void* qscale,
                             unsigned long long* qcounters, void* qcol, void* qscale_col) {
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FP8Q_ERR_SHAPE;
    const bool mx = A.kind == FP8Q_MXFP8_1x32;
    const bool pt = A.kind == FP8Q_PERTENSOR_CURRENT || A.kind == FP8Q_PERTENSOR_DELAYED;
    const bool pc = A.kind == FP8Q_PERCHANNEL_CURRENT;
    static_assert(Cfg<REC_MX>::BN == Cfg<REC_PT>::BN && Cfg<REC_B2D>::BN == Cfg<REC_B1D>::BN, "tile widths");
    const int bn = (mx || pt || pc) ? Cfg<REC_PT>::BN : Cfg<REC_B2D>::BN;
    CUtensorMap maps[7];
    memset(maps, 0, sizeof(maps));
    Params2 p;
    memset(&p, 0, sizeof(p));
    p.hasD = D != nullptr;
    p.wait_ns = wait_limit_ns();
    p.stall = take_stall();
    p.qscale = (uint8_t*)qscale;
    p.qscale_col = qscale_col;
    p.qcounters = qcounters;
    if (qkind >= 0 && qcounters != nullptr && cudaMemsetAsync(qcounters, 0, 3 * sizeof(unsigned long long), s) != cudaSuccess)
        return FP8Q_ERR_CUDA;
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_m2 = (M + 255) / 256;
    p.tiles_n = (N + bn - 1) / bn;
    p.nkb = (K + BK - 1) / BK;
    p.nkbq = p.nkb;
    p.nbnq = (N + 127) / 128;
    p.tiles_m128 = (M + 127) / 128;
    p.nbn128 = (N + 127) / 128;
    p.Mp = p.tiles_m128 * 128;
    p.Np = p.nbn128 * 128;
    if (p.Mp * p.nkb >= ((int64_t)1 << 31) || p.Np * p.nkb >= ((int64_t)1 << 31)) return FP8Q_ERR_SHAPE;
    if (!make_map_2d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A.data, M, K, 128, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B.data, N, K, 128, bn / 2, CU_TENSOR_MAP_SWIZZLE_128B))
        return FP8Q_ERR_CUDA;
    const uint32_t shape = ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
    const uint32_t fmts = ((uint32_t)A.fmt << 7) | ((uint32_t)B.fmt << 10);
    if (mx) {
        // scale tiles as rows of 128 uint32 (512 bytes): [row tiles x K-block groups][128]
        if (!make_map_2d(&maps[3], CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, A.scale, p.tiles_m128 * p.nkb, 128, 128, 1,
                         CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_map_2d(&maps[4], CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, B.scale, p.nbn128 * p.nkb, 128, 128, 1,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return FP8Q_ERR_CUDA;
        p.idesc = shape | fmts | (1u << 23);
        return launch2_rec<REC_MX>(maps, p, D, out_dtype, qkind, qfmt, qdata, qcol, s);
    }
    maps[3] = maps[0];
    maps[4] = maps[1];
    p.idesc = shape | fmts | (1u << 4);
    if (pt) {
        p.sa_inv = A.scale_inv;
        p.sb_inv = B.scale_inv;
        return launch2_rec<REC_PT>(maps, p, D, out_dtype, qkind, qfmt, qdata, qcol, s);
    }
    if (pc) {  // the copies' per-row factors, fp32 padded to 128 entries
        if (((uintptr_t)A.scale | (uintptr_t)B.scale) & 15) return FP8Q_ERR_ARG;
        p.bsa = (const float*)A.scale;
        p.bsb = (const float*)B.scale;
        return launch2_rec<REC_PC>(maps, p, D, out_dtype, qkind, qfmt, qdata, qcol, s);
    }
    // blockwise scale rows are fetched by bulk copies: 16-byte aligned bases
    if (((uintptr_t)A.scale | (uintptr_t)B.scale) & 15) return FP8Q_ERR_ARG;
    p.bsa = (const float*)A.scale;
    p.bsb = (const float*)B.scale;
    const int kbs = A.kblock;  // the scales' K block: 128, or a generic 32, 64, 256
    p.nkbq = (K + kbs - 1) / kbs;
    p.nbnq = (N + kbs - 1) / kbs;
    if (p.Mp * p.nkbq >= ((int64_t)1 << 31) || p.Np * p.nkbq >= ((int64_t)1 << 31)) return FP8Q_ERR_SHAPE;
    const bool b2 = B.kind == FP8Q_BLOCK_128x128;
    if (kbs == 128)
        return b2 ? launch2_rec<REC_B2D>(maps, p, D, out_dtype, qkind, qfmt, qdata, qcol, s)
                  : launch2_rec<REC_B1D>(maps, p, D, out_dtype, qkind, qfmt, qdata, qcol, s);
    if (qkind >= 0) return FP8Q_ERR_UNSUPPORTED;  // the fused output quantize takes 128-wide K blocks
    if (D == nullptr) return FP8Q_ERR_ARG;
    const bool f32 = out_dtype == 1;
    if (!make_map_2d(&maps[2], f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f32 ? 4 : 2,
                     D, p.M, p.N, f32 ? 8 : 16, 32, CU_TENSOR_MAP_SWIZZLE_32B))
        return FP8Q_ERR_CUDA;
    switch (kbs * 2 + (b2 ? 1 : 0)) {
#define FP8Q_KB_CASE(KBV)                                                                                     \
    case KBV * 2 + 1:                                                                                         \
        return f32 ? launch2_t<REC_B2D, true, 0, KBV>(maps, p, s) : launch2_t<REC_B2D, false, 0, KBV>(maps, p, s); \
    case KBV * 2:                                                                                             \
        return f32 ? launch2_t<REC_B1D, true, 0, KBV>(maps, p, s) : launch2_t<REC_B1D, false, 0, KBV>(maps, p, s);
        FP8Q_KB_CASE(32)
        FP8Q_KB_CASE(64)
        FP8Q_KB_CASE(256)
#undef FP8Q_KB_CASE
        default:
            return FP8Q_ERR_UNSUPPORTED;
    }
}

}  // namespace fp8q
