// Scaled FP8 GEMM on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// D[M][N] = A_q[M][K] . B_q[N][K]^T, both operands K-contiguous ("2025 FP8
// quantized-training guide", sec. 3.1: fprop / dgrad / wgrad take quantized
// inputs, outputs stay BF16 / FP32).  Three scale treatments:
//   per-tensor   one MMA chain per tile, D = s_inv_A * s_inv_B * acc in the
//                epilogue (sec. 2.1);
//   MXFP8        kind::mxf8f6f4.block_scale: the tensor core applies the E8M0
//                scale of every 32-wide K block itself (sec. 2.3; "mastering FP8
//                LLM training", strategy 4: hardware-native on Blackwell);
//   blockwise    each 128-wide K block is its own MMA chain into one of two
//                TMEM buffers; the epilogue warps scale that partial by
//                d_A[m][kb] * d_B[n(/128)][kb] and add it to fp32 register
//                accumulators (sec. 2.2 1x128 x 128x128 tiles, or 1x128 x 1x128).
//
// Persistent kernel, one CTA per SM, 576 threads:
//   warp 0      TMA producer: A box 128x128 B, B box 256x128 B (128-byte
//               swizzle) per stage (4 stages), plus the MX scale tiles (bulk copies);
//   warp 1      TMEM allocator and single-thread MMA issuer (M128 N256 K32);
//   warps 2-17  epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (its rows)
//               and columns 64 ((w - 2) / 4) .. +63, and writes them through a
//               swizzled shared-memory box and a TMA store.
// Every mbarrier wait is bounded (about one second of %globaltimer); a wait
// that gives up sets bit 0 of g_device_errors, raises a CTA-wide abort flag,
// and the CTA drains its in-flight copies and MMAs (bounded) and frees TMEM.
#include <cuda.h>

#include "fp8q_internal.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace fp8q {

__device__ unsigned int g_device_errors = 0;

namespace {

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 4;
constexpr int kEpiWarps = 16;
constexpr int kEpiCols = BN / (kEpiWarps / 4);  // accumulator columns per epilogue warp
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t A_STAGE = BM * BK, B_STAGE = BN * BK;
constexpr uint32_t SFA_STAGE = 512, SFB_STAGE = 1024;
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_STAGE;
constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_STAGE;
constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_STAGE;
constexpr uint32_t OFF_SBW = OFF_SFB + STAGES * SFB_STAGE;      // per-epilogue-warp 1x128 B scales
constexpr uint32_t OFF_STG = (OFF_SBW + kEpiWarps * kEpiCols * 4 + 1023) / 1024 * 1024;
constexpr uint32_t STG_WARP = 32 * 32;                           // one 32-row x 32-byte output box per warp
constexpr uint32_t OFF_BAR = OFF_STG + kEpiWarps * STG_WARP;
constexpr uint32_t NBARS = 2 * STAGES + 5;
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * NBARS;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;            // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_TMEM_COL = 256;                            // MX scale slots: 12 columns per stage

enum { REC_PT = 0, REC_MX = 1, REC_B2D = 2, REC_B1D = 3 };

struct Params {
    int64_t M, N, K;
    int64_t tiles_m, tiles_n, nkb;
    void* D;
    const float* sa_inv;    // per-tensor
    const float* sb_inv;
    const uint8_t* sfa;     // MX packed tiles
    const uint8_t* sfb;
    const float* bsa;       // blockwise [nkb][Mp]
    const float* bsb;       // [nkb][Np] (1x128) or [ceil(N/128)][nkb] (128x128)
    int64_t Mp, Np, nbn128;
    uint32_t idesc;
    uint64_t wait_ns;  // bounded-wait limit
    int stall;         // 1: the producer issues no loads (diagnostic)
};

// ------------------------------------------------------------ PTX wrappers

// The phase is usually complete already: test it inline (no call, so no
// register save / restore around it) and only fall back to the bounded loop.
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, volatile int* abort_flag, uint64_t limit_ns) {
    if (mbar_try(a, parity)) return true;
    return mbar_wait_bounded(a, parity, abort_flag, &g_device_errors, 1u, limit_ns);
}

__device__ __forceinline__ void tc_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar) : "memory");
}

__device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_mx(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
            d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc));
}
__device__ __forceinline__ void tc_cp_32x128b(uint32_t taddr, uint64_t desc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc));
}

template <int REC, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmD, const Params p) {
    constexpr uint32_t kAcc = (REC == REC_PT) ? 2u : 1u;  // TMEM accumulator buffers of 256 columns
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(smem);
    auto full = [&](int s) { return sb + OFF_BAR + 8u * s; };
    auto empty = [&](int s) { return sb + OFF_BAR + 8u * (STAGES + s); };
    auto tfull = [&](int b) { return sb + OFF_BAR + 8u * (2 * STAGES + b); };
    auto tempty = [&](int b) { return sb + OFF_BAR + 8u * (2 * STAGES + 2 + b); };
    const uint32_t mma_done = sb + OFF_BAR + 8u * (2 * STAGES + 4);
    uint32_t* tmem_slot = (uint32_t*)(smem + OFF_MISC);
    volatile int* abort_flag = (volatile int*)(smem + OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), kEpiWarps);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_map(&tmA);
        prefetch_map(&tmB);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int64_t ntiles = p.tiles_m * p.tiles_n;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && !p.stall) {  // a stalled launch (diagnostic) loads nothing
            int s = 0;
            uint32_t ph = 0;
            uint32_t filled = 0, fill_par = 0;  // per-stage bits for the abort drain
            bool ok = true;
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                int64_t mb, nb;
                tile_coords(t, p.tiles_m, p.tiles_n, mb, nb);
                const bool b2 = (2 * nb + 1) < p.nbn128;  // second 128-row scale tile of B exists
                for (int64_t kb = 0; kb < p.nkb; ++kb) {
                    if (!mbar_wait(empty(s), ph ^ 1u, abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    uint32_t bytes = A_STAGE + B_STAGE;
                    if (REC == REC_MX) bytes += SFA_STAGE + (b2 ? 1024u : 512u);
                    mbar_expect_tx(full(s), bytes);
                    tma_load_2d(sb + OFF_A + s * A_STAGE, &tmA, (int)(kb * BK), (int)(mb * BM), full(s));
                    tma_load_2d(sb + OFF_B + s * B_STAGE, &tmB, (int)(kb * BK), (int)(nb * BN), full(s));
                    if (REC == REC_MX) {
                        bulk_load(sb + OFF_SFA + s * SFA_STAGE, p.sfa + (mb * p.nkb + kb) * 512, 512, full(s));
                        bulk_load(sb + OFF_SFB + s * SFB_STAGE, p.sfb + (2 * nb * p.nkb + kb) * 512, 512, full(s));
                        if (b2)
                            bulk_load(sb + OFF_SFB + s * SFB_STAGE + 512, p.sfb + ((2 * nb + 1) * p.nkb + kb) * 512,
                                      512, full(s));
                    }
                    filled |= 1u << s;
                    fill_par = (fill_par & ~(1u << s)) | (ph << s);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // let copies already issued land before the CTA exits (bounded)
                for (int i = 0; i < STAGES; ++i)
                    if (filled >> i & 1u) mbar_drain(full(i), (fill_par >> i) & 1u, p.wait_ns / 10);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t tile_i = 0;
            uint64_t kbg = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++tile_i) {
                if (REC == REC_PT || REC == REC_MX) {
                    // per-tensor: two accumulator buffers, so the epilogue of tile i
                    // overlaps the MMAs of tile i + 1; MX: one (its scale slots use the rest)
                    if (!mbar_wait(tempty(tile_i % kAcc), ((tile_i / kAcc) & 1u) ^ 1u, abort_flag, p.wait_ns)) break;
                    tc_fence_after();
                }
                for (int64_t kb = 0; kb < p.nkb; ++kb) {
                    uint32_t dcol = (REC == REC_PT) ? (tile_i % kAcc) * BN : 0;
                    if (REC == REC_B2D || REC == REC_B1D) {
                        const uint32_t buf = (uint32_t)(kbg & 1u);
                        if (!mbar_wait(tempty(buf), (uint32_t)((kbg >> 1) & 1u) ^ 1u, abort_flag, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        dcol = buf * BN;
                    }
                    if (!mbar_wait(full(s), ph, abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sb + OFF_A + s * A_STAGE, b0 = sb + OFF_B + s * B_STAGE;
                    if (REC == REC_MX) {
                        const uint32_t sfa_t = tmem + SF_TMEM_COL + 12u * s;
                        tc_cp_32x128b(sfa_t, smem_desc(sb + OFF_SFA + s * SFA_STAGE, 0, 128, 0));
                        tc_cp_32x128b(sfa_t + 4, smem_desc(sb + OFF_SFB + s * SFB_STAGE, 0, 128, 0));
                        tc_cp_32x128b(sfa_t + 8, smem_desc(sb + OFF_SFB + s * SFB_STAGE + 512, 0, 128, 0));
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k) {
                            const uint32_t idesc = p.idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29);
                            mma_mx(tmem, desc_sw128(a0 + 32 * k), desc_sw128(b0 + 32 * k), idesc, sfa_t, sfa_t + 4,
                                   (kb > 0 || k > 0) ? 1u : 0u);
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k) {
                            const uint32_t acc = (REC == REC_PT) ? ((kb > 0 || k > 0) ? 1u : 0u) : (k > 0 ? 1u : 0u);
                            mma_f8(tmem + dcol, desc_sw128(a0 + 32 * k), desc_sw128(b0 + 32 * k), p.idesc, acc);
                        }
                    }
                    tc_commit(empty(s));
                    if (REC == REC_B2D || REC == REC_B1D) {
                        tc_commit(tfull((uint32_t)(kbg & 1u)));
                        ++kbg;
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                if (REC == REC_PT || REC == REC_MX) tc_commit(tfull(tile_i % kAcc));
            }
            // every MMA / copy this thread issued has completed once mma_done fires
            tc_commit(mma_done);
            mbar_drain(mma_done, 0, p.wait_ns);
        }
    } else {
        // ------------------------------------------------ epilogue warps
        // warp w owns TMEM lanes 32 (w % 4) .. +31 (its rows) and columns
        // 64 j .. 64 j + 63, j = (w - 2) / 4, of the 256-column accumulator
        const int ew = warp - 2, q = warp & 3, j = ew >> 2;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        float sab = 1.0f;
        if (REC == REC_PT) sab = __fmul_rn(*p.sa_inv, *p.sb_inv);
        float* sbw = (float*)(smem + OFF_SBW) + ew * kEpiCols;
        uint8_t* stg = smem + OFF_STG + ew * STG_WARP;
        const uint32_t stg_s = sb + OFF_STG + ew * STG_WARP;
        uint32_t tile_i = 0;
        uint32_t kbg = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++tile_i) {
            int64_t mb, nb;
            tile_coords(t, p.tiles_m, p.tiles_n, mb, nb);
            const int64_t row = mb * BM + 32 * q + lane;
            const int64_t col0 = nb * BN + kEpiCols * j;
            const uint32_t tcol = (uint32_t)(kEpiCols * j);
            if (REC == REC_PT || REC == REC_MX) {
                const uint32_t abuf = tile_i % kAcc;
                if (!mbar_wait(tfull(abuf), (tile_i / kAcc) & 1u, abort_flag, p.wait_ns)) break;
                tc_fence_after();
                // drain this warp's 64 columns into registers, hand TMEM back, then store
                uint32_t r[64];
                FP8Q_LD32(tmem + lane_base + abuf * BN + tcol, r);
                FP8Q_LD32(tmem + lane_base + abuf * BN + tcol + 32, (r + 32));
                tc_wait_ld();
                reg_fence32(r);
                reg_fence32(r + 32);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty(abuf));
                float vf[64];
#pragma unroll
                for (int i = 0; i < 64; ++i) vf[i] = __uint_as_float(r[i]);
                store_slice<OUT_F32>(&tmD, stg, stg_s, lane, (int)col0, (int)(mb * BM + 32 * q), (int)p.N, (int)p.M, vf,
                                     sab);
            } else {
                float acc[kEpiCols];
#pragma unroll
                for (int i = 0; i < kEpiCols; ++i) acc[i] = 0.0f;
                const bool cvalid = (col0 < p.N);
                // the next K block's scales are loaded one iteration ahead (32-bit offsets:
                // the host checks that the scale arrays index below 2^31)
                const int nkb = (int)p.nkb;
                const int nblk = (int)((nb * BN + kEpiCols * j) / 128);
                const bool bvalid = nblk < (int)p.nbn128;
                const int Mp = (int)p.Mp, Np = (int)p.Np;
                const float* pa = p.bsa + (int)row;                                   // [kb][Mp]
                const float* pb = p.bsb + (bvalid ? nblk * nkb : 0);                  // 128x128: [nblk][kb]
                const float* pv = p.bsb + (cvalid ? (int)col0 : 0) + 2 * lane;        // 1x128: [kb][Np]
                float sa_n = __ldg(pa), sb_n = (REC == REC_B2D && bvalid) ? __ldg(pb) : 0.0f;
                float2 sv_n = make_float2(0.f, 0.f);
                if (REC == REC_B1D && cvalid) sv_n = __ldg((const float2*)pv);
                bool ok = true;
                for (int kb = 0; kb < nkb; ++kb, ++kbg) {
                    const float sa = sa_n, sbk = sb_n;
                    const float2 sv = sv_n;
                    if (kb + 1 < nkb) {
                        sa_n = __ldg(pa + (kb + 1) * Mp);
                        if (REC == REC_B2D && bvalid) sb_n = __ldg(pb + kb + 1);
                        if (REC == REC_B1D && cvalid) sv_n = __ldg((const float2*)(pv + (kb + 1) * Np));
                    }
                    if (REC == REC_B1D) {
                        __syncwarp();
                        *(float2*)(sbw + 2 * lane) = sv;  // B scales of this warp's 64 columns
                        __syncwarp();
                    }
                    const float sc = __fmul_rn(sa, sbk);
                    const uint32_t buf = (uint32_t)(kbg & 1u);
                    if (!mbar_wait(tfull(buf), (uint32_t)((kbg >> 1) & 1u), abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t base = tmem + lane_base + buf * BN + tcol;
                    // 16-column chunks; the four warps sharing an SM sub-partition
                    // hide each other's TMEM load latency
#pragma unroll
                    for (int c = 0; c < kEpiCols / 16; ++c) {
                        uint32_t r[16];
                        FP8Q_LD16(base + 16 * c, r);
                        tc_wait_ld();
                        reg_fence16(r);
                        if (REC == REC_B2D) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[16 * c + i] = fmaf(__uint_as_float(r[i]), sc, acc[16 * c + i]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; i += 4) {
                                // d_A[m][kb] (this thread's row) x d_B[n][kb] (shared by the warp)
                                const float4 s4 = *(const float4*)(sbw + 16 * c + i);
                                acc[16 * c + i] = fmaf(__uint_as_float(r[i]), __fmul_rn(sa, s4.x), acc[16 * c + i]);
                                acc[16 * c + i + 1] =
                                    fmaf(__uint_as_float(r[i + 1]), __fmul_rn(sa, s4.y), acc[16 * c + i + 1]);
                                acc[16 * c + i + 2] =
                                    fmaf(__uint_as_float(r[i + 2]), __fmul_rn(sa, s4.z), acc[16 * c + i + 2]);
                                acc[16 * c + i + 3] =
                                    fmaf(__uint_as_float(r[i + 3]), __fmul_rn(sa, s4.w), acc[16 * c + i + 3]);
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty(buf));
                }
                if (!ok) break;
                store_slice<OUT_F32>(&tmD, stg, stg_s, lane, (int)col0, (int)(mb * BM + 32 * q), (int)p.N, (int)p.M, acc,
                                     1.0f);
            }
        }
    }

    if (warp >= 2 && lane == 0) bulk_wait_all();  // this warp's output boxes are written
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ------------------------------------------------------------------ host

// 2-D map over a K-contiguous uint8 matrix [rows][K], box 128 bytes x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t K, uint32_t box_rows) {
    return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, K, 128, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int REC, bool F32>
fp8q_status launch_t(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md, const Params& p,
                     cudaStream_t s) {
    auto kern = gemm_kernel<REC, F32>;
    static PerDevice<bool> attr;
    if (!smem_opt_in(attr, kern, SMEM_BYTES)) return FP8Q_ERR_CUDA;
    const int sms = sm_count();
    if (sms < 1) return FP8Q_ERR_CUDA;
    const int64_t ntiles = p.tiles_m * p.tiles_n;
    const int grid = (int)(ntiles < sms ? ntiles : sms);
    kern<<<grid, kThreads, SMEM_BYTES, s>>>(ma, mb, md, p);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

template <int REC>
fp8q_status launch_rec(const CUtensorMap& ma, const CUtensorMap& mb, const Params& p, int out_dtype, cudaStream_t s) {
    // D [M][N] row-major: 32-row boxes of 32 bytes (16 bf16 / 8 fp32) in the 32-byte swizzle
    CUtensorMap md;
    const bool f32 = out_dtype == 1;
    if (!make_map_2d(&md, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f32 ? 4 : 2, p.D,
                     p.M, p.N, f32 ? 8 : 16, 32, CU_TENSOR_MAP_SWIZZLE_32B))
        return FP8Q_ERR_CUDA;
    return f32 ? launch_t<REC, true>(ma, mb, md, p, s) : launch_t<REC, false>(ma, mb, md, p, s);
}

}  // namespace

fp8q_status read_device_errors(unsigned int* flags, cudaStream_t s) {
    if (cudaStreamSynchronize(s) != cudaSuccess) return FP8Q_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_errors, sizeof(v)) != cudaSuccess) return FP8Q_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_device_errors, &zero, sizeof(zero)) != cudaSuccess) return FP8Q_ERR_CUDA;
    *flags = v;
    return FP8Q_OK;
}

int g_gemm_variant = 0;

fp8q_status launch_gemm(const GemmOperand& A, const GemmOperand& B, void* D, int out_dtype, int64_t M, int64_t N,
                        int64_t K, cudaStream_t s) {
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FP8Q_ERR_SHAPE;
    // SM pairs once there are enough 256 x 256 tiles to occupy the GPU's SMs
    // in pairs (and, for blockwise scales, which the pair kernel fetches with
    // bulk copies, 16-byte aligned scale arrays)
    const bool scales_aligned =
        A.kind != FP8Q_BLOCK_1x128 || ((((uintptr_t)A.scale) | ((uintptr_t)B.scale)) & 15) == 0;
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    // per-channel scales only on SM pairs
    // per-channel scales and K blocks other than 128 only on SM pairs
    if (A.kind == FP8Q_PERCHANNEL_CURRENT || (A.kblock != 0 && A.kblock != 128) || g_gemm_variant == 2 ||
        (g_gemm_variant == 0 && scales_aligned && pair_tiles >= 64))
        return launch_gemm_pair(A, B, D, out_dtype, M, N, K, s);
    CUtensorMap ma, mb;
    if (!make_map(&ma, A.data, M, K, BM) || !make_map(&mb, B.data, N, K, BN)) return FP8Q_ERR_CUDA;
    Params p;
    memset(&p, 0, sizeof(p));
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_m = (M + BM - 1) / BM;
    p.tiles_n = (N + BN - 1) / BN;
    p.nkb = (K + BK - 1) / BK;
    p.D = D;
    p.wait_ns = wait_limit_ns();
    p.stall = take_stall();
    p.Mp = p.tiles_m * BM;
    if (p.Mp * p.nkb >= ((int64_t)1 << 31) || ((N + 127) / 128 * 128) * p.nkb >= ((int64_t)1 << 31))
        return FP8Q_ERR_SHAPE;  // the blockwise epilogue indexes its scales with 32-bit offsets
    p.Np = (N + 127) / 128 * 128;
    p.nbn128 = (N + 127) / 128;
    const bool pt = A.kind == FP8Q_PERTENSOR_CURRENT || A.kind == FP8Q_PERTENSOR_DELAYED;
    // instruction descriptor: M = 128 (bits 24-28: M >> 4), N = 256 (bits 17-22: N >> 3),
    // A / B formats at bits 7-9 / 10-12 (0 = E4M3, 1 = E5M2)
    const uint32_t shape = ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
    const uint32_t fmts = ((uint32_t)A.fmt << 7) | ((uint32_t)B.fmt << 10);
    if (A.kind == FP8Q_MXFP8_1x32) {
        p.sfa = (const uint8_t*)A.scale;
        p.sfb = (const uint8_t*)B.scale;
        p.idesc = shape | fmts | (1u << 23);  // scale type UE8M0; scale-factor ids added per MMA
        return launch_rec<REC_MX>(ma, mb, p, out_dtype, s);
    }
    p.idesc = shape | fmts | (1u << 4);  // D format F32
    if (pt) {
        p.sa_inv = A.scale_inv;
        p.sb_inv = B.scale_inv;
        return launch_rec<REC_PT>(ma, mb, p, out_dtype, s);
    }
    p.bsa = (const float*)A.scale;
    p.bsb = (const float*)B.scale;
    if (B.kind == FP8Q_BLOCK_128x128) return launch_rec<REC_B2D>(ma, mb, p, out_dtype, s);
    return launch_rec<REC_B1D>(ma, mb, p, out_dtype, s);
}

}  // namespace fp8q
