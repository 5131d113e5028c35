// tcgen05 / TMA helpers shared by the GEMM kernels of libfp8q: TMEM fences
// and loads, shared-memory matrix descriptors, bf16 packing, TMA stores of the
// output through swizzled staging boxes, and the persistent tile order.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fp8q {

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: start >> 4, leading byte offset >> 4,
// stride byte offset >> 4, fixed 0b001 at bit 46, swizzle mode at bit 61.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swz << 61);
}
// K-major operand tile, rows of 128 bytes in the 128-byte swizzle: 8-row
// groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) { return smem_desc(addr, 16, 1024, 2); }

#define FP8Q_LD32(addr, r)                                                                                          \
    asm volatile(                                                                                                   \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18," \
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                              \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),         \
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),    \
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),  \
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])   \
        : "r"(addr))

#define FP8Q_LD16(addr, r)                                                                                     \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, " \
                 "[%16];"                                                                                      \
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),          \
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),      \
                   "=r"(r[14]), "=r"(r[15])                                                                     \
                 : "r"(addr))

// 16 columns of TMEM, waited for, as 8 column pairs in 64-bit registers (the
// operands of the two-lane fp32 instructions): the load, its wait and the
// packing in one asm block, so the pairs are formed from completed registers.
#define FP8Q_LD16_PAIRS(addr, d)                                                                                \
    asm volatile(                                                                                               \
        "{\n .reg .b32 t<16>;\n"                                                                                \
        " tcgen05.ld.sync.aligned.32x32b.x16.b32 {t0,t1,t2,t3,t4,t5,t6,t7,t8,t9,t10,t11,t12,t13,t14,t15}, [%8];\n" \
        " tcgen05.wait::ld.sync.aligned;\n"                                                                      \
        " mov.b64 %0, {t0,t1};\n mov.b64 %1, {t2,t3};\n mov.b64 %2, {t4,t5};\n mov.b64 %3, {t6,t7};\n"            \
        " mov.b64 %4, {t8,t9};\n mov.b64 %5, {t10,t11};\n mov.b64 %6, {t12,t13};\n mov.b64 %7, {t14,t15};\n}\n"  \
        : "=l"(d[0]), "=l"(d[1]), "=l"(d[2]), "=l"(d[3]), "=l"(d[4]), "=l"(d[5]), "=l"(d[6]), "=l"(d[7])          \
        : "r"(addr)                                                                                             \
        : "memory")

__device__ __forceinline__ float2 u64_as_float2(uint64_t u) {
    union {
        uint64_t u;
        float2 f;
    } x;
    x.u = u;
    return x.f;
}

// Registers written by tcgen05.ld are valid only after tcgen05.wait::ld; this
// empty asm, placed after the wait, keeps the compiler from hoisting their
// uses above it.
__device__ __forceinline__ void reg_fence16(uint32_t* r) {
    asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]));
}
__device__ __forceinline__ void reg_fence32(uint32_t* r) {
    reg_fence16(r);
    reg_fence16(r + 16);
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Tile order: groups of 8 M-blocks, N-blocks outer inside a group, so the
// CTAs working at one time share A and B panels in L2.
__device__ __forceinline__ void tile_coords(int64_t t, int64_t tiles_m, int64_t tiles_n, int64_t& mb, int64_t& nb) {
    const int64_t G = 8;
    const int64_t group = t / (G * tiles_n);
    const int64_t first = group * G;
    const int64_t gs = (tiles_m - first) < G ? (tiles_m - first) : G;
    const int64_t in = t - group * G * tiles_n;
    mb = first + in % gs;
    nb = in / gs;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x),
                 "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// all but the most recent bulk group have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Stores this warp's 32 rows x 64 columns of D (v: the lane's row, scaled by
// `scale`) through its 1 KB shared-memory staging box and TMA stores, in
// rounds of 32-byte row pieces (16 bf16 / 8 fp32) in the 32-byte swizzle
// (16-byte chunk c of row r at r*32 + (c ^ ((r / 4) % 2))*16, so the lanes'
// writes do not conflict).  The TMA clips rows / columns outside D; boxes
// wholly outside D are skipped.
template <bool OUT_F32>
__device__ __forceinline__ void store_slice(const CUtensorMap* mapD, uint8_t* stg, uint32_t stg_s, int lane, int x0,
                                            int y0, int n_extent, int m_extent, const float* v, float scale) {
    const int r = lane;
    constexpr int kCols = OUT_F32 ? 8 : 16;  // columns per 32-byte piece
#pragma unroll
    for (int rd = 0; rd < 64 / kCols; ++rd) {
        bulk_wait_read();  // the previous box has been read out of stg
        __syncwarp();
        const float* q = v + kCols * rd;
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
        const int sw = (r >> 2) & 1;
        *(uint4*)(stg + r * 32 + ((0 ^ sw) << 4)) = c0;
        *(uint4*)(stg + r * 32 + ((1 ^ sw) << 4)) = c1;
        fence_async_smem();
        __syncwarp();
        if (lane == 0 && x0 + kCols * rd < n_extent && y0 < m_extent) {
            tma_store_2d(mapD, x0 + kCols * rd, y0, stg_s);
            bulk_commit();
        }
    }
}

}  // namespace fp8q
