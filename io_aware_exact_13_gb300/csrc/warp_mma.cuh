// warp_mma.cuh -- warp-level 16x8x16 MMA and ldmatrix wrappers for the
// small-tile (decoding) kernels: one-instruction inline-PTX wrappers written
// from the PTX ISA description of each instruction.
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace fa {

// D(16x8, fp32) += A(16x16, row) * B(16x8, col), 16-bit inputs. Fragments (per
// lane, g = lane / 4, c = lane % 4): A a0 = (row g, cols 2c, 2c+1), a1 = row g+8,
// a2 = cols + 8, a3 = row g+8 and cols + 8; B b0 = (rows 2c, 2c+1, col g), b1 =
// rows + 8; D d0, d1 = (row g, cols 2c, 2c+1), d2, d3 = row g+8.
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (BF16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 16-bit matrices from shared memory: lane i gives the address of row
// i % 8 of matrix i / 8, and register j receives matrix j as (row lane / 4,
// cols 2 (lane % 4), +1). The .trans form delivers each matrix transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                              uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// cp_async16, cp_async_commit and cp_async_wait live in ptx.cuh.

}  // namespace fa
