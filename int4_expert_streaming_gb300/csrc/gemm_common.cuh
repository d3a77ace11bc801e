// gemm_common.cuh -- device helpers shared by the prefill grouped GEMMs:
// exact int4/int8 dequantisation to bf16 (magic-number code conversion and
// packed fp32x2 arithmetic), shared-memory and cp.async wrappers, TMA loads,
// the pre-swizzled SwiGLU buffer layout, tensor-memory loads and vector
// reductions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "umma.cuh"

namespace moe {
namespace gemmc {

using namespace umma;

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// packed fp32 pairs (one register pair, two IEEE operations per instruction)
__device__ __forceinline__ uint64_t f2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint32_t bf16x2_of(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return pack_bf16(lo, hi);
}

// code byte i of v as the bits of the float 2^23 + q (exact)
__device__ __forceinline__ uint32_t code_bits(uint32_t v, int i) { return __byte_perm(v, 0x4B000000u, 0x7440u | i); }

// bf16(fma(s, q, b)) of code bytes (x byte i, y byte j) as a bf16 pair;
// m2 = (-2^23, -2^23)
__device__ __forceinline__ uint32_t dq_pair(uint32_t x, int i, uint32_t y, int j, uint64_t s2, uint64_t b2,
                                            uint64_t m2) {
    return bf16x2_of(fma_f2(s2, add_f2(f2(code_bits(x, i), code_bits(y, j)), m2), b2));
}

// 8 consecutive int4 columns (one code word, column c in nibble c)
__device__ __forceinline__ uint4 dq8_int4(uint32_t wd, uint64_t s2, uint64_t b2, uint64_t m2) {
    const uint32_t lo = wd & 0x0F0F0F0Fu, hi = (wd >> 4) & 0x0F0F0F0Fu;  // even / odd columns
    return make_uint4(dq_pair(lo, 0, hi, 0, s2, b2, m2), dq_pair(lo, 1, hi, 1, s2, b2, m2),
                      dq_pair(lo, 2, hi, 2, s2, b2, m2), dq_pair(lo, 3, hi, 3, s2, b2, m2));
}

// int4 code byte i of v as the bits of the float 128 + q (exact: q sits in
// mantissa bits 16-19 under the exponent of 128)
__device__ __forceinline__ uint32_t code128_bits(uint32_t v, int i) {
    return __byte_perm(v, 0x43000000u, 0x7044u | ((uint32_t)i << 8));
}

// 8 consecutive int4 columns as fma(s, 128 + q, c) with c = b - 128 s exact,
// which equals fma(s, q, b): both round the same exact value s*q + b once
__device__ __forceinline__ uint4 dq8_int4_fast(uint32_t wd, uint64_t s2, uint64_t c2) {
    const uint32_t lo = wd & 0x0F0F0F0Fu, hi = (wd >> 4) & 0x0F0F0F0Fu;
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = bf16x2_of(fma_f2(s2, f2(code128_bits(lo, i), code128_bits(hi, i)), c2));
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// c = b - 128 s in fp32; true if that subtraction was exact (TwoSum error 0,
// -128 s itself being exact)
__device__ __forceinline__ bool shifted_bias(float s, float b, float& c) {
    const float t = __fmul_rn(-128.0f, s);
    c = __fadd_rn(b, t);
    const float bv = __fsub_rn(c, b), av = __fsub_rn(c, bv);
    return __fadd_rn(__fsub_rn(b, av), __fsub_rn(t, bv)) == 0.0f;
}

// 8 consecutive int8 columns (two code words, column c in byte c)
__device__ __forceinline__ uint4 dq8_int8(uint32_t w0, uint32_t w1, uint64_t s2, uint64_t b2, uint64_t m2) {
    return make_uint4(dq_pair(w0, 0, w0, 1, s2, b2, m2), dq_pair(w0, 2, w0, 3, s2, b2, m2),
                      dq_pair(w1, 0, w1, 1, s2, b2, m2), dq_pair(w1, 2, w1, 3, s2, b2, m2));
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// TMA: the box at (column x, row y) of a 2D map to shared memory, completion
// counted on the mbarrier
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* b) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(b))
        : "memory");
}
__device__ __forceinline__ void bar_arrive_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
                     smem_u32(b)),
                 "r"(bytes)
                 : "memory");
}

// element offset of (row, col) in a pre-swizzled SwiGLU buffer: planes of 64
// columns, [plane][row][64], 16-byte chunks swizzled by row & 7
__device__ __forceinline__ size_t h_offset(int rows, int row, int col) {
    return ((size_t)(col >> 6) * rows + row) * 64 + ((((col >> 3) ^ row) & 7) << 3) + (col & 7);
}

// 32 lanes x 16 consecutive 32-bit tensor-memory columns
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

// y[0..3] += (a, b, c, d): one 16-byte fp32 reduction in L2
__device__ __forceinline__ void red_add_v4(float* y, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(y), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

}  // namespace gemmc
}  // namespace moe
