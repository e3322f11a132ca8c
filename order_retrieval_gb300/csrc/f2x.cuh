// f2x.cuh -- pairs of f32 values held in one 64-bit register, the operand form
// of the Blackwell f32x2 instructions (add/sub/mul/fma.rn.f32x2).  Keeping a
// pair packed from its load to its last use leaves the register allocator no
// halves to gather into aligned pairs before each packed instruction.
#pragma once

#include <cstdint>

namespace zeta {

struct F2 {
    uint64_t v;
};

__device__ __forceinline__ F2 f2_pack(float lo, float hi) {
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ F2 f2_pack_u(uint32_t lo, uint32_t hi) {
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ F2 f2_dup(float x) { return f2_pack(x, x); }
__device__ __forceinline__ void f2_unpack(F2 a, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
    F2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) {
    F2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
    F2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
    F2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
}
// Approximate reciprocal of both halves (the MUFU result, denormals flushed).
__device__ __forceinline__ F2 f2_rcp_approx(F2 a) {
    F2 r;
    asm("{\n .reg .f32 l, h;\n mov.b64 {l, h}, %1;\n rcp.approx.ftz.f32 l, l;\n"
        " rcp.approx.ftz.f32 h, h;\n mov.b64 %0, {l, h};\n}\n"
        : "=l"(r.v)
        : "l"(a.v));
    return r;
}
// Both halves rounded to bf16, the low half in the low 16 bits.
__device__ __forceinline__ uint32_t f2_bf16x2(F2 a) {
    uint32_t r;
    asm("{\n .reg .f32 l, h;\n mov.b64 {l, h}, %1;\n cvt.rn.bf16x2.f32 %0, h, l;\n}\n"
        : "=r"(r)
        : "l"(a.v));
    return r;
}
// Two pairs (four consecutive f32) from shared memory.
__device__ __forceinline__ void f2_lds2(uint32_t addr, F2 &a, F2 &b) {
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a.v), "=l"(b.v) : "r"(addr));
}

}  // namespace zeta
