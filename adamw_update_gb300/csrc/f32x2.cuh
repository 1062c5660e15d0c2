// f32x2.cuh -- packed pairs of binary32 operations (sm_100 and later).
//
// add.rn.f32x2, mul.rn.f32x2 and fma.rn.f32x2 apply the binary32 operation to
// both lanes of a 64-bit register pair, each lane rounded once to nearest
// even, with subnormal operands and results kept (no .ftz): lane for lane the
// same results as the scalar __fadd_rn / __fmul_rn / __fmaf_rn, for half the
// instructions.  The update is issue-bound wherever HBM is not the limit, so
// pairing two independent operations -- two elements, or the first- and
// second-moment lanes of one element -- into one instruction is a direct gain.
#pragma once

namespace pa {

__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// a + b in both lanes.  Use add2x instead when either operand is a product:
// ptxas may fuse the multiply into this add.
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// a*b + c, each lane rounded once
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c);

// 1.0 in constant memory: the compiler cannot fold its value, so fma2(x, one,
// y) stays a fused operation whose exact product x*1 = x is added to y and
// rounded once -- RN(x + y), signed zeros included -- and no multiply feeding
// x or y can be fused into it.  (ptxas was seen, on GB300 with --fmad false, to
// fuse a packed multiply into a packed add that consumed it, changing the
// rounding; so a packed sum of products is always written with add2x.)
__constant__ float c_one_f32x2 = 1.0f;

__device__ __forceinline__ float2 one_pair()
{
    const float o = c_one_f32x2;
    return make_float2(o, o);
}

// x + y in both lanes, each rounded once, immune to contraction (see above)
__device__ __forceinline__ float2 add2x(float2 x, float2 y, float2 one)
{
    return fma2(x, one, y);
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

}  // namespace pa
