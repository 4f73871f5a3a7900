// NVFP4 encoding of bf16 activations, for GEMM2's A after the SwiGLU step
// of the MoE expert block (page "LLM-Assisted Kernel Development in CuTe
// DSL, Gluon, Helion and Triton", mixture-of-experts section: each expert
// runs GEMM1, SwiGLU, GEMM2).  The pages give no quantisation recipe; the
// one used here keeps the NVFP4 format of the GEMM's operands and picks each
// 16-element block's scale so that its largest magnitude meets the largest
// code.  Per block, every step in fp32 with round-to-nearest-even:
//
//     z_i = x_i * q            (q: the caller's pre-scale for the row)
//     sf  = e4m3(max_i |z_i| / 6), saturating at 448;  d = value of sf
//     c_i = e2m1(z_i / d), saturating at 6, or 0 when d == 0
//
// so x_i ~ c_i * d / q (GEMM2's alpha carries 1 / q).  Codes are packed two
// per byte, the even element in the low nibble; a zero code is written as +0.
// The hardware conversions (cvt.rn.satfinite to e4m3x2 and e2m1x2) round
// to nearest even and saturate, as the recipe asks.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace nvfp4gg {

// e4m3 byte of the block scale for block maximum |z| = amax, and its value d.
// amax / 6 rounded to nearest even from RN(1 / 6) and one residual
// correction (the steps and the theorem of nvfp4_code_quad below); when the
// residual underflows, amax / 6 is below 2^-126 and its e4m3 byte is 0
// either way, and an infinite amax is passed through (inf / 6 = inf).
__device__ __forceinline__ uint32_t nvfp4_block_scale(float amax, float& d) {
    const float y6 = __uint_as_float(0x3E2AAAABu);   // RN(1 / 6)
    const float q0 = __fmul_rn(amax, y6);
    const float q1 = __fmaf_rn(__fmaf_rn(-q0, 6.0f, amax), y6, q0);
    const float s = amax == __uint_as_float(0x7F800000u) ? amax : q1;
    const uint32_t sf = __nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3);
    d = __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(sf), __NV_E4M3)));
    return sf;
}

// (a0 * b, a1 * b) for fp32 bit patterns a0, a1, from one packed fp32
// multiply (each element rounded to nearest even, as a scalar multiply);
// b2 holds b in both halves.
__device__ __forceinline__ void mul2_rn(uint32_t a0, uint32_t a1, uint64_t b2, uint32_t& r0,
                                        uint32_t& r1) {
    asm("{\n\t.reg .b64 a, r;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mul.rn.f32x2 r, a, %4;\n\t"
        "mov.b64 {%0, %1}, r;\n\t}"
        : "=r"(r0), "=r"(r1)
        : "r"(a0), "r"(a1), "l"(b2));
}

// Four code bytes: byte j encodes (ze[j] / d, zo[j] / d), the even element
// in the low nibble, with y2 = (y, y), y = RN(1 / d), and nd2 = (-d, -d).
// Each quotient z / d, rounded to nearest even, comes from the rounded
// reciprocal: q0 = RN(z y), the residual r = z - q0 d (exact with one fused
// multiply-add), q1 = RN(q0 + r y).  Markstein's theorem (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990; also Muller et al., "Handbook of
// Floating-Point Arithmetic", on division from a correctly rounded
// reciprocal) makes q1 the correctly rounded quotient when no step
// underflows or overflows.  Here d is an e4m3 value (>= 2^-9) and a quotient
// small enough for the residual to underflow is far below 0.25, so its e2m1
// code is 0 either way; a quotient never overflows (d saturates at 448).
// The steps run two elements per packed fp32 instruction (each element
// rounded as the scalar instruction would), then the saturating e2m1
// conversions; -0 codes become +0 on all eight nibbles at once (a nibble
// keeps its sign bit only if its magnitude bits are not all zero).
__device__ __forceinline__ uint32_t nvfp4_code_quad(const uint32_t (&ze)[4],
                                                    const uint32_t (&zo)[4], uint64_t y2,
                                                    uint64_t nd2) {
    uint32_t out;
    asm("{\n\t.reg .b64 z, q0, r, q1;\n\t.reg .b32 l, h;\n\t.reg .b8 t0, t1, t2, t3;\n\t"
        "mov.b64 z, {%1, %2};\n\t"
        "mul.rn.f32x2 q0, z, %9;\n\t"
        "fma.rn.f32x2 r, q0, %10, z;\n\t"
        "fma.rn.f32x2 q1, r, %9, q0;\n\t"
        "mov.b64 {l, h}, q1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, h, l;\n\t"
        "mov.b64 z, {%3, %4};\n\t"
        "mul.rn.f32x2 q0, z, %9;\n\t"
        "fma.rn.f32x2 r, q0, %10, z;\n\t"
        "fma.rn.f32x2 q1, r, %9, q0;\n\t"
        "mov.b64 {l, h}, q1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, h, l;\n\t"
        "mov.b64 z, {%5, %6};\n\t"
        "mul.rn.f32x2 q0, z, %9;\n\t"
        "fma.rn.f32x2 r, q0, %10, z;\n\t"
        "fma.rn.f32x2 q1, r, %9, q0;\n\t"
        "mov.b64 {l, h}, q1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t2, h, l;\n\t"
        "mov.b64 z, {%7, %8};\n\t"
        "mul.rn.f32x2 q0, z, %9;\n\t"
        "fma.rn.f32x2 r, q0, %10, z;\n\t"
        "fma.rn.f32x2 q1, r, %9, q0;\n\t"
        "mov.b64 {l, h}, q1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t3, h, l;\n\t"
        "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
        : "=r"(out)
        : "r"(ze[0]), "r"(zo[0]), "r"(ze[1]), "r"(zo[1]), "r"(ze[2]), "r"(zo[2]), "r"(ze[3]),
          "r"(zo[3]), "l"(y2), "l"(nd2));
    const uint32_t mag = out & 0x77777777u;
    return mag | (out & ((mag + 0x77777777u) & 0x88888888u));
}

// Half a block for two cooperating lanes (lane pairs l, l ^ 1, all 32 lanes
// active): this lane's 8 bf16 values (one uint4), the partner's 8 complete
// the block.  Same steps and bits as nvfp4_quant_block16, the per-element
// arithmetic two elements per packed fp32 instruction; returns the scale
// byte and this lane's 4 code bytes (elements 8h .. 8h + 7 of the block).
__device__ __forceinline__ uint32_t nvfp4_quant_half8(const uint4& v, float q, uint32_t& codes) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint32_t qb = __float_as_uint(q);
    const uint64_t q2 = ((uint64_t)qb << 32) | qb;
    uint32_t ze[4], zo[4];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        mul2_rn(w[j] << 16, w[j] & 0xFFFF0000u, q2, ze[j], zo[j]);
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(ze[j])), fabsf(__uint_as_float(zo[j]))));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    float d;
    const uint32_t s = nvfp4_block_scale(amax, d);
    if (!(d > 0.f)) {
        codes = 0u;
        return s;
    }
    const uint32_t yb = __float_as_uint(__frcp_rn(d)), ndb = __float_as_uint(-d);
    codes = nvfp4_code_quad(ze, zo, ((uint64_t)yb << 32) | yb, ((uint64_t)ndb << 32) | ndb);
    return s;
}

// One 16-element block: bf16 values in v0 (elements 0..7) and v1 (8..15),
// two per 32-bit word, low half first; pre-scale q.  Returns the scale byte
// and leaves the 8 code bytes in codes.  The same steps and helpers as
// nvfp4_quant_half8, one thread per block.
__device__ __forceinline__ uint32_t nvfp4_quant_block16(const uint4& v0, const uint4& v1, float q,
                                                        uint2& codes) {
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    const uint32_t qb = __float_as_uint(q);
    const uint64_t q2 = ((uint64_t)qb << 32) | qb;
    uint32_t ze[2][4], zo[2][4];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        mul2_rn(w[j] << 16, w[j] & 0xFFFF0000u, q2, ze[j >> 2][j & 3], zo[j >> 2][j & 3]);
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(ze[j >> 2][j & 3])),
                                 fabsf(__uint_as_float(zo[j >> 2][j & 3]))));
    }
    float d;
    const uint32_t s = nvfp4_block_scale(amax, d);
    if (!(d > 0.f)) {
        codes = make_uint2(0u, 0u);
        return s;
    }
    const uint32_t yb = __float_as_uint(__frcp_rn(d)), ndb = __float_as_uint(-d);
    const uint64_t y2 = ((uint64_t)yb << 32) | yb, nd2 = ((uint64_t)ndb << 32) | ndb;
    codes = make_uint2(nvfp4_code_quad(ze[0], zo[0], y2, nd2), nvfp4_code_quad(ze[1], zo[1], y2, nd2));
    return s;
}

// Standalone encoder: x bf16 [R][L] row-major (L % 16 == 0), row r scaled by
// qscale[r / rows_per_scale]; codes u8 [R][L/2], sf u8 [R][L/16].  One thread
// per 16-element block: 32 bytes read, 9 written, blocks in row-major order
// so a warp's loads and stores are contiguous.
__global__ void __launch_bounds__(256) quantize_bf16_kernel(const __nv_bfloat16* __restrict__ x,
                                                            const float* __restrict__ qscale,
                                                            uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ sf, long long blocks,
                                                            int L, int rows_per_scale) {
    const int bpr = L >> 4;   // blocks per row
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < blocks;
         b += (long long)gridDim.x * blockDim.x) {
        const long long row = b / bpr;
        const float q = __ldg(qscale + row / rows_per_scale);
        const uint4* src = reinterpret_cast<const uint4*>(x) + 2 * b;
        uint2 c;
        const uint32_t s = nvfp4_quant_block16(__ldg(src), __ldg(src + 1), q, c);
        *reinterpret_cast<uint2*>(codes + 8 * b) = c;
        sf[b] = static_cast<uint8_t>(s);
    }
}

}  // namespace nvfp4gg
