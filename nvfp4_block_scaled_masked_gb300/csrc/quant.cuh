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
__device__ __forceinline__ uint32_t nvfp4_block_scale(float amax, float& d) {
    const float s = __fdiv_rn(amax, 6.0f);
    const uint32_t sf = __nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3);
    d = __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(sf), __NV_E4M3)));
    return sf;
}

// z / d rounded to nearest even, from y = RN(1 / d): q0 = RN(z y), the
// residual z - q0 d (exact with one fused multiply-add), q1 = RN(q0 + r y).
// Markstein's theorem (P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990; also
// Muller et al., "Handbook of Floating-Point Arithmetic", on division from a
// correctly rounded reciprocal) makes q1 the correctly rounded quotient when
// no step underflows or overflows.  Here d is an e4m3 value (>= 2^-9) and a
// quotient small enough for the residual to underflow is far below 0.25, so
// its e2m1 code is 0 either way; a quotient never overflows (d saturates at
// 448).  Three instructions per element instead of a full division.
__device__ __forceinline__ float div_rn_by_recip(float z, float d, float y) {
    const float q0 = __fmul_rn(z, y);
    const float r = __fmaf_rn(-q0, d, z);
    return __fmaf_rn(r, y, q0);
}

// One byte of two e2m1 codes: z_even / d in the low nibble, z_odd / d in the
// high one (y = RN(1 / d)); both +0 when d == 0.
__device__ __forceinline__ uint32_t nvfp4_code_pair(float z_even, float z_odd, float d, float y) {
    if (!(d > 0.f)) return 0u;
    const float lo = div_rn_by_recip(z_even, d, y), hi = div_rn_by_recip(z_odd, d, y);
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tmov.b16 %0, {t, 0};\n\t}"
        : "=h"(r)
        : "f"(lo), "f"(hi));
    uint32_t b = r & 0xFFu;
    if ((b & 0x07u) == 0) b &= 0xF0u;   // -0 -> +0
    if ((b & 0x70u) == 0) b &= 0x0Fu;
    return b;
}

// One 16-element block: bf16 values in v0 (elements 0..7) and v1 (8..15),
// two per 32-bit word, low half first; pre-scale q.  Returns the scale byte
// and leaves the 8 code bytes in codes.
__device__ __forceinline__ uint32_t nvfp4_quant_block16(const uint4& v0, const uint4& v1, float q,
                                                        uint2& codes) {
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float z[16];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        z[2 * j] = __fmul_rn(__uint_as_float(w[j] << 16), q);
        z[2 * j + 1] = __fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), q);
        amax = fmaxf(amax, fmaxf(fabsf(z[2 * j]), fabsf(z[2 * j + 1])));
    }
    float d;
    const uint32_t s = nvfp4_block_scale(amax, d);
    const float y = d > 0.f ? __frcp_rn(d) : 0.f;
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j)
        out[j >> 2] |= nvfp4_code_pair(z[2 * j], z[2 * j + 1], d, y) << (8 * (j & 3));
    codes = make_uint2(out[0], out[1]);
    return s;
}

// Half a block for two cooperating lanes (lane pairs l, l ^ 1, all 32 lanes
// active): this lane's 8 bf16 values (one uint4), the partner's 8 complete
// the block.  Same steps and bits as nvfp4_quant_block16; returns the scale
// byte and this lane's 4 code bytes (elements 8h .. 8h + 7 of the block).
__device__ __forceinline__ uint32_t nvfp4_quant_half8(const uint4& v, float q, uint32_t& codes) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float z[8];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        z[2 * j] = __fmul_rn(__uint_as_float(w[j] << 16), q);
        z[2 * j + 1] = __fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), q);
        amax = fmaxf(amax, fmaxf(fabsf(z[2 * j]), fabsf(z[2 * j + 1])));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    float d;
    const uint32_t s = nvfp4_block_scale(amax, d);
    const float y = d > 0.f ? __frcp_rn(d) : 0.f;
    uint32_t out = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) out |= nvfp4_code_pair(z[2 * j], z[2 * j + 1], d, y) << (8 * j);
    codes = out;
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
