// W4A16 GEMV for decode (M <= 8 tokens): NVFP4 weights, bf16 activations,
// the nvfp4_gemv workload (its W4A16 form) in the kernel table of the page
// listing Helion's pretuned_kernels directory, a one-token decode GEMV over
// model projection shapes.  For every token m < M and weight row n < N:
//
//     y[m][n] = bf16( alpha * sum_k x[m][k] * B[n][k] )
//
// where B[n][k] = e2m1 code times the e4m3 scale of its 16-element K block
// (raw row-major layout: codes [N][K/2], scales [N][K/16]) and x, y are bf16.
//
// Each weight byte is read once, so the kernel streams HBM: one warp per
// group of R weight rows (2 up to four tokens, else 1; groups grid-strided
// over all warps), every lane loading 16-byte chunks of the row (32 codes)
// with coalesced, evict-first loads.  The tokens are staged once per CTA in
// shared memory as f16 with a power-of-two factor per 16-element block: the
// block's largest value is moved to [2^14, 2^15), so every bf16 value down
// to 2^-31 of it is exact in f16 (8 significant bits) and only smaller ones,
// far below the fp32 accumulation error, are rounded.  32 values per K chunk
// are padded to 80 bytes (lanes read different chunks: rows 5 x 16 bytes
// apart keep the 16-byte loads of a warp free of bank conflicts).  Codes are
// converted with the hardware e2m1x2 -> f16x2 conversion and multiplied with
// mixed-precision FMAs (f16 factors, fp32 accumulator: the code-times-token
// product is exact), so no conversion to fp32 sits on the per-code path; at
// one token the instruction stream, not only HBM, bounds this kernel.  Block
// scale times token factor is applied once per 16 products; a warp reduction
// ends the row.  No tensor cores: two FLOPs per weight byte and a half cannot
// use them.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace nvfp4gg {

constexpr int kGemvMaxTokens = 8;
constexpr int kGemvThreads = 256;
constexpr int kGemvMaxSmem = 192 * 1024;   // staged tokens: 2.75 bytes per token value
constexpr int kGemvRowBytes = 80;          // 32 f16 tokens + 16 bytes of padding per K chunk
constexpr int kGemvBatch = 4;              // chunks per lane and row loaded before use

// shared memory of M staged tokens of K values: f16 chunks and block factors
inline long long gemv_smem_bytes(int M, int K) {
    return (long long)M * (K / 32) * kGemvRowBytes + (long long)M * (K / 16) * 4;
}

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3)));
}

// acc + sum over the 8 codes of word w (byte j: codes 2j, 2j+1, low nibble
// first) times the 8 f16 tokens in x01, x23, x45, x67 (two per register, low
// half first).  e2m1x2 -> f16x2 conversions, then mixed-precision FMAs with
// f16 factors and an fp32 accumulator: each product (at most 10 significant
// bits) is exact, one rounding per addition, no f16 -> f32 conversions.
__device__ __forceinline__ float dot8(uint32_t w, uint32_t x01, uint32_t x23, uint32_t x45,
                                      uint32_t x67, float acc) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        ".reg .b32 h0, h1, h2, h3;\n\t"
        ".reg .b16 c0, c1, c2, c3, c4, c5, c6, c7, y0, y1, y2, y3, y4, y5, y6, y7;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 h0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 h2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
        "mov.b32 {c0, c1}, h0;\n\tmov.b32 {c2, c3}, h1;\n\t"
        "mov.b32 {c4, c5}, h2;\n\tmov.b32 {c6, c7}, h3;\n\t"
        "mov.b32 {y0, y1}, %2;\n\tmov.b32 {y2, y3}, %3;\n\t"
        "mov.b32 {y4, y5}, %4;\n\tmov.b32 {y6, y7}, %5;\n\t"
        "fma.rn.f32.f16 %0, c0, y0, %0;\n\tfma.rn.f32.f16 %0, c1, y1, %0;\n\t"
        "fma.rn.f32.f16 %0, c2, y2, %0;\n\tfma.rn.f32.f16 %0, c3, y3, %0;\n\t"
        "fma.rn.f32.f16 %0, c4, y4, %0;\n\tfma.rn.f32.f16 %0, c5, y5, %0;\n\t"
        "fma.rn.f32.f16 %0, c6, y6, %0;\n\tfma.rn.f32.f16 %0, c7, y7, %0;\n\t}"
        : "+f"(acc)
        : "r"(w), "r"(x01), "r"(x23), "r"(x45), "r"(x67));
    return acc;
}

// Sum over the 16 codes of words w0, w1 times the 16 staged f16 tokens at xh
// (16-byte aligned: two 16-byte loads).
__device__ __forceinline__ float block16(uint32_t w0, uint32_t w1, const uint4* xh) {
    const uint4 xa = xh[0], xb = xh[1];
    float p = dot8(w0, xa.x, xa.y, xa.z, xa.w, 0.f);
    return dot8(w1, xb.x, xb.y, xb.z, xb.w, p);
}

// A warp's work is a sequence of items (row group, chunk batch): the loads of
// item i + 1 are issued before the arithmetic of item i, and the first
// item's loads before the tokens are staged, so loads and arithmetic overlap.
template <int R>
struct GemvBatch {
    uint4 q[kGemvBatch][R];
    uint32_t t[kGemvBatch][R];
};

template <int R>
__device__ __forceinline__ void gemv_load(GemvBatch<R>& b, const uint8_t* __restrict__ B,
                                          const uint8_t* __restrict__ B_sf, int n0, int N, int K,
                                          int c0, int chunks) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int n = n0 + r < N ? n0 + r : n0;   // past N: repeat row n0, not stored
        const uint4* row = reinterpret_cast<const uint4*>(B + (size_t)n * (K >> 1));
        const uint16_t* srow = reinterpret_cast<const uint16_t*>(B_sf + (size_t)n * (K >> 4));
#pragma unroll
        for (int u = 0; u < kGemvBatch; ++u) {
            const int c = c0 + 32 * u;
            if (c < chunks) {
                b.q[u][r] = __ldcs(row + c);
                b.t[u][r] = __ldcs(srow + c);
            }
        }
    }
}

template <int M, int R>
__global__ void __launch_bounds__(kGemvThreads, 2)
gemv_w4a16_kernel(const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ B,
                  const uint8_t* __restrict__ B_sf, const float* __restrict__ alpha,
                  __nv_bfloat16* __restrict__ y, int N, int K) {
    // tokens staged as f16 times 2^-e per 16-element block (e from the block's
    // largest exponent), 2^e kept beside it: [M][K/32] rows of 32 halves + 8
    // halves of padding (80 bytes), then [M][K/16] fp32 block factors
    extern __shared__ __align__(16) uint8_t gemv_smem[];
    const int chunks = K >> 5;                 // 16-byte chunks (32 codes) per row
    float* xf = reinterpret_cast<float*>(gemv_smem + (size_t)M * chunks * kGemvRowBytes);
    const int lane = threadIdx.x & 31;
    const int wid = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int warps = (int)((gridDim.x * blockDim.x) >> 5);
    const int groups = (N + R - 1) / R;
    const int nbat = (chunks + 32 * kGemvBatch - 1) / (32 * kGemvBatch);   // batches per row group
    const int mine = wid < groups ? (groups - 1 - wid) / warps + 1 : 0;    // row groups of this warp
    const int items = mine * nbat;
    GemvBatch<R> cur, nxt;
    if (items > 0) gemv_load<R>(cur, B, B_sf, R * wid, N, K, lane, chunks);
    for (int blk = threadIdx.x; blk < (M * K) >> 4; blk += blockDim.x) {
        const uint4* src = reinterpret_cast<const uint4*>(x) + 2 * blk;
        const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t emax = 0;   // largest biased exponent of the block
#pragma unroll
        for (int j = 0; j < 8; ++j)
            emax = max(emax, max((w[j] >> 7) & 0xFFu, (w[j] >> 23) & 0xFFu));
        // the largest value, in [2^(emax-127), 2^(emax-126)), goes to [2^14,
        // 2^15); blocks below 2^-111 (zero, subnormal) use e = -126 instead,
        // which keeps both factors normal fp32 powers of two
        const int e = max((int)emax - 141, -126);
        const float down = __uint_as_float((uint32_t)(127 - e) << 23);
        const float up = __uint_as_float((uint32_t)(127 + e) << 23);
        __half2 hv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            hv[j] = __floats2half2_rn(__uint_as_float(w[j] << 16) * down,
                                      __uint_as_float(w[j] & 0xFFFF0000u) * down);
        const int mrow = blk / (K >> 4), kb = blk - mrow * (K >> 4);   // token, 16-block
        uint4* dst = reinterpret_cast<uint4*>(gemv_smem + ((size_t)mrow * chunks + (kb >> 1)) * kGemvRowBytes +
                                              (kb & 1) * 32);
        dst[0] = make_uint4(*reinterpret_cast<uint32_t*>(&hv[0]), *reinterpret_cast<uint32_t*>(&hv[1]),
                            *reinterpret_cast<uint32_t*>(&hv[2]), *reinterpret_cast<uint32_t*>(&hv[3]));
        dst[1] = make_uint4(*reinterpret_cast<uint32_t*>(&hv[4]), *reinterpret_cast<uint32_t*>(&hv[5]),
                            *reinterpret_cast<uint32_t*>(&hv[6]), *reinterpret_cast<uint32_t*>(&hv[7]));
        xf[blk] = up;
    }
    __syncthreads();
    const float al = __ldg(alpha);
    float acc[R][M];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.f;
    for (int it = 0; it < items; ++it) {
        const int k = it / nbat, bat = it - k * nbat;
        const int n0 = R * (wid + k * warps);
        const int c0 = lane + 32 * kGemvBatch * bat;
        if (it + 1 < items) {
            const int k1 = (it + 1) / nbat, bat1 = (it + 1) - k1 * nbat;
            gemv_load<R>(nxt, B, B_sf, R * (wid + k1 * warps), N, K, lane + 32 * kGemvBatch * bat1, chunks);
        }
#pragma unroll
        for (int u = 0; u < kGemvBatch; ++u) {
            const int c = c0 + 32 * u;
            if (c < chunks) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float s0 = e4m3_to_float(cur.t[u][r] & 0xFFu), s1 = e4m3_to_float(cur.t[u][r] >> 8);
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const uint4* xk = reinterpret_cast<const uint4*>(
                            gemv_smem + ((size_t)m * chunks + c) * kGemvRowBytes);
                        const float2 f = *reinterpret_cast<const float2*>(xf + (size_t)m * (K >> 4) + 2 * c);
                        acc[r][m] = fmaf(block16(cur.q[u][r].x, cur.q[u][r].y, xk), s0 * f.x, acc[r][m]);
                        acc[r][m] = fmaf(block16(cur.q[u][r].z, cur.q[u][r].w, xk + 2), s1 * f.y, acc[r][m]);
                    }
                }
            }
        }
        if (bat == nbat - 1) {   // the row group is complete
#pragma unroll
            for (int r = 0; r < R; ++r) {
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    float v = acc[r][m];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0 && n0 + r < N) y[(size_t)m * N + n0 + r] = __float2bfloat16_rn(al * v);
                    acc[r][m] = 0.f;
                }
            }
        }
        cur = nxt;
    }
}

}  // namespace nvfp4gg
