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
// pair of weight rows (pairs grid-strided over all warps), every lane loading 16-byte
// chunks of the row (32 codes) with coalesced, evict-first loads; the tokens
// are staged once per CTA in shared memory as fp32, 32 values per K chunk
// padded to 36 (lanes read different chunks: rows 144 bytes apart keep the
// 16-byte loads of a warp free of bank conflicts).  Codes and scales are
// converted with CUDA's fp4 / fp8 conversion intrinsics; products are summed
// in fp32 per 16-element block and the block scale applied once; a warp
// reduction ends the row.  No tensor cores: two FLOPs per weight byte and a
// half cannot use them.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace nvfp4gg {

constexpr int kGemvMaxTokens = 8;
constexpr int kGemvThreads = 256;
constexpr int kGemvMaxSmem = 192 * 1024;   // tokens staged as fp32: M * (K / 32) * 144 bytes
constexpr int kGemvRow = 36;               // floats per staged 32-value chunk
constexpr int kGemvBatch = 4;              // chunks per lane and row loaded before use

// Two e2m1 codes (low nibble = even element) as floats.
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte) {
    const __half2 h = __half2(__nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>(byte), __NV_E2M1));
    return __half22float2(h);
}

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte), __NV_E4M3)));
}

// Sum over the 16 codes of words w0, w1 (8 codes each) times x[0..15]
// (16-byte aligned in shared memory).
__device__ __forceinline__ float block16(uint32_t w0, uint32_t w1, const float* xs) {
    const float4* x4 = reinterpret_cast<const float4*>(xs);
    float p = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t w = h ? w1 : w0;
        const float4 xa = x4[2 * h], xb = x4[2 * h + 1];
        const float2 c0 = e2m1x2_to_float2(w & 0xFFu), c1 = e2m1x2_to_float2((w >> 8) & 0xFFu);
        const float2 c2 = e2m1x2_to_float2((w >> 16) & 0xFFu), c3 = e2m1x2_to_float2(w >> 24);
        p = fmaf(c0.x, xa.x, p);
        p = fmaf(c0.y, xa.y, p);
        p = fmaf(c1.x, xa.z, p);
        p = fmaf(c1.y, xa.w, p);
        p = fmaf(c2.x, xb.x, p);
        p = fmaf(c2.y, xb.y, p);
        p = fmaf(c3.x, xb.z, p);
        p = fmaf(c3.y, xb.w, p);
    }
    return p;
}

template <int M>
__global__ void __launch_bounds__(kGemvThreads, 2)
gemv_w4a16_kernel(const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ B,
                  const uint8_t* __restrict__ B_sf, const float* __restrict__ alpha,
                  __nv_bfloat16* __restrict__ y, int N, int K) {
    extern __shared__ __align__(16) float xs[];   // [M][K/32][36] fp32
    const int chunks = K >> 5;                 // 16-byte chunks (32 codes) per row
    // stage the tokens: 8 bf16 per 16-byte load
    for (int i = threadIdx.x; i < (M * K) >> 3; i += blockDim.x) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x) + i);
        float* dst = xs + ((i << 3) >> 5) * kGemvRow + ((i << 3) & 31);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            dst[2 * j] = __uint_as_float(w[j] << 16);
            dst[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int warps = (int)((gridDim.x * blockDim.x) >> 5);
    const float al = __ldg(alpha);
    // each warp streams two rows at once (twice the loads in flight)
    for (int n0 = 2 * (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); n0 < N; n0 += 2 * warps) {
        const bool two = n0 + 1 < N;
        const int n1 = two ? n0 + 1 : n0;
        const uint4* row0 = reinterpret_cast<const uint4*>(B + (size_t)n0 * (K >> 1));
        const uint4* row1 = reinterpret_cast<const uint4*>(B + (size_t)n1 * (K >> 1));
        const uint16_t* srow0 = reinterpret_cast<const uint16_t*>(B_sf + (size_t)n0 * (K >> 4));
        const uint16_t* srow1 = reinterpret_cast<const uint16_t*>(B_sf + (size_t)n1 * (K >> 4));
        float acc0[M], acc1[M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc0[m] = acc1[m] = 0.f;
        // batches of kGemvBatch chunks per lane and row: all loads of a batch
        // are issued before any of its arithmetic
        for (int cb = lane; cb < chunks; cb += 32 * kGemvBatch) {
            uint4 q0[kGemvBatch], q1[kGemvBatch];
            uint32_t t0[kGemvBatch], t1[kGemvBatch];
#pragma unroll
            for (int u = 0; u < kGemvBatch; ++u) {
                const int c = cb + 32 * u;
                if (c < chunks) {
                    q0[u] = __ldcs(row0 + c);
                    q1[u] = __ldcs(row1 + c);
                    t0[u] = __ldcs(srow0 + c);
                    t1[u] = __ldcs(srow1 + c);
                }
            }
#pragma unroll
            for (int u = 0; u < kGemvBatch; ++u) {
                const int c = cb + 32 * u;
                if (c < chunks) {
                    const float s00 = e4m3_to_float(t0[u] & 0xFFu), s01 = e4m3_to_float(t0[u] >> 8);
                    const float s10 = e4m3_to_float(t1[u] & 0xFFu), s11 = e4m3_to_float(t1[u] >> 8);
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const float* xk = xs + (m * chunks + c) * kGemvRow;
                        acc0[m] = fmaf(block16(q0[u].x, q0[u].y, xk), s00, acc0[m]);
                        acc0[m] = fmaf(block16(q0[u].z, q0[u].w, xk + 16), s01, acc0[m]);
                        acc1[m] = fmaf(block16(q1[u].x, q1[u].y, xk), s10, acc1[m]);
                        acc1[m] = fmaf(block16(q1[u].z, q1[u].w, xk + 16), s11, acc1[m]);
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float v0 = acc0[m], v1 = acc1[m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                v0 += __shfl_xor_sync(0xffffffffu, v0, o);
                v1 += __shfl_xor_sync(0xffffffffu, v1, o);
            }
            if (lane == 0) {
                y[(size_t)m * N + n0] = __float2bfloat16_rn(al * v0);
                if (two) y[(size_t)m * N + n1] = __float2bfloat16_rn(al * v1);
            }
        }
    }
}

}  // namespace nvfp4gg
