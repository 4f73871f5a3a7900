// Persistent, warp-specialised tcgen05 kernel for the masked, block-scaled
// NVFP4 grouped GEMM-NT (FlashInfer's grouped_gemm_nt_masked as described on
// "The CuteDSL Gamble: Chasing Kernel Efficiency on Blackwell GPUs", "The
// Message": per expert g and row m < masked_m[g],
// C[g][m][n] = bf16(alpha[g] * sum_k A[g][m][k] B[g][n][k])).
//
// Orientation ("swap-AB"): the MMA's M = 128 rows are weight rows n (B), its
// N dimension is a tile of tokens m (A) whose width w is chosen per expert at
// run time (a multiple of 16, up to TT_MAX).  So the weight stream fills the
// 128-row tensor-core tile even for decode-sized masked_m, and a ragged
// masked_m wastes at most 15 token columns per tile.
//
// Roles (352 threads).  An asynchronous instruction (TMA copy, mbarrier
// operation, tcgen05 copy/MMA/commit) occupies its issuing thread for tens of
// cycles (hundreds under load), so the per-stage work is spread over several
// issuing threads:
//   warp 0      weight producer (one lane): bulk copies of the stage's
//               weight tiles (16 KB per 256-code K-tile, KSUB K-tiles per
//               stage, contiguous in the prepared layout) and their scale
//               atoms (2 KB per K-tile) into the shared ring.
//   warp 1      TMEM owner; MMA warp: walks the stages as a warp, one
//               elected lane issues 4 x tcgen05.mma (K = 64 each) per K-tile
//               and the commit of the stage back to the producers.
//   warp 2      token producer (one lane): per K-tile one tiled TMA for the
//               w token rows and one for their scale rows (a tensor map per
//               width w).
//   warps 3, 4, 9, 10  scale warps, one per TMEM lane quarter: every stage,
//               each lane loads its scale words from shared memory and the
//               warp writes them into its quarter with tcgen05.st (no
//               tcgen05.cp: one thread issuing a dozen copies per stage was
//               measured to be the bound of compute-bound tiles).
//   warps 5..8  epilogue: tcgen05.ld of the fp32 accumulator (lane = n,
//               column = token), x alpha[g], bf16 round-to-nearest, a per-warp
//               shared-memory transpose, 16-byte stores of rows m < masked_m[g].
// Tiles are walked persistently: CTA b takes tiles b, b + grid, ...; the
// tile list holds, per expert in order, ceil(N/128) weight blocks times the
// token tiles of that expert, and experts with masked_m = 0 contribute none.
//
// Scale factors in TMEM: the MMA reads the scale of operand row r from TMEM
// lane r % 32 (every lane quarter holds the same words), column
// base + r / 32, byte = 16-element K block; the base must be a multiple of 4
// columns.  So lane i, column base + c holds the 4 scale bytes of one K chunk
// of 64 for row 32c + i: for the weights that is word c of row i of a
// 512-byte atom of the prepared scales, for the tokens word (K chunk) of the
// plain scale row 32c + i loaded by TMA.
//
// Every wait on an mbarrier is bounded (time limit in the parameters); on
// expiry the waiter records NVFP4GG_ERR_TIMEOUT in the error word, raises a
// shared abort flag that makes the other roles stop, in-flight copies and
// MMAs are drained with bounded waits, TMEM is freed and the kernel returns.
#pragma once
#include <cuda_bf16.h>
#include "ptx.cuh"
#include "quant.cuh"
#include "nvfp4gg.h"

namespace nvfp4gg {

constexpr int kGroupsMax = NVFP4GG_MAX_GROUPS;
constexpr int kThreads = 352;
constexpr int kMaxWidths = 16;   // token tile widths 16, 32, ..., 256 rows

// Scalar arguments of every GEMM kernel.
struct GemmArgs {
    const uint8_t* wq;               // prepared codes: [G][NT][K/256][16384], pre-swizzled tiles
    const uint8_t* wsf;              // prepared scales: [G][NT][K/64][512]
    const float* alpha;
    const int* masked_m;
    __nv_bfloat16* C;
    int* err;
    int G, M_max, N, K, NT, KS;
    unsigned long long timeout_ns;
    // split-K (decode kernel): each tile's K stages are cut into `split`
    // contiguous ranges computed by different CTAs; with split > 1 every range
    // leaves an fp32 partial in ws_part[(tile*split + range)][TT_MAX][128] and
    // the last range to finish (counter ws_cnt[tile]) sums them in range order
    int split;
    float* ws_part;
    unsigned long long* ws_cnt;
    // split-K within a thread-block cluster (csplit != 0, split <= 8): the
    // grid is a multiple of split, cluster rank = K range, and the ranges of
    // a tile reduce through distributed shared memory (no workspace)
    int csplit;
    // per-expert completion signals (null: none): signals[g] is incremented
    // once per call after all of expert g's valid rows of C are stored;
    // sig_cnt[G] counts finished tile parts
    int* signals;
    unsigned long long* sig_cnt;
    // a number unique to this call (never 0): arrival counters are tagged
    // with it, so they need no clearing between calls (epoch_arrive)
    unsigned long long epoch;
    // packed-rows layout (contiguous != 0): A, A_sf and C hold only valid
    // rows, expert g's from row off[g] = sum_{h<g} masked_m[h], M_total rows
    // in all; token tensor maps are over [M_total] rows with one group
    int contiguous;
    int M_total;
    // SwiGLU epilogue only: also encode the bf16 output as NVFP4 for GEMM2
    // (qa non-null): codes qa [G][M_max][N/4], scales qsf [G][M_max][N/32],
    // expert g pre-scaled by qscale[g]; C may then be null (no bf16 store)
    uint8_t* qa;
    uint8_t* qsf;
    const float* qscale;
};

// Kernel parameters: the scalars and the token tensor maps of NW tile widths,
// tm_a[i] / tm_asf[i] for 16 (i + 1) rows (the host picks which widths a
// kernel variant can address).  Only these travel with a launch: a parameter
// block of 32 maps (4 KB) was measured to add about a microsecond to every
// call's launch.
template <int NW>
struct GemmParams : GemmArgs {
    CUtensorMap tm_a[NW];    // A codes u8 [G][M_max][K/2], box 128 x rows, SW128
    CUtensorMap tm_asf[NW];  // A_sf u8 [G][M_max][K/16], box 16 x rows
};

// Row of C holding token `tok` of expert g: g * M_max + tok in the masked
// layout; off[g] + tok in the packed-rows layout, -1 past its M_total rows.
__device__ __forceinline__ long long out_row(const GemmArgs& p, const int* off, int g, int tok) {
    if (!p.contiguous) return (long long)g * p.M_max + tok;
    const int r = off[g] + tok;
    return r < p.M_total ? r : -1;
}

// K stages [kb, ke) of split range sp of S over KS stages (balanced;
// S <= 16 and KS <= 4096, so 32-bit products suffice).  The unsplit call
// takes no division: it sits on the path to each CTA's first weight copy.
__device__ __forceinline__ void k_range(int sp, int S, int KS, int& kb, int& ke) {
    if (S == 1) {
        kb = 0;
        ke = KS;
        return;
    }
    kb = (sp * KS) / S;
    ke = ((sp + 1) * KS) / S;
}

__host__ __device__ constexpr int pow2_cols(int n) {
    return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512;
}

// A ring stage holds KSUB K-tiles of 256 codes.  Every stage costs a fixed
// few hundred nanoseconds of barrier hand-offs (producer, scale warps, MMA
// warp) whatever its size, so when few CTAs share the weight stream the
// bytes per stage set each SM's share of it: two K-tiles per stage move
// twice the bytes per hand-off.
template <int TT_MAX, int STAGES, int KSUB = 1>
struct KCfg {
    static_assert(TT_MAX % 32 == 0 && TT_MAX <= 256, "token tile");
    static_assert(STAGES >= 3 || (KSUB > 1 && STAGES >= 2), "ring depth");
    static_assert(KSUB == 1 || KSUB == 2, "K-tiles per stage");
    static constexpr int W_TILE = 128 * 128;         // one K-tile: 128 weight rows x 256 codes
    static constexpr int T_TILE = TT_MAX * 128;      // one K-tile: TT_MAX token rows x 256 codes
    static constexpr int WSF_TILE = 4 * 512;         // one K-tile: 4 weight-scale atoms
    static constexpr int TSF_PLAIN = TT_MAX * 16;    // one K-tile: token scales, 16 bytes per row
    static constexpr int W_STAGE = KSUB * W_TILE;
    static constexpr int T_STAGE = KSUB * T_TILE;
    static constexpr int WSF_STAGE = KSUB * WSF_TILE;
    static constexpr int TSF_STAGE = KSUB * TSF_PLAIN;
    static constexpr int NA = (TT_MAX + 127) / 128;  // 128-row token groups per MMA
    static constexpr int ACC_BUFS = 2;
    static constexpr int SFW_COLS = 16 * KSUB;       // 4 MMAs x 4 columns per K-tile
    static constexpr int SFT_COLS = 16 * NA * KSUB;
    static constexpr int SF_COLS = SFW_COLS + SFT_COLS;
    // Scale-factor TMEM regions, used round-robin by stage count.  With one
    // region per ring stage a region is rewritten only after the stage's next
    // full barrier, i.e. after the MMAs that read it completed.  Where TMEM
    // holds fewer (wide token tiles), the scale warps wait for those MMAs
    // (the empty barrier of the stage that last used the region).
    static constexpr int SF_FIT = (512 - ACC_BUFS * TT_MAX) / SF_COLS;
    static constexpr int SF_BUFS = SF_FIT < STAGES ? SF_FIT : STAGES;
    static_assert(SF_BUFS >= 2, "TMEM budget");
    static constexpr int TMEM_NEED = ACC_BUFS * TT_MAX + SF_BUFS * SF_COLS;
    // Scale-factor operands of tcgen05.mma are addressed in groups of 4 TMEM
    // columns: every scale address below is a multiple of 4 columns.
    static_assert(TT_MAX % 4 == 0 && SF_COLS % 4 == 0 && SFW_COLS % 4 == 0, "SF alignment");
    static_assert(TMEM_NEED <= 512, "TMEM budget");
    static constexpr int TMEM_COLS = pow2_cols(TMEM_NEED);

    static constexpr int OFF_W = 0;
    static constexpr int OFF_T = OFF_W + STAGES * W_STAGE;
    static constexpr int OFF_WSF = OFF_T + STAGES * T_STAGE;
    static constexpr int OFF_TSFP = OFF_WSF + STAGES * WSF_STAGE;
    static constexpr int OFF_EPI = OFF_TSFP + STAGES * TSF_STAGE;   // 4 warps x 16 tokens x 32 n bf16
    static constexpr int EPI_BYTES = 4 * 16 * 32 * 2;
    // cluster split-K (decode tiles): this K range's fp32 partial,
    // [TT_MAX tokens][128 weight rows], read by the cluster's CTAs
    static constexpr int PART_BYTES = TT_MAX <= 32 ? TT_MAX * 128 * 4 : 0;
    static constexpr int OFF_PART = OFF_EPI + EPI_BYTES;
    static constexpr int OFF_BAR = OFF_PART + PART_BYTES;
    // full, sfull, empty, sfready per stage; acc full/empty per buffer; MMA
    // drain; cluster split-K: partials ready, partials read
    static constexpr int NUM_BARS = 4 * STAGES + 2 * ACC_BUFS + 3;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_TAB = (OFF_MISC + 16 + 15) & ~15;
    // cum[kGroupsMax + 1] (tile prefix), gm[kGroupsMax] (clamped masked_m),
    // off[kGroupsMax + 1] (row prefix, packed-rows layout)
    static constexpr int TAB_BYTES = (3 * kGroupsMax + 2) * 4;
    static constexpr int SMEM_BYTES = OFF_TAB + TAB_BYTES + 1024;   // + alignment slack
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(OFF_T % 1024 == 0 && T_TILE % 1024 == 0, "128-byte swizzle alignment");
};

// Barrier among `threads` threads (whole warps) on hardware barrier `id`.
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void record_error(int* err, int code) {
    atomicCAS(err, 0, code);
}

// Bounded wait for the phase of `bar` with parity `parity`.  Gives up when
// the shared abort flag is raised by another role, or after timeout_ns, in
// which case it records the timeout and raises the flag itself.  Between
// checks the thread sleeps in try_wait (woken when the phase completes), so
// waiting warps leave the issue slots to the working ones.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, int* err,
                                             unsigned long long timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
        if ((it & 31u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                record_error(err, NVFP4GG_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// wait_bounded for a barrier that CTAs of the cluster arrive on with
// release: the completed phase is observed with a cluster-scope acquire.
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                     volatile int* abort_flag, int* err,
                                                     unsigned long long timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster_sleep(bar, parity, 1000u)) return true;
        if ((it & 31u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                record_error(err, NVFP4GG_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

struct TileCoord {
    int g, nt, t0, w, m;
};

template <int TT_MAX>
__device__ __forceinline__ int token_tiles(int m);

// Arrival on a counter shared by the CTAs of one call, without clearing it
// between calls: the counter holds epoch * span + arrivals, and the first
// arrival of a call finds another epoch's value (an earlier call's, or
// whatever the memory held) and restarts the count.  Returns this arrival's
// number (1-based).  A lock-free CAS loop: a retry means another arrival
// succeeded, and a call has at most `span` - 1 arrivals per counter.
__device__ __forceinline__ unsigned long long epoch_arrive(unsigned long long* c,
                                                           unsigned long long epoch,
                                                           unsigned long long span) {
    const unsigned long long base = epoch * span;
    unsigned long long seen = *reinterpret_cast<volatile unsigned long long*>(c);
    for (;;) {
        const unsigned long long next = (seen >= base && seen - base < span) ? seen + 1 : base + 1;
        const unsigned long long prev = atomicCAS(c, seen, next);
        if (prev == seen) return next - base;
        seen = prev;
    }
}

// After one epilogue warp stored its part of a tile of expert tc.g: count the
// part; the last of the expert's 4 x (tiles) parts increments the expert's
// signal.  Each lane fences its own stores first.
template <int TT_MAX>
__device__ __forceinline__ void signal_tile_part(const GemmArgs& p, const TileCoord& tc, int lane) {
    if (!p.signals) return;
    __threadfence();
    __syncwarp();
    if (lane == 0) {
        const unsigned long long parts = 4ull * token_tiles<TT_MAX>(tc.m) * p.NT;
        if (epoch_arrive(p.sig_cnt + tc.g, p.epoch, 1ull << 32) == parts) {
            __threadfence();
            atomicAdd(p.signals + tc.g, 1);
        }
    }
}

// Token tiles of an expert with m valid rows: ntt = ceil(m / TT_MAX) tiles of
// equal width w = ceil(m / ntt) rounded up to 16 (the MMA's N granularity).
template <int TT_MAX>
__device__ __forceinline__ int token_tiles(int m) { return (m + TT_MAX - 1) / TT_MAX; }
__device__ __forceinline__ int token_width(int m, int ntt) {
    return ntt ? (((m + ntt - 1) / ntt + 15) & ~15) : 0;
}

// Tile id -> (expert, weight block, first token, token width, masked_m).
template <int TT_MAX>
__device__ __forceinline__ TileCoord decode_tile(const int* cum, const int* gm, int G, int tile) {
    int lo = 0, hi = G - 1;   // the last g with cum[g] <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    TileCoord c;
    c.g = lo;
    c.m = gm[lo];
    const int local = tile - cum[lo];
    const int ntt = token_tiles<TT_MAX>(c.m);
    if (ntt == 1) {   // the common decode case: no divisions
        c.w = (c.m + 15) & ~15;
        c.nt = local;
        c.t0 = 0;
        return c;
    }
    c.w = token_width(c.m, ntt);
    c.nt = local / ntt;
    c.t0 = (local - c.nt * ntt) * c.w;
    return c;
}

// The SwiGLU epilogue of one tile on the swap-AB kernels (TMEM lane = prepared
// weight row, column = token): 16-token chunks; lane l < 16 combines its
// h_gate = alpha * acc with lane l + 16's h_up into silu(h_gate) * h_up for
// output column 64 * block + 16 * quad + l, where `block` is the tile's
// 128-row weight block; the [16 tokens][16 columns] bf16 chunk is staged in
// `stage_buf` (512 bytes) and stored, and with qa set lane t < 16 also
// encodes token t's 16 columns as one NVFP4 block of GEMM2's K.
// silu(g) u = g u / (1 + exp(-g)) for two (g, u) pairs, two elements per
// packed fp32 instruction where the arithmetic allows: exp(-g) as
// 2^(-g log2 e) from the approximate base-2 exponential, the quotient
// through the approximate reciprocal (the SwiGLU output is held to the
// GEMM's tolerance, not to a correctly rounded result), both flushing
// subnormal results to zero (an exponential below 2^-126 leaves 1 + e at 1;
// a reciprocal below 2^-126 leaves y far under the tolerance).  For
// g -> -inf the denominator overflows and the reciprocal gives 0.
__device__ __forceinline__ void silu_mul2(float ga, float gb, float ua, float ub, float& ya,
                                          float& yb) {
    const uint64_t neg_log2e2 = 0xBFB8AA3BBFB8AA3Bull;   // (-log2 e, -log2 e)
    const uint64_t one2 = 0x3F8000003F800000ull;         // (1, 1)
    asm("{\n\t.reg .b64 g, u, t, e, d, n, y;\n\t.reg .b32 ta, tb, ea, eb, ra, rb;\n\t"
        "mov.b64 g, {%2, %3};\n\t"
        "mov.b64 u, {%4, %5};\n\t"
        "mul.rn.f32x2 t, g, %6;\n\t"
        "mov.b64 {ta, tb}, t;\n\t"
        "ex2.approx.ftz.f32 ea, ta;\n\t"
        "ex2.approx.ftz.f32 eb, tb;\n\t"
        "mov.b64 e, {ea, eb};\n\t"
        "add.rn.f32x2 d, e, %7;\n\t"
        "mov.b64 {ta, tb}, d;\n\t"
        "rcp.approx.ftz.f32 ra, ta;\n\t"
        "rcp.approx.ftz.f32 rb, tb;\n\t"
        "mul.rn.f32x2 n, g, u;\n\t"
        "mov.b64 d, {ra, rb};\n\t"
        "mul.rn.f32x2 y, n, d;\n\t"
        "mov.b64 {%0, %1}, y;\n\t}"
        : "=f"(ya), "=f"(yb)
        : "f"(ga), "f"(gb), "f"(ua), "f"(ub), "l"(neg_log2e2), "l"(one2));
}

template <int TT_MAX>
__device__ __forceinline__ void swiglu_tile_store(const GemmArgs& p, const int* off,
                                                  const TileCoord& tc, uint32_t tbase, int block,
                                                  int quad, int lane, float al,
                                                  uint8_t* stage_buf) {
    const int NO = p.N >> 1;
    const int oc0 = block * 64 + quad * 16;
    const int t_end = min(tc.t0 + tc.w, tc.m);
    const bool quant = p.qa != nullptr;
    const float qs = quant ? __ldg(p.qscale + tc.g) : 0.f;
    const uint64_t al2 = ((uint64_t)__float_as_uint(al) << 32) | __float_as_uint(al);
    __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(stage_buf);
#pragma unroll 1
    for (int c = 0; c < TT_MAX / 16; ++c) {
        if (c * 16 >= tc.w) break;
        uint32_t r[16];
        tmem_ld_32x32b_x16(tbase + c * 16, r);
        tmem_wait_ld();
        // all 32 lanes compute: lane l < 16 token 2j of column l (its own
        // gate, lane l + 16's up), lane l + 16 token 2j + 1 of the same
        // column (lane l's gate, its own up)
        const bool lo = lane < 16;
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            float gate[2], up[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                uint32_t h0b, h1b;
                mul2_rn(r[2 * (j + k)], r[2 * (j + k) + 1], al2, h0b, h1b);   // x alpha
                const float h0 = __uint_as_float(h0b), h1 = __uint_as_float(h1b);
                const float p0 = __shfl_xor_sync(0xffffffffu, h0, 16);
                const float p1 = __shfl_xor_sync(0xffffffffu, h1, 16);
                gate[k] = lo ? h0 : p1;
                up[k] = lo ? p0 : h1;
            }
            float y0, y1;
            silu_mul2(gate[0], gate[1], up[0], up[1], y0, y1);
            sb[(2 * j + (lo ? 0 : 1)) * 16 + (lane & 15)] = __float2bfloat16_rn(y0);
            sb[(2 * j + 2 + (lo ? 0 : 1)) * 16 + (lane & 15)] = __float2bfloat16_rn(y1);
        }
        __syncwarp();
        const int t = lane >> 1, hh = lane & 1;
        const int tok = tc.t0 + c * 16 + t;
        const uint4 v = *reinterpret_cast<const uint4*>(stage_buf + t * 32 + hh * 16);
        const long long row = out_row(p, off, tc.g, tok);
        if (p.C && tok < t_end && oc0 < NO && row >= 0)
            *reinterpret_cast<uint4*>(p.C + row * NO + oc0 + 8 * hh) = v;
        if (quant) {
            // lanes 2t, 2t + 1: the two halves of token t's block (the
            // 16-byte piece this lane just stored)
            uint32_t qc;
            const uint32_t qsb = nvfp4_quant_half8(v, qs, qc);
            if (tok < t_end && oc0 < NO && row >= 0) {
                *reinterpret_cast<uint32_t*>(p.qa + row * (NO >> 1) + (oc0 >> 1) + 4 * hh) = qc;
                if (hh == 0) p.qsf[row * (NO >> 4) + (oc0 >> 4)] = static_cast<uint8_t>(qsb);
            }
        }
        __syncwarp();
    }
}

// SWIGLU: the fused GEMM1 epilogue.  The weights are prepared with gate and
// up rows interleaved (nvfp4_prepare_weights_swiglu): in each 32-row lane
// quarter of a 128-row block, rows 0..15 are gate rows and rows 16..31 the
// up rows of the same 16 output columns.  Lane l < 16 then combines its
// h_gate = alpha * acc with lane l + 16's h_up into silu(h_gate) * h_up, and
// C is bf16 [G][M_max][N/2], output column = 64 * block + 16 * quarter + l.
template <int TT_MAX, int STAGES, bool SWIGLU = false, int KSUB = 1>
__global__ void __launch_bounds__(kThreads, 1)
gemm_nt_masked_kernel(const __grid_constant__ GemmParams<TT_MAX / 16> p) {
    using Cfg = KCfg<TT_MAX, STAGES, KSUB>;
    // ring stages per tile: K-tiles of 256 codes, KSUB per stage (the host
    // picks KSUB = 2 only where it divides K / 256)
    const int KSS = p.KS / KSUB;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Decode tiles: the first weight stages of this CTA's first unit are
    // requested into L2 at once, before masked_m and the tile tables (a
    // couple of microseconds) are known.  The unit is guessed as if every
    // expert held one token tile (an unsplit decode call with no empty
    // expert: then exact); a wrong guess only warms other weights.
    if (TT_MAX <= 32 && warp == 0 && lane == 0) {
        const int tile = blockIdx.x / p.split;
        const int g = tile / p.NT;
        if (g < p.G) {
            int kb, ke;
            k_range(blockIdx.x - tile * p.split, p.split, KSS, kb, ke);
            const size_t wtile = ((size_t)g * p.NT + (tile - g * p.NT)) * (size_t)p.KS;
            const uint8_t* src = p.wq + wtile * Cfg::W_TILE + (size_t)kb * Cfg::W_STAGE;
            const int n = min(ke - kb, STAGES);
            prefetch_l2_bulk(src, (uint32_t)n * Cfg::W_STAGE);
        }
    }

    const uint32_t bar_full = base + Cfg::OFF_BAR;               // operand tiles: 2 producers + bytes
    const uint32_t bar_sfull = bar_full + 8 * STAGES;            // scale rows: 2 producers + bytes
    const uint32_t bar_empty = bar_sfull + 8 * STAGES;           // MMA commit
    const uint32_t bar_sfready = bar_empty + 8 * STAGES;         // 4 scale warps
    const uint32_t bar_accf = bar_sfready + 8 * STAGES;          // MMA commit, last stage
    const uint32_t bar_acce = bar_accf + 8 * Cfg::ACC_BUFS;      // 4 epilogue warps
    const uint32_t bar_done = bar_acce + 8 * Cfg::ACC_BUFS;      // MMA thread's drain
    const uint32_t bar_pready = bar_done + 8;                    // cluster split-K: partials stored
    const uint32_t bar_pfree = bar_pready + 8;                   // cluster split-K: partials read
    uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + Cfg::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    volatile int* epi_flag = reinterpret_cast<volatile int*>(misc + 2);   // split-K: last range
    volatile int* epi_stop = reinterpret_cast<volatile int*>(misc + 3);   // split-K: leave the loop
    int* cum = reinterpret_cast<int*>(sbase + Cfg::OFF_TAB);
    int* gm = cum + kGroupsMax + 1;
    int* off = gm + kGroupsMax;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 2);
            mbar_init(bar_sfull + 8 * s, 2);
            mbar_init(bar_empty + 8 * s, 1);
            mbar_init(bar_sfready + 8 * s, 4);
        }
        for (int b = 0; b < Cfg::ACC_BUFS; ++b) {
            mbar_init(bar_accf + 8 * b, 1);
            mbar_init(bar_acce + 8 * b, 4);
        }
        mbar_init(bar_done, 1);
        // every CTA of the cluster arrives once per tile on each
        mbar_init(bar_pready, p.csplit ? p.split : 1);
        mbar_init(bar_pfree, p.csplit ? p.split : 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(base + Cfg::OFF_MISC, Cfg::TMEM_COLS);
        tmem_relinquish();   // this CTA allocates nothing else: let others allocate
    }
    if (warp == 2 && lane == 0) {
        for (int i = 0; i < TT_MAX / 16; ++i) {
            prefetch_tmap(&p.tm_a[i]);
            prefetch_tmap(&p.tm_asf[i]);
        }
    }

    // Per-expert tables: valid rows (clamped), then the exclusive prefix of
    // tile counts (token tiles x weight blocks per expert).
    for (int g = threadIdx.x; g < p.G; g += kThreads) {
        int m = __ldg(p.masked_m + g);
        if (m < 0 || m > p.M_max) {
            record_error(p.err, NVFP4GG_ERR_MASK);
            m = m < 0 ? 0 : p.M_max;
        }
        gm[g] = m;
        // an expert without valid rows is complete from the start
        if (p.signals && m == 0 && blockIdx.x == 0) atomicAdd(p.signals + g, 1);
    }
    __syncthreads();
    // cluster split-K: every CTA's barriers are initialised before any CTA
    // of the cluster arrives on them.  Every thread arrives here; only the
    // epilogue warps, which arrive remotely, wait at once (their first
    // remote arrive is microseconds away), the others at the kernel's end.
    // Thread 0 published the initialisation with fence.mbarrier_init, so a
    // relaxed arrive suffices.
    if (p.csplit) cluster_arrive_relaxed();
    if (warp == 0) {
        // Both prefixes in one pass: tile counts (the tile list) and valid
        // rows (row offsets of the packed-rows layout).  It sits on the path
        // to every CTA's first weight copy: the two shuffle chains run side
        // by side and each parameter is read once.
        const int G = p.G, NT = p.NT;
        const int per = (G + 31) / 32;
        const int lo = lane * per;
        const int hi = min(G, lo + per);
        int sum = 0, rs = 0;
        for (int g = lo; g < hi; ++g) {
            const int m = gm[g];
            sum += token_tiles<TT_MAX>(m) * NT;
            rs += m;
        }
        int incl = sum, rincl = rs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            const int w = __shfl_up_sync(0xffffffffu, rincl, o);
            if (lane >= o) {
                incl += v;
                rincl += w;
            }
        }
        int run = incl - sum, rrun = rincl - rs;
        for (int g = lo; g < hi; ++g) {
            const int m = gm[g];
            cum[g] = run;
            off[g] = rrun;
            run += token_tiles<TT_MAX>(m) * NT;
            rrun += m;
        }
        if (lane == 31) {
            cum[G] = incl;
            off[G] = rincl;
            if (p.contiguous && rincl > p.M_total) record_error(p.err, NVFP4GG_ERR_MASK);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const int total = cum[p.G];
    const int units = total * p.split;   // (tile, K range) work units
    // TMEM map: accumulators [0, ACC_BUFS*TT_MAX), then SF_BUFS regions of 16
    // weight-scale + 16*NA token-scale columns
    const uint32_t tmem_sf = tmem + Cfg::ACC_BUFS * TT_MAX;

    if (warp == 0 || warp == 2) {
        // ------------------------------------------- producers (weights / tokens)
        // As the MMA warp: the warp walks the stages, the elected lane issues.
        const bool weights = warp == 0;
        const uint64_t pol_stream = policy_evict_first();
        int s = 0;
        uint32_t ph = 0;
        long long issued = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const int tile = p.split == 1 ? u : u / p.split;
            int kb, ke;
            k_range(u - tile * p.split, p.split, KSS, kb, ke);
            const TileCoord tc = decode_tile<TT_MAX>(cum, gm, p.G, tile);
            const size_t wtile = ((size_t)tc.g * p.NT + tc.nt) * (size_t)p.KS;
            const uint8_t* wq_tile = p.wq + wtile * Cfg::W_TILE;
            const uint8_t* wsf_tile = p.wsf + wtile * Cfg::WSF_TILE;
            const int box = (tc.w >> 4) - 1;   // tensor map of this token width
            for (int ks = kb; ks < ke; ++ks) {
                ok = __all_sync(0xffffffffu, wait_bounded(bar_empty + 8 * s, ph ^ 1u, abort_flag,
                                                          p.err, p.timeout_ns));
                if (!ok) break;
                // scales first (small: the scale warps start on them while the
                // operand tiles are still in flight), then the operand tile
                const uint32_t fb = bar_full + 8 * s;
                const uint32_t sb = bar_sfull + 8 * s;
                // (the stage's KSUB K-tiles of weights and of their scale
                // atoms are contiguous in the prepared layout: one copy each)
                if (!elect_one()) {
                } else if (weights) {
                    mbar_arrive_expect_tx(sb, Cfg::WSF_STAGE);
                    bulk_load_hint(base + Cfg::OFF_WSF + s * Cfg::WSF_STAGE,
                                   wsf_tile + (size_t)ks * Cfg::WSF_STAGE, Cfg::WSF_STAGE, sb,
                                   pol_stream);
                    mbar_arrive_expect_tx(fb, Cfg::W_STAGE);
                    bulk_load_hint(base + Cfg::OFF_W + s * Cfg::W_STAGE,
                                   wq_tile + (size_t)ks * Cfg::W_STAGE, Cfg::W_STAGE, fb, pol_stream);
                } else {
                    mbar_arrive_expect_tx(sb, tc.w * 16 * KSUB);
                    mbar_arrive_expect_tx(fb, tc.w * 128 * KSUB);
                    const int ty = p.contiguous ? off[tc.g] + tc.t0 : tc.t0;
                    const int tz = p.contiguous ? 0 : tc.g;
#pragma unroll
                    for (int i = 0; i < KSUB; ++i) {
                        const int kt = ks * KSUB + i;   // K-tile
                        tma_load_3d(base + Cfg::OFF_TSFP + s * Cfg::TSF_STAGE + i * Cfg::TSF_PLAIN,
                                    &p.tm_asf[box], sb, kt * 16, ty, tz);
                        tma_load_3d(base + Cfg::OFF_T + s * Cfg::T_STAGE + i * Cfg::T_TILE,
                                    &p.tm_a[box], fb, kt * 128, ty, tz);
                    }
                }
                __syncwarp();
                ++issued;
                if (++s == STAGES) { s = 0; ph ^= 1u; }
            }
        }
        // Drain: every stage's last issued copy must have landed before the
        // CTA may exit (normally already consumed; bounded on abort).
        for (int st = 0; st < STAGES; ++st) {
            if (st >= issued) break;
            const long long last = st + (long long)STAGES * ((issued - 1 - st) / STAGES);
            const uint32_t par = (uint32_t)((last / STAGES) & 1);
            volatile int no_abort = 0;
            wait_bounded(bar_full + 8 * st, par, &no_abort, p.err, p.timeout_ns);
            wait_bounded(bar_sfull + 8 * st, par, &no_abort, p.err, p.timeout_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA warp
        // All 32 lanes walk the loop, so every operand is warp-uniform; the
        // elected lane issues the MMAs and the commits that track them.
        int s = 0;
        uint32_t ph = 0;
        int r = 0;   // scale region
        int acc = 0;
        uint32_t aph = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const int tile = p.split == 1 ? u : u / p.split;
            int kb, ke;
            k_range(u - tile * p.split, p.split, KSS, kb, ke);
            const TileCoord tc = decode_tile<TT_MAX>(cum, gm, p.G, tile);
            ok = __all_sync(0xffffffffu, wait_bounded(bar_acce + 8 * acc, aph ^ 1u, abort_flag,
                                                      p.err, p.timeout_ns));
            if (!ok) break;
            const uint32_t idesc = idesc_mxf4nvf4((uint32_t)tc.w);
            const uint32_t d_tmem = tmem + acc * TT_MAX;
            for (int ks = kb; ks < ke; ++ks) {
                // both scale sets are in TMEM and the operand tiles have
                // landed: the four scale warps arrive after their stores,
                // one of them only after the stage's full barrier, so one
                // wait covers both (one wait less in the issuing thread)
                ok = __all_sync(0xffffffffu, wait_bounded(bar_sfready + 8 * s, ph, abort_flag,
                                                          p.err, p.timeout_ns));
                if (!ok) break;
                tc_fence_after();
                const uint32_t sfw0 = tmem_sf + r * Cfg::SF_COLS;
                const uint32_t sft0 = sfw0 + Cfg::SFW_COLS;
                if (elect_one()) {
#pragma unroll
                    for (int i = 0; i < KSUB; ++i) {
                        // K-tile i of the stage: its operand tiles, 16 weight-
                        // and 16 NA token-scale columns
                        const uint64_t ad =
                            sdesc_k_sw128(base + Cfg::OFF_W + s * Cfg::W_STAGE + i * Cfg::W_TILE);
                        const uint64_t bd =
                            sdesc_k_sw128(base + Cfg::OFF_T + s * Cfg::T_STAGE + i * Cfg::T_TILE);
                        const uint32_t sfw = sfw0 + 16 * i;
                        const uint32_t sft = sft0 + 16 * Cfg::NA * i;
                        const uint32_t acc_in = (ks != kb || i > 0) ? 1u : 0u;
                        umma_mxf4nvf4(d_tmem, ad, bd, idesc, sfw, sft, acc_in);
                        umma_mxf4nvf4(d_tmem, ad + 2, bd + 2, idesc, sfw + 4, sft + 4 * Cfg::NA, 1u);
                        umma_mxf4nvf4(d_tmem, ad + 4, bd + 4, idesc, sfw + 8, sft + 8 * Cfg::NA, 1u);
                        umma_mxf4nvf4(d_tmem, ad + 6, bd + 6, idesc, sfw + 12, sft + 12 * Cfg::NA, 1u);
                    }
                    umma_commit(bar_empty + 8 * s);
                    if (ks == ke - 1) umma_commit(bar_accf + 8 * acc);
                }
                __syncwarp();
                if (++s == STAGES) { s = 0; ph ^= 1u; }
                if (++r == Cfg::SF_BUFS) r = 0;
            }
            if (++acc == Cfg::ACC_BUFS) { acc = 0; aph ^= 1u; }
        }
        // Drain the tensor pipe before TMEM is freed.
        if (elect_one()) umma_commit(bar_done);
        __syncwarp();
        volatile int no_abort = 0;
        wait_bounded(bar_done, 0, &no_abort, p.err, p.timeout_ns);
    } else if (warp == 3 || warp == 4 || warp == 9 || warp == 10) {
        // ------------------------------- scale warps (one per TMEM lane quarter)
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        int s = 0;
        uint32_t ph = 0;
        int r = 0;              // scale region
        long long cnt = 0;      // stages walked
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const int tile = p.split == 1 ? u : u / p.split;
            int kb, ke;
            k_range(u - tile * p.split, p.split, KSS, kb, ke);
            for (int ks = kb; ks < ke; ++ks) {
                ok = __all_sync(0xffffffffu, wait_bounded(bar_sfull + 8 * s, ph, abort_flag,
                                                          p.err, p.timeout_ns));
                if (!ok) break;
                if (Cfg::SF_BUFS < STAGES && cnt >= Cfg::SF_BUFS) {
                    // the MMAs of the stage that last used region r are done
                    const long long prev = cnt - Cfg::SF_BUFS;
                    ok = __all_sync(0xffffffffu,
                                    wait_bounded(bar_empty + 8 * (int)(prev % STAGES),
                                                 (uint32_t)((prev / STAGES) & 1), abort_flag,
                                                 p.err, p.timeout_ns));
                    if (!ok) break;
                }
                // (With a region per stage, the MMAs that read this stage's
                // scale columns in the previous round completed before its
                // loads were issued: empty barrier.)
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < KSUB; ++i) {
                    // K-tile i of the stage.  Weights: column 4q + c = word c
                    // of row `lane` of atom q
                    const uint8_t* wsf = sbase + Cfg::OFF_WSF + s * Cfg::WSF_STAGE +
                                         i * Cfg::WSF_TILE + lane * 16;
                    uint32_t w[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 v = *reinterpret_cast<const uint4*>(wsf + 512 * q);
                        w[4 * q] = v.x;
                        w[4 * q + 1] = v.y;
                        w[4 * q + 2] = v.z;
                        w[4 * q + 3] = v.w;
                    }
                    // tokens: column 4(q NA + a) + c = word q of plain row
                    // 128a + 32c + lane (rows past TT_MAX: zero, never read)
                    const uint8_t* plain = sbase + Cfg::OFF_TSFP + s * Cfg::TSF_STAGE +
                                           i * Cfg::TSF_PLAIN + lane * 16;
                    uint32_t t[16 * Cfg::NA];
#pragma unroll
                    for (int a = 0; a < Cfg::NA; ++a) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint4 v = make_uint4(0u, 0u, 0u, 0u);
                            if (128 * a + 32 * c < TT_MAX)
                                v = *reinterpret_cast<const uint4*>(plain + (128 * a + 32 * c) * 16);
                            t[4 * (0 * Cfg::NA + a) + c] = v.x;
                            t[4 * (1 * Cfg::NA + a) + c] = v.y;
                            t[4 * (2 * Cfg::NA + a) + c] = v.z;
                            t[4 * (3 * Cfg::NA + a) + c] = v.w;
                        }
                    }
                    const uint32_t sfw = tmem_sf + r * Cfg::SF_COLS + lane_off + 16 * i;
                    const uint32_t sft = tmem_sf + r * Cfg::SF_COLS + lane_off + Cfg::SFW_COLS +
                                         16 * Cfg::NA * i;
                    tmem_st_32x32b_x16(sfw, w);
#pragma unroll
                    for (int h = 0; h < Cfg::NA; ++h)
                        tmem_st_32x32b_x16(sft + 16 * h, t + 16 * h);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                // warp 3 also waits for the stage's operand tiles, so that the
                // completed sfready phase tells the MMA thread both
                if (warp == 3) {
                    ok = __all_sync(0xffffffffu, wait_bounded(bar_full + 8 * s, ph, abort_flag,
                                                              p.err, p.timeout_ns));
                    if (!ok) break;
                }
                if (lane == 0) mbar_arrive(bar_sfready + 8 * s);
                if (++s == STAGES) { s = 0; ph ^= 1u; }
                if (++r == Cfg::SF_BUFS) r = 0;
                ++cnt;
            }
        }
    } else if (warp >= 5 && warp <= 8) {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 5;     // epilogue warp 0..3
        const int quad = warp & 3;   // TMEM lane quarter this warp may access
        uint8_t* stage_buf = sbase + Cfg::OFF_EPI + ew * (16 * 32 * 2);
        int acc = 0;
        uint32_t aph = 0;
        uint32_t ntile = 0;   // tiles reduced (cluster split-K barrier phases)
        if (p.csplit) cluster_wait();
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
            const int tile = u / p.split;
            const int sp = u - tile * p.split;
            const TileCoord tc = decode_tile<TT_MAX>(cum, gm, p.G, tile);
            const bool ok = __all_sync(0xffffffffu, wait_bounded(bar_accf + 8 * acc, aph, abort_flag,
                                                                 p.err, p.timeout_ns));
            if (!ok && p.split == 1) break;
            tc_fence_after();
            const float al = __ldg(p.alpha + tc.g);
            const int n0 = tc.nt * 128 + quad * 32;   // first of this warp's 32 weight rows
            const int t_end = min(tc.t0 + tc.w, tc.m);
            const uint32_t tbase = tmem + acc * TT_MAX + ((uint32_t)(quad * 32) << 16);
            // each lane later stores 16 bytes: token row (lane >> 2) (+8),
            // weight rows n0 + 8*(lane & 3) .. +7
            const int tr = lane >> 2, tq = lane & 3;
            const bool n_ok = n0 + 8 * tq < p.N;
            __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(stage_buf);
            if (SWIGLU) {
                swiglu_tile_store<TT_MAX>(p, off, tc, tbase, tc.nt, quad, lane, al, stage_buf);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_acce + 8 * acc);
                signal_tile_part<TT_MAX>(p, tc, lane);
            } else if (p.split == 1) {
#pragma unroll 1
                for (int c = 0; c < TT_MAX / 16; ++c) {
                    if (c * 16 >= tc.w) break;
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(tbase + c * 16, r);
                    tmem_wait_ld();
                    // lane = weight row n0 + lane; column t = token; transpose via
                    // shared memory into [token][32 rows] bf16
#pragma unroll
                    for (int t = 0; t < 16; ++t) sb[t * 32 + lane] = __float2bfloat16_rn(al * __uint_as_float(r[t]));
                    __syncwarp();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int t = tr + 8 * h;
                        const int tok = tc.t0 + c * 16 + t;
                        const uint4 v = *reinterpret_cast<const uint4*>(stage_buf + t * 64 + tq * 16);
                        const long long row = out_row(p, off, tc.g, tok);
                        if (tok < t_end && n_ok && row >= 0)
                            *reinterpret_cast<uint4*>(p.C + row * p.N + n0 + 8 * tq) = v;
                    }
                    __syncwarp();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_acce + 8 * acc);
                signal_tile_part<TT_MAX>(p, tc, lane);
            } else if (p.csplit) {
                // split-K in a cluster: the CTA of cluster rank sp computed K
                // range sp of this tile.  Each CTA leaves its fp32 partial in
                // its own shared memory; CTA sp then sums token rows sp,
                // sp + split, ... over all ranks in rank order (the order of
                // the workspace reduction below) and stores them.  All CTAs
                // of a cluster walk the same tiles, so the per-tile arrivals
                // pair up.  As below, the 4 epilogue warps pass the same
                // named barriers on every tile and leave together on a flag
                // set under a barrier; after a timeout the peers' waits run
                // out in turn, and the kernel's closing cluster barrier keeps
                // every CTA's shared memory alive while peers may read it.
                const uint32_t ph_t = ntile & 1u;
                bool go = ok;
                if (go && ntile > 0)   // peers have read this CTA's previous partial
                    go = __all_sync(0xffffffffu, wait_bounded_cluster(bar_pfree, ph_t ^ 1u, abort_flag,
                                                                      p.err, p.timeout_ns));
                if (go) {
                    // partial [token][128 weight rows]: lane = row, so each
                    // token's 32 rows of this warp are one 128-byte row piece
                    float* part = reinterpret_cast<float*>(sbase + Cfg::OFF_PART) + quad * 32 + lane;
#pragma unroll 1
                    for (int c = 0; c < TT_MAX / 16; ++c) {
                        if (c * 16 >= tc.w) break;
                        uint32_t r[16];
                        tmem_ld_32x32b_x16(tbase + c * 16, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int t = 0; t < 16; ++t) part[(c * 16 + t) * 128] = __uint_as_float(r[t]);
                    }
                }
                if (ok) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_acce + 8 * acc);   // TMEM no longer needed
                }
                named_barrier_sync(1, 128);   // the 4 warps' partial rows are stored
                if (ew == 0) {
                    const int stop = __shfl_sync(0xffffffffu, lane == 0 ? *abort_flag : 0, 0);
                    if (lane == 0) *epi_stop = stop;
                    // lane q tells rank q; release at cluster scope publishes
                    // the CTA's partial (ordered before it by the barrier).
                    // One arrive per lane: a release arrive takes hundreds of
                    // cycles, so they run side by side
                    if (!stop && lane < p.split)
                        mbar_arrive_remote_release(mapa_shared(bar_pready, (uint32_t)lane));
                }
                named_barrier_sync(1, 128);
                if (*epi_stop) break;
                const bool rd = __all_sync(0xffffffffu, wait_bounded_cluster(bar_pready, ph_t, abort_flag,
                                                                             p.err, p.timeout_ns));
                if (rd) {
                    // token rows t = sp + split (ew + 4 i); lane: weight rows
                    // 4 lane .. 4 lane + 3 (16-byte loads from every rank)
                    const int ng = tc.nt * 128 + 4 * lane;
                    const uint32_t part0 = base + Cfg::OFF_PART + 16u * lane;
                    for (int t = sp + p.split * ew; t < tc.w; t += 4 * p.split) {
                        const uint32_t a = part0 + (uint32_t)t * 512u;
                        float4 v[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            if (q < p.split) v[q] = ld_shared_cluster_v4(mapa_shared(a, (uint32_t)q));
                        float4 sum = v[0];
#pragma unroll
                        for (int q = 1; q < 8; ++q)
                            if (q < p.split) {
                                sum.x += v[q].x;
                                sum.y += v[q].y;
                                sum.z += v[q].z;
                                sum.w += v[q].w;
                            }
                        const int tok = tc.t0 + t;
                        const long long row = out_row(p, off, tc.g, tok);
                        if (tok < t_end && ng < p.N && row >= 0) {
                            uint2 o;
                            o.x = pack_bf16x2(al * sum.x, al * sum.y);
                            o.y = pack_bf16x2(al * sum.z, al * sum.w);
                            *reinterpret_cast<uint2*>(p.C + row * p.N + ng) = o;
                        }
                    }
                }
                named_barrier_sync(1, 128);   // the 4 warps' reads of the partials are done
                if (ew == 0) {
                    const int stop = __shfl_sync(0xffffffffu, lane == 0 ? *abort_flag : 0, 0);
                    if (lane == 0) *epi_stop = stop;
                    // the reads completed (their values are stored): relaxed
                    // arrives free the peers' partials, lane q for rank q
                    if (!stop && lane < p.split)
                        mbar_arrive_remote_relaxed(mapa_shared(bar_pfree, (uint32_t)lane));
                }
                named_barrier_sync(1, 128);
                if (*epi_stop) break;
                ++ntile;
            } else {
                // split-K.  The 4 epilogue warps pass the same named-barrier
                // sequence on every unit, even after a timeout (then they skip
                // the work), and leave the loop together on a flag set under
                // the barrier, so no warp can wait on a barrier another left.
                if (ok) {
                    // leave this range's fp32 partial, [column][128 rows]
                    float* part = p.ws_part + ((size_t)tile * p.split + sp) * (TT_MAX * 128) + quad * 32 + lane;
#pragma unroll 1
                    for (int c = 0; c < TT_MAX / 16; ++c) {
                        if (c * 16 >= tc.w) break;
                        uint32_t r[16];
                        tmem_ld_32x32b_x16(tbase + c * 16, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int t = 0; t < 16; ++t) part[(c * 16 + t) * 128] = __uint_as_float(r[t]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_acce + 8 * acc);   // TMEM no longer needed
                }
                // the barrier orders the 4 warps' partial stores before the
                // ticket; one device-scope fence by the ticket's thread then
                // publishes them all (a fence in every thread waited for each
                // thread's own stores to be acknowledged, microseconds per
                // unit under a saturated memory system)
                named_barrier_sync(1, 128);                          // the 4 epilogue warps
                if (ew == 0 && lane == 0) {
                    const int stop = *abort_flag;
                    *epi_stop = stop;
                    __threadfence();
                    *epi_flag = (!stop && epoch_arrive(p.ws_cnt + tile, p.epoch, 64) ==
                                              (unsigned long long)p.split) ? 1 : 0;
                    __threadfence();   // acquire: the other ranges' partials, for the last range
                }
                named_barrier_sync(1, 128);
                if (*epi_flag) {
                    // the last range: sum all ranges' partials in range order
                    const float* base_part = p.ws_part + (size_t)tile * p.split * (TT_MAX * 128) + quad * 32 + lane;
#pragma unroll 1
                    for (int c = 0; c < TT_MAX / 16; ++c) {
                        if (c * 16 >= tc.w) break;
                        // every range's value of a column is loaded before
                        // any is added (split <= 16), so the loads overlap
                        // instead of each waiting for the previous sum; the
                        // sum is still taken in range order
#pragma unroll 2
                        for (int t = 0; t < 16; ++t) {
                            float v[16];
#pragma unroll
                            for (int r2 = 0; r2 < 16; ++r2)
                                v[r2] = r2 < p.split ? __ldcg(base_part + (size_t)r2 * (TT_MAX * 128) +
                                                              (c * 16 + t) * 128)
                                                     : 0.f;
                            float acc_v = v[0];
#pragma unroll
                            for (int r2 = 1; r2 < 16; ++r2)
                                if (r2 < p.split) acc_v += v[r2];
                            sb[t * 32 + lane] = __float2bfloat16_rn(al * acc_v);
                        }
                        __syncwarp();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int t = tr + 8 * h;
                            const int tok = tc.t0 + c * 16 + t;
                            const uint4 v = *reinterpret_cast<const uint4*>(stage_buf + t * 64 + tq * 16);
                            const long long row = out_row(p, off, tc.g, tok);
                            if (tok < t_end && n_ok && row >= 0)
                                *reinterpret_cast<uint4*>(p.C + row * p.N + n0 + 8 * tq) = v;
                        }
                        __syncwarp();
                    }
                }
                const bool stop = *epi_stop != 0;
                named_barrier_sync(1, 128);   // epi_flag / epi_stop are reused by the next unit
                if (stop) break;
            }
            if (++acc == Cfg::ACC_BUFS) { acc = 0; aph ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
    // cluster split-K: no CTA leaves while another may still read its
    // partial or arrive on its barriers
    if (p.csplit) {
        if (warp < 5 || warp > 8) cluster_wait();   // the epilogue warps waited already
        cluster_arrive();
        cluster_wait();
    }
}

// One CTA waits on a barrier that nothing completes; the bounded wait gives
// up after timeout_ns and records NVFP4GG_ERR_TIMEOUT.
__global__ void watchdog_selftest_kernel(int* err, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        wait_bounded(smem_u32(&bar), 0, &abort_flag, err, timeout_ns);
    __syncthreads();
}

// Tensor-pipe throughput probe: every CTA issues `iters` x 4 block-scaled
// MMAs (M = 128, N = n, K = 64 each) on resident shared-memory operands
// (zero codes, unit scales) into one TMEM accumulator, from one thread, then
// waits for the tensor pipe with a bounded wait.  FLOPs per CTA:
// iters * 4 * 2 * 128 * n * 64.
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int n, int* err,
                                                          unsigned long long timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw);
    // [0, 16K) A tile, [16K, 48K) B tile (256 rows), [48K, 50K) 4 scale
    // atoms shared by A and B, then the barrier and the TMEM slot
    constexpr int OFF_SF = 49152, OFF_BAR = 51200, OFF_SLOT = 51208;
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < OFF_SF / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(sbase)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < 2048 / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(sbase + OFF_SF)[i] = 0x38383838u;   // e4m3 1.0
    if (threadIdx.x == 0) {
        mbar_init(base + OFF_BAR, 1);
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(base + OFF_SLOT, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sbase + OFF_SLOT);
    if (threadIdx.x == 0) {
        const uint32_t sfa = tmem + 256, sfb = tmem + 272;
        for (int q = 0; q < 4; ++q) {
            tmem_cp_32x128b_x4(sfa + 4 * q, sdesc_rows16(base + OFF_SF + 512 * q));
            tmem_cp_32x128b_x4(sfb + 8 * q, sdesc_rows16(base + OFF_SF + 512 * q));
            tmem_cp_32x128b_x4(sfb + 8 * q + 4, sdesc_rows16(base + OFF_SF + 512 * q));
        }
        const uint32_t idesc = idesc_mxf4nvf4((uint32_t)n);
        const uint64_t ad = sdesc_k_sw128(base);
        const uint64_t bd = sdesc_k_sw128(base + 16384);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                umma_mxf4nvf4(tmem, ad + 2 * q, bd + 2 * q, idesc, sfa + 4 * q, sfb + 8 * q,
                              (it | q) != 0);
        }
        umma_commit(base + OFF_BAR);
        volatile int no_abort = 0;
        wait_bounded(base + OFF_BAR, 0, &no_abort, err, timeout_ns);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Where the rows of the logical weight [G][N][*] live: row r of expert g is
// row r of src0 for r < split, else row r - split of src1, each source
// holding `stride` rows per expert.  One weight: src0 = src1, split = stride
// = N.  The dual GEMM's two operands (gate B1 and up B2 of N/2 rows each):
// src0 = B1, src1 = B2, split = stride = N/2.
struct WeightSource {
    const uint8_t* src0;
    const uint8_t* src1;
    int split;
    int stride;
};

__device__ __forceinline__ const uint8_t* weight_row(const WeightSource& w, int g, int r,
                                                     size_t row_bytes) {
    return r < w.split ? w.src0 + ((size_t)g * w.stride + r) * row_bytes
                       : w.src1 + ((size_t)g * w.stride + (r - w.split)) * row_bytes;
}

// Source row of prepared weight row n: the identity, or with `swiglu` the
// gate/up interleave the fused SwiGLU epilogue reads (N % 128 == 0): in
// 128-row block b, lane quarter q, row l of 32 holds gate row
// 64b + 16q + l (l < 16) or up row N/2 + 64b + 16q + (l - 16).
__device__ __forceinline__ int prepared_source_row(int n, int N, int swiglu) {
    if (!swiglu) return n;
    const int b = n >> 7, q = (n >> 5) & 3, l = n & 31;
    const int col = 64 * b + 16 * q + (l & 15);
    return l < 16 ? col : (N >> 1) + col;
}

// Weight-scale re-layout: B_sf u8 [G][N][K/16] -> atoms [G][NT][K/64][32][4][4]
// where atom byte (i, j, b) is the scale of row 128*nt + 32*j + i, K block
// 4*kc + b (zero for rows >= N).  One thread per 16-byte atom row.
__global__ void relayout_weight_scales_kernel(const WeightSource bsf, uint8_t* __restrict__ out,
                                              int G, int N, int K, int swiglu) {
    const int NT = (N + 127) / 128;
    const int KC = K / 64;
    const long long rows = (long long)G * NT * KC * 32;
    const int ks16 = K / 16;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < rows;
         idx += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(idx & 31);
        long long rest = idx >> 5;
        const int kc = (int)(rest % KC);
        rest /= KC;
        const int nt = (int)(rest % NT);
        const int g = (int)(rest / NT);
        uint32_t wv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = nt * 128 + 32 * j + i;
            wv[j] = n < N ? *reinterpret_cast<const uint32_t*>(
                                weight_row(bsf, g, prepared_source_row(n, N, swiglu), ks16) + 4 * kc)
                          : 0u;
        }
        *reinterpret_cast<uint4*>(out + idx * 16) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
}

// Weight-code re-layout: B u8 [G][N][K/2] -> tiles [G][NT][K/256][128][128]
// holding rows 128*nt .. +127 and bytes 128*ks .. +127 of each row, stored
// the way a 128-byte-swizzled TMA load would leave them in shared memory
// (16-byte chunk c of row r at chunk c ^ (r % 8)), zero for rows >= N.  One
// thread per 16-byte chunk.
__global__ void relayout_weight_codes_kernel(const WeightSource b, uint8_t* __restrict__ out,
                                             int G, int N, int K, int swiglu) {
    const int NT = (N + 127) / 128;
    const int KS = K / 256;
    const long long chunks = (long long)G * NT * KS * 1024;
    const size_t row_bytes = (size_t)K / 2;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < chunks;
         idx += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(idx & 7);
        const int r = (int)((idx >> 3) & 127);
        long long rest = idx >> 10;
        const int ks = (int)(rest % KS);
        rest /= KS;
        const int nt = (int)(rest % NT);
        const int g = (int)(rest / NT);
        const int n = nt * 128 + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n < N)
            v = *reinterpret_cast<const uint4*>(weight_row(b, g, prepared_source_row(n, N, swiglu), row_bytes) +
                                                (size_t)ks * 128 + c * 16);
        *reinterpret_cast<uint4*>(out + (idx >> 3) * 128 + ((c ^ (r & 7)) * 16)) = v;
    }
}

}  // namespace nvfp4gg
