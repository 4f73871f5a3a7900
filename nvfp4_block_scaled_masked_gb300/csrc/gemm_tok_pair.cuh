// Token-major CTA-pair kernel for compute-bound experts of the masked,
// block-scaled NVFP4 grouped GEMM-NT (grouped_gemm_nt_masked on "The CuteDSL
// Gamble: Chasing Kernel Efficiency on Blackwell GPUs", "The Message").
//
// For experts with many valid rows the weight stream no longer dominates:
// the tensor pipe does.  Here the two CTAs of a 2-CTA cluster run
// tcgen05.mma.cta_group::2 with M = 256 tokens (128 per CTA, the TMEM lanes)
// and N = 256 weight rows (two 128-row weight blocks, one staged by each
// CTA), the largest block-scaled NVFP4 MMA.  Per SM a ring stage then
// carries 32 KB of operands for 4 x 136 tensor cycles, and five stages fit:
// the ring covers more load latency than the swap-AB kernels' 192-token
// tiles can.  The accumulator holds 256 fp32 columns (one buffer), so
// five TMEM scale-factor regions fit beside it: one per ring stage.
//
// Roles (512 threads per CTA; a role's warp walks the stages with
// warp-uniform values and an elected lane issues the single-thread
// instructions).  Each producer issues one copy per stage: measured on
// GB300, a thread's copies per stage, not their bytes, bound the ring.
//   warp 0        weight producer: this CTA's 16 KB weight tile (tiled TMA
//                 whose completion is counted on the leader's `full`).
//   warp 2        token producer: this CTA's 128 token rows (same).
//   warp 15       scale producer: its weight block's 2 KB of scale atoms,
//                 multicast to both CTAs (each CTA's scale warps need all
//                 256 rows' scales), and its 128 token scale rows; both
//                 complete this CTA's `sfull`.
//   warp 1        TMEM (allocated for the pair).  Leader: the MMA warp, 4
//                 pair MMAs per stage after one wait on `full` (both CTAs'
//                 operand tiles) and one on `sfready` (both CTAs' scale
//                 factors), commits multicast to both CTAs.
//   warps 3..6    scale warps, one per TMEM lane quarter: token scales
//                 (this CTA's rows, regrouped) and the 256 weight rows'
//                 scales into this CTA's TMEM with tcgen05.st, then an
//                 arrive on the leader's `sfready` (remote from the peer).
//   warps 7..14   epilogue, two warps per lane quarter (one per half of the
//                 256 columns): tcgen05.ld of the whole quarter-half (lane =
//                 token, column = weight row), x alpha, bf16 pairs held in
//                 registers; the accumulator is released once the last
//                 load has landed, so the stores overlap the next tile's
//                 main loop.  Stores go
//                 through a per-warp [32 rows][64 B] transpose in shared
//                 memory: each instruction writes 8 rows x 64 contiguous
//                 bytes; rows m >= masked_m are skipped.
// Every wait is bounded; on expiry the waiter records NVFP4GG_ERR_TIMEOUT
// and raises the CTA's abort flag; copies and MMAs in flight are drained,
// then TMEM is freed.
#pragma once
#include "gemm.cuh"
#include "gemm_pair.cuh"

namespace nvfp4gg {

constexpr int kTokThreads = 512;

struct TokPairCfg {
    static constexpr int STAGES = 5;
    static constexpr int T_TILE = 128 * 128;       // this CTA's 128 token rows x 256 codes
    static constexpr int W_TILE = 128 * 128;       // this CTA's 128 weight rows x 256 codes
    static constexpr int TSF_STAGE = 128 * 16;     // this CTA's token scale rows (plain)
    static constexpr int WSF_STAGE = 2 * 4 * 512;  // both weight blocks' scale atoms
    static constexpr int ACC_COLS = 256;
    // scale region per stage: 16 token-scale columns (4 per K chunk) then 32
    // weight-scale columns (8 per K chunk)
    static constexpr int SFA_COLS = 16;
    static constexpr int SF_COLS = SFA_COLS + 32;
    static_assert(ACC_COLS + STAGES * SF_COLS <= 512, "TMEM budget");
    static_assert(SF_COLS % 4 == 0 && SFA_COLS % 4 == 0 && ACC_COLS % 4 == 0, "SF alignment");
    static constexpr int TMEM_COLS = 512;

    static constexpr int OFF_T = 0;
    static constexpr int OFF_W = OFF_T + STAGES * T_TILE;
    static constexpr int OFF_TSF = OFF_W + STAGES * W_TILE;
    static constexpr int OFF_WSF = OFF_TSF + STAGES * TSF_STAGE;
    // epilogue staging: per epilogue warp 32 token rows x 32 columns of bf16
    static constexpr int EPI_WARP_BYTES = 32 * 64;
    static constexpr int OFF_EPI = OFF_WSF + STAGES * WSF_STAGE;
    static constexpr int OFF_BAR = OFF_EPI + 8 * EPI_WARP_BYTES;
    // full, sfull, empty, sfready per stage; accf, acce; the MMA drain
    static constexpr int NUM_BARS = 4 * STAGES + 3;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_TAB = (OFF_MISC + 16 + 15) & ~15;
    // cum[G + 1], gm[G]: sized per launch (plus alignment slack)
    static constexpr int SMEM_FIXED = OFF_TAB + 4 + 1024;
    static constexpr int SMEM_LIMIT = 232448;
    static_assert(SMEM_FIXED + 8 <= SMEM_LIMIT, "shared memory budget");
    static constexpr int MAX_GROUPS = (SMEM_LIMIT - SMEM_FIXED) / 8;
    static int smem_bytes(int G) { return SMEM_FIXED + 8 * G; }
    static_assert(OFF_W % 1024 == 0 && OFF_T % 1024 == 0, "128-byte swizzle alignment");
};

// Tile id -> (expert, weight-block pair, first token of the 256, masked_m).
// Within an expert the weight-block pair runs fastest: the CTAs working at
// one time then share one or two token tiles and cycle through all of the
// expert's weights, which stay in L2 for its next token tiles (with the
// token tile fastest, every round of tiles would start on weights that no
// CTA has read yet, all fetched from DRAM at the same moment).
__device__ __forceinline__ TileCoord decode_tok_tile(const int* cum, const int* gm, int G, int NP,
                                                     int tile) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    TileCoord c;
    c.g = lo;
    c.m = gm[lo];
    const int local = tile - cum[lo];
    const int tt = local / NP;
    c.w = 256;
    c.nt = local - tt * NP;          // weight-block pair
    c.t0 = tt * 256;
    return c;
}

__global__ void __launch_bounds__(kTokThreads, 1)
gemm_nt_masked_tok_pair_kernel(const __grid_constant__ GemmParams<1> p,
                               const __grid_constant__ CUtensorMap tm_w) {
    using Cfg = TokPairCfg;
    constexpr int STAGES = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();   // 0 = leader, 1 = peer
    const bool leader = rank == 0;

    const uint32_t bar_full = base + Cfg::OFF_BAR;         // leader: both CTAs' operand tiles
    const uint32_t bar_sfull = bar_full + 8 * STAGES;      // this CTA's scale rows
    const uint32_t bar_empty = bar_sfull + 8 * STAGES;     // leader's multicast commit
    const uint32_t bar_sfready = bar_empty + 8 * STAGES;   // leader: 4 local + 4 peer scale warps
    const uint32_t bar_accf = bar_sfready + 8 * STAGES;    // leader's multicast commit
    const uint32_t bar_acce = bar_accf + 8;                // leader: 8 local + 8 peer epilogue warps
    const uint32_t bar_done = bar_acce + 8;                // MMA drain
    uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + Cfg::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    int* cum = reinterpret_cast<int*>(sbase + Cfg::OFF_TAB);
    int* gm = cum + p.G + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 2);
            mbar_init(bar_sfull + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
            mbar_init(bar_sfready + 8 * s, 8);
        }
        mbar_init(bar_accf, 1);
        mbar_init(bar_acce, 16);
        mbar_init(bar_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(base + Cfg::OFF_MISC, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    if (warp == 2 && lane == 0) {
        prefetch_tmap(&p.tm_a[0]);
        prefetch_tmap(&p.tm_asf[0]);
        prefetch_tmap(&tm_w);
    }
    for (int g = threadIdx.x; g < p.G; g += kTokThreads) {
        int m = __ldg(p.masked_m + g);
        if (m < 0 || m > p.M_max) {
            record_error(p.err, NVFP4GG_ERR_MASK);
            m = m < 0 ? 0 : p.M_max;
        }
        gm[g] = m;
    }
    const int NP = p.NT / 2;
    __syncthreads();
    if (warp == 0) {
        const int per = (p.G + 31) / 32;
        const int lo = lane * per;
        const int hi = min(p.G, lo + per);
        int sum = 0;
        for (int g = lo; g < hi; ++g) sum += ((gm[g] + 255) >> 8) * NP;
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int g = lo; g < hi; ++g) {
            cum[g] = run;
            run += ((gm[g] + 255) >> 8) * NP;
        }
        if (lane == 31) cum[p.G] = incl;
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // both CTAs' barriers initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const int total = cum[p.G];
    const int cid = blockIdx.x >> 1;
    const int ncl = gridDim.x >> 1;
    const uint32_t tmem_sf = tmem + Cfg::ACC_COLS;
    // the leader's full barriers, as addresses this CTA's TMA can signal
    const uint32_t full_leader = leader ? bar_full : mapa_shared(bar_full, 0);

    if (warp == 0 || warp == 2 || warp == 15) {
        // ----------------------------------------------------------- producers
        // One copy per stage per producer warp: an issuing thread with
        // several copies per stage was measured to be the ring's bound.
        //   warp 0:  this CTA's weight tile (leader's `full`)
        //   warp 2:  this CTA's token tile (leader's `full`)
        //   warp 15: this CTA's weight block's scale atoms, multicast to both
        //            CTAs, and its token scale rows (this CTA's `sfull`, which
        //            also receives the peer's atoms)
        const int role = warp == 0 ? 0 : warp == 2 ? 1 : 2;
        const uint64_t pol_stream = policy_evict_first();
        int s = 0;
        uint32_t ph = 0;
        long long issued = 0;
        bool ok = true;
        for (int tile = cid; tile < total && ok; tile += ncl) {
            const TileCoord tc = decode_tok_tile(cum, gm, p.G, NP, tile);
            const int nt = 2 * tc.nt + (int)rank;                // this CTA's weight block
            const size_t wsf0 = ((size_t)tc.g * p.NT + nt) * (size_t)(p.KS * 4);   // atom index
            // row of this CTA's weight tile in the prepared-tile map, stage 0
            const int wrow = (int)((((size_t)tc.g * p.NT + nt) * p.KS) * 128);
            const int trow = tc.t0 + 128 * (int)rank;
            for (int ks = 0; ks < p.KS; ++ks) {
                ok = __all_sync(0xffffffffu, wait_bounded(bar_empty + 8 * s, ph ^ 1u, abort_flag,
                                                          p.err, p.timeout_ns));
                if (!ok) break;
                const uint32_t fl = full_leader + 8 * s;
                if (!elect_one()) {
                } else if (role == 0) {
                    if (leader) mbar_arrive_expect_tx(bar_full + 8 * s, 2 * Cfg::W_TILE);
                    tma_load_2d_pair(base + Cfg::OFF_W + s * Cfg::W_TILE, &tm_w, fl, 0,
                                     wrow + 128 * ks);
                } else if (role == 1) {
                    if (leader) mbar_arrive_expect_tx(bar_full + 8 * s, 2 * Cfg::T_TILE);
                    tma_load_3d_pair(base + Cfg::OFF_T + s * Cfg::T_TILE, &p.tm_a[0], fl, ks * 128,
                                     trow, tc.g);
                } else {
                    // the peer's empty barrier completed with this one (same
                    // multicast commit), so its slot s is free as well
                    const uint32_t sb = bar_sfull + 8 * s;
                    mbar_arrive_expect_tx(sb, Cfg::WSF_STAGE + Cfg::TSF_STAGE);
                    bulk_load_multicast(base + Cfg::OFF_WSF + s * Cfg::WSF_STAGE + rank * 2048,
                                        p.wsf + (wsf0 + 4 * (size_t)ks) * 512, 2048, sb, 0x3);
                    tma_load_3d(base + Cfg::OFF_TSF + s * Cfg::TSF_STAGE, &p.tm_asf[0], sb, ks * 16,
                                trow, tc.g);
                }
                __syncwarp();
                ++issued;
                if (++s == STAGES) { s = 0; ph ^= 1u; }
            }
        }
        // Drain: this CTA's scale copies (its own and the peer's multicast
        // atoms), and (leader) every operand copy of both CTAs, must have
        // landed before the CTAs may exit; the final cluster barrier keeps
        // both CTAs alive until then.
        for (int st = 0; st < STAGES; ++st) {
            if (st >= issued) break;
            const long long last = st + (long long)STAGES * ((issued - 1 - st) / STAGES);
            const uint32_t par = (uint32_t)((last / STAGES) & 1);
            volatile int no_abort = 0;
            if (role == 2) wait_bounded(bar_sfull + 8 * st, par, &no_abort, p.err, p.timeout_ns);
            else if (leader) wait_bounded(bar_full + 8 * st, par, &no_abort, p.err, p.timeout_ns);
        }
    } else if (warp == 1 && leader) {
        // ---------------------------------------------------- MMA warp (leader)
        int s = 0;
        uint32_t ph = 0;
        uint32_t aph = 0;
        bool ok = true;
        const uint32_t idesc = idesc_mxf4nvf4_pair(256u);
        for (int tile = cid; tile < total && ok; tile += ncl) {
            // the epilogue has read the previous tile's accumulator
            ok = __all_sync(0xffffffffu, wait_bounded(bar_acce, aph ^ 1u, abort_flag, p.err,
                                                      p.timeout_ns));
            if (!ok) break;
            tc_fence_after();
            for (int ks = 0; ks < p.KS; ++ks) {
                ok = __all_sync(0xffffffffu, wait_bounded(bar_full + 8 * s, ph, abort_flag, p.err,
                                                          p.timeout_ns) &&
                                                 wait_bounded(bar_sfready + 8 * s, ph, abort_flag,
                                                              p.err, p.timeout_ns));
                if (!ok) break;
                tc_fence_after();
                const uint32_t sfa = tmem_sf + s * Cfg::SF_COLS;
                const uint32_t sfb = sfa + Cfg::SFA_COLS;
                const uint64_t ad = sdesc_k_sw128(base + Cfg::OFF_T + s * Cfg::T_TILE);
                const uint64_t bd = sdesc_k_sw128(base + Cfg::OFF_W + s * Cfg::W_TILE);
                const uint32_t acc_in = ks != 0;
                if (elect_one()) {
                    umma_pair_mxf4nvf4(tmem, ad, bd, idesc, sfa, sfb, acc_in);
                    umma_pair_mxf4nvf4(tmem, ad + 2, bd + 2, idesc, sfa + 4, sfb + 8, 1u);
                    umma_pair_mxf4nvf4(tmem, ad + 4, bd + 4, idesc, sfa + 8, sfb + 16, 1u);
                    umma_pair_mxf4nvf4(tmem, ad + 6, bd + 6, idesc, sfa + 12, sfb + 24, 1u);
                    umma_commit_pair_multicast(bar_empty + 8 * s, 0x3);
                    if (ks == p.KS - 1) umma_commit_pair_multicast(bar_accf, 0x3);
                }
                __syncwarp();
                if (++s == STAGES) { s = 0; ph ^= 1u; }
            }
            aph ^= 1u;
        }
        if (elect_one()) umma_commit_pair(bar_done);
        __syncwarp();
        volatile int no_abort = 0;
        wait_bounded(bar_done, 0, &no_abort, p.err, p.timeout_ns);
    } else if (warp >= 3 && warp <= 6) {
        // ------------------------------- scale warps (one per TMEM lane quarter)
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t sfready_target = leader ? bar_sfready : mapa_shared(bar_sfready, 0);
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int tile = cid; tile < total && ok; tile += ncl) {
            for (int ks = 0; ks < p.KS; ++ks) {
                // region s was last read by the MMAs of this slot's previous
                // stage, which completed before its copies were reissued
                ok = __all_sync(0xffffffffu, wait_bounded(bar_sfull + 8 * s, ph, abort_flag,
                                                          p.err, p.timeout_ns));
                if (!ok) break;
                tc_fence_after();
                // tokens (this CTA's 128 rows): column 4q + c = word q of
                // plain row 32c + lane
                const uint8_t* plain = sbase + Cfg::OFF_TSF + s * Cfg::TSF_STAGE + lane * 16;
                uint32_t a[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4*>(plain + c * 32 * 16);
                    a[c] = v.x;
                    a[4 + c] = v.y;
                    a[8 + c] = v.z;
                    a[12 + c] = v.w;
                }
                // weights (256 rows, two blocks): column 8q + j = word (j & 3)
                // of row `lane` of block (j >> 2)'s atom q
                const uint8_t* wsf = sbase + Cfg::OFF_WSF + s * Cfg::WSF_STAGE + lane * 16;
                uint32_t w[32];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const uint4 v = *reinterpret_cast<const uint4*>(wsf + b * 2048 + q * 512);
                        w[8 * q + 4 * b] = v.x;
                        w[8 * q + 4 * b + 1] = v.y;
                        w[8 * q + 4 * b + 2] = v.z;
                        w[8 * q + 4 * b + 3] = v.w;
                    }
                }
                const uint32_t sfa = tmem_sf + s * Cfg::SF_COLS + lane_off;
                tmem_st_32x32b_x16(sfa, a);
                tmem_st_32x32b_x16(sfa + Cfg::SFA_COLS, w);
                tmem_st_32x32b_x16(sfa + Cfg::SFA_COLS + 16, w + 16);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (leader) mbar_arrive(sfready_target + 8 * s);
                    else mbar_arrive_remote_relaxed(sfready_target + 8 * s);
                }
                if (++s == STAGES) { s = 0; ph ^= 1u; }
            }
        }
    } else if (warp >= 7 && warp <= 14) {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 7;          // 0..7
        const int quad = warp & 3;        // TMEM lane quarter this warp may access
        const int half = ew >> 2;         // columns [128 half, 128 half + 128)
        const uint32_t acce_target = leader ? bar_acce : mapa_shared(bar_acce, 0);
        uint8_t* stage = sbase + Cfg::OFF_EPI + ew * Cfg::EPI_WARP_BYTES;
        uint32_t aph = 0;
        for (int tile = cid; tile < total; tile += ncl) {
            const TileCoord tc = decode_tok_tile(cum, gm, p.G, NP, tile);
            const bool ok = __all_sync(0xffffffffu, wait_bounded(bar_accf, aph, abort_flag, p.err,
                                                                 p.timeout_ns));
            if (!ok) break;
            tc_fence_after();
            const uint32_t alb = __float_as_uint(__ldg(p.alpha + tc.g));
            const uint64_t al2 = ((uint64_t)alb << 32) | alb;
            const uint32_t tbase = tmem + ((uint32_t)(quad * 32) << 16) + 128 * half;
            // the whole accumulator quarter-half into registers as bf16 pairs,
            // in 16-column loads, each issued before the previous one is
            // converted (the conversion overlaps the next load's latency); the
            // accumulator is released as soon as the last load has landed,
            // before the last 16 columns are converted: the next tile's MMAs
            // wait for that release, the stores below overlap them
            uint32_t o[64];
            uint32_t ra[16], rb[16];
            tmem_ld_32x32b_x16(tbase, ra);
#pragma unroll
            for (int c = 0; c < 8; c += 2) {
                tmem_wait_ld_regs(ra);
                tmem_ld_32x32b_x16(tbase + 16 * (c + 1), rb);
#pragma unroll
                for (int j = 0; j < 8; ++j) o[8 * c + j] = scale_pack_bf16x2(ra[2 * j], ra[2 * j + 1], al2);
                tmem_wait_ld_regs(rb);
                if (c + 2 < 8) {
                    tmem_ld_32x32b_x16(tbase + 16 * (c + 2), ra);
                } else {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (leader) mbar_arrive(acce_target);
                        else mbar_arrive_remote_relaxed(acce_target);
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    o[8 * (c + 1) + j] = scale_pack_bf16x2(rb[2 * j], rb[2 * j + 1], al2);
            }
            // stores: per 32-column chunk, a [32 rows][64 B] transpose in this
            // warp's staging buffer (16-byte units XOR-swizzled by row), then
            // each instruction writes 8 rows x 64 contiguous bytes
            const int row0 = tc.t0 + 128 * (int)rank + 32 * quad;   // this warp's first token
            __nv_bfloat16* cbase = p.C + ((size_t)tc.g * p.M_max) * p.N + (size_t)tc.nt * 256 + 128 * half;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int slot = u ^ ((lane >> 1) & 3);
                    *reinterpret_cast<uint4*>(stage + lane * 64 + slot * 16) =
                        make_uint4(o[16 * c + 4 * u], o[16 * c + 4 * u + 1], o[16 * c + 4 * u + 2],
                                   o[16 * c + 4 * u + 3]);
                }
                __syncwarp();
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int row = 8 * t + (lane >> 2);
                    const int u = lane & 3;
                    const uint4 v = *reinterpret_cast<const uint4*>(stage + row * 64 +
                                                                    (u ^ ((row >> 1) & 3)) * 16);
                    const int tok = row0 + row;
                    if (tok < tc.m)
                        *reinterpret_cast<uint4*>(cbase + (size_t)tok * p.N + 32 * c + 8 * u) = v;
                }
                __syncwarp();
            }
            aph ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // the leader's MMAs and copies are drained; no remote arrive in flight
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
    }
}

}  // namespace nvfp4gg
