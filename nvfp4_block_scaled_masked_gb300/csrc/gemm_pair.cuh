// CTA-pair variant of the masked, block-scaled NVFP4 grouped GEMM-NT for
// prefill-sized experts (the operation of grouped_gemm_nt_masked on "The
// CuteDSL Gamble: Chasing Kernel Efficiency on Blackwell GPUs", "The
// Message").
//
// The two CTAs of a 2-CTA cluster run one tcgen05 MMA of M = 256 weight rows
// (128 per CTA: weight blocks 2*np and 2*np + 1) by N = w tokens, the token
// rows split half per CTA.  Per SM this halves the token bytes staged per
// stage for the same MMA work, so a deeper ring fits in shared memory: the
// single-CTA kernel is bound by how many bytes its 4-stage ring keeps in
// flight against the load latency.
//
// Roles (352 threads, both CTAs unless noted; as in the single-CTA kernel,
// a role's warp walks the stages with warp-uniform values and an elected
// lane issues the single-thread instructions):
//   warps 0, 2        weight / token producers: the scale atoms (2 KB) then
//                     the 16 KB tile of this CTA's weight block; all w token
//                     scale rows then this CTA's half of the w token rows.
//   warp 1            TMEM (allocated for the pair).  Leader CTA: the MMA
//                     warp, 4 pair MMAs per stage, multicast commit of the
//                     stage to both CTAs.  Peer CTA: idle.
//   warps 3, 4, 9, 10 scale warps, one per TMEM lane quarter, in each CTA:
//                     this CTA's weight scales and all token scales into its
//                     own TMEM with tcgen05.st; then an arrive on the
//                     leader's sfready barrier (8 arrivals: the peer's are
//                     remote).  Warp 3 first waits for its CTA's operand
//                     tiles, so one barrier tells the MMA warp everything.
//   warps 5..8        epilogue, as in the single-CTA kernel, on this CTA's
//                     128 weight rows; the peer's warps release the
//                     accumulator to the leader with remote arrives.
// Cross-CTA signals are relaxed remote mbarrier arrives (tens of cycles; a
// release arrive costs hundreds).  Each reports an event the signalling
// thread has already observed complete -- tiles landed (it waited on the TMA
// barrier), scale factors stored (tcgen05.wait::st), TMEM read
// (tcgen05.wait::ld) -- and the receiver acts on it only through the tensor
// core after seeing the arrive.  Every wait is bounded.
#pragma once
#include "gemm.cuh"

namespace nvfp4gg {

constexpr int kPairThreads = 352;

template <int TT_MAX, int STAGES>
struct PairCfg {
    static_assert(TT_MAX % 32 == 0 && TT_MAX <= 256, "token tile");
    static_assert(STAGES >= 3, "ring depth");
    static constexpr int W_TILE = 128 * 128;            // this CTA's 128 weight rows x 256 codes
    static constexpr int T_TILE = (TT_MAX / 2) * 128;   // this CTA's half of the token rows
    static constexpr int WSF_STAGE = 4 * 512;
    static constexpr int TSF_PLAIN = TT_MAX * 16;       // all token scale rows
    static constexpr int NA = (TT_MAX + 127) / 128;
    static constexpr int ACC_BUFS = 2;
    static constexpr int SFW_COLS = 16;
    static constexpr int SFT_COLS = 16 * NA;
    static constexpr int SF_COLS = SFW_COLS + SFT_COLS;
    static constexpr int SF_FIT = (512 - ACC_BUFS * TT_MAX) / SF_COLS;
    // TMEM scale regions, used round-robin by stage count; a region is
    // rewritten only after the MMAs that read it completed.
    static constexpr int SF_BUFS = SF_FIT < STAGES ? SF_FIT : STAGES;
    static_assert(SF_BUFS >= 2, "TMEM budget");
    static constexpr int TMEM_NEED = ACC_BUFS * TT_MAX + SF_BUFS * SF_COLS;
    static_assert(TT_MAX % 4 == 0 && SF_COLS % 4 == 0, "SF alignment");
    static_assert(TMEM_NEED <= 512, "TMEM budget");
    static constexpr int TMEM_COLS = pow2_cols(TMEM_NEED);

    static constexpr int OFF_W = 0;
    static constexpr int OFF_T = OFF_W + STAGES * W_TILE;
    static constexpr int OFF_WSF = OFF_T + STAGES * T_TILE;
    static constexpr int OFF_TSFP = OFF_WSF + STAGES * WSF_STAGE;
    static constexpr int OFF_EPI = OFF_TSFP + STAGES * TSF_PLAIN;
    static constexpr int EPI_BYTES = 4 * 16 * 32 * 2;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    // full, sfull, empty, sfready per stage; accf, acce per buffer; the MMA drain
    static constexpr int NUM_BARS = 4 * STAGES + 2 * ACC_BUFS + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_TAB = (OFF_MISC + 16 + 15) & ~15;
    static constexpr int TAB_BYTES = (3 * kGroupsMax + 2) * 4;   // cum, gm, off (as the single-CTA kernel)
    static constexpr int SMEM_BYTES = OFF_TAB + TAB_BYTES + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(OFF_T % 1024 == 0 && T_TILE % 1024 == 0, "128-byte swizzle alignment");
};

// Pair tiles round token widths up to 32 (16 token rows per CTA at least).
__device__ __forceinline__ int token_width_pair(int m, int ntt) {
    return ntt ? (((m + ntt - 1) / ntt + 31) & ~31) : 0;
}

// Tile id -> (expert, weight-block pair, first token, token width, masked_m).
template <int TT_MAX>
__device__ __forceinline__ TileCoord decode_pair_tile(const int* cum, const int* gm, int G,
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
    const int ntt = token_tiles<TT_MAX>(c.m);
    c.w = token_width_pair(c.m, ntt);
    c.nt = local / ntt;              // weight-block pair index
    c.t0 = (local - c.nt * ntt) * c.w;
    return c;
}

// SWIGLU: the fused GEMM1 epilogue of the single-CTA kernels (weights
// prepared with gate and up rows interleaved per lane quarter), on this
// CTA's weight block 2 nt + rank.
template <int TT_MAX, int STAGES, bool SWIGLU = false>
__global__ void __launch_bounds__(kPairThreads, 1)
gemm_nt_masked_pair_kernel(const __grid_constant__ GemmParams<TT_MAX / 16> p) {
    using Cfg = PairCfg<TT_MAX, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();   // 0 = leader, 1 = peer
    const bool leader = rank == 0;

    const uint32_t bar_full = base + Cfg::OFF_BAR;          // this CTA's tiles: 2 producers + bytes
    const uint32_t bar_sfull = bar_full + 8 * STAGES;       // this CTA's scale rows
    const uint32_t bar_empty = bar_sfull + 8 * STAGES;      // leader's multicast commit
    const uint32_t bar_sfready = bar_empty + 8 * STAGES;    // leader: 4 local + 4 peer scale warps
    const uint32_t bar_accf = bar_sfready + 8 * STAGES;     // leader's multicast commit
    const uint32_t bar_acce = bar_accf + 8 * Cfg::ACC_BUFS; // leader: 4 local + 4 peer epilogue warps
    const uint32_t bar_done = bar_acce + 8 * Cfg::ACC_BUFS; // MMA drain
    uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + Cfg::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    int* cum = reinterpret_cast<int*>(sbase + Cfg::OFF_TAB);
    int* gm = cum + kGroupsMax + 1;
    int* off = gm + kGroupsMax;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 2);
            mbar_init(bar_sfull + 8 * s, 2);
            mbar_init(bar_empty + 8 * s, 1);
            mbar_init(bar_sfready + 8 * s, 8);
        }
        for (int b = 0; b < Cfg::ACC_BUFS; ++b) {
            mbar_init(bar_accf + 8 * b, 1);
            mbar_init(bar_acce + 8 * b, 8);
        }
        mbar_init(bar_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(base + Cfg::OFF_MISC, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    if (warp == 2 && lane == 0) {
        for (int i = 0; i < TT_MAX / 16; ++i) {
            prefetch_tmap(&p.tm_a[i]);
            prefetch_tmap(&p.tm_asf[i]);
        }
    }
    for (int g = threadIdx.x; g < p.G; g += kPairThreads) {
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
        for (int g = lo; g < hi; ++g) sum += token_tiles<TT_MAX>(gm[g]) * NP;
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int g = lo; g < hi; ++g) {
            cum[g] = run;
            run += token_tiles<TT_MAX>(gm[g]) * NP;
        }
        if (lane == 31) cum[p.G] = incl;
        int rs = 0;
        for (int g = lo; g < hi; ++g) rs += gm[g];
        int rincl = rs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, rincl, o);
            if (lane >= o) rincl += v;
        }
        int rrun = rincl - rs;
        for (int g = lo; g < hi; ++g) {
            off[g] = rrun;
            rrun += gm[g];
        }
        if (lane == 31) {
            off[p.G] = rincl;
            if (p.contiguous && rincl > p.M_total) record_error(p.err, NVFP4GG_ERR_MASK);
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // both CTAs' barriers initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const int total = cum[p.G];
    const int cid = blockIdx.x >> 1;      // cluster id
    const int ncl = gridDim.x >> 1;
    const uint32_t tmem_sf = tmem + Cfg::ACC_BUFS * TT_MAX;

    if (warp == 0 || warp == 2) {
        // ----------------------------------------------------------- producers
        const bool weights = warp == 0;
        const uint64_t pol_stream = policy_evict_first();
        int s = 0;
        uint32_t ph = 0;
        long long issued = 0;
        bool ok = true;
        for (int tile = cid; tile < total && ok; tile += ncl) {
            const TileCoord tc = decode_pair_tile<TT_MAX>(cum, gm, p.G, tile);
            const int nt = 2 * tc.nt + (int)rank;
            const size_t wtile = ((size_t)tc.g * p.NT + nt) * (size_t)p.KS;
            const uint8_t* wq_tile = p.wq + wtile * Cfg::W_TILE;
            const uint8_t* wsf_tile = p.wsf + wtile * Cfg::WSF_STAGE;
            const int half = tc.w >> 1;
            for (int ks = 0; ks < p.KS; ++ks) {
                ok = __all_sync(0xffffffffu, wait_bounded(bar_empty + 8 * s, ph ^ 1u, abort_flag,
                                                          p.err, p.timeout_ns));
                if (!ok) break;
                const uint32_t fb = bar_full + 8 * s;
                const uint32_t sb = bar_sfull + 8 * s;
                if (!elect_one()) {
                } else if (weights) {
                    mbar_arrive_expect_tx(sb, Cfg::WSF_STAGE);
                    bulk_load_hint(base + Cfg::OFF_WSF + s * Cfg::WSF_STAGE,
                                   wsf_tile + (size_t)ks * Cfg::WSF_STAGE, Cfg::WSF_STAGE, sb,
                                   pol_stream);
                    mbar_arrive_expect_tx(fb, Cfg::W_TILE);
                    bulk_load_hint(base + Cfg::OFF_W + s * Cfg::W_TILE,
                                   wq_tile + (size_t)ks * Cfg::W_TILE, Cfg::W_TILE, fb, pol_stream);
                } else {
                    mbar_arrive_expect_tx(sb, tc.w * 16);
                    const int ty = p.contiguous ? off[tc.g] + tc.t0 : tc.t0;
                    const int tz = p.contiguous ? 0 : tc.g;
                    tma_load_3d(base + Cfg::OFF_TSFP + s * Cfg::TSF_PLAIN, &p.tm_asf[(tc.w >> 4) - 1],
                                sb, ks * 16, ty, tz);
                    mbar_arrive_expect_tx(fb, half * 128);
                    tma_load_3d(base + Cfg::OFF_T + s * Cfg::T_TILE, &p.tm_a[(half >> 4) - 1], fb,
                                ks * 128, ty + (int)rank * half, tz);
                }
                __syncwarp();
                ++issued;
                if (++s == STAGES) { s = 0; ph ^= 1u; }
            }
        }
        for (int st = 0; st < STAGES; ++st) {
            if (st >= issued) break;
            const long long last = st + (long long)STAGES * ((issued - 1 - st) / STAGES);
            const uint32_t par = (uint32_t)((last / STAGES) & 1);
            volatile int no_abort = 0;
            wait_bounded(bar_full + 8 * st, par, &no_abort, p.err, p.timeout_ns);
            wait_bounded(bar_sfull + 8 * st, par, &no_abort, p.err, p.timeout_ns);
        }
    } else if (warp == 1 && leader) {
        // ---------------------------------------------------- MMA warp (leader)
        int s = 0;
        uint32_t ph = 0;
        int r = 0;   // scale region
        int acc = 0;
        uint32_t aph = 0;
        bool ok = true;
        for (int tile = cid; tile < total && ok; tile += ncl) {
            const TileCoord tc = decode_pair_tile<TT_MAX>(cum, gm, p.G, tile);
            ok = __all_sync(0xffffffffu, wait_bounded(bar_acce + 8 * acc, aph ^ 1u, abort_flag,
                                                      p.err, p.timeout_ns));
            if (!ok) break;
            const uint32_t idesc = idesc_mxf4nvf4_pair((uint32_t)tc.w);
            const uint32_t d_tmem = tmem + acc * TT_MAX;
            for (int ks = 0; ks < p.KS; ++ks) {
                // both CTAs' tiles landed and all eight scale warps stored
                ok = __all_sync(0xffffffffu, wait_bounded(bar_sfready + 8 * s, ph, abort_flag,
                                                          p.err, p.timeout_ns));
                if (!ok) break;
                tc_fence_after();
                const uint32_t sfw = tmem_sf + r * Cfg::SF_COLS;
                const uint32_t sft = sfw + Cfg::SFW_COLS;
                const uint64_t ad = sdesc_k_sw128(base + Cfg::OFF_W + s * Cfg::W_TILE);
                const uint64_t bd = sdesc_k_sw128(base + Cfg::OFF_T + s * Cfg::T_TILE);
                const uint32_t acc_in = ks != 0;
                if (elect_one()) {
                    umma_pair_mxf4nvf4(d_tmem, ad, bd, idesc, sfw, sft, acc_in);
                    umma_pair_mxf4nvf4(d_tmem, ad + 2, bd + 2, idesc, sfw + 4, sft + 4 * Cfg::NA, 1u);
                    umma_pair_mxf4nvf4(d_tmem, ad + 4, bd + 4, idesc, sfw + 8, sft + 8 * Cfg::NA, 1u);
                    umma_pair_mxf4nvf4(d_tmem, ad + 6, bd + 6, idesc, sfw + 12, sft + 12 * Cfg::NA, 1u);
                    umma_commit_pair_multicast(bar_empty + 8 * s, 0x3);
                    if (ks == p.KS - 1) umma_commit_pair_multicast(bar_accf + 8 * acc, 0x3);
                }
                __syncwarp();
                if (++s == STAGES) { s = 0; ph ^= 1u; }
                if (++r == Cfg::SF_BUFS) r = 0;
            }
            if (++acc == Cfg::ACC_BUFS) { acc = 0; aph ^= 1u; }
        }
        if (elect_one()) umma_commit_pair(bar_done);
        __syncwarp();
        volatile int no_abort = 0;
        wait_bounded(bar_done, 0, &no_abort, p.err, p.timeout_ns);
    } else if (warp == 3 || warp == 4 || warp == 9 || warp == 10) {
        // ------------------------------- scale warps (one per TMEM lane quarter)
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t sfready_target = leader ? bar_sfready : mapa_shared(bar_sfready, 0);
        int s = 0;
        uint32_t ph = 0;
        int r = 0;
        long long cnt = 0;
        bool ok = true;
        for (int tile = cid; tile < total && ok; tile += ncl) {
            for (int ks = 0; ks < p.KS; ++ks) {
                ok = __all_sync(0xffffffffu, wait_bounded(bar_sfull + 8 * s, ph, abort_flag,
                                                          p.err, p.timeout_ns));
                if (!ok) break;
                if (Cfg::SF_BUFS < STAGES && cnt >= Cfg::SF_BUFS) {
                    // the MMAs of the stage that last used region r are done
                    // (the leader's commit reaches both CTAs' empty barriers)
                    const long long prev = cnt - Cfg::SF_BUFS;
                    ok = __all_sync(0xffffffffu,
                                    wait_bounded(bar_empty + 8 * (int)(prev % STAGES),
                                                 (uint32_t)((prev / STAGES) & 1), abort_flag,
                                                 p.err, p.timeout_ns));
                    if (!ok) break;
                }
                tc_fence_after();
                // weights (this CTA's 128 rows): column 4q + c = word c of row
                // `lane` of atom q
                const uint8_t* wsf = sbase + Cfg::OFF_WSF + s * Cfg::WSF_STAGE + lane * 16;
                uint32_t w[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v = *reinterpret_cast<const uint4*>(wsf + 512 * q);
                    w[4 * q] = v.x;
                    w[4 * q + 1] = v.y;
                    w[4 * q + 2] = v.z;
                    w[4 * q + 3] = v.w;
                }
                // tokens (all w rows): column 4(q NA + a) + c = word q of plain
                // row 128a + 32c + lane
                const uint8_t* plain = sbase + Cfg::OFF_TSFP + s * Cfg::TSF_PLAIN + lane * 16;
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
                const uint32_t sfw = tmem_sf + r * Cfg::SF_COLS + lane_off;
                tmem_st_32x32b_x16(sfw, w);
#pragma unroll
                for (int h = 0; h < Cfg::NA; ++h)
                    tmem_st_32x32b_x16(sfw + Cfg::SFW_COLS + 16 * h, t + 16 * h);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (warp == 3) {   // this CTA's operand tiles landed, too
                    ok = __all_sync(0xffffffffu, wait_bounded(bar_full + 8 * s, ph, abort_flag,
                                                              p.err, p.timeout_ns));
                    if (!ok) break;
                }
                if (lane == 0) {
                    if (leader) mbar_arrive(sfready_target + 8 * s);
                    else mbar_arrive_remote_relaxed(sfready_target + 8 * s);
                }
                if (++s == STAGES) { s = 0; ph ^= 1u; }
                if (++r == Cfg::SF_BUFS) r = 0;
                ++cnt;
            }
        }
    } else if (warp >= 5 && warp <= 8) {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 5;
        const int quad = warp & 3;
        uint8_t* stage_buf = sbase + Cfg::OFF_EPI + ew * (16 * 32 * 2);
        const uint32_t acce_target = leader ? bar_acce : mapa_shared(bar_acce, 0);
        int acc = 0;
        uint32_t aph = 0;
        for (int tile = cid; tile < total; tile += ncl) {
            const TileCoord tc = decode_pair_tile<TT_MAX>(cum, gm, p.G, tile);
            const bool ok = __all_sync(0xffffffffu, wait_bounded(bar_accf + 8 * acc, aph,
                                                                 abort_flag, p.err, p.timeout_ns));
            if (!ok) break;
            tc_fence_after();
            const float al = __ldg(p.alpha + tc.g);
            const int n0 = (2 * tc.nt + (int)rank) * 128 + quad * 32;
            const int t_end = min(tc.t0 + tc.w, tc.m);
            const uint32_t tbase = tmem + acc * TT_MAX + ((uint32_t)(quad * 32) << 16);
            const int tr = lane >> 2, tq = lane & 3;
            const bool n_ok = n0 + 8 * tq < p.N;
            if (SWIGLU)
                swiglu_tile_store<TT_MAX>(p, off, tc, tbase, 2 * tc.nt + (int)rank, quad, lane, al,
                                          stage_buf);
#pragma unroll 1
            for (int c = 0; c < (SWIGLU ? 0 : TT_MAX / 16); ++c) {
                if (c * 16 >= tc.w) break;
                uint32_t rr[16];
                tmem_ld_32x32b_x16(tbase + c * 16, rr);
                tmem_wait_ld();
                __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(stage_buf);
#pragma unroll
                for (int t = 0; t < 16; ++t) sb[t * 32 + lane] = __float2bfloat16_rn(al * __uint_as_float(rr[t]));
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
            if (lane == 0) {
                if (leader) mbar_arrive(acce_target + 8 * acc);
                else mbar_arrive_remote_relaxed(acce_target + 8 * acc);
            }
            if (++acc == Cfg::ACC_BUFS) { acc = 0; aph ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // the leader's MMAs are drained; no remote arrive is in flight
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
    }
}

// Tensor-pipe throughput probe for CTA pairs: each 2-CTA cluster issues
// `iters` x 4 pair MMAs (M = 256: 128 rows per CTA, N = n, K = 64) from the
// leader's thread 0 on resident shared-memory operands (zero codes, unit
// scales written into each CTA's TMEM with tcgen05.st), then both CTAs wait
// for the multicast commit with a bounded wait.  FLOPs per cluster:
// iters * 4 * 2 * 256 * n * 64.
__global__ void __launch_bounds__(128, 1) mma_peak_pair_kernel(int iters, int n, int* err,
                                                               unsigned long long timeout_ns) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw);
    // [0, 16K) this CTA's 128 A rows, [16K, 32K) its (at most 128) B rows,
    // then the barrier and the TMEM slot
    constexpr int OFF_BAR = 32768, OFF_SLOT = 32776;
    const int warp = threadIdx.x >> 5;
    const bool leader = cluster_ctarank() == 0;
    for (int i = threadIdx.x; i < OFF_BAR / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(sbase)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        mbar_init(base + OFF_BAR, 1);
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc_pair(base + OFF_SLOT, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sbase + OFF_SLOT);
    // scale factors: columns 256..271 (A: 4 K chunks x 4) and 272..303
    // (B: 4 K chunks x 8), e4m3 1.0 in every byte, in this warp's lane quarter
    {
        uint32_t ones[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) ones[i] = 0x38383838u;
        const uint32_t q = tmem + ((uint32_t)(warp * 32) << 16);
        tmem_st_32x32b_x16(q + 256, ones);
        tmem_st_32x32b_x16(q + 272, ones);
        tmem_st_32x32b_x16(q + 288, ones);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // both CTAs' operands, scales and barriers are ready
    tc_fence_after();
    if (leader && threadIdx.x == 0) {
        const uint32_t sfa = tmem + 256, sfb = tmem + 272;
        const uint32_t idesc = idesc_mxf4nvf4_pair((uint32_t)n);
        const uint64_t ad = sdesc_k_sw128(base);
        const uint64_t bd = sdesc_k_sw128(base + 16384);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                umma_pair_mxf4nvf4(tmem, ad + 2 * q, bd + 2 * q, idesc, sfa + 4 * q, sfb + 8 * q,
                                   (it | q) != 0);
        }
        umma_commit_pair_multicast(base + OFF_BAR, 0x3);
    }
    if (threadIdx.x == 0) {
        volatile int no_abort = 0;
        wait_bounded(base + OFF_BAR, 0, &no_abort, err, timeout_ns);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

}  // namespace nvfp4gg
