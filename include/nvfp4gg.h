/*
 * nvfp4gg — masked, block-scaled NVFP4 grouped GEMM-NT for GB300 (sm_103a).
 *
 * The operation is the one FlashInfer exposes as grouped_gemm_nt_masked, as
 * described on the page "The CuteDSL Gamble: Chasing Kernel Efficiency on
 * Blackwell GPUs" (sections "The Message" and "Output Knowledge Created"):
 * a masked, batched GEMM whose operands each come as (data, block scale
 * factors), with one valid-row count masked_m[g] per expert and an optional
 * alpha applied at the output.  For every expert g < G, every row
 * m < masked_m[g] and every n < N:
 *
 *     C[g][m][n] = bf16( alpha[g] * sum_{k<K} A[g][m][k] * B[g][n][k] )
 *
 * where each A/B element is an e2m1 (FP4) code times the e4m3 scale of its
 * 16-element block along K (sf_vec_size = 16, i.e. NVFP4).  "NT" means both
 * operands are K-major: A is [G][M_max][K], B is [G][N][K].  Rows of C at or
 * past masked_m[g] are never written.
 *
 * Encodings (the pages name NVFP4 but do not define it; these are the OCP
 * Microscaling readings):
 *   e2m1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa; two codes
 *         per byte, element k of a row in byte k/2, even k in the low nibble.
 *   e4m3: one byte per 16 K-elements, positive finite values (bit 7 clear,
 *         not 0x7F).
 *   C:    bf16, round to nearest even.
 *
 * Conventions for every call:
 *   - All buffers are owned by the caller, except the static scratch of
 *     nvfp4_grouped_gemm_nt_masked_splitk_noalloc.  The library allocates no
 *     device memory in any call.
 *   - Device pointers must be 16-byte aligned (alpha and masked_m: 4-byte).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and never synchronise the host, except
 *     nvfp4_gg_check_error.  masked_m is never read on the host.
 *   - Every entry point checks its arguments on the host first and returns a
 *     negative nvfp4gg_status without launching anything when they are bad.
 *   - Calls on one stream are thread-compatible; the SM cap set by
 *     nvfp4_gg_set_sm_count is process-wide.
 *   - Per device the library looks up, on its first call there, the device
 *     addresses of its static __device__ arrays (error word, signal
 *     counters, split-K scratch), sets its kernels' shared-memory limits and
 *     caches tensor maps; it keeps all of it until nvfp4_gg_shutdown.  A
 *     cudaDeviceReset invalidates it: call nvfp4_gg_shutdown after resetting
 *     a device before calling into the library there again.
 */
#ifndef NVFP4GG_H
#define NVFP4GG_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4GG_OK = 0,
    NVFP4GG_ERR_NULL = -1,      /* a required pointer is NULL                        */
    NVFP4GG_ERR_SHAPE = -2,     /* G, M_max, N or K outside the supported set         */
    NVFP4GG_ERR_ALIGN = -3,     /* a pointer is not aligned as required              */
    NVFP4GG_ERR_ARCH = -4,      /* the current device is not compute capability 10.3 */
    NVFP4GG_ERR_CUDA = -5,      /* a CUDA runtime/driver call failed                 */
    NVFP4GG_ERR_TIMEOUT = -6,   /* a device-side wait ran past its limit (error word) */
    NVFP4GG_ERR_MASK = -7,      /* masked_m[g] outside [0, M_max] seen on the device  */
    NVFP4GG_ERR_SCRATCH = -8    /* split needs more than the library's static scratch */
} nvfp4gg_status;

/* Shape limits of nvfp4_grouped_gemm_nt_masked. */
#define NVFP4GG_MAX_GROUPS 1024   /* 1 <= G <= 1024                                  */
#define NVFP4GG_K_ALIGN 256       /* K % 256 == 0 (a 16-byte row of A_sf per 256 K)   */
#define NVFP4GG_N_ALIGN 16        /* N % 16 == 0                                      */

/*
 * Sizes of the prepared weight buffers that nvfp4_prepare_weights writes.
 *   *b_bytes  = G * ceil(N/128) * 128 * K / 2        (codes, tiled)
 *   *sf_bytes = G * ceil(N/128) * (K/64) * 512       (scales in MMA atom order)
 * Returns NVFP4GG_OK or NVFP4GG_ERR_NULL / NVFP4GG_ERR_SHAPE.
 */
int nvfp4_prepared_weight_bytes(int G, int N, int K, size_t* b_bytes, size_t* sf_bytes);

/*
 * One-time weight re-layout (run once per weight set, outside the timed GEMM).
 *   B         device u8 [G][N][K/2]   e2m1 codes, K-major
 *   B_sf      device u8 [G][N][K/16]  e4m3 scales, row-major
 *   B_prep    device, b_bytes: the codes as contiguous 16384-byte tiles, one
 *             per (expert g, 128-row block nb, 256-element K block ks), in
 *             that order; tile byte r*128 + 16*(c ^ (r % 8)) + i holds byte
 *             128*ks + 16*c + i of row 128*nb + r (the 128-byte swizzle the
 *             tensor core reads; zero past row N)
 *   B_sf_prep device, sf_bytes: the scales regrouped into 512-byte atoms, one
 *             per (expert, 128-row block of N, 64-element block of K): byte
 *             (i*16 + j*4 + b) of an atom holds the scale of row
 *             128*nb + 32*j + i and K block 4*kc + b (zero past row N)
 * Asynchronous on `stream`.  The outputs must not alias the inputs
 * (NVFP4GG_ERR_SHAPE otherwise).
 */
int nvfp4_prepare_weights(const void* B, const void* B_sf, int G, int N, int K,
                          void* B_prep, void* B_sf_prep, void* stream);

/*
 * The grouped GEMM.
 *   A        device u8 [G][M_max][K/2]   e2m1 activations (rows >= masked_m[g]
 *            may hold anything, including NaN scales; they are ignored)
 *   A_sf     device u8 [G][M_max][K/16]  e4m3 activation scales, row-major
 *   B        device, prepared codes  (nvfp4_prepare_weights)
 *   B_sf     device, prepared scales (nvfp4_prepare_weights)
 *   alpha    device f32 [G]
 *   masked_m device i32 [G], 0 <= masked_m[g] <= M_max (values outside are
 *            clamped and flagged NVFP4GG_ERR_MASK in the error word)
 *   C        device bf16 [G][M_max][N], row-major; rows m >= masked_m[g] keep
 *            their previous contents bit for bit
 * Limits: 1 <= G <= NVFP4GG_MAX_GROUPS, M_max >= 1, N % 16 == 0,
 * K % 256 == 0.  Asynchronous on `stream`; device-side failures (a wait past
 * its time limit, a bad masked_m) are recorded in the error word read by
 * nvfp4_gg_check_error.
 * Decode calls (M_max <= 64) with K >= 6144 and at most SMs/4 weight tiles
 * (G * ceil(M_max/32) * ceil(N/128), every expert counted full) split K as
 * nvfp4_grouped_gemm_nt_masked_splitk with split_k = 0 does, reducing within
 * thread-block clusters (no workspace); the result is deterministic and
 * agrees with an unsplit call up to fp32 summation order.
 */
int nvfp4_grouped_gemm_nt_masked(const void* A, const void* A_sf, const void* B,
                                 const void* B_sf, const float* alpha, const int* masked_m,
                                 void* C, int G, int M_max, int N, int K, void* stream);

/*
 * Split-K variant for decode-sized calls (M_max <= 64), the swap-AB path's
 * split-K: each weight tile's K range is cut into split_k contiguous ranges
 * computed by different CTAs, and their fp32 partials are summed in range
 * order (so results are deterministic), scaled by alpha and stored as bf16.
 * This keeps more SMs streaming weights when there are fewer weight tiles
 * than SMs (few non-empty experts, small N).  Up to 8 ranges run as one
 * thread-block cluster per tile and reduce through distributed shared
 * memory: the workspace is then not touched.  Larger splits, or an SM cap
 * (nvfp4_gg_set_sm_count) below the split, reduce through the workspace:
 * the last range of a tile to finish sums the partials.  Both reductions
 * add in the same order, so they give the same bits.
 *   split_k    1..16, or 0 to choose from the tile count: floor(SMs / tiles),
 *              at most 6 and at most K/1024
 *   workspace  device scratch owned by the caller, 256-byte aligned, at least
 *              nvfp4_splitk_workspace_bytes(G, M_max, N, K, split_k) bytes
 *              (fp32 partials, then one 8-byte arrival counter per tile);
 *              it needs no initial value and no clearing between calls (the
 *              counters are tagged with a number unique to each call); calls
 *              that run at the same time must not share it
 * Other arguments as in nvfp4_grouped_gemm_nt_masked.  With M_max > 64 the
 * call runs unsplit and the workspace is not touched.  Results agree with the
 * unsplit call up to fp32 summation order.
 */
size_t nvfp4_splitk_workspace_bytes(int G, int M_max, int N, int K, int split_k);
int nvfp4_grouped_gemm_nt_masked_splitk(const void* A, const void* A_sf, const void* B,
                                        const void* B_sf, const float* alpha, const int* masked_m,
                                        void* C, int G, int M_max, int N, int K, int split_k,
                                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Split-K without a caller workspace.  This entry point has no counterpart
 * on the pages that define the operation; it exists for callers that cannot
 * allocate device memory at call time: a serving loop that has handed all of
 * HBM to weights and KV cache before it starts, code that must not hit the
 * device-wide synchronisation of cudaFree, or a C caller with no device
 * allocator of its own.  It allocates nothing.  It computes exactly what
 * nvfp4_grouped_gemm_nt_masked_splitk computes with the same split (the same
 * kernel and reduction order, so the same bits), using a scratch buffer that
 * is a static __device__ array of the library, reserved once per device when
 * the library's module is loaded there:
 *   NVFP4GG_NOALLOC_MAX_SLOTS fp32 partial tiles of 32 x 128 (16 KiB each,
 *   4 MiB in all) plus one 8-byte arrival counter per slot (2 KiB).
 * A split call uses tiles x split slots, tiles = G * ceil(M_max/32) *
 * ceil(N/128) (every expert counted full); a split the cluster reduction
 * takes (up to 8 ranges, see nvfp4_grouped_gemm_nt_masked_splitk) leaves the
 * scratch untouched, but the slot limit below applies all the same.
 *   split_k  0: the automatic split of the workspace variant, lowered until
 *               tiles x split fits the scratch (1 = unsplit when even 2 does
 *               not fit);
 *            1: unsplit, the scratch is not touched;
 *            2..16: that split (capped at K/256); NVFP4GG_ERR_SCRATCH, with
 *               nothing launched, when tiles x split exceeds
 *               NVFP4GG_NOALLOC_MAX_SLOTS.
 * With M_max > 64 the call runs unsplit.  Other arguments as in
 * nvfp4_grouped_gemm_nt_masked.
 * State: neither the partials nor the counters need an initial value or
 * clearing between calls: every call tags the counters it uses with a
 * number unique to the call (the first arrival of a call restarts a counter
 * that holds another call's number), so a call that ended in a device-side
 * timeout leaves nothing for the next call to clean up.  Nothing besides
 * the GEMM kernel is launched.
 * The first call on a device looks up the scratch's device address
 * (cudaGetSymbolAddress) and sets the kernel's shared-memory limit: make one
 * call on each device before capturing a stream.
 * Calls that may run at the same time on one device (different streams, or
 * host threads that do not order their calls) share the scratch and race on
 * it: their results are undefined.  Order them on one stream, or give each
 * stream its own workspace through nvfp4_grouped_gemm_nt_masked_splitk.
 */
#define NVFP4GG_NOALLOC_MAX_SLOTS 256
int nvfp4_grouped_gemm_nt_masked_splitk_noalloc(const void* A, const void* A_sf, const void* B,
                                                const void* B_sf, const float* alpha,
                                                const int* masked_m, void* C, int G, int M_max,
                                                int N, int K, int split_k, void* stream);

/*
 * W4A16 GEMV for decode: NVFP4 weights, bf16 activations, the "nvfp4_gemv"
 * workload (W4A16) in the kernel table of the page listing Helion's
 * pretuned_kernels directory (a one-token decode GEMV over model
 * projection shapes).  For m < M, n < N:
 *     y[m][n] = bf16( alpha[0] * sum_k x[m][k] * B[n][k] )     (fp32 accumulation)
 *   x      device bf16 [M][K], 16-byte aligned
 *   B      device u8 [N][K/2] e2m1 codes, the raw row-major layout (no
 *          nvfp4_prepare_weights), 16-byte aligned
 *   B_sf   device u8 [N][K/16] e4m3 scales, row-major
 *   alpha  device f32 [1]
 *   y      device bf16 [M][N]
 * Limits: 1 <= M <= 8, K % 32 == 0, M * K <= 71493 (the tokens are staged
 * in shared memory, 2.75 bytes per value), N <= 2^24.  The W4A4 form (NVFP4 activations)
 * is nvfp4_grouped_gemm_nt_masked with G = 1.
 */
int nvfp4_gemv_w4a16(const void* x, const void* B, const void* B_sf, const float* alpha, void* y,
                     int M, int N, int K, void* stream);

/*
 * The GEMM on the packed-rows ("contiguous") grouped layout: the activations
 * and the output hold only valid rows, expert after expert, instead of M_max
 * rows per expert.  Expert g's rows start at row off[g] = masked_m[0] + ... +
 * masked_m[g-1] (computed on the device from masked_m).
 *   A        device u8 [M_total][K/2], A_sf device u8 [M_total][K/16]
 *   C        device bf16 [M_total][N]; rows off[g] .. off[g] + masked_m[g] - 1
 *            are written, no other row
 *   M_max    bound on every masked_m[g] (picks the kernel family; values above
 *            it are clamped and flagged NVFP4GG_ERR_MASK), M_max <= M_total
 *   M_total  rows of A, A_sf and C (1 .. 2^24); a sum of masked_m above it is
 *            flagged NVFP4GG_ERR_MASK and rows past M_total are not written
 * Other arguments as in nvfp4_grouped_gemm_nt_masked (same prepared weights).
 * The pages name this layout for a grouped baseline (DeepGEMM's contiguous
 * grouped GEMM, in the kernel table of the page listing Helion's
 * pretuned_kernels directory); the operation is the same.
 */
int nvfp4_grouped_gemm_nt_contiguous(const void* A, const void* A_sf, const void* B,
                                     const void* B_sf, const float* alpha, const int* masked_m,
                                     void* C, int G, int M_max, int M_total, int N, int K,
                                     void* stream);

/*
 * The GEMM with per-expert completion signals: the dst_signals argument of
 * grouped_gemm_nt_masked on "The CuteDSL Gamble: Chasing Kernel Efficiency
 * on Blackwell GPUs" ("The Message"), whose behaviour the page does not
 * describe (reading taken: a consumer may start on expert g as soon as its
 * output is complete, without waiting for the whole call).
 *   dst_signals  device i32 [G], owned by the caller.  Each call increments
 *                dst_signals[g] by exactly 1 after every valid row of expert
 *                g's C has been stored, a device-scope fence in between;
 *                experts with masked_m[g] = 0 are signalled at kernel start.
 *                A consumer that sees the new value must load C with
 *                acquire ordering (or fence) before reading it.
 * Other arguments as in nvfp4_grouped_gemm_nt_masked; runs on the single-CTA
 * kernels.  The per-expert counters behind the signals are a static array of
 * the library (NVFP4GG_MAX_GROUPS 8-byte counters per device), tagged with
 * a number unique to each call (no clearing between calls): calls of this
 * entry point that overlap on one device race on them.
 */
int nvfp4_grouped_gemm_nt_masked_signals(const void* A, const void* A_sf, const void* B,
                                         const void* B_sf, const float* alpha, const int* masked_m,
                                         void* C, int G, int M_max, int N, int K, int* dst_signals,
                                         void* stream);

/*
 * GEMM1 of an MoE expert block with its SwiGLU activation fused into the
 * epilogue: the step that follows this GEMM on the page "LLM-Assisted Kernel
 * Development in CuTe DSL, Gluon, Helion and Triton" (mixture-of-experts
 * section: each expert runs GEMM1, then SwiGLU, then GEMM2; I = 2048).  B is GEMM1's
 * weight [G][N][K] with N = 2 I: rows 0 .. I-1 the gate projection, rows
 * I .. 2I-1 the up projection (the page does not fix the order; this is the
 * reading taken).  For m < masked_m[g] and j < I:
 *     h(row)     = alpha[g] * sum_k A[g][m][k] * B[g][row][k]   (fp32 accumulation)
 *     C[g][m][j] = bf16( silu(h(j)) * h(I + j) ),   silu(x) = x / (1 + e^-x)
 * C is bf16 [G][M_max][N/2], row-major; rows m >= masked_m[g] are never
 * written.  B and B_sf must come from nvfp4_prepare_weights_swiglu (same
 * sizes as nvfp4_prepare_weights), which interleaves gate and up rows so that
 * one weight tile holds both halves of the outputs it produces.  N % 128 == 0
 * (NVFP4GG_ERR_SHAPE otherwise); other arguments and limits as in
 * nvfp4_grouped_gemm_nt_masked.  Runs on the single-CTA kernels (no CTA
 * pairs, no split-K).
 */
int nvfp4_prepare_weights_swiglu(const void* B, const void* B_sf, int G, int N, int K,
                                 void* B_prep, void* B_sf_prep, void* stream);
int nvfp4_grouped_gemm_nt_masked_swiglu(const void* A, const void* A_sf, const void* B,
                                        const void* B_sf, const float* alpha, const int* masked_m,
                                        void* C, int G, int M_max, int N, int K, void* stream);

/*
 * Dual GEMM: two GEMMs that share the activation operand A, with separate
 * weights B1 (gate) and B2 (up) -- the "NVFP4 dual GEMM" problem of the page
 * "LLM-Assisted Kernel Development in CuTe DSL, Gluon, Helion and Triton"
 * (one A tile feeding two B operands; the page's derivation stacks the two
 * B operands).  This one-time re-layout writes the prepared weights of the
 * stacked operand straight from the two separate ones, so the caller never
 * builds [B1; B2] itself:
 *   B1, B2        device u8 [G][N1][K/2]   e2m1 codes of each operand
 *   B1_sf, B2_sf  device u8 [G][N1][K/16]  their e4m3 scales
 *   interleave 0: the layout of nvfp4_prepare_weights for the stacked
 *                 weight [B1; B2] (N = 2 N1): nvfp4_grouped_gemm_nt_masked
 *                 with N = 2 N1 then writes C[g][m][0 .. N1-1] = A B1^T and
 *                 C[g][m][N1 .. 2N1-1] = A B2^T (each times alpha[g])
 *   interleave 1: the layout of nvfp4_prepare_weights_swiglu for the same
 *                 stacked weight (needs N1 % 64 == 0):
 *                 nvfp4_grouped_gemm_nt_masked_swiglu (and _swiglu_quant)
 *                 with N = 2 N1 then writes silu(alpha A B1^T) * (alpha A B2^T)
 *   B_prep, B_sf_prep  outputs, sized by nvfp4_prepared_weight_bytes(G, 2 N1, K)
 * The bytes written equal those of nvfp4_prepare_weights(_swiglu) on the
 * stacked weight.  Limits: N1 % 16 == 0, 2 N1 within the GEMM's N limits,
 * K % 256 == 0; the outputs must not overlap any input (NVFP4GG_ERR_SHAPE).
 * Asynchronous on `stream`.
 */
int nvfp4_prepare_weights_dual(const void* B1, const void* B1_sf, const void* B2,
                               const void* B2_sf, int G, int N1, int K, int interleave,
                               void* B_prep, void* B_sf_prep, void* stream);

/*
 * NVFP4 encoding of bf16 activations, GEMM2's A after the SwiGLU step (the
 * MoE expert block of the page "LLM-Assisted Kernel Development in CuTe DSL,
 * Gluon, Helion and Triton" runs GEMM1, SwiGLU, GEMM2 per expert; the pages
 * give no quantisation recipe, so this is the reading).  Per 16-element
 * block of a row, in fp32 with round-to-nearest-even:
 *     z_i = x_i * q;  sf = e4m3(max|z_i| / 6) (saturating at 448);
 *     d = value(sf);  code_i = e2m1(z_i / d) (saturating at 6), 0 if d == 0
 * so x_i ~ code_i * d / q: a GEMM2 on these codes takes alpha / q.  Zero
 * codes are written as +0.
 *   x        device bf16 [R][L] row-major, 16-byte aligned, finite
 *   qscale   device f32; row r uses qscale[r / rows_per_scale]
 *            (rows_per_scale = R: one per tensor; = M_max: one per expert)
 *   codes    device u8 [R][L/2] (low nibble = even element), 8-byte aligned
 *   sf       device u8 [R][L/16]
 * Limits: R >= 1, L % 16 == 0, R * L <= 2^40.  The layouts match A and
 * A_sf of nvfp4_grouped_gemm_nt_masked (K = L).
 */
int nvfp4_quantize_bf16(const void* x, const float* qscale, void* codes, void* sf, int R, int L,
                        int rows_per_scale, void* stream);

/*
 * nvfp4_grouped_gemm_nt_masked_swiglu whose epilogue also encodes its bf16
 * output as NVFP4 for GEMM2, by the recipe of nvfp4_quantize_bf16 with one
 * pre-scale per expert: the codes are those nvfp4_quantize_bf16 gives for
 * the bf16 values C holds (rows_per_scale = M_max).
 *   C        bf16 [G][M_max][N/2] as in the SwiGLU entry, or NULL (then only
 *            the NVFP4 output is written)
 *   qscale   device f32 [G], expert g's pre-scale
 *   A2       device u8 [G][M_max][N/4], 16-byte aligned: GEMM2's A codes
 *   A2_sf    device u8 [G][M_max][N/32]: GEMM2's A_sf
 * Rows m >= masked_m[g] of C, A2 and A2_sf are never written.  GEMM2 is then
 * nvfp4_grouped_gemm_nt_masked(A2, A2_sf, W2 prepared, ..., K = N/2) with
 * alpha2[g] / qscale[g].  Other arguments and limits as in the SwiGLU entry.
 */
int nvfp4_grouped_gemm_nt_masked_swiglu_quant(const void* A, const void* A_sf, const void* B,
                                              const void* B_sf, const float* alpha,
                                              const int* masked_m, void* C, const float* qscale,
                                              void* A2, void* A2_sf, int G, int M_max, int N, int K,
                                              void* stream);

/*
 * End-to-end variant for callers whose activations live in host memory.
 *   h_A, h_A_sf, h_alpha, h_masked_m: HOST buffers laid out as above (pinned
 *       memory gives asynchronous copies)
 *   B, B_sf: DEVICE prepared weights
 *   h_C: HOST bf16 [G][M_max][N]; only rows m < h_masked_m[g] are written
 *   d_staging: DEVICE scratch of at least nvfp4_host_staging_bytes(...) bytes,
 *       16-byte aligned, owned by the caller
 * Copies h_A and h_A_sf host->device, runs the GEMM and delivers the valid
 * rows of C, all on `stream`.  Buffers in pinned (page-locked) host memory,
 * which the device can address, are used in place: the kernel reads h_alpha
 * and h_masked_m directly, and its epilogue stores the valid rows of C
 * straight into h_C (16-byte aligned) over the CPU-GPU link.  Pageable
 * buffers go through d_staging instead: one copy each for alpha and
 * masked_m, and one device->host copy of C per non-empty expert.  Calls with
 * M_max > 64 and at least 2 MiB of activations copy them in 2 to 4 expert
 * chunks of growing size (1 : 4 : 16 : 64) on a library-owned stream, each
 * chunk's GEMM waiting (by an event) for its own copy only, so that later
 * chunks cross the link while earlier ones compute; the copies wait for the
 * work queued on `stream` before the call, and the results equal the
 * unchunked call's bit for bit.  Returns
 * when the work is queued; synchronise `stream` (which then covers the
 * side stream's copies) before reading h_C, and do not modify the inputs
 * before then.  While `stream` is being captured into a CUDA graph, no
 * other thread may call this entry point with a chunked shape.
 */
size_t nvfp4_host_staging_bytes(int G, int M_max, int N, int K);
int nvfp4_grouped_gemm_nt_masked_host(const void* h_A, const void* h_A_sf,
                                      const float* h_alpha, const int* h_masked_m,
                                      const void* B, const void* B_sf, void* h_C,
                                      int G, int M_max, int N, int K,
                                      void* d_staging, size_t staging_bytes, void* stream);

/*
 * Caps the number of SMs (persistent CTAs) a GEMM launch uses; 0 = all SMs.
 * This is the sm_count argument of grouped_gemm_nt_masked on the same page
 * ("The Message").  Process-wide.  Returns NVFP4GG_ERR_SHAPE if negative.
 */
int nvfp4_gg_set_sm_count(int sm_count);

/*
 * Kernel family for experts with M_max > 64 (prefill sizes).
 *   mode 0: one CTA per 128 weight rows (token tiles of up to 192).
 *   mode 1: when N is a multiple of 256, the two CTAs of a 2-CTA cluster
 *           share one MMA of 256 weight rows (each CTA stages 128 weight
 *           rows and half of the token rows).
 *   mode 2 (default): automatic.  N % 256 == 0 and M_max <= 256: mode 1;
 *           N % 256 == 0 and M_max > 256: mode 3; else mode 0.  Measured on
 *           GB300: pairs are ~8 % faster on bandwidth-bound prefill shapes
 *           (few token tiles per expert); compute-heavy experts run fastest
 *           on the token-major pairs.
 *   mode 3: when N is a multiple of 256 and M_max >= 128, token-major CTA
 *           pairs: one MMA of 256 tokens (128 per CTA) by 256 weight rows,
 *           for experts with many valid rows.
 * Calls with per-expert signals, the SwiGLU epilogue or the packed-rows
 * layout, and calls capped to one SM, run on the single-CTA kernels.
 * Results are equal up to fp32 summation order.  Process-wide.
 * NVFP4GG_ERR_SHAPE unless 0, 1, 2 or 3.
 */
int nvfp4_gg_set_pair_mode(int mode);

/*
 * Drops every host-side cache of the library: per-device state (SM count,
 * error-word and scratch addresses, kernel attributes, cluster fits) and
 * the tensor-map caches, and forgets the host-buffer entry's side stream
 * and events without destroying them (after a cudaDeviceReset they are
 * gone with the context; otherwise the context releases them when it is
 * destroyed).  The library holds no device allocation, so nothing is freed
 * on the device; the next call on a device sets it up again.  Call it after
 * a cudaDeviceReset, or when done with the library.  It must not run while
 * another thread is inside a library call.  Returns NVFP4GG_OK.
 */
int nvfp4_gg_shutdown(void);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns NVFP4GG_OK, NVFP4GG_ERR_TIMEOUT, NVFP4GG_ERR_MASK, or
 * NVFP4GG_ERR_CUDA if a CUDA call failed.
 */
int nvfp4_gg_check_error(void* stream);

/*
 * Launches one CTA that waits on a barrier nothing ever completes, with the
 * same bounded-wait code the GEMM uses and the given limit in nanoseconds
 * (1e3 .. 1e10).  The wait gives up, records NVFP4GG_ERR_TIMEOUT in the
 * error word and the kernel returns; nvfp4_gg_check_error then reports it.
 * Used to test the watchdog without faulting or hanging the GPU.
 */
int nvfp4_gg_selftest_watchdog(long long timeout_ns, void* stream);

/*
 * Tensor-pipe throughput probe (measurement only; computes nothing useful).
 * Launches `ctas` CTAs (0 = one per SM), each issuing iters x 4 block-scaled
 * NVFP4 MMAs of M = 128, N = n (16..256, multiple of 16), K = 64 on resident
 * shared-memory operands.  FLOPs of one launch: ctas * iters * 4 * 2*128*n*64.
 * Time it with events on `stream` to get the dense NVFP4 tensor rate.
 */
int nvfp4_gg_mma_peak_probe(int iters, int n, int ctas, void* stream);

/*
 * The same probe for CTA pairs (tcgen05 cta_group::2, the two SMs of a 2-CTA
 * cluster sharing one MMA): `clusters` clusters (0 = one per pair of SMs),
 * each issuing iters x 4 block-scaled NVFP4 MMAs of M = 256, N = n (16..256,
 * multiple of 16), K = 64 from the leader CTA.  FLOPs of one launch:
 * clusters * iters * 4 * 2*256*n*64.  The pair form is the one the pages'
 * Blackwell grouped kernels use for large tiles ("LLM-Assisted Kernel
 * Development in CuTe DSL, Gluon, Helion and Triton", NVFP4 grouped GEMM).
 */
int nvfp4_gg_mma_peak_probe_pair(int iters, int n, int clusters, void* stream);

/* Human-readable name of a status code (static string). */
const char* nvfp4_gg_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4GG_H */
