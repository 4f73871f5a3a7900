"""GPU parity of the NVFP4 activation encoder and the GEMM1 -> GEMM2 chain.

* nvfp4_quantize_bf16 against the oracle's quantize_nvfp4: codes and scale
  bytes bit-identical on seeded inputs (random magnitudes, zero, tiny,
  subnormal, midpoint and saturating blocks).
* nvfp4_grouped_gemm_nt_masked_swiglu_quant: its bf16 output bit-identical
  to the SwiGLU entry's; its NVFP4 output equal to nvfp4_quantize_bf16 of
  that bf16 output (one recipe, two kernels); decoded values within half an
  e2m1 step (at most d) of the oracle's pre-scaled SwiGLU output plus the
  GEMM tolerance; rows m >= masked_m[g] untouched.
* The chain: GEMM2 on those codes (alpha2 / q) element by element against
  the oracle GEMM on the same codes and scales (the GEMM tolerance), and
  against the oracle's fp64 chain without quantisation, within the NVFP4
  quantisation noise.
Calls go through the C-ABI."""
import numpy as np
import pytest

from oracle import oracle
from nvfp4_block_scaled_masked_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SENT = 0xAB   # prefill of the NVFP4 outputs


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_block_scaled_masked_gb300 import build, binding
    build.build()
    binding.load()
    assert binding.nvfp4_gg_check_error() == 0
    return binding


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_quantize(lib, x_bits, q, rows_per_scale):
    R, L = x_bits.shape
    codes = torch.full((R, L // 2), SENT, dtype=torch.uint8, device="cuda")
    sf = torch.full((R, L // 16), SENT, dtype=torch.uint8, device="cuda")
    lib.nvfp4_quantize_bf16(dev(x_bits.view(np.int16)), dev(np.asarray(q, np.float32)), codes, sf, R, L,
                            rows_per_scale)
    assert lib.nvfp4_gg_check_error() == 0
    return codes.cpu().numpy(), sf.cpu().numpy()


def bf16_pattern(rng, shape, exp_lo, exp_hi):
    sign = rng.integers(0, 2, shape).astype(np.uint16)
    exp = rng.integers(exp_lo, exp_hi + 1, shape).astype(np.uint16)
    return (sign << 15) | (exp << 7) | rng.integers(0, 128, shape).astype(np.uint16)


def special_rows(rng, R, L):
    """Rows of 16-element blocks of several kinds, block by block: random
    magnitudes, all zero, tiny (scale underflows to 0), bf16 subnormals,
    exact midpoints of the e2m1 grid times a power-of-two scale (ties), and
    blocks whose scale rounds down (codes saturate at 6)."""
    x = bf16_pattern(rng, (R, L), 118, 136).reshape(R, L // 16, 16)
    kind = rng.integers(0, 6, (R, L // 16))
    x[kind == 1] = 0
    x[kind == 2] = bf16_pattern(rng, x[kind == 2].shape, 30, 40)
    x[kind == 3] = bf16_pattern(rng, x[kind == 3].shape, 0, 1)
    mids = np.float32([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -2.5, -3.5, -5.0, 4.0, 0.5])
    n3 = int((kind == 4).sum())
    if n3:
        scale = np.float32(2.0) ** rng.integers(-8, 6, (n3, 1)).astype(np.float32)
        perm = np.argsort(rng.random((n3, 16)), axis=1)
        vals = (mids[perm] * scale).astype(np.float32)
        x[kind == 4] = (vals.view(np.uint32) >> 16).astype(np.uint16)
    n4 = int((kind == 5).sum())
    if n4:
        vals = np.full((n4, 16), 1.0, np.float32)
        vals[:, 0] = 6.25                               # amax / 6 = 1.04: scale 1.0, w = 6.25 -> 6
        x[kind == 5] = (vals.view(np.uint32) >> 16).astype(np.uint16)
    return x.reshape(R, L)


@pytest.mark.parametrize("R,L,rps,kind,qkind", [
    (37, 4096, 1, "random", "pow2"),
    (64, 2048, 16, "special", "pow2"),
    (64, 2048, 64, "special", "odd"),
    (3, 16, 3, "special", "one"),
    (1024, 7168, 8, "random", "odd"),
    (5, 7168, 1, "special", "odd"),
])
def test_quantize_matches_oracle(lib, R, L, rps, kind, qkind):
    rng = np.random.default_rng(R * 31 + L + rps)
    x = bf16_pattern(rng, (R, L), 110, 140) if kind == "random" else special_rows(rng, R, L)
    nq = (R + rps - 1) // rps
    if qkind == "pow2":
        q = np.float32(2.0) ** rng.integers(-12, -4, nq).astype(np.float32)
    elif qkind == "odd":
        q = rng.uniform(0.001, 0.05, nq).astype(np.float32)
    else:
        q = np.ones(nq, np.float32)
    codes, sf = gpu_quantize(lib, x, q, rps)
    q_row = np.repeat(q, rps)[:R]
    want_c, want_sf = oracle.quantize_nvfp4(x, q_row)
    np.testing.assert_array_equal(sf, want_sf)
    np.testing.assert_array_equal(codes, want_c)


def test_quantize_near_ties_for_every_scale(lib):
    """Quotients z / d at, and one to three float32 ulps around, every
    midpoint of the e2m1 grid, for every positive finite e4m3 scale d: each
    block's largest element is 6, so with the pre-scale q = d (1 + k 2^-23)
    the block scale is d and element m gives z / d ~ m (1 + k 2^-23).  Codes
    and scales must match the oracle's correctly rounded float32 division
    and e2m1 rounding bit for bit (the encoder divides through one rounded
    reciprocal per block and a residual correction)."""
    mids = np.float32([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0,
                       -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, 0.5])
    xb = (mids.view(np.uint32) >> 16).astype(np.uint16)          # exact in bf16
    ds = oracle.E4M3_TABLE[1:0x7F].astype(np.float64)             # 126 scales
    ks = np.arange(-3, 4, dtype=np.float64)
    q = (ds[:, None] * (1.0 + ks[None, :] * 2.0 ** -23)).astype(np.float32).ravel()
    x = np.tile(xb, (q.size, 1))
    codes, sf = gpu_quantize(lib, x, q, 1)
    want_c, want_sf = oracle.quantize_nvfp4(x, q)
    np.testing.assert_array_equal(sf, want_sf)
    np.testing.assert_array_equal(codes, want_c)


def test_block_scale_near_e4m3_midpoints(lib):
    """Blocks whose amax / 6 lies at, and one to three float32 ulps around,
    every midpoint between consecutive positive e4m3 values (and above the
    largest, where the scale saturates): scale bytes and codes bit for bit
    against the oracle's correctly rounded float32 quotient (the encoder
    divides by 6 through RN(1/6) and one residual correction).  Each block's
    largest magnitude is 6, so with the pre-scale q, amax / 6 ~ q."""
    vals = oracle.E4M3_TABLE[1:0x7F].astype(np.float64)          # 126 positive finite
    mids = np.concatenate([(vals[:-1] + vals[1:]) / 2.0, [464.0, 672.0]])
    ks = np.arange(-3, 4, dtype=np.float64)
    q = (mids[:, None] * (1.0 + ks[None, :] * 2.0 ** -23)).astype(np.float32).ravel()
    row = np.float32([6.0, -3.0, 1.5, -0.75, 0.5, 2.0, -6.0, 0.25,
                      4.0, -1.0, 3.0, 0.0, 5.0, -2.5, 1.0, -0.5])
    x = np.tile((row.view(np.uint32) >> 16).astype(np.uint16), (q.size, 1))
    codes, sf = gpu_quantize(lib, x, q, 1)
    want_c, want_sf = oracle.quantize_nvfp4(x, q)
    np.testing.assert_array_equal(sf, want_sf)
    np.testing.assert_array_equal(codes, want_c)


def _pow2_prescale(y_max):
    """Power of two that brings the block maxima near the top of the NVFP4
    range (448 * 6), from the oracle's output."""
    return np.float32(2.0) ** np.floor(np.log2(2688.0 / max(y_max, 1e-30))).astype(np.float32)


@pytest.mark.parametrize("case", ["narrow", "wide", "wide_pair", "decode_gemm1"])
def test_swiglu_quant_and_chain(lib, case):
    # "wide": the single-CTA prefill kernel (pair mode 0); "wide_pair": the
    # same shape on CTA pairs (automatic mode, N % 256 == 0)
    lib.nvfp4_gg_set_pair_mode(0 if case == "wide" else lib.PAIR_AUTO)
    try:
        _swiglu_quant_and_chain(lib, case)
    finally:
        lib.nvfp4_gg_set_pair_mode(lib.PAIR_AUTO)


def _swiglu_quant_and_chain(lib, case):
    if case == "narrow":
        d = W.generate(W.custom(3, 40, 512, 512, masked_m=[40, 0, 17]), seed=91)
    elif case in ("wide", "wide_pair"):
        d = W.generate(W.custom(2, 200, 512, 1024, masked_m=[200, 77]), seed=92)
    else:
        d = W.generate(W.CONFIGS["c2"])
    cfg = d["cfg"]
    G, M, N, K = cfg.G, cfg.M_max, cfg.N, cfg.K
    I = N // 2
    mm = d["masked_m"]
    valid = np.zeros((G, M), dtype=bool)
    for g in range(G):
        valid[g, :mm[g]] = True

    # oracle: GEMM1 in fp64, SwiGLU, per-expert power-of-two pre-scale
    _, ref64 = oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], mm, d["C_init"], G, M, N, K)
    _, y64 = oracle.swiglu(ref64, mm, np.full((G, M, I), W.SENTINEL_BF16, np.uint16))
    q = np.array([_pow2_prescale(np.nanmax(np.abs(y64[g, :mm[g]])) if mm[g] else 1.0) for g in range(G)],
                 np.float32)

    A, A_sf, B, B_sf = dev(d["A"]), dev(d["A_sf"]), dev(d["B"]), dev(d["B_sf"])
    alpha, mmd, qd = dev(d["alpha"]), dev(mm.astype(np.int32)), dev(q)
    bb, sb = lib.nvfp4_prepared_weight_bytes(G, N, K)
    Bp = torch.empty(bb, dtype=torch.uint8, device="cuda")
    Bsp = torch.empty(sb, dtype=torch.uint8, device="cuda")
    lib.nvfp4_prepare_weights_swiglu(B, B_sf, G, N, K, Bp, Bsp)

    C1 = torch.full((G, M, I), W.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    lib.nvfp4_grouped_gemm_nt_masked_swiglu(A, A_sf, Bp, Bsp, alpha, mmd, C1, G, M, N, K)
    C2 = torch.full((G, M, I), W.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    A2 = torch.full((G, M, I // 2), SENT, dtype=torch.uint8, device="cuda")
    A2sf = torch.full((G, M, I // 16), SENT, dtype=torch.uint8, device="cuda")
    lib.nvfp4_grouped_gemm_nt_masked_swiglu_quant(A, A_sf, Bp, Bsp, alpha, mmd, C2, qd, A2, A2sf, G, M, N, K)
    A2n = torch.full((G, M, I // 2), SENT, dtype=torch.uint8, device="cuda")
    A2sfn = torch.full((G, M, I // 16), SENT, dtype=torch.uint8, device="cuda")
    lib.nvfp4_grouped_gemm_nt_masked_swiglu_quant(A, A_sf, Bp, Bsp, alpha, mmd, None, qd, A2n, A2sfn,
                                                  G, M, N, K)
    assert lib.nvfp4_gg_check_error() == 0
    c1 = C1.cpu().numpy().view(np.uint16)
    c2 = C2.cpu().numpy().view(np.uint16)
    a2, a2sf = A2.cpu().numpy(), A2sf.cpu().numpy()

    # the bf16 output is the SwiGLU entry's; C = NULL changes nothing else
    np.testing.assert_array_equal(c2, c1)
    np.testing.assert_array_equal(A2n.cpu().numpy(), a2)
    np.testing.assert_array_equal(A2sfn.cpu().numpy(), a2sf)
    # rows past masked_m untouched
    assert np.all(a2[~valid] == SENT) and np.all(a2sf[~valid] == SENT)
    if not valid.any():
        return
    # one recipe: the fused codes are the standalone encoder's on C
    sc, ssf = gpu_quantize(lib, c2.reshape(G * M, I), q, M)
    np.testing.assert_array_equal(a2[valid], sc.reshape(G, M, I // 2)[valid])
    np.testing.assert_array_equal(a2sf[valid], ssf.reshape(G, M, I // 16)[valid])

    # against the oracle: decoded codes within d of q * y (plus the GEMM tolerance)
    dec = oracle.decode_numpy(a2[valid], a2sf[valid], I)
    dsc = np.repeat(oracle.E4M3_TABLE[a2sf[valid]], 16, axis=-1)
    qr = np.repeat(q[:, None], M, axis=1)[valid][:, None].astype(np.float64)
    yv = y64[valid]
    z = qr * yv
    slack = qr * (8e-3 * np.abs(yv) + 1e-4 * np.abs(yv).max())
    assert np.all(np.abs(dec - z) <= dsc * (1 + 1e-6) + slack)

    # the chain: GEMM2 (K = N/2) on the GPU's codes with alpha2 / q.  Element
    # by element against the oracle GEMM on those same codes and scales (the
    # GEMM's own tolerance), and, as a whole, within the NVFP4 quantisation
    # noise of the fp64 chain without quantisation
    N2 = 512
    d2 = W.generate(W.custom(G, M, N2, I, masked_m=list(mm)), seed=G + N2 + I)
    bb2, sb2 = lib.nvfp4_prepared_weight_bytes(G, N2, I)
    W2p = torch.empty(bb2, dtype=torch.uint8, device="cuda")
    W2sp = torch.empty(sb2, dtype=torch.uint8, device="cuda")
    lib.nvfp4_prepare_weights(dev(d2["B"]), dev(d2["B_sf"]), G, N2, I, W2p, W2sp)
    alpha2 = (d2["alpha"] / q).astype(np.float32)
    C3 = torch.full((G, M, N2), W.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    lib.nvfp4_grouped_gemm_nt_masked(A2, A2sf, W2p, W2sp, dev(alpha2), mmd, C3, G, M, N2, I)
    assert lib.nvfp4_gg_check_error() == 0
    c3 = C3.cpu().numpy().view(np.uint16)
    assert np.all(c3[~valid] == W.SENTINEL_BF16)
    init2 = np.full((G, M, N2), W.SENTINEL_BF16, np.uint16)
    _, ref2 = oracle.gemm(a2, a2sf, d2["B"], d2["B_sf"], alpha2, mm, init2, G, M, N2, I)
    got = (c3[valid].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r2 = ref2[valid]
    ok = oracle.tolerance_ok(got, r2, np.abs(r2).max())
    assert ok.all(), f"GEMM2: {(~ok).sum()} of {ok.size} outputs outside tolerance"
    W2d = oracle.decode_numpy(d2["B"].reshape(G, N2, I // 2), d2["B_sf"].reshape(G, N2, I // 16), I)
    for g in range(G):
        m = int(mm[g])
        if m == 0:
            continue
        ref = np.float64(d2["alpha"][g]) * (y64[g, :m] @ W2d[g].T)
        got_g = (c3[g, :m].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        rel = np.linalg.norm(got_g - ref) / np.linalg.norm(ref)
        assert rel < 0.2, f"expert {g}: relative RMS error {rel:.3f} against the unquantised chain"
