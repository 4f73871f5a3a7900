"""GPU parity over the whole NVFP4 input domain, element by element.

The seeded benchmark workloads draw scale bytes from seven powers of two and
leave out the negative-zero code.  Here every e2m1 code (0x8 = -0 included)
and every finite non-negative e4m3 scale byte 0x00..0x7E (zero, the
subnormals 0x01..0x07, mantissa bits, up to 448) reach the tensor cores of
each kernel family: the decode kernel (token tiles of 32), the 192-wide
single-CTA kernel, the CTA-pair kernel and the token-major CTA-pair kernel,
including K = 7168.  Scale
regimes run as separate calls (all bytes; subnormal x subnormal; subnormal x
large; large x large), so a kernel that mis-decoded subnormal or large scales
could not hide behind the tolerance's absolute term (1e-4 of the call's
largest output).  The operand encodings are the OCP Microscaling ones the
page "The CuteDSL Gamble: Chasing Kernel Efficiency on Blackwell GPUs" names
for grouped_gemm_nt_masked ("The Message": NVFP4 operands with one e4m3
scale per 16 elements, sf_vec_size = 16).

Bar: |gpu - ref| <= 4e-3 |ref| + 1e-4 max|ref| per output, ref the oracle's
unrounded fp64 value; rows m >= masked_m[g] bit-identical to the 0x7FC0
prefill."""
import numpy as np
import pytest

from oracle import oracle
from nvfp4_block_scaled_masked_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

REGIMES = [("all", "all"), ("subnormal", "subnormal"), ("subnormal", "large"),
           ("large", "large")]


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_block_scaled_masked_gb300 import build, binding
    build.build()
    binding.load()
    assert binding.nvfp4_gg_check_error() == 0
    return binding


def _check(d, C_gpu):
    cfg = d["cfg"]
    _, ref = oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], d["masked_m"],
                         d["C_init"], cfg.G, cfg.M_max, cfg.N, cfg.K)
    mm = d["masked_m"]
    valid = np.zeros((cfg.G, cfg.M_max), dtype=bool)
    for g in range(cfg.G):
        valid[g, :mm[g]] = True
    assert np.all(C_gpu[~valid] == W.SENTINEL_BF16), "rows >= masked_m were written"
    vals = (C_gpu[valid].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = ref[valid]
    assert np.all(np.isfinite(vals))
    max_abs = np.abs(r).max()
    assert max_abs > 0
    ok = oracle.tolerance_ok(vals, r, max_abs)
    if not ok.all():
        bad = np.flatnonzero(~ok.ravel())
        pytest.fail(f"{bad.size} of {ok.size} outside tolerance; first gpu "
                    f"{vals.ravel()[bad[:4]]} ref {r.ravel()[bad[:4]]} (max {max_abs:g})")
    return vals, r


def _run(lib, d, pair_mode):
    from nvfp4_block_scaled_masked_gb300.device import Problem
    lib.nvfp4_gg_set_pair_mode(pair_mode)
    try:
        prob = Problem(d)
        prob.run()
        rc = lib.nvfp4_gg_check_error()
        assert rc == 0, lib.status_string(rc)
        return prob.C_bits()
    finally:
        lib.nvfp4_gg_set_pair_mode(lib.PAIR_AUTO)


# (kernel family, G, M_max, N, K, masked_m, pair mode)
SHAPES = [
    ("decode", 3, 16, 384, 7168, [16, 5, 0], 2),
    ("decode", 2, 64, 272, 1024, [64, 37], 2),
    ("wide", 2, 192, 384, 2048, [192, 77], 0),
    ("wide", 2, 200, 512, 7168, [200, 129], 0),
    ("pair", 2, 200, 512, 7168, [200, 129], 1),
    ("pair", 3, 256, 768, 1024, [256, 31, 0], 1),
    ("token-major pair", 2, 300, 512, 7168, [300, 129], 3),
]


@pytest.mark.parametrize("a_sc,b_sc", REGIMES)
@pytest.mark.parametrize("kind,G,M_max,N,K,masked,pair", SHAPES)
def test_full_domain_parity(lib, kind, G, M_max, N, K, masked, pair, a_sc, b_sc):
    cfg = W.custom(G, M_max, N, K, masked_m=masked)
    seed = 7919 * G + 31 * N + K + 1009 * REGIMES.index((a_sc, b_sc))
    d = W.generate_full_range(cfg, seed, a_sc, b_sc)
    _check(d, _run(lib, d, pair))


def test_negative_zero_codes_and_zero_scales(lib):
    """Every code -0 (0x8) in one expert, every scale 0x00 in another, a
    single non-zero element in a third: the first two give exact zeros, the
    third the one product."""
    cfg = W.custom(3, 32, 256, 512, masked_m=[32, 32, 1])
    d = W.generate_full_range(cfg, 5, "all", "all")
    d["A"][0] = 0x88
    d["B_sf"][1] = 0x00
    d["A"][2] = 0
    d["A"][2, 0, 100] = 0x70           # element 201 of row 0: code 0x7 (= 6)
    d["A_sf"][2, 0, 201 // 16] = 0x7E  # 448
    C = _run(lib, d, 2)
    vals = (C.astype(np.uint32) << 16).view(np.float32)
    assert np.all(vals[0] == 0) and np.all(vals[1] == 0)
    _check(d, C)
    # expert 2, row 0: alpha * 6 * 448 * b(n, 201), a single product; the
    # kernel rounds alpha * acc to fp32 and then to bf16, so it may differ
    # from the one fp64 -> bf16 rounding by one bf16 unit on a tie
    b_codes = d["B"][2, :, 100] >> 4
    b_val = oracle.E2M1_TABLE[b_codes] * oracle.E4M3_TABLE[d["B_sf"][2, :, 201 // 16]]
    want = np.float64(d["alpha"][2]) * 6.0 * 448.0 * b_val
    got = vals[2, 0].astype(np.float64)
    assert np.all((want == 0) == (got == 0))
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want))
