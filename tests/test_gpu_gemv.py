"""GPU parity of the W4A16 decode GEMV (nvfp4_gemv_w4a16) against the oracle:
every output within |gpu - ref| <= 4e-3 |ref| + 1e-4 max|ref| of the fp64
value, most of them the correctly rounded bf16; two calls bit-identical."""
import numpy as np
import pytest

from oracle import oracle
from nvfp4_block_scaled_masked_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_block_scaled_masked_gb300 import build, binding
    build.build()
    binding.load()
    assert binding.nvfp4_gg_check_error() == 0
    return binding


def run(lib, d):
    cfg = d["cfg"]
    M, N, K = cfg.M_max, cfg.N, cfg.K
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    x = dev(d["x"].view(np.int16))
    B, Bsf, al = dev(d["B"]), dev(d["B_sf"]), dev(d["alpha"])
    outs = []
    for _ in range(2):
        y = torch.full((M, N), W.SENTINEL_BF16, dtype=torch.int16, device="cuda")
        lib.nvfp4_gemv_w4a16(x, B, Bsf, al, y, M, N, K)
        assert lib.nvfp4_gg_check_error() == 0
        outs.append(y.cpu().numpy().view(np.uint16))
    np.testing.assert_array_equal(outs[0], outs[1])
    return outs[0]


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (3, 1000, 2048), (8, 130, 4096), (1, 37, 32),
                                   (2, 4096, 14336), (1, 7, 256), (4, 5000, 1024), (5, 153, 768),
                                   (1, 151, 2304)])
def test_gemv_matches_oracle(lib, M, N, K):
    cfg = W.Config("v0", f"gemv {M}x{N}x{K}", 1, M, N, K, "fixed", masked_list=(M,),
                   kind="gemv_w4a16")
    d = W.generate_gemv(cfg, seed=M * 1000 + N + K)
    y = run(lib, d)
    bits, ref = oracle.gemv_w4a16(d["x"], d["B"], d["B_sf"], d["alpha"][0], K)
    vals = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ok = oracle.tolerance_ok(vals, ref, np.abs(ref).max())
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside tolerance"
    assert np.mean(y == bits) > 0.9


def test_gemv_llama_projection_full(lib):
    d = W.generate_gemv(W.lookup("v1"))
    y = run(lib, d)
    _, ref = oracle.gemv_w4a16(d["x"], d["B"], d["B_sf"], d["alpha"][0], d["cfg"].K)
    vals = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert oracle.tolerance_ok(vals, ref, np.abs(ref).max()).all()


def _bf16_pattern(rng, shape, exp_lo, exp_hi):
    """Random bf16 bit patterns: random sign, biased exponent in [exp_lo,
    exp_hi] (0 = subnormal or zero), random 7-bit mantissa."""
    sign = rng.integers(0, 2, shape).astype(np.uint16)
    exp = rng.integers(exp_lo, exp_hi + 1, shape).astype(np.uint16)
    man = rng.integers(0, 128, shape).astype(np.uint16)
    return (sign << 15) | (exp << 7) | man


def test_gemv_activation_range(lib):
    """Activations over bf16's whole finite range, one token per kind, each
    token checked against its own largest output: zero blocks between normal
    ones, subnormal and near-subnormal values, values near 1e30, and blocks
    mixing 2^-40 .. 2^10 (the staging's per-block factor at its limits)."""
    M, N, K = 5, 300, 2048
    cfg = W.Config("v0", f"gemv {M}x{N}x{K}", 1, M, N, K, "fixed", masked_list=(M,),
                   kind="gemv_w4a16")
    d = W.generate_gemv(cfg, seed=77)
    rng = np.random.default_rng(78)
    x = np.empty((M, K), np.uint16)
    x[0] = _bf16_pattern(rng, K, 120, 130)
    x[0].reshape(-1, 16)[::3] = 0                       # every third block all zero
    x[1] = _bf16_pattern(rng, K, 0, 0)                  # subnormal (and some zeros)
    x[2] = _bf16_pattern(rng, K, 0, 3)                  # straddles the normal boundary
    x[3] = _bf16_pattern(rng, K, 215, 226)              # about 1e28 .. 1e31
    x[4] = _bf16_pattern(rng, K, 127 - 40, 127 + 10)    # 50 binades inside each block
    d["x"] = x
    y = run(lib, d)
    _, ref = oracle.gemv_w4a16(x, d["B"], d["B_sf"], d["alpha"][0], K)
    vals = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for m in range(M):
        ok = oracle.tolerance_ok(vals[m], ref[m], np.abs(ref[m]).max())
        assert ok.all(), f"token {m}: {(~ok).sum()} of {N} outside tolerance"


@pytest.mark.parametrize("M,K", [(8, 8928), (1, 71488)])
def test_gemv_largest_staging(lib, M, K):
    """The largest token staging shared memory takes (M * K <= 71493)."""
    N = 97
    cfg = W.Config("v0", f"gemv {M}x{N}x{K}", 1, M, N, K, "fixed", masked_list=(M,),
                   kind="gemv_w4a16")
    d = W.generate_gemv(cfg, seed=M + K)
    y = run(lib, d)
    _, ref = oracle.gemv_w4a16(d["x"], d["B"], d["B_sf"], d["alpha"][0], K)
    vals = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert oracle.tolerance_ok(vals, ref, np.abs(ref).max()).all()
