"""GPU parity of the fused GEMM1 + SwiGLU entry point against the oracle.

nvfp4_grouped_gemm_nt_masked_swiglu on weights prepared by
nvfp4_prepare_weights_swiglu, compared element by element with the oracle's
swiglu step applied to its fp64 GEMM1 output: valid rows within
|gpu - ref| <= 4e-3 |ref| + 1e-4 max|ref| (ref unrounded fp64), rows
m >= masked_m[g] bit-identical to the prefill.  Calls go through the C-ABI."""
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


def run_swiglu(lib, d, calls=2):
    cfg = d["cfg"]
    G, M, N, K = cfg.G, cfg.M_max, cfg.N, cfg.K
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    A, A_sf, B, B_sf = dev(d["A"]), dev(d["A_sf"]), dev(d["B"]), dev(d["B_sf"])
    alpha, mm = dev(d["alpha"]), dev(d["masked_m"].astype(np.int32))
    bb, sb = lib.nvfp4_prepared_weight_bytes(G, N, K)
    Bp = torch.empty(bb, dtype=torch.uint8, device="cuda")
    Bsp = torch.empty(sb, dtype=torch.uint8, device="cuda")
    lib.nvfp4_prepare_weights_swiglu(B, B_sf, G, N, K, Bp, Bsp)
    outs = []
    for _ in range(calls):
        C = torch.full((G, M, N // 2), W.SENTINEL_BF16, dtype=torch.int16, device="cuda")
        lib.nvfp4_grouped_gemm_nt_masked_swiglu(A, A_sf, Bp, Bsp, alpha, mm, C, G, M, N, K)
        rc = lib.nvfp4_gg_check_error()
        assert rc == 0, lib.status_string(rc)
        outs.append(C.cpu().numpy().view(np.uint16))
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])
    return outs[0]


def check(d, C_gpu):
    cfg = d["cfg"]
    G, M, N = cfg.G, cfg.M_max, cfg.N
    _, ref64 = oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], d["masked_m"],
                           d["C_init"], G, M, N, cfg.K)
    init = np.full((G, M, N // 2), W.SENTINEL_BF16, np.uint16)
    C_ref, out = oracle.swiglu(ref64, d["masked_m"], init)
    mm = d["masked_m"]
    valid = np.zeros((G, M), dtype=bool)
    for g in range(G):
        valid[g, :mm[g]] = True
    assert np.all(C_gpu[~valid] == W.SENTINEL_BF16), "rows >= masked_m were written"
    if not valid.any():
        return
    vals = (C_gpu[valid].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = out[valid]
    assert np.all(np.isfinite(vals))
    ok = oracle.tolerance_ok(vals, r, np.abs(r).max())
    assert ok.all(), (f"{(~ok).sum()} of {ok.size} outside tolerance; first gpu="
                      f"{vals[~ok][:4]} ref={r[~ok][:4]}")
    same = np.mean(C_gpu[valid] == C_ref[valid])
    assert same > 0.9, f"only {same:.3f} bit-identical to the correctly rounded oracle"


@pytest.mark.parametrize("pair", [0, 2])         # single-CTA kernels; automatic (CTA pairs where N % 256 == 0)
@pytest.mark.parametrize("G,M_max,N,K,masked", [
    (3, 40, 256, 512, [40, 0, 17]),              # decode kernel, two token tiles, an empty expert
    (2, 200, 384, 1024, [200, 77]),              # prefill kernel, ragged token tiles
    (2, 200, 512, 1024, [200, 77]),              # prefill, N % 256 == 0: CTA pairs in mode 2
    (3, 300, 768, 2048, [300, 0, 129]),          # several token tiles per expert, an empty expert
    (1, 1, 128, 256, [1]),                       # minimum sizes
])
def test_swiglu_shapes(lib, G, M_max, N, K, masked, pair):
    d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=G * 7 + N + K)
    lib.nvfp4_gg_set_pair_mode(pair)
    try:
        C = run_swiglu(lib, d)
    finally:
        lib.nvfp4_gg_set_pair_mode(lib.PAIR_AUTO)
    check(d, C)


def test_swiglu_decode_gemm1_full(lib):
    """The decode GEMM1 workload (G=32, N = 2 x 2048, K = 7168), every output."""
    d = W.generate(W.CONFIGS["c2"])
    check(d, run_swiglu(lib, d, calls=1))


def test_swiglu_rejects_n_not_multiple_of_128(lib):
    with pytest.raises(lib.NVFP4GGError) as e:
        lib.nvfp4_grouped_gemm_nt_masked_swiglu(256, 256, 256, 256, 256, 256, 256, 1, 16, 192, 256)
    assert e.value.status == lib.ERR_SHAPE
