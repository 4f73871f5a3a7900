"""GPU checks of two API extensions built on the GEMM kernels.

* Per-expert completion signals (nvfp4_grouped_gemm_nt_masked_signals): each
  call adds exactly 1 to every expert's signal, empty experts included, and
  C is bit-identical to the plain single-CTA call.
* The dual GEMM (one A operand used by two GEMMs, on the page "LLM-Assisted Kernel
  Development in CuTe DSL, Gluon, Helion and Triton"): with B1 and B2 stacked
  along N one call computes both, each equal to its own oracle
  GEMM; with the SwiGLU entry point it computes silu(A B1^T) * (A B2^T)."""
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


def _within(d_like, C_bits, ref64, mm):
    G, M = C_bits.shape[:2]
    valid = np.zeros((G, M), dtype=bool)
    for g in range(G):
        valid[g, :mm[g]] = True
    assert np.all(C_bits[~valid] == W.SENTINEL_BF16)
    vals = (C_bits[valid].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = ref64[valid]
    assert oracle.tolerance_ok(vals, r, np.abs(r).max()).all()


@pytest.mark.parametrize("G,M_max,N,K,masked", [
    (5, 40, 272, 512, [40, 0, 17, 33, 0]),      # decode kernel, empty experts
    (3, 200, 512, 512, [200, 0, 65]),           # prefill shape (pairs would apply: not here)
])
def test_signals_count_once_per_call_and_results_match(lib, G, M_max, N, K, masked):
    from nvfp4_block_scaled_masked_gb300.device import Problem
    d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=G * 31 + N)
    prob = Problem(d)
    lib.nvfp4_gg_set_pair_mode(0)
    try:
        prob.run()
        want = prob.C_bits()
    finally:
        lib.nvfp4_gg_set_pair_mode(lib.PAIR_AUTO)
    sig = torch.full((G,), 7, dtype=torch.int32, device="cuda")
    for call in range(2):
        prob.reset_C()
        lib.nvfp4_grouped_gemm_nt_masked_signals(prob.A, prob.A_sf, prob.B_prep, prob.B_sf_prep,
                                                 prob.alpha, prob.masked_m, prob.C, G, M_max, N, K,
                                                 sig)
        assert lib.nvfp4_gg_check_error() == 0
        np.testing.assert_array_equal(sig.cpu().numpy(), np.full(G, 8 + call))
        np.testing.assert_array_equal(prob.C_bits(), want)
    _, ref = oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], d["masked_m"],
                         d["C_init"], G, M_max, N, K)
    _within(d, want, ref, d["masked_m"])


def test_dual_gemm_merged_b_and_swiglu(lib):
    """A [M, K] shared; B1, B2 [N1, K]: the call on B1 and B2 stacked equals the two oracle
    GEMMs column block by column block, and the SwiGLU call equals
    silu(A B1^T) * (A B2^T) from the same oracle outputs."""
    from nvfp4_block_scaled_masked_gb300.device import Problem
    M, N1, K = 96, 256, 1024
    d = W.generate(W.custom(1, M, 2 * N1, K, masked_m=[M]), seed=99)
    B1, B1sf = d["B"][:, :N1], d["B_sf"][:, :N1]
    B2, B2sf = d["B"][:, N1:], d["B_sf"][:, N1:]
    init = np.full((1, M, N1), W.SENTINEL_BF16, np.uint16)
    _, r1 = oracle.gemm(d["A"], d["A_sf"], B1, B1sf, d["alpha"], d["masked_m"], init, 1, M, N1, K)
    _, r2 = oracle.gemm(d["A"], d["A_sf"], B2, B2sf, d["alpha"], d["masked_m"], init, 1, M, N1, K)
    prob = Problem(d)                       # B = [B1; B2] along N
    prob.run()
    C = prob.C_bits()
    _within(d, np.ascontiguousarray(C[:, :, :N1]), r1, d["masked_m"])
    _within(d, np.ascontiguousarray(C[:, :, N1:]), r2, d["masked_m"])
    # combined: silu(A B1^T) * (A B2^T)
    bb, sb = lib.nvfp4_prepared_weight_bytes(1, 2 * N1, K)
    Bp = torch.empty(bb, dtype=torch.uint8, device="cuda")
    Bsp = torch.empty(sb, dtype=torch.uint8, device="cuda")
    raw_B = torch.from_numpy(np.ascontiguousarray(d["B"])).cuda()
    raw_Bsf = torch.from_numpy(np.ascontiguousarray(d["B_sf"])).cuda()
    lib.nvfp4_prepare_weights_swiglu(raw_B, raw_Bsf, 1, 2 * N1, K, Bp, Bsp)
    Cs = torch.full((1, M, N1), W.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    lib.nvfp4_grouped_gemm_nt_masked_swiglu(prob.A, prob.A_sf, Bp, Bsp, prob.alpha, prob.masked_m,
                                            Cs, 1, M, 2 * N1, K)
    assert lib.nvfp4_gg_check_error() == 0
    want = oracle.silu(r1) * r2
    _within(d, Cs.cpu().numpy().view(np.uint16), want, d["masked_m"])
