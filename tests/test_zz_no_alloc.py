"""GPU checks of nvfp4_grouped_gemm_nt_masked_splitk_noalloc, the split-K call
whose scratch is a static device array of the library (it allocates nothing).

Its results are compared with the existing entry points on the same inputs:
bit for bit with nvfp4_grouped_gemm_nt_masked_splitk at the same split (same
kernel, same reduction order), and within the parity tolerance with the
unsplit nvfp4_grouped_gemm_nt_masked; two calls in a row each time, so that a
counter the first call left behind would show in the second.  The file is
named to be collected last, so it runs both alone and after the other tests
have used the library on the same device."""
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


def bf16_to_f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def _checked(lib):
    rc = lib.nvfp4_gg_check_error()
    assert rc == 0, lib.status_string(rc)


def _noalloc(lib, prob, split_k):
    cfg = prob.cfg
    prob.reset_C()
    lib.nvfp4_grouped_gemm_nt_masked_splitk_noalloc(prob.A, prob.A_sf, prob.B_prep,
                                                    prob.B_sf_prep, prob.alpha, prob.masked_m,
                                                    prob.C, cfg.G, cfg.M_max, cfg.N, cfg.K,
                                                    split_k)
    _checked(lib)
    return prob.C_bits()


def _workspace(lib, prob, split_k):
    cfg = prob.cfg
    nbytes = lib.nvfp4_splitk_workspace_bytes(cfg.G, cfg.M_max, cfg.N, cfg.K, split_k)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    prob.reset_C()
    lib.nvfp4_grouped_gemm_nt_masked_splitk(prob.A, prob.A_sf, prob.B_prep, prob.B_sf_prep,
                                            prob.alpha, prob.masked_m, prob.C, cfg.G, cfg.M_max,
                                            cfg.N, cfg.K, split_k, ws, nbytes)
    _checked(lib)
    return prob.C_bits()


def _unsplit(lib, prob):
    prob.reset_C()
    prob.run()
    _checked(lib)
    return prob.C_bits()


def _within_tolerance(d, got, want):
    """Valid rows within |got - want| <= 4e-3 |want| + 1e-4 max|want| (the
    unsplit result standing in for the reference); other rows untouched."""
    cfg, mm = d["cfg"], d["masked_m"]
    valid = np.zeros((cfg.G, cfg.M_max), dtype=bool)
    for g in range(cfg.G):
        valid[g, :mm[g]] = True
    assert np.all(got[~valid] == W.SENTINEL_BF16), "rows >= masked_m were written"
    if valid.any():
        w = bf16_to_f64(want[valid])
        ok = oracle.tolerance_ok(bf16_to_f64(got[valid]), w, np.abs(w).max())
        assert ok.all(), f"{int((~ok).sum())} of {ok.size} outside tolerance"


@pytest.mark.parametrize("G,M_max,N,K,masked,split", [
    (1, 8, 4096, 7168, [7], 0),                  # one expert, automatic split
    (1, 16, 4096, 7168, [16], 8),                # 32 tiles x 8 = all 256 slots
    (3, 40, 144, 1280, [40, 0, 9], 3),           # N tail, two token tiles per expert
    (4, 64, 384, 512, [64, 33, 0, 1], 16),       # split capped at K/256 = 2
])
def test_noalloc_matches_existing_entry_points(lib, G, M_max, N, K, masked, split):
    from nvfp4_block_scaled_masked_gb300.device import Problem
    d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=1009 * G + K)
    prob = Problem(d)
    ref_ws = _workspace(lib, prob, split)
    ref_unsplit = _unsplit(lib, prob)
    for _ in range(2):
        got = _noalloc(lib, prob, split)
        np.testing.assert_array_equal(got, ref_ws)
        _within_tolerance(d, got, ref_unsplit)


def test_noalloc_unsplit_cases_equal_the_plain_call(lib):
    """split_k = 1, prefill shapes (M_max > 64) and an automatic split with
    more weight tiles than SMs all run the unsplit kernel: same bits as the
    plain call."""
    from nvfp4_block_scaled_masked_gb300.device import Problem
    for G, M_max, N, K, masked, split in [(2, 16, 512, 1024, [16, 3], 1),
                                         (2, 96, 256, 512, [96, 50], 4),
                                         (32, 16, 4096, 512, [5] * 32, 0)]:
        d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=G + M_max + K)
        prob = Problem(d)
        want = _unsplit(lib, prob)
        for _ in range(2):
            np.testing.assert_array_equal(_noalloc(lib, prob, split), want)


def test_noalloc_oversized_split_is_refused_without_launch(lib):
    from nvfp4_block_scaled_masked_gb300.device import Problem
    d = W.generate(W.custom(8, 16, 4096, 1024, masked_m=[16] * 8), seed=5)   # 256 tiles
    prob = Problem(d)
    with pytest.raises(lib.NVFP4GGError) as e:
        _noalloc(lib, prob, 2)
    assert e.value.status == lib.ERR_SCRATCH
    assert np.all(prob.C_bits() == W.SENTINEL_BF16)
    _checked(lib)
