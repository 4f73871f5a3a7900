"""GPU parity of the packed-rows ("contiguous") layout entry point.

The masked-layout inputs are packed expert after expert (rows m <
masked_m[g] only) into A [M_total][K/2] and A_sf [M_total][K/16];
nvfp4_grouped_gemm_nt_contiguous must write exactly the packed valid rows of
C, bit-identical to the masked-layout call (same kernel, same token tiles),
within tolerance of the oracle, and leave every other row untouched."""
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


def pack(d, M_total):
    cfg, mm = d["cfg"], d["masked_m"]
    A = np.zeros((M_total, cfg.K // 2), np.uint8)
    Asf = np.full((M_total, cfg.K // 16), 0x38, np.uint8)
    r = 0
    for g in range(cfg.G):
        A[r:r + mm[g]] = d["A"][g, :mm[g]]
        Asf[r:r + mm[g]] = d["A_sf"][g, :mm[g]]
        r += mm[g]
    return A, Asf


@pytest.mark.parametrize("G,M_max,N,K,masked,spare", [
    (5, 40, 272, 512, [40, 0, 17, 33, 1], 9),     # decode kernel; tiles overhang into the next expert
    (3, 200, 384, 1024, [200, 65, 0], 0),         # prefill, single CTAs (N % 256 != 0), exact capacity
    (3, 200, 512, 512, [129, 200, 31], 40),       # prefill on CTA pairs (automatic mode)
])
def test_contiguous_matches_masked_layout(lib, G, M_max, N, K, masked, spare):
    from nvfp4_block_scaled_masked_gb300.device import Problem
    d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=G * 13 + N + K)
    prob = Problem(d)
    prob.run()
    want = prob.C_bits()
    mm = d["masked_m"]
    M_total = int(mm.sum()) + spare
    A, Asf = pack(d, M_total)
    dA, dAsf = torch.from_numpy(A).cuda(), torch.from_numpy(Asf).cuda()
    C = torch.full((M_total, N), W.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    for _ in range(2):
        lib.nvfp4_grouped_gemm_nt_contiguous(dA, dAsf, prob.B_prep, prob.B_sf_prep, prob.alpha,
                                             prob.masked_m, C, G, M_max, M_total, N, K)
        assert lib.nvfp4_gg_check_error() == 0
        got = C.cpu().numpy().view(np.uint16)
        r = 0
        for g in range(G):
            np.testing.assert_array_equal(got[r:r + mm[g]], want[g, :mm[g]])
            r += mm[g]
        assert np.all(got[r:] == W.SENTINEL_BF16), "rows past the packed valid rows were written"
    _, ref = oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], mm, d["C_init"],
                         G, M_max, N, K)
    valid = np.concatenate([ref[g, :mm[g]] for g in range(G)])
    vals = (got[:int(mm.sum())].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert oracle.tolerance_ok(vals, valid, np.abs(valid).max()).all()


def test_contiguous_capacity_overflow_is_flagged(lib):
    """sum(masked_m) > M_total: the error word says NVFP4GG_ERR_MASK and no row
    past M_total is written (the buffer is padded to see it)."""
    from nvfp4_block_scaled_masked_gb300.device import Problem
    G, M_max, N, K = 2, 40, 128, 256
    d = W.generate(W.custom(G, M_max, N, K, masked_m=[40, 30]), seed=4)
    prob = Problem(d)
    M_total = 50
    A, Asf = pack(d, 70)
    dA, dAsf = torch.from_numpy(A).cuda(), torch.from_numpy(Asf).cuda()
    C = torch.full((80, N), W.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    lib.nvfp4_grouped_gemm_nt_contiguous(dA, dAsf, prob.B_prep, prob.B_sf_prep, prob.alpha,
                                         prob.masked_m, C, G, M_max, M_total, N, K)
    assert lib.nvfp4_gg_check_error() == lib.ERR_MASK
    got = C.cpu().numpy().view(np.uint16)
    assert np.all(got[M_total:] == W.SENTINEL_BF16)
