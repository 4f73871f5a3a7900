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


def test_signals_arrive_before_the_call_ends(lib):
    """dst_signals exist so that a consumer can start on an expert while the
    call is still running.  The consumer here is the copy engine driven from
    the host (no kernel spins on another kernel's flag): while the GEMM runs
    on one stream, a second stream repeatedly copies dst_signals to pinned
    host memory; for each expert whose signal is seen, its valid rows of C
    are copied out right then.  Experts of very different sizes, and one
    persistent CTA (sm_count = 1), so that experts finish one after another.
    Passes if some snapshot shows part of the non-empty experts signalled and
    the rest not (the signal came before the call's end), signals never go
    back or past +1, and every early copy equals the final C bit for bit."""
    import time
    from nvfp4_block_scaled_masked_gb300.device import Problem
    G, M_max, N, K = 8, 192, 4096, 7168
    masked = [192, 0, 17, 192, 5, 192, 64, 130]
    d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=2024)
    prob = Problem(d)
    init = 40
    sig = torch.full((G,), init, dtype=torch.int32, device="cuda")
    snap = torch.empty(G, dtype=torch.int32).pin_memory()
    early = {}
    nonempty = [g for g in range(G) if masked[g] > 0]
    partial_seen = False
    history = []
    gemm_stream = torch.cuda.Stream()
    copy_stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    lib.nvfp4_gg_set_sm_count(1)
    try:
        with torch.cuda.stream(gemm_stream):
            lib.nvfp4_grouped_gemm_nt_masked_signals(prob.A, prob.A_sf, prob.B_prep, prob.B_sf_prep,
                                                     prob.alpha, prob.masked_m, prob.C, G, M_max, N,
                                                     K, sig, gemm_stream)
            done = torch.cuda.Event()
            done.record(gemm_stream)
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 30.0:
            finished = done.query()           # taken before the snapshot is copied
            with torch.cuda.stream(copy_stream):
                snap.copy_(sig, non_blocking=True)
            copy_stream.synchronize()
            s = snap.numpy().copy()
            history.append(s)
            got = [g for g in nonempty if s[g] == init + 1]
            if not finished and 0 < len(got) < len(nonempty):
                partial_seen = True
            for g in got:
                if g not in early:
                    host = torch.empty((masked[g], N), dtype=torch.int16).pin_memory()
                    with torch.cuda.stream(copy_stream):
                        host.copy_(prob.C[g, :masked[g]], non_blocking=True)
                    copy_stream.synchronize()
                    early[g] = host.numpy().view(np.uint16).copy()
            if finished:
                break
        gemm_stream.synchronize()
    finally:
        lib.nvfp4_gg_set_sm_count(0)
    assert lib.nvfp4_gg_check_error() == 0
    h = np.array(history)
    assert np.all(np.diff(h, axis=0) >= 0) and np.all((h == init) | (h == init + 1))
    np.testing.assert_array_equal(sig.cpu().numpy(), np.full(G, init + 1))
    final = prob.C_bits()
    for g, rows in early.items():
        np.testing.assert_array_equal(rows, final[g, :masked[g]])
    assert partial_seen, f"no snapshot caught the call part-way ({len(history)} snapshots)"
    # the final C is the plain call's
    lib.nvfp4_gg_set_pair_mode(0)
    try:
        prob.reset_C()
        prob.run()
        np.testing.assert_array_equal(prob.C_bits(), final)
    finally:
        lib.nvfp4_gg_set_pair_mode(lib.PAIR_AUTO)


@pytest.mark.parametrize("G,M_max,N1,K,masked", [
    (2, 96, 256, 1024, [96, 41]),       # prefill-sized experts
    (3, 16, 512, 2048, [16, 0, 7]),     # decode-sized experts, one empty
])
def test_dual_gemm_entry_point_from_separate_operands(lib, G, M_max, N1, K, masked):
    """nvfp4_prepare_weights_dual takes B1 and B2 as separate buffers.  Its
    stacked layout gives both products in one GEMM call, each against its own
    oracle GEMM; its interleaved layout gives silu(A B1^T) * (A B2^T) through
    the SwiGLU entry point.  Both prepared buffers are byte-identical to the
    single-operand re-layouts of [B1; B2]."""
    cfg = W.custom(G, M_max, 2 * N1, K, masked_m=masked)
    d = W.generate(cfg, seed=G * 7 + N1 + K)
    mm = d["masked_m"]
    B1, B1sf = np.ascontiguousarray(d["B"][:, :N1]), np.ascontiguousarray(d["B_sf"][:, :N1])
    B2, B2sf = np.ascontiguousarray(d["B"][:, N1:]), np.ascontiguousarray(d["B_sf"][:, N1:])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    A, A_sf, alpha, mmd = dev(d["A"]), dev(d["A_sf"]), dev(d["alpha"]), dev(mm.astype(np.int32))
    bb, sb = lib.nvfp4_prepared_weight_bytes(G, 2 * N1, K)
    init = np.full((G, M_max, N1), W.SENTINEL_BF16, np.uint16)
    _, r1 = oracle.gemm(d["A"], d["A_sf"], B1, B1sf, d["alpha"], mm, init, G, M_max, N1, K)
    _, r2 = oracle.gemm(d["A"], d["A_sf"], B2, B2sf, d["alpha"], mm, init, G, M_max, N1, K)
    for interleave in (0, 1):
        Bp = torch.empty(bb, dtype=torch.uint8, device="cuda")
        Bsp = torch.empty(sb, dtype=torch.uint8, device="cuda")
        lib.nvfp4_prepare_weights_dual(dev(B1), dev(B1sf), dev(B2), dev(B2sf), G, N1, K, interleave,
                                       Bp, Bsp)
        # the same bytes as preparing the stacked operand
        Rp = torch.empty(bb, dtype=torch.uint8, device="cuda")
        Rsp = torch.empty(sb, dtype=torch.uint8, device="cuda")
        prep = lib.nvfp4_prepare_weights_swiglu if interleave else lib.nvfp4_prepare_weights
        prep(dev(d["B"]), dev(d["B_sf"]), G, 2 * N1, K, Rp, Rsp)
        assert torch.equal(Bp, Rp) and torch.equal(Bsp, Rsp)
        if interleave == 0:
            C = torch.full((G, M_max, 2 * N1), W.SENTINEL_BF16, dtype=torch.int16, device="cuda")
            lib.nvfp4_grouped_gemm_nt_masked(A, A_sf, Bp, Bsp, alpha, mmd, C, G, M_max, 2 * N1, K)
            assert lib.nvfp4_gg_check_error() == 0
            c = C.cpu().numpy().view(np.uint16)
            _within(d, np.ascontiguousarray(c[:, :, :N1]), r1, mm)
            _within(d, np.ascontiguousarray(c[:, :, N1:]), r2, mm)
        else:
            C = torch.full((G, M_max, N1), W.SENTINEL_BF16, dtype=torch.int16, device="cuda")
            lib.nvfp4_grouped_gemm_nt_masked_swiglu(A, A_sf, Bp, Bsp, alpha, mmd, C, G, M_max,
                                                    2 * N1, K)
            assert lib.nvfp4_gg_check_error() == 0
            _within(d, C.cpu().numpy().view(np.uint16), oracle.silu(r1) * r2, mm)
