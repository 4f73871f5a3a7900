"""GPU parity: the CUDA path against the CPU oracle, element by element.

Bar (the stated acceptance test): for every valid (g, m, n),
|gpu - ref| <= 4e-3 |ref| + 1e-4 max|ref|, ref the oracle's unrounded fp64
value and max taken over the call; rows m >= masked_m[g] bit-identical to the
0x7FC0 prefill.  Calls go through the C-ABI (ctypes binding)."""
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


def run_gpu(d):
    from nvfp4_block_scaled_masked_gb300.device import Problem
    from nvfp4_block_scaled_masked_gb300 import binding
    prob = Problem(d)
    prob.run()
    rc = binding.nvfp4_gg_check_error()
    assert rc == 0, binding.status_string(rc)
    return prob.C_bits()


def check_full(d, C_gpu):
    cfg = d["cfg"]
    C_ref, ref = oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], d["masked_m"],
                             d["C_init"], cfg.G, cfg.M_max, cfg.N, cfg.K)
    mm = d["masked_m"]
    valid = np.zeros((cfg.G, cfg.M_max), dtype=bool)
    for g in range(cfg.G):
        valid[g, :mm[g]] = True
    # invariants: untouched rows bit-identical to the prefill
    assert np.all(C_gpu[~valid] == W.SENTINEL_BF16), "rows >= masked_m were written"
    if not valid.any():
        return
    vals = bf16_to_f64(C_gpu[valid])
    r = ref[valid]
    assert np.all(np.isfinite(vals))
    max_abs = np.abs(r).max()
    ok = oracle.tolerance_ok(vals, r, max_abs)
    if not ok.all():
        bad = np.flatnonzero(~ok.ravel())
        idx = np.argwhere(valid)
        cols = bad % cfg.N
        rows = idx[bad // cfg.N]
        msg = [f"{len(bad)} of {ok.size} outside tolerance; first:"]
        for b, (g, m), n in list(zip(bad, rows, cols))[:8]:
            msg.append(f"  g={g} m={m} n={n} gpu={vals.ravel()[b]!r} ref={r.ravel()[b]!r}")
        pytest.fail("\n".join(msg))
    # most values should be the correctly rounded bf16 (fp32 accumulation order
    # only rarely moves a value across a rounding boundary)
    same = np.mean(C_gpu[valid] == C_ref[valid])
    assert same > 0.9, f"only {same:.3f} bit-identical to the correctly rounded oracle"


def check_sampled(d, C_gpu, rows_per_group=6, cols=96, seed=0):
    """Every non-empty expert: its first and last valid row plus random rows,
    each at `cols` random n; fp64 sampled oracle.  Invariants checked in full."""
    cfg = d["cfg"]
    mm = d["masked_m"]
    for g in range(cfg.G):
        assert np.all(C_gpu[g, mm[g]:] == W.SENTINEL_BF16), f"expert {g}: rows >= masked_m written"
    rng = np.random.default_rng(seed)
    idx = []
    for g in range(cfg.G):
        if mm[g] == 0:
            continue
        rows = {0, mm[g] - 1} | set(rng.integers(0, mm[g], rows_per_group).tolist())
        for m in rows:
            for n in rng.choice(cfg.N, size=min(cols, cfg.N), replace=False):
                idx.append((g, m, n))
    idx = np.array(idx, dtype=np.int64)
    ref = oracle.gemm_sampled(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], idx,
                              cfg.G, cfg.M_max, cfg.N, cfg.K)
    vals = bf16_to_f64(C_gpu[idx[:, 0], idx[:, 1], idx[:, 2]])
    max_abs = np.abs(ref).max()
    ok = oracle.tolerance_ok(vals, ref, max_abs)
    assert ok.all(), (f"{(~ok).sum()} of {ok.size} sampled outputs outside tolerance; "
                      f"first {idx[~ok][:4].tolist()} gpu={vals[~ok][:4]} ref={ref[~ok][:4]}")


def test_c1_small_masked(lib):
    d = W.generate(W.CONFIGS["c1"])
    check_full(d, run_gpu(d))


def test_c1_poisoned_rows_ignored(lib):
    d = W.generate(W.CONFIGS["c1"], poison=True)
    check_full(d, run_gpu(d))


@pytest.mark.parametrize("G,M_max,N,K,masked", [
    (3, 16, 128, 256, [1, 16, 0]),                          # one stage, narrow tiles
    (5, 40, 144, 512, [40, 33, 32, 17, 0]),                 # N tail, 2 token tiles, 2 stages
    (2, 64, 256, 1024, [64, 31]),                           # narrow kernel, M_max = 64
    (4, 200, 272, 768, [200, 129, 128, 1]),                 # wide kernel, ragged widths
    (2, 256, 384, 512, [256, 255]),                         # wide kernel, 2 x 128 tiles
    (2, 192, 384, 2048, [192, 177]),                        # wide single-CTA kernel (N % 256
                                                            # != 0), full 192-row tile, 8 stages
                                                            # over 2 scale regions
    (1, 1, 16, 256, [1]),                                   # minimum sizes
    (6, 24, 128, 256, [0, 0, 0, 0, 0, 0]),                  # every expert empty
])
def test_shapes_ragged_and_edges(lib, G, M_max, N, K, masked):
    d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=G * 1000 + N)
    check_full(d, run_gpu(d))


@pytest.mark.parametrize("G,M_max,N,K,masked", [
    (3, 200, 512, 512, [200, 33, 1]),          # CTA pairs: 2 token tiles, widths 128 / 64 / 32
    (2, 161, 256, 256, [161, 160]),             # widths rounded to 32, one k-stage
    (4, 96, 768, 1024, [96, 0, 65, 31]),        # empty expert, 3 weight-block pairs, 4 k-stages
])
@pytest.mark.parametrize("pair", [True, False])
def test_prefill_variants_pair_and_single(lib, G, M_max, N, K, masked, pair):
    d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=G + N + K)
    lib.nvfp4_gg_set_pair_mode(pair)
    try:
        check_full(d, run_gpu(d))
    finally:
        lib.nvfp4_gg_set_pair_mode(lib.PAIR_AUTO)


@pytest.mark.parametrize("G,M_max,N,K,masked", [
    (3, 300, 512, 1536, [300, 0, 129]),      # 2 token tiles (the second CTA's rows of the
                                             # last one wholly past M_max), 6 stages > ring
    (2, 256, 768, 2048, [256, 200]),         # 3 weight-block pairs, 8 stages
    (1, 128, 256, 256, [1]),                 # one stage, one valid row
    (4, 512, 256, 7168, [512, 511, 0, 257]),  # 28 stages, ragged token tiles, empty expert
])
def test_token_major_pair_kernel(lib, G, M_max, N, K, masked):
    """Token-major CTA pairs (256 tokens x 256 weight rows per MMA), forced
    with pair mode 3 on small shapes; chosen automatically for M_max > 256."""
    d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=3 * G + N + K)
    lib.nvfp4_gg_set_pair_mode(lib.PAIR_TOKEN_MAJOR)
    try:
        check_full(d, run_gpu(d))
    finally:
        lib.nvfp4_gg_set_pair_mode(lib.PAIR_AUTO)


@pytest.mark.parametrize("key", ["c4", "c5"])
def test_full_size_sampled_pair_kernel(lib, key):
    lib.nvfp4_gg_set_pair_mode(True)
    try:
        d = W.generate(W.CONFIGS[key])
        check_sampled(d, run_gpu(d), rows_per_group=3, cols=48)
    finally:
        lib.nvfp4_gg_set_pair_mode(lib.PAIR_AUTO)


def run_gpu_splitk(d, split_k):
    from nvfp4_block_scaled_masked_gb300.device import Problem
    from nvfp4_block_scaled_masked_gb300 import binding
    cfg = d["cfg"]
    prob = Problem(d)
    nbytes = binding.nvfp4_splitk_workspace_bytes(cfg.G, cfg.M_max, cfg.N, cfg.K, split_k)
    # the workspace needs no initial value: arbitrary bytes in it (counters
    # included) must not change the result
    ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):      # deterministic: two calls give the same bits
        prob.reset_C()
        binding.nvfp4_grouped_gemm_nt_masked_splitk(prob.A, prob.A_sf, prob.B_prep, prob.B_sf_prep,
                                                    prob.alpha, prob.masked_m, prob.C, cfg.G,
                                                    cfg.M_max, cfg.N, cfg.K, split_k, ws, nbytes)
        rc = binding.nvfp4_gg_check_error()
        assert rc == 0, binding.status_string(rc)
        outs.append(prob.C_bits())
    np.testing.assert_array_equal(outs[0], outs[1])
    return outs[0]


@pytest.mark.parametrize("G,M_max,N,K,masked,split", [
    (3, 16, 256, 768, [5, 0, 16], 2),           # 3 k-stages split 1 + 2
    (2, 40, 144, 1280, [40, 7], 3),             # N tail, 2 token tiles, 5 stages split 1/2/2
    (1, 8, 4096, 7168, [7], 0),                 # one expert: automatic split (all SMs)
    (4, 64, 384, 512, [64, 33, 0, 1], 16),      # split capped at K/256 = 2
])
def test_splitk_decode(lib, G, M_max, N, K, masked, split):
    d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=31 * G + K)
    check_full(d, run_gpu_splitk(d, split))


# Splits of up to 8 ranges reduce inside a thread-block cluster (distributed
# shared memory), larger ones through the workspace.  Several tiles per
# cluster exercise the per-tile hand-offs; an SM cap below the split falls
# back to the workspace; ragged N and token tails are stored by the cluster
# epilogue.
@pytest.mark.parametrize("G,M_max,N,K,masked,split,cap", [
    (4, 64, 2048, 4096, [64, 33, 0, 50], 8, 0),   # 96 tiles on 19 clusters of 8
    (2, 40, 1040, 7168, [40, 7], 5, 0),           # clusters of 5 (grid 150), N tail
    (1, 32, 4096, 7168, [32], 12, 0),             # more than 8 ranges: workspace
    (3, 48, 512, 2048, [48, 1, 17], 4, 6),        # SM cap 6: one cluster of 4
    (2, 16, 256, 1024, [16, 9], 4, 3),            # SM cap 3 < split: workspace
])
def test_splitk_cluster_and_workspace(lib, G, M_max, N, K, masked, split, cap):
    d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=7 * G + N + K)
    lib.nvfp4_gg_set_sm_count(cap)
    try:
        check_full(d, run_gpu_splitk(d, split))
    finally:
        lib.nvfp4_gg_set_sm_count(0)


@pytest.mark.parametrize("G,N,masked", [
    (1, 2048, [7]),          # 16 tiles: 6 ranges per tile
    (1, 4096, [32]),         # 32 tiles: 4 ranges
    (2, 1040, [5, 0]),       # 18 tiles (N tail, one expert empty)
])
def test_plain_entry_splits_few_tile_decode_calls(lib, G, N, masked):
    """The plain entry point splits decode calls with at most SMs/4 tiles
    and K >= 6144 over thread-block clusters: within the tolerance, rows
    past masked_m untouched, two calls bit-identical; under SM caps (10: 2
    ranges of a single... or fewer; 3: too few SMs to split) the results stay
    within the tolerance."""
    from nvfp4_block_scaled_masked_gb300.device import Problem
    d = W.generate(W.custom(G, 32, N, 7168, masked_m=masked), seed=G * 7 + N)
    prob = Problem(d)
    outs = []
    for cap in (0, 0, 70, 3):
        lib.nvfp4_gg_set_sm_count(cap)
        try:
            prob.reset_C()
            prob.run()
            rc = lib.nvfp4_gg_check_error()
            assert rc == 0, lib.status_string(rc)
            outs.append(prob.C_bits())
        finally:
            lib.nvfp4_gg_set_sm_count(0)
    np.testing.assert_array_equal(outs[0], outs[1])
    for C in outs:
        check_full(d, C)


def test_splitk_cluster_equals_workspace_bits(lib):
    """Four ranges reduce in a cluster when 4 SMs or more are allowed, through
    the workspace under an SM cap of 3; both add the same partials in range
    order, so the bits agree."""
    d = W.generate(W.custom(2, 40, 1296, 7168, masked_m=[40, 19]), seed=4242)
    cluster = run_gpu_splitk(d, 4)
    lib.nvfp4_gg_set_sm_count(3)
    try:
        workspace = run_gpu_splitk(d, 4)
    finally:
        lib.nvfp4_gg_set_sm_count(0)
    np.testing.assert_array_equal(cluster, workspace)
    check_full(d, cluster)


def test_c2_decode_full(lib):
    d = W.generate(W.CONFIGS["c2"])
    check_full(d, run_gpu(d))


@pytest.mark.parametrize("key", ["c3", "c4", "c5"])
def test_full_size_sampled(lib, key):
    d = W.generate(W.CONFIGS[key])
    check_sampled(d, run_gpu(d))


def test_alpha_power_of_two_linearity_on_gpu(lib):
    d = W.generate(W.CONFIGS["c1"])
    C1 = run_gpu(d)
    d2 = dict(d)
    d2["alpha"] = (d["alpha"] * np.float32(0.25)).astype(np.float32)
    C2 = run_gpu(d2)
    mm = d["masked_m"]
    for g in range(len(mm)):
        np.testing.assert_array_equal(bf16_to_f64(C2[g, :mm[g]]), bf16_to_f64(C1[g, :mm[g]]) * 0.25)


def test_watchdog_reports_timeout(lib):
    lib.nvfp4_gg_selftest_watchdog(2_000_000)      # 2 ms limit on a barrier nobody completes
    assert lib.nvfp4_gg_check_error() == lib.ERR_TIMEOUT
    assert lib.nvfp4_gg_check_error() == 0          # the word was cleared
    d = W.generate(W.CONFIGS["c1"])                 # the context is still usable
    check_full(d, run_gpu(d))


@pytest.mark.parametrize("pinned_in,pinned_out", [(True, True), (False, False), (True, False)])
def test_host_buffer_entry_point_matches_device_path(lib, pinned_in, pinned_out):
    """nvfp4_grouped_gemm_nt_masked_host: host inputs in, valid rows of C out;
    bit-identical to the device-buffer call, other host rows untouched.
    Pinned buffers are used in place (alpha, masked_m read and C written by
    the kernel); pageable ones go through the device staging buffer."""
    from nvfp4_block_scaled_masked_gb300.device import Problem
    cfg = W.custom(5, 40, 272, 512, masked_m=[40, 0, 17, 33, 1])
    d = W.generate(cfg, seed=77)
    prob = Problem(d)
    prob.run()
    want = prob.C_bits()

    def host(arr, pinned):
        t = torch.from_numpy(np.ascontiguousarray(arr))
        return t.pin_memory() if pinned else t

    h = {k: host(d[k], pinned_in) for k in ("A", "A_sf", "alpha")}
    h["masked_m"] = host(d["masked_m"].astype(np.int32), pinned_in)
    hC = host(np.full((cfg.G, cfg.M_max, cfg.N), W.SENTINEL_BF16, dtype=np.int16), pinned_out)
    nbytes = lib.nvfp4_host_staging_bytes(cfg.G, cfg.M_max, cfg.N, cfg.K)
    staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        lib.nvfp4_grouped_gemm_nt_masked_host(h["A"], h["A_sf"], h["alpha"], h["masked_m"],
                                              prob.B_prep, prob.B_sf_prep, hC, cfg.G, cfg.M_max,
                                              cfg.N, cfg.K, staging, nbytes)
        torch.cuda.synchronize()
        assert lib.nvfp4_gg_check_error() == 0
        np.testing.assert_array_equal(hC.numpy().view(np.uint16), want)
    check_full(d, hC.numpy().view(np.uint16))


@pytest.mark.parametrize("G,M_max,N,K,pinned_in,pinned_out", [
    (40, 128, 256, 4096, True, True),     # CTA pairs, 3 chunks of 2, 8, 30 experts
    (40, 128, 256, 4096, True, False),    # the same with pageable C (staged, copied per expert)
    (40, 128, 256, 4096, False, True),    # pageable activations, alpha and masked_m
    (120, 128, 256, 4096, True, True),    # 4 chunks of 1, 6, 23, 90 experts
    (12, 384, 256, 2048, True, True),     # token-major pairs, 2 chunks of 2, 10 experts
])
def test_host_buffer_entry_point_chunked_copies(lib, G, M_max, N, K, pinned_in, pinned_out):
    """Large host-buffer calls copy the activations in expert chunks on a
    side stream, each chunk's GEMM waiting for its own copy: the bits equal
    the device-buffer call's and rows >= masked_m stay untouched.  A second
    call on other inputs is queued right behind the first, through the same
    staging buffer: its copies must wait for the first call's GEMMs, or the
    first call's output would mix the two problems."""
    from nvfp4_block_scaled_masked_gb300.device import Problem
    rng = np.random.default_rng(G * 1000 + M_max)
    masked = [int(x) for x in rng.integers(1, M_max + 1, G)]
    masked[0], masked[5], masked[-1] = 0, M_max, 0
    cfg = W.custom(G, M_max, N, K, masked_m=masked)
    calls = []
    for seed in (G + M_max, G + M_max + 1):
        d = W.generate(cfg, seed=seed)
        prob = Problem(d)
        prob.run()
        h = {k: torch.from_numpy(np.ascontiguousarray(d[k])) for k in ("A", "A_sf", "alpha")}
        h["masked_m"] = torch.from_numpy(d["masked_m"].astype(np.int32))
        if pinned_in:
            h = {k: v.pin_memory() for k, v in h.items()}
        hC = torch.from_numpy(np.full((cfg.G, cfg.M_max, cfg.N), W.SENTINEL_BF16, dtype=np.int16))
        calls.append((d, prob, prob.C_bits(), h, hC.pin_memory() if pinned_out else hC))
    nbytes = lib.nvfp4_host_staging_bytes(cfg.G, cfg.M_max, cfg.N, cfg.K)
    staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    for _, prob, _, h, hC in calls:
        lib.nvfp4_grouped_gemm_nt_masked_host(h["A"], h["A_sf"], h["alpha"], h["masked_m"],
                                              prob.B_prep, prob.B_sf_prep, hC, cfg.G, cfg.M_max,
                                              cfg.N, cfg.K, staging, nbytes)
    torch.cuda.synchronize()
    assert lib.nvfp4_gg_check_error() == 0
    for _, _, want, _, hC in calls:
        np.testing.assert_array_equal(hC.numpy().view(np.uint16), want)
    check_full(calls[0][0], calls[0][4].numpy().view(np.uint16))


@pytest.mark.parametrize("G,M_max,N,K,masked", [
    (3, 200, 384, 512, [200, 5, 130]),      # single-CTA wide kernel (N % 256 != 0)
    (3, 200, 512, 768, [200, 5, 130]),      # CTA-pair kernel (automatic mode)
])
def test_sm_count_cap_gives_identical_results(lib, G, M_max, N, K, masked):
    """The sm_count cap bounds the CTAs of a launch.  Caps of 7 and 152 run
    the same kernel family (pairs: 6 CTAs), so the bits equal the uncapped
    call's; a cap of 1 leaves no room for a pair and runs the single-CTA
    kernel, equal within the tolerance."""
    from nvfp4_block_scaled_masked_gb300.device import Problem
    d = W.generate(W.custom(G, M_max, N, K, masked_m=masked), seed=8 + N)
    prob = Problem(d)
    prob.run()
    ref = prob.C_bits()
    pair_shape = N % 256 == 0
    try:
        for cap in (1, 7):
            lib.nvfp4_gg_set_sm_count(cap)
            prob.reset_C()
            prob.run()
            assert lib.nvfp4_gg_check_error() == 0
            if cap == 1 and pair_shape:
                check_full(d, prob.C_bits())
            else:
                np.testing.assert_array_equal(prob.C_bits(), ref)
    finally:
        lib.nvfp4_gg_set_sm_count(0)
    check_full(d, ref)


def test_calls_after_shutdown_set_the_device_up_again(lib):
    """After nvfp4_gg_shutdown the next calls rebuild the device state, the
    kernels' shared-memory limits and the tensor maps: a decode call split
    in clusters and a prefill call on CTA pairs give the same bits as before
    it."""
    from nvfp4_block_scaled_masked_gb300.device import Problem
    ds = [W.generate(W.custom(1, 8, 2048, 7168, masked_m=[5]), seed=3),      # cluster split
          W.generate(W.custom(3, 200, 512, 768, masked_m=[200, 5, 130]), seed=4)]   # pairs
    probs = [Problem(d) for d in ds]
    before = []
    for prob in probs:
        prob.run()
        assert lib.nvfp4_gg_check_error() == 0
        before.append(prob.C_bits())
    lib.nvfp4_gg_shutdown()
    for d, prob, ref in zip(ds, probs, before):
        prob.reset_C()
        prob.run()
        assert lib.nvfp4_gg_check_error() == 0
        np.testing.assert_array_equal(prob.C_bits(), ref)
        check_full(d, ref)


def test_mma_peak_probe_runs_clean(lib):
    lib.nvfp4_gg_mma_peak_probe(64, 256)
    lib.nvfp4_gg_mma_peak_probe(64, 16, 3)
    lib.nvfp4_gg_mma_peak_probe_pair(64, 256)
    lib.nvfp4_gg_mma_peak_probe_pair(64, 32, 3)
    assert lib.nvfp4_gg_check_error() == 0


def test_masked_m_out_of_range_is_flagged(lib):
    from nvfp4_block_scaled_masked_gb300.device import Problem
    d = W.generate(W.custom(2, 16, 128, 256, masked_m=[16, 3]))
    prob = Problem(d)
    prob.masked_m.copy_(torch.tensor([17, 3], dtype=torch.int32))
    prob.run()
    assert lib.nvfp4_gg_check_error() == lib.ERR_MASK
    # clamped to M_max: the result equals the masked_m = [16, 3] result
    check_full(d, prob.C_bits())


def test_prepare_weights_roundtrip(lib):
    """Re-layout, then the inverse permutations on the CPU, gives back B and
    B_sf; rows past N are zero."""
    from nvfp4_block_scaled_masked_gb300 import binding
    G, N, K = 3, 272, 512
    rng = np.random.default_rng(4)
    bsf = rng.integers(0, 256, (G, N, K // 16), dtype=np.uint8)
    b = rng.integers(0, 256, (G, N, K // 2), dtype=np.uint8)
    bb, sb = binding.nvfp4_prepared_weight_bytes(G, N, K)
    dB, dBsf = torch.from_numpy(b).cuda(), torch.from_numpy(bsf).cuda()
    oB = torch.empty(bb, dtype=torch.uint8, device="cuda")
    oS = torch.empty(sb, dtype=torch.uint8, device="cuda")
    binding.nvfp4_prepare_weights(dB, dBsf, G, N, K, oB, oS)
    torch.cuda.synchronize()
    NT, KC, KS = (N + 127) // 128, K // 64, K // 256
    tiles = oB.cpu().numpy().reshape(G, NT, KS, 128, 8, 16)     # [g][nt][ks][r][chunk][byte]
    r = np.arange(128)[:, None]
    unswz = tiles[:, :, :, r, (np.arange(8)[None, :] ^ (r % 8)), :]   # chunk c read from c ^ r%8
    back_b = unswz.transpose(0, 1, 3, 2, 4, 5).reshape(G, NT * 128, K // 2)
    np.testing.assert_array_equal(back_b[:, :N], b)
    assert np.all(back_b[:, N:] == 0)
    atoms = oS.cpu().numpy().reshape(G, NT, KC, 32, 4, 4)      # [g][nt][kc][i][j][b]
    back = atoms.transpose(0, 1, 4, 3, 2, 5).reshape(G, NT * 128, KC * 4)   # row = 128nt+32j+i
    np.testing.assert_array_equal(back[:, :N], bsf)
    assert np.all(back[:, N:] == 0)
