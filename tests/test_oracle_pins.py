"""Pins for the CPU oracle: each test checks it against something other than
itself (a library routine, exact rational arithmetic, a published table, an
invariant of the mathematics), chosen so that a plausible slip anywhere in the
oracle (a wrong table entry, nibble order, scale index, sign, dropped term,
transposed operand, double rounding) fails at least one of them.

The operation is FlashInfer's grouped_gemm_nt_masked as the page "The
CuteDSL Gamble: Chasing Kernel Efficiency on Blackwell GPUs" describes it
(sections "The Message" and "Output Knowledge Created").
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle
from nvfp4_block_scaled_masked_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# e2m1 magnitudes as printed in the OCP Microscaling Formats (MX) v1.0
# specification's FP4 (E2M1) element format (see tests/golden/ocp_formats.json)
with open(os.path.join(GOLDEN, "ocp_formats.json")) as f:
    OCP = json.load(f)


# ---------------------------------------------------------------- P1 tables

def test_e2m1_all_codes_match_ocp_table():
    mags = [Fraction(x) for x in OCP["e2m1_magnitudes_by_low3bits"]]
    for code in range(16):
        want = mags[code & 7] * (-1 if code & 8 else 1)
        got = oracle.e2m1_value(code)
        assert got == float(want), (code, got, want)
        assert np.copysign(1.0, got) == (-1.0 if code & 8 else 1.0)
    np.testing.assert_array_equal(oracle.E2M1_TABLE, [oracle.e2m1_value(c) for c in range(16)])


def test_e2m1_decode_table_matches_ocp_and_bit_fields():
    """The C oracle decodes elements through a 16-entry table; every entry
    equals the OCP magnitude with the code's sign and the bit-field closed
    form, signed zero included."""
    mags = [Fraction(x) for x in OCP["e2m1_magnitudes_by_low3bits"]]
    for code in range(16):
        t = oracle.e2m1_table_value(code)
        assert t == float(mags[code & 7] * (-1 if code & 8 else 1)), code
        assert np.copysign(1.0, t) == (-1.0 if code & 8 else 1.0), code
        assert t == oracle.e2m1_value(code)


def test_e4m3_all_bytes_match_torch_float8_e4m3fn():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(b) for b in range(256)])
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(got), nan)
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF]
    np.testing.assert_array_equal(got[~nan], lib[~nan])
    np.testing.assert_array_equal(oracle.E4M3_TABLE[~nan], lib[~nan])


def test_e4m3_spot_values_from_ocp():
    for hexbyte, val in OCP["e4m3_spot_values"].items():
        assert oracle.e4m3_value(int(hexbyte, 16)) == float(Fraction(val)), hexbyte


def test_bf16_rne_matches_torch_on_float32_values():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(1000),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        np.array([1.0, -1.0, 3.0, 65504.0, 1e38, -1e38, 2.0 ** -126], dtype=np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in x], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)
    # the NumPy restatement agrees on the normal range
    normal = np.abs(x) >= 2.0 ** -126
    np.testing.assert_array_equal(oracle.bf16_bits_numpy(x[normal].astype(np.float64)), want[normal])


def test_bf16_rne_rounds_once_from_fp64():
    # 1 + 2^-8 is exactly halfway between bf16 1.0 and 1 + 2^-7: ties to even
    assert oracle.bf16_rne(1.0 + 2.0 ** -8) == 0x3F80
    # slightly above the tie must round up; going through fp32 first would
    # lose the 2^-30 and round down to even
    assert oracle.bf16_rne(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert oracle.bf16_rne(-(1.0 + 2.0 ** -8 + 2.0 ** -30)) == 0xBF81
    # odd neighbour: 1 + 3*2^-8 ties to the even 1 + 2^-6
    assert oracle.bf16_rne(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # carry into the next binade
    assert oracle.bf16_rne(2.0 - 2.0 ** -9) == 0x4000
    assert oracle.bf16_rne(0.0) == 0 and oracle.bf16_rne(-0.0) == 0x8000


# ------------------------------------------------ exact rational brute force

def _bf16_exact(fr: Fraction) -> int:
    """bf16 bits of the exact rational, one rounding, ties to even."""
    if fr == 0:
        return 0
    sign = 0x8000 if fr < 0 else 0
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q = Fraction(2) ** (max(e, -126) - 7)
    r = round(a / q) * q          # Fraction round(): half to even
    bits = np.array([float(r)], dtype=np.float32).view(np.uint32)[0] >> 16
    return sign | int(bits)


def _elem_exact(codes_row, sf_row, k):
    byte = int(codes_row[k // 2])
    code = (byte >> 4) if k % 2 else (byte & 15)
    mag = Fraction(OCP["e2m1_magnitudes_by_low3bits"][code & 7])
    s = int(sf_row[k // 16])
    e, m = (s >> 3) & 15, s & 7
    sc = Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7)
    return (-mag if code & 8 else mag) * sc


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_oracle_equals_exact_rational_arithmetic(seed):
    """Tiny shapes, any finite positive e4m3 scale (subnormals included), any
    codes: the oracle's fp64 value must equal alpha times the exact rational
    sum correctly rounded, and C its bf16 rounding."""
    rng = np.random.default_rng(seed)
    G, M, N, K = 2, 3, 4, 48
    A = rng.integers(0, 256, (G, M, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, (G, N, K // 2), dtype=np.uint8)
    A_sf = rng.integers(0, 0x7F, (G, M, K // 16), dtype=np.uint8)   # 0x00..0x7E
    B_sf = rng.integers(0, 0x7F, (G, N, K // 16), dtype=np.uint8)
    alpha = rng.uniform(0.5, 2.0, G).astype(np.float32)
    mm = np.array([3, 2], dtype=np.int32)
    C0 = np.full((G, M, N), 0x7FC0, dtype=np.uint16)
    C, ref = oracle.gemm(A, A_sf, B, B_sf, alpha, mm, C0, G, M, N, K)
    for g in range(G):
        for m in range(M):
            for n in range(N):
                if m >= mm[g]:
                    assert C[g, m, n] == 0x7FC0 and np.isnan(ref[g, m, n])
                    continue
                s = sum(_elem_exact(A[g, m], A_sf[g, m], k) * _elem_exact(B[g, n], B_sf[g, n], k)
                        for k in range(K))
                exact = Fraction(float(alpha[g])) * s
                assert ref[g, m, n] == float(exact)
                assert C[g, m, n] == _bf16_exact(exact), (g, m, n)


def test_single_nonzero_brute_force():
    """Every code pair x every scale pair of the workload set x every position
    k of a K=32 row, one non-zero per row: C must be the exact product (<= 4
    significant bits, so bf16-exact), which pins nibble order and the k/16
    scale index."""
    codes = np.arange(16)
    sc = W.SCALE_BYTES
    ca, cb, ia, ib, pos = np.meshgrid(codes, codes, np.arange(len(sc)), np.arange(len(sc)),
                                      np.arange(32), indexing="ij")
    ca, cb, ia, ib, pos = (x.ravel() for x in (ca, cb, ia, ib, pos))
    G = ca.size
    K = 32
    A = np.zeros((G, 1, K // 2), dtype=np.uint8)
    B = np.zeros((G, 1, K // 2), dtype=np.uint8)
    rows = np.arange(G)
    shift = (pos % 2) * 4
    A[rows, 0, pos // 2] = (ca << shift).astype(np.uint8)
    B[rows, 0, pos // 2] = (cb << shift).astype(np.uint8)
    # the block holding pos gets the drawn scale; the other block a decoy
    A_sf = np.full((G, 1, 2), 0x48, dtype=np.uint8)
    B_sf = np.full((G, 1, 2), 0x18, dtype=np.uint8)
    A_sf[rows, 0, pos // 16] = sc[ia]
    B_sf[rows, 0, pos // 16] = sc[ib]
    alpha = np.ones(G, dtype=np.float32)
    mm = np.ones(G, dtype=np.int32)
    C, ref = oracle.gemm(A, A_sf, B, B_sf, alpha, mm, np.zeros((G, 1, 1), np.uint16), G, 1, 1, K)
    e2m1 = np.array([float(Fraction(OCP["e2m1_magnitudes_by_low3bits"][c & 7])) * (-1 if c & 8 else 1)
                     for c in range(16)])
    e4m3 = torch.from_numpy(sc.copy()).view(torch.float8_e4m3fn).double().numpy()
    want = e2m1[ca] * e2m1[cb] * e4m3[ia] * e4m3[ib]
    np.testing.assert_array_equal(ref[:, 0, 0], want)
    want_bits = torch.from_numpy(want).float().to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = C[:, 0, 0]
    # +0 and -0 are both correct for an exact zero
    zero = want == 0
    np.testing.assert_array_equal(got[~zero], want_bits[~zero])
    assert np.all((got[zero] == 0) | (got[zero] == 0x8000))


def test_integer_special_case_is_int64_matmul():
    """All scales 1.0 (0x38), alpha 1, codes for 0, 1, -1, 2: C must be the
    integer matrix product (numpy int64 matmul), rounded to bf16."""
    rng = np.random.default_rng(11)
    G, M, N, K = 3, 5, 7, 64
    vals = np.array([0, 1, -1, 2])
    codes = np.array([0x0, 0x2, 0xA, 0x4], dtype=np.uint8)
    ia = rng.integers(0, 4, (G, M, K))
    ib = rng.integers(0, 4, (G, N, K))
    pack = lambda i: (codes[i[..., 0::2]] | (codes[i[..., 1::2]] << 4)).astype(np.uint8)
    A, B = pack(ia), pack(ib)
    A_sf = np.full((G, M, K // 16), 0x38, np.uint8)
    B_sf = np.full((G, N, K // 16), 0x38, np.uint8)
    mm = np.array([5, 0, 3], dtype=np.int32)
    C, ref = oracle.gemm(A, A_sf, B, B_sf, np.ones(G, np.float32), mm,
                         np.full((G, M, N), 0x7FC0, np.uint16), G, M, N, K)
    for g in range(G):
        want = vals[ia[g]].astype(np.int64) @ vals[ib[g]].astype(np.int64).T
        np.testing.assert_array_equal(ref[g, :mm[g]], want[:mm[g]])
        bits = torch.from_numpy(want[:mm[g]]).float().to(torch.bfloat16).view(torch.int16).numpy()
        np.testing.assert_array_equal(C[g, :mm[g]], bits.astype(np.uint16))
        assert np.all(C[g, mm[g]:] == 0x7FC0)


def test_short_k_float32_sum_is_exact():
    """With the workload's power-of-two scales and K <= 28 every partial sum
    is exact in fp32 too: the oracle's fp64 result equals a float32 BLAS
    product of the decoded operands bit for bit (the exactness argument)."""
    cfg = W.custom(2, 6, 8, 16, masked_m=[6, 4])
    d = W.generate(cfg, seed=5)
    C, ref = oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"], np.ones(2, np.float32),
                         d["masked_m"], d["C_init"], 2, 6, 8, 16)
    Ad = oracle.decode_numpy(d["A"], d["A_sf"], 16).astype(np.float32)
    Bd = oracle.decode_numpy(d["B"], d["B_sf"], 16).astype(np.float32)
    for g in range(2):
        m = d["masked_m"][g]
        f32 = (Ad[g, :m] @ Bd[g].T).astype(np.float64)
        np.testing.assert_array_equal(ref[g, :m], f32)


# ------------------------------------------------------- second implementation

@pytest.mark.parametrize("key", ["c1"])
def test_c_oracle_matches_numpy_restatement(key):
    cfg = W.CONFIGS[key]
    d = W.generate(cfg)
    args = (d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], d["masked_m"], d["C_init"],
            cfg.G, cfg.M_max, cfg.N, cfg.K)
    C1, r1 = oracle.gemm(*args)
    C2, r2 = oracle.gemm_numpy(*args)
    np.testing.assert_array_equal(C1, C2)
    np.testing.assert_array_equal(r1, r2)


def test_sampled_matches_full():
    cfg = W.CONFIGS["c1"]
    d = W.generate(cfg)
    C, ref = oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], d["masked_m"],
                         d["C_init"], cfg.G, cfg.M_max, cfg.N, cfg.K)
    rng = np.random.default_rng(0)
    idx = []
    for g in range(cfg.G):
        for _ in range(50):
            if d["masked_m"][g]:
                idx.append((g, rng.integers(d["masked_m"][g]), rng.integers(cfg.N)))
    idx = np.array(idx)
    s = oracle.gemm_sampled(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], idx,
                            cfg.G, cfg.M_max, cfg.N, cfg.K)
    np.testing.assert_array_equal(s, ref[idx[:, 0], idx[:, 1], idx[:, 2]])


# ------------------------------------------------------------------ invariants

def _run(d, cfg, alpha=None):
    return oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"],
                       d["alpha"] if alpha is None else alpha, d["masked_m"], d["C_init"],
                       cfg.G, cfg.M_max, cfg.N, cfg.K)


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("j", [-2, 1])
def test_alpha_power_of_two_linearity(j):
    cfg = W.CONFIGS["c1"]
    d = W.generate(cfg)
    C, _ = _run(d, cfg)
    Cj, _ = _run(d, cfg, alpha=(d["alpha"] * np.float32(2.0 ** j)).astype(np.float32))
    for g in range(cfg.G):
        m = d["masked_m"][g]
        np.testing.assert_array_equal(_bf16_to_f64(Cj[g, :m]), _bf16_to_f64(C[g, :m]) * 2.0 ** j)


def test_masked_rows_and_empty_groups_untouched_and_poison_ignored():
    cfg = W.CONFIGS["c1"]
    d = W.generate(cfg)
    p = W.generate(cfg, poison=True)
    C, _ = _run(d, cfg)
    Cp, _ = _run(p, cfg)
    for g in range(cfg.G):
        m = d["masked_m"][g]
        assert np.all(C[g, m:] == W.SENTINEL_BF16)
        valid = C[g, :m]
        assert not np.any(valid == W.SENTINEL_BF16)
        assert np.all(np.isfinite(_bf16_to_f64(valid)))
    np.testing.assert_array_equal(C, Cp)
    assert d["masked_m"][0] == 0 and np.all(C[0] == W.SENTINEL_BF16)


def test_permutation_symmetry():
    cfg = W.custom(3, 8, 32, 64, masked_m=[8, 3, 5])
    d = W.generate(cfg, seed=3)
    C, _ = _run(d, cfg)
    perm = np.array([2, 0, 1])
    q = {k: (v[perm] if isinstance(v, np.ndarray) and v.shape[:1] == (3,) else v) for k, v in d.items()}
    cfgp = W.custom(3, 8, 32, 64, masked_m=d["masked_m"][perm])
    Cp, _ = _run(q, cfgp)
    np.testing.assert_array_equal(Cp, C[perm])
    # permuting the rows of B permutes the columns of C
    cols = np.random.default_rng(0).permutation(32)
    r = dict(d)
    r["B"], r["B_sf"] = d["B"][:, cols], d["B_sf"][:, cols]
    Cc, _ = _run(r, cfg)
    np.testing.assert_array_equal(Cc, C[:, :, cols])


def test_oracle_rejects_bad_arguments():
    cfg = W.custom(1, 4, 8, 32, masked_m=[5])   # masked_m > M_max
    with pytest.raises(AssertionError):
        W.generate(cfg)
    d = W.generate(W.custom(1, 4, 8, 32, masked_m=[4]))
    with pytest.raises(ValueError):
        oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], np.array([5], np.int32),
                    d["C_init"], 1, 4, 8, 32)


# --------------------------------------------------------------- golden fixture

def test_golden_tiny_case_regression():
    """A tiny case frozen by tests/golden/make_golden.py (which calls only the
    oracle): inputs and expected output bits are stored as hex text."""
    with open(os.path.join(GOLDEN, "tiny_case.json")) as f:
        gd = json.load(f)
    G, M, N, K = gd["G"], gd["M_max"], gd["N"], gd["K"]
    h = lambda s, shape: np.frombuffer(bytes.fromhex(s), dtype=np.uint8).reshape(shape)
    A, A_sf = h(gd["A"], (G, M, K // 2)), h(gd["A_sf"], (G, M, K // 16))
    B, B_sf = h(gd["B"], (G, N, K // 2)), h(gd["B_sf"], (G, N, K // 16))
    alpha = np.array(gd["alpha"], dtype=np.float32)
    mm = np.array(gd["masked_m"], dtype=np.int32)
    C, ref = oracle.gemm(A, A_sf, B, B_sf, alpha, mm, np.full((G, M, N), 0x7FC0, np.uint16),
                         G, M, N, K)
    np.testing.assert_array_equal(C.ravel(), np.array(gd["C_bits"], dtype=np.uint16))


# ------------------------------------------------ SwiGLU step after GEMM1

def test_silu_closed_forms():
    """sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4 give silu(+-ln 3) in closed
    form; silu(x) - silu(-x) = x for every x; the limits at +-infinity."""
    ln3 = np.log(3.0)
    assert oracle.silu(0.0) == 0.0
    np.testing.assert_allclose(oracle.silu(ln3), 0.75 * ln3, rtol=4e-16)
    np.testing.assert_allclose(oracle.silu(-ln3), -0.25 * ln3, rtol=4e-16)
    x = np.random.default_rng(3).normal(0, 20, 1000)
    np.testing.assert_allclose(oracle.silu(x) - oracle.silu(-x), x, rtol=1e-12, atol=1e-12)
    assert oracle.silu(1000.0) == 1000.0
    assert oracle.silu(-1000.0) == 0.0


def _one_token_gemm1(gate_vals, up_vals):
    """G=1, one token with the value 1 at k = 0 (scale 1.0); weight row j holds
    its value at k = 0 (e2m1 code times an e4m3 scale), so h_j is that value."""
    N, K = 2 * len(gate_vals), 16
    enc = {1: (0x2, 0x38), 3: (0x5, 0x38), 6: (0x7, 0x38), 24: (0x7, 0x48), -24: (0xF, 0x48)}
    A = np.zeros((1, 1, K // 2), np.uint8)
    A[0, 0, 0] = 0x2
    A_sf = np.full((1, 1, K // 16), 0x38, np.uint8)
    B = np.zeros((1, N, K // 2), np.uint8)
    B_sf = np.full((1, N, K // 16), 0x38, np.uint8)
    for j, v in enumerate(list(gate_vals) + list(up_vals)):
        B[0, j, 0], B_sf[0, j, 0] = enc[v]
    mm = np.array([1], np.int32)
    _, ref = oracle.gemm(A, A_sf, B, B_sf, np.ones(1, np.float32), mm,
                         np.zeros((1, 1, N), np.uint16), 1, 1, N, K)
    return ref, mm


def test_swiglu_gate_is_the_first_half():
    """h = [gate | up] = [24, -24 | 3, 6]: out = silu(24)*3 rounds to exactly 72
    (the swapped reading would give silu(3)*24 = 68.6), and silu(-24)*6 is a
    tiny negative number, not silu(6)*(-24) = -143.6."""
    ref, mm = _one_token_gemm1([24, -24], [3, 6])
    np.testing.assert_array_equal(ref[0, 0], [24.0, -24.0, 3.0, 6.0])
    C, out = oracle.swiglu(ref, mm, np.zeros((1, 1, 2), np.uint16))
    assert C[0, 0, 0] == 0x4290                    # bf16(72.0)
    assert -1e-8 < out[0, 0, 1] < 0


def test_swiglu_is_linear_in_up_and_not_in_gate():
    """Doubling every up-row scale (e4m3 exponent + 1) doubles the output
    exactly; doubling the gate-row scales does not."""
    G, M, N, K = 2, 6, 64, 256
    d = W.generate(W.custom(G, M, N, K, masked_m=[6, 3]), seed=21)
    init = np.full((G, M, N // 2), 0x7FC0, np.uint16)

    def run(B_sf):
        _, ref = oracle.gemm(d["A"], d["A_sf"], d["B"], B_sf, d["alpha"], d["masked_m"],
                             d["C_init"], G, M, N, K)
        return oracle.swiglu(ref, d["masked_m"], init)

    C0, y0 = run(d["B_sf"])
    up2 = d["B_sf"].copy()
    up2[:, N // 2:] += 8
    C1, y1 = run(up2)
    gate2 = d["B_sf"].copy()
    gate2[:, :N // 2] += 8
    _, y2 = run(gate2)
    for g in range(G):
        m = d["masked_m"][g]
        np.testing.assert_array_equal(y1[g, :m], 2.0 * y0[g, :m])
        assert not np.allclose(y2[g, :m], 2.0 * y0[g, :m])
        assert np.all(C0[g, m:] == 0x7FC0) and np.all(C1[g, m:] == 0x7FC0)


def test_bf16_bits_any_subnormal_grid():
    vals = np.array([1.0, -2.0 ** -130, 1.5 * 2.0 ** -133, 2.5 * 2.0 ** -133, 128 * 2.0 ** -133, -0.0])
    want = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    np.testing.assert_array_equal(oracle.bf16_bits_any(vals), want.astype(np.uint16))


# ---------------------------------------------------- W4A16 decode GEMV

def test_gemv_one_hot_reads_one_weight_column():
    """x = 2^j at position k, zero elsewhere: y[n] = alpha * 2^j * code * scale
    of weight element (n, k), from the OCP tables by hand."""
    N, K = 4, 64
    B = np.zeros((N, K // 2), np.uint8)
    B_sf = np.full((N, K // 16), 0x38, np.uint8)
    k = 37                                     # odd: high nibble of byte 18, scale block 2
    codes = [0x5, 0xF, 0x1, 0x0]               # 3, -6, 0.5, 0
    scales = [0x40, 0x30, 0x48, 0x38]          # 2, 0.5, 4, 1
    for n in range(N):
        B[n, k // 2] = codes[n] << 4
        B_sf[n, k // 16] = scales[n]
    x = np.zeros((1, K), np.uint16)
    x[0, k] = 0x4000                           # 2.0
    bits, y = oracle.gemv_w4a16(x, B, B_sf, 0.75, K)
    np.testing.assert_array_equal(y[0], 0.75 * 2.0 * np.array([3 * 2, -6 * 0.5, 0.5 * 4, 0]))
    want = torch.tensor(y[0], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy()
    np.testing.assert_array_equal(bits[0], want.astype(np.uint16))


def test_gemv_integer_case_is_int64_matmul():
    rng = np.random.default_rng(5)
    M, N, K = 3, 9, 96
    vals = np.array([0, 1, -1, 2])
    codes = np.array([0x0, 0x2, 0xA, 0x4], dtype=np.uint8)
    ib = rng.integers(0, 4, (N, K))
    B = (codes[ib[:, 0::2]] | (codes[ib[:, 1::2]] << 4)).astype(np.uint8)
    B_sf = np.full((N, K // 16), 0x38, np.uint8)
    xi = rng.integers(-3, 4, (M, K))
    x = torch.from_numpy(xi.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    _, y = oracle.gemv_w4a16(x, B, B_sf, 1.0, K)
    np.testing.assert_array_equal(y, (xi.astype(np.int64) @ vals[ib].T).astype(np.float64))


# ---------------------------------------------------------------- NVFP4 quantiser

def _bf16_bits_exact(v):
    """bf16 bits of float32 values that bf16 holds exactly (asserted)."""
    f = np.asarray(v, dtype=np.float32)
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def test_e4m3_encode_matches_torch_in_range():
    """Round to nearest even on the e4m3 grid, checked against torch's
    float32 -> float8_e4m3fn conversion for values within [0, 448]."""
    rng = np.random.default_rng(5)
    s = np.concatenate([rng.uniform(0, 448, 20000), 2.0 ** rng.uniform(-12, 8.8, 20000),
                        oracle._E4M3_POS[:-1] + np.diff(oracle._E4M3_POS) / 2]).astype(np.float32)
    s = s[s <= 448]
    ref = torch.from_numpy(s).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(s), ref)


def test_e4m3_encode_ties_and_saturation():
    cases = {1.0625: 0x38, 1.1875: 0x3A, 2.0 ** -10: 0x00, 3 * 2.0 ** -10: 0x02, 448.0: 0x7E,
             463.0: 0x7E, 500.0: 0x7E, 1e30: 0x7E, 0.0: 0x00}
    got = oracle.e4m3_encode(np.float32(list(cases)))
    assert list(got) == list(cases.values())


def test_e2m1_encode_ties_signs_saturation():
    # midpoints go to the even code: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0,
    # 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4; beyond 6 saturates; -0 is +0
    w = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 1e9, -0.25, -0.3, -5.0, -7.0, 0.0, -0.0])
    want = [0, 2, 2, 4, 4, 6, 6, 7, 7, 0, 9, 14, 15, 0, 0]
    assert list(oracle.e2m1_encode(w)) == want


def _exact_blocks(rng, R, L, sf_lo=0x01, sf_hi=0x70):
    """Blocks code * d with one element of every block at +-6 (so the block's
    scale is d exactly), codes != -0, d a positive e4m3 value."""
    codes = rng.integers(0, 15, (R, L)).astype(np.uint8)
    codes[codes >= 8] += 1                             # skip 0x8 (-0)
    blk = codes.reshape(R, L // 16, 16)
    pos = rng.integers(0, 16, (R, L // 16))
    sign = rng.integers(0, 2, (R, L // 16)).astype(np.uint8) << 3
    np.put_along_axis(blk, pos[..., None], (7 | sign)[..., None], axis=-1)
    sf = rng.integers(sf_lo, sf_hi + 1, (R, L // 16)).astype(np.uint8)
    vals = oracle.E2M1_TABLE[codes] * np.repeat(oracle.E4M3_TABLE[sf], 16, axis=-1)
    return codes, sf, _bf16_bits_exact(vals.astype(np.float32))


def test_quantize_round_trips_exact_blocks():
    """Encoding values that are exactly code * d, with the block maximum at
    6 d, returns those codes and d's byte (subnormal scales included); this
    fixes the block grouping, the nibble order and the code table."""
    rng = np.random.default_rng(11)
    codes, sf, x = _exact_blocks(rng, 7, 256)
    got_c, got_sf = oracle.quantize_nvfp4(x, np.ones(7, np.float32))
    np.testing.assert_array_equal(got_sf, sf)
    np.testing.assert_array_equal(got_c, (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))


def test_quantize_midpoints_round_to_even_codes():
    d = 0.5                                            # byte 0x30
    m = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -2.5, -5.0, 4.0, -6.0, 0.0, 1.0]
    want = [7, 0, 2, 2, 4, 4, 6, 6, 0, 10, 12, 14, 6, 15, 0, 2]
    x = _bf16_bits_exact(np.float32(m) * np.float32(d))[None, :]
    c, sf = oracle.quantize_nvfp4(x, np.ones(1, np.float32))
    assert sf[0, 0] == 0x30
    got = [int(c[0, j // 2] >> (4 * (j & 1)) & 15) for j in range(16)]
    assert got == want


def test_quantize_prescale_power_of_two_shifts_the_scale_byte():
    """q -> 2^j q leaves the codes and moves the scale byte by 8 j (one e4m3
    exponent step per factor 2) while the scale stays normal and unsaturated."""
    rng = np.random.default_rng(12)
    _, _, x = _exact_blocks(rng, 3, 64, sf_lo=0x30, sf_hi=0x48)
    c0, s0 = oracle.quantize_nvfp4(x, np.ones(3, np.float32))
    for j in (-2, 1, 3):
        c, s = oracle.quantize_nvfp4(x, np.full(3, 2.0 ** j, np.float32))
        np.testing.assert_array_equal(c, c0)
        np.testing.assert_array_equal(s.astype(int), s0.astype(int) + 8 * j)


def test_quantize_zero_tiny_and_saturating_blocks():
    x = np.zeros((1, 48), np.uint16)
    x[0, 16:32] = _bf16_bits_exact(np.full(16, 2.0 ** -20, np.float32))     # amax / 6 < 2^-10
    blk = np.full(16, 1.0, np.float32)
    blk[3] = 6.25                                      # amax / 6 = 1.04 -> scale 1.0, w = 6.25 -> 6
    x[0, 32:] = _bf16_bits_exact(blk)
    c, sf = oracle.quantize_nvfp4(x, np.ones(1, np.float32))
    assert list(sf[0]) == [0, 0, 0x38]
    assert np.all(c[0, :16] == 0)
    third = [int(c[0, 16 + j // 2] >> (4 * (j & 1)) & 15) for j in range(16)]
    assert third == [2, 2, 2, 7] + [2] * 12


def test_quantize_error_bound():
    """Every decoded element lies within half a grid step of z = x q: at
    most d / 4 where |z| <= 2 d, at most d elsewhere (steps 0.5, 1, 2 times d;
    saturation adds at most 0.375 d, covered by the second bound since
    amax / d <= 6 * (1 + 1/16))."""
    rng = np.random.default_rng(13)
    R, L = 9, 512
    sign = rng.integers(0, 2, (R, L)).astype(np.uint16)
    exp = rng.integers(120, 135, (R, L)).astype(np.uint16)          # 2^-7 .. 2^8
    x = (sign << 15) | (exp << 7) | rng.integers(0, 128, (R, L)).astype(np.uint16)
    q = np.float32(2.0) ** rng.integers(-6, 3, R).astype(np.float32)   # scales stay in range
    c, sf = oracle.quantize_nvfp4(x, q)
    z = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64) * q[:, None].astype(np.float64)
    dec = oracle.decode_numpy(c, sf, L)
    d = np.repeat(oracle.E4M3_TABLE[sf], 16, axis=-1)
    assert np.all(d > 0) and np.all(sf < 0x7E)
    err = np.abs(dec - z)
    small = np.abs(z) <= 2 * d
    assert np.all(err[small] <= d[small] / 4 * (1 + 1e-6))
    assert np.all(err <= d * (1 + 1e-6))


def _nearest_even(v: Fraction, grid):
    """Brute force over every grid point (exact rationals): the nearest one,
    ties to the even index, beyond the last point the last."""
    if v >= grid[-1]:
        return len(grid) - 1
    best, best_d = 0, abs(v - grid[0])
    for i, g in enumerate(grid[1:], 1):
        d = abs(v - g)
        if d < best_d or (d == best_d and i % 2 == 0):
            best, best_d = i, d
    return best


def test_quantize_matches_scalar_rational_brute_force():
    """A second, scalar restatement of the encoder: float32 steps with numpy
    scalars, every grid decision by exhaustive search in exact rationals."""
    e4 = [Fraction(float(v)) for v in oracle._E4M3_POS]
    e2 = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    rng = np.random.default_rng(14)
    R, L = 4, 64
    sign = rng.integers(0, 2, (R, L)).astype(np.uint16)
    exp = rng.integers(100, 140, (R, L)).astype(np.uint16)
    x = (sign << 15) | (exp << 7) | rng.integers(0, 128, (R, L)).astype(np.uint16)
    x[1, 16:32] = 0                                        # a zero block
    x[2, :16] = _bf16_bits_exact(np.float32([6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5] * 2) * np.float32(0.125))
    q = np.float32([1.0, 0.37, 2.0 ** -3, 3.1])
    c, sf = oracle.quantize_nvfp4(x, q)
    for r in range(R):
        for b in range(L // 16):
            z = []
            for i in range(16):
                xi = np.uint32(int(x[r, 16 * b + i]) << 16).view(np.float32)
                z.append(np.float32(xi * q[r]))
            amax = max(abs(v) for v in z)
            s = np.float32(np.float32(amax) / np.float32(6.0))
            sb = _nearest_even(Fraction(float(s)), e4)
            assert sf[r, b] == sb
            d = np.float32(float(e4[sb]))
            for i in range(16):
                if d > 0:
                    w = np.float32(z[i] / d)
                    m = _nearest_even(Fraction(abs(float(w))), e2)
                    code = m | (8 if (w < 0 and m > 0) else 0)
                else:
                    code = 0
                got = int(c[r, 8 * b + i // 2]) >> (4 * (i & 1)) & 15
                assert got == code, (r, b, i, float(w), got, code)
