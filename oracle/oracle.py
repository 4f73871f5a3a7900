"""CPU oracle for the masked, block-scaled NVFP4 grouped GEMM-NT.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA library and never imports it.

Two implementations live here, written independently of each other:

* ``gemm`` / ``gemm_sampled`` call the plain C oracle (``nvfp4_oracle.c``),
  fp64, built with gcc (OpenMP over independent output rows only).
* ``gemm_numpy`` is a second, NumPy fp64 restatement used to cross-check the
  C oracle on small shapes (table lookup, scale broadcast, ``einsum``).
* ``gemv_w4a16`` is the decode GEMV with bf16 activations, the plain fp64
  product of the decoded weights and the activations.
* ``swiglu`` applies the MoE block's SwiGLU step to GEMM1's unrounded fp64
  output (``silu(gate) * up``, one bf16 rounding), for the fused GEMM1
  epilogue.
* ``quantize_nvfp4`` encodes bf16 activations as NVFP4 for GEMM2's A
  (float32 steps, each rounded as IEEE prescribes; see its docstring).

The operation is the one the page "The CuteDSL Gamble: Chasing Kernel
Efficiency on Blackwell GPUs" describes for FlashInfer's
``grouped_gemm_nt_masked`` (sections "The Message" and "Output Knowledge
Created"): per expert g and row m < masked_m[g],
``C[g,m,n] = bf16(alpha[g] * sum_k A[g,m,k] * B[g,n,k])`` with NVFP4 operands
(e2m1 codes, one e4m3 scale per 16 K-elements); rows at or past masked_m[g]
are not written.  The NVFP4 encodings are not defined on the pages; the
readings (OCP e2m1 / e4m3, low nibble = even k, fp64 -> bf16 round to nearest
even) are stated in ``nvfp4_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libnvfp4_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (strict IEEE: no fast-math, no FMA
    contraction, so x86 and Arm builds round identically)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.nvfp4o_e2m1_value.restype = ctypes.c_double
        lib.nvfp4o_e2m1_value.argtypes = [ctypes.c_int]
        lib.nvfp4o_e2m1_table.restype = ctypes.c_double
        lib.nvfp4o_e2m1_table.argtypes = [ctypes.c_int]
        lib.nvfp4o_e4m3_value.restype = ctypes.c_double
        lib.nvfp4o_e4m3_value.argtypes = [ctypes.c_int]
        lib.nvfp4o_bf16_rne.restype = ctypes.c_uint16
        lib.nvfp4o_bf16_rne.argtypes = [ctypes.c_double]
        lib.nvfp4o_max_threads.restype = ctypes.c_int
        lib.nvfp4o_gemm.restype = ctypes.c_int
        lib.nvfp4o_gemm.argtypes = [u8p, u8p, u8p, u8p, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p] + [ctypes.c_int] * 5
        lib.nvfp4o_gemm_sampled.restype = ctypes.c_int
        lib.nvfp4o_gemm_sampled.argtypes = [u8p, u8p, u8p, u8p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int64,
                                            ctypes.c_void_p] + [ctypes.c_int] * 5
        _lib = lib
    return _lib


def _u8(a):
    a = np.ascontiguousarray(a, dtype=np.uint8)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


def e2m1_value(code: int) -> float:
    """e2m1 value from the code's bit fields (sign, exponent, mantissa)."""
    return _load().nvfp4o_e2m1_value(int(code))


def e2m1_table_value(code: int) -> float:
    """Entry `code` of the C oracle's 16-entry e2m1 table, through which it
    decodes every element."""
    return _load().nvfp4o_e2m1_table(int(code))


def e4m3_value(byte: int) -> float:
    return _load().nvfp4o_e4m3_value(int(byte))


def bf16_rne(x: float) -> int:
    return int(_load().nvfp4o_bf16_rne(float(x)))


def max_threads() -> int:
    return int(_load().nvfp4o_max_threads())


def gemm(A, A_sf, B, B_sf, alpha, masked_m, C_init, G, M_max, N, K,
         nthreads: int = 0, want_ref64: bool = True):
    """Full oracle.  Returns (C bf16 bits as uint16 [G,M_max,N], ref64 f64
    [G,M_max,N] or None).  C starts as a copy of C_init (uint16 bits); only
    rows m < masked_m[g] are written.  ref64 holds NaN where not written."""
    lib = _load()
    A, pA = _u8(A)
    A_sf, pAs = _u8(A_sf)
    B, pB = _u8(B)
    B_sf, pBs = _u8(B_sf)
    alpha = np.ascontiguousarray(alpha, dtype=np.float32)
    masked_m = np.ascontiguousarray(masked_m, dtype=np.int32)
    C = np.array(C_init, dtype=np.uint16, copy=True).reshape(G, M_max, N)
    ref = np.full((G, M_max, N), np.nan) if want_ref64 else None
    rc = lib.nvfp4o_gemm(pA, pAs, pB, pBs, alpha.ctypes.data, masked_m.ctypes.data,
                         C.ctypes.data, ref.ctypes.data if ref is not None else None,
                         G, M_max, N, K, nthreads)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return C, ref


def gemm_sampled(A, A_sf, B, B_sf, alpha, idx, G, M_max, N, K, nthreads: int = 0):
    """Unrounded fp64 alpha*sum for each (g, m, n) row of idx (int64 [n,3])."""
    lib = _load()
    A, pA = _u8(A)
    A_sf, pAs = _u8(A_sf)
    B, pB = _u8(B)
    B_sf, pBs = _u8(B_sf)
    alpha = np.ascontiguousarray(alpha, dtype=np.float32)
    idx = np.ascontiguousarray(idx, dtype=np.int64).reshape(-1, 3)
    out = np.empty(idx.shape[0], dtype=np.float64)
    rc = lib.nvfp4o_gemm_sampled(pA, pAs, pB, pBs, alpha.ctypes.data, idx.ctypes.data,
                                 idx.shape[0], out.ctypes.data, G, M_max, N, K, nthreads)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return out


# ---------------------------------------------------------------------------
# Second implementation (NumPy fp64), independent of the C code above.
# ---------------------------------------------------------------------------

# e2m1 magnitudes by the 3 low bits (OCP FP4 E2M1): subnormal 0, 0.5; then
# 1, 1.5, 2, 3, 4, 6.  Bit 3 is the sign.
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
E2M1_TABLE = np.concatenate([_E2M1_MAG, -_E2M1_MAG])


def _e4m3_table() -> np.ndarray:
    t = np.empty(256)
    for b in range(256):
        s, e, m = b >> 7, (b >> 3) & 15, b & 7
        if e == 15 and m == 7:
            t[b] = np.nan
            continue
        v = m * 2.0 ** -9 if e == 0 else (8 + m) * 2.0 ** (e - 10)
        t[b] = -v if s else v
    return t


E4M3_TABLE = _e4m3_table()


def decode_numpy(codes, sf, K):
    """Dense fp64 [..., rows, K] from packed codes [..., rows, K/2] and scales
    [..., rows, K/16]."""
    codes = np.asarray(codes, dtype=np.uint8)
    lo = E2M1_TABLE[codes & 15]
    hi = E2M1_TABLE[codes >> 4]
    vals = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], K)
    scale = np.repeat(E4M3_TABLE[np.asarray(sf, dtype=np.uint8)], 16, axis=-1)
    return vals * scale


def gemm_numpy(A, A_sf, B, B_sf, alpha, masked_m, C_init, G, M_max, N, K):
    """NumPy fp64 restatement: returns (C bits uint16, ref64 with NaN where
    not written).  The bf16 rounding works on the fp64 bit pattern directly
    (a different method from the C oracle's scale-and-nearbyint)."""
    Ad = decode_numpy(np.asarray(A).reshape(G, M_max, K // 2),
                      np.asarray(A_sf).reshape(G, M_max, K // 16), K)
    Bd = decode_numpy(np.asarray(B).reshape(G, N, K // 2),
                      np.asarray(B_sf).reshape(G, N, K // 16), K)
    C = np.array(C_init, dtype=np.uint16, copy=True).reshape(G, M_max, N)
    ref = np.full((G, M_max, N), np.nan)
    for g in range(G):
        mm = int(masked_m[g])
        if mm == 0:
            continue
        acc = np.einsum("mk,nk->mn", Ad[g, :mm], Bd[g])
        v = np.float64(np.float32(alpha[g])) * acc
        ref[g, :mm] = v
        C[g, :mm] = bf16_bits_numpy(v)
    return C, ref


def bf16_bits_numpy(x) -> np.ndarray:
    """fp64 -> bf16 bits, round to nearest even, computed on the fp64 bit
    pattern (52-bit mantissa, keep 7).  Finite normal inputs in bf16's normal
    range only; anything else raises."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    if np.any(~np.isfinite(x)) or np.any((ax != 0) & (ax < 2.0 ** -126)) or np.any(ax >= 2.0 ** 128):
        raise ValueError("bf16_bits_numpy: value outside the normal bf16 range")
    bits = x.view(np.uint64)
    sign = (bits >> np.uint64(63)).astype(np.uint64)
    exp = ((bits >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64)
    man = bits & np.uint64((1 << 52) - 1)
    keep = man >> np.uint64(45)                  # top 7 mantissa bits
    rest = man & np.uint64((1 << 45) - 1)
    half = np.uint64(1 << 44)
    up = (rest > half) | ((rest == half) & ((keep & np.uint64(1)) == 1))
    mant = keep + up.astype(np.uint64)
    e = exp - 1023 + 127
    carry = mant >> np.uint64(7)
    mant = mant & np.uint64(0x7F)
    e = e + carry.astype(np.int64)
    out = (sign << np.uint64(15)) | (e.astype(np.uint64) << np.uint64(7)) | mant
    out = np.where(ax == 0, sign << np.uint64(15), out)
    if np.any(e >= 255):
        raise ValueError("bf16_bits_numpy: overflow")
    return out.astype(np.uint16)


def bf16_bits_any(x) -> np.ndarray:
    """fp64 -> bf16 bits, round to nearest even, over bf16's whole finite range:
    the normal range as bf16_bits_numpy, below 2^-126 onto bf16's subnormal
    grid (multiples of 2^-133, ties to even; 128 * 2^-133 is the smallest
    normal)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    tiny = np.abs(x) < 2.0 ** -126
    if np.any(~tiny):
        out[~tiny] = bf16_bits_numpy(x[~tiny])
    if np.any(tiny):
        k = np.rint(np.abs(x[tiny]) / 2.0 ** -133).astype(np.uint16)   # rint: ties to even
        out[tiny] = (np.signbit(x[tiny]).astype(np.uint16) << np.uint16(15)) | k
    return out


def silu(x):
    """silu(x) = x * sigmoid(x) = x / (1 + e^-x), fp64 (e^-x overflowing to
    inf gives the limit 0)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def swiglu(ref64, masked_m, C_init_half):
    """The SwiGLU step after GEMM1 in the MoE expert block of the page
    "LLM-Assisted Kernel Development in CuTe DSL, Gluon, Helion and Triton"
    (mixture-of-experts section: each expert runs GEMM1, SwiGLU, GEMM2).  From
    GEMM1's unrounded fp64 output ref64 [G, M_max, N] (N = 2I; reading: the
    first I columns are the gate projection, the last I the up projection):
    out[g, m, j] = silu(ref64[g, m, j]) * ref64[g, m, I + j] in fp64, rounded
    once to bf16.  Returns (C bits uint16 [G, M_max, I], a copy of
    C_init_half with rows m < masked_m[g] written; out64 with NaN elsewhere)."""
    G, M_max, N = ref64.shape
    I = N // 2
    C = np.array(C_init_half, dtype=np.uint16, copy=True).reshape(G, M_max, I)
    out = np.full((G, M_max, I), np.nan)
    for g in range(G):
        m = int(masked_m[g])
        if m == 0:
            continue
        y = silu(ref64[g, :m, :I]) * ref64[g, :m, I:]
        out[g, :m] = y
        C[g, :m] = bf16_bits_any(y)
    return C, out


# Non-negative finite e4m3 values, byte 0x00 .. 0x7E in increasing order.
_E4M3_POS = E4M3_TABLE[:127].copy()


def _round_to_grid(v, grid):
    """Index of the nearest grid point to each v >= 0 (grid ascending, exact
    in fp64; v float32 or fp64), ties to the even index, values beyond the
    last point to the last (saturation)."""
    v = np.asarray(v, dtype=np.float64)
    hi = np.clip(np.searchsorted(grid, v, side="left"), 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_lo = v - grid[lo]
    d_hi = grid[hi] - v
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    return np.where(v >= grid[-1], len(grid) - 1, idx)


def e4m3_encode(s):
    """e4m3 byte of each s >= 0 (float32): round to nearest, ties to even
    (the even byte: its low bit is the mantissa's), saturating at 448."""
    return _round_to_grid(s, _E4M3_POS).astype(np.uint8)


def e2m1_encode(w):
    """e2m1 code of each w (float32): |w| to the nearest of 0, 0.5, 1, 1.5,
    2, 3, 4, 6 (ties to the even code), saturating at 6; the sign bit for
    negative non-zero results; a zero result is +0 (code 0)."""
    w = np.asarray(w, dtype=np.float64)
    mag = _round_to_grid(np.abs(w), _E2M1_MAG).astype(np.uint8)
    neg = (w < 0) & (mag > 0)
    return (mag | (neg.astype(np.uint8) << 3)).astype(np.uint8)


def quantize_nvfp4(x_bits, qscale):
    """NVFP4 encoding of bf16 activations (bits uint16 [R, L], L % 16 == 0)
    with one float32 pre-scale per row (qscale [R]), for GEMM2's A after the
    MoE block's SwiGLU step (page "LLM-Assisted Kernel Development in CuTe
    DSL, Gluon, Helion and Triton", mixture-of-experts section: GEMM1,
    SwiGLU, GEMM2 per expert).  The pages give no quantisation recipe;
    reading (the NVFP4 format used everywhere here, scale chosen so that the
    block's largest magnitude meets the largest code), per 16-element block,
    every step in float32 with IEEE round-to-nearest-even:
      z_i   = x_i * q                  (x widened to float32 exactly)
      amax  = max_i |z_i|
      sf    = e4m3(amax / 6)           (e4m3_encode: nearest, saturating)
      d     = the value of sf
      code_i = e2m1(z_i / d) if d > 0 else 0   (e2m1_encode)
    So x_i ~ code_i * d / q; GEMM2's alpha carries the 1/q.  Returns (codes
    uint8 [R, L/2], low nibble = even element; sf uint8 [R, L/16])."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    R, L = x_bits.shape
    assert L % 16 == 0
    x = (x_bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    q = np.asarray(qscale, dtype=np.float32).reshape(R, 1)
    z = (x * q).astype(np.float32)                       # float32 products
    assert np.all(np.isfinite(z)), "finite activations only"
    zb = z.reshape(R, L // 16, 16)
    amax = np.abs(zb).max(axis=-1)
    s = (amax / np.float32(6.0)).astype(np.float32)      # float32 quotient
    sf = e4m3_encode(s)
    d = E4M3_TABLE[sf].astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        w = (zb / d[..., None]).astype(np.float32)
    w = np.where(d[..., None] > 0, w, np.float32(0.0))
    codes = e2m1_encode(w).reshape(R, L)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, sf.reshape(R, L // 16)


def gemv_w4a16(x_bits, B, B_sf, alpha, K):
    """The W4A16 decode GEMV ("nvfp4_gemv", W4A16, in the kernel table of the
    page listing Helion's pretuned_kernels directory): y[m, n] = alpha *
    sum_k x[m, k] * B[n, k], x bf16 (bits uint16 [M, K]), B NVFP4 in the raw
    layout (codes [N, K/2], scales [N, K/16]) decoded by decode_numpy; fp64,
    one bf16 rounding.  Returns (y bits uint16 [M, N], y64)."""
    xd = (np.asarray(x_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Bd = decode_numpy(B, B_sf, K)
    y64 = float(alpha) * (xd @ Bd.T)
    return bf16_bits_any(y64), y64


def tolerance_ok(gpu_vals, ref64, max_abs):
    """The acceptance test: |gpu - ref| <= 4e-3*|ref| + 1e-4*max_abs, with ref
    the unrounded fp64 value and max_abs the largest |ref| of the call."""
    gpu_vals = np.asarray(gpu_vals, dtype=np.float64)
    ref64 = np.asarray(ref64, dtype=np.float64)
    err = np.abs(gpu_vals - ref64)
    bound = 4e-3 * np.abs(ref64) + 1e-4 * max_abs
    return err <= bound
