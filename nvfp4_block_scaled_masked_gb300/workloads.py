"""Seeded synthetic workloads for the masked NVFP4 grouped GEMM-NT.

This module only draws inputs: it holds none of the GEMM's arithmetic (no
decoding, no products, no rounding), so both the CUDA path's tests and the CPU
oracle can take their inputs from it.

The shapes come from the DeepSeek-V3 MoE dimensions that the page
"LLM-Assisted Kernel Development in CuTe DSL, Gluon, Helion and Triton"
lists for its MoE reference (section "MoE": H=7168, I=2048, 256 experts):
GEMM1 (gate+up) has N=4096, K=7168; GEMM2 has N=7168, K=2048.  The pages'
real workloads (a serving trace, model weights) are not available, so these
seeded inputs stand in for them.

Recipe (all configs):
  * masked_m: fixed list, uniform integers, or the per-expert counts of top-8
    routing where each token picks 8 distinct experts uniformly at random;
  * alpha_g: uniform in [0.5, 2) as fp32 (1.0 for the compute-bound config);
  * A, B codes: e2m1 codes uniform over the 15 codes other than negative zero
    (0x8), two per byte;
  * A_sf, B_sf: e4m3 bytes uniform over {0x18,0x20,...,0x48} = 2^-4 .. 2^2;
  * C is prefilled with the bf16 NaN 0x7FC0 so untouched rows are visible;
  * rows >= masked_m of A are drawn like the others (or poisoned: NaN scales).
Draw order: masked_m, alpha, A codes, A_sf, B codes, B_sf.
"""
from __future__ import annotations

import dataclasses

import numpy as np

SENTINEL_BF16 = 0x7FC0
SCALE_BYTES = np.array([0x18, 0x20, 0x28, 0x30, 0x38, 0x40, 0x48], dtype=np.uint8)
# the 15 e2m1 codes other than 0x8 (negative zero)
CODES = np.array([c for c in range(16) if c != 8], dtype=np.uint8)
# packed byte for a uniform index i in [0, 225): low nibble (the even element)
# CODES[i % 15], high nibble CODES[i // 15]
_PAIR_LUT = (CODES[np.arange(225) % 15] | (CODES[np.arange(225) // 15] << 4)).astype(np.uint8)


@dataclasses.dataclass(frozen=True)
class Config:
    key: str
    name: str
    G: int
    M_max: int
    N: int
    K: int
    masked: str                   # "fixed" | "uniform" | "topk" | "full"
    masked_list: tuple = ()
    masked_hi: int = 0            # for "uniform": masked_m ~ U{0..masked_hi}
    tokens: int = 0               # for "topk"
    topk: int = 0
    alpha_one: bool = False
    kind: str = "gemm"            # "gemm" | "gemv_w4a16" (M_max tokens of bf16 activations)

    @property
    def seed(self) -> int:
        return 0x4E5646340000 + int(self.key[1:])


CONFIGS = {
    "c1": Config("c1", "small-masked G=4 M_max=128 N=256 K=256", 4, 128, 256, 256,
                 "fixed", masked_list=(0, 17, 64, 128)),
    "c2": Config("c2", "decode GEMM1 G=32 M_max=16 N=4096 K=7168", 32, 16, 4096, 7168,
                 "uniform", masked_hi=8),
    "c3": Config("c3", "decode GEMM1 MoE G=256 64 tokens top-8 M_max=64 N=4096 K=7168",
                 256, 64, 4096, 7168, "topk", tokens=64, topk=8),
    "c4": Config("c4", "prefill GEMM2 G=256 4096 tokens top-8 M_max=256 N=7168 K=2048",
                 256, 256, 7168, 2048, "topk", tokens=4096, topk=8),
    "c5": Config("c5", "compute-bound G=8 M=2048 N=7168 K=4096", 8, 2048, 7168, 4096,
                 "full", alpha_one=True),
}


# Extra workloads beyond the five above (not benchmark headlines): a decode
# call whose experts are all empty (the fixed cost of a call), and one with a
# single non-empty expert, where the unsplit kernel has only 32 weight tiles
# for the GPU's SMs (the case split-K is for).
EXTRA = {
    "x0": Config("x0", "decode GEMM1 all experts empty G=32 N=4096 K=7168", 32, 16, 4096, 7168,
                 "fixed", masked_list=(0,) * 32),
    "x1": Config("x1", "decode GEMM1 one expert G=1 masked_m=7 N=4096 K=7168", 1, 16, 4096, 7168,
                 "fixed", masked_list=(7,)),
    # W4A16 decode GEMV, one token, Llama-3-8B MLP projection shapes (the
    # pages' nvfp4_gemv workload names Llama-3 / Qwen projections)
    "v1": Config("v1", "decode GEMV W4A16 M=1 N=14336 K=4096", 1, 1, 14336, 4096,
                 "fixed", masked_list=(1,), kind="gemv_w4a16"),
    "v2": Config("v2", "decode GEMV W4A16 M=1 N=4096 K=14336", 1, 1, 4096, 14336,
                 "fixed", masked_list=(1,), kind="gemv_w4a16"),
}


def generate_gemv(cfg: Config, seed: int | None = None) -> dict:
    """Inputs of the W4A16 GEMV: x bf16 bits u16[M, K] (M = cfg.M_max) built
    directly as bf16 patterns (random sign, exponent 2^-3 .. 2^1, 7-bit
    mantissa: no rounding), B u8[N, K/2] and B_sf u8[N, K/16] in the raw layout
    drawn like the GEMM's weights, alpha f32 uniform in [0.5, 2)."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    M, N, K = cfg.M_max, cfg.N, cfg.K
    sign = rng.integers(0, 2, (M, K)).astype(np.uint16)
    exp = rng.integers(127 - 3, 127 + 2, (M, K)).astype(np.uint16)
    man = rng.integers(0, 128, (M, K)).astype(np.uint16)
    x = (sign << 15) | (exp << 7) | man
    alpha = np.float32(rng.uniform(0.5, 2.0))
    B = draw_codes(rng, (N, K // 2))
    B_sf = draw_scales(rng, (N, K // 16))
    return dict(cfg=cfg, x=x.astype(np.uint16), B=B, B_sf=B_sf, alpha=np.array([alpha], np.float32))


def lookup(key: str) -> Config:
    return CONFIGS[key] if key in CONFIGS else EXTRA[key]


def custom(G, M_max, N, K, masked_m=None, key="c0", alpha_one=False) -> Config:
    """An ad-hoc config (tests): masked_m fixed if given, else uniform 0..M_max."""
    if masked_m is not None:
        return Config(key, f"custom G={G} M_max={M_max} N={N} K={K}", G, M_max, N, K,
                      "fixed", masked_list=tuple(int(x) for x in masked_m),
                      alpha_one=alpha_one)
    return Config(key, f"custom G={G} M_max={M_max} N={N} K={K}", G, M_max, N, K,
                  "uniform", masked_hi=M_max, alpha_one=alpha_one)


def draw_masked_m(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    if cfg.masked == "fixed":
        mm = np.array(cfg.masked_list, dtype=np.int32)
        assert mm.shape == (cfg.G,)
    elif cfg.masked == "uniform":
        mm = rng.integers(0, cfg.masked_hi + 1, size=cfg.G).astype(np.int32)
    elif cfg.masked == "topk":
        # each token picks topk distinct experts uniformly: the first topk of a
        # uniformly random permutation (argsort of iid uniforms)
        picks = np.argsort(rng.random((cfg.tokens, cfg.G)), axis=1)[:, :cfg.topk]
        mm = np.bincount(picks.ravel(), minlength=cfg.G).astype(np.int32)
    elif cfg.masked == "full":
        mm = np.full(cfg.G, cfg.M_max, dtype=np.int32)
    else:
        raise ValueError(cfg.masked)
    if mm.max(initial=0) > cfg.M_max or mm.min(initial=0) < 0:
        raise AssertionError("generated masked_m outside [0, M_max]")
    return mm


_CHUNK = 1 << 24


def _uniform_index(rng: np.random.Generator, n: int, k: int) -> np.ndarray:
    """n iid integers uniform on [0, k) as uint8 (k <= 256): raw 32-bit words
    reduced mod k, drawn in chunks (the bias of the reduction is below
    k / 2^32 < 1e-7)."""
    out = np.empty(n, dtype=np.uint8)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        w = rng.integers(0, 1 << 32, size=e - s, dtype=np.uint32)
        np.remainder(w, np.uint32(k), out=w)
        out[s:e] = w
    return out


def draw_codes(rng: np.random.Generator, shape_bytes) -> np.ndarray:
    """Packed e2m1 bytes, both nibbles uniform over the 15 allowed codes."""
    n = int(np.prod(shape_bytes))
    return _PAIR_LUT[_uniform_index(rng, n, 225)].reshape(shape_bytes)


def draw_scales(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return SCALE_BYTES[_uniform_index(rng, n, len(SCALE_BYTES))].reshape(shape)


# Scale-byte sets for the full-range inputs: every finite non-negative e4m3
# byte (0x00 zero, 0x01..0x07 subnormal, up to 0x7E = 448; 0x7F is NaN), the
# subnormals with zero, and the top binades.
SCALE_SETS = {
    "all": np.arange(0x00, 0x7F, dtype=np.uint8),
    "subnormal": np.arange(0x00, 0x08, dtype=np.uint8),
    "large": np.arange(0x70, 0x7F, dtype=np.uint8),
    "powers": SCALE_BYTES,
}


def generate_full_range(cfg: Config, seed: int, a_scales: str = "all",
                        b_scales: str = "all") -> dict:
    """Inputs over the whole NVFP4 domain, in the layouts of generate(): both
    nibbles of every code byte uniform over all 16 e2m1 codes (negative zero
    0x8 included), scale bytes uniform over SCALE_SETS[a_scales] for A_sf and
    SCALE_SETS[b_scales] for B_sf, alpha uniform in [0.5, 2).  masked_m as the
    config says; C prefilled with 0x7FC0."""
    G, M, N, K = cfg.G, cfg.M_max, cfg.N, cfg.K
    rng = np.random.default_rng(seed)
    masked_m = draw_masked_m(cfg, rng)
    alpha = rng.uniform(0.5, 2.0, size=G).astype(np.float32)
    sa, sb = SCALE_SETS[a_scales], SCALE_SETS[b_scales]
    A = rng.integers(0, 256, size=(G, M, K // 2), dtype=np.uint8)
    A_sf = sa[_uniform_index(rng, G * M * (K // 16), len(sa))].reshape(G, M, K // 16)
    B = rng.integers(0, 256, size=(G, N, K // 2), dtype=np.uint8)
    B_sf = sb[_uniform_index(rng, G * N * (K // 16), len(sb))].reshape(G, N, K // 16)
    return dict(cfg=cfg, masked_m=masked_m, alpha=alpha, A=A, A_sf=A_sf, B=B, B_sf=B_sf,
                C_init=np.full((G, M, N), SENTINEL_BF16, dtype=np.uint16))


def generate(cfg: Config, seed: int | None = None, poison: bool = False,
             with_b: bool = True) -> dict:
    """All inputs of one call, as NumPy arrays in the plain layouts:
    A u8[G,M_max,K/2], A_sf u8[G,M_max,K/16], B u8[G,N,K/2], B_sf u8[G,N,K/16],
    alpha f32[G], masked_m i32[G], C_init u16[G,M_max,N] (all 0x7FC0).
    poison=True puts the NaN scale byte 0x7F in every row >= masked_m of A_sf."""
    G, M, N, K = cfg.G, cfg.M_max, cfg.N, cfg.K
    assert K % 16 == 0
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    masked_m = draw_masked_m(cfg, rng)
    if cfg.alpha_one:
        alpha = np.ones(G, dtype=np.float32)
    else:
        alpha = rng.uniform(0.5, 2.0, size=G).astype(np.float32)
    A = draw_codes(rng, (G, M, K // 2))
    A_sf = draw_scales(rng, (G, M, K // 16))
    if poison:
        for g in range(G):
            A_sf[g, masked_m[g]:] = 0x7F
    out = dict(cfg=cfg, masked_m=masked_m, alpha=alpha, A=A, A_sf=A_sf)
    if with_b:
        out["B"] = draw_codes(rng, (G, N, K // 2))
        out["B_sf"] = draw_scales(rng, (G, N, K // 16))
    out["C_init"] = np.full((G, M, N), SENTINEL_BF16, dtype=np.uint16)
    return out


def algorithmic_counts(cfg: Config, masked_m) -> dict:
    """FLOPs and the bytes the method must move: weights + scales of non-empty
    experts, activations + scales of valid rows, bf16 output of valid rows."""
    mm = np.asarray(masked_m, dtype=np.int64)
    rows = int(mm.sum())
    nonempty = int((mm > 0).sum())
    N, K = cfg.N, cfg.K
    w_bytes = nonempty * N * (K // 2 + K // 16)
    a_bytes = rows * (K // 2 + K // 16)
    c_bytes = rows * N * 2
    return dict(flops=2 * rows * N * K, rows=rows, nonempty=nonempty,
                weight_bytes=w_bytes, act_bytes=a_bytes, out_bytes=c_bytes,
                bytes=w_bytes + a_bytes + c_bytes)
