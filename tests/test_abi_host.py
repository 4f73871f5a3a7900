"""Host-side checks of the C-ABI library: it builds for sm_103a, loads, exports
every entry point include/nvfp4gg.h declares, and rejects bad arguments with
the documented status before touching the GPU (no GPU needed)."""
import os
import re

import pytest

from nvfp4_block_scaled_masked_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "nvfp4gg.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"{n} declared in nvfp4gg.h but not exported"
    assert sorted(binding.EXPORTS) == names


def test_status_strings(lib):
    for s in range(0, -9, -1):
        assert binding.status_string(s).startswith("NVFP4GG_")
    assert "unknown" in binding.status_string(42)


def test_prepared_weight_bytes(lib):
    b, s = binding.nvfp4_prepared_weight_bytes(32, 4096, 7168)
    assert b == 32 * 4096 * 3584
    assert s == 32 * 32 * (7168 // 64) * 512 == 32 * 4096 * 7168 // 16
    b, s = binding.nvfp4_prepared_weight_bytes(2, 144, 512)   # N tail padded to 256 rows
    assert b == 2 * 256 * 256
    assert s == 2 * 2 * 8 * 512
    for bad in [(0, 128, 256), (1025, 128, 256), (1, 120, 256), (1, 128, 320), (1, 128, 0)]:
        with pytest.raises(binding.NVFP4GGError) as e:
            binding.nvfp4_prepared_weight_bytes(*bad)
        assert e.value.status == binding.ERR_SHAPE


FAKE = 0x10000   # aligned, never dereferenced: every call below fails its checks first


def gemm(lib, A=FAKE, A_sf=FAKE, B=FAKE, B_sf=FAKE, alpha=FAKE, mask=FAKE, C=FAKE,
         G=4, M=16, N=256, K=256):
    return lib.nvfp4_grouped_gemm_nt_masked(A, A_sf, B, B_sf, alpha, mask, C, G, M, N, K, None)


@pytest.mark.parametrize("field", ["A", "A_sf", "B", "B_sf", "alpha", "mask", "C"])
def test_null_pointers_rejected(lib, field):
    assert gemm(lib, **{field: None}) == binding.ERR_NULL


@pytest.mark.parametrize("shape", [
    dict(G=0), dict(G=1025), dict(M=0), dict(N=0), dict(N=8), dict(N=136),
    dict(K=0), dict(K=128), dict(K=320), dict(G=-3),
])
def test_bad_shapes_rejected(lib, shape):
    assert gemm(lib, **shape) == binding.ERR_SHAPE


@pytest.mark.parametrize("field,addr", [("A", FAKE + 8), ("A_sf", FAKE + 4), ("B", FAKE + 1),
                                        ("B_sf", FAKE + 2), ("C", FAKE + 2),
                                        ("alpha", FAKE + 2), ("mask", FAKE + 1)])
def test_misaligned_pointers_rejected(lib, field, addr):
    assert gemm(lib, **{field: addr}) == binding.ERR_ALIGN


def test_prepare_weights_argument_checks(lib):
    f = lib.nvfp4_prepare_weights
    assert f(None, FAKE, 1, 128, 256, FAKE, FAKE + 4096, None) == binding.ERR_NULL
    assert f(FAKE, FAKE, 1, 100, 256, FAKE, FAKE + 4096, None) == binding.ERR_SHAPE
    assert f(FAKE + 1, FAKE, 1, 128, 256, FAKE, FAKE + 4096, None) == binding.ERR_ALIGN
    assert f(FAKE, FAKE + 64, 1, 128, 256, FAKE + 128, FAKE + 64, None) == binding.ERR_SHAPE
    assert f(FAKE, FAKE + 64, 1, 128, 256, FAKE, FAKE + 128, None) == binding.ERR_SHAPE


def test_host_variant_argument_checks(lib):
    need = binding.nvfp4_host_staging_bytes(4, 16, 256, 256)
    up = lambda x: (x + 255) // 256 * 256
    assert need == up(4 * 16 * 256 * 2) + up(4 * 16 * 128) + up(4 * 16 * 16) + 2 * up(16)
    assert binding.nvfp4_host_staging_bytes(0, 16, 256, 256) == 0
    f = lib.nvfp4_grouped_gemm_nt_masked_host
    args = [FAKE] * 7 + [4, 16, 256, 256, FAKE, need, None]
    a = list(args); a[0] = None
    assert f(*a) == binding.ERR_NULL
    a = list(args); a[12] = need - 1
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[11] = FAKE + 8
    assert f(*a) == binding.ERR_ALIGN


def test_splitk_argument_checks(lib):
    f = lib.nvfp4_grouped_gemm_nt_masked_splitk
    need = binding.nvfp4_splitk_workspace_bytes(4, 16, 256, 512, 2)
    tiles = 4 * 1 * 2
    assert need == (tiles * 2 * 32 * 128 * 4 + 255) // 256 * 256 + tiles * 8
    assert binding.nvfp4_splitk_workspace_bytes(4, 16, 256, 512, 17) == 0
    args = [FAKE] * 7 + [4, 16, 256, 512, 2, FAKE, need, None]
    a = list(args); a[12] = None
    assert f(*a) == binding.ERR_NULL
    a = list(args); a[11] = 17
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[12] = FAKE + 16
    assert f(*a) == binding.ERR_ALIGN
    a = list(args); a[13] = need - 1
    assert f(*a) == binding.ERR_SHAPE


def test_noalloc_splitk_argument_checks(lib):
    """The static-scratch split-K call: bad arguments and splits that do not
    fit its NVFP4GG_NOALLOC_MAX_SLOTS scratch slots are refused before any
    CUDA call."""
    f = lib.nvfp4_grouped_gemm_nt_masked_splitk_noalloc
    slots = 256
    # G=8, M_max=16, N=4096: 8 * 1 * 32 = 256 tiles
    args = [FAKE] * 7 + [8, 16, 4096, 7168, 2, None]
    a = list(args); a[0] = None
    assert f(*a) == binding.ERR_NULL
    a = list(args); a[11] = 17
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[11] = -1
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[10] = 7000          # K % 256 != 0
    assert f(*a) == binding.ERR_SHAPE
    assert 256 * 2 > slots
    assert f(*args) == binding.ERR_SCRATCH
    a = list(args); a[7] = 4; a[11] = 3     # 128 tiles x 3 > 256
    assert f(*a) == binding.ERR_SCRATCH
    a = list(args); a[7] = 1; a[9] = 16384; a[11] = 16   # 128 tiles x 16
    assert f(*a) == binding.ERR_SCRATCH
    assert "NOALLOC_MAX_SLOTS" in binding.status_string(binding.ERR_SCRATCH)


def test_sm_cap_and_watchdog_argument_checks(lib):
    assert lib.nvfp4_gg_set_sm_count(-1) == binding.ERR_SHAPE
    assert lib.nvfp4_gg_set_sm_count(0) == binding.OK
    assert lib.nvfp4_gg_set_pair_mode(4) == binding.ERR_SHAPE
    assert lib.nvfp4_gg_set_pair_mode(-1) == binding.ERR_SHAPE
    assert lib.nvfp4_gg_set_pair_mode(3) == binding.OK   # token-major pairs
    assert lib.nvfp4_gg_set_pair_mode(1) == binding.OK
    assert lib.nvfp4_gg_set_pair_mode(0) == binding.OK
    assert lib.nvfp4_gg_set_pair_mode(2) == binding.OK   # the default: automatic
    assert lib.nvfp4_gg_selftest_watchdog(10, None) == binding.ERR_SHAPE
    assert lib.nvfp4_gg_selftest_watchdog(10 ** 11, None) == binding.ERR_SHAPE


def test_shutdown_is_host_only_and_repeatable(lib):
    """nvfp4_gg_shutdown touches no device: it works here, with no GPU, and
    twice in a row; the settings (SM cap, pair mode) are not caches and stay."""
    assert lib.nvfp4_gg_shutdown() == binding.OK
    assert lib.nvfp4_gg_shutdown() == binding.OK


def test_library_targets_sm103a_only():
    assert build.ARCH_FLAGS == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_swiglu_argument_checks(lib):
    f = lib.nvfp4_grouped_gemm_nt_masked_swiglu
    args = [FAKE] * 7 + [2, 16, 256, 512, None]
    a = list(args); a[9] = 192                    # N % 128 != 0
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[0] = None
    assert f(*a) == binding.ERR_NULL
    p = lib.nvfp4_prepare_weights_swiglu
    assert p(FAKE, FAKE, 2, 192, 512, FAKE + 4096, FAKE + 8192, None) == binding.ERR_SHAPE
    assert p(None, FAKE, 2, 256, 512, FAKE + 4096, FAKE + 8192, None) == binding.ERR_NULL


def test_swiglu_quant_argument_checks(lib):
    f = lib.nvfp4_grouped_gemm_nt_masked_swiglu_quant
    # A, A_sf, B, B_sf, alpha, masked_m, C, qscale, A2, A2_sf, G, M_max, N, K, stream
    args = [FAKE] * 10 + [2, 16, 256, 512, None]
    for k in (7, 8, 9):                           # qscale, A2, A2_sf required
        a = list(args); a[k] = None
        assert f(*a) == binding.ERR_NULL
    a = list(args); a[0] = None
    assert f(*a) == binding.ERR_NULL
    a = list(args); a[12] = 192                   # N % 128 != 0
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[8] = FAKE + 8               # A2 not 16-byte aligned
    assert f(*a) == binding.ERR_ALIGN
    a = list(args); a[7] = FAKE + 2               # qscale not 4-byte aligned
    assert f(*a) == binding.ERR_ALIGN


def test_quantize_argument_checks(lib):
    f = lib.nvfp4_quantize_bf16
    args = [FAKE] * 4 + [4, 256, 4, None]
    for k in range(4):
        a = list(args); a[k] = None
        assert f(*a) == binding.ERR_NULL
    for k, v in ((4, 0), (5, 8), (5, 264), (6, 0)):   # R < 1, L < 16, L % 16, rows_per_scale < 1
        a = list(args); a[k] = v
        assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[0] = FAKE + 8               # x not 16-byte aligned
    assert f(*a) == binding.ERR_ALIGN
    a = list(args); a[2] = FAKE + 4               # codes not 8-byte aligned
    assert f(*a) == binding.ERR_ALIGN


def test_signals_argument_checks(lib):
    f = lib.nvfp4_grouped_gemm_nt_masked_signals
    args = [FAKE] * 7 + [2, 16, 256, 512, FAKE, None]
    a = list(args); a[11] = None
    assert f(*a) == binding.ERR_NULL
    a = list(args); a[11] = FAKE + 2
    assert f(*a) == binding.ERR_ALIGN
    a = list(args); a[10] = 100
    assert f(*a) == binding.ERR_SHAPE


def test_contiguous_argument_checks(lib):
    f = lib.nvfp4_grouped_gemm_nt_contiguous
    args = [FAKE] * 7 + [4, 32, 64, 256, 512, None]
    a = list(args); a[9] = 0                      # M_total < 1
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[8] = 65                     # M_max > M_total
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[10] = 100                   # N % 16 != 0
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[6] = None
    assert f(*a) == binding.ERR_NULL


def test_gemv_argument_checks(lib):
    f = lib.nvfp4_gemv_w4a16
    args = [FAKE] * 5 + [1, 4096, 4096, None]
    a = list(args); a[5] = 0
    assert f(*a) == binding.ERR_SHAPE            # M < 1
    a = list(args); a[5] = 9
    assert f(*a) == binding.ERR_SHAPE            # M > 8
    a = list(args); a[7] = 4008
    assert f(*a) == binding.ERR_SHAPE            # K % 32 != 0
    a = list(args); a[5] = 8; a[7] = 8960
    assert f(*a) == binding.ERR_SHAPE            # tokens do not fit shared memory
    a = list(args); a[5] = 1; a[7] = 71520
    assert f(*a) == binding.ERR_SHAPE            # M * K = 71520 > 71493
    a = list(args); a[1] = FAKE + 8
    assert f(*a) == binding.ERR_ALIGN
    a = list(args); a[4] = None
    assert f(*a) == binding.ERR_NULL


def test_prepare_weights_dual_argument_checks(lib):
    f = lib.nvfp4_prepare_weights_dual
    # B1, B1_sf, B2, B2_sf, G, N1, K, interleave, B_prep, B_sf_prep, stream
    big = 1 << 24
    args = [FAKE, FAKE + big, FAKE + 2 * big, FAKE + 3 * big, 2, 128, 512, 1,
            FAKE + 4 * big, FAKE + 5 * big, None]
    for k in (0, 1, 2, 3, 8, 9):
        a = list(args); a[k] = None
        assert f(*a) == binding.ERR_NULL
    a = list(args); a[5] = 72                     # N1 % 16 != 0
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[5] = 96                     # interleaved needs 2 N1 % 128 == 0
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[7] = 2                      # interleave is 0 or 1
    assert f(*a) == binding.ERR_SHAPE
    a = list(args); a[2] = FAKE + 2 * big + 8     # misaligned B2
    assert f(*a) == binding.ERR_ALIGN
    a = list(args); a[8] = FAKE + 2 * big + 4096  # output overlaps B2
    assert f(*a) == binding.ERR_SHAPE
