"""Python binding of libnvfp4gg (include/nvfp4gg.h): argument marshalling only.

Every function takes device buffers as torch tensors (their data_ptr is
passed) or as raw integer addresses, and a CUDA stream (a torch.cuda.Stream,
a raw cudaStream_t integer, or None for torch's current stream).  All work
runs in the library's CUDA kernels; if the library is not built this module
raises instead of computing anything another way.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

_lib = None

OK = 0
ERR_NULL = -1
ERR_SHAPE = -2
ERR_ALIGN = -3
ERR_ARCH = -4
ERR_CUDA = -5
ERR_TIMEOUT = -6
ERR_MASK = -7
ERR_SCRATCH = -8

# every symbol the header declares
EXPORTS = (
    "nvfp4_prepared_weight_bytes",
    "nvfp4_prepare_weights",
    "nvfp4_grouped_gemm_nt_masked",
    "nvfp4_splitk_workspace_bytes",
    "nvfp4_grouped_gemm_nt_masked_splitk",
    "nvfp4_grouped_gemm_nt_masked_splitk_noalloc",
    "nvfp4_grouped_gemm_nt_contiguous",
    "nvfp4_gemv_w4a16",
    "nvfp4_grouped_gemm_nt_masked_signals",
    "nvfp4_prepare_weights_swiglu",
    "nvfp4_prepare_weights_dual",
    "nvfp4_grouped_gemm_nt_masked_swiglu",
    "nvfp4_grouped_gemm_nt_masked_swiglu_quant",
    "nvfp4_quantize_bf16",
    "nvfp4_host_staging_bytes",
    "nvfp4_grouped_gemm_nt_masked_host",
    "nvfp4_gg_set_sm_count",
    "nvfp4_gg_set_pair_mode",
    "nvfp4_gg_shutdown",
    "nvfp4_gg_check_error",
    "nvfp4_gg_selftest_watchdog",
    "nvfp4_gg_mma_peak_probe",
    "nvfp4_gg_mma_peak_probe_pair",
    "nvfp4_gg_status_string",
)


class NVFP4GGError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Open libnvfp4gg.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.nvfp4_prepared_weight_bytes.argtypes = [i, i, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.nvfp4_prepared_weight_bytes.restype = i
    lib.nvfp4_prepare_weights.argtypes = [vp, vp, i, i, i, vp, vp, vp]
    lib.nvfp4_prepare_weights.restype = i
    lib.nvfp4_grouped_gemm_nt_masked.argtypes = [vp] * 7 + [i] * 4 + [vp]
    lib.nvfp4_grouped_gemm_nt_masked.restype = i
    lib.nvfp4_splitk_workspace_bytes.argtypes = [i] * 5
    lib.nvfp4_splitk_workspace_bytes.restype = sz
    lib.nvfp4_grouped_gemm_nt_masked_splitk.argtypes = [vp] * 7 + [i] * 5 + [vp, sz, vp]
    lib.nvfp4_grouped_gemm_nt_masked_splitk.restype = i
    lib.nvfp4_grouped_gemm_nt_masked_splitk_noalloc.argtypes = [vp] * 7 + [i] * 5 + [vp]
    lib.nvfp4_grouped_gemm_nt_masked_splitk_noalloc.restype = i
    lib.nvfp4_gemv_w4a16.argtypes = [vp] * 5 + [i] * 3 + [vp]
    lib.nvfp4_gemv_w4a16.restype = i
    lib.nvfp4_grouped_gemm_nt_contiguous.argtypes = [vp] * 7 + [i] * 5 + [vp]
    lib.nvfp4_grouped_gemm_nt_contiguous.restype = i
    lib.nvfp4_grouped_gemm_nt_masked_signals.argtypes = [vp] * 7 + [i] * 4 + [vp, vp]
    lib.nvfp4_grouped_gemm_nt_masked_signals.restype = i
    lib.nvfp4_prepare_weights_swiglu.argtypes = [vp, vp, i, i, i, vp, vp, vp]
    lib.nvfp4_prepare_weights_swiglu.restype = i
    lib.nvfp4_prepare_weights_dual.argtypes = [vp] * 4 + [i] * 4 + [vp, vp, vp]
    lib.nvfp4_prepare_weights_dual.restype = i
    lib.nvfp4_grouped_gemm_nt_masked_swiglu.argtypes = [vp] * 7 + [i] * 4 + [vp]
    lib.nvfp4_grouped_gemm_nt_masked_swiglu.restype = i
    lib.nvfp4_grouped_gemm_nt_masked_swiglu_quant.argtypes = [vp] * 10 + [i] * 4 + [vp]
    lib.nvfp4_grouped_gemm_nt_masked_swiglu_quant.restype = i
    lib.nvfp4_quantize_bf16.argtypes = [vp] * 4 + [i] * 3 + [vp]
    lib.nvfp4_quantize_bf16.restype = i
    lib.nvfp4_host_staging_bytes.argtypes = [i] * 4
    lib.nvfp4_host_staging_bytes.restype = sz
    lib.nvfp4_grouped_gemm_nt_masked_host.argtypes = [vp] * 7 + [i] * 4 + [vp, sz, vp]
    lib.nvfp4_grouped_gemm_nt_masked_host.restype = i
    lib.nvfp4_gg_set_sm_count.argtypes = [i]
    lib.nvfp4_gg_set_sm_count.restype = i
    lib.nvfp4_gg_set_pair_mode.argtypes = [i]
    lib.nvfp4_gg_set_pair_mode.restype = i
    lib.nvfp4_gg_shutdown.argtypes = []
    lib.nvfp4_gg_shutdown.restype = i
    lib.nvfp4_gg_check_error.argtypes = [vp]
    lib.nvfp4_gg_check_error.restype = i
    lib.nvfp4_gg_selftest_watchdog.argtypes = [ctypes.c_longlong, vp]
    lib.nvfp4_gg_selftest_watchdog.restype = i
    lib.nvfp4_gg_mma_peak_probe.argtypes = [i, i, i, vp]
    lib.nvfp4_gg_mma_peak_probe.restype = i
    lib.nvfp4_gg_mma_peak_probe_pair.argtypes = [i, i, i, vp]
    lib.nvfp4_gg_mma_peak_probe_pair.restype = i
    lib.nvfp4_gg_status_string.argtypes = [i]
    lib.nvfp4_gg_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):          # numpy array (host buffers)
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


_raw_stream = None


def _stream(s):
    if s is None:
        global _raw_stream
        if _raw_stream is None:
            import torch
            raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
            if raw is not None:
                _raw_stream = lambda: raw(torch.cuda.current_device())
            else:
                _raw_stream = lambda: torch.cuda.current_stream().cuda_stream
        return _raw_stream()
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, what: str):
    if rc != OK:
        raise NVFP4GGError(rc, what)


def status_string(status: int) -> str:
    return load().nvfp4_gg_status_string(int(status)).decode()


def nvfp4_prepared_weight_bytes(G: int, N: int, K: int):
    b, s = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().nvfp4_prepared_weight_bytes(G, N, K, ctypes.byref(b), ctypes.byref(s)),
           "nvfp4_prepared_weight_bytes")
    return b.value, s.value


def nvfp4_prepare_weights(B, B_sf, G, N, K, B_prep, B_sf_prep, stream=None):
    _check(load().nvfp4_prepare_weights(_ptr(B), _ptr(B_sf), G, N, K, _ptr(B_prep),
                                        _ptr(B_sf_prep), _stream(stream)),
           "nvfp4_prepare_weights")


def nvfp4_grouped_gemm_nt_masked(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K,
                                 stream=None):
    _check(load().nvfp4_grouped_gemm_nt_masked(_ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf),
                                               _ptr(alpha), _ptr(masked_m), _ptr(C),
                                               G, M_max, N, K, _stream(stream)),
           "nvfp4_grouped_gemm_nt_masked")


def nvfp4_gemv_w4a16(x, B, B_sf, alpha, y, M, N, K, stream=None):
    _check(load().nvfp4_gemv_w4a16(_ptr(x), _ptr(B), _ptr(B_sf), _ptr(alpha), _ptr(y), M, N, K,
                                   _stream(stream)),
           "nvfp4_gemv_w4a16")


def nvfp4_grouped_gemm_nt_contiguous(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, M_total,
                                     N, K, stream=None):
    _check(load().nvfp4_grouped_gemm_nt_contiguous(
        _ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf), _ptr(alpha), _ptr(masked_m), _ptr(C),
        G, M_max, M_total, N, K, _stream(stream)),
        "nvfp4_grouped_gemm_nt_contiguous")


def nvfp4_grouped_gemm_nt_masked_signals(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K,
                                         dst_signals, stream=None):
    _check(load().nvfp4_grouped_gemm_nt_masked_signals(
        _ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf), _ptr(alpha), _ptr(masked_m), _ptr(C),
        G, M_max, N, K, _ptr(dst_signals), _stream(stream)),
        "nvfp4_grouped_gemm_nt_masked_signals")


def nvfp4_prepare_weights_swiglu(B, B_sf, G, N, K, B_prep, B_sf_prep, stream=None):
    _check(load().nvfp4_prepare_weights_swiglu(_ptr(B), _ptr(B_sf), G, N, K, _ptr(B_prep),
                                               _ptr(B_sf_prep), _stream(stream)),
           "nvfp4_prepare_weights_swiglu")


def nvfp4_prepare_weights_dual(B1, B1_sf, B2, B2_sf, G, N1, K, interleave, B_prep, B_sf_prep,
                               stream=None):
    _check(load().nvfp4_prepare_weights_dual(
        _ptr(B1), _ptr(B1_sf), _ptr(B2), _ptr(B2_sf), G, N1, K, int(interleave), _ptr(B_prep),
        _ptr(B_sf_prep), _stream(stream)), "nvfp4_prepare_weights_dual")


def nvfp4_grouped_gemm_nt_masked_swiglu(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K,
                                        stream=None):
    _check(load().nvfp4_grouped_gemm_nt_masked_swiglu(_ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf),
                                                      _ptr(alpha), _ptr(masked_m), _ptr(C),
                                                      G, M_max, N, K, _stream(stream)),
           "nvfp4_grouped_gemm_nt_masked_swiglu")


def nvfp4_grouped_gemm_nt_masked_swiglu_quant(A, A_sf, B, B_sf, alpha, masked_m, C, qscale, A2,
                                              A2_sf, G, M_max, N, K, stream=None):
    """SwiGLU GEMM1 whose epilogue also writes GEMM2's NVFP4 A (A2, A2_sf);
    C may be None."""
    _check(load().nvfp4_grouped_gemm_nt_masked_swiglu_quant(
        _ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf), _ptr(alpha), _ptr(masked_m), _ptr(C),
        _ptr(qscale), _ptr(A2), _ptr(A2_sf), G, M_max, N, K, _stream(stream)),
        "nvfp4_grouped_gemm_nt_masked_swiglu_quant")


def nvfp4_quantize_bf16(x, qscale, codes, sf, R, L, rows_per_scale, stream=None):
    """NVFP4 encoding of bf16 rows x [R][L] (qscale[r // rows_per_scale])."""
    _check(load().nvfp4_quantize_bf16(_ptr(x), _ptr(qscale), _ptr(codes), _ptr(sf), R, L,
                                      rows_per_scale, _stream(stream)),
           "nvfp4_quantize_bf16")


def nvfp4_splitk_workspace_bytes(G, M_max, N, K, split_k=0) -> int:
    return int(load().nvfp4_splitk_workspace_bytes(G, M_max, N, K, split_k))


def nvfp4_grouped_gemm_nt_masked_splitk(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max, N, K,
                                        split_k, workspace, workspace_bytes, stream=None):
    _check(load().nvfp4_grouped_gemm_nt_masked_splitk(
        _ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf), _ptr(alpha), _ptr(masked_m), _ptr(C),
        G, M_max, N, K, split_k, _ptr(workspace), workspace_bytes, _stream(stream)),
        "nvfp4_grouped_gemm_nt_masked_splitk")


def nvfp4_grouped_gemm_nt_masked_splitk_noalloc(A, A_sf, B, B_sf, alpha, masked_m, C, G, M_max,
                                                N, K, split_k, stream=None):
    _check(load().nvfp4_grouped_gemm_nt_masked_splitk_noalloc(
        _ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf), _ptr(alpha), _ptr(masked_m), _ptr(C),
        G, M_max, N, K, split_k, _stream(stream)),
        "nvfp4_grouped_gemm_nt_masked_splitk_noalloc")


def nvfp4_host_staging_bytes(G, M_max, N, K) -> int:
    return int(load().nvfp4_host_staging_bytes(G, M_max, N, K))


def nvfp4_grouped_gemm_nt_masked_host(h_A, h_A_sf, h_alpha, h_masked_m, B, B_sf, h_C,
                                      G, M_max, N, K, d_staging, staging_bytes, stream=None):
    _check(load().nvfp4_grouped_gemm_nt_masked_host(
        _ptr(h_A), _ptr(h_A_sf), _ptr(h_alpha), _ptr(h_masked_m), _ptr(B), _ptr(B_sf),
        _ptr(h_C), G, M_max, N, K, _ptr(d_staging), staging_bytes, _stream(stream)),
        "nvfp4_grouped_gemm_nt_masked_host")


def nvfp4_gg_set_sm_count(sm_count: int):
    _check(load().nvfp4_gg_set_sm_count(sm_count), "nvfp4_gg_set_sm_count")


PAIR_OFF, PAIR_ON, PAIR_AUTO, PAIR_TOKEN_MAJOR = 0, 1, 2, 3


def nvfp4_gg_set_pair_mode(mode):
    """0 / False: single-CTA tiles; 1 / True: CTA pairs where N % 256 == 0;
    2: automatic (the library's default)."""
    m = (1 if mode else 0) if isinstance(mode, bool) else int(mode)
    _check(load().nvfp4_gg_set_pair_mode(m), "nvfp4_gg_set_pair_mode")


def nvfp4_gg_shutdown():
    """Drops the library's host-side caches (after a device reset, or when
    done); the next call sets the device up again."""
    _check(load().nvfp4_gg_shutdown(), "nvfp4_gg_shutdown")


def nvfp4_gg_check_error(stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device error word."""
    return int(load().nvfp4_gg_check_error(_stream(stream)))


def nvfp4_gg_mma_peak_probe(iters: int, n: int, ctas: int = 0, stream=None):
    _check(load().nvfp4_gg_mma_peak_probe(iters, n, ctas, _stream(stream)),
           "nvfp4_gg_mma_peak_probe")


def nvfp4_gg_mma_peak_probe_pair(iters: int, n: int, clusters: int = 0, stream=None):
    _check(load().nvfp4_gg_mma_peak_probe_pair(iters, n, clusters, _stream(stream)),
           "nvfp4_gg_mma_peak_probe_pair")


def nvfp4_gg_selftest_watchdog(timeout_ns: int, stream=None):
    _check(load().nvfp4_gg_selftest_watchdog(int(timeout_ns), _stream(stream)),
           "nvfp4_gg_selftest_watchdog")
