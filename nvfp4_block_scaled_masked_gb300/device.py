"""Device-memory plumbing around the C-ABI: copies seeded host inputs into
torch CUDA tensors, prepares the weights once, and calls the GEMM.  Torch only
allocates memory and supplies streams; every step of the GEMM runs in
libnvfp4gg's kernels."""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from .workloads import SENTINEL_BF16


def to_device(arr: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.to(device, non_blocking=False)


class Problem:
    """One call's device buffers: activations, prepared weights, alpha,
    masked_m and a C buffer prefilled with the bf16 sentinel."""

    def __init__(self, d: dict, device="cuda", stream=None, keep_raw_weights=False):
        cfg = d["cfg"]
        self.cfg = cfg
        self.G, self.M_max, self.N, self.K = cfg.G, cfg.M_max, cfg.N, cfg.K
        self.A = to_device(d["A"], device)
        self.A_sf = to_device(d["A_sf"], device)
        self.alpha = to_device(d["alpha"], device)
        self.masked_m = to_device(d["masked_m"].astype(np.int32), device)
        b_bytes, sf_bytes = B.nvfp4_prepared_weight_bytes(self.G, self.N, self.K)
        raw_B = to_device(d["B"], device)
        raw_Bsf = to_device(d["B_sf"], device)
        self.B_prep = torch.empty(b_bytes, dtype=torch.uint8, device=device)
        self.B_sf_prep = torch.empty(sf_bytes, dtype=torch.uint8, device=device)
        B.nvfp4_prepare_weights(raw_B, raw_Bsf, self.G, self.N, self.K, self.B_prep,
                                self.B_sf_prep, stream)
        if keep_raw_weights:
            self.raw_B, self.raw_Bsf = raw_B, raw_Bsf
        else:
            self.raw_B = self.raw_Bsf = None
            del raw_B, raw_Bsf
        self.C = torch.full((self.G, self.M_max, self.N), SENTINEL_BF16, dtype=torch.int16,
                            device=device)

    def reset_C(self):
        self.C.fill_(SENTINEL_BF16)

    def run(self, stream=None, C=None):
        B.nvfp4_grouped_gemm_nt_masked(self.A, self.A_sf, self.B_prep, self.B_sf_prep, self.alpha,
                                       self.masked_m, self.C if C is None else C, self.G,
                                       self.M_max, self.N, self.K, stream)

    def C_bits(self) -> np.ndarray:
        return self.C.cpu().numpy().view(np.uint16)
