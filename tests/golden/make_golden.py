"""Writes tests/golden/tiny_case.json: a tiny seeded case and the oracle's
output bits for it.  Calls only the oracle and the seeded input generator."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
from oracle import oracle  # noqa: E402
from nvfp4_block_scaled_masked_gb300 import workloads as W  # noqa: E402


def main():
    G, M, N, K = 2, 4, 4, 32
    cfg = W.custom(G, M, N, K, masked_m=[3, 0])
    d = W.generate(cfg, seed=20261202)
    C, _ = oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], d["masked_m"],
                       d["C_init"], G, M, N, K)
    out = dict(G=G, M_max=M, N=N, K=K, masked_m=[int(x) for x in d["masked_m"]],
               alpha=[float(x) for x in d["alpha"]],
               A=d["A"].tobytes().hex(), A_sf=d["A_sf"].tobytes().hex(),
               B=d["B"].tobytes().hex(), B_sf=d["B_sf"].tobytes().hex(),
               C_bits=[int(x) for x in C.ravel()])
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_case.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
