"""Write tests/golden/tiny_layer_oracle.json from the CPU oracle alone.

Run from the repository root: python tests/golden/gen_golden.py
The file records digests and a few values of the oracle's result on the tiny
layer (M=16, K=2048, N=256, seed 0) so that an unintended change to the
oracle's arithmetic shows up as a test failure.
"""

import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from oracle import ternary_linear as O  # noqa: E402
from quantized_linear_layers_block_gb300 import synth  # noqa: E402


def digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def compute() -> dict:
    L = synth.config_inputs("tiny")
    r = O.layer(L.x_bits, L.codes, L.s)
    packed, qT, sw = O.pack_weights(L.codes, L.s)
    return {
        "inputs": {"codes": digest(L.codes), "s": digest(L.s), "x_bits": digest(L.x_bits)},
        "packed": digest(packed), "qT": digest(qT), "sw": digest(sw),
        "xq": digest(r["xq"]), "sx": digest(r["sx"]),
        "acc": digest(r["acc"].astype(np.int32)), "y32": digest(r["y32"]), "ybf": digest(r["ybf"]),
        "acc_00_01_10": [int(r["acc"][0, 0]), int(r["acc"][0, 1]), int(r["acc"][1, 0])],
        "sx_0": float(r["sx"][0]),
        "rel_fro_vs_fp64": O.rel_fro(r["y32"], O.reference_fp64(L.x_bits, L.codes, L.s)),
    }


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_layer_oracle.json")
    with open(out, "w") as f:
        json.dump(compute(), f, indent=1, sort_keys=True)
        f.write("\n")
    print("wrote", out)
