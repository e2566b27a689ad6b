"""Writes the stored expected values under tests/golden/ from the CPU oracle.

Run from the repository root:  python tests/golden/make_golden.py

Only oracle/ computes the values; the inputs come from the seeded generator.
The pages print no worked numeric example, so these files are regression pins
of the oracle on the small workload (B=1, H=1, N=128, d=64, seed 0, both
masks) plus checksums that pin the generator's output bits.
"""
from __future__ import annotations

import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from exact_softmax_attention_fattn_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402

ROWS = [0, 1, 2, 63, 64, 65, 126, 127]


def digest(a) -> str:
    return hashlib.sha256(a.tobytes()).hexdigest()


def golden_for(name: str) -> dict:
    w = WORKLOADS[name]
    x = make_inputs(w)
    o, lse = oracle.forward(x.q, x.k, x.v, w.softmax_scale, w.causal, key_len=x.key_len)
    return {
        "workload": name,
        "shape": [w.B, w.H, w.N, w.d],
        "causal": w.causal,
        "scale": w.softmax_scale,
        "seed": w.seed,
        "sha256_q_bits": digest(x.q),
        "sha256_k_bits": digest(x.k),
        "sha256_v_bits": digest(x.v),
        "first_q_bits": [int(b) for b in x.q.reshape(-1)[:8]],
        "rows": ROWS,
        "o_rows": [[float.hex(float(t)) for t in o[0, 0, r]] for r in ROWS],
        "lse": [float.hex(float(t)) for t in lse[0, 0]],
    }


def main() -> None:
    for name in ("b1h1n128d64", "b1h1n128d64_causal"):
        path = os.path.join(HERE, f"{name}.json")
        with open(path, "w") as f:
            json.dump(golden_for(name), f, indent=1)
            f.write("\n")
        print("wrote", path)


if __name__ == "__main__":
    main()
