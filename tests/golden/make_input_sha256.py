"""Writes ``input_sha256.json``: the SHA-256 of every seeded input tensor of the attention workloads.

The record pins the generator: a change to the stream, the distributions, the rounding or the fill
order changes a digest, and the test ``tests/test_synth_inputs.py`` fails until this script is run
again on purpose.  Only the input generator is called; no attention arithmetic is involved.

Normal draws go through the host's fp64 ``log1p``, ``cos`` and ``sin``; a last-place difference in those can
flip the fp32 rounding of a rare element, so every machine type (``platform.machine()``) keeps its own
digests.  The script replaces the entry of the machine it runs on and keeps the others.

Run from the repository root:  python tests/golden/make_input_sha256.py [output path]
(default: the record next to this script; another path starts from that record's contents).
"""

from __future__ import annotations

import hashlib
import json
import os
import platform
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import synth  # noqa: E402


def digests(w: synth.Workload) -> dict:
    q, k, v = synth.make_workload(w)
    out = {}
    for name, a in (("Q", q), ("K", k), ("V", v)):
        out[name] = {"shape": "x".join(str(s) for s in a.shape), "element": w.dtype,
                     "sha256": hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()}
    return out


RECORD = os.path.join(HERE, "input_sha256.json")


def main() -> None:
    out = sys.argv[1] if len(sys.argv) > 1 else RECORD
    try:
        with open(RECORD) as f:
            record = json.load(f)
    except OSError:
        record = {}
    record.setdefault("what", "SHA-256 of the bytes of Q, K and V (row-major [B,H,S,D]; bf16 as uint16 bit "
                              "patterns, f32 as float32, little-endian) for each seeded workload")
    record.setdefault("note", "normal draws go through the host's fp64 log1p, cos and sin; a last-place "
                              "difference in those can flip the fp32 rounding of a rare element, so each "
                              "machine type keeps its own digests")
    record.setdefault("machines", {})[platform.machine()] = {
        "numpy": np.__version__,
        "workloads": {name: digests(w) for name, w in synth.WORKLOADS.items()},
    }
    with open(out, "w") as f:
        json.dump(record, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
