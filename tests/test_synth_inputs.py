"""The seeded inputs are the recorded ones: SHA-256 of every workload's Q, K and V.

The parity tests, the bench and the stored traffic figures all run on these tensors; the record in
``tests/golden/input_sha256.json`` (written by ``tests/golden/make_input_sha256.py``) makes a silent
change of the generator visible.  Normal draws pass through the host's fp64 ``log1p``, ``cos`` and
``sin``, so the digests are checked only on the machine type they were written on.
"""

from __future__ import annotations

import hashlib
import json
import os
import platform

import numpy as np
import pytest

import synth

with open(os.path.join(os.path.dirname(__file__), "golden", "input_sha256.json")) as f:
    RECORD = json.load(f)


def test_record_covers_every_workload():
    assert sorted(RECORD["workloads"]) == sorted(synth.WORKLOADS)


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_input_digests(name):
    if platform.machine() != RECORD["machine"]:
        pytest.skip(f"digests recorded on {RECORD['machine']}")
    w = synth.WORKLOADS[name]
    for tname, a in zip("QKV", synth.make_workload(w)):
        want = RECORD["workloads"][name][tname]
        assert "x".join(str(s) for s in a.shape) == want["shape"], f"{name} {tname} shape"
        got = hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()
        assert got == want["sha256"], f"{name} {tname}: inputs differ from the recorded ones"
