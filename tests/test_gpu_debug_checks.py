"""The debug build's bounds checks on the GPU (the stand-in for a memory checker,
which is closed on this machine).  libfathom_debug.so is the library compiled with
-DFATHOM_DEBUG: every scan, gather and attention access whose index comes from
data first checks that it lies inside the buffer the call was given, and
records the first failure per kernel file.  A child process loads that build
(FATHOM_LIB), checks that a planted self-test record is reported, clears the
records, runs the parity cases below through the oracle comparison, and
reports the records, which must all be zero."""
import json
import os
import subprocess
import sys

import pytest
import torch

from bit_plane_kv_gb300 import build as BUILD

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = r"""
import json, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np, torch
from bit_plane_kv_gb300 import binding as B, synth
import fathom_cases as FC
assert B.LIB_PATH.endswith("libfathom_debug.so"), B.LIB_PATH
planted = B.fathom_debug_status(2)
B.fathom_debug_status(1)
w = synth.shrink(synth.WORKLOADS["qwen3_32k"], n=6481)
inp = FC.Inputs(w, [0, 1, 2], 6481)
for regime in ("hbm", "host", "fused"):
    r = FC.run_gpu(inp, k=300, budget=[40, 48, 56], regime=regime)
    for ui in range(3):
        FC.check_unit(inp, r, ui, 300, [40, 48, 56])
r = FC.run_gpu(inp, k=300, budget=48, fixed=(32, 4), regime="host")
FC.check_unit(inp, r, 0, 300, 48, fixed=(32, 4))
w1 = synth.shrink(synth.WORKLOADS["host_1m"], n=1 << 17, layers=1)
inp1 = FC.Inputs(w1, list(range(8)), 1 << 17)
r = FC.run_gpu(inp1, k=512, budget=48, regime="fused", want_scores=False)
torch.cuda.synchronize()
print("DEBUG_STATUS " + json.dumps({{"planted": planted, "after": B.fathom_debug_status(0)}}))
"""


def test_debug_build_checks_stay_silent_on_the_parity_cases():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = BUILD.build(debug=True)
    env = dict(os.environ, FATHOM_LIB=lib)
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, tests=HERE)], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = [x for x in r.stdout.splitlines() if x.startswith("DEBUG_STATUS ")][-1]
    st = json.loads(line.split(" ", 1)[1])
    assert st["planted"] == [(15 << 48) | 0x5E1F] * 3          # the reporting path works in every file
    assert st["after"] == [0, 0, 0], [hex(x) for x in st["after"]]
