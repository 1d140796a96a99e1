"""Bounded-wait error path on the GPU, without a fault, trap or hang.

A child process sets WST_FAULT_INJECT=drop_load (the first dense GEMM launch
leaves one K-block unloaded) and a 200 ms wait limit.  The MMA issuer's
bounded wait must run out, the kernel must exit, wst_sync_status must report
WST_ERR_TIMEOUT, and the next call on the same context must be correct."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, torch
sys.path.insert(0, %r); sys.path.insert(0, %r)
import oracle, synthetic
import warp_specialized_tensor_gb300 as wst
from gpu_util import amax, assert_parity
d = synthetic.dense(128, 256, 256, seed=51)
A, B = d["A"].cuda(), d["B"].cuda()
C = torch.zeros(128, 256, dtype=torch.float32, device="cuda")
ws = wst.workspace()
wst.wst_gemm_bf16(A, B, C, workspace=ws)          # injected: one K-block never arrives
st = wst.wst_sync_status(ws)
print("first_status", st)
wst.wst_gemm_bf16(A, B, C, workspace=ws)          # normal
st2 = wst.wst_sync_status(ws)
print("second_status", st2)
assert_parity(C, oracle.gemm(d["A"], d["B"]), 256, amax(d["A"]), amax(d["B"]), False, what="after timeout")
print("ok")
''' % (ROOT, os.path.join(ROOT, "tests"))


def test_bounded_wait_times_out_and_context_survives():
    env = dict(os.environ, WST_FAULT_INJECT="drop_load", WST_TIMEOUT_MS="200")
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, capture_output=True, text=True,
                       timeout=300)
    out = r.stdout + r.stderr
    assert r.returncode == 0, out
    assert "first_status 5" in out, out      # WST_ERR_TIMEOUT
    assert "second_status 0" in out, out
    assert out.rstrip().endswith("ok"), out
