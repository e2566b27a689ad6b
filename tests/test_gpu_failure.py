"""Failure detection without a GPU fault.

Every wait inside the kernel is bounded.  A child process sets the bound to
1 microsecond, far below the latency of the first tile load, so the waits run
out for real; the kernel must record the time-out (status, role, barrier,
work unit), drain its own copies and MMAs, free tensor memory and return, and
the host must read FATTN_ERR_TIMEOUT from fattn_last_error.  The child then
runs ordinary CUDA work to show the context is still usable.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
case = sys.argv[2]
from exact_softmax_attention_fattn_gb300 import binding
from exact_softmax_attention_fattn_gb300.inputs import Workload, make_inputs
# shapes whose waits run well past 1 us: the 256-column kernel, whose CTAs
# each hold one query tile, gets a non-causal problem (every CTA 64 key tiles)
shapes = {"fwd": (1, 4, 2048, 128, True), "split": (1, 2, 4096, 128, True), "d256": (1, 8, 4096, 256, False),
          "d256split": (1, 2, 4096, 256, False), "bwd256": (1, 2, 1024, 256, True),
          "bwd": (1, 2, 1024, 128, True), "bwdfused": (1, 2, 1024, 128, True), "noalloc": (1, 4, 2048, 128, True),
          "linear": (2, 4, 4096, 64, True)}
B, H, N, d, causal = shapes[case]
x = make_inputs(Workload("to", B, H, N, d, causal, 50))
dev = torch.device("cuda:0")
q, k, v = (torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16) for a in (x.q, x.k, x.v))
o = torch.zeros_like(q); lse = torch.zeros((B, H, N), dtype=torch.float32, device=dev)
if case in ("bwd", "bwd256", "bwdfused"):
    binding.last_error()                  # start clean
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    binding.backward_into(q, k, v, o, lse, q, dq, dk, dv, causal=causal)
elif case == "linear":
    # causal linear attention on the tensor cores (fp32 Q, K, V; E = M = 64)
    lq, lk, lv = (torch.randn(B, H, N, d, device=dev) for _ in range(3))
    binding.linear_forward(lq, lk, lv)
elif case == "noalloc":
    # the no-alloc entry point records its time-out in the word after its
    # static array; fattn_last_error must report it like the others
    st0 = binding.noalloc_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                              1.0 / d ** 0.5, int(causal), None, torch.cuda.current_stream().cuda_stream)
    assert st0 == 0, st0
else:
    binding.forward_into(q, k, v, o, lse, causal=causal, n_splits=4 if case in ("split", "d256split") else None)
st, detail = binding.last_error()
again, _ = binding.last_error()          # the flag is cleared once read
a = torch.randn(512, 512, device=dev)
ok = bool(torch.isfinite(a @ a).all().item())
torch.cuda.synchronize()
print(json.dumps({"status": st, "detail": detail, "again": again, "context_ok": ok}))
"""


@pytest.mark.parametrize("case", ["fwd", "split", "d256", "d256split", "bwd", "bwd256", "bwdfused", "noalloc", "linear"])
def test_bounded_wait_times_out_and_reports(cuda_device, case):
    """Each kernel family (the forward, its split-KV instantiation, the
    256-column forward, the backward's kernels (and the single-kernel
    backward), the tensor-core linear
    attention kernels) and the no-alloc entry point (its error word lives
    after its static array) times out for real and reports; the backward runs on zero O and LSE (values do not matter
    here)."""
    env = dict(os.environ, FATTN_WAIT_LIMIT_US="1")
    if case == "bwdfused":
        env["FATTN_BWD_FUSED"] = "1"  # the single-kernel backward
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, case], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["status"] == 4  # FATTN_ERR_TIMEOUT
    status, role, barrier, unit = res["detail"]
    assert status == 4 and role in (1, 2, 3) and barrier >= 0 and unit >= 0
    assert res["again"] == 0
    assert res["context_ok"]
