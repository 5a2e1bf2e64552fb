"""DS4A_NVTX=1 wraps every C-ABI op in an NVTX range named after it (for
Nsight Systems timelines); with the variable unset nothing is recorded.  Either
way the results must be the same, bit for bit.  The variable is read once per
process, so each setting runs in a process of its own."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCRIPT = r"""
import hashlib, sys
sys.path.insert(0, sys.argv[1])
import torch
import deepseek_v4_sparse_indexer_gb300 as P
from deepseek_v4_sparse_indexer_gb300.workloads import make_decode_inputs
x = make_decode_inputs(3, 40000, device="cuda", seed=5, n_rows=[40000, 39000, 700])
st = P.DecodeStep(3, 40000, 512)
st(x, 0.044194173824159216)
torch.cuda.synchronize()
h = hashlib.sha256()
for t in (st.scores, st.idx, st.count, st.out, st.lse):
    h.update(t.cpu().numpy().tobytes())
print(h.hexdigest(), P.ds4a_get_device_status()[0])
"""


def _run(nvtx):
    env = dict(os.environ)
    env.pop("DS4A_NVTX", None)
    if nvtx:
        env["DS4A_NVTX"] = "1"
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout.split()


def test_nvtx_ranges_leave_results_unchanged():
    a, b = _run(False), _run(True)
    assert a[1] == "0" and b[1] == "0"
    assert a[0] == b[0]
