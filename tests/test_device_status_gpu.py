"""The device-side failure path without a fault: a bounded wait that nothing
completes gives up, sets DS4A_DEV_TIMEOUT in the device status word, and the
context stays usable (the compute kernels' waits behave the same way when a
producer never arrives)."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_sparse_indexer_gb300 import _binding as B

pytestmark = pytest.mark.gpu


def test_a_wait_nothing_completes_reports_a_timeout_and_the_context_stays_usable(cuda_lib):
    st, flags = B.ds4a_get_device_status()                  # start clean
    B.ds4a_debug_wait_timeout(2000)                          # 2 ms
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_EDEVICE and flags == B.DS4A_DEV_TIMEOUT
    st, flags = B.ds4a_get_device_status()                  # read once, then cleared
    assert st == B.DS4A_OK and flags == 0
    # the next op runs normally on the same context
    x = torch.randn(2, 1, 3000, device="cuda")
    n = torch.tensor([3000, 1234], dtype=torch.int32, device="cuda")
    idx = torch.empty(2, 1, 64, dtype=torch.int32, device="cuda")
    cnt = torch.empty(2, 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.ds4a_workspace_bytes(B.DS4A_OP_TOPK_SELECT, 2, 1, 3000, 64), dtype=torch.uint8, device="cuda")
    B.ds4a_topk_select(x, n, 64, idx, cnt, ws)
    st, flags = B.ds4a_get_device_status()
    assert st == B.DS4A_OK and flags == 0
    xs = x.cpu().numpy()
    for u, m in ((0, 3000), (1, 1234)):
        want, _ = oracle.topk_select(xs[u, 0, :m].astype(np.float64), 64)
        assert np.array_equal(idx[u, 0].cpu().numpy(), want)


def test_wait_hook_rejects_out_of_range_limits(cuda_lib):
    for bad in (0, 100001):
        with pytest.raises(B.Ds4aError) as e:
            B.ds4a_debug_wait_timeout(bad)
        assert e.value.status == B.DS4A_EINVAL
