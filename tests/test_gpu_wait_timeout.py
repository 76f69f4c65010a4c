"""The kernels' bounded barrier wait, made to run out on the GPU: one thread
waits for a barrier phase that nothing completes.  The wait must give up
after its limit, report TREEWY_STATUS_TIMEOUT through the status word, and
leave the CUDA context usable for the next verification."""
import numpy as np
import pytest
import torch

from gdn_speculative_tree_gb300 import binding
from gdn_speculative_tree_gb300 import workloads as wl
from tests.gpu_helpers import CudaRun, assert_within, compare

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_us", [2_000, 50_000])
def test_wait_gives_up_and_reports(cuda_lib, limit_us):
    status = torch.zeros(3, dtype=torch.int32, device="cuda")
    binding.treewy_selftest_wait_timeout(status, limit_us)
    torch.cuda.synchronize()
    s = status.cpu().numpy().astype(np.int64)
    assert s[0] == binding.STATUS_TIMEOUT
    waited_ns = (s[1] & 0xFFFFFFFF) | (s[2] << 32)
    assert limit_us * 1000 <= waited_ns < limit_us * 1000 + 5_000_000, waited_ns

    # the context still runs the hot path correctly afterwards
    w = wl.generate(wl.CONFIGS["binary"], R=4).to("cuda")
    run = CudaRun(w)
    assert not run.status.any()
    assert_within(compare(w, run, range(w.R)), "after a timed-out wait")
