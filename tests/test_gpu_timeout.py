"""Failure detection without a GPU fault: the tensor-core kernels' bounded
pipeline wait, run against a barrier that nothing completes, gives up after
its cycle limit, writes LORA_ERR_TIMEOUT to the status word and returns; the
context stays usable (a packed forward right after it matches the oracle)."""
import time

import pytest
import torch

import adapter_sgmv_gb300 as lora
import workloads as wl
from lora_testlib import FWD_TOL, GpuCase, assert_close, dev_to_f64, oracle_all

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lora.build_library()
    lora.lib()


def test_stalled_wait_ends_with_timeout_status_and_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    lora.lora_check_wait_timeout(status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == 7  # LORA_ERR_TIMEOUT
    assert 0.5 < elapsed < 30.0  # 4e9 SM cycles: about 2 s at GB300 clocks
    # a status already set is kept (first error wins)
    status.fill_(4)
    lora.lora_check_wait_timeout(status)
    torch.cuda.synchronize()
    assert int(status.item()) == 4
    # the context still runs the path
    spec = wl.tiny()
    host = wl.host_inputs(spec, y0="randn")
    case = GpuCase(spec, host)
    y, H = case.fwd()
    torch.cuda.synchronize()
    assert lora.lora_query_status(case.segs) == 0
    ref = oracle_all(spec, host)
    assert_close(dev_to_f64(y), ref["y"], FWD_TOL, "y")

