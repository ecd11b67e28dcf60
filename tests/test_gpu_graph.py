"""The library's calls under CUDA graph capture: the decode forward (two
launches chained by programmatic dependent launch) and the packed backward
(dB and dA forked onto side streams and joined) replay to the same results
as eager calls."""
import numpy as np
import pytest
import torch

import adapter_sgmv_gb300 as lora
import workloads as wl
from lora_testlib import GpuCase

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lora.build_library()
    lora.lib()


def _spec(T):
    ranks = [16, 64, 128]
    rng = np.random.default_rng(T)
    ids = rng.integers(0, 3, T).astype(np.int32)
    return wl.custom(f"graph{T}", 512, 640, ranks, [2.0 * r for r in ranks], ids)


@pytest.mark.parametrize("T", [200, 1500])  # decode kernels / packed kernels
def test_captured_step_replays_eager_results(T):
    spec = _spec(T)
    case = GpuCase(spec, wl.host_inputs(spec, y0="randn", dX0="randn"))
    y_ref, H_ref = case.fwd()
    dX_ref, dA_ref, dB_ref = case.bwd(H_ref)
    torch.cuda.synchronize()

    y = torch.empty_like(y_ref)
    H = torch.empty_like(H_ref)
    dX = torch.empty_like(dX_ref)
    dA = torch.empty_like(dA_ref)
    dB = torch.empty_like(dB_ref)
    stream = torch.cuda.Stream()

    def step():
        y.copy_(case.inp["y0"])
        dX.copy_(case.inp["dX0"])
        lora.lora_packed_fwd(y, H, case.inp["x"], case.table, case.segs, case.ws, stream=stream)
        lora.lora_packed_bwd(dX, dA, dB, case.inp["dY"], case.inp["x"], H, case.table, case.segs, case.ws,
                             stream=stream)

    with torch.cuda.stream(stream):
        step()  # first calls (side streams, kernel attributes) outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    for _ in range(2):
        y.zero_()
        dA.zero_()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        assert lora.lora_query_status(case.segs) == 0
        for got, ref in ((y, y_ref), (H, H_ref), (dX, dX_ref), (dA, dA_ref), (dB, dB_ref)):
            assert torch.equal(got, ref)
