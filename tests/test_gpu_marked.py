"""The measurement entry points (lora_packed_fwd_marked / _bwd_marked) launch
the same kernels as the plain calls: identical results, and one event pair
recorded per kernel in the documented order."""
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


def _events(n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _case(T):
    ranks = [16, 32, 128]
    lengths = [T // 2, T // 4, T - T // 2 - T // 4]
    ids = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lengths)])
    spec = wl.custom(f"marked{T}", 512, 384, ranks, [32.0] * 3, ids)
    return spec, GpuCase(spec, wl.host_inputs(spec, y0="randn", dX0="randn"))


@pytest.mark.parametrize("T,fwd_kernels", [(945, 2), (300, 1)])
def test_marked_calls_match_plain_calls(T, fwd_kernels):
    spec, case = _case(T)
    y1, H1 = case.fwd()
    dX1, dA1, dB1 = case.bwd(H1)

    y2 = case.inp["y0"].clone()
    H2 = torch.zeros_like(H1)
    ev = _events(6)
    n = lora.lora_packed_fwd_marked(y2, H2, case.inp["x"], case.table, case.segs, case.ws, ev)
    assert n == 2 * fwd_kernels
    dX2 = case.inp["dX0"].clone()
    dA2 = torch.full_like(dA1, float("nan"))
    dB2 = torch.full_like(dB1, float("nan"))
    evb = _events(10)
    nb = lora.lora_packed_bwd_marked(dX2, dA2, dB2, case.inp["dY"], case.inp["x"], H2, case.table, case.segs,
                                     case.ws, evb)
    assert nb == 10  # H to bf16, dB, dh, dA, dX
    torch.cuda.synchronize()
    assert lora.lora_query_status(case.segs) == 0
    for a, b in ((y1, y2), (H1, H2), (dX1, dX2), (dA1, dA2), (dB1, dB2)):
        assert torch.equal(a, b)
    for k in range(0, n, 2):
        assert ev[k].elapsed_time(ev[k + 1]) >= 0.0
    for k in range(0, nb, 2):
        assert evb[k].elapsed_time(evb[k + 1]) >= 0.0


def test_marked_backward_with_fewer_events_than_kernels():
    spec, case = _case(945)
    y, H = case.fwd()
    dX1, dA1, dB1 = case.bwd(None)  # recomputes H: five kernels
    dX2 = case.inp["dX0"].clone()
    dA2 = torch.full_like(dA1, float("nan"))
    dB2 = torch.full_like(dB1, float("nan"))
    ev = _events(3)
    n = lora.lora_packed_bwd_marked(dX2, dA2, dB2, case.inp["dY"], case.inp["x"], None, case.table, case.segs,
                                    case.ws, ev)
    torch.cuda.synchronize()
    assert n == 3
    assert torch.equal(dX1, dX2) and torch.equal(dA1, dA2) and torch.equal(dB1, dB2)
