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


def test_captured_fused_layer_and_multi_projection_replay_eager_results():
    # the fused base + delta launch (cooperative, with its counter reset) and a
    # multi-projection decode call, captured together
    lengths = [300, 130, 270]
    ids = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lengths)])
    spec = wl.custom("graphfb", 320, 512, [16, 64, 128], [64.0, 256.0, 512.0], ids)
    case = GpuCase(spec, wl.host_inputs(spec))
    W = torch.from_numpy(wl.base_weight(spec).view(np.int16)).cuda().view(torch.bfloat16)
    ws_f = torch.empty(lora.lora_fused_base_workspace_bytes(case.table, spec.n_tokens), dtype=torch.uint8,
                       device="cuda")
    dec_ids = np.random.default_rng(9).integers(0, 3, 64).astype(np.int32)
    d1 = wl.custom("graphm1", 320, 256, [16, 64, 128], [32.0] * 3, dec_ids, with_bwd=False)
    d2 = wl.custom("graphm2", 320, 128, [8, 8, 32], [16.0] * 3, dec_ids, with_bwd=False)
    c1 = GpuCase(d1, wl.host_inputs(d1, y0="randn"))
    c2 = GpuCase(d2, wl.host_inputs(d2, y0="randn"))
    x_dec = c1.inp["x"]
    ws_m = torch.empty(lora.lora_multi_workspace_bytes([c1.table, c2.table], 64), dtype=torch.uint8, device="cuda")

    def run(y, H, ys):
        lora.lora_fused_base_fwd(y, H, case.inp["x"], W, case.table, case.segs, ws_f, stream=stream)
        ys[0].copy_(c1.inp["y0"])
        ys[1].copy_(c2.inp["y0"])
        lora.lora_multi_fwd(ys, None, x_dec, [c1.table, c2.table], c1.segs, ws_m, stream=stream)

    stream = torch.cuda.Stream()
    mk = lambda: (torch.empty((spec.n_tokens, spec.d_out), dtype=torch.bfloat16, device="cuda"),
                  torch.empty((spec.n_tokens, spec.r_max), dtype=torch.float32, device="cuda"),
                  [torch.empty_like(c1.inp["y0"]), torch.empty_like(c2.inp["y0"])])
    y_ref, H_ref, ys_ref = mk()
    with torch.cuda.stream(stream):
        run(y_ref, H_ref, ys_ref)
    torch.cuda.synchronize()
    y, H, ys = mk()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run(y, H, ys)
    for _ in range(2):
        y.zero_()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        assert lora.lora_query_status(case.segs) == 0 and lora.lora_query_status(c1.segs) == 0
        assert torch.equal(y, y_ref) and torch.equal(H, H_ref)
        assert torch.equal(ys[0], ys_ref[0]) and torch.equal(ys[1], ys_ref[1])
