"""lora_packed_bwd_concurrent: the packed backward with dB and dA on side
streams the caller owns.

Its results must be those of lora_packed_bwd bit for bit (the same kernels,
only the streams differ), and independent callers must not share anything:
two host threads, each with its own stream, side streams, workspace and
segments, run forward and backward at the same time and both match the fp64
oracle."""
import threading

import numpy as np
import pytest
import torch

import adapter_sgmv_gb300 as lora
import workloads as wl
from lora_testlib import FWD_TOL, GRAD_TOL, GpuCase, assert_close, check_blocks, dev_to_f64, oracle_all

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lora.build_library()
    lora.lib()


def spec_of(seed, T=900):
    rng = np.random.default_rng(300 + seed)
    ranks = [8, 16, 32, 64, 128, 24]
    ids = rng.integers(0, len(ranks), T).astype(np.int32)
    if seed % 2 == 0:
        ids = np.sort(ids)
    return wl.custom(f"conc{seed}", 264, 328, ranks, [2.0 * r for r in ranks], ids, seed=seed)


def run_bwd(case, H, side=None, stream=None):
    s = case.spec
    dX = case.inp["dX0"].clone()
    dA = torch.full((s.sum_r, s.d_in), float("nan"), dtype=torch.float32, device="cuda")
    dB = torch.full((s.sum_r, s.d_out), float("nan"), dtype=torch.float32, device="cuda")
    if side is None:
        lora.lora_packed_bwd(dX, dA, dB, case.inp["dY"], case.inp["x"], H, case.table, case.segs, case.ws,
                             stream=stream)
    else:
        lora.lora_packed_bwd_concurrent(dX, dA, dB, case.inp["dY"], case.inp["x"], H, case.table, case.segs,
                                        case.ws, side, stream=stream)
    return dX, dA, dB


@pytest.mark.parametrize("saved", [True, False])
def test_concurrent_backward_equals_serial_backward_bitwise(saved):
    spec = spec_of(0)
    case = GpuCase(spec, wl.host_inputs(spec, dX0="randn"))
    y, H = case.fwd()
    h = H if saved else None
    ref = run_bwd(case, h)
    side = lora.SideStreams()
    for _ in range(3):  # the same side streams and events, reused call after call
        got = run_bwd(case, h, side)
        torch.cuda.synchronize()
        for g, r, what in zip(got, ref, ("dX", "dA", "dB")):
            assert torch.equal(g, r), what  # every adapter here has one span: dA / dB are bit-reproducible
    assert lora.lora_query_status(case.segs) == 0


def test_concurrent_backward_rejects_bad_side_streams():
    import ctypes

    spec = spec_of(0, T=64)
    case = GpuCase(spec, wl.host_inputs(spec))
    _, H = case.fwd()
    side = lora.SideStreams()
    cur = torch.cuda.current_stream()

    def call_with(c):  # a modified copy of the owned set; the set itself stays intact
        s = spec
        dX = case.inp["dX0"].clone()
        dA = torch.empty((s.sum_r, s.d_in), dtype=torch.float32, device="cuda")
        dB = torch.empty((s.sum_r, s.d_out), dtype=torch.float32, device="cuda")
        P = lambda t: ctypes.c_void_p(t.data_ptr())
        return lora.lib().lora_packed_bwd_concurrent(
            P(dX), P(dA), P(dB), P(case.inp["dY"]), P(case.inp["x"]), P(H), ctypes.byref(case.table.c),
            ctypes.byref(case.segs.c), P(case.ws), case.ws.numel(), ctypes.byref(c), ctypes.c_void_p(cur.cuda_stream))

    def copy():
        c = lora.c_side_streams()
        ctypes.memmove(ctypes.addressof(c), ctypes.addressof(side.c), ctypes.sizeof(c))
        return c

    bad = copy()
    bad.stream[1] = bad.stream[0]  # the two side streams coincide
    assert call_with(bad) == 1
    bad = copy()
    bad.stream[0] = cur.cuda_stream  # a side stream is the caller's stream
    assert call_with(bad) == 1
    bad = copy()
    bad.event[3] = bad.event[0]  # two events coincide
    assert call_with(bad) == 1
    bad = copy()
    bad.event[2] = None
    assert call_with(bad) == 1
    assert call_with(copy()) == 0  # the intact set works
    run_bwd(case, H, side)
    torch.cuda.synchronize()
    assert lora.lora_query_status(case.segs) == 0


def test_side_streams_are_fresh_and_distinct():
    """Sets made by lora_side_streams_create never coincide with each other or
    with streams torch hands out (torch's stream pool recycles its streams)."""
    pool = [torch.cuda.Stream() for _ in range(40)]
    sets = [lora.SideStreams() for _ in range(6)]
    handles = [h for st in sets for h in st.c.stream]
    assert len(set(handles)) == len(handles)
    assert not set(handles) & {p.cuda_stream for p in pool}
    events = [h for st in sets for h in st.c.event]
    assert len(set(events)) == len(events) and all(events)
    del sets
    torch.cuda.synchronize()


def test_two_host_threads_run_backward_at_once():
    specs = [spec_of(1), spec_of(2, T=1400)]
    hosts = [wl.host_inputs(s, y0="zero", dX0="zero") for s in specs]
    results = [None, None]
    errors = []
    start = threading.Barrier(2)

    def worker(k):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                case = GpuCase(specs[k], hosts[k])
                side = lora.SideStreams()
                torch.cuda.synchronize()
                start.wait()
                for _ in range(20):  # many calls, so the two threads' work interleaves on the GPU
                    y, H = case.fwd()
                    dX, dA, dB = run_bwd(case, H, side, stream=stream)
                stream.synchronize()
                results[k] = (case, y, H, dX, dA, dB, lora.lora_query_status(case.segs, stream=stream))
        except Exception as e:  # surfaced in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k in range(2):
        case, y, H, dX, dA, dB, st = results[k]
        assert st == 0
        ref = oracle_all(specs[k], hosts[k])
        assert_close(dev_to_f64(y), ref["y"], FWD_TOL, f"y[{k}]")
        assert_close(dev_to_f64(H), ref["H"], FWD_TOL, f"H[{k}]")
        assert_close(dev_to_f64(dX), ref["dX"], GRAD_TOL, f"dX[{k}]")
        check_blocks(specs[k], dev_to_f64(dA), dev_to_f64(dB), ref["dA"], ref["dB"])
