"""The ordered backward (lora_packed_bwd_ex with LORA_BWD_DETERMINISTIC): dA
and dB are bit-identical from run to run also for adapters of more than two
spans of LORA_SPAN_TOKENS tokens, where the default backward may add the span
partials in any order, and they still match the fp64 oracle."""
import numpy as np
import pytest
import torch

import adapter_sgmv_gb300 as lora
import workloads as wl
from lora_testlib import GRAD_TOL, GpuCase, assert_close, check_blocks, dev_to_f64, oracle_all

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lora.build_library()
    lora.lib()


def bwd(case, H, side=None, deterministic=True):
    s = case.spec
    dX = case.inp["dX0"].clone()
    dA = torch.full((s.sum_r, s.d_in), float("nan"), dtype=torch.float32, device="cuda")
    dB = torch.full((s.sum_r, s.d_out), float("nan"), dtype=torch.float32, device="cuda")
    lora.lora_packed_bwd_ex(dX, dA, dB, case.inp["dY"], case.inp["x"], H, case.table, case.segs, case.ws,
                            side=side, deterministic=deterministic)
    return dX, dA, dB


@pytest.mark.parametrize("route", ["auto", "ids"])
@pytest.mark.parametrize("concurrent", [False, True])
def test_ordered_backward_is_bit_identical_and_matches_oracle(route, concurrent):
    # adapters of 5, 4 and 4 spans (and one of two), ranks 16..128, a d_out
    # whose last 512-column range is ragged
    lengths = [5000, 4000, 3288, 1500]
    ranks = [16, 64, 128, 8]
    ids = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lengths)])
    if route == "ids":
        ids = np.random.default_rng(4).permutation(ids)
    spec = wl.custom("ordered", 1024, 1544, ranks, [2.0 * r for r in ranks], ids)
    host = wl.host_inputs(spec, y0="zero", dX0="zero")
    case = GpuCase(spec, host, route=route)
    _, H = case.fwd()
    side = lora.SideStreams() if concurrent else None
    first = bwd(case, H, side)
    for _ in range(4):
        again = bwd(case, H, side)
        torch.cuda.synchronize()
        for g, r, what in zip(again, first, ("dX", "dA", "dB")):
            assert torch.equal(g, r), f"{what} differs between runs of the ordered backward"
    assert lora.lora_query_status(case.segs) == 0
    ref = oracle_all(spec, host)
    assert_close(dev_to_f64(first[0]), ref["dX"], GRAD_TOL, "dX")
    check_blocks(spec, dev_to_f64(first[1]), dev_to_f64(first[2]), ref["dA"], ref["dB"])
    # the default order gives the same sums up to rounding
    dflt = bwd(case, H, side, deterministic=False)
    torch.cuda.synchronize()
    check_blocks(spec, dev_to_f64(dflt[1]), dev_to_f64(dflt[2]), ref["dA"], ref["dB"])


def test_ordered_backward_full_packed_batch_repeats():
    # the packed training batch the bench times: 8 adapters of 4096 tokens (four spans each)
    spec = wl.packed4096()
    inp = wl.device_inputs(spec, torch.device("cuda"), y0="zero", dX0="zero")
    case = GpuCase(spec, inp)
    _, H = case.fwd()
    side = lora.SideStreams()
    _, dA1, dB1 = bwd(case, H, side)
    _, dA2, dB2 = bwd(case, H, side)
    torch.cuda.synchronize()
    assert lora.lora_query_status(case.segs) == 0
    assert torch.equal(dA1, dA2) and torch.equal(dB1, dB2)
    # every adapter's blocks against the oracle on that adapter's tokens
    A, B = dev_to_f64(inp["A"]), dev_to_f64(inp["B"])
    for i in (0, 7):
        toks = np.flatnonzero(spec.ids == i)
        rows = lambda t: t[torch.from_numpy(toks).cuda()].float().cpu().numpy().astype(np.float64)
        host_i = {"A": A, "B": B, "x": rows(inp["x"]), "dY": rows(inp["dY"]),
                  "y0": np.zeros((toks.size, spec.d_out)), "dX0": np.zeros((toks.size, spec.d_in))}
        sub = wl.custom(spec.name, spec.d_in, spec.d_out, spec.ranks, spec.alphas, spec.ids[toks], sorted_=False)
        ref = oracle_all(sub, host_i)
        check_blocks(spec, dev_to_f64(dA1), dev_to_f64(dB1), ref["dA"], ref["dB"], adapters=[i])


def test_unknown_flag_bits_are_rejected():
    import ctypes

    spec = wl.tiny()
    case = GpuCase(spec, wl.host_inputs(spec))
    _, H = case.fwd()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    dA = torch.empty((spec.sum_r, spec.d_in), dtype=torch.float32, device="cuda")
    st = lora.lib().lora_packed_bwd_ex(None, P(dA), None, P(case.inp["dY"]), P(case.inp["x"]), P(H),
                                       ctypes.byref(case.table.c), ctypes.byref(case.segs.c), P(case.ws),
                                       case.ws.numel(), None, 6, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 1
