"""lora_packed_bwd_noalloc: the packed backward for callers that cannot
allocate device memory (its scratch sits in a fixed array inside the library).

It is checked through the C ABI on the same inputs, on two calls in a row:
against lora_packed_bwd (the workspace version, which runs the same kernels)
bit for bit -- dX always, dA and dB because every adapter here has at most two
spans of tokens -- and against the fp64 oracle at the tolerance the other
gradient tests use.  This file is collected last so that a failure here comes
after every other test has run."""
import ctypes

import numpy as np
import pytest
import torch

import adapter_sgmv_gb300 as lora
import workloads as wl
from lora_testlib import GRAD_TOL, GpuCase, check_blocks, dev_to_f64, assert_close, oracle_all

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lora.build_library()
    lora.lib()


def outputs(case, fn, H):
    s = case.spec
    dX = case.inp["dX0"].clone()
    dA = torch.full((s.sum_r, s.d_in), float("nan"), dtype=torch.float32, device="cuda")
    dB = torch.full((s.sum_r, s.d_out), float("nan"), dtype=torch.float32, device="cuda")
    fn(dX, dA, dB, H)
    torch.cuda.synchronize()
    return dX, dA, dB


@pytest.mark.parametrize("name", ["tiny", "ragged_unsorted"])
def test_noalloc_backward_matches_workspace_backward_twice(name):
    if name == "tiny":
        spec = wl.tiny()
    else:
        rng = np.random.default_rng(21)
        ranks = [8, 16, 24, 64, 128]
        spec = wl.custom("ragged", 136, 200, ranks, [2.0 * r for r in ranks],
                         rng.integers(0, 5, 333).astype(np.int32))
    assert spec.n_tokens <= 2 * 1024  # at most two spans per adapter: dA / dB are bit-reproducible
    host = wl.host_inputs(spec, dX0="randn")
    case = GpuCase(spec, host)
    y, H = case.fwd()
    # the reference per mode: a saved H (here from the decode-size forward) and
    # an H recomputed by the backward's own shrink may differ in their last bits
    ws_bwd = lambda dX, dA, dB, h: lora.lora_packed_bwd(dX, dA, dB, case.inp["dY"], case.inp["x"], h, case.table,
                                                        case.segs, case.ws)
    refs = {True: outputs(case, ws_bwd, H), False: outputs(case, ws_bwd, None)}
    orc = oracle_all(spec, host)
    for call in range(2):
        for saved in (H, None):
            tag = f"call {call}, H {'saved' if saved is not None else 'recomputed'}"
            got = outputs(case, lambda dX, dA, dB, h: lora.lora_packed_bwd_noalloc(
                dX, dA, dB, case.inp["dY"], case.inp["x"], h, case.table, case.segs), saved)
            for g, r, what in zip(got, refs[saved is not None], ("dX", "dA", "dB")):
                assert torch.equal(g, r), f"{what} ({tag}) differs from lora_packed_bwd"
            assert_close(dev_to_f64(got[0]), orc["dX"], GRAD_TOL, f"dX ({tag})")
            check_blocks(spec, dev_to_f64(got[1]), dev_to_f64(got[2]), orc["dA"], orc["dB"])
    assert lora.lora_query_status(case.segs) == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    T = 16500  # two bf16 hand-off copies of [T, 128]: 2 * 16500 * 128 * 2 bytes = 8.45 MB > 8 MiB
    spec = wl.custom("big", 64, 64, [128], [256.0], np.zeros(T, np.int32))
    dev = torch.device("cuda")
    A = torch.zeros((128, 64), dtype=torch.bfloat16, device=dev)
    B = torch.zeros((128, 64), dtype=torch.bfloat16, device=dev)
    table = lora.AdapterTable(A, B, [128], [2.0], 64, 64)
    segs = lora.lora_build_segments(seg_offsets=torch.tensor([0, T], dtype=torch.int32, device=dev),
                                    n_tokens=T, n_adapters=1)
    dY = torch.zeros((T, 64), dtype=torch.bfloat16, device=dev)
    X = torch.zeros((T, 64), dtype=torch.bfloat16, device=dev)
    st = lora.lib().lora_packed_bwd_noalloc(None, None, None, ctypes.c_void_p(dY.data_ptr()),
                                           ctypes.c_void_p(X.data_ptr()), None, ctypes.byref(table.c),
                                           ctypes.byref(segs.c), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 5  # LORA_ERR_WORKSPACE_TOO_SMALL
    assert spec.n_tokens == T
    # a batch of rank-128 adapters that fits: two copies of 16256 x 128 bf16 (8,323,072 bytes)
    # plus a 256-byte block of work-claim counters and one of tickets, below 8 MiB
    T = 16256
    segs = lora.lora_build_segments(seg_offsets=torch.tensor([0, T], dtype=torch.int32, device=dev),
                                    n_tokens=T, n_adapters=1)
    st = lora.lib().lora_packed_bwd_noalloc(None, None, None, ctypes.c_void_p(dY.data_ptr()),
                                           ctypes.c_void_p(X.data_ptr()), None, ctypes.byref(table.c),
                                           ctypes.byref(segs.c), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    assert lora.lora_query_status(segs) == 0
