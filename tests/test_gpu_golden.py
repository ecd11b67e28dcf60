"""The CUDA path on the hand-worked example of tests/golden/worked_two_adapters.json:
every value is a small integer, exact in bf16 and fp32, so y, H, dH, dX, dA
and dB must match bit for bit.  Three tokens take the decode-size forward; the
same batch repeated 200 times (600 tokens, unsorted) takes the tensor-core
kernels, with dA / dB 200 times the single batch's (integers below 2^24, so
exact in any summation order)."""
import numpy as np
import pytest
import torch

import adapter_sgmv_gb300 as lora
from lora_testlib import worked_example

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lora.build_library()
    lora.lib()


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(torch.bfloat16)


@pytest.mark.parametrize("repeat", [1, 200])
def test_hand_worked_example_bit_exact(repeat):
    g = worked_example()
    ids = np.tile(g["ids"], repeat)
    T, pad, r_max = ids.size, g["x"].shape[1], g["r_max"]
    table = lora.AdapterTable(_bf16(g["A"]), _bf16(g["B"]), g["ranks"].tolist(),
                              torch.from_numpy(g["scales"].astype(np.float32)), pad, pad)
    segs = lora.lora_build_segments(ids=torch.from_numpy(ids).cuda(), n_adapters=len(g["ranks"]))
    ws = lora.workspace(table, T)
    x, dY = _bf16(np.tile(g["x"], (repeat, 1))), _bf16(np.tile(g["dY"], (repeat, 1)))
    y = torch.zeros((T, pad), dtype=torch.bfloat16, device="cuda")
    H = torch.full((T, r_max), float("nan"), dtype=torch.float32, device="cuda")
    lora.lora_packed_fwd(y, H, x, table, segs, ws)
    dX = torch.zeros((T, pad), dtype=torch.bfloat16, device="cuda")
    dA = torch.full(g["dA"].shape, float("nan"), dtype=torch.float32, device="cuda")
    dB = torch.full(g["dB"].shape, float("nan"), dtype=torch.float32, device="cuda")
    lora.lora_packed_bwd(dX, dA, dB, dY, x, H, table, segs, ws)
    torch.cuda.synchronize()
    assert lora.lora_query_status(segs) == 0
    host = lambda t: t.float().cpu().numpy().astype(np.float64)
    for name, got, want in (("y", y, np.tile(g["y"], (repeat, 1))), ("H", H, np.tile(g["H"], (repeat, 1))),
                            ("dX", dX, np.tile(g["dX"], (repeat, 1))), ("dA", dA, repeat * g["dA"]),
                            ("dB", dB, repeat * g["dB"])):
        assert np.array_equal(host(got), want), name
