"""The fused base projection + packed LoRA delta (lora_fused_base_fwd) against
the fp64 oracle's layer forward y = x W^T + s_i (x A_i^T) B_i^T.

Small cases span several 256-column blocks, a ragged last column block, a
ragged K (d_in not a multiple of 64), routing tiles cut short at segment ends
and an odd number of routing tiles (a pair with one half); the scale s_i is
large so the delta is as large as the base and cannot hide inside the
tolerance.  W = 0 isolates the delta, B = 0 the base.  At the full packed
size, sampled rows are compared with the oracle run on those rows alone (the
layer is per token)."""
import numpy as np
import pytest
import torch

import adapter_sgmv_gb300 as lora
import oracle
import workloads as wl
from lora_testlib import FWD_TOL, GpuCase, assert_close, bits_to_dev, dev_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lora.build_library()
    lora.lib()


def _spec(name, d_in, d_out, ranks, lengths, alpha_per_rank=64.0, seed=0):
    ids = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lengths)])
    return wl.custom(name, d_in, d_out, ranks, [alpha_per_rank * r for r in ranks], ids, seed=seed)


def _run(case, W, with_H=True):
    s = case.spec
    y = torch.full((s.n_tokens, s.d_out), float("nan"), dtype=torch.bfloat16, device="cuda")
    H = torch.full((s.n_tokens, s.r_max), float("nan"), dtype=torch.float32, device="cuda") if with_H else None
    ws = torch.empty(max(16, lora.lora_fused_base_workspace_bytes(case.table, s.n_tokens)), dtype=torch.uint8,
                     device="cuda")
    lora.lora_fused_base_fwd(y, H, case.inp["x"], W, case.table, case.segs, ws)
    torch.cuda.synchronize()
    assert lora.lora_query_status(case.segs) == 0
    return y, H


def _oracle(spec, h, W_bits):
    P = {k: wl.bf16_bits_to_f64(v) for k, v in h.items()}
    tab = oracle.Table(spec.ranks, spec.scales.astype(np.float64))
    return oracle.base_lora_fwd(tab, spec.ids, wl.bf16_bits_to_f64(W_bits), P["A"], P["B"], P["x"])


CASES = [
    # d_in, d_out, ranks, segment lengths
    (200, 600, [8, 16, 128, 40], [300, 5, 128, 77]),      # ragged K, ragged column block, 6 routing tiles
    (512, 256, [64, 32, 16], [129, 256, 1]),               # one column block, 5 routing tiles (a half-empty pair)
    (320, 1032, [128, 128], [640, 200]),                   # rank 128 on both halves, d_out = 4 x 256 + 8
]


@pytest.mark.parametrize("d_in,d_out,ranks,lengths", CASES)
def test_fused_base_matches_oracle(d_in, d_out, ranks, lengths):
    spec = _spec(f"fb{d_in}x{d_out}", d_in, d_out, ranks, lengths, seed=d_in)
    h = wl.host_inputs(spec)
    Wb = wl.base_weight(spec)
    case = GpuCase(spec, h)
    y, H = _run(case, bits_to_dev(Wb))
    y_ref, H_ref = _oracle(spec, h, Wb)
    assert_close(dev_to_f64(H), H_ref, FWD_TOL, "H")
    assert_close(dev_to_f64(y), y_ref, FWD_TOL, "y")
    # the delta is not negligible against the base in these cases
    base = oracle.base(wl.bf16_bits_to_f64(Wb), wl.bf16_bits_to_f64(h["x"]))
    assert np.max(np.abs(y_ref - base)) > 0.2 * np.max(np.abs(base))


def test_fused_base_zero_weight_is_the_packed_delta_and_zero_B_the_base():
    spec = _spec("fb_parts", 256, 512, [16, 64, 8], [200, 130, 60], alpha_per_rank=2.0, seed=7)
    h = wl.host_inputs(spec)
    case = GpuCase(spec, h)
    y, _ = _run(case, torch.zeros((spec.d_out, spec.d_in), dtype=torch.bfloat16, device="cuda"), with_H=False)
    P = {k: wl.bf16_bits_to_f64(v) for k, v in h.items()}
    tab = oracle.Table(spec.ranks, spec.scales.astype(np.float64))
    y_d, _ = oracle.fwd(tab, spec.ids, P["A"], P["B"], P["x"], np.zeros((spec.n_tokens, spec.d_out)))
    assert_close(dev_to_f64(y), y_d, FWD_TOL, "y (W = 0)")

    h0 = dict(h)
    h0["B"] = np.zeros_like(h["B"])
    case0 = GpuCase(spec, h0)
    Wb = wl.base_weight(spec)
    y0, _ = _run(case0, bits_to_dev(Wb), with_H=False)
    assert_close(dev_to_f64(y0), oracle.base(wl.bf16_bits_to_f64(Wb), P["x"]), FWD_TOL, "y (B = 0)")


def test_fused_base_is_deterministic_and_matches_packed_fwd_H():
    spec = _spec("fb_det", 384, 768, [32, 128, 16, 64], [500, 260, 3, 400], seed=9)
    h = wl.host_inputs(spec)
    case = GpuCase(spec, h)
    W = bits_to_dev(wl.base_weight(spec))
    y1, H1 = _run(case, W)
    y2, H2 = _run(case, W)
    assert torch.equal(y1, y2) and torch.equal(H1, H2)
    # H equals the packed forward's H (the same shrink definition)
    _, H_p = case.fwd()
    assert_close(dev_to_f64(H1), dev_to_f64(H_p), 1e-5, "H vs lora_packed_fwd")


def test_fused_base_full_packed_size_sampled_rows():
    spec = wl.packed4096()
    dev = torch.device("cuda")
    inp = wl.device_inputs(spec, dev, need={"A", "B", "x", "W"})
    case = GpuCase(spec, inp)
    y, H = _run(case, inp["W"])
    rng = np.random.default_rng(5)
    T = spec.n_tokens
    # segment ends and starts, tile boundaries, and random rows
    edges = np.concatenate([spec.seg_offsets[1:-1] - 1, spec.seg_offsets[1:-1], [0, 127, 128, 255, T - 1]])
    rows = np.unique(np.concatenate([edges, rng.integers(0, T, 40)]))
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    x_rows = wl.bf16_bits_to_f64(bits(inp["x"][torch.from_numpy(rows).to(dev)]))
    tab = oracle.Table(spec.ranks, spec.scales.astype(np.float64))
    y_ref, H_ref = oracle.base_lora_fwd(tab, spec.ids[rows], wl.bf16_bits_to_f64(bits(inp["W"])),
                                        wl.bf16_bits_to_f64(bits(inp["A"])), wl.bf16_bits_to_f64(bits(inp["B"])),
                                        x_rows)
    assert_close(dev_to_f64(H)[rows], H_ref, FWD_TOL, "H rows")
    assert_close(dev_to_f64(y)[rows], y_ref, FWD_TOL, "y rows")
    assert torch.isfinite(y.float()).all()


def test_fused_base_rejects_unsorted_batches_and_small_workspace():
    ids = np.array([1, 0, 1, 0, 0, 1] * 20, np.int32)
    spec = wl.custom("fb_unsorted", 64, 64, [8, 16], [16.0, 32.0], ids)
    h = wl.host_inputs(spec)
    case = GpuCase(spec, h, route="ids")
    W = bits_to_dev(wl.base_weight(spec))
    y = torch.empty((spec.n_tokens, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(lora.lora_fused_base_workspace_bytes(case.table, spec.n_tokens), dtype=torch.uint8,
                     device="cuda")
    with pytest.raises(lora.LoraError) as e:
        lora.lora_fused_base_fwd(y, None, case.inp["x"], W, case.table, case.segs, ws)
    assert e.value.status == 6  # LORA_ERR_UNSUPPORTED
    srt = _spec("fb_small_ws", 64, 64, [8], [100])
    c2 = GpuCase(srt, wl.host_inputs(srt))
    with pytest.raises(lora.LoraError) as e:
        lora.lora_fused_base_fwd(torch.empty((100, 64), dtype=torch.bfloat16, device="cuda"), None, c2.inp["x"],
                                 bits_to_dev(wl.base_weight(srt)), c2.table, c2.segs,
                                 torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 5  # LORA_ERR_WORKSPACE_TOO_SMALL
