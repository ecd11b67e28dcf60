"""Several projections that read the same x in one call (lora_multi_fwd):
every projection's y and H against the fp64 oracle, and bit-equal to
lora_packed_fwd run on that projection alone (the same kernels and the same
summation order, only the launches are shared).  Shapes are a Qwen3-4B
layer's decode projections: q / k / v (2560 -> 4096, 1024, 1024) and
gate / up (2560 -> 9728, 9728), with ranks that differ per projection and per
adapter; a batch above the decode size takes the per-projection path."""
import numpy as np
import pytest
import torch

import adapter_sgmv_gb300 as lora
import oracle
import workloads as wl
from lora_testlib import FWD_TOL, assert_close, bits_to_dev, dev_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lora.build_library()
    lora.lib()


def _projection(name, d_out, ranks, ids, d_in=2560, seed=0):
    ranks = np.asarray(ranks, np.int32)
    return wl.custom(name, d_in, d_out, ranks, 2.0 * ranks, ids, seed=seed, with_bwd=False)


def _setup(specs):
    dev = torch.device("cuda")
    x_bits = wl.host_inputs(specs[0])["x"]  # the shared input
    host, tables, y0 = [], [], []
    for s in specs:
        h = wl.host_inputs(s, y0="randn")
        h["x"] = x_bits
        host.append(h)
        tables.append(lora.AdapterTable(bits_to_dev(h["A"]), bits_to_dev(h["B"]), s.ranks.tolist(),
                                        torch.from_numpy(s.scales), s.d_in, s.d_out))
        y0.append(bits_to_dev(h["y0"]))
    s0 = specs[0]
    if s0.sorted:
        segs = lora.lora_build_segments(seg_offsets=torch.from_numpy(s0.seg_offsets).to(dev), n_tokens=s0.n_tokens,
                                        n_adapters=s0.n_adapters, device=dev)
    else:
        segs = lora.lora_build_segments(ids=torch.from_numpy(s0.ids).to(dev), n_adapters=s0.n_adapters, device=dev)
    return bits_to_dev(x_bits), host, tables, y0, segs


def _check(specs):
    x, host, tables, y0, segs = _setup(specs)
    T = specs[0].n_tokens
    ys = [y.clone() for y in y0]
    Hs = [torch.full((T, s.r_max), float("nan"), dtype=torch.float32, device="cuda") for s in specs]
    ws = torch.empty(max(16, lora.lora_multi_workspace_bytes(tables, T)), dtype=torch.uint8, device="cuda")
    lora.lora_multi_fwd(ys, Hs, x, tables, segs, ws)
    torch.cuda.synchronize()
    assert lora.lora_query_status(segs) == 0
    for p, s in enumerate(specs):
        # alone through lora_packed_fwd: the same bits
        y1 = y0[p].clone()
        H1 = torch.full((T, s.r_max), float("nan"), dtype=torch.float32, device="cuda")
        lora.lora_packed_fwd(y1, H1, x, tables[p], segs, lora.workspace(tables[p], T))
        torch.cuda.synchronize()
        assert torch.equal(ys[p], y1) and torch.equal(Hs[p], H1), f"projection {p} differs from lora_packed_fwd"
        # and the oracle
        P = {k: wl.bf16_bits_to_f64(v) for k, v in host[p].items()}
        tab = oracle.Table(s.ranks, s.scales.astype(np.float64))
        y_ref, H_ref = oracle.fwd(tab, s.ids, P["A"], P["B"], P["x"], P["y0"])
        assert_close(dev_to_f64(Hs[p]), H_ref, FWD_TOL, f"H[{p}]")
        assert_close(dev_to_f64(ys[p]), y_ref, FWD_TOL, f"y[{p}]")


def test_attention_projections_q_k_v_decode_batch():
    ids = np.random.default_rng(3).integers(0, 8, 256).astype(np.int32)
    specs = [_projection("q", 4096, [32, 16, 64, 8, 32, 128, 16, 32], ids, seed=1),
             _projection("k", 1024, [16, 16, 32, 8, 16, 64, 8, 16], ids, seed=2),
             _projection("v", 1024, [64, 32, 32, 16, 64, 128, 32, 64], ids, seed=3)]
    _check(specs)


def test_mlp_projections_gate_up_decode_batch():
    ids = np.random.default_rng(4).integers(0, 8, 96).astype(np.int32)
    specs = [_projection("gate", 9728, [32] * 8, ids, seed=4), _projection("up", 9728, [16, 64] * 4, ids, seed=5)]
    _check(specs)


def test_large_batch_takes_the_per_projection_path():
    ids = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate([300, 200, 201])])
    specs = [_projection("q", 1024, [16, 32, 64], ids, d_in=512, seed=6),
             _projection("k", 256, [8, 8, 16], ids, d_in=512, seed=7)]
    _check(specs)


def test_multi_rejects_mismatched_tables():
    ids = np.zeros(16, np.int32)
    a = _projection("a", 256, [8], ids, d_in=256)
    b = _projection("b", 256, [8], ids, d_in=512)
    x, host, tables, y0, segs = _setup([a])
    _, _, tables_b, y0_b, _ = _setup([b])
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(lora.LoraError) as e:
        lora.lora_multi_fwd([y0[0], y0_b[0]], None, x, [tables[0], tables_b[0]], segs, ws)
    assert e.value.status == 2  # LORA_ERR_SHAPE: d_in differs
    with pytest.raises(lora.LoraError) as e:
        lora.lora_multi_fwd([y0[0]] * 9, None, x, [tables[0]] * 9, segs, ws)
    assert e.value.status == 2  # more than LORA_MAX_PROJECTIONS


def test_attention_projections_low_rank():
    # ranks <= 32: the decode buffers sized for a rank-padded 32
    ids = np.random.default_rng(8).integers(0, 8, 256).astype(np.int32)
    specs = [_projection("q", 4096, [32, 16, 8, 32, 24, 32, 16, 8], ids, seed=11),
             _projection("k", 1024, [8, 16, 32, 8, 16, 32, 8, 16], ids, seed=12),
             _projection("v", 1024, [32] * 8, ids, seed=13)]
    _check(specs)
