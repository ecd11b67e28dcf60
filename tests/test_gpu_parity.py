"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Small cases run the whole oracle; the full-size workloads (the ones the bench
times, in the same launch configuration) are checked on sampled token rows
and on whole adapters for dA / dB."""
import numpy as np
import pytest
import torch

import adapter_sgmv_gb300 as lora
import workloads as wl
from lora_testlib import (FWD_TOL, GRAD_TOL, GpuCase, assert_close, check_blocks, dev_to_f64,
                          oracle_all)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lora.build_library()
    lora.lib()


def full_check(spec, y0="zero", dX0="zero", route="auto", saved_H=True):
    host = wl.host_inputs(spec, y0=y0, dX0=dX0)
    case = GpuCase(spec, host, route=route)
    y, H = case.fwd()
    dX, dA, dB = case.bwd(H if saved_H else None)
    torch.cuda.synchronize()
    assert lora.lora_query_status(case.segs) == 0
    ref = oracle_all(spec, host)
    valid = (spec.ids >= 0) & (spec.ids < spec.n_adapters)
    e = {}
    e["y"] = assert_close(dev_to_f64(y)[valid], ref["y"][valid], FWD_TOL, "y")
    e["H"] = assert_close(dev_to_f64(H)[valid], ref["H"][valid], FWD_TOL, "H")
    e["dH"] = assert_close(dev_to_f64(case.dH_workspace())[valid], ref["dH"][valid], GRAD_TOL, "dH")
    e["dX"] = assert_close(dev_to_f64(dX)[valid], ref["dX"][valid], GRAD_TOL, "dX")
    e.update(check_blocks(spec, dev_to_f64(dA), dev_to_f64(dB), ref["dA"], ref["dB"]))
    return e


def test_tiny_config_sorted_offsets():
    full_check(wl.tiny())


def test_tiny_config_routed_by_ids():
    full_check(wl.tiny(), route="ids")


def test_tiny_config_accumulates_into_nonzero_outputs():
    full_check(wl.tiny(), y0="randn", dX0="randn")


def test_tiny_config_recomputes_H_when_not_saved():
    full_check(wl.tiny(), saved_H=False)


@pytest.mark.parametrize("seed", [0, 1])
def test_ragged_unsorted_mixed_ranks(seed):
    rng = np.random.default_rng(100 + seed)
    T, N = 333, 6
    ranks = [4, 8, 16, 24, 64, 128]
    ids = rng.integers(0, N, T).astype(np.int32)
    spec = wl.custom("ragged", 136, 200, ranks, [2.0 * r for r in ranks], ids, seed=seed)
    full_check(spec, y0="randn", dX0="randn")


def test_long_segments_several_tiles_with_ragged_tail():
    ranks = [16, 32, 128]
    lengths = [300, 128, 517]
    ids = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lengths)])
    spec = wl.custom("long", 512, 384, ranks, [32.0, 32.0, 32.0], ids)
    full_check(spec)


@pytest.mark.parametrize("route", ["auto", "ids"])
def test_wide_projection_sorted_three_thousand_tokens(route):
    # d_in and d_out above 2048, so case ii works through whole 1024-column
    # items and a ragged last one (d_out = 3080 also ends 8 columns into a
    # 64-column block); sorted, the case ii epilogue runs on eight warps, by
    # ids on four; full tiles, ragged tails and a rank below 16
    ranks = [16, 64, 128, 8, 32]
    lengths = [700, 1100, 512, 300, 388]
    ids = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lengths)])
    spec = wl.custom("wide", 2112, 3080, ranks, [2.0 * r for r in ranks], ids)
    full_check(spec, route=route)


def test_two_ctas_per_sm_shapes_ragged():
    # A sorted batch sized so that, on 152 SMs, case i has 1.5+ tiles per SM
    # (three-stage ring, two CTAs per SM) and cases iii/iv 1.5 to 3 items per
    # SM (two CTAs per SM, 256-column items): 45 adapters, T = 30720, d_in and
    # d_out ending 8 columns into their last 256-column range (and into a
    # 64-column block, so the activations come by 2-D boxes); an empty
    # adapter, one of a single token, one of three spans, ranks 8..128 with
    # 24 and 40 among them
    rng = np.random.default_rng(31)
    n = 45
    ranks = [[8, 16, 24, 32, 40, 64, 128, 16, 8][i % 9] for i in range(n)]
    lengths = rng.integers(300, 1000, n)
    lengths[3], lengths[7], lengths[11], lengths[20] = 0, 1, 2500, 129
    lengths[-1] += 30720 - lengths.sum()
    ids = np.concatenate([np.full(m, i, np.int32) for i, m in enumerate(lengths)])
    spec = wl.custom("two_cta", 1032, 1288, ranks, [2.0 * r for r in ranks], ids)
    full_check(spec)


def test_zipf_runs_unsorted_small():
    rng = np.random.default_rng(8)
    runs = []
    total = 0
    while total < 1500:
        n = int(min(rng.zipf(1.2), 300))
        runs.append((min(n, 1500 - total), int(rng.integers(0, 8))))
        total += runs[-1][0]
    ids = np.concatenate([np.full(n, a, np.int32) for n, a in runs])
    ranks = [8, 16, 32, 64, 128, 8, 16, 32]
    spec = wl.custom("zipf", 256, 448, ranks, [2.0 * r for r in ranks], ids)
    full_check(spec)


@pytest.mark.parametrize("route", ["auto", "ids"])
def test_five_thousand_adapters_sorted(route):
    # more adapters than the one-launch routing build holds (4095): sorted
    # offsets take the build that scans in global memory, ids the counting
    # sort; a quarter of the adapters empty, one spanning several tiles
    rng = np.random.default_rng(11)
    N = 5000
    lens = rng.integers(0, 4, N)
    lens[rng.random(N) < 0.25] = 0
    lens[17] = 700
    ids = np.repeat(np.arange(N, dtype=np.int32), lens)
    ranks = rng.choice(np.array([1, 4, 8, 16, 40]), size=N).astype(np.int32)
    spec = wl.custom("many", 64, 72, ranks, 2.0 * ranks, ids, seed=3)
    full_check(spec, y0="randn", dX0="randn", route=route)


def test_empty_adapters_get_zero_gradients():
    ids = np.array([0] * 40 + [3] * 70, np.int32)  # adapters 1 and 2 have no token
    spec = wl.custom("empty", 64, 96, [8, 16, 32, 16], [16.0] * 4, ids)
    full_check(spec)


def test_bad_ids_report_status_and_leave_rows_untouched():
    ids = np.array([0, 1, 9, 1, -1, 0, 1, 2], np.int32)
    spec = wl.custom("bad", 64, 64, [8, 16, 8], [16.0] * 3, ids)
    host = wl.host_inputs(spec, y0="randn", dX0="randn")
    case = GpuCase(spec, host, route="ids")
    y, H = case.fwd()
    dX, dA, dB = case.bwd(H)
    assert lora.lora_query_status(case.segs) == 4
    y0, dX0 = dev_to_f64(case.inp["y0"]), dev_to_f64(case.inp["dX0"])
    for t in (2, 4):
        assert np.array_equal(dev_to_f64(y)[t], y0[t])
        assert np.array_equal(dev_to_f64(dX)[t], dX0[t])
    ref = oracle_all(spec, host)
    ok = np.array([0, 1, 3, 5, 6, 7])
    assert_close(dev_to_f64(y)[ok], ref["y"][ok], FWD_TOL, "y")
    check_blocks(spec, dev_to_f64(dA), dev_to_f64(dB), ref["dA"], ref["dB"])


def test_optional_outputs_can_be_skipped():
    spec = wl.tiny()
    host = wl.host_inputs(spec)
    case = GpuCase(spec, host)
    y, H = case.fwd()
    dA = torch.zeros((spec.sum_r, spec.d_in), device="cuda")
    lora.lora_packed_bwd(None, dA, None, case.inp["dY"], case.inp["x"], H, case.table, case.segs, case.ws)
    ref = oracle_all(spec, host)
    assert_close(dev_to_f64(dA), ref["dA"], GRAD_TOL, "dA")


def test_decode_path_full_tiles_rank_128_ragged_edges():
    # T = 512 still takes the decode kernels: 128-row tiles at rank 128, a d_in
    # whose last slice ends 8 columns into a k16 step, a d_out with an 8-column tail
    ranks = [128, 64, 8]
    lengths = [300, 150, 62]
    rng = np.random.default_rng(5)
    ids = rng.permutation(np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lengths)]))
    spec = wl.custom("decode_edges", 4104, 776, ranks, [2.0 * r for r in ranks], ids)
    full_check(spec, y0="randn")


@pytest.mark.parametrize("route", ["ids", "auto"])
def test_decode_path_ragged_edges(route):
    # a decode-size batch (T <= 512): an adapter spanning two tiles, ragged
    # tiles, ranks 1 and 33 (padding to 16 and 48), d_in = 3000 (slices of 256,
    # the last 184 wide) and d_out = 1000 (four 256-column expand slices, the
    # last 232 wide)
    ranks = [64, 48, 8, 1, 33]
    lengths = [200, 150, 100, 40, 10]
    rng = np.random.default_rng(9)
    ids = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lengths)])
    if route == "ids":
        ids = rng.permutation(ids)
    spec = wl.custom("decode_edges2", 3000, 1000, ranks, [2.0 * r for r in ranks], ids)
    full_check(spec, y0="zero")
    host = wl.host_inputs(spec, y0="randn")
    case = GpuCase(spec, host)
    y1, H1 = case.fwd()
    y2, H2 = case.fwd()
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(H1, H2)
    ref = oracle_all(spec, host)
    assert_close(dev_to_f64(y1), ref["y"], FWD_TOL, "y (accumulated)")


@pytest.mark.parametrize("proj", [0, 1, 2])
def test_decode_batch_shrink_expand(proj):
    spec = wl.decode(proj)
    host = wl.host_inputs(spec, y0="zero")
    case = GpuCase(spec, host)
    T = spec.n_tokens
    H = torch.zeros((T, spec.r_max), dtype=torch.float32, device="cuda")
    lora.lora_sgmv_shrink(H, case.inp["x"], case.table, case.segs)
    y = case.inp["y0"].clone()
    lora.lora_sgmv_expand(y, H, case.table, case.segs)
    y2, H2 = case.fwd()
    torch.cuda.synchronize()
    ref = oracle_all(spec, host)
    assert_close(dev_to_f64(H), ref["H"], FWD_TOL, "H")
    assert_close(dev_to_f64(y), ref["y"], FWD_TOL, "y")
    assert_close(dev_to_f64(y2), ref["y"], FWD_TOL, "y(packed_fwd)")
    assert_close(dev_to_f64(H2), ref["H"], FWD_TOL, "H(packed_fwd)")


def test_repeated_runs_are_identical():
    spec = wl.tiny()
    host = wl.host_inputs(spec)
    case = GpuCase(spec, host)
    y1, H1 = case.fwd()
    y2, H2 = case.fwd()
    assert torch.equal(y1, y2) and torch.equal(H1, H2)


# ---------------------------------------------------------------------------- full size
def sampled_rows(spec, rng, per_adapter=3):
    rows = set()
    seg = np.flatnonzero(np.r_[True, np.diff(spec.ids) != 0])
    ends = np.r_[seg[1:], spec.n_tokens] - 1
    for a, b in list(zip(seg, ends))[:: max(1, len(seg) // 24)]:
        rows.update([int(a), int(b)])
    for i in range(spec.n_adapters):
        idx = np.flatnonzero(spec.ids == i)
        if idx.size:
            rows.update(int(v) for v in rng.choice(idx, size=min(per_adapter, idx.size), replace=False))
    rows.update([0, spec.n_tokens - 1])
    return np.array(sorted(rows))


def host_rows(dev, rows):
    return dev[torch.from_numpy(rows).to(dev.device)].float().cpu().numpy().astype(np.float64)


FULL = {
    "packed4096": lambda: wl.packed4096(),
    "sweep2": lambda: wl.sweep(2),
    "sweep32": lambda: wl.sweep(32),
    "skewed": lambda: wl.skewed(),
}


def adapter_rows(spec, i):
    return np.flatnonzero(spec.ids == i)


@pytest.mark.parametrize("name", sorted(FULL))
def test_full_size_pure_delta_every_adapter(name):
    """The workloads the bench times, at full size and in its launch
    configuration, with y0 = dX0 = 0 so that the tolerance binds the delta
    itself: for every adapter, all of its tokens' rows of y, H, dH and dX and
    its dA_i / dB_i blocks against the oracle run on that adapter's tokens."""
    spec = FULL[name]()
    dev = torch.device("cuda")
    inp = wl.device_inputs(spec, dev, y0="zero", dX0="zero")
    case = GpuCase(spec, inp)
    y, H = case.fwd()
    dX, dA, dB = case.bwd(H, side=lora.SideStreams())  # as the bench runs it
    torch.cuda.synchronize()
    assert lora.lora_query_status(case.segs) == 0
    dH = case.dH_workspace()
    A, B = dev_to_f64(inp["A"]), dev_to_f64(inp["B"])
    dA_h, dB_h = dev_to_f64(dA), dev_to_f64(dB)
    checked = 0
    for i in range(spec.n_adapters):
        toks = adapter_rows(spec, i)
        if toks.size == 0:
            continue
        host_i = {"A": A, "B": B, "x": host_rows(inp["x"], toks), "dY": host_rows(inp["dY"], toks),
                  "y0": np.zeros((toks.size, spec.d_out)), "dX0": np.zeros((toks.size, spec.d_in))}
        sub = wl.custom(spec.name, spec.d_in, spec.d_out, spec.ranks, spec.alphas, spec.ids[toks], sorted_=False)
        ref = oracle_all(sub, host_i)
        assert_close(host_rows(y, toks), ref["y"], FWD_TOL, f"y (adapter {i})")
        assert_close(H[torch.from_numpy(toks).cuda()].cpu().numpy(), ref["H"], FWD_TOL, f"H (adapter {i})")
        assert_close(host_rows(dH, toks), ref["dH"], GRAD_TOL, f"dH (adapter {i})")
        assert_close(host_rows(dX, toks), ref["dX"], GRAD_TOL, f"dX (adapter {i})")
        check_blocks(spec, dA_h, dB_h, ref["dA"], ref["dB"], adapters=[i])
        checked += 1
    # adapters without tokens get zero gradients
    for i in range(spec.n_adapters):
        if adapter_rows(spec, i).size == 0:
            a0, a1 = int(spec.row_off[i]), int(spec.row_off[i + 1])
            assert not dA_h[a0:a1].any() and not dB_h[a0:a1].any()
    assert checked > 0


def test_full_size_accumulates_into_nonzero_outputs():
    """Accumulation semantics at full size (y += delta, dX += delta on
    unit-variance y0 / dX0), on sampled rows of the packed training batch."""
    spec = FULL["packed4096"]()
    dev = torch.device("cuda")
    inp = wl.device_inputs(spec, dev, y0="randn", dX0="randn")
    case = GpuCase(spec, inp)
    y, H = case.fwd()
    dX, dA, dB = case.bwd(H)
    torch.cuda.synchronize()
    assert lora.lora_query_status(case.segs) == 0
    rng = np.random.default_rng(0)
    rows = sampled_rows(spec, rng)
    host = {"A": dev_to_f64(inp["A"]), "B": dev_to_f64(inp["B"]),
            "x": host_rows(inp["x"], rows), "dY": host_rows(inp["dY"], rows),
            "y0": host_rows(inp["y0"], rows), "dX0": host_rows(inp["dX0"], rows)}
    sub = wl.custom(spec.name, spec.d_in, spec.d_out, spec.ranks, spec.alphas, spec.ids[rows], sorted_=False)
    ref = oracle_all(sub, host)
    assert_close(host_rows(y, rows), ref["y"], FWD_TOL, "y")
    assert_close(host_rows(dX, rows), ref["dX"], GRAD_TOL, "dX")
