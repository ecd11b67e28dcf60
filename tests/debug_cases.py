"""Cases for the library's debug build (device-side index checks), run as a
child process with LORA_SGMV_LIB pointing at liblora_sgmv_debug.so:

    python tests/debug_cases.py OUT_DIR

Every call the path has (routing from offsets and from ids, the decode
forward, the packed forward with and without the split along d, the packed
backward serial / ordered / with side streams, the fused base layer, the
multi-projection decode) runs on small ragged batches; the outputs go to
OUT_DIR/<case>.npz with the status word and the check site after each case.
The parent test runs the same cases on the release build and compares.

Then three batches whose perm holds one token index past T (a corruption the
builder never makes) run through the debug build's decode and packed paths (split and not);
their x / y / H / dY / dX buffers carry 64 spare rows, so even an unchecked
read or write of that row would stay inside its buffer.  The checks must
report LORA_ERR_INDEX and where."""
from __future__ import annotations

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def specs():
    import workloads as wl

    out = {"tiny": wl.tiny()}
    # sorted: five adapters, one empty and one of a single token; adapter 0
    # spans three LORA_SPAN_TOKENS spans (the ordered backward's tickets); 27
    # routing tiles, so case i is cut along d_in (two parts)
    lengths, ranks = [2300, 700, 1, 129, 0], [16, 64, 128, 8, 32]
    ids = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lengths)])
    alphas = [2.0 * r for r in ranks]
    out["ragged_sorted"] = wl.custom("ragged_sorted", 1032, 520, ranks, alphas, ids)
    out["ragged_ids"] = wl.custom("ragged_ids", 1032, 520, ranks, alphas,
                                  np.random.default_rng(11).permutation(ids), sorted_=False)
    # enough tiles (87) that case i is not split along d
    lengths2, ranks2 = [4000, 3000, 1500, 1, 1739, 0], [32, 128, 16, 64, 8, 16]
    ids2 = np.concatenate([np.full(n, i, np.int32) for i, n in enumerate(lengths2)])
    alphas2 = [2.0 * r for r in ranks2]
    out["many_tiles_sorted"] = wl.custom("many_tiles_sorted", 256, 392, ranks2, alphas2, ids2)
    out["many_tiles_ids"] = wl.custom("many_tiles_ids", 256, 392, ranks2, alphas2,
                                      np.random.default_rng(13).permutation(ids2), sorted_=False)
    # decode-sized, unsorted (the decode kernels)
    dec_ranks = [16, 32, 8, 128, 24]
    out["decode_ids"] = wl.custom("decode_ids", 264, 392, dec_ranks, [2.0 * r for r in dec_ranks],
                                  np.random.default_rng(12).integers(0, 5, size=37).astype(np.int32), sorted_=False)
    return out


def run_case(spec, host):
    """Every entry point on one batch; returns named outputs as numpy arrays."""
    import torch

    import adapter_sgmv_gb300 as lora
    from lora_testlib import GpuCase

    case = GpuCase(spec, host)
    res = {}
    y, H = case.fwd()
    res["y"], res["H"] = y, H
    # backward: serial (H saved), ordered with side streams, ordered with H recomputed
    dX, dA, dB = case.bwd(H)
    res["dX"] = dX
    side = lora.SideStreams()
    for tag, h, sd in (("ord", H, side), ("ord_recompute", None, None)):
        dX2 = case.inp["dX0"].clone()
        dA2 = torch.full((spec.sum_r, spec.d_in), float("nan"), dtype=torch.float32, device="cuda")
        dB2 = torch.full((spec.sum_r, spec.d_out), float("nan"), dtype=torch.float32, device="cuda")
        lora.lora_packed_bwd_ex(dX2, dA2, dB2, case.inp["dY"], case.inp["x"], h, case.table, case.segs, case.ws,
                                side=sd, deterministic=True)
        res[f"dX_{tag}"], res[f"dA_{tag}"], res[f"dB_{tag}"] = dX2, dA2, dB2
    torch.cuda.synchronize()
    del side
    # the fused base layer (segment-sorted batches only)
    if spec.sorted:
        g = torch.Generator(device="cuda").manual_seed(5)
        W = (torch.randn((spec.d_out, spec.d_in), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
        yb = torch.full((spec.n_tokens, spec.d_out), float("nan"), dtype=torch.bfloat16, device="cuda")
        Hb = torch.full((spec.n_tokens, spec.r_max), float("nan"), dtype=torch.float32, device="cuda")
        wsb = torch.empty(max(16, lora.lora_fused_base_workspace_bytes(case.table, spec.n_tokens)),
                          dtype=torch.uint8, device="cuda")
        lora.lora_fused_base_fwd(yb, Hb, case.inp["x"], W, case.table, case.segs, wsb)
        res["W"], res["y_base"], res["H_base"] = W, yb, Hb
    # two projections sharing x in one call (decode kernels for <= 512 tokens)
    B2 = case.inp["B"].flip(1).contiguous()
    t2 = lora.AdapterTable(case.inp["A"], B2, spec.ranks.tolist(), torch.from_numpy(spec.scales), spec.d_in,
                           spec.d_out)
    ys = [torch.zeros((spec.n_tokens, spec.d_out), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    Hs = [torch.zeros((spec.n_tokens, spec.r_max), dtype=torch.float32, device="cuda") for _ in range(2)]
    wsm = torch.empty(max(16, lora.lora_multi_workspace_bytes([case.table, t2], spec.n_tokens)), dtype=torch.uint8,
                      device="cuda")
    lora.lora_multi_fwd(ys, Hs, case.inp["x"], [case.table, t2], case.segs, wsm)
    res["y_multi0"], res["y_multi1"], res["H_multi1"] = ys[0], ys[1], Hs[1]
    torch.cuda.synchronize()
    st, where = lora.lora_query_index_check(case.segs)
    out = {}
    for k, v in res.items():
        v = v.detach()
        out[k] = v.view(torch.int16).cpu().numpy() if v.dtype == torch.bfloat16 else v.cpu().numpy()
    return out, st, where


def run_corrupted(spec, host):
    """perm[k] = T + 5 for one k inside a tile; forward and backward through
    the debug build.  Returns (status, where) after each."""
    import torch

    import adapter_sgmv_gb300 as lora
    from lora_testlib import GpuCase

    T, pad = spec.n_tokens, 64
    case = GpuCase(spec, host)

    def padded(t):  # the same rows plus `pad` spare rows past T
        p = torch.zeros((T + pad,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        p[:T] = t
        return p

    x, dY = padded(case.inp["x"]), padded(case.inp["dY"])
    y = padded(case.inp["y0"])
    dX = padded(case.inp["dX0"])
    H = torch.zeros((T + pad, spec.r_max), dtype=torch.float32, device="cuda")
    k = int(case.segs.seg_start[1].item()) + 3  # the fourth token of adapter 1's group
    case.segs.perm[k] = T + 5
    torch.cuda.synchronize()
    out = {}
    lora.lora_packed_fwd(y, H, x, case.table, case.segs, case.ws)
    out["fwd"] = lora.lora_query_index_check(case.segs)
    lora.lora_reset_status(case.segs)
    dA = torch.zeros((spec.sum_r, spec.d_in), dtype=torch.float32, device="cuda")
    dB = torch.zeros((spec.sum_r, spec.d_out), dtype=torch.float32, device="cuda")
    lora.lora_packed_bwd(dX, dA, dB, dY, x, H, case.table, case.segs, case.ws)
    out["bwd"] = lora.lora_query_index_check(case.segs)
    return out


def main(out_dir):
    sys.path[:0] = [ROOT, HERE]
    import torch

    import adapter_sgmv_gb300 as lora
    import workloads as wl

    assert lora.lora_debug_checks(), "the debug build is not the library loaded"
    summary = {"debug_checks": True, "cases": {}, "corrupted": {}}
    for name, spec in specs().items():
        host = wl.host_inputs(spec)
        out, st, where = run_case(spec, host)
        np.savez(os.path.join(out_dir, f"{name}.npz"), **out)
        summary["cases"][name] = {"status": st, "where": where}
    for name in ("decode_ids", "ragged_ids", "many_tiles_ids"):
        spec = specs()[name]
        summary["corrupted"][name] = run_corrupted(spec, wl.host_inputs(spec))
    torch.cuda.synchronize()
    with open(os.path.join(out_dir, "summary.json"), "w") as f:
        json.dump(summary, f)


if __name__ == "__main__":
    main(sys.argv[1])
