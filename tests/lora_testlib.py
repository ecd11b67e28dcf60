"""Helpers shared by the GPU tests: move seeded inputs to the device, run the
library through its C ABI, run the fp64 oracle on the same inputs, compare.

Tolerances (fp32 accumulation of bf16 inputs): forward outputs (y, H)
max|err| <= 5e-3 * max|ref|; gradients (dH, dA, dB, dX) <= 1e-2 * max|ref|,
dA / dB checked per adapter block so a small-rank adapter cannot hide behind
a large one."""
from __future__ import annotations

import numpy as np
import torch

import adapter_sgmv_gb300 as lora
import oracle
import workloads as wl

FWD_TOL = 5e-3
GRAD_TOL = 1e-2


def bits_to_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def dev_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    if scale == 0.0:
        return 0.0 if err == 0.0 else float("inf")
    return err / scale


def assert_close(got, ref, tol, what):
    e = rel_err(got, ref)
    assert e <= tol, f"{what}: max|err|/max|ref| = {e:.3e} > {tol:.1e}"
    return e


class GpuCase:
    """A spec's inputs on the device, its adapter table and its segments."""

    def __init__(self, spec: wl.Spec, inputs: dict, device="cuda", route="auto"):
        self.spec = spec
        dev = torch.device(device)
        self.inp = {k: (v if isinstance(v, torch.Tensor) else bits_to_dev(v, dev)) for k, v in inputs.items()}
        self.table = lora.AdapterTable(self.inp["A"], self.inp["B"], spec.ranks.tolist(),
                                       torch.from_numpy(spec.scales), spec.d_in, spec.d_out)
        use_offsets = spec.sorted if route == "auto" else route == "offsets"
        if use_offsets:
            self.segs = lora.lora_build_segments(seg_offsets=torch.from_numpy(spec.seg_offsets).to(dev),
                                                 n_tokens=spec.n_tokens, n_adapters=spec.n_adapters,
                                                 device=dev)
        else:
            self.segs = lora.lora_build_segments(ids=torch.from_numpy(spec.ids).to(dev),
                                                 n_adapters=spec.n_adapters, device=dev)
        self.ws = lora.workspace(self.table, spec.n_tokens, dev)
        self.device = dev

    def fwd(self):
        T, r_max = self.spec.n_tokens, self.spec.r_max
        y = self.inp["y0"].clone()
        H = torch.zeros((T, r_max), dtype=torch.float32, device=self.device)
        lora.lora_packed_fwd(y, H, self.inp["x"], self.table, self.segs, self.ws)
        return y, H

    def bwd(self, H=None, side=None):
        """Packed backward; with ``side`` (lora.SideStreams) the concurrent
        variant, dB and dA on the side streams (the bench's configuration)."""
        s = self.spec
        dX = self.inp["dX0"].clone()
        dA = torch.full((s.sum_r, s.d_in), float("nan"), dtype=torch.float32, device=self.device)
        dB = torch.full((s.sum_r, s.d_out), float("nan"), dtype=torch.float32, device=self.device)
        if side is None:
            lora.lora_packed_bwd(dX, dA, dB, self.inp["dY"], self.inp["x"], H, self.table, self.segs, self.ws)
        else:
            lora.lora_packed_bwd_concurrent(dX, dA, dB, self.inp["dY"], self.inp["x"], H, self.table, self.segs,
                                            self.ws, side)
        return dX, dA, dB

    def dH_workspace(self):
        """dH as left in the workspace by the last backward, in token order
        (implementation detail, for diagnosis): the second hand-off buffer,
        bf16 [T, rw] rows in perm order, of which a row holds its adapter's
        r_i columns (zero up to r_i rounded to 16, unwritten past that)."""
        s = self.spec
        rw = 64 if s.r_max <= 64 else 128
        region = ((s.n_tokens * rw * 2) + 255) & ~255
        dhb = self.ws[region:region + s.n_tokens * rw * 2].view(torch.bfloat16).view(s.n_tokens, rw)
        n_valid = int(self.segs.seg_start[-1].item())
        perm = self.segs.perm[:n_valid].long()
        out = torch.zeros((s.n_tokens, s.r_max), dtype=torch.float32, device=self.device)
        out[perm] = dhb[:n_valid, :s.r_max].float()
        ids = np.asarray(s.ids)
        ok = (ids >= 0) & (ids < s.n_adapters)
        rank = np.where(ok, np.asarray(s.ranks)[np.where(ok, ids, 0)], 0)
        keep = torch.arange(s.r_max, device=self.device)[None, :] < torch.from_numpy(rank).to(self.device)[:, None]
        return torch.where(keep, out, torch.zeros_like(out))


def oracle_all(spec: wl.Spec, host: dict, rows=None):
    """fp64 oracle on the tokens ``rows`` (all when None) of a host-input dict."""
    tab = oracle.Table(spec.ranks, spec.scales.astype(np.float64))
    sel = slice(None) if rows is None else rows
    f = lambda k: wl.bf16_bits_to_f64(host[k]) if host[k].dtype == np.uint16 else host[k]
    ids = spec.ids[sel]
    A, B = f("A"), f("B")
    x, dY, y0, dX0 = f("x")[sel], f("dY")[sel], f("y0")[sel], f("dX0")[sel]
    y, H = oracle.fwd(tab, ids, A, B, x, y0)
    dH, dA, dB, dX = oracle.bwd(tab, ids, A, B, x, H, dY, dX0)
    return dict(y=y, H=H, dH=dH, dA=dA, dB=dB, dX=dX)


def check_blocks(spec, got_dA, got_dB, ref_dA, ref_dB, adapters=None):
    errs = {}
    d_in, d_out = spec.d_in, spec.d_out
    off = spec.row_off
    for i in (range(spec.n_adapters) if adapters is None else adapters):
        a0, a1 = int(off[i]), int(off[i + 1])
        errs[f"dA[{i}]"] = assert_close(got_dA[a0:a1], ref_dA[a0:a1], GRAD_TOL, f"dA_{i}")
        errs[f"dB[{i}]"] = assert_close(got_dB[a0:a1], ref_dB[a0:a1], GRAD_TOL, f"dB_{i}")
    return errs


def worked_example(pad: int = 8) -> dict:
    """The hand-worked two-adapter example of tests/golden/worked_two_adapters.json
    as stacked arrays (A and B_i^T stacked by rank rows, dA / dB likewise), d_in
    and d_out padded to ``pad`` with zero columns.  All values are small
    integers (exact in bf16 / fp32 / fp64)."""
    import json
    import os

    with open(os.path.join(os.path.dirname(__file__), "golden", "worked_two_adapters.json")) as f:
        g = json.load(f)
    ranks = np.asarray(g["ranks"], np.int32)
    T = len(g["ids"])
    sum_r = int(ranks.sum())
    A = np.zeros((sum_r, pad))
    B = np.zeros((sum_r, pad))
    dA = np.zeros((sum_r, pad))
    dB = np.zeros((sum_r, pad))
    row = 0
    for i, r in enumerate(ranks):
        Ai = np.asarray(g["A_i"][str(i)], float)
        Bi = np.asarray(g["B_i (d_out x r_i)"][str(i)], float)
        dBi = np.asarray(g["expected"]["dB_i (d_out x r_i)"][str(i)], float)
        dAi = np.asarray(g["expected"]["dA_i (r_i x d_in)"][str(i)], float)
        A[row:row + r, :Ai.shape[1]] = Ai
        B[row:row + r, :Bi.shape[0]] = Bi.T
        dA[row:row + r, :dAi.shape[1]] = dAi
        dB[row:row + r, :dBi.shape[0]] = dBi.T
        row += r

    def padded(key, width):
        v = np.asarray(key, float)
        out = np.zeros((v.shape[0], width))
        out[:, :v.shape[1]] = v
        return out

    e = g["expected"]
    return {"ranks": ranks, "alphas": np.asarray(g["alphas"], float), "scales": np.asarray(g["scales"], float),
            "ids": np.asarray(g["ids"], np.int32), "A": A, "B": B, "x": padded(g["x"], pad),
            "dY": padded(g["dy"], pad), "T": T, "r_max": int(ranks.max()),
            "H": padded(e["H (T x r_max, zero past r_i)"], int(ranks.max())), "y": padded(e["y (y0 = 0)"], pad),
            "dH": padded(e["dH"], int(ranks.max())), "dX": padded(e["dX (dX0 = 0)"], pad), "dA": dA, "dB": dB}
