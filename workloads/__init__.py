"""Seeded synthetic inputs for the multi-adapter LoRA delta.

This module only draws random numbers and rounds them to bf16; it holds none
of the LoRA arithmetic.  Both the CUDA path (tests, bench) and the fp64
oracle read the inputs it produces, which is the only thing they share.

The five workloads follow the shapes of the pages' model families: Qwen3-4B
projections for the decode batch (C-LoRA report, "I numeri sul campo"),
Qwen-2.5 / LLaMA-3 projections for the packed training batches (PLoRA
technical summary, "Resultaten"), with per-adapter rank and scaling factor
varying as in PLoRA's search space.  None of them needs a dataset or trained
weights: the delta is a linear map, so only shapes and value ranges matter.

Value recipe (every tensor bf16, rounded to nearest-even from fp32):
  x, dY, y0, dX0 ~ N(0, 1); A_i ~ U(-1/sqrt(d_in), +1/sqrt(d_in)); B_i ~ N(0, 0.02^2);
  the frozen base weight W [d_out, d_in] ~ U(-1/sqrt(d_in), +1/sqrt(d_in)).
Layouts: A [sum_r, d_in] (A_i stacked); B [sum_r, d_out] (B_i transposed,
stacked the same way: row row_off[i] + k is column k of B_i).
Each tensor draws from its own stream, numpy ``default_rng([seed, k])`` on
the host or a ``torch.Generator`` seeded ``seed * 1000 + k`` on a device.
"""
from __future__ import annotations

import dataclasses
import json
import math
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SKEWED_FIXTURE = os.path.join(_HERE, "skewed_seed0.json")

# stream indices, one per tensor
_S_A, _S_B, _S_X, _S_DY, _S_Y0, _S_DX0, _S_W = 1, 2, 3, 4, 5, 6, 7


# ----------------------------------------------------------------------------
# bf16 <-> fp32 bit conversions (round to nearest, ties to even)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    out = ((u + (((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF))) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(b) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


# ----------------------------------------------------------------------------
# problem specifications (cheap: ranks, scales, routing)
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Spec:
    name: str
    d_in: int
    d_out: int
    ranks: np.ndarray          # int32 [N]
    alphas: np.ndarray         # float64 [N]
    ids: np.ndarray            # int32 [T], adapter of every token
    sorted: bool               # tokens already grouped by adapter, ascending
    seed: int = 0
    with_bwd: bool = True

    @property
    def n_tokens(self) -> int:
        return int(self.ids.shape[0])

    @property
    def n_adapters(self) -> int:
        return int(self.ranks.shape[0])

    @property
    def scales(self) -> np.ndarray:
        """s_i = alpha_i / r_i, formed in fp64 and rounded once to fp32."""
        return (self.alphas / self.ranks.astype(np.float64)).astype(np.float32)

    @property
    def row_off(self) -> np.ndarray:
        off = np.zeros(self.n_adapters + 1, dtype=np.int64)
        off[1:] = np.cumsum(self.ranks, dtype=np.int64)
        return off

    @property
    def sum_r(self) -> int:
        return int(self.ranks.sum())

    @property
    def r_max(self) -> int:
        return int(self.ranks.max())

    @property
    def seg_offsets(self) -> np.ndarray | None:
        """[N+1] group offsets when tokens are sorted by adapter, else None."""
        if not self.sorted:
            return None
        counts = np.bincount(self.ids, minlength=self.n_adapters)
        off = np.zeros(self.n_adapters + 1, dtype=np.int32)
        off[1:] = np.cumsum(counts)
        return off

    def runs(self):
        """(start, length, adapter) of maximal runs of equal ids, in token order."""
        ids = self.ids
        if ids.size == 0:
            return []
        cut = np.flatnonzero(np.diff(ids)) + 1
        starts = np.concatenate([[0], cut])
        ends = np.concatenate([cut, [ids.size]])
        return [(int(s), int(e - s), int(ids[s])) for s, e in zip(starts, ends)]


def _sorted_ids(lengths) -> np.ndarray:
    return np.concatenate([np.full(int(n), i, dtype=np.int32) for i, n in enumerate(lengths)])


def tiny(seed: int = 0) -> Spec:
    """N=4, ranks {4,8,8,16}, alpha=2r, d_in=d_out=256, T=64 in sorted segments {8,16,24,16}."""
    ranks = np.array([4, 8, 8, 16], dtype=np.int32)
    return Spec("tiny", 256, 256, ranks, 2.0 * ranks, _sorted_ids([8, 16, 24, 16]), True, seed)


DECODE_PROJECTIONS = ((2560, 4096), (2560, 9728), (9728, 2560))


def decode(proj: int = 0, seed: int = 0, n_tokens: int = 256) -> Spec:
    """Decode batch: one token per request, adapter id uniform over 8 (unsorted), r=32, alpha=64."""
    d_in, d_out = DECODE_PROJECTIONS[proj]
    rng = np.random.default_rng([seed, 0])
    ids = rng.integers(0, 8, size=n_tokens).astype(np.int32)
    ranks = np.full(8, 32, dtype=np.int32)
    return Spec(f"decode{d_in}x{d_out}", d_in, d_out, ranks, np.full(8, 64.0), ids, False, seed, False)


def packed4096(seed: int = 0, tokens_per_adapter: int = 4096) -> Spec:
    """4096->4096, N=8, ranks {8,16,16,32,32,64,64,128}, alpha 16 (even i) / 32 (odd i), sorted."""
    ranks = np.array([8, 16, 16, 32, 32, 64, 64, 128], dtype=np.int32)
    alphas = np.array([16.0 if i % 2 == 0 else 32.0 for i in range(8)])
    return Spec("packed4096", 4096, 4096, ranks, alphas, _sorted_ids([tokens_per_adapter] * 8), True, seed)


def sweep(n_adapters: int, seed: int = 0, tokens_per_adapter: int = 2048) -> Spec:
    """3584->18944, rank 16, alpha 32, N adapters of 2048 tokens each, sorted."""
    ranks = np.full(n_adapters, 16, dtype=np.int32)
    return Spec(f"sweep{n_adapters}", 3584, 18944, ranks, np.full(n_adapters, 32.0),
                _sorted_ids([tokens_per_adapter] * n_adapters), True, seed)


def draw_skewed(seed: int = 0, n_tokens: int = 16384, n_adapters: int = 32, cap: int = 1024):
    """Ranks uniform over {8..128} powers of two, then Zipf(1.2) run lengths
    (values above ``cap`` redrawn), each run's adapter uniform; runs appended
    in draw order until ``n_tokens`` (the last one clipped)."""
    rng = np.random.default_rng(seed)
    ranks = rng.choice(np.array([8, 16, 32, 64, 128]), size=n_adapters).astype(np.int32)
    runs = []
    total = 0
    while total < n_tokens:
        n = int(rng.zipf(1.2))
        while n > cap:
            n = int(rng.zipf(1.2))
        a = int(rng.integers(0, n_adapters))
        n = min(n, n_tokens - total)
        runs.append((n, a))
        total += n
    return ranks, runs


def write_skewed_fixture(path: str = SKEWED_FIXTURE, seed: int = 0) -> None:
    ranks, runs = draw_skewed(seed)
    with open(path, "w") as f:
        json.dump({"seed": seed, "n_tokens": 16384, "ranks": [int(r) for r in ranks],
                   "runs": [[int(n), int(a)] for n, a in runs]}, f)
        f.write("\n")


def skewed(seed: int = 0) -> Spec:
    """4096->14336, N=32, T=16384 in Zipf(1.2) runs (unsorted ids), alpha=2r.
    The seed-0 draw is read from a committed fixture so that it does not
    depend on the numpy version."""
    if seed == 0 and os.path.exists(SKEWED_FIXTURE):
        with open(SKEWED_FIXTURE) as f:
            fx = json.load(f)
        ranks = np.array(fx["ranks"], dtype=np.int32)
        runs = [(int(n), int(a)) for n, a in fx["runs"]]
    else:
        ranks, runs = draw_skewed(seed)
    ids = np.concatenate([np.full(n, a, dtype=np.int32) for n, a in runs])
    return Spec("skewed", 4096, 14336, ranks, 2.0 * ranks, ids, False, seed)


def custom(name, d_in, d_out, ranks, alphas, ids, seed=0, sorted_=None, with_bwd=True) -> Spec:
    ids = np.asarray(ids, dtype=np.int32)
    if sorted_ is None:
        sorted_ = bool(ids.size == 0 or np.all(np.diff(ids) >= 0))
    return Spec(name, int(d_in), int(d_out), np.asarray(ranks, dtype=np.int32),
                np.asarray(alphas, dtype=np.float64), ids, sorted_, seed, with_bwd)


def random_spec(rng, T, N, d_in, d_out, rank_choices=(8, 16, 32), sorted_=False, name="random") -> Spec:
    ranks = rng.choice(np.asarray(rank_choices), size=N).astype(np.int32)
    alphas = rng.choice(np.array([8.0, 16.0, 32.0]), size=N)
    ids = rng.integers(0, N, size=T).astype(np.int32)
    if sorted_:
        ids = np.sort(ids)
    return custom(name, d_in, d_out, ranks, alphas, ids, sorted_=sorted_)


# ----------------------------------------------------------------------------
# materialisation
# ----------------------------------------------------------------------------
def host_inputs(spec: Spec, y0: str = "zero", dX0: str = "zero") -> dict:
    """bf16 bit arrays (uint16) drawn on the host with numpy.

    Keys: A [sum_r, d_in], B [sum_r, d_out] (B_i transposed, stacked like A),
    x [T, d_in], dY [T, d_out], y0 [T, d_out], dX0 [T, d_in].
    ``y0`` / ``dX0`` are "zero" or "randn"."""
    T, d_in, d_out, sr, s = spec.n_tokens, spec.d_in, spec.d_out, spec.sum_r, spec.seed

    def rng(k):
        return np.random.default_rng([s, k])

    lim = 1.0 / math.sqrt(d_in)
    out = {
        "A": f32_to_bf16_bits(rng(_S_A).uniform(-lim, lim, size=(sr, d_in)).astype(np.float32)),
        "B": f32_to_bf16_bits(rng(_S_B).normal(0.0, 0.02, size=(sr, d_out)).astype(np.float32)),
        "x": f32_to_bf16_bits(rng(_S_X).standard_normal(size=(T, d_in), dtype=np.float32)),
    }
    out["dY"] = f32_to_bf16_bits(rng(_S_DY).standard_normal(size=(T, d_out), dtype=np.float32))
    if y0 == "randn":
        out["y0"] = f32_to_bf16_bits(rng(_S_Y0).standard_normal(size=(T, d_out), dtype=np.float32))
    else:
        out["y0"] = np.zeros((T, d_out), dtype=np.uint16)
    if dX0 == "randn":
        out["dX0"] = f32_to_bf16_bits(rng(_S_DX0).standard_normal(size=(T, d_in), dtype=np.float32))
    else:
        out["dX0"] = np.zeros((T, d_in), dtype=np.uint16)
    return out


def base_weight(spec: Spec) -> np.ndarray:
    """bf16 bits of the frozen base weight W [d_out, d_in] (row-major, the
    layout of a linear layer's weight), drawn on the host."""
    lim = 1.0 / math.sqrt(spec.d_in)
    g = np.random.default_rng([spec.seed, _S_W])
    return f32_to_bf16_bits(g.uniform(-lim, lim, size=(spec.d_out, spec.d_in)).astype(np.float32))


def device_inputs(spec: Spec, device, y0: str = "zero", dX0: str = "zero", need=None) -> dict:
    """The same recipe drawn on a torch device (bf16 tensors), for sizes too
    large to draw on the host.  ``need`` restricts the keys produced; the
    base weight "W" is produced only when asked for."""
    import torch

    T, d_in, d_out, sr, s = spec.n_tokens, spec.d_in, spec.d_out, spec.sum_r, spec.seed
    keys = set(need) if need is not None else {"A", "B", "x", "dY", "y0", "dX0"}

    def gen(k):
        g = torch.Generator(device=device)
        g.manual_seed(s * 1000 + k)
        return g

    out = {}
    lim = 1.0 / math.sqrt(d_in)
    if "A" in keys:
        a = torch.rand((sr, d_in), generator=gen(_S_A), device=device, dtype=torch.float32)
        out["A"] = (a * (2 * lim) - lim).to(torch.bfloat16)
    if "B" in keys:
        out["B"] = (torch.randn((sr, d_out), generator=gen(_S_B), device=device) * 0.02).to(torch.bfloat16)
    if "x" in keys:
        out["x"] = torch.randn((T, d_in), generator=gen(_S_X), device=device).to(torch.bfloat16)
    if "dY" in keys:
        out["dY"] = torch.randn((T, d_out), generator=gen(_S_DY), device=device).to(torch.bfloat16)
    if "y0" in keys:
        if y0 == "randn":
            out["y0"] = torch.randn((T, d_out), generator=gen(_S_Y0), device=device).to(torch.bfloat16)
        else:
            out["y0"] = torch.zeros((T, d_out), device=device, dtype=torch.bfloat16)
    if "W" in keys:
        w = torch.rand((d_out, d_in), generator=gen(_S_W), device=device, dtype=torch.float32)
        out["W"] = (w * (2 * lim) - lim).to(torch.bfloat16)
    if "dX0" in keys:
        if dX0 == "randn":
            out["dX0"] = torch.randn((T, d_in), generator=gen(_S_DX0), device=device).to(torch.bfloat16)
        else:
            out["dX0"] = torch.zeros((T, d_in), device=device, dtype=torch.bfloat16)
    return out
