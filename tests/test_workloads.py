"""The seeded input recipe (no GPU): shapes and value distributions of the
synthetic inputs, the bf16 rounding, and the committed draw of the skewed
batch.  The generators hold no LoRA arithmetic; these checks pin the recipe
stated for the inputs (standard deviation 0.02 for B, uniform +-1/sqrt(d_in)
for A, N(0, 1) activations, fp32 draws rounded to bf16 nearest-even, Zipf(1.2)
run lengths capped at 1024)."""
import json

import numpy as np
import torch

import workloads as wl


def test_bf16_rounding_is_nearest_even():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 65504.0, 1e-40], np.float32)
    bits = wl.f32_to_bf16_bits(f)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, want)
    assert bits[1] == wl.f32_to_bf16_bits(np.array([1.0], np.float32))[0]  # tie to even (down)
    assert bits[2] == wl.f32_to_bf16_bits(np.array([1.0 + 4 * 2 ** -8], np.float32))[0]  # tie to even (up)


def test_host_recipe_distributions():
    spec = wl.custom("dist", 512, 640, [64, 64], [128.0, 128.0], np.zeros(4096, np.int32))
    h = wl.host_inputs(spec, y0="randn", dX0="randn")
    f = {k: wl.bf16_bits_to_f64(v) for k, v in h.items()}
    lim = 1.0 / np.sqrt(512)
    assert f["A"].shape == (128, 512) and np.all(np.abs(f["A"]) <= lim * (1 + 2 ** -8))
    assert abs(f["A"].std() - lim / np.sqrt(3)) < 0.02 * lim  # uniform on [-lim, lim]
    assert f["B"].shape == (128, 640) and abs(f["B"].std() - 0.02) < 0.0005
    for k in ("x", "dY", "y0", "dX0"):
        assert abs(f[k].mean()) < 0.01 and abs(f[k].std() - 1.0) < 0.01, k
    # seeded: the same spec draws the same bits, another seed other bits
    assert np.array_equal(wl.host_inputs(spec)["x"], h["x"])
    other = wl.custom("dist", 512, 640, [64, 64], [128.0, 128.0], np.zeros(4096, np.int32), seed=1)
    assert not np.array_equal(wl.host_inputs(other)["x"], h["x"])


def test_skewed_fixture_is_the_seed0_draw_of_its_recipe():
    with open(wl.SKEWED_FIXTURE) as f:
        fx = json.load(f)
    ranks, runs = wl.draw_skewed(0)
    assert fx["ranks"] == [int(r) for r in ranks] and fx["runs"] == [[int(n), int(a)] for n, a in runs]
    n = np.array([r[0] for r in fx["runs"]])
    assert n.sum() == 16384 and n.max() <= 1024 and len(n) == 259 and int((n == 1).sum()) == 51
    spec = wl.skewed()
    assert int(spec.sum_r) == 1816 and set(spec.ranks.tolist()) <= {8, 16, 32, 64, 128}
    assert np.array_equal(spec.alphas, 2.0 * spec.ranks)
