"""The fused per-adapter AdamW step (lora_adamw_step) against the fp64 oracle:
fp32 masters and moments within a tolerance over several steps, the table's
bf16 weights bit-equal to the round-to-nearest-even of the new fp32 masters,
per-adapter learning rates and step numbers, an adapter with lr = 0 left
unchanged."""
import numpy as np
import pytest
import torch

import adapter_sgmv_gb300 as lora
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 1e-5  # fp32 arithmetic against fp64: max|err| <= TOL * max|ref| per array


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lora.build_library()
    lora.lib()


def _rel(got, ref):
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


@pytest.mark.parametrize("d_in,d_out", [(320, 200), (4096, 4096)])
def test_adamw_step_matches_oracle(d_in, d_out):
    ranks = [8, 16, 128, 32]
    n = len(ranks)
    sum_r = sum(ranks)
    rng = np.random.default_rng(d_in)
    dev = torch.device("cuda")
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    wA0 = rng.standard_normal((sum_r, d_in)).astype(np.float32) * 0.05
    wB0 = rng.standard_normal((sum_r, d_out)).astype(np.float32) * 0.02
    mA0 = rng.standard_normal(wA0.shape).astype(np.float32) * 1e-3
    mB0 = rng.standard_normal(wB0.shape).astype(np.float32) * 1e-3
    vA0 = (rng.standard_normal(wA0.shape).astype(np.float32) * 1e-3) ** 2
    vB0 = (rng.standard_normal(wB0.shape).astype(np.float32) * 1e-3) ** 2
    lr = np.array([1e-3, 2e-4, 5e-3, 0.0], dtype=np.float32)
    step0 = np.array([1, 4, 10, 2], dtype=np.int32)
    hp = dict(beta1=0.9, beta2=0.98, eps=1e-6, weight_decay=0.01)

    wA, wB, mA, mB, vA, vB = (f32(a) for a in (wA0, wB0, mA0, mB0, vA0, vB0))
    A_bf = torch.zeros((sum_r, d_in), dtype=torch.bfloat16, device=dev)
    B_bf = torch.zeros((sum_r, d_out), dtype=torch.bfloat16, device=dev)
    table = lora.AdapterTable(A_bf, B_bf, ranks, torch.ones(n, dtype=torch.float32), d_in, d_out)
    lr_d = f32(lr)
    step_d = torch.from_numpy(step0.copy()).to(dev)

    tab = oracle.Table(ranks, np.ones(n))
    ref = {"wA": wA0.astype(np.float64), "wB": wB0.astype(np.float64), "mA": mA0.astype(np.float64),
           "mB": mB0.astype(np.float64), "vA": vA0.astype(np.float64), "vB": vB0.astype(np.float64)}
    step = step0.copy()
    for k in range(3):
        gA = rng.standard_normal(wA0.shape).astype(np.float32) * 1e-2
        gB = rng.standard_normal(wB0.shape).astype(np.float32) * 1e-2
        lora.lora_adamw_step(table, wA, wB, f32(gA), f32(gB), mA, vA, mB, vB, lr_d, step_d, **hp)
        ref["wA"], ref["mA"], ref["vA"] = oracle.adamw(tab, ref["wA"], gA, ref["mA"], ref["vA"], lr, step, **hp)
        ref["wB"], ref["mB"], ref["vB"] = oracle.adamw(tab, ref["wB"], gB, ref["mB"], ref["vB"], lr, step, **hp)
        step += 1
        step_d += 1
    torch.cuda.synchronize()
    got = {k: t.cpu().numpy().astype(np.float64) for k, t in
           (("wA", wA), ("wB", wB), ("mA", mA), ("mB", mB), ("vA", vA), ("vB", vB))}
    for k in got:
        assert _rel(got[k], ref[k]) <= TOL, (k, _rel(got[k], ref[k]))
    # lr = 0 (last adapter): masters unchanged
    r0 = sum(ranks[:-1])
    assert np.array_equal(wA.cpu().numpy()[r0:], wA0[r0:]) and np.array_equal(wB.cpu().numpy()[r0:], wB0[r0:])
    # the table's bf16 weights are the rounding of the new masters, bit for bit
    for t_bf, t32 in ((A_bf, wA), (B_bf, wB)):
        want = wl.f32_to_bf16_bits(t32.cpu().numpy())
        have = t_bf.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(have, want)


def test_adamw_step_rejects_bad_hyper_parameters():
    ranks = [8]
    dev = torch.device("cuda")
    A_bf = torch.zeros((8, 64), dtype=torch.bfloat16, device=dev)
    B_bf = torch.zeros((8, 64), dtype=torch.bfloat16, device=dev)
    table = lora.AdapterTable(A_bf, B_bf, ranks, torch.ones(1), 64, 64)
    z = lambda: torch.zeros((8, 64), dtype=torch.float32, device=dev)
    lr = torch.ones(1, device=dev)
    step = torch.ones(1, dtype=torch.int32, device=dev)
    with pytest.raises(lora.LoraError) as e:
        lora.lora_adamw_step(table, z(), z(), z(), z(), z(), z(), z(), z(), lr, step, beta1=1.0)
    assert e.value.status == 1
