"""Pins for the fp64 oracle, checked against things other than the oracle itself.

The pages print no worked example and no formula for the LoRA delta, so the
oracle is pinned by closed forms and invariants the method fixes:
  * routing equals numpy's stable argsort (a library routine);
  * with one adapter the packed delta is an ordinary LoRA matmul (numpy ``@``);
  * brute-force Python loops on tiny inputs, written per adapter rather than
    per token;
  * central finite differences of L = sum(dY * y) (exact, L being linear in
    every single entry of A, B and x);
  * B_i = 0, token permutation, packing == sequential, rank padding,
    splitting an adapter into two identical ones, linearity in s_i, bad ids.
Each one is chosen so that a plausible slip (a dropped scale, a transposed
block, a wrong ragged offset, an unstable sort) fails at least one test.
"""
import numpy as np
import pytest

import oracle
import workloads as wl


def f64(bits):
    return wl.bf16_bits_to_f64(bits)


def make(spec, y0="zero", dX0="zero"):
    h = wl.host_inputs(spec, y0=y0, dX0=dX0)
    P = {k: f64(v) for k, v in h.items()}
    P["tab"] = oracle.Table(spec.ranks, spec.scales.astype(np.float64))
    P["ids"] = spec.ids
    return P


def run_all(P, r_max=None):
    tab = P["tab"]
    y, H = oracle.fwd(tab, P["ids"], P["A"], P["B"], P["x"], P["y0"], r_max)
    dH, dA, dB, dX = oracle.bwd(tab, P["ids"], P["A"], P["B"], P["x"], H, P["dY"], P["dX0"], r_max)
    return dict(y=y, H=H, dH=dH, dA=dA, dB=dB, dX=dX)


def close(a, b, rel=1e-12):
    a = np.asarray(a)
    b = np.asarray(b)
    scale = max(1e-300, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= rel * scale, f"max|err|={err:.3e} > {rel:.1e} * {scale:.3e}"


def B_block(P, i, d_out):
    """B_i as the d_out x r_i matrix (stored transposed: rows of B are columns of B_i)."""
    tab = P["tab"]
    r = int(tab.rank[i])
    a0 = int(tab.row_off[i])
    return P["B"][a0:a0 + r].T


# ---------------------------------------------------------------- routing
def test_route_matches_numpy_stable_argsort():
    rng = np.random.default_rng(7)
    for T, N in [(1, 1), (17, 3), (1000, 8), (4096, 37)]:
        ids = rng.integers(-2, N + 2, size=T).astype(np.int32)
        perm, seg, bad = oracle.route(ids, N)
        valid = (ids >= 0) & (ids < N)
        idx = np.flatnonzero(valid)
        want = idx[np.argsort(ids[valid], kind="stable")]
        assert bad == int((~valid).sum())
        assert np.array_equal(perm, want)
        cnt = np.bincount(ids[valid], minlength=N)
        assert np.array_equal(seg, np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32))


def test_route_sorted_input_is_identity():
    spec = wl.tiny()
    perm, seg, bad = oracle.route(spec.ids, spec.n_adapters)
    assert bad == 0
    assert np.array_equal(perm, np.arange(spec.n_tokens))
    assert np.array_equal(seg, spec.seg_offsets)


def test_route_empty_and_all_one_adapter():
    perm, seg, bad = oracle.route(np.zeros(0, np.int32), 4)
    assert perm.size == 0 and np.all(seg == 0) and bad == 0
    ids = np.full(33, 2, np.int32)
    perm, seg, bad = oracle.route(ids, 4)
    assert np.array_equal(perm, np.arange(33)) and seg.tolist() == [0, 0, 0, 33, 33]


# ---------------------------------------------------------------- I1: N = 1 closed form
@pytest.mark.parametrize("r,d_in,d_out,T", [(1, 8, 16, 5), (16, 64, 48, 40), (37, 24, 72, 19)])
def test_single_adapter_is_plain_lora_matmul(r, d_in, d_out, T):
    spec = wl.custom("n1", d_in, d_out, [r], [2.0 * r + 3.0], np.zeros(T, np.int32), seed=3)
    P = make(spec, y0="randn", dX0="randn")
    out = run_all(P)
    s = float(spec.scales[0])
    A, x, dY = P["A"], P["x"], P["dY"]
    B = P["B"].T  # B_i, d_out x r (stored as its transpose)
    H = x @ A.T
    close(out["H"], H)
    close(out["y"], P["y0"] + s * (H @ B.T))
    dH = s * (dY @ B)
    close(out["dH"], dH)
    close(out["dB"].T, s * (dY.T @ H))
    close(out["dA"], dH.T @ x)
    close(out["dX"], P["dX0"] + dH @ A)


# ---------------------------------------------------------------- I2: brute force loops
def brute_force(P, spec):
    """Per-adapter Python loops over explicit token lists."""
    T, N, d_in, d_out = spec.n_tokens, spec.n_adapters, spec.d_in, spec.d_out
    r_max = spec.r_max
    ranks, off = spec.ranks, spec.row_off
    s = spec.scales.astype(np.float64)
    A, Bf, x, dY = P["A"], P["B"], P["x"], P["dY"]
    y = P["y0"].copy()
    dX = P["dX0"].copy()
    H = np.zeros((T, r_max))
    dH = np.zeros((T, r_max))
    dA = np.zeros_like(A)
    dB = np.zeros_like(Bf)
    for i in range(N):
        toks = [t for t in range(T) if spec.ids[t] == i]
        r = int(ranks[i])
        a0 = int(off[i])
        for t in toks:
            for k in range(r):
                acc = 0.0
                for j in range(d_in):
                    acc += A[off[i] + k, j] * x[t, j]
                H[t, k] = acc
            for o in range(d_out):
                acc = 0.0
                for k in range(r):
                    acc += Bf[a0 + k, o] * H[t, k]
                y[t, o] += s[i] * acc
            for k in range(r):
                acc = 0.0
                for o in range(d_out):
                    acc += dY[t, o] * Bf[a0 + k, o]
                dH[t, k] = s[i] * acc
            for j in range(d_in):
                acc = 0.0
                for k in range(r):
                    acc += dH[t, k] * A[off[i] + k, j]
                dX[t, j] += acc
        for o in range(d_out):
            for k in range(r):
                dB[a0 + k, o] = s[i] * sum(dY[t, o] * H[t, k] for t in toks)
        for k in range(r):
            for j in range(d_in):
                dA[off[i] + k, j] = sum(dH[t, k] * x[t, j] for t in toks)
    return dict(y=y, H=H, dH=dH, dA=dA, dB=dB, dX=dX)


def test_bruteforce_tiny_random():
    ids = np.array([2, 0, 0, 5, 1, 2, 2, -1], np.int32)  # 5 and -1 belong to no adapter
    spec = wl.custom("bf", 5, 6, [1, 2, 3], [3.0, 2.0, 12.0], ids, seed=11)
    P = make(spec, y0="randn", dX0="randn")
    want = brute_force(P, spec)
    got = run_all(P)
    for k in want:
        close(got[k], want[k])


def test_bruteforce_configs_tiny():
    spec = wl.tiny()
    P = make(spec, y0="randn", dX0="randn")
    want = brute_force(P, spec)
    got = run_all(P)
    for k in want:
        close(got[k], want[k])


# ---------------------------------------------------------------- I5: finite differences
def test_gradients_match_central_differences():
    spec = wl.tiny()
    P = make(spec)
    tab, ids = P["tab"], P["ids"]
    out = run_all(P)
    dY = P["dY"]

    def L(A, B, x):
        y, _ = oracle.fwd(tab, ids, A, B, x, np.zeros_like(P["y0"]))
        return float(np.sum(dY * y))

    rng = np.random.default_rng(5)
    step = 0.5  # L is linear in each single entry: any step gives the exact slope
    for name, grad in (("A", out["dA"]), ("B", out["dB"]), ("x", out["dX"])):
        base = P[name]
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in base.shape)
            plus, minus = base.copy(), base.copy()
            plus[idx] += step
            minus[idx] -= step
            args = {"A": P["A"], "B": P["B"], "x": P["x"]}
            args[name] = plus
            lp = L(**args)
            args[name] = minus
            lm = L(**args)
            fd = (lp - lm) / (2 * step)
            g = float(grad[idx])
            assert abs(fd - g) <= 1e-9 * max(1.0, abs(g)), (name, idx, fd, g)


# ---------------------------------------------------------------- I3: B_i = 0
def test_zero_B_adapter_contributes_nothing():
    spec = wl.tiny()
    P = make(spec, y0="randn", dX0="randn")
    i = 2
    a0, a1 = int(spec.row_off[i]), int(spec.row_off[i + 1])
    P["B"][a0:a1] = 0.0
    out = run_all(P)
    rows = spec.ids == i
    close(out["y"][rows], P["y0"][rows], 0.0)
    assert np.all(out["dH"][rows] == 0.0)
    assert np.all(out["dA"][a0:a1] == 0.0)
    close(out["dX"][rows], P["dX0"][rows], 0.0)
    assert np.any(out["dB"][a0:a1] != 0.0)  # dB_i = s dY^T H is not zero
    assert np.any(out["y"][~rows] != P["y0"][~rows])


# ---------------------------------------------------------------- I4: permutation
def test_token_permutation_equivariance():
    rng = np.random.default_rng(9)
    spec = wl.random_spec(rng, 50, 5, 40, 24, rank_choices=(3, 8, 16))
    P = make(spec, y0="randn", dX0="randn")
    out = run_all(P)
    p = rng.permutation(spec.n_tokens)
    Q = dict(P)
    for k in ("x", "dY", "y0", "dX0"):
        Q[k] = P[k][p]
    Q["ids"] = P["ids"][p]
    outp = run_all(Q)
    for k in ("y", "H", "dH", "dX"):
        close(outp[k], out[k][p], 0.0)
    close(outp["dA"], out["dA"], 1e-13)
    close(outp["dB"], out["dB"], 1e-13)
    perm_a, seg_a, _ = oracle.route(P["ids"], 5)
    perm_b, seg_b, _ = oracle.route(Q["ids"], 5)
    assert np.array_equal(seg_a, seg_b)
    assert np.array_equal(P["ids"][perm_a], Q["ids"][perm_b])


# ---------------------------------------------------------------- I6: packing == sequential
def test_packing_equals_sequential_single_adapter_runs():
    rng = np.random.default_rng(4)
    spec = wl.random_spec(rng, 60, 4, 32, 40, rank_choices=(2, 8, 16))
    P = make(spec, y0="randn", dX0="randn")
    out = run_all(P)
    d_in, d_out = spec.d_in, spec.d_out
    for i in range(spec.n_adapters):
        rows = np.flatnonzero(spec.ids == i)
        r = int(spec.ranks[i])
        a0 = int(spec.row_off[i])
        tab1 = oracle.Table([r], [float(spec.scales[i])])
        ids1 = np.zeros(rows.size, np.int32)
        A1 = P["A"][a0:a0 + r]
        B1 = P["B"][a0:a0 + r]
        y, H = oracle.fwd(tab1, ids1, A1, B1, P["x"][rows], P["y0"][rows])
        dH, dA, dB, dX = oracle.bwd(tab1, ids1, A1, B1, P["x"][rows], H, P["dY"][rows], P["dX0"][rows])
        close(out["y"][rows], y, 0.0)
        close(out["H"][rows, :r], H, 0.0)
        close(out["dX"][rows], dX, 0.0)
        close(out["dA"][a0:a0 + r], dA, 1e-13)
        close(out["dB"][a0:a0 + r], dB, 1e-13)
        assert d_in == P["x"].shape[1]


# ---------------------------------------------------------------- I7: rank padding
def test_zero_rank_padding_changes_nothing():
    rng = np.random.default_rng(12)
    spec = wl.random_spec(rng, 30, 3, 16, 24, rank_choices=(2, 4, 5))
    P = make(spec, y0="randn", dX0="randn")
    out = run_all(P)
    pad = 3
    d_in, d_out = spec.d_in, spec.d_out
    ranks2 = spec.ranks + pad
    A2, B2 = [], []
    for i in range(spec.n_adapters):
        r = int(spec.ranks[i])
        a0 = int(spec.row_off[i])
        A2.append(np.vstack([P["A"][a0:a0 + r], np.zeros((pad, d_in))]))
        B2.append(np.vstack([P["B"][a0:a0 + r], np.zeros((pad, d_out))]))
    Q = dict(P)
    Q["A"] = np.vstack(A2)
    Q["B"] = np.vstack(B2)
    Q["tab"] = oracle.Table(ranks2, spec.scales.astype(np.float64))  # s_i held fixed
    outp = run_all(Q, r_max=int(ranks2.max()))
    close(outp["y"], out["y"], 0.0)
    close(outp["dX"], out["dX"], 0.0)
    for i in range(spec.n_adapters):
        r = int(spec.ranks[i])
        a0, b0 = int(spec.row_off[i]), int(Q["tab"].row_off[i])
        rows = spec.ids == i
        close(outp["H"][rows, :r], out["H"][rows, :r], 0.0)
        assert np.all(outp["H"][rows, r:] == 0.0)
        close(outp["dA"][b0:b0 + r], out["dA"][a0:a0 + r], 0.0)
        assert np.all(outp["dA"][b0 + r:b0 + r + pad] == 0.0)


# ---------------------------------------------------------------- I8: split an adapter in two
def test_splitting_an_adapter_into_two_identical_ones():
    spec = wl.tiny()
    P = make(spec, y0="randn", dX0="randn")
    out = run_all(P)
    i = 2  # duplicate adapter 2 as a new adapter 4; route every other of its tokens there
    d_out = spec.d_out
    r = int(spec.ranks[i])
    a0 = int(spec.row_off[i])
    ranks2 = np.concatenate([spec.ranks, [r]])
    scales2 = np.concatenate([spec.scales, [spec.scales[i]]]).astype(np.float64)
    Q = dict(P)
    Q["A"] = np.vstack([P["A"], P["A"][a0:a0 + r]])
    Q["B"] = np.vstack([P["B"], P["B"][a0:a0 + r]])
    Q["tab"] = oracle.Table(ranks2, scales2)
    ids2 = P["ids"].copy()
    rows = np.flatnonzero(ids2 == i)
    ids2[rows[1::2]] = 4
    Q["ids"] = ids2
    outp = run_all(Q)
    for k in ("y", "H", "dH", "dX"):
        close(outp[k], out[k], 0.0)
    s0 = int(spec.sum_r)
    close(outp["dA"][a0:a0 + r] + outp["dA"][s0:s0 + r], out["dA"][a0:a0 + r], 1e-13)
    close(outp["dB"][a0:a0 + r] + outp["dB"][s0:s0 + r], out["dB"][a0:a0 + r], 1e-13)


# ---------------------------------------------------------------- I9: linearity in s_i
def test_doubling_alpha_doubles_the_adapters_contribution():
    spec = wl.tiny()
    P = make(spec, y0="randn", dX0="zero")
    out = run_all(P)
    i = 1
    sc = spec.scales.astype(np.float64).copy()
    sc[i] *= 2.0
    Q = dict(P)
    Q["tab"] = oracle.Table(spec.ranks, sc)
    outp = run_all(Q)
    rows = spec.ids == i
    close(outp["y"][rows] - P["y0"][rows], 2.0 * (out["y"][rows] - P["y0"][rows]), 1e-14)
    close(outp["y"][~rows], out["y"][~rows], 0.0)
    b0, b1 = int(spec.row_off[i]), int(spec.row_off[i + 1])
    close(outp["dB"][b0:b1], 2.0 * out["dB"][b0:b1], 0.0)
    close(outp["dH"][rows], 2.0 * out["dH"][rows], 0.0)
    # dA_i = dH^T X and dX pick up s_i through dH
    a0, a1 = int(spec.row_off[i]), int(spec.row_off[i + 1])
    close(outp["dA"][a0:a1], 2.0 * out["dA"][a0:a1], 0.0)


# ---------------------------------------------------------------- bad ids / empty adapters
def test_tokens_without_adapter_and_empty_adapters():
    ids = np.array([0, 7, 0, -3, 0], np.int32)  # adapter 1 has no token
    spec = wl.custom("bad", 16, 8, [4, 8], [8.0, 16.0], ids, seed=2)
    P = make(spec, y0="randn", dX0="randn")
    out = run_all(P)
    for t in (1, 3):
        close(out["y"][t], P["y0"][t], 0.0)
        close(out["dX"][t], P["dX0"][t], 0.0)
        assert np.all(out["H"][t] == 0.0) and np.all(out["dH"][t] == 0.0)
    assert np.all(out["dA"][4:12] == 0.0)
    assert np.all(out["dB"][4:12] == 0.0)


# ---------------------------------------------------------------- optimizer step
def test_adamw_first_step_closed_form():
    # t = 1 from zero moments: m_hat = g and v_hat = g^2, so the step is
    # w (1 - lr wd) - lr g / (|g| + eps)
    tab = oracle.Table([3, 5], [1.0, 1.0])
    rng = np.random.default_rng(11)
    w = rng.standard_normal((8, 16))
    g = rng.standard_normal((8, 16))
    lr = np.array([1e-3, 5e-3])
    w1, m1, v1 = oracle.adamw(tab, w, g, np.zeros_like(w), np.zeros_like(w), lr, 1, beta1=0.9, beta2=0.99,
                              eps=1e-6, weight_decay=0.1)
    lr_rows = np.repeat(lr, [3, 5])[:, None]
    ref = w * (1 - lr_rows * 0.1) - lr_rows * g / (np.abs(g) + 1e-6)
    assert np.allclose(w1, ref, rtol=1e-13, atol=1e-15)
    assert np.allclose(m1, 0.1 * g, rtol=1e-14) and np.allclose(v1, 0.01 * g * g, rtol=1e-13)


def test_adamw_matches_torch_optimizer_over_several_steps():
    torch = pytest.importorskip("torch")
    ranks = [2, 4, 3]
    tab = oracle.Table(ranks, [1.0] * 3)
    rng = np.random.default_rng(12)
    d = 24
    w = rng.standard_normal((sum(ranks), d))
    lrs = [1e-2, 3e-3, 7e-4]
    params = [torch.tensor(w[o:o + r].copy(), dtype=torch.float64, requires_grad=True)
              for o, r in zip(tab.row_off[:-1], ranks)]
    opt = torch.optim.AdamW([{"params": [p], "lr": lr} for p, lr in zip(params, lrs)], betas=(0.9, 0.95), eps=1e-7,
                            weight_decay=0.05)
    m = np.zeros_like(w)
    v = np.zeros_like(w)
    for t in range(1, 5):
        g = rng.standard_normal(w.shape)
        for p, o, r in zip(params, tab.row_off[:-1], ranks):
            p.grad = torch.tensor(g[o:o + r].copy(), dtype=torch.float64)
        opt.step()
        w, m, v = oracle.adamw(tab, w, g, m, v, lrs, t, beta1=0.9, beta2=0.95, eps=1e-7, weight_decay=0.05)
    ref = np.concatenate([p.detach().numpy() for p in params])
    assert np.allclose(w, ref, rtol=1e-12, atol=1e-14)


def test_adamw_zero_learning_rate_keeps_weights_and_moves_moments():
    tab = oracle.Table([4, 4], [1.0, 1.0])
    rng = np.random.default_rng(13)
    w = rng.standard_normal((8, 8))
    g = rng.standard_normal((8, 8))
    w1, m1, _ = oracle.adamw(tab, w, g, np.zeros_like(w), np.zeros_like(w), [0.0, 1e-3], [3, 7], weight_decay=0.1)
    assert np.array_equal(w1[:4], w[:4]) and not np.array_equal(w1[4:], w[4:])
    assert np.allclose(m1, 0.1 * g, rtol=1e-14)


# ---------------------------------------------------------------- base projection + delta
def test_base_matches_numpy_matmul():
    rng = np.random.default_rng(21)
    W = rng.standard_normal((13, 9))
    x = rng.standard_normal((6, 9))
    assert np.allclose(oracle.base(W, x), x @ W.T, rtol=1e-13, atol=1e-13)


def test_base_identity_and_permutation_weights_are_exact():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((7, 10))
    assert np.array_equal(oracle.base(np.eye(10), x), x)
    p = rng.permutation(10)
    P = np.eye(10)[p]  # row o of W picks input p[o]
    assert np.array_equal(oracle.base(P, x), x[:, p])


def test_base_rank_one_weight_closed_form():
    # W = u v^T: y_t = u (v . x_t); a transposed W or swapped loop bound fails
    rng = np.random.default_rng(23)
    u = rng.standard_normal(11)
    v = rng.standard_normal(5)
    x = rng.standard_normal((4, 5))
    assert np.allclose(oracle.base(np.outer(u, v), x), np.outer(x @ v, u), rtol=1e-13, atol=1e-13)


def test_layer_forward_is_base_plus_single_adapter_lora():
    # one adapter: y = x W^T + s x A^T B^T with numpy @ (the plain LoRA layer)
    spec = wl.custom("layer1", 24, 40, [6], [18.0], np.zeros(9, np.int32), seed=5)
    P = make(spec)
    W = f64(wl.base_weight(spec))
    y, H = oracle.base_lora_fwd(P["tab"], P["ids"], W, P["A"], P["B"], P["x"])
    s = float(spec.scales[0])
    close(H, P["x"] @ P["A"].T)
    close(y, P["x"] @ W.T + s * (P["x"] @ P["A"].T) @ P["B"])


def test_layer_forward_reduces_to_its_parts():
    # W = 0: the packed delta alone; A = 0: the base alone
    ids = np.array([1, 1, 0, 2, 0, 1, 2, 2, 2, 0], np.int32)
    spec = wl.custom("layer3", 16, 24, [2, 5, 3], [4.0, 10.0, 3.0], ids, seed=6)
    P = make(spec)
    W = f64(wl.base_weight(spec))
    y, H = oracle.base_lora_fwd(P["tab"], P["ids"], np.zeros_like(W), P["A"], P["B"], P["x"])
    y_d, H_d = oracle.fwd(P["tab"], P["ids"], P["A"], P["B"], P["x"], np.zeros((10, 24)))
    assert np.array_equal(y, y_d) and np.array_equal(H, H_d)
    y0, _ = oracle.base_lora_fwd(P["tab"], P["ids"], W, np.zeros_like(P["A"]), P["B"], P["x"])
    close(y0, P["x"] @ W.T)


# ---------------------------------------------------------------- hand-worked example
def test_oracle_reproduces_the_hand_worked_example_exactly():
    # tests/golden/worked_two_adapters.json: two adapters of rank 1 and 2, three
    # unsorted tokens, every product worked out by hand in small integers
    from lora_testlib import worked_example

    g = worked_example()
    tab = oracle.Table(g["ranks"], g["scales"])
    y, H = oracle.fwd(tab, g["ids"], g["A"], g["B"], g["x"], np.zeros_like(g["y"]))
    dH, dA, dB, dX = oracle.bwd(tab, g["ids"], g["A"], g["B"], g["x"], H, g["dY"], np.zeros_like(g["dX"]))
    for name, got, want in (("y", y, g["y"]), ("H", H, g["H"]), ("dH", dH, g["dH"]), ("dA", dA, g["dA"]),
                            ("dB", dB, g["dB"]), ("dX", dX, g["dX"])):
        assert np.array_equal(got, want), name
