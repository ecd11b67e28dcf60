"""Segment-metadata builder on the GPU: bit-exact against the oracle's stable
counting sort, tiles checked for validity, device-side error reporting."""
import numpy as np
import pytest
import torch

import adapter_sgmv_gb300 as lora
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lora.build_library()
    lora.lib()


def expected_pieces(seg_start, perm, length):
    out = []
    for i in range(len(seg_start) - 1):
        n = int(seg_start[i + 1] - seg_start[i])
        for q in range(0, n, length):
            b = int(seg_start[i]) + q
            rows = min(length, n - q)
            out.append((i, b, rows, int(perm[b + rows - 1] - perm[b] == rows - 1)))
    return out


def check_tiles(segs, seg_start, perm):
    """Tiles (128 tokens) and spans (1024 tokens): every adapter's group cut in
    order, nothing straddling adapters, contiguity flags right."""
    for length, n_dev, lst in ((128, segs.n_tiles, segs.tiles), (1024, segs.n_spans, segs.spans)):
        n = int(n_dev.item())
        got = [tuple(int(v) for v in t) for t in lst[:n].cpu().numpy()]
        assert got == expected_pieces(seg_start, perm, length)


def run_ids(ids_np, N):
    ids = torch.from_numpy(np.asarray(ids_np, dtype=np.int32)).cuda()
    segs = lora.lora_build_segments(ids=ids, n_adapters=N, n_tokens=len(ids_np))
    st = lora.lora_query_status(segs)
    return segs, st


ID_CASES = {
    "decode256x8": lambda: (wl.decode(0).ids, 8),
    "skewed16384x32": lambda: (wl.skewed().ids, 32),
    "one_token": lambda: (np.array([3], np.int32), 4),
    "all_one_adapter": lambda: (np.full(300, 2, np.int32), 4),
    "sparse_many_adapters": lambda: (np.random.default_rng(1).integers(0, 3000, 2000).astype(np.int32), 3000),
    "runs_and_singletons": lambda: (np.concatenate([np.full(129, 1), [0], np.full(257, 1), [2, 0, 2]]).astype(np.int32), 3),
    "odd_length_random": lambda: (np.random.default_rng(2).integers(0, 7, 4099).astype(np.int32), 7),
    "ten_thousand_adapters": lambda: (np.random.default_rng(3).integers(0, 10000, 5000).astype(np.int32), 10000),
    # the one-launch build holds the ids, their permutation, N x 32 counts and
    # two tables of N + 1 in 200 KB of shared memory: at the limit, and just
    # past it (the six-launch build)
    "one_launch_limit": lambda: (np.random.default_rng(4).integers(0, 542, 16384).astype(np.int32), 542),
    "past_one_launch_limit": lambda: (np.random.default_rng(5).integers(0, 543, 16384).astype(np.int32), 543),
}


@pytest.mark.parametrize("name", sorted(ID_CASES))
def test_route_from_ids_is_bit_exact(name):
    ids, N = ID_CASES[name]()
    segs, st = run_ids(ids, N)
    assert st == 0
    perm_o, seg_o, bad = oracle.route(ids, N)
    seg = segs.seg_start.cpu().numpy()
    perm = segs.perm.cpu().numpy()[: seg[-1]]
    assert np.array_equal(seg, seg_o)
    assert np.array_equal(perm, perm_o)
    check_tiles(segs, seg, perm)


def test_route_bad_ids_reported_and_left_out():
    rng = np.random.default_rng(3)
    ids = rng.integers(-2, 7, 1000).astype(np.int32)  # N = 5: -2, -1, 5, 6 are bad
    segs, st = run_ids(ids, 5)
    assert st == lora.LoraError(4, "").status
    perm_o, seg_o, bad = oracle.route(ids, 5)
    seg = segs.seg_start.cpu().numpy()
    assert np.array_equal(seg, seg_o)
    assert np.array_equal(segs.perm.cpu().numpy()[: seg[-1]], perm_o)
    lora.lora_reset_status(segs)
    assert lora.lora_query_status(segs) == 0


def test_route_empty_batch():
    segs = lora.lora_build_segments(ids=torch.zeros(0, dtype=torch.int32, device="cuda"), n_adapters=4,
                                    n_tokens=0)
    assert lora.lora_query_status(segs) == 0
    assert segs.seg_start.cpu().tolist() == [0] * 5
    assert int(segs.n_tiles.item()) == 0


@pytest.mark.parametrize("offsets", [[0, 8, 24, 48, 64], [0, 0, 5, 5, 10], [0, 4096 * 8], [0, 129, 130, 400]])
def test_route_from_sorted_offsets(offsets):
    off = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    N, T = len(offsets) - 1, offsets[-1]
    segs = lora.lora_build_segments(seg_offsets=off, n_tokens=T, n_adapters=N)
    assert lora.lora_query_status(segs) == 0
    assert segs.seg_start.cpu().tolist() == offsets
    perm = segs.perm.cpu().numpy()
    assert np.array_equal(perm, np.arange(T))
    check_tiles(segs, np.array(offsets), perm)


def random_offsets(N, seed, max_len=9):
    # segment lengths 0..max_len (a quarter of the adapters empty), first 0, last T
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, max_len + 1, N)
    lens[rng.random(N) < 0.25] = 0
    lens[rng.integers(0, N)] += 300  # one segment of several tiles
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


@pytest.mark.parametrize("N", [4095, 4096, 9000])
def test_route_from_sorted_offsets_many_adapters(N):
    # 4095 adapters: the one-launch build at its shared-memory capacity; above
    # it the build that scans the offsets in global memory
    offsets = random_offsets(N, seed=N)
    T = int(offsets[-1])
    off = torch.from_numpy(offsets).cuda()
    segs = lora.lora_build_segments(seg_offsets=off, n_tokens=T, n_adapters=N)
    assert lora.lora_query_status(segs) == 0
    assert np.array_equal(segs.seg_start.cpu().numpy(), offsets)
    perm = segs.perm.cpu().numpy()
    assert np.array_equal(perm, np.arange(T))
    check_tiles(segs, offsets, perm)


@pytest.mark.parametrize("N", [4095, 5000])
def test_route_inconsistent_offsets_many_adapters(N):
    offsets = random_offsets(N, seed=7 + N)
    offsets[N // 2] = offsets[N // 2 + 1] + 1  # one segment ends before it starts
    T = int(offsets[-1])
    off = torch.from_numpy(offsets).cuda()
    segs = lora.lora_build_segments(seg_offsets=off, n_tokens=T, n_adapters=N)
    assert lora.lora_query_status(segs) == 9
    assert int(segs.n_tiles.item()) == 0 and int(segs.n_spans.item()) == 0


@pytest.mark.parametrize("offsets,T", [([0, 9, 5, 12], 12), ([1, 4, 12], 12), ([0, 4, 11], 12)])
def test_route_inconsistent_offsets_yield_no_work(offsets, T):
    off = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    segs = lora.lora_build_segments(seg_offsets=off, n_tokens=T, n_adapters=len(offsets) - 1)
    assert lora.lora_query_status(segs) == 9
    assert int(segs.n_tiles.item()) == 0 and int(segs.n_spans.item()) == 0
    assert np.all(segs.seg_start.cpu().numpy() == 0)
