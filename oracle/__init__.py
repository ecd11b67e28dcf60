"""fp64 CPU oracle for the multi-adapter LoRA delta (test infrastructure).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` import this
package.  The CUDA library and its Python binding never import it, and it
shares no code with them: the arithmetic lives in ``lora_oracle.c`` (plain C
loops in IEEE double, see its header for the definitions and the passages of
the pages they follow); this module only compiles that file with gcc and
marshals numpy arrays through ctypes.

Inputs are bf16 values widened exactly to float64 by the caller (see
``workloads.bf16_bits_to_f32``); every output is float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblora_oracle.so")

_lib = None
_lock = threading.Lock()

_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile ``lora_oracle.c`` into ``oracle/_build/liblora_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.lora_oracle_threads.restype = ctypes.c_int
        lib.lora_oracle_set_threads.argtypes = [ctypes.c_int]
        lib.lora_oracle_route.restype = ctypes.c_int64
        lib.lora_oracle_route.argtypes = [ctypes.c_int64, ctypes.c_int32, _i32p, _i32p, _i32p]
        common = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _i32p, _i64p]
        lib.lora_oracle_shrink.argtypes = common + [_i32p, _f64p, _f64p, _f64p]
        lib.lora_oracle_expand.argtypes = common + [_f64p, _i32p, _f64p, _f64p, _f64p]
        lib.lora_oracle_dh.argtypes = common + [_f64p, _i32p, _f64p, _f64p, _f64p]
        lib.lora_oracle_db.argtypes = common + [_f64p, _i32p, _f64p, _f64p, _f64p]
        lib.lora_oracle_da.argtypes = common + [_i32p, _f64p, _f64p, _f64p]
        lib.lora_oracle_dx.argtypes = common + [_i32p, _f64p, _f64p, _f64p]
        lib.lora_oracle_adamw.argtypes = [ctypes.c_int32, ctypes.c_int32, _i32p, _i64p, _f64p, _i32p,
                                          ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                          _f64p, _f64p, _f64p, _f64p]
        lib.lora_oracle_base.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _f64p, _f64p, _f64p]
        for name in ("shrink", "expand", "dh", "db", "da", "dx", "adamw", "base"):
            getattr(lib, f"lora_oracle_{name}").restype = None
        _lib = lib
        return lib


def threads() -> int:
    """Number of OpenMP threads the oracle uses."""
    return int(_load().lora_oracle_threads())


def set_threads(n: int) -> None:
    _load().lora_oracle_set_threads(int(n))


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a, ptype):
    return a.ctypes.data_as(ptype)


class Table:
    """Per-adapter ranks, scales and row offsets (row_off[i] = sum_{j<i} r_j)."""

    def __init__(self, ranks, scales):
        self.rank = _c(ranks, np.int32)
        self.scale = _c(scales, np.float64)
        if self.rank.ndim != 1 or self.scale.shape != self.rank.shape:
            raise ValueError("ranks and scales must be 1-D of equal length")
        if np.any(self.rank < 1):
            raise ValueError("every rank must be >= 1")
        self.row_off = np.zeros(len(self.rank) + 1, dtype=np.int64)
        self.row_off[1:] = np.cumsum(self.rank, dtype=np.int64)

    @property
    def n(self) -> int:
        return int(len(self.rank))

    @property
    def sum_r(self) -> int:
        return int(self.row_off[-1])

    @property
    def r_max(self) -> int:
        return int(self.rank.max())


def route(ids, n_adapters: int):
    """Stable grouping of tokens by adapter: (perm, seg_start, n_bad)."""
    lib = _load()
    ids = _c(ids, np.int32)
    T = ids.shape[0]
    perm = np.full(T, -1, dtype=np.int32)
    seg_start = np.zeros(n_adapters + 1, dtype=np.int32)
    bad = lib.lora_oracle_route(T, n_adapters, _p(ids, _i32p), _p(perm, _i32p), _p(seg_start, _i32p))
    return perm[: seg_start[-1]].copy(), seg_start, int(bad)


def _hdr(tab: Table, T: int, d: int, r_max: int):
    return (T, tab.n, d, r_max, _p(tab.rank, _i32p), _p(tab.row_off, _i64p))


def shrink(tab: Table, ids, A, x, r_max: int | None = None):
    """H[T, r_max] with H[t, :r_i] = A_i x_t."""
    lib = _load()
    r_max = tab.r_max if r_max is None else r_max
    ids = _c(ids, np.int32)
    A = _c(A, np.float64)
    x = _c(x, np.float64)
    T, d_in = x.shape
    H = np.zeros((T, r_max), dtype=np.float64)
    lib.lora_oracle_shrink(*_hdr(tab, T, d_in, r_max), _p(ids, _i32p), _p(A, _f64p), _p(x, _f64p), _p(H, _f64p))
    return H


def expand(tab: Table, ids, B, H, y0):
    """y = y0 + s_i B_i h_t per token (y0 is copied, not modified).
    ``B`` is Bt_cat [sum_r, d_out] (B_i transposed, stacked like A)."""
    lib = _load()
    ids = _c(ids, np.int32)
    B = _c(B, np.float64)
    H = _c(H, np.float64)
    y = np.array(y0, dtype=np.float64, copy=True, order="C")
    T, d_out = y.shape
    lib.lora_oracle_expand(*_hdr(tab, T, d_out, H.shape[1]), _p(tab.scale, _f64p), _p(ids, _i32p),
                           _p(B, _f64p), _p(H, _f64p), _p(y, _f64p))
    return y


def dh(tab: Table, ids, B, dY, r_max: int | None = None):
    lib = _load()
    r_max = tab.r_max if r_max is None else r_max
    ids = _c(ids, np.int32)
    B = _c(B, np.float64)
    dY = _c(dY, np.float64)
    T, d_out = dY.shape
    out = np.zeros((T, r_max), dtype=np.float64)
    lib.lora_oracle_dh(*_hdr(tab, T, d_out, r_max), _p(tab.scale, _f64p), _p(ids, _i32p),
                       _p(B, _f64p), _p(dY, _f64p), _p(out, _f64p))
    return out


def db(tab: Table, ids, dY, H):
    lib = _load()
    ids = _c(ids, np.int32)
    dY = _c(dY, np.float64)
    H = _c(H, np.float64)
    T, d_out = dY.shape
    out = np.zeros((tab.sum_r, d_out), dtype=np.float64)
    lib.lora_oracle_db(*_hdr(tab, T, d_out, H.shape[1]), _p(tab.scale, _f64p), _p(ids, _i32p),
                       _p(dY, _f64p), _p(H, _f64p), _p(out, _f64p))
    return out


def da(tab: Table, ids, dH, X):
    lib = _load()
    ids = _c(ids, np.int32)
    dH = _c(dH, np.float64)
    X = _c(X, np.float64)
    T, d_in = X.shape
    out = np.zeros((tab.sum_r, d_in), dtype=np.float64)
    lib.lora_oracle_da(*_hdr(tab, T, d_in, dH.shape[1]), _p(ids, _i32p),
                       _p(dH, _f64p), _p(X, _f64p), _p(out, _f64p))
    return out


def dx(tab: Table, ids, A, dH, dX0):
    lib = _load()
    ids = _c(ids, np.int32)
    A = _c(A, np.float64)
    dH = _c(dH, np.float64)
    out = np.array(dX0, dtype=np.float64, copy=True, order="C")
    T, d_in = out.shape
    lib.lora_oracle_dx(*_hdr(tab, T, d_in, dH.shape[1]), _p(ids, _i32p),
                       _p(A, _f64p), _p(dH, _f64p), _p(out, _f64p))
    return out


def fwd(tab: Table, ids, A, B, x, y0, r_max: int | None = None):
    """Packed forward: (y, H) with H = shrink and y = y0 + expand(H)."""
    H = shrink(tab, ids, A, x, r_max)
    return expand(tab, ids, B, H, y0), H


def bwd(tab: Table, ids, A, B, X, H, dY, dX0, r_max: int | None = None):
    """Packed backward: (dH, dA, dB, dX) from saved H and incoming dY."""
    g = dh(tab, ids, B, dY, r_max if r_max is not None else H.shape[1])
    return g, da(tab, ids, g, X), db(tab, ids, dY, H), dx(tab, ids, A, g, dX0)


def adamw(tab: Table, w, g, m, v, lr, step, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
          weight_decay: float = 0.0):
    """One AdamW step per adapter over a [sum_r, d] weight matrix (rows of
    adapter i at tab.row_off[i]); returns the new (w, m, v) in fp64."""
    lib = _load()
    w = np.array(w, dtype=np.float64, copy=True, order="C")
    m = np.array(m, dtype=np.float64, copy=True, order="C")
    v = np.array(v, dtype=np.float64, copy=True, order="C")
    g = _c(g, np.float64)
    lr = _c(np.broadcast_to(np.asarray(lr, dtype=np.float64), (tab.n,)), np.float64)
    step = _c(np.broadcast_to(np.asarray(step, dtype=np.int32), (tab.n,)), np.int32)
    d = w.shape[1]
    lib.lora_oracle_adamw(tab.n, d, _p(tab.rank, _i32p), _p(tab.row_off, _i64p),
                          _p(lr, _f64p), _p(step, _i32p), beta1, beta2, eps, weight_decay, _p(w, _f64p), _p(g, _f64p),
                          _p(m, _f64p), _p(v, _f64p))
    return w, m, v


def base(W, x):
    """Base projection y = x W^T (W is [d_out, d_in], x is [T, d_in])."""
    lib = _load()
    W = _c(W, np.float64)
    x = _c(x, np.float64)
    T, d_in = x.shape
    d_out = W.shape[0]
    assert W.shape[1] == d_in
    y = np.zeros((T, d_out), dtype=np.float64)
    lib.lora_oracle_base(T, d_in, d_out, _p(W, _f64p), _p(x, _f64p), _p(y, _f64p))
    return y


def base_lora_fwd(tab: Table, ids, W, A, B, x, r_max: int | None = None):
    """A LoRA layer's forward: (y, H) with H = shrink(x) and
    y = x W^T + expand(H), i.e. the base projection plus the delta."""
    return fwd(tab, ids, A, B, x, base(W, x), r_max)
