"""Python binding of ``liblora_sgmv.so``, the GB300 multi-adapter LoRA delta library.

Argument marshalling only: every function here forwards torch tensors' device
pointers and the current CUDA stream to the C ABI declared in
``include/lora_sgmv.h`` and raises ``LoraError`` on a non-OK status.  All
arithmetic runs in the library's CUDA kernels; there is no CPU path.  The
functions carry the C names:

    lora_build_segments, lora_sgmv_shrink, lora_sgmv_expand,
    lora_packed_fwd, lora_packed_bwd, lora_query_status, ...

PyTorch provides device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

from ._build import DEBUG_LIB_PATH, LIB_PATH, build as build_library  # noqa: F401

__all__ = [
    "LoraError", "AdapterTable", "Segments", "lib", "lora_abi_version", "lora_status_string",
    "lora_segments_bytes", "lora_build_segments", "lora_workspace_bytes", "lora_sgmv_shrink",
    "lora_sgmv_expand", "lora_packed_fwd", "lora_packed_bwd", "lora_packed_bwd_concurrent", "lora_packed_bwd_ex", "SideStreams",
    "LORA_BWD_DETERMINISTIC",
    "lora_packed_fwd_marked", "lora_packed_bwd_marked",
    "lora_packed_bwd_noalloc", "lora_adamw_step", "lora_fused_base_workspace_bytes", "lora_fused_base_fwd",
    "lora_multi_workspace_bytes", "lora_multi_fwd", "lora_plan_pack",
    "lora_query_status", "lora_reset_status", "lora_check_wait_timeout", "lora_debug_checks",
    "lora_query_index_check",
    "STATUS",
]

STATUS = {
    0: "LORA_OK", 1: "LORA_ERR_INVALID_ARG", 2: "LORA_ERR_SHAPE", 3: "LORA_ERR_ALIGNMENT",
    4: "LORA_ERR_BAD_ADAPTER_ID", 5: "LORA_ERR_WORKSPACE_TOO_SMALL", 6: "LORA_ERR_UNSUPPORTED",
    7: "LORA_ERR_TIMEOUT", 8: "LORA_ERR_BAD_TABLE", 9: "LORA_ERR_BAD_SEGMENTS", 10: "LORA_ERR_CUDA",
    11: "LORA_ERR_INDEX",
}


class LoraError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)}")


class c_table(ctypes.Structure):
    _fields_ = [("n_adapters", ctypes.c_int32), ("d_in", ctypes.c_int32), ("d_out", ctypes.c_int32),
                ("r_max", ctypes.c_int32), ("sum_r", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("rank", ctypes.c_void_p), ("row_off", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("A", ctypes.c_void_p), ("B", ctypes.c_void_p)]


class c_segments(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int32), ("n_adapters", ctypes.c_int32), ("max_tiles", ctypes.c_int32),
                ("sorted", ctypes.c_int32), ("perm", ctypes.c_void_p), ("seg_start", ctypes.c_void_p),
                ("tiles", ctypes.c_void_p), ("n_tiles", ctypes.c_void_p), ("status", ctypes.c_void_p),
                ("scratch", ctypes.c_void_p), ("scratch_words", ctypes.c_int64), ("max_spans", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("spans", ctypes.c_void_p), ("n_spans", ctypes.c_void_p)]


class c_side_streams(ctypes.Structure):
    _fields_ = [("stream", ctypes.c_void_p * 2), ("event", ctypes.c_void_p * 4)]


class c_plan_config(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32), ("tokens_per_step", ctypes.c_int32), ("steps", ctypes.c_int64),
                ("mem_bytes", ctypes.c_int64)]


class c_plan_cost(ctypes.Structure):
    _fields_ = [("step_overhead_s", ctypes.c_double), ("base_s_per_token", ctypes.c_double),
                ("lora_s_per_token", ctypes.c_double), ("lora_s_per_token_rank", ctypes.c_double),
                ("gpu_mem_bytes", ctypes.c_int64), ("job_mem_bytes", ctypes.c_int64),
                ("mem_unit_bytes", ctypes.c_int64), ("n_gpus", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class c_plan_job(ctypes.Structure):
    _fields_ = [("gpu", ctypes.c_int32), ("n_configs", ctypes.c_int32), ("start_s", ctypes.c_double),
                ("duration_s", ctypes.c_double), ("step_s", ctypes.c_double)]


_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t

# name -> (restype, argtypes), mirrors include/lora_sgmv.h
SIGNATURES = {
    "lora_abi_version": (_I32, []),
    "lora_status_string": (ctypes.c_char_p, [_I32]),
    "lora_segments_bytes": (_SZ, [_I32, _I32]),
    "lora_build_segments": (_I32, [_P, _P, _I32, _I32, _P, _SZ, ctypes.POINTER(c_segments), _P]),
    "lora_workspace_bytes": (_SZ, [ctypes.POINTER(c_table), _I32]),
    "lora_sgmv_shrink": (_I32, [_P, _P, ctypes.POINTER(c_table), ctypes.POINTER(c_segments), _P]),
    "lora_sgmv_expand": (_I32, [_P, _P, ctypes.POINTER(c_table), ctypes.POINTER(c_segments), _P]),
    "lora_packed_fwd": (_I32, [_P, _P, _P, ctypes.POINTER(c_table), ctypes.POINTER(c_segments), _P, _SZ, _P]),
    "lora_packed_bwd": (_I32, [_P, _P, _P, _P, _P, _P, ctypes.POINTER(c_table), ctypes.POINTER(c_segments),
                               _P, _SZ, _P]),
    "lora_side_streams_create": (_I32, [ctypes.POINTER(c_side_streams)]),
    "lora_side_streams_destroy": (_I32, [ctypes.POINTER(c_side_streams)]),
    "lora_packed_bwd_ex": (_I32, [_P, _P, _P, _P, _P, _P, ctypes.POINTER(c_table), ctypes.POINTER(c_segments), _P,
                                  _SZ, ctypes.POINTER(c_side_streams), ctypes.c_uint32, _P]),
    "lora_packed_bwd_concurrent": (_I32, [_P, _P, _P, _P, _P, _P, ctypes.POINTER(c_table),
                                          ctypes.POINTER(c_segments), _P, _SZ, ctypes.POINTER(c_side_streams), _P]),
    "lora_packed_fwd_marked": (_I32, [_P, _P, _P, ctypes.POINTER(c_table), ctypes.POINTER(c_segments), _P, _SZ,
                                      _P, ctypes.POINTER(_P), _I32, ctypes.POINTER(_I32)]),
    "lora_packed_bwd_marked": (_I32, [_P, _P, _P, _P, _P, _P, ctypes.POINTER(c_table), ctypes.POINTER(c_segments),
                                      _P, _SZ, _P, ctypes.POINTER(_P), _I32, ctypes.POINTER(_I32)]),
    "lora_packed_bwd_noalloc": (_I32, [_P, _P, _P, _P, _P, _P, ctypes.POINTER(c_table),
                                       ctypes.POINTER(c_segments), _P]),
    "lora_adamw_step": (_I32, [ctypes.POINTER(c_table), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_float,
                                ctypes.c_float, ctypes.c_float, ctypes.c_float, _P]),
    "lora_multi_workspace_bytes": (_SZ, [_I32, ctypes.POINTER(c_table), _I32]),
    "lora_multi_fwd": (_I32, [_I32, ctypes.POINTER(_P), ctypes.POINTER(_P), _P, ctypes.POINTER(c_table),
                              ctypes.POINTER(c_segments), _P, _SZ, _P]),
    "lora_fused_base_workspace_bytes": (_SZ, [ctypes.POINTER(c_table), _I32]),
    "lora_fused_base_fwd": (_I32, [_P, _P, _P, _P, ctypes.POINTER(c_table), ctypes.POINTER(c_segments), _P, _SZ,
                                   _P]),
    "lora_plan_pack": (_I32, [ctypes.POINTER(c_plan_config), _I32, ctypes.POINTER(c_plan_cost),
                              ctypes.POINTER(_I32), ctypes.POINTER(c_plan_job), ctypes.POINTER(_I32),
                              ctypes.POINTER(ctypes.c_double)]),
    "lora_query_status": (_I32, [ctypes.POINTER(c_segments), _P]),
    "lora_query_index_check": (_I32, [ctypes.POINTER(c_segments), _P, ctypes.POINTER(_I32)]),
    "lora_debug_checks": (_I32, []),
    "lora_reset_status": (_I32, [ctypes.POINTER(c_segments), _P]),
    "lora_check_wait_timeout": (_I32, [_P, _P]),
}


def lib(path: str | None = None):
    """Load the CUDA library (it must have been built: ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("LORA_SGMV_LIB", LIB_PATH)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first (python -c "
                           "'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(st: int, where: str):
    if st != 0:
        raise LoraError(st, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def lora_abi_version() -> int:
    return int(lib().lora_abi_version())


def lora_status_string(st: int) -> str:
    return lib().lora_status_string(int(st)).decode()


def lora_segments_bytes(n_tokens: int, n_adapters: int) -> int:
    return int(lib().lora_segments_bytes(int(n_tokens), int(n_adapters)))


class AdapterTable:
    """Device-resident stacked adapter table (keeps its tensors alive).

    ``A``: bf16 [sum_r, d_in] (A_i stacked); ``B``: bf16 [sum_r, d_out]
    (B_i transposed, stacked the same way: row row_off[i] + k = column k of B_i);
    ``ranks`` / ``scales``: per-adapter rank and s_i = alpha_i / r_i."""

    def __init__(self, A, B, ranks, scales, d_in: int, d_out: int):
        import torch

        dev = A.device
        ranks = [int(r) for r in ranks]
        self.rank = torch.tensor(ranks, dtype=torch.int32, device=dev)
        off = [0]
        for r in ranks:
            off.append(off[-1] + r)
        self.row_off = torch.tensor(off, dtype=torch.int32, device=dev)
        self.scale = torch.as_tensor(scales, dtype=torch.float32).to(dev)
        self.A = A
        self.B = B
        self.ranks = ranks
        self.d_in, self.d_out = int(d_in), int(d_out)
        self.c = c_table(len(ranks), self.d_in, self.d_out, max(ranks), off[-1], 0,
                         self.rank.data_ptr(), self.row_off.data_ptr(), self.scale.data_ptr(),
                         A.data_ptr(), B.data_ptr())

    @property
    def n_adapters(self):
        return self.c.n_adapters

    @property
    def r_max(self):
        return self.c.r_max

    @property
    def sum_r(self):
        return self.c.sum_r


class Segments:
    """Routing metadata of one batch; owns its device storage."""

    def __init__(self, storage, c: c_segments):
        self.storage = storage
        self.c = c

    def _i32(self, attr, n):
        import torch

        base = self.storage.data_ptr()
        off = (getattr(self.c, attr) - base) // 4
        return self.storage.view(torch.int32)[off:off + n]

    @property
    def perm(self):
        return self._i32("perm", self.c.n_tokens)

    @property
    def seg_start(self):
        return self._i32("seg_start", self.c.n_adapters + 1)

    @property
    def n_tiles(self):
        return self._i32("n_tiles", 1)

    @property
    def tiles(self):
        return self._i32("tiles", 4 * self.c.max_tiles).view(-1, 4)

    @property
    def n_spans(self):
        return self._i32("n_spans", 1)

    @property
    def spans(self):
        return self._i32("spans", 4 * self.c.max_spans).view(-1, 4)


def lora_build_segments(ids=None, seg_offsets=None, n_tokens=None, n_adapters=None, device=None,
                        stream=None, storage=None) -> Segments:
    """Build routing metadata from per-token ``ids`` (int32 [T], any order) or
    sorted ``seg_offsets`` (int32 [N+1])."""
    import torch

    src = ids if ids is not None else seg_offsets
    if n_tokens is None:
        n_tokens = int(ids.numel()) if ids is not None else int(seg_offsets[-1].item())
    if device is None:
        device = src.device if src is not None else torch.device("cuda")
    nbytes = lora_segments_bytes(n_tokens, n_adapters)
    if nbytes == 0:
        raise LoraError(2, "lora_segments_bytes")
    if storage is None:
        storage = torch.empty(nbytes, dtype=torch.uint8, device=device)
    c = c_segments()
    st = lib().lora_build_segments(_ptr(ids), _ptr(seg_offsets), int(n_tokens), int(n_adapters),
                                   _ptr(storage), storage.numel(), ctypes.byref(c), _stream(stream))
    _check(st, "lora_build_segments")
    return Segments(storage, c)


def lora_workspace_bytes(table: AdapterTable, n_tokens: int) -> int:
    return int(lib().lora_workspace_bytes(ctypes.byref(table.c), int(n_tokens)))


def workspace(table: AdapterTable, n_tokens: int, device=None):
    import torch

    n = lora_workspace_bytes(table, n_tokens)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or table.A.device)


def lora_sgmv_shrink(H, x, table: AdapterTable, segs: Segments, stream=None):
    _check(lib().lora_sgmv_shrink(_ptr(H), _ptr(x), ctypes.byref(table.c), ctypes.byref(segs.c),
                                  _stream(stream)), "lora_sgmv_shrink")
    return H


def lora_sgmv_expand(y, H, table: AdapterTable, segs: Segments, stream=None):
    _check(lib().lora_sgmv_expand(_ptr(y), _ptr(H), ctypes.byref(table.c), ctypes.byref(segs.c),
                                  _stream(stream)), "lora_sgmv_expand")
    return y


def lora_packed_fwd(y, H_save, x, table: AdapterTable, segs: Segments, ws=None, stream=None):
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().lora_packed_fwd(_ptr(y), _ptr(H_save), _ptr(x), ctypes.byref(table.c), ctypes.byref(segs.c),
                                 _ptr(ws), wsb, _stream(stream)), "lora_packed_fwd")
    return y


def lora_packed_bwd(dX, dA, dB, dY, X, H_saved, table: AdapterTable, segs: Segments, ws, stream=None):
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().lora_packed_bwd(_ptr(dX), _ptr(dA), _ptr(dB), _ptr(dY), _ptr(X), _ptr(H_saved),
                                 ctypes.byref(table.c), ctypes.byref(segs.c), _ptr(ws), wsb, _stream(stream)),
           "lora_packed_bwd")


class SideStreams:
    """Two CUDA streams and four events owned by the caller, on which
    lora_packed_bwd_concurrent runs dB and dA beside dh and dX; made on the
    current device by lora_side_streams_create (fresh streams, so they never
    coincide with a stream torch hands out) and released when the object is
    collected.  One set per host thread that runs backward calls at the same
    time."""

    def __init__(self, device=None):
        import torch

        self.c = c_side_streams()
        with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
            _check(lib().lora_side_streams_create(ctypes.byref(self.c)), "lora_side_streams_create")

    def __del__(self):
        if getattr(self, "c", None) is not None and _lib is not None:
            _lib.lora_side_streams_destroy(ctypes.byref(self.c))
            self.c = None


def lora_packed_bwd_concurrent(dX, dA, dB, dY, X, H_saved, table: AdapterTable, segs: Segments, ws,
                               side: SideStreams, stream=None):
    """lora_packed_bwd with dB and dA on the caller's side streams (same results)."""
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().lora_packed_bwd_concurrent(_ptr(dX), _ptr(dA), _ptr(dB), _ptr(dY), _ptr(X), _ptr(H_saved),
                                            ctypes.byref(table.c), ctypes.byref(segs.c), _ptr(ws), wsb,
                                            ctypes.byref(side.c), _stream(stream)), "lora_packed_bwd_concurrent")


LORA_BWD_DETERMINISTIC = 1


def lora_packed_bwd_ex(dX, dA, dB, dY, X, H_saved, table: AdapterTable, segs: Segments, ws, side=None,
                       deterministic=False, stream=None):
    """Packed backward with options: dB / dA on the caller's side streams
    (``side``: SideStreams) and/or dA / dB summed in a fixed span order
    (``deterministic``: bit-identical from run to run)."""
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().lora_packed_bwd_ex(_ptr(dX), _ptr(dA), _ptr(dB), _ptr(dY), _ptr(X), _ptr(H_saved),
                                    ctypes.byref(table.c), ctypes.byref(segs.c), _ptr(ws), wsb,
                                    None if side is None else ctypes.byref(side.c),
                                    LORA_BWD_DETERMINISTIC if deterministic else 0, _stream(stream)),
           "lora_packed_bwd_ex")


def _events(events, stream):
    """ctypes array of the cudaEvent_t handles of torch.cuda.Event objects
    (an event that was never recorded is recorded once so that it exists)."""
    import torch

    for e in events:
        if e.cuda_event == 0:
            e.record(stream if stream is not None else torch.cuda.current_stream())
    return (_P * max(1, len(events)))(*[e.cuda_event for e in events])


def lora_packed_fwd_marked(y, H_save, x, table: AdapterTable, segs: Segments, ws, events, stream=None) -> int:
    """lora_packed_fwd recording ``events`` (torch.cuda.Event) around its
    kernels: events[2k] before and events[2k + 1] after kernel k.  Returns the
    number of events recorded."""
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    arr = _events(events, stream)
    n = ctypes.c_int32(0)
    _check(lib().lora_packed_fwd_marked(_ptr(y), _ptr(H_save), _ptr(x), ctypes.byref(table.c), ctypes.byref(segs.c),
                                        _ptr(ws), wsb, _stream(stream), arr, len(events), ctypes.byref(n)),
           "lora_packed_fwd_marked")
    return int(n.value)


def lora_packed_bwd_marked(dX, dA, dB, dY, X, H_saved, table: AdapterTable, segs: Segments, ws, events,
                           stream=None) -> int:
    """lora_packed_bwd recording ``events`` around its kernels (see
    lora_packed_fwd_marked).  Returns the number of events recorded."""
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    arr = _events(events, stream)
    n = ctypes.c_int32(0)
    _check(lib().lora_packed_bwd_marked(_ptr(dX), _ptr(dA), _ptr(dB), _ptr(dY), _ptr(X), _ptr(H_saved),
                                        ctypes.byref(table.c), ctypes.byref(segs.c), _ptr(ws), wsb, _stream(stream),
                                        arr, len(events), ctypes.byref(n)),
           "lora_packed_bwd_marked")
    return int(n.value)


def lora_packed_bwd_noalloc(dX, dA, dB, dY, X, H_saved, table: AdapterTable, segs: Segments, stream=None):
    """lora_packed_bwd with its scratch in the library's fixed device array
    (no workspace argument; for callers that cannot allocate)."""
    _check(lib().lora_packed_bwd_noalloc(_ptr(dX), _ptr(dA), _ptr(dB), _ptr(dY), _ptr(X), _ptr(H_saved),
                                         ctypes.byref(table.c), ctypes.byref(segs.c), _stream(stream)),
           "lora_packed_bwd_noalloc")


def lora_adamw_step(table: AdapterTable, wA, wB, gA, gB, mA, vA, mB, vB, lr, step, beta1=0.9, beta2=0.999,
                    eps=1e-8, weight_decay=0.0, stream=None):
    """One AdamW step per adapter (lr: fp32 [N], step: int32 [N] device
    tensors); also rewrites the table's bf16 A / B from the new masters."""
    _check(lib().lora_adamw_step(ctypes.byref(table.c), _ptr(wA), _ptr(wB), _ptr(gA), _ptr(gB), _ptr(mA), _ptr(vA),
                                 _ptr(mB), _ptr(vB), _ptr(lr), _ptr(step), beta1, beta2, eps, weight_decay,
                                 _stream(stream)), "lora_adamw_step")


def _tables(tables):
    return (c_table * len(tables))(*[t.c for t in tables])


def lora_multi_workspace_bytes(tables, n_tokens: int) -> int:
    """Workspace of lora_multi_fwd for these AdapterTables and T tokens."""
    return int(lib().lora_multi_workspace_bytes(len(tables), _tables(tables), int(n_tokens)))


def lora_multi_fwd(ys, H_saves, x, tables, segs: Segments, ws, stream=None):
    """Packed forward of len(tables) projections sharing x (one y / table per
    projection; H_saves: None or a list with None entries allowed)."""
    n = len(tables)
    if len(ys) != n or (H_saves is not None and len(H_saves) != n):
        raise ValueError("one y (and H_save) per table")
    y_arr = (_P * n)(*[_ptr(y) for y in ys])
    h_arr = None if H_saves is None else (_P * n)(*[_ptr(h) for h in H_saves])
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().lora_multi_fwd(n, y_arr, h_arr, _ptr(x), _tables(tables), ctypes.byref(segs.c), _ptr(ws), wsb,
                                _stream(stream)), "lora_multi_fwd")
    return ys


def lora_fused_base_workspace_bytes(table: AdapterTable, n_tokens: int) -> int:
    return int(lib().lora_fused_base_workspace_bytes(ctypes.byref(table.c), int(n_tokens)))


def lora_fused_base_fwd(y, H_save, x, W, table: AdapterTable, segs: Segments, ws, stream=None):
    """y = x W^T + the packed LoRA delta, in one launch (segment-sorted batch;
    H_save may be None).  ws: at least lora_fused_base_workspace_bytes bytes."""
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().lora_fused_base_fwd(_ptr(y), _ptr(H_save), _ptr(x), _ptr(W), ctypes.byref(table.c),
                                     ctypes.byref(segs.c), _ptr(ws), wsb, _stream(stream)), "lora_fused_base_fwd")
    return y


def lora_plan_pack(configs, cost: dict) -> dict:
    """Packing planner (host).  configs: sequence of dicts with rank,
    tokens_per_step, steps, mem_bytes; cost: dict with the lora_plan_cost
    fields.  Returns {"job_of": [...], "jobs": [{gpu, n_configs, start_s,
    duration_s, step_s}, ...], "makespan_s": float}."""
    n = len(configs)
    arr = (c_plan_config * n)(*[c_plan_config(int(c["rank"]), int(c["tokens_per_step"]), int(c["steps"]),
                                              int(c["mem_bytes"])) for c in configs])
    cc = c_plan_cost(float(cost.get("step_overhead_s", 0.0)), float(cost.get("base_s_per_token", 0.0)),
                     float(cost.get("lora_s_per_token", 0.0)), float(cost.get("lora_s_per_token_rank", 0.0)),
                     int(cost["gpu_mem_bytes"]), int(cost.get("job_mem_bytes", 0)),
                     int(cost.get("mem_unit_bytes", 1 << 20)), int(cost.get("n_gpus", 1)), 0)
    job_of = (_I32 * n)()
    jobs = (c_plan_job * n)()
    nj = _I32(0)
    mk = ctypes.c_double(0.0)
    _check(lib().lora_plan_pack(arr, n, ctypes.byref(cc), job_of, jobs, ctypes.byref(nj), ctypes.byref(mk)),
           "lora_plan_pack")
    return {"job_of": list(job_of), "makespan_s": mk.value,
            "jobs": [{"gpu": j.gpu, "n_configs": j.n_configs, "start_s": j.start_s, "duration_s": j.duration_s,
                      "step_s": j.step_s} for j in jobs[:nj.value]]}


def lora_query_status(segs: Segments, stream=None) -> int:
    return int(lib().lora_query_status(ctypes.byref(segs.c), _stream(stream)))


def lora_debug_checks() -> bool:
    """True when the loaded library is the debug build (device-side index checks)."""
    return bool(lib().lora_debug_checks())


def lora_query_index_check(segs: Segments, stream=None) -> tuple[int, int]:
    """(status, where): the status word and, after LORA_ERR_INDEX in the debug
    build, the failed check's source file number << 16 | line."""
    where = _I32(0)
    st = int(lib().lora_query_index_check(ctypes.byref(segs.c), _stream(stream), ctypes.byref(where)))
    return st, int(where.value)


def lora_reset_status(segs: Segments, stream=None):
    _check(lib().lora_reset_status(ctypes.byref(segs.c), _stream(stream)), "lora_reset_status")


def lora_check_wait_timeout(status, stream=None):
    """Run the bounded pipeline wait against a barrier nothing completes; the
    device int32 tensor ``status`` receives LORA_ERR_TIMEOUT (7) after ~2 s."""
    _check(lib().lora_check_wait_timeout(_ptr(status), _stream(stream)), "lora_check_wait_timeout")
