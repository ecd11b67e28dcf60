"""CPU-only checks of the C ABI: the library builds for sm_103a, loads, exports
every entry point include/lora_sgmv.h declares, and rejects bad arguments on
the host before any CUDA call.  Nothing here runs a kernel."""
import ctypes
import os
import re
import subprocess

import pytest

import adapter_sgmv_gb300 as lora

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora_sgmv.h")


@pytest.fixture(scope="module")
def L():
    lora.build_library()
    return lora.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z_]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("lora_sgmv_shrink", "lora_sgmv_expand", "lora_packed_fwd", "lora_packed_bwd",
              "lora_build_segments"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", lora.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = sorted(set(re.findall(r"\bT (lora_\w+)", out)))
    assert exported == names, (exported, names)
    assert set(lora.SIGNATURES) == set(names)


def test_debug_build_exports_the_same_symbols(L):
    # the device-side index checks are a compile-time switch: same sources, same ABI
    path = lora.build_library(debug=True)
    D = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(D, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    assert sorted(set(re.findall(r"\bT (lora_\w+)", out))) == declared_functions()
    D.lora_debug_checks.restype = ctypes.c_int32
    assert D.lora_debug_checks() == 1
    assert L.lora_debug_checks() == 0
    assert lora.lora_debug_checks() is False


def test_version_and_status_strings(L):
    assert lora.lora_abi_version() == 2
    for code, name in lora.STATUS.items():
        assert lora.lora_status_string(code) == name
    assert lora.lora_status_string(999) == "LORA_ERR_UNKNOWN"


def test_segment_storage_sizes(L):
    a = lora.lora_segments_bytes(256, 8)
    b = lora.lora_segments_bytes(16384, 32)
    assert 0 < a < b
    assert a % 256 == 0
    assert lora.lora_segments_bytes(0, 1) > 0
    assert lora.lora_segments_bytes(-1, 4) == 0
    assert lora.lora_segments_bytes(10, 0) == 0
    assert lora.lora_segments_bytes(10, 70000) == 0


def fake_table(**kw):
    f = dict(n_adapters=4, d_in=256, d_out=256, r_max=16, sum_r=36, reserved=0,
             rank=0x10000, row_off=0x20000, scale=0x30000, A=0x40000, B=0x50000)
    f.update(kw)
    return lora.c_table(*[f[k] for k, _ in lora.c_table._fields_])


def test_workspace_bytes_and_table_checks(L):
    t = fake_table()
    n = L.lora_workspace_bytes(ctypes.byref(t), 64)
    assert n >= 2 * 64 * 16 * 4
    for bad in (dict(d_in=12), dict(d_out=0), dict(r_max=129), dict(r_max=0), dict(n_adapters=0),
                dict(sum_r=8), dict(A=0), dict(B=0x50008)):
        tb = fake_table(**bad)
        assert L.lora_workspace_bytes(ctypes.byref(tb), 64) == 0, bad


def fake_segs(**kw):
    f = dict(n_tokens=64, n_adapters=4, max_tiles=5, sorted=1, perm=0x1000, seg_start=0x2000, tiles=0x3000,
             n_tiles=0x4000, status=0x5000, scratch=0x6000, scratch_words=0, max_spans=5, reserved=0,
             spans=0x7000, n_spans=0x8000)
    f.update(kw)
    return lora.c_segments(*[f[k] for k, _ in lora.c_segments._fields_])


def test_host_side_rejections_return_before_any_cuda_call(L):
    segs = lora.c_segments()
    # no storage / no output struct
    assert L.lora_build_segments(None, None, 4, 2, None, 0, ctypes.byref(segs), None) == 1
    # both ids and offsets given
    assert L.lora_build_segments(0x1000, 0x2000, 4, 2, 0x3000, 1 << 20, ctypes.byref(segs), None) == 1
    # misaligned storage
    assert L.lora_build_segments(0x1000, None, 4, 2, 0x3008, 1 << 20, ctypes.byref(segs), None) == 3
    # storage too small
    assert L.lora_build_segments(0x1000, None, 4, 2, 0x3000, 16, ctypes.byref(segs), None) == 5
    t = fake_table()
    s = fake_segs()
    assert L.lora_sgmv_shrink(None, 0x1000, ctypes.byref(t), ctypes.byref(s), None) == 1
    assert L.lora_sgmv_shrink(0x1004, 0x1000, ctypes.byref(t), ctypes.byref(s), None) == 3
    assert L.lora_sgmv_expand(0x1000, 0x2000, None, ctypes.byref(s), None) == 1
    s_bad = fake_segs(n_adapters=3)
    assert L.lora_sgmv_expand(0x1000, 0x2000, ctypes.byref(t), ctypes.byref(s_bad), None) == 2
    assert L.lora_packed_fwd(0x1000, None, 0x2000, ctypes.byref(t), ctypes.byref(s), None, 0, None) == 5
    assert L.lora_packed_bwd(None, None, None, 0x1000, 0x2000, None, ctypes.byref(t), ctypes.byref(s),
                             0x3000, 16, None) == 5
    assert L.lora_packed_bwd(None, None, None, None, 0x2000, None, ctypes.byref(t), ctypes.byref(s),
                             0x3000, 1 << 20, None) == 1
    assert L.lora_query_status(None, None) == 1
    # segments missing a pointer the kernels read on the device, or with a
    # negative capacity: rejected on the host by every entry point
    for bad, code in ((dict(n_tiles=0), 1), (dict(spans=0), 1), (dict(n_spans=0), 1), (dict(status=0), 1),
                      (dict(max_tiles=-1), 2), (dict(max_spans=-1), 2), (dict(tiles=0x3008), 3)):
        sb = fake_segs(**bad)
        assert L.lora_sgmv_shrink(0x1000, 0x1000, ctypes.byref(t), ctypes.byref(sb), None) == code, bad
        assert L.lora_packed_fwd(0x1000, None, 0x2000, ctypes.byref(t), ctypes.byref(sb), 0x3000, 1 << 20,
                                 None) == code, bad
        assert L.lora_packed_bwd(None, None, None, 0x1000, 0x2000, None, ctypes.byref(t), ctypes.byref(sb),
                                 0x3000, 1 << 20, None) == code, bad
    assert L.lora_check_wait_timeout(None, None) == 1
    assert L.lora_check_wait_timeout(0x1002, None) == 3


def test_noalloc_backward_checks_its_arguments_like_the_workspace_backward(L):
    """The entry point without a workspace makes the same host-side checks as
    lora_packed_bwd, in the same order: a malformed table or segment struct is
    a status code, never a launch that dereferences it on the device."""
    t = fake_table()
    s = fake_segs()
    call = lambda tb, sg, dY=0x1000, X=0x2000, dX=None: L.lora_packed_bwd_noalloc(
        dX, None, None, dY, X, None, ctypes.byref(tb) if tb is not None else None,
        ctypes.byref(sg) if sg is not None else None, None)
    ws_call = lambda tb, sg, dY=0x1000, X=0x2000, dX=None: L.lora_packed_bwd(
        dX, None, None, dY, X, None, ctypes.byref(tb) if tb is not None else None,
        ctypes.byref(sg) if sg is not None else None, 0x3000, 1 << 20, None)
    cases = [(None, s, {}), (t, None, {}),
             (fake_table(rank=0), s, {}), (fake_table(row_off=0x20002), s, {}), (fake_table(scale=0x30001), s, {}),
             (fake_table(d_in=12), s, {}), (fake_table(sum_r=8), s, {}),
             (t, fake_segs(n_tiles=0), {}), (t, fake_segs(seg_start=0), {}), (t, fake_segs(spans=0), {}),
             (t, fake_segs(max_tiles=-1), {}), (t, fake_segs(max_spans=-1), {}), (t, fake_segs(n_adapters=3), {}),
             (t, fake_segs(n_tokens=-1), {}), (t, fake_segs(perm=0x1002), {}),
             (t, s, dict(dY=None)), (t, s, dict(X=0x2008)), (t, s, dict(dX=0x4004))]
    for tb, sg, kw in cases:
        got = call(tb, sg, **kw)
        assert got in (1, 2, 3), (tb, sg, kw, got)
        assert got == ws_call(tb, sg, **kw), (tb, sg, kw)


def test_binding_fails_loudly_without_the_library():
    with pytest.raises(RuntimeError):
        lora._lib = None
        try:
            lora.lib(path="/nonexistent/liblora_sgmv.so")
        finally:
            lora._lib = None


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "adapter_sgmv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "lora_oracle" not in src, f
