"""The debug build (liblora_sgmv_debug.so, device-side index checks).

A child process loads the debug build and runs every entry point on the
tiny batch and on ragged batches (an empty adapter, a one-token adapter, an
adapter of three spans, sorted and id-routed, a decode-sized one): the
status word must stay clean, and every output must be bit-identical to the
release build's on the same inputs (the checks change no arithmetic) and
within tolerance of the fp64 oracle.  Then one perm entry is set past T (the
buffers have spare rows there, so nothing leaves its allocation even
unchecked): the checks must report LORA_ERR_INDEX, and where."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import adapter_sgmv_gb300 as lora
import debug_cases as dc
import workloads as wl
from lora_testlib import FWD_TOL, GRAD_TOL, assert_close, check_blocks, oracle_all

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
LORA_ERR_INDEX = 11
FILE_NUMBER = {"route.cu": 1, "tc_rowproj.cu": 2, "tc_colproj.cu": 3, "tc_tokred.cu": 4, "decode.cu": 5,
               "tc_base.cu": 6}


@pytest.fixture(scope="module")
def debug_run(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    path = lora.build_library(debug=True)
    out = tmp_path_factory.mktemp("debug_build")
    env = dict(os.environ, LORA_SGMV_LIB=path)
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_cases.py"), str(out)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout[-4000:], r.stderr[-4000:])
    with open(out / "summary.json") as f:
        return out, json.load(f)


def test_debug_build_is_clean_and_bit_identical_to_release(debug_run):
    out, summary = debug_run
    assert summary["debug_checks"]
    lora.build_library()
    assert not lora.lora_debug_checks()
    for name, spec in dc.specs().items():
        assert summary["cases"][name] == {"status": 0, "where": 0}, name
        host = wl.host_inputs(spec)
        rel, st, where = dc.run_case(spec, host)
        assert (st, where) == (0, 0), name
        dbg = np.load(out / f"{name}.npz")
        assert sorted(dbg.files) == sorted(rel), name
        for k, v in rel.items():
            assert np.array_equal(dbg[k], v, equal_nan=True), f"{name}: {k} differs between debug and release"
        # the debug build's outputs against the oracle
        ref = oracle_all(spec, host)
        bf = lambda a: (a.astype(np.int32) << 16).view(np.float32).astype(np.float64)
        assert_close(bf(dbg["y"]), ref["y"], FWD_TOL, f"{name}: y")
        assert_close(dbg["H"], ref["H"], FWD_TOL, f"{name}: H")
        for tag in ("ord", "ord_recompute"):
            assert_close(bf(dbg[f"dX_{tag}"]), ref["dX"], GRAD_TOL, f"{name}: dX_{tag}")
            check_blocks(spec, dbg[f"dA_{tag}"].astype(np.float64), dbg[f"dB_{tag}"].astype(np.float64),
                         ref["dA"], ref["dB"], adapters=[i for i in range(spec.n_adapters)
                                                         if np.any(spec.ids == i)])
        assert_close(bf(dbg["y_multi0"]), ref["y"], FWD_TOL, f"{name}: y of the first projection")


def test_debug_build_reports_a_bad_perm_entry(debug_run):
    _, summary = debug_run
    c = summary["corrupted"]
    # decode-sized batch: the decode shrink finds it first; the backward's
    # first reader of perm is the bf16 copy of H (tc_rowproj.cu)
    st, where = c["decode_ids"]["fwd"]
    assert st == LORA_ERR_INDEX and where >> 16 == FILE_NUMBER["decode.cu"] and where & 0xffff > 0, (st, where)
    st, where = c["decode_ids"]["bwd"]
    assert st == LORA_ERR_INDEX and where >> 16 == FILE_NUMBER["tc_rowproj.cu"], (st, where)
    # packed batch of few tiles (case i split along d, two launches): the shrink reads perm first
    st, where = c["ragged_ids"]["fwd"]
    assert st == LORA_ERR_INDEX and where >> 16 == FILE_NUMBER["tc_rowproj.cu"] and where & 0xffff > 0, (st, where)
    st, where = c["ragged_ids"]["bwd"]
    assert st == LORA_ERR_INDEX and where >> 16 == FILE_NUMBER["tc_rowproj.cu"], (st, where)
    # a batch of many tiles (case i not split): the shrink reads it first
    st, where = c["many_tiles_ids"]["fwd"]
    assert st == LORA_ERR_INDEX and where >> 16 == FILE_NUMBER["tc_rowproj.cu"] and where & 0xffff > 0, (st, where)
    st, where = c["many_tiles_ids"]["bwd"]
    assert st == LORA_ERR_INDEX and where >> 16 == FILE_NUMBER["tc_rowproj.cu"], (st, where)
