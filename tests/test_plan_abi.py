"""The library's C++ plan builder against the independent Python builder, bit for bit
(host code: runs without a GPU)."""
import json
import os

import numpy as np
import pytest

from oracle import plan_oracle as po
from kv_cache_decode_02_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_cases.json")
with open(GOLDEN) as f:
    PLAN = json.load(f)


def both(kvattn, seqs, capacity, stride=None):
    got_plan, got_lens = kvattn.build_cell_plan([np.asarray(s, np.int64) for s in seqs], capacity,
                                                plan_stride=stride)
    want_plan, want_lens = po.build_cell_plan(seqs, capacity, plan_stride=stride)
    return got_plan, got_lens, want_plan, want_lens


@pytest.mark.parametrize("case", PLAN["cases"] + PLAN["ok_edges"], ids=lambda c: c["name"])
def test_golden_cases_bit_exact(kvattn, case):
    gp, gl, wp, wl = both(kvattn, case["seqs"], case["capacity"])
    assert np.array_equal(gl, wl)
    assert np.array_equal(gp, wp)


@pytest.mark.parametrize("case", PLAN["errors"], ids=lambda c: c["name"])
def test_capacity_errors(kvattn, case):
    with pytest.raises(kvattn.KvattnError) as e:
        kvattn.build_cell_plan([np.asarray(s, np.int64) for s in case["seqs"]], case["capacity"])
    assert e.value.status == kvattn.KVATTN_ERR_CAPACITY


def test_stride_overflow_and_padding(kvattn):
    seqs = PLAN["cases"][1]["seqs"]
    gp, gl, wp, wl = both(kvattn, seqs, 1024, stride=640)
    assert np.array_equal(gp, wp) and gp.shape == (2, 640)
    with pytest.raises(kvattn.KvattnError) as e:
        kvattn.build_cell_plan([np.asarray(s, np.int64) for s in seqs], 1024, plan_stride=300)
    assert e.value.status == kvattn.KVATTN_ERR_CAPACITY


def test_bad_offsets_rejected(kvattn):
    cells = np.arange(10, dtype=np.int64)
    lens = np.zeros(2, np.int32)
    plan = np.zeros((2, 256), np.int32)
    for offs in ([1, 5, 10], [0, 6, 5]):
        rc = kvattn.lib.kvattn_build_cell_plan(cells.ctypes.data, np.array(offs, np.int64).ctypes.data, 2,
                                               1024, plan.ctypes.data, 256, lens.ctypes.data)
        assert rc == kvattn.KVATTN_ERR_INVALID_ARG
    rc = kvattn.lib.kvattn_build_cell_plan(cells.ctypes.data, np.array([0, 5, 10], np.int64).ctypes.data, 2,
                                           0, plan.ctypes.data, 256, lens.ctypes.data)
    assert rc == kvattn.KVATTN_ERR_INVALID_ARG


def test_random_cases_bit_exact(kvattn):
    rng = np.random.default_rng(2024)
    for trial in range(400):
        capacity = int(rng.integers(1, 5000))
        n_seq = int(rng.integers(0, 5))
        seqs = []
        for _ in range(n_seq):
            n = int(rng.integers(0, 300))
            phys = rng.integers(0, capacity, size=n)
            tags = rng.integers(0, 1 << 20, size=n)
            seqs.append(((tags << 32) | phys).astype(np.int64))
        if n_seq == 0:
            continue
        gp, gl, wp, wl = both(kvattn, seqs, capacity)
        assert np.array_equal(gl, wl), trial
        assert np.array_equal(gp, wp), trial


def test_multislot_layout_bit_exact(kvattn):
    w = inputs.MULTISLOT_PLAN
    lay = inputs.make_unified_layout(w)
    gp, gl, wp, wl = both(kvattn, lay.encoded_cells, w.n_cells)
    assert gl.tolist() == list(w.seq_lens)
    assert np.array_equal(gp, wp)
