"""Pins for the Python plan builder and descriptor mirror (oracle side).

Hand-worked fixtures under tests/golden/ (each states the passage it follows) plus the
structural properties the pages require of a compact plan.
"""
import json
import os

import numpy as np
import pytest

from oracle import plan_oracle as po
from kv_cache_decode_02_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def expand(spec: str):
    """'a-b' -> a..b inclusive, '-1xN' -> N holes, 'c' -> c."""
    out = []
    for tok in spec.split():
        if tok.startswith("-1x"):
            out.extend([-1] * int(tok[3:]))
        elif "-" in tok[1:]:
            a, b = tok.split("-")
            out.extend(range(int(a), int(b) + 1))
        else:
            out.append(int(tok))
    return out


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


PLAN = load("plan_cases.json")
DESC = load("descriptor_cases.json")


@pytest.mark.parametrize("case", PLAN["cases"] + PLAN["ok_edges"], ids=lambda c: c["name"])
def test_plan_golden(case):
    plan, lens = po.build_cell_plan(case["seqs"], case["capacity"])
    assert lens.tolist() == case["seq_lens"]
    for s, spec in enumerate(case["plan"]):
        want = expand(spec)
        assert len(want) == case["seq_lens"][s]
        assert plan[s, :len(want)].tolist() == want
        assert np.all(plan[s, len(want):] == -1)


@pytest.mark.parametrize("case", PLAN["errors"], ids=lambda c: c["name"])
def test_plan_golden_errors(case):
    with pytest.raises(po.CapacityError):
        po.build_cell_plan(case["seqs"], case["capacity"])


def test_plan_stride_padding_and_overflow():
    case = PLAN["cases"][1]
    plan, lens = po.build_cell_plan(case["seqs"], case["capacity"], plan_stride=512)
    assert plan.shape == (2, 512)
    assert np.all(plan[0, 384:] == -1) and np.all(plan[1, 256:] == -1)
    with pytest.raises(po.CapacityError):
        po.build_cell_plan(case["seqs"], case["capacity"], plan_stride=300)


@pytest.mark.parametrize("case", DESC["cases"], ids=lambda c: c["name"])
def test_descriptor_golden(case):
    if "plan_case" in case:
        pc = next(c for c in PLAN["cases"] if c["name"] == case["plan_case"])
        plan, lens = po.build_cell_plan(pc["seqs"], pc["capacity"])
    else:
        plan = np.array(case["plan_rows"], dtype=np.int32)
        lens = np.array(case["seq_lens"], dtype=np.int32)
    d = po.descriptors(plan, lens, case["max_len"], case["split"], case["n_cells_phys"])
    assert d.tolist() == case["desc"]


def test_plan_structure_on_the_multislot_layout():
    """Every selected cell appears once, at its positional slot of its record's segment;
    records ascend; nothing unselected appears; lengths are 128 x records."""
    w = inputs.MULTISLOT_PLAN
    lay = inputs.make_unified_layout(w)
    plan, lens = po.build_cell_plan(lay.encoded_cells, w.n_cells)
    assert lens.tolist() == list(w.seq_lens)
    for s in range(w.n_seq):
        row = plan[s, :lens[s]]
        segs = row.reshape(-1, 128)
        recs = []
        for seg in segs:
            valid = seg[seg >= 0]
            assert valid.size > 0
            r = valid[0] // 128
            recs.append(r)
            j = np.nonzero(seg >= 0)[0]
            assert np.array_equal(seg[j], r * 128 + j)
        assert recs == sorted(recs) and len(set(recs)) == len(recs)
        got = np.sort(row[row >= 0])
        assert np.array_equal(got, lay.selected[s])
    holes = (plan[:, :] == -1).sum() - sum(plan.shape[1] - L for L in lens)
    frac = holes / lens.sum()
    assert 0.07 < frac < 0.13  # ~10 % holes


def test_descriptor_properties_random():
    rng = np.random.default_rng(1)
    S, stride, Np = 3, 700, 4096
    plan = rng.integers(-1, Np, size=(S, stride)).astype(np.int32)
    plan[0, 100:300] = np.arange(1000, 1200)  # one linear run
    plan[0, 128:140] = -1
    lens = np.array([650, 0, 700], dtype=np.int32)
    d = po.descriptors(plan, lens, 700, 64, Np)
    for s in range(S):
        for p in range(d.shape[1]):
            i0, i1 = p * 64, min(p * 64 + 64, lens[s])
            seg = plan[s, i0:max(i0, i1)]
            v = seg[(seg >= 0) & (seg < Np)]
            assert d[s, p, 0] == v.size
            if v.size:
                assert d[s, p, 1] == v.min() and d[s, p, 2] == v.max()
    # split [128, 192) of sequence 0 lies in the linear run with holes
    assert d[0, 2, 3] & po.FLAG_LINEAR
    assert d[1, :, 3].tolist() == [po.FLAG_EMPTY | po.FLAG_BEYOND] * d.shape[1]
