"""One-warp CTAs for the quantised head_dim-256 single-query kernels (real head_dim 256 and
head_dim 128 as KV-head pairs).

A call whose work units (sequence, split, KV head or pair) overflow one wave of the two-warp
CTAs (608 on GB300) but fit one wave of one-warp CTAs (eight per SM: 1216) runs a unit per
warp with no end-of-unit exchange between warps (launch mode 4 in the trace).  These tests
run such shapes -- every quantised type, ragged and short sequences, a compact plan with
holes, the no-workspace entry point -- check through the launch trace (KVATTN_LOG=1) that
mode 4 was taken, and compare with the oracle, and so is the same call on two-warp CTAs
(KVATTN_ONE_WARP=0).
"""
import re

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu

ORACLE = {"q8": oracle.decode_q8_0, "q8q4": oracle.decode_q8_0_q4_0, "q4": oracle.decode_q4_0}
KV_TYPE = {"q8": "KVATTN_KV_Q8_0", "q8q4": "KVATTN_KV_Q8_0_Q4_0", "q4": "KVATTN_KV_Q4_0"}


def quant_cache(rng, kind, lead, D):
    """(k values, k scales, v values, v scales) in the value ranges of the workloads."""
    lead = tuple(lead)
    if kind == "q4":
        kq = rng.integers(0, 256, lead + (D // 2,), dtype=np.uint8)
        kd = rng.uniform(0.001, 0.3, lead + (D // 32,)).astype(np.float16)
    else:
        kq = rng.integers(-127, 128, lead + (D,), dtype=np.int8)
        kd = rng.uniform(0.001, 0.02, lead + (D // 32,)).astype(np.float16)
    if kind == "q8":
        vq = rng.integers(-127, 128, lead + (D,), dtype=np.int8)
        vd = rng.uniform(0.001, 0.02, lead + (D // 32,)).astype(np.float16)
    else:
        vq = rng.integers(0, 256, lead + (D // 2,), dtype=np.uint8)
        vd = rng.uniform(0.001, 0.3, lead + (D // 32,)).astype(np.float16)
    return kq, kd, vq, vd


def traced(kvattn, capfd, monkeypatch, fn, one_warp_env=None):
    """Runs fn with the launch trace on; returns the fields of its decode line."""
    import torch
    monkeypatch.setenv("KVATTN_LOG", "1")
    if one_warp_env is not None:
        monkeypatch.setenv("KVATTN_ONE_WARP", one_warp_env)
    capfd.readouterr()
    fn()
    torch.cuda.synchronize()
    err = capfd.readouterr().err
    monkeypatch.delenv("KVATTN_LOG")
    if one_warp_env is not None:
        monkeypatch.delenv("KVATTN_ONE_WARP")
    lines = [ln for ln in err.splitlines() if ln.startswith("kvattn: decode ")]
    assert len(lines) == 1, err
    return dict(re.findall(r"(\w+)=(\S+)", lines[0]))


CASES = [
    # kind, D, G, Hk, lens, split  (units = sequences x splits x KV heads, or pairs at D 128)
    ("q8", 128, 4, 2, [100000], 128),            # one KV-head pair: 782 units
    ("q8", 256, 4, 2, [50000], 128),             # 782 units
    ("q8", 256, 7, 1, [38900, 3000], 64),        # G = 7 (rows padded to 8), 1216 units: a full wave
    ("q8q4", 128, 2, 2, [70000, 5000], 128),     # 1094 units, the second sequence ends early
    ("q8q4", 256, 3, 1, [38976], 64),            # 609 units: one more than the two-warp CTAs
    ("q4", 128, 4, 4, [50000, 17], 256),         # two KV-head pairs, a 17-cell sequence
    ("q4", 256, 5, 2, [20000, 333, 0], 128),     # G = 5, an empty sequence: 942 units
]


def _inputs(rng, kind, D, G, Hk, lens):
    S, N = len(lens), max(lens)
    H = G * Hk
    q = rng.standard_normal((S, H, D), dtype=np.float32).astype(np.float16)
    cache = quant_cache(rng, kind, (S, N, Hk), D)
    return q, cache, S, N, H


@pytest.mark.parametrize("kind,D,G,Hk,lens,split", CASES)
def test_one_warp_ctas_match_the_oracle(kvattn, capfd, monkeypatch, kind, D, G, Hk, lens, split):
    import torch
    rng = np.random.default_rng([71, D, G, Hk, len(lens)])
    q, cache, S, N, H = _inputs(rng, kind, D, G, Hk, lens)
    kq, kd, vq, vd = cache
    args = (dev(q), dev(kq), dev(vq), dev(kd), dev(vd), getattr(kvattn, KV_TYPE[kind]), N, None, 0,
            dev(np.asarray(lens, np.int32)), S, N, H, Hk, D, split, 1.0 / np.sqrt(D))
    wo, wl = ORACLE[kind](q, *cache, lens)
    nbytes = kvattn.kvattn_decode_workspace_bytes(S, H, D, N, split)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")

    out = torch.full((S, H, D), float("nan"), device="cuda")
    lse = torch.full((S, H), float("nan"), device="cuda")
    f = traced(kvattn, capfd, monkeypatch, lambda: kvattn.kvattn_decode(*args, out, lse, ws, nbytes))
    assert f["mode"] == "4" and f["grid"] == f["units"] and f["tma"] == "1", f
    assert 608 < int(f["units"]) <= 1216, f
    assert_close(out, lse, wo, wl)
    # a second call on the same workspace
    out.fill_(float("nan"))
    kvattn.kvattn_decode(*args, out, lse, ws, nbytes)
    torch.cuda.synchronize()
    assert_close(out, lse, wo, wl)

    # two warps per CTA: the same result
    out_w = torch.full((S, H, D), float("nan"), device="cuda")
    lse_w = torch.full((S, H), float("nan"), device="cuda")
    f = traced(kvattn, capfd, monkeypatch, lambda: kvattn.kvattn_decode(*args, out_w, lse_w, ws, nbytes), "0")
    assert f["mode"] == "0", f
    assert_close(out_w, lse_w, wo, wl)


def test_few_units_keep_two_warps_per_cta(kvattn, capfd, monkeypatch):
    """One wave of two-warp CTAs already holds every unit: each unit keeps both warps."""
    import torch
    rng = np.random.default_rng(72)
    kind, D, G, Hk, lens, split = "q8", 128, 4, 8, [16384], 256  # 64 splits x 4 pairs = 256 units
    q, cache, S, N, H = _inputs(rng, kind, D, G, Hk, lens)
    kq, kd, vq, vd = cache
    nbytes = kvattn.kvattn_decode_workspace_bytes(S, H, D, N, split)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full((S, H, D), float("nan"), device="cuda")
    lse = torch.full((S, H), float("nan"), device="cuda")
    f = traced(kvattn, capfd, monkeypatch, lambda: kvattn.kvattn_decode(
        dev(q), dev(kq), dev(vq), dev(kd), dev(vd), kvattn.KVATTN_KV_Q8_0, N, None, 0,
        dev(np.asarray(lens, np.int32)), S, N, H, Hk, D, split, 1.0 / np.sqrt(D), out, lse, ws, nbytes))
    assert f["mode"] == "0" and f["units"] == "256", f
    wo, wl = ORACLE[kind](q, *cache, lens)
    assert_close(out, lse, wo, wl)


def test_one_warp_ctas_through_a_plan_with_holes(kvattn, capfd, monkeypatch):
    """Two sequences read through a compact cell plan over 128-cell records, ~20 % of the
    cells -1 holes (descriptors from their own launch, fully masked splits skipped)."""
    import torch
    rng = np.random.default_rng(73)
    D, G, Hk, pool, split = 128, 4, 2, 800, 128
    H = G * Hk
    n_cells = pool * 128
    perm = rng.permutation(pool)
    encoded = []
    for recs in (perm[:420], perm[420:790]):
        cells = (recs[:, None] * 128 + np.arange(128)[None]).reshape(-1)
        encoded.append(cells[rng.random(cells.size) >= 0.2].astype(np.int64))
    plan, plens = kvattn.build_cell_plan(encoded, n_cells)
    S, stride = plan.shape
    q = rng.standard_normal((S, H, D), dtype=np.float32).astype(np.float16)
    cache = quant_cache(rng, "q8", (n_cells, Hk), D)
    kq, kd, vq, vd = cache
    nbytes = kvattn.kvattn_decode_workspace_bytes(S, H, D, stride, split)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full((S, H, D), float("nan"), device="cuda")
    lse = torch.full((S, H), float("nan"), device="cuda")
    f = traced(kvattn, capfd, monkeypatch, lambda: kvattn.kvattn_decode(
        dev(q), dev(kq), dev(vq), dev(kd), dev(vd), kvattn.KVATTN_KV_Q8_0, n_cells, dev(plan), stride, dev(plens),
        S, stride, H, Hk, D, split, 1.0 / np.sqrt(D), out, lse, ws, nbytes))
    assert f["mode"] == "4" and f["plan"] == "1", f
    wo, wl = oracle.decode_q8_0(q, *cache, plens.tolist(), plan=plan)
    assert_close(out, lse, wo, wl)


def test_one_warp_ctas_without_a_workspace(kvattn, capfd, monkeypatch):
    """kvattn_decode_noalloc takes the same route."""
    import torch
    kind, D, G, Hk, lens, split = CASES[0]
    rng = np.random.default_rng(74)
    q, cache, S, N, H = _inputs(rng, kind, D, G, Hk, lens)
    kq, kd, vq, vd = cache
    out = torch.full((S, H, D), float("nan"), device="cuda")
    lse = torch.full((S, H), float("nan"), device="cuda")
    f = traced(kvattn, capfd, monkeypatch, lambda: kvattn.kvattn_decode_noalloc(
        dev(q), dev(kq), dev(vq), dev(kd), dev(vd), kvattn.KVATTN_KV_Q8_0, N, None, 0,
        dev(np.asarray(lens, np.int32)), S, N, H, Hk, D, split, 1.0 / np.sqrt(D), out, lse))
    assert f["mode"] == "4", f
    wo, wl = ORACLE[kind](q, *cache, lens)
    assert_close(out, lse, wo, wl)
