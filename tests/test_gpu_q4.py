"""GPU parity of the 4-bit decode kernels -- Q8_0 keys with Q4_0 values, and Q4_0 keys and
values -- against the fp64 oracle:
compact plans with holes (one-run chunks through TMA boxes, the 4-bit V rows in one box),
scattered plans (per-row copies into plain rows), several sequences with ragged and empty
lengths, fully masked splits, the automatic split, the no-allocation entry point and the
full-size long-context workloads.

Unselected cells carry NaN scales: a masked cell whose scale reached the arithmetic would
turn its row's output into NaN.
"""
import numpy as np
import pytest

import oracle
from kv_cache_decode_02_gb300 import inputs
from oracle import plan_oracle as po
from tests.gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu


KINDS = ["q8k_q4v", "q4kv"]


def q8q4_cache(rng, n_cells, Hk, D, kind="q8k_q4v"):
    if kind == "q4kv":
        kq = rng.integers(0, 256, (n_cells, Hk, D // 2), dtype=np.uint8)
        kd = rng.uniform(0.001, 0.3, (n_cells, Hk, D // 32)).astype(np.float16)
    else:
        kq = rng.integers(-127, 128, (n_cells, Hk, D), dtype=np.int8)
        kd = rng.uniform(0.001, 0.02, (n_cells, Hk, D // 32)).astype(np.float16)
    v4 = rng.integers(0, 256, (n_cells, Hk, D // 2), dtype=np.uint8)
    vd = rng.uniform(0.001, 0.3, (n_cells, Hk, D // 32)).astype(np.float16)
    return kq, v4, kd, vd


def kv_type_of(K, kq, v4):
    return K.KVATTN_KV_Q4_0 if kq.dtype == np.uint8 else K.KVATTN_KV_Q8_0_Q4_0


def want(q, kq, kd, v4, vd, lens, plan=None):
    f = oracle.decode_q4_0 if kq.dtype == np.uint8 else oracle.decode_q8_0_q4_0
    return f(q, kq, kd, v4, vd, lens, plan=plan)


def run(K, q, kq, v4, kd, vd, lens, split, plan=None, n_cells=None, max_len=None):
    import torch
    out, lse = K.decode(dev(q), dev(kq), dev(v4), dev(np.asarray(lens, np.int32)), split=split,
                        k_scales=dev(kd), v_scales=dev(vd), cell_plan=None if plan is None else dev(plan),
                        n_cells=n_cells, max_len=max_len, kv_type=kv_type_of(K, kq, v4))
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("D,G,split", [(128, 4, 128), (128, 6, 256), (256, 8, 128), (256, 1, 64), (128, 8, 32)])
def test_q8q4_compact_plan_with_holes(kvattn, D, G, split, kind):
    rng = np.random.default_rng(700 + D + G)
    Hk, pool = 2, 24
    H = Hk * G
    n_cells = pool * 128
    kq, v4, kd, vd = q8q4_cache(rng, n_cells, Hk, D, kind)
    perm = rng.permutation(pool)
    owned = [perm[0:5], perm[5:6], perm[6:14]]
    encoded, selected = [], []
    for recs in owned:
        cells = (recs[:, None] * 128 + np.arange(128)[None]).reshape(-1)
        keep = rng.random(cells.size) >= 0.25
        sel = cells[keep]
        encoded.append(sel.astype(np.int64)[rng.permutation(sel.size)])
        selected.append(sel)
    unused = np.setdiff1d(np.arange(n_cells), np.concatenate(selected))
    kd[unused] = np.nan
    vd[unused] = np.nan
    plan, lens = kvattn.build_cell_plan(encoded, n_cells)
    wplan, wlens = po.build_cell_plan([e.tolist() for e in encoded], n_cells)
    assert np.array_equal(plan, wplan) and np.array_equal(lens, wlens)
    q = rng.standard_normal((3, H, D), dtype=np.float32).astype(np.float16)
    out, lse = run(kvattn, q, kq, v4, kd, vd, lens, split, plan=plan, n_cells=n_cells, max_len=plan.shape[1])
    wo, wl = want(q, kq, kd, v4, vd, lens.tolist(), plan=plan)
    assert_close(out, lse, wo, wl)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("D", [128, 256])
def test_q8q4_scattered_plan(kvattn, D, kind):
    """Plan entries in random order (most chunks are not one run: per-row copies into plain
    rows), -1 holes, a fully masked split, an empty sequence."""
    rng = np.random.default_rng(800 + D)
    Hk, G, split = 4, 4, 64
    H = Hk * G
    n_cells = 3000
    kq, v4, kd, vd = q8q4_cache(rng, n_cells, Hk, D, kind)
    stride = 700
    lens = np.array([700, 0, 333, 64], np.int32)
    plan = np.full((4, stride), -1, np.int32)
    used = np.zeros(n_cells, bool)
    for s, L in enumerate(lens):
        cells = rng.choice(n_cells, size=L, replace=False).astype(np.int32)
        cells[rng.random(L) < 0.2] = -1
        plan[s, :L] = cells
        used[cells[cells >= 0]] = True
    plan[0, 128:192] = -1
    plan[2, 32:48] = np.arange(1000, 1016, dtype=np.int32)   # one chunk that is a run
    used[1000:1016] = True
    kd[~used] = np.nan
    vd[~used] = np.nan
    q = rng.standard_normal((4, H, D), dtype=np.float32).astype(np.float16)
    out, lse = run(kvattn, q, kq, v4, kd, vd, lens, split, plan=plan, n_cells=n_cells, max_len=stride)
    wo, wl = want(q, kq, kd, v4, vd, lens.tolist(), plan=plan)
    assert_close(out, lse, wo, wl)
    assert np.all(np.isneginf(lse.cpu().numpy()[1]))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("D", [128, 256])
def test_q8q4_multi_sequence_ragged(kvattn, D, kind):
    rng = np.random.default_rng(900 + D)
    S, N, Hk, G, split = 3, 1100, 2, 5, 128
    H = Hk * G
    kq, v4, kd, vd = q8q4_cache(rng, S * N, Hk, D, kind)
    kq, v4 = kq.reshape((S, N) + kq.shape[1:]), v4.reshape(S, N, Hk, D // 2)
    kd, vd = kd.reshape(S, N, Hk, D // 32), vd.reshape(S, N, Hk, D // 32)
    lens = [1100, 0, 17]
    q = rng.standard_normal((S, H, D), dtype=np.float32).astype(np.float16)
    out, lse = run(kvattn, q, kq, v4, kd, vd, lens, split, n_cells=N, max_len=N)
    wo, wl = want(q, kq, kd, v4, vd, lens)
    assert_close(out, lse, wo, wl)


@pytest.mark.parametrize("D", [128, 256])
def test_q8q4_every_nibble_and_extreme_scales(kvattn, D):
    """Every 4-bit value in both halves of every byte position, scales of both signs from
    0.001 to 8 (values up to 64 in magnitude), one cell per sequence so that O is V itself:
    P = 1 and every product is exact, so the kernel must reproduce V bit for bit."""
    Hk = 1
    n = 16
    v4 = np.zeros((n, Hk, D // 2), np.uint8)
    for c in range(n):
        for j in range(D // 2):
            v4[c, 0, j] = ((c + j) % 16) | (((c + 3 * j + 7) % 16) << 4)
    pattern = [0.5, -8.0, 0.001, 3.0, -0.25, 1.0, 7.5, -0.002]
    vd = np.array(pattern[:D // 32], np.float16).reshape(1, 1, 1, D // 32).repeat(n, 0)
    kq = np.ones((n, 1, Hk, D), np.int8)
    kd = np.full((n, 1, Hk, D // 32), 0.01, np.float16)
    q = np.ones((n, Hk, D), np.float16)
    v4 = v4.reshape(n, 1, Hk, D // 2)
    out, lse = run(kvattn, q, kq, v4, kd, vd, [1] * n, 32, n_cells=1, max_len=1)
    wo, wl = oracle.decode_q8_0_q4_0(q, kq, kd, v4, vd, [1] * n)
    np.testing.assert_array_equal(out.cpu().numpy().reshape(wo.shape), wo)
    assert np.max(np.abs(lse.cpu().numpy() - wl)) <= 1e-4


def test_q8q4_auto_split_and_noalloc(kvattn):
    import torch
    rng = np.random.default_rng(950)
    N, Hk, G, D = 5000, 8, 4, 128
    H = Hk * G
    kq, v4, kd, vd = q8q4_cache(rng, N, Hk, D)
    q = rng.standard_normal((1, H, D), dtype=np.float32).astype(np.float16)
    wo, wl = oracle.decode_q8_0_q4_0(q, kq, kd, v4, vd, [N])
    lens = dev(np.array([N], np.int32))
    split = kvattn.kvattn_select_split(kvattn.KVATTN_KV_Q8_0_Q4_0, 1, N, Hk, D)
    assert split >= 64
    out, lse = run(kvattn, q, kq, v4, kd, vd, [N], 0)
    assert_close(out, lse, wo, wl)
    out2 = torch.empty((1, H, D), dtype=torch.float32, device="cuda")
    lse2 = torch.empty((1, H), dtype=torch.float32, device="cuda")
    kvattn.kvattn_decode_noalloc(dev(q), dev(kq), dev(v4), dev(kd), dev(vd), kvattn.KVATTN_KV_Q8_0_Q4_0, N, None, 0,
                                 lens, 1, N, H, Hk, D, 0, 1 / np.sqrt(D), out2, lse2, None)
    torch.cuda.synchronize()
    assert_close(out2, lse2, wo, wl)


def test_q4_keys_every_nibble(kvattn):
    """Q4_0 keys: each cell's key is one element of value scale * (n - 8) at one position and
    8 (zero) elsewhere, with q = 1, so the logit of cell c is scale_c * (n_c - 8) / sqrt(D):
    every nibble value in every position of both halves of a block reaches the score."""
    import torch
    D, Hk = 128, 1
    n = 64
    k4 = np.full((n, 1, Hk, D // 2), 0x88, np.uint8)
    for c in range(n):
        pos = (7 * c) % D
        nib = c % 16
        blk, j = pos // 32, pos % 32
        byte = 16 * blk + (j % 16)
        k4[c, 0, 0, byte] = (0x80 | nib) if j < 16 else (0x08 | (nib << 4))
    kd = np.full((n, 1, Hk, D // 32), 0.5, np.float16)
    v4 = np.full((n, 1, Hk, D // 2), 0x99, np.uint8)  # every value 1 * scale
    vd = np.full((n, 1, Hk, D // 32), 0.25, np.float16)
    q = np.ones((n, Hk, D), np.float16)
    out, lse = run(kvattn, q, k4, v4, kd, vd, [1] * n, 32, n_cells=1, max_len=1)
    wo, wl = oracle.decode_q4_0(q, k4, kd, v4, vd, [1] * n)
    logits = np.array([0.5 * ((c % 16) - 8) / np.sqrt(D) for c in range(n)])
    np.testing.assert_allclose(wl[:, 0], logits, rtol=0, atol=1e-12)
    assert np.max(np.abs(lse.cpu().numpy()[:, 0] - wl[:, 0])) <= 1e-5
    np.testing.assert_array_equal(out.cpu().numpy().reshape(wo.shape), wo)
    torch.cuda.synchronize()


@pytest.mark.parametrize("w", [inputs.Q8Q4_LONG_D128, inputs.Q8Q4_LONG_D256, inputs.Q4_LONG_D128,
                               inputs.Q4_LONG_D256], ids=lambda w: w.name)
def test_q8q4_long_context(kvattn, w):
    import torch
    q = inputs.make_q(w)
    (kq, kd), (v4, vd) = inputs.make_kv_q4(w) if w.kv_type == "q4_0" else inputs.make_kv_q8q4(w)
    out, lse = kvattn.decode(dev(q), dev(kq), dev(v4), dev(np.array(w.seq_lens, np.int32)), split=w.split,
                             k_scales=dev(kd), v_scales=dev(vd))
    torch.cuda.synchronize()
    wo, wl = want(q, kq, kd, v4, vd, list(w.seq_lens))
    assert_close(out, lse, wo, wl)


@pytest.mark.parametrize("kind", KINDS)
def test_q4_bounded_wait_reports_timeout_and_context_survives(kvattn, monkeypatch, kind):
    import torch
    rng = np.random.default_rng(960)
    N, Hk, G, D = 512, 2, 4, 128
    H = Hk * G
    kq, v4, kd, vd = q8q4_cache(rng, N, Hk, D, kind)
    q = rng.standard_normal((1, H, D), dtype=np.float32).astype(np.float16)
    ws = kvattn.decode_workspace(1, H, D, N, 128)
    monkeypatch.setenv("KVATTN_DEBUG_STALL_TX", "16")
    monkeypatch.setenv("KVATTN_DEBUG_WAIT_MS", "20")
    kvattn.decode(dev(q), dev(kq), dev(v4), dev(np.array([N], np.int32)), split=128, k_scales=dev(kd),
                  v_scales=dev(vd), ws=ws, kv_type=kv_type_of(kvattn, kq, v4))
    torch.cuda.synchronize()
    assert kvattn.kvattn_workspace_status(ws, clear=True) & kvattn.KVATTN_DEVICE_WAIT_TIMEOUT
    monkeypatch.delenv("KVATTN_DEBUG_STALL_TX")
    out, lse = kvattn.decode(dev(q), dev(kq), dev(v4), dev(np.array([N], np.int32)), split=128, k_scales=dev(kd),
                             v_scales=dev(vd), ws=ws, kv_type=kv_type_of(kvattn, kq, v4))
    torch.cuda.synchronize()
    assert kvattn.kvattn_workspace_status(ws) == 0
    wo, wl = want(q, kq, kd, v4, vd, [N])
    assert_close(out, lse, wo, wl)
