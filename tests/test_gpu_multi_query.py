"""GPU parity of causal multi-query decode (kvattn_decode_multi) against the fp64 oracle:
n_q new tokens per sequence, token t seeing logical positions 0 .. L - n_q + t, the
G x n_q query rows of a KV head in one 16-row MMA tile (up to 16 rows: the two consumer warps
split the cells) or two (17 to 32 rows: they split the rows); at f16 head_dim 128, 33 to 128
rows, and 17 to 32 rows when the call's units fit about one wave of its CTAs, run on the
tcgen05 kernel (its own cases in test_gpu_multi_query_tc.py, which also runs the mma.sync
layouts that serve them with KVATTN_TC=0); at head_dim 256 each consumer warp takes 8 of up
to 16 rows."""
import numpy as np
import pytest

import oracle
from oracle import plan_oracle as po
from tests.gpu_util import TOL_LSE, TOL_O, TOL_RMSE_O, dev

pytestmark = pytest.mark.gpu


def rand_f16(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def check(out, lse, wo, wl):
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert o.shape == wo.shape and l.shape == wl.shape
    assert np.array_equal(np.isneginf(l), np.isneginf(wl))
    fin = np.isfinite(wl)
    assert np.max(np.abs(l[fin] - wl[fin]), initial=0.0) <= TOL_LSE
    assert np.max(np.abs(o - wo)) <= TOL_O
    assert np.sqrt(np.mean((o.astype(np.float64) - wo) ** 2)) <= TOL_RMSE_O
    assert np.all(o[~fin] == 0)


@pytest.mark.parametrize("n_q,G,Hk,lens,split", [
    (1, 4, 2, [1000, 37], 128),         # one token: the single-query kernels
    (2, 4, 2, [1000, 1], 128),          # 8 rows (single-query kernels, per-row causal masks); sequence 1 shorter than n_q
    (3, 2, 4, [515, 2, 0], 64),         # 6 rows, ragged, an empty sequence
    (8, 1, 2, [97, 8], 32),             # MHA, 8 tokens: 8 rows
    (4, 4, 2, [777, 4, 3], 64),         # 16 rows per KV head
    (8, 2, 4, [513, 300], 256),
    (16, 1, 4, [100, 16], 32),          # MHA, 16 tokens
    (3, 5, 2, [2049, 0], 512),          # 15 rows, an empty sequence
    (8, 4, 2, [1500, 9, 5], 128),       # 32 rows: each warp takes 16 rows over all cells
    (5, 5, 2, [640, 33], 64),           # 25 rows: the second warp's last 7 rows are padding
    (17, 1, 2, [300, 17], 32),          # MHA, 17 tokens
    (3, 6, 2, [2047], 256),             # 18 rows (GQA-6)
    (9, 4, 2, [1000, 9, 4], 128),       # 36 rows: two row groups (32 + 4)
    (8, 6, 2, [1537, 0], 64),           # 48 rows (GQA-6 verifying 8 tokens), an empty sequence
    (8, 8, 1, [700, 3], 256),           # 64 rows (GQA-8 verifying 8 tokens), a sequence shorter than n_q
    (16, 4, 2, [300, 16], 32),          # 64 rows: 16 tokens at GQA-4
    (33, 1, 2, [200, 40], 32),          # MHA, 33 tokens: the second group holds one row
])
def test_multi_query_contiguous(kvattn, n_q, G, Hk, lens, split):
    import torch
    rng = np.random.default_rng(n_q * 100 + G)
    S, D = len(lens), 128
    N = max(max(lens), 1)
    H = G * Hk
    q = rand_f16(rng, (S, n_q, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    out, lse = kvattn.decode_multi(dev(q), dev(k), dev(v), dev(np.array(lens, np.int32)), split=split,
                                   n_cells=N, max_len=N)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_multi(oracle.decode_f16, q, lens, k, v)
    check(out, lse, wo, wl)


@pytest.mark.parametrize("n_q,G,Hk,lens,split", [
    (1, 2, 2, [1000, 37], 128),
    (2, 8, 1, [700, 1], 128),           # sequence 1 shorter than n_q: token 0 sees nothing
    (4, 4, 2, [777, 4, 3], 64),         # 16 rows: each warp takes 8
    (3, 3, 2, [513, 0], 256),           # 9 rows (the second warp holds one), an empty sequence
    (16, 1, 2, [100, 16], 32),          # MHA, 16 tokens
    (5, 2, 4, [2049], 512),             # 10 rows over a ragged last split
    (5, 4, 2, [300, 5, 2], 32),         # 20 rows: row groups of 16 and 4
    (8, 4, 2, [777, 8], 128),           # 32 rows (GQA-4 verifying 8 tokens): two row groups
    (8, 8, 1, [500, 3, 0], 64),         # 64 rows: four row groups, short and empty sequences
    (16, 8, 1, [300, 16, 2], 64),       # 128 rows (16 tokens at GQA-8): eight row groups
])
def test_multi_query_contiguous_d256(kvattn, n_q, G, Hk, lens, split):
    """head_dim 256 (Gemma-family layers): 8 query rows per consumer warp, row groups of 16
    beyond 16 rows."""
    import torch
    rng = np.random.default_rng(n_q * 100 + G + 3)
    S, D = len(lens), 256
    N = max(max(lens), 1)
    H = G * Hk
    q = rand_f16(rng, (S, n_q, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    out, lse = kvattn.decode_multi(dev(q), dev(k), dev(v), dev(np.array(lens, np.int32)), split=split,
                                   n_cells=N, max_len=N)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_multi(oracle.decode_f16, q, lens, k, v)
    check(out, lse, wo, wl)


@pytest.mark.parametrize("n_q,D,G", [(4, 128, 4), (8, 128, 4), (4, 256, 4), (8, 128, 6), (16, 128, 4),
                                     (8, 256, 4)])
def test_multi_query_plan_with_holes(kvattn, n_q, D, G):
    import torch
    rng = np.random.default_rng(9)
    Hk = 4
    H = Hk * G
    pool = 30
    n_cells = pool * 128
    k = rand_f16(rng, (n_cells, Hk, D))
    v = rand_f16(rng, (n_cells, Hk, D))
    perm = rng.permutation(pool)
    encoded, selected = [], []
    for recs in (perm[:4], perm[4:5], perm[5:12]):
        cells = (recs[:, None] * 128 + np.arange(128)[None]).reshape(-1)
        sel = cells[rng.random(cells.size) >= 0.2]
        encoded.append(sel.astype(np.int64)[rng.permutation(sel.size)])
        selected.append(sel)
    unused = np.setdiff1d(np.arange(n_cells), np.concatenate(selected))
    k[unused] = np.nan
    v[unused] = np.nan
    plan, lens = kvattn.build_cell_plan(encoded, n_cells)
    q = rand_f16(rng, (3, n_q, H, D))
    out, lse = kvattn.decode_multi(dev(q), dev(k), dev(v), dev(lens), split=128, cell_plan=dev(plan),
                                   n_cells=n_cells)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_multi(oracle.decode_f16, q, lens.tolist(), k, v, plan=plan)
    check(out, lse, wo, wl)


@pytest.mark.parametrize("D", [128, 256])
def test_one_token_equals_single_query_decode(kvattn, D):
    import torch
    rng = np.random.default_rng(10)
    S, N, H, Hk = 2, 3000, 32, 8
    q = rand_f16(rng, (S, 1, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    lens = dev(np.array([3000, 1234], np.int32))
    mo, ml = kvattn.decode_multi(dev(q), dev(k), dev(v), lens, split=256, n_cells=N, max_len=N)
    so, sl = kvattn.decode(dev(q[:, 0]), dev(k), dev(v), lens, split=256, n_cells=N, max_len=N)
    torch.cuda.synchronize()
    # head_dim 128 runs the same cell order in both kernels; at 256 the multi-query warp walks
    # both halves of a tile (the single-query warps split them and merge), so the running
    # maxima, and with them the f16 roundings of P, differ: agreement to rounding, not bits
    tol = 1e-5 if D == 128 else 1e-4
    assert np.max(np.abs(mo.cpu().numpy()[:, 0] - so.cpu().numpy())) <= tol
    assert np.max(np.abs(ml.cpu().numpy()[:, 0] - sl.cpu().numpy())) <= 1e-5


@pytest.mark.parametrize("n_q", [4, 8])
def test_speculative_verify_qwen3_layer(kvattn, n_q):
    """The Qwen3-8B-shaped layer verifying 4 or 8 draft tokens: 16 or 32 query rows per KV
    head."""
    import torch
    from kv_cache_decode_02_gb300 import inputs
    w = inputs.QWEN3_8B_LAYER
    rng = np.random.default_rng(11)
    q = rand_f16(rng, (1, n_q, w.n_head, w.head_dim))
    k, v = inputs.make_kv_f16(w, layer=0)
    lens = list(w.seq_lens)
    out, lse = kvattn.decode_multi(dev(q), dev(k), dev(v), dev(np.array(lens, np.int32)), split=w.split)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_multi(oracle.decode_f16, q, lens, k, v)
    check(out, lse, wo, wl)


def q8_cache(rng, shape, kind="q8"):
    """Quantised K and V planes: kind q8 (int8 K and V), q8k_q4v (int8 K, 4-bit V) or q4kv."""
    *lead, D = shape
    lead = tuple(lead)
    if kind == "q4kv":
        kq = rng.integers(0, 256, lead + (D // 2,), dtype=np.uint8)
        kd = rng.uniform(0.001, 0.3, lead + (D // 32,)).astype(np.float16)
    else:
        kq = rng.integers(-127, 128, shape, dtype=np.int8)
        kd = rng.uniform(0.001, 0.02, lead + (D // 32,)).astype(np.float16)
    if kind == "q8":
        vq = rng.integers(-127, 128, shape, dtype=np.int8)
        vd = rng.uniform(0.001, 0.02, lead + (D // 32,)).astype(np.float16)
    else:
        vq = rng.integers(0, 256, lead + (D // 2,), dtype=np.uint8)
        vd = rng.uniform(0.001, 0.3, lead + (D // 32,)).astype(np.float16)
    return kq, kd, vq, vd


ORACLE = {"q8": oracle.decode_q8_0, "q8k_q4v": oracle.decode_q8_0_q4_0, "q4kv": oracle.decode_q4_0}


@pytest.mark.parametrize("kind", ["q8", "q8k_q4v", "q4kv"])
@pytest.mark.parametrize("n_q,G,Hk,lens,split", [
    (1, 4, 2, [1000, 37], 128),
    (2, 4, 2, [1000, 1], 128),          # sequence 1 shorter than n_q
    (4, 4, 2, [777, 4, 3], 64),         # 16 rows per KV head
    (8, 2, 4, [513, 300], 256),
    (16, 1, 2, [100, 16], 32),          # MHA, 16 tokens
    (3, 5, 2, [2049, 0], 512),          # 15 rows, an empty sequence
    (5, 4, 2, [300, 5, 2], 32),         # 20 rows: row groups of 16 and 4
    (8, 4, 2, [777, 8, 3], 64),         # 32 rows (GQA-4 verifying 8 tokens): two row groups
    (8, 8, 1, [513, 0], 128),           # 64 rows: four row groups, an empty sequence
    (16, 8, 1, [400, 16], 64),          # 128 rows: eight row groups
])
def test_multi_query_quantised_contiguous(kvattn, n_q, G, Hk, lens, split, kind):
    """Quantised caches: the self-loading kernels with the whole 16-row M of the MMA, row
    groups of 16 beyond 16 rows."""
    import torch
    rng = np.random.default_rng(n_q * 100 + G + 7)
    S, D = len(lens), 128
    N = max(max(lens), 1)
    H = G * Hk
    q = rand_f16(rng, (S, n_q, H, D))
    kq, kd, vq, vd = q8_cache(rng, (S, N, Hk, D), kind)
    out, lse = kvattn.decode_multi(dev(q), dev(kq), dev(vq), dev(np.array(lens, np.int32)), split=split,
                                   n_cells=N, max_len=N, k_scales=dev(kd), v_scales=dev(vd))
    torch.cuda.synchronize()
    wo, wl = oracle.decode_multi(ORACLE[kind], q, lens, kq, kd, vq, vd)
    check(out, lse, wo, wl)


@pytest.mark.parametrize("n_q", [4, 8])
@pytest.mark.parametrize("kind", ["q8", "q8k_q4v", "q4kv"])
def test_multi_query_quantised_plan_with_holes(kvattn, kind, n_q):
    """Scattered and record-aligned plan entries with -1 holes over NaN-scaled cells."""
    import torch
    rng = np.random.default_rng(19)
    Hk, G, D = 4, 4, 128
    H = Hk * G
    pool = 30
    n_cells = pool * 128
    kq, kd, vq, vd = q8_cache(rng, (n_cells, Hk, D), kind)
    perm = rng.permutation(pool)
    encoded, selected = [], []
    for recs in (perm[:4], perm[4:5], perm[5:12]):
        cells = (recs[:, None] * 128 + np.arange(128)[None]).reshape(-1)
        sel = cells[rng.random(cells.size) >= 0.2]
        encoded.append(sel.astype(np.int64)[rng.permutation(sel.size)])
        selected.append(sel)
    unused = np.setdiff1d(np.arange(n_cells), np.concatenate(selected))
    kd[unused] = np.nan
    vd[unused] = np.nan
    plan, lens = kvattn.build_cell_plan(encoded, n_cells)
    plan[0, 40:200] = plan[0, 40:200][rng.permutation(160)]  # no longer one physical run: per-row copies
    q = rand_f16(rng, (3, n_q, H, D))
    out, lse = kvattn.decode_multi(dev(q), dev(kq), dev(vq), dev(lens), split=128, cell_plan=dev(plan),
                                   n_cells=n_cells, k_scales=dev(kd), v_scales=dev(vd))
    torch.cuda.synchronize()
    wo, wl = oracle.decode_multi(ORACLE[kind], q, lens.tolist(), kq, kd, vq, vd, plan=plan)
    check(out, lse, wo, wl)


@pytest.mark.parametrize("kind", ["q8", "q8k_q4v", "q4kv"])
@pytest.mark.parametrize("n_q,G,Hk,lens,split", [
    (1, 4, 2, [1000, 37], 128),         # 4 rows
    (2, 4, 2, [700, 1], 64),            # 8 rows, a sequence shorter than n_q
    (4, 4, 2, [777, 4, 3], 64),         # 16 rows: two 8-row groups
    (3, 5, 2, [2049, 0], 512),          # 15 rows, an empty sequence
    (5, 2, 4, [300], 32),               # 10 rows: groups of 8 and 2
    (8, 8, 1, [500, 3], 64),            # 64 rows: eight groups
    (16, 8, 1, [260, 7], 64),           # 128 rows: sixteen groups
])
def test_multi_query_quantised_d256(kvattn, n_q, G, Hk, lens, split, kind):
    """head_dim 256 over the quantised caches: 8-row units on the single-query geometry,
    each lane's cells cut at its row's causal limit."""
    import torch
    rng = np.random.default_rng(n_q * 100 + G + 11)
    S, D = len(lens), 256
    N = max(max(lens), 1)
    H = G * Hk
    q = rand_f16(rng, (S, n_q, H, D))
    kq, kd, vq, vd = q8_cache(rng, (S, N, Hk, D), kind)
    out, lse = kvattn.decode_multi(dev(q), dev(kq), dev(vq), dev(np.array(lens, np.int32)), split=split,
                                   n_cells=N, max_len=N, k_scales=dev(kd), v_scales=dev(vd))
    torch.cuda.synchronize()
    wo, wl = oracle.decode_multi(ORACLE[kind], q, lens, kq, kd, vq, vd)
    check(out, lse, wo, wl)


@pytest.mark.parametrize("kind", ["q8", "q8k_q4v", "q4kv"])
def test_multi_query_quantised_d256_plan_with_holes(kvattn, kind):
    import torch
    rng = np.random.default_rng(29)
    Hk, G, n_q, D = 2, 4, 4, 256
    H = Hk * G
    pool = 20
    n_cells = pool * 128
    kq, kd, vq, vd = q8_cache(rng, (n_cells, Hk, D), kind)
    perm = rng.permutation(pool)
    encoded, selected = [], []
    for recs in (perm[:3], perm[3:4], perm[4:9]):
        cells = (recs[:, None] * 128 + np.arange(128)[None]).reshape(-1)
        sel = cells[rng.random(cells.size) >= 0.2]
        encoded.append(sel.astype(np.int64)[rng.permutation(sel.size)])
        selected.append(sel)
    unused = np.setdiff1d(np.arange(n_cells), np.concatenate(selected))
    kd[unused] = np.nan
    vd[unused] = np.nan
    plan, lens = kvattn.build_cell_plan(encoded, n_cells)
    q = rand_f16(rng, (3, n_q, H, D))
    out, lse = kvattn.decode_multi(dev(q), dev(kq), dev(vq), dev(lens), split=128, cell_plan=dev(plan),
                                   n_cells=n_cells, k_scales=dev(kd), v_scales=dev(vd))
    torch.cuda.synchronize()
    wo, wl = oracle.decode_multi(ORACLE[kind], q, lens.tolist(), kq, kd, vq, vd, plan=plan)
    check(out, lse, wo, wl)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("kind", ["q8", "q8k_q4v", "q4kv"])
def test_multi_query_quantised_one_token_equals_single_query(kvattn, kind, D):
    import torch
    rng = np.random.default_rng(20)
    S, N, H, Hk = 2, 3000, 32, 8
    q = rand_f16(rng, (S, 1, H, D))
    kq, kd, vq, vd = q8_cache(rng, (S, N, Hk, D), kind)
    lens = dev(np.array([3000, 1234], np.int32))
    mo, ml = kvattn.decode_multi(dev(q), dev(kq), dev(vq), lens, split=256, n_cells=N, max_len=N,
                                 k_scales=dev(kd), v_scales=dev(vd))
    so, sl = kvattn.decode(dev(q[:, 0]), dev(kq), dev(vq), lens, split=256, n_cells=N, max_len=N,
                           k_scales=dev(kd), v_scales=dev(vd))
    torch.cuda.synchronize()
    assert np.max(np.abs(mo.cpu().numpy()[:, 0] - so.cpu().numpy())) <= 1e-4
    assert np.max(np.abs(ml.cpu().numpy()[:, 0] - sl.cpu().numpy())) <= 1e-5


@pytest.mark.parametrize("kind", ["f16", "f16_d256", "q8", "f16_8rows", "f16_48rows", "f16_128rows"])
def test_multi_query_bounded_wait_reports_timeout_and_context_survives(kvattn, monkeypatch, kind):
    """The multi-query kernels' pipeline waits are bounded: a first tile that expects bytes
    no copy delivers (host test switch) ends in the timeout status bit, and the next call is
    clean.  (f16_8rows: 8 query rows per KV head, the single-query kernels' multi-query mode;
    f16_48rows and f16_128rows: the tcgen05 kernel with two and four row warps.)"""
    import torch
    rng = np.random.default_rng(23)
    S, N, H, Hk = 1, 600, 16, 4
    n_q = {"f16_8rows": 2, "f16_48rows": 12, "f16_128rows": 32}.get(kind, 4)
    D = 256 if kind == "f16_d256" else 128
    q = rand_f16(rng, (S, n_q, H, D))
    if kind.startswith("f16"):
        k, v = rand_f16(rng, (S, N, Hk, D)), rand_f16(rng, (S, N, Hk, D))
        extra = {}
        want = oracle.decode_multi(oracle.decode_f16, q, [N], k, v)
    else:
        k, kd, v, vd = q8_cache(rng, (S, N, Hk, D))
        extra = {"k_scales": dev(kd), "v_scales": dev(vd)}
        want = oracle.decode_multi(oracle.decode_q8_0, q, [N], k, kd, v, vd)
    ws = torch.zeros(kvattn.kvattn_decode_multi_workspace_bytes(S, n_q, H, D, N, 128), dtype=torch.uint8,
                     device="cuda")
    lens = dev(np.array([N], np.int32))
    monkeypatch.setenv("KVATTN_DEBUG_STALL_TX", "16")
    monkeypatch.setenv("KVATTN_DEBUG_WAIT_MS", "20")
    kvattn.decode_multi(dev(q), dev(k), dev(v), lens, split=128, n_cells=N, max_len=N, ws=ws, **extra)
    torch.cuda.synchronize()
    assert kvattn.kvattn_workspace_status(ws, clear=True) & kvattn.KVATTN_DEVICE_WAIT_TIMEOUT
    monkeypatch.delenv("KVATTN_DEBUG_STALL_TX")
    out, lse = kvattn.decode_multi(dev(q), dev(k), dev(v), lens, split=128, n_cells=N, max_len=N, ws=ws, **extra)
    torch.cuda.synchronize()
    assert kvattn.kvattn_workspace_status(ws) == 0
    check(out, lse, *want)
