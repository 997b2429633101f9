"""GPU parity of causal multi-query decode on the fifth-generation tensor cores (f16 cache,
head_dim 128, 17 to 128 query rows per KV head: every row of a KV head in one work unit, S,
P and O in tensor memory) against the fp64 oracle -- contiguous caches with ragged and
empty sequences, many work units per CTA, plans whose tiles are whole runs, runs with holes
and scattered cells over NaN-filled unused cells, the per-split descriptors such a call
leaves in the workspace, the automatic split, and the mma.sync kernels that serve the same
calls when the tcgen05 path is switched off (KVATTN_TC=0)."""
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


CONTIGUOUS = [
    # n_q, G, Hk, lens, split   (rows per KV head = n_q * G)
    (11, 3, 2, [2047, 11, 1], 64),     # 33 rows; a sequence of one cell: ten tokens see nothing
    (9, 4, 2, [1000, 9, 4], 128),      # 36 rows; sequences no longer than n_q
    (8, 6, 2, [1537, 0], 64),          # 48 rows (GQA-6 verifying 8 tokens), an empty sequence
    (10, 5, 3, [777, 301], 96),        # 50 rows, a ragged last tile in every sequence
    (16, 4, 1, [700, 3, 16], 32),      # 64 rows, one KV head
    (8, 8, 2, [9000, 4100], 32),       # 64 rows over 428 splits: several units per CTA
    (12, 6, 2, [1100, 5], 128),        # 72 rows: three row warps
    (13, 7, 1, [700, 13, 2], 32),      # 91 rows
    (16, 8, 1, [900, 10], 64),         # 128 rows (16 tokens at GQA-8): every TMEM lane
    (16, 8, 2, [5000, 16], 32),        # 128 rows over 314 splits
]


@pytest.mark.parametrize("n_q,G,Hk,lens,split", CONTIGUOUS)
def test_tc_contiguous(kvattn, n_q, G, Hk, lens, split):
    import torch
    rng = np.random.default_rng([41, n_q, G, Hk, split])
    S, D = len(lens), 128
    N = max(max(lens), 1)
    H = G * Hk
    q = rand_f16(rng, (S, n_q, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    out, lse = kvattn.decode_multi(dev(q), dev(k), dev(v), dev(np.array(lens, np.int32)), split=split,
                                   n_cells=N, max_len=N)
    torch.cuda.synchronize()
    check(out, lse, *oracle.decode_multi(oracle.decode_f16, q, lens, k, v))


def plan_cache(kvattn, rng, kind, Hk, D, pool=24, plan_stride=None):
    """A unified cache of pool x 128 cells, three sequences and their plan.  kind: 'runs' --
    whole records (every 32-entry tile one physical run); 'holes' -- records with a fifth of
    their cells dropped (runs with holes: the plan keeps a record's positions); 'scattered'
    -- a hand-made plan listing the sequences' cells in random order (no tile is a run).
    Cells no sequence holds are NaN.  Returns k, v, plan, lens, n_cells."""
    n_cells = pool * 128
    k = rand_f16(rng, (n_cells, Hk, D))
    v = rand_f16(rng, (n_cells, Hk, D))
    perm = rng.permutation(pool)
    encoded = []
    for recs in (perm[:5], perm[5:6], perm[6:15]):
        cells = (recs[:, None] * 128 + np.arange(128)[None]).reshape(-1)
        if kind == "holes":
            cells = cells[rng.random(cells.size) >= 0.2]
        encoded.append(cells.astype(np.int64))
    unused = np.setdiff1d(np.arange(n_cells), np.concatenate(encoded))
    k[unused] = np.nan
    v[unused] = np.nan
    if kind == "scattered":
        lens = np.array([e.size for e in encoded], np.int32)
        plan = np.full((3, plan_stride or int(lens.max())), -1, np.int32)
        for s_, e in enumerate(encoded):
            plan[s_, :e.size] = e[rng.permutation(e.size)]
    else:
        plan, lens = kvattn.build_cell_plan(encoded, n_cells, plan_stride=plan_stride)
    return k, v, plan, lens, n_cells


@pytest.mark.parametrize("kind", ["runs", "holes", "scattered"])
@pytest.mark.parametrize("n_q,G", [(8, 6), (16, 4), (12, 3), (16, 8)])
def test_tc_plan(kvattn, kind, n_q, G):
    import torch
    rng = np.random.default_rng([42, n_q, G, ["runs", "holes", "scattered"].index(kind)])
    Hk, D = 2, 128
    k, v, plan, lens, n_cells = plan_cache(kvattn, rng, kind, Hk, D)
    q = rand_f16(rng, (3, n_q, G * Hk, D))
    out, lse = kvattn.decode_multi(dev(q), dev(k), dev(v), dev(lens), split=128, cell_plan=dev(plan),
                                   n_cells=n_cells)
    torch.cuda.synchronize()
    check(out, lse, *oracle.decode_multi(oracle.decode_f16, q, lens.tolist(), k, v, plan=plan))


def test_tc_plan_leaves_the_split_descriptors_in_the_workspace(kvattn):
    """The tcgen05 producer writes every split's descriptor (count, smallest and largest
    cell, one-run and out-of-range flags) into the workspace as kvattn_build_descriptors
    computes them: out-of-range entries, a fully masked split, splits past a length."""
    import torch
    rng = np.random.default_rng(43)
    Hk, D, G, n_q = 2, 128, 6, 8
    k, v, plan, lens, n_cells = plan_cache(kvattn, rng, "holes", Hk, D, plan_stride=1280)
    plan[0, 5] = -7
    plan[2, 300] = n_cells + 3
    plan[2, 128:256] = -1
    masked = plan.copy()
    masked[(masked < -1) | (masked >= n_cells)] = -1
    S, H = plan.shape[0], G * Hk
    q = rand_f16(rng, (S, n_q, H, D))
    for split, max_len in [(128, 1280), (64, 1100)]:
        n_split = -(-max_len // split)
        ws = torch.zeros(kvattn.kvattn_decode_multi_workspace_bytes(S, n_q, H, D, max_len, split), dtype=torch.uint8,
                         device="cuda")
        out, lse = kvattn.decode_multi(dev(q), dev(k), dev(v), dev(lens), split=split, cell_plan=dev(plan),
                                       n_cells=n_cells, max_len=max_len, ws=ws)
        torch.cuda.synchronize()
        status = kvattn.kvattn_workspace_status(ws, clear=True)
        assert status == kvattn.KVATTN_DEVICE_BAD_PLAN_ENTRY
        got = ws[256:256 + S * n_split * 16].view(torch.int32).view(S, n_split, 4).cpu().numpy()
        assert np.array_equal(got, po.descriptors(plan, lens, max_len, split, n_cells))
        check(out, lse, *oracle.decode_multi(oracle.decode_f16, q, np.minimum(lens, max_len).tolist(), k, v,
                                             plan=masked))


@pytest.mark.parametrize("n_q,G,Hk,lens,split", [CONTIGUOUS[0], CONTIGUOUS[2], CONTIGUOUS[4], CONTIGUOUS[8],
                                                 (17, 1, 2, [300, 17], 32),        # 17 rows
                                                 (5, 5, 2, [640, 33], 64),         # 25 rows
                                                 (8, 4, 2, [1500, 9, 5], 128)])    # 32 rows
def test_mma_path_for_the_same_rows(kvattn, monkeypatch, n_q, G, Hk, lens, split):
    """With the tcgen05 path off the mma.sync kernels (the two consumer warps splitting 17 to
    32 rows, three consumer warps, row groups) serve the same calls; both agree with the
    oracle and with each other to rounding."""
    import torch
    rng = np.random.default_rng([44, n_q, G])
    S, D = len(lens), 128
    N = max(max(lens), 1)
    H = G * Hk
    q = rand_f16(rng, (S, n_q, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    args = (dev(q), dev(k), dev(v), dev(np.array(lens, np.int32)))
    o_tc, l_tc = kvattn.decode_multi(*args, split=split, n_cells=N, max_len=N)
    monkeypatch.setenv("KVATTN_TC", "0")
    o_mma, l_mma = kvattn.decode_multi(*args, split=split, n_cells=N, max_len=N)
    torch.cuda.synchronize()
    want = oracle.decode_multi(oracle.decode_f16, q, lens, k, v)
    check(o_mma, l_mma, *want)
    check(o_tc, l_tc, *want)
    fin = np.isfinite(l_tc.cpu().numpy())
    assert np.max(np.abs(o_tc.cpu().numpy() - o_mma.cpu().numpy())) <= 1e-3
    assert np.max(np.abs(l_tc.cpu().numpy()[fin] - l_mma.cpu().numpy()[fin]), initial=0.0) <= 1e-4


def test_tc_split_zero_selects_one_wave_of_its_units(kvattn):
    """split 0 on the tcgen05 path picks the split for the kernel's own two CTAs per SM (the
    smallest power of two whose units fit one wave): the result is bit-identical to an
    explicit call at that split, and matches the oracle."""
    import torch
    rng = np.random.default_rng(45)
    S, N, Hk, G, n_q, D = 2, 6000, 4, 6, 8, 128
    H = G * Hk
    q = rand_f16(rng, (S, n_q, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    lens = dev(np.array([N, 2500], np.int32))
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    sp = kvattn.kvattn_select_split_for(S, N, Hk, 2 * sm)
    o0, l0 = kvattn.decode_multi(dev(q), dev(k), dev(v), lens, split=0, n_cells=N, max_len=N)
    o1, l1 = kvattn.decode_multi(dev(q), dev(k), dev(v), lens, split=sp, n_cells=N, max_len=N)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    check(o0, l0, *oracle.decode_multi(oracle.decode_f16, q, [N, 2500], k, v))


def test_q_not_16_byte_aligned_takes_the_mma_path(kvattn):
    """The tcgen05 kernel copies query rows 16 bytes at a time; a q that is only 4-byte
    aligned (as the entry point allows) is served by the mma.sync layouts, still exact."""
    import torch
    rng = np.random.default_rng(46)
    S, N, Hk, G, n_q, D = 2, 900, 2, 6, 8, 128      # 48 rows per KV head
    H = G * Hk
    q = rand_f16(rng, (S, n_q, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    buf = torch.empty(q.size + 2, dtype=torch.float16, device="cuda")
    qd = buf[2:].view(S, n_q, H, D)                 # 4 bytes past a 16-byte boundary
    qd.copy_(dev(q))
    assert qd.data_ptr() % 16 == 4
    out, lse = kvattn.decode_multi(qd, dev(k), dev(v), dev(np.array([N, 333], np.int32)), split=128, n_cells=N,
                                   max_len=N)
    torch.cuda.synchronize()
    check(out, lse, *oracle.decode_multi(oracle.decode_f16, q, [N, 333], k, v))
