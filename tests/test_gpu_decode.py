"""GPU parity of the split-KV decode path (through the C ABI) against the fp64 oracle.

Small cases span several 32-cell tiles, several splits and ragged tails; edge cases
cover a single cell, an empty sequence, G = 1..8, head_dim 128/256, Q8_0, and plans with
holes over NaN-filled cells.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import plan_oracle as po
from tests.gpu_util import TOL_LSE, TOL_O, assert_close, dev

pytestmark = pytest.mark.gpu


def rand_f16(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def run_contiguous(K, q, k, v, lens, split, max_len=None):
    import torch
    S, H, D = q.shape
    n_cells = k.shape[1] if k.ndim == 4 else k.shape[0]
    out, lse = K.decode(dev(q), dev(k), dev(v), dev(np.asarray(lens, np.int32)), split=split,
                        max_len=n_cells if max_len is None else max_len, n_cells=n_cells)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("N,H,Hk,D,split", [
    (1, 8, 8, 128, 32),          # one cell, MHA
    (31, 8, 2, 128, 32),         # shorter than a tile
    (33, 8, 2, 128, 32),         # one cell into the second tile
    (1000, 12, 2, 128, 64),      # GQA-6, ragged tail
    (4097, 40, 8, 128, 256),     # GQA-5, ragged
    (777, 8, 1, 256, 128),       # GQA-8, head_dim 256
    (2048, 4, 4, 256, 512),      # MHA, head_dim 256
    (129, 16, 2, 128, 128),      # GQA-8
    (3000, 28, 4, 128, 96),      # GQA-7, split of three tiles
])
def test_f16_contiguous(kvattn, N, H, Hk, D, split):
    rng = np.random.default_rng(N * 7 + H)
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    out, lse = run_contiguous(kvattn, q, k, v, [N], split)
    wo, wl = oracle.decode_f16(q, k, v, [N])
    assert_close(out, lse, wo, wl)


def test_tiny_workload(kvattn):
    from kv_cache_decode_02_gb300 import inputs
    w = inputs.TINY
    q = inputs.make_q(w)
    k, v = inputs.make_kv_f16(w)
    out, lse = run_contiguous(kvattn, q, k, v, list(w.seq_lens), w.split)
    wo, wl = oracle.decode_f16(q, k, v, list(w.seq_lens))
    assert_close(out, lse, wo, wl)


def test_multi_sequence_ragged_with_empty(kvattn):
    rng = np.random.default_rng(5)
    S, N, H, Hk, D = 4, 1500, 32, 8, 128
    q = rand_f16(rng, (S, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    lens = [1500, 0, 1, 777]
    out, lse = run_contiguous(kvattn, q, k, v, lens, 256)
    wo, wl = oracle.decode_f16(q, k, v, lens)
    assert_close(out, lse, wo, wl)
    lse_h = lse.cpu().numpy()
    assert np.all(np.isneginf(lse_h[1])) and np.all(out.cpu().numpy()[1] == 0)


def test_lengths_clamped_to_max_len(kvattn):
    rng = np.random.default_rng(6)
    N, H, Hk, D = 640, 8, 2, 128
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    out, lse = run_contiguous(kvattn, q, k, v, [N], 64, max_len=300)
    wo, wl = oracle.decode_f16(q, k[:300], v[:300], [300])
    assert_close(out, lse, wo, wl)


@pytest.mark.parametrize("D,N,split,G", [(128, 1000, 128, 4), (256, 1000, 512, 4), (128, 97, 32, 6),
                                          (256, 300, 64, 8)])
def test_q8_0(kvattn, D, N, split, G):
    import torch
    rng = np.random.default_rng(D + N)
    Hk = 2
    H = Hk * G
    q = rand_f16(rng, (1, H, D))
    kq = rng.integers(-127, 128, (N, Hk, D), dtype=np.int8)
    vq = rng.integers(-127, 128, (N, Hk, D), dtype=np.int8)
    kd = rng.uniform(0.001, 0.02, (N, Hk, D // 32)).astype(np.float16)
    vd = rng.uniform(0.001, 0.02, (N, Hk, D // 32)).astype(np.float16)
    out, lse = kvattn.decode(dev(q), dev(kq), dev(vq), dev(np.array([N], np.int32)), split=split,
                             k_scales=dev(kd), v_scales=dev(vd))
    torch.cuda.synchronize()
    wo, wl = oracle.decode_q8_0(q, kq, kd, vq, vd, [N])
    assert_close(out, lse, wo, wl)


def small_unified(rng, S=3, pool_records=40, H=24, Hk=4, D=128, hole=0.25):
    """A unified cache of pool_records x 128 cells, sequences owning scattered records."""
    n_cells = pool_records * 128
    perm = rng.permutation(pool_records)
    owned = [perm[0:3], perm[3:10], perm[10:11]][:S]
    encoded, selected = [], []
    for recs in owned:
        cells = (recs[:, None] * 128 + np.arange(128)[None]).reshape(-1)
        keep = rng.random(cells.size) >= hole
        keep[0] = True
        sel = cells[keep]
        enc = np.concatenate([sel, sel[: sel.size // 10]])
        rng.shuffle(enc)
        encoded.append((rng.integers(0, 8, enc.size).astype(np.int64) << 32) | enc.astype(np.int64))
        selected.append(sel)
    k = rand_f16(rng, (n_cells, Hk, D))
    v = rand_f16(rng, (n_cells, Hk, D))
    unused = np.setdiff1d(np.arange(n_cells), np.concatenate(selected))
    k[unused] = np.nan
    v[unused] = np.nan
    q = rand_f16(rng, (S, H, D))
    return q, k, v, encoded, n_cells


@pytest.mark.parametrize("split", [32, 128, 256])
def test_plan_with_holes_over_nan_cells(kvattn, split):
    import torch
    rng = np.random.default_rng(split)
    q, k, v, encoded, n_cells = small_unified(rng)
    plan, lens = kvattn.build_cell_plan(encoded, n_cells)
    wplan, wlens = po.build_cell_plan([e.tolist() for e in encoded], n_cells)
    assert np.array_equal(plan, wplan) and np.array_equal(lens, wlens)
    out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(lens), split=split, cell_plan=dev(plan),
                             n_cells=n_cells)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_f16(q, k, v, lens.tolist(), plan=plan)
    assert_close(out, lse, wo, wl)


def test_descriptors_bit_exact(kvattn):
    import torch
    rng = np.random.default_rng(9)
    q, k, v, encoded, n_cells = small_unified(rng)
    plan, lens = kvattn.build_cell_plan(encoded, n_cells, plan_stride=1200)
    plan[0, 5] = -7              # out-of-range entries: masked and flagged
    plan[1, 300] = n_cells + 3
    for split, max_len in [(128, 1200), (96, 1100), (64, 500)]:
        n_split = -(-max_len // split)
        desc = torch.zeros((plan.shape[0], n_split, 4), dtype=torch.int32, device="cuda")
        kvattn.kvattn_build_descriptors(dev(plan), plan.shape[1], dev(lens), plan.shape[0], max_len, split,
                                        n_cells, desc)
        torch.cuda.synchronize()
        want = po.descriptors(plan, lens, max_len, split, n_cells)
        assert np.array_equal(desc.cpu().numpy(), want)


@pytest.mark.parametrize("kv", ["f16", "q8_0"])
def test_decode_leaves_the_split_descriptors_in_the_workspace(kvattn, kv):
    """kvattn_decode with a plan leaves every split's descriptor at byte 256 of the
    workspace, bit-exact with the CPU mirror (the f16 kernels compute them in their producer
    warp, the quantised ones read them from a descriptor launch): out-of-range entries, a
    fully masked split, splits past a sequence's length, max_len below the plan stride."""
    import torch
    rng = np.random.default_rng(12)
    q, k, v, encoded, n_cells = small_unified(rng)
    plan, lens = kvattn.build_cell_plan(encoded, n_cells, plan_stride=1200)
    plan[0, 5] = -7
    plan[1, 300] = n_cells + 3
    plan[1, 128:256] = -1        # a fully masked split (128..255 of a 896-entry row)
    S, H, D = q.shape
    Hk = k.shape[1]
    masked = plan.copy()
    masked[(masked < -1) | (masked >= n_cells)] = -1
    for split, max_len in [(128, 1200), (64, 1100), (32, 500)]:
        n_split = -(-max_len // split)
        ws = kvattn.decode_workspace(S, H, D, max_len, split)
        ws.fill_(0xEE)
        ws[:256].zero_()
        if kv == "f16":
            out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(lens), split=split, cell_plan=dev(plan),
                                     n_cells=n_cells, max_len=max_len, ws=ws)
            wo, wl = oracle.decode_f16(q, k, v, np.minimum(lens, max_len).tolist(), plan=masked)
        else:
            kq = rng.integers(-127, 128, (n_cells, Hk, D), dtype=np.int8)
            vq = rng.integers(-127, 128, (n_cells, Hk, D), dtype=np.int8)
            kd = rng.uniform(0.001, 0.02, (n_cells, Hk, D // 32)).astype(np.float16)
            vd = rng.uniform(0.001, 0.02, (n_cells, Hk, D // 32)).astype(np.float16)
            out, lse = kvattn.decode(dev(q), dev(kq), dev(vq), dev(lens), split=split, cell_plan=dev(plan),
                                     n_cells=n_cells, max_len=max_len, ws=ws, k_scales=dev(kd), v_scales=dev(vd))
            wo, wl = oracle.decode_q8_0(q, kq, kd, vq, vd, np.minimum(lens, max_len).tolist(), plan=masked)
        torch.cuda.synchronize()
        got = ws[256:256 + S * n_split * 16].view(torch.int32).view(S, n_split, 4).cpu().numpy()
        want = po.descriptors(plan, lens, max_len, split, n_cells)
        assert np.array_equal(got, want), (split, max_len)
        assert kvattn.kvattn_workspace_status(ws) & kvattn.KVATTN_DEVICE_BAD_PLAN_ENTRY
        assert_close(out, lse, wo, wl)


def test_bad_plan_entries_are_masked_and_flagged(kvattn):
    import torch
    rng = np.random.default_rng(10)
    q, k, v, encoded, n_cells = small_unified(rng)
    plan, lens = kvattn.build_cell_plan(encoded, n_cells)
    bad = plan.copy()
    bad[0, 3] = -9
    bad[1, 130] = n_cells + 100
    ws = kvattn.decode_workspace(q.shape[0], q.shape[1], q.shape[2], bad.shape[1], 128)
    out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(lens), split=128, cell_plan=dev(bad),
                             n_cells=n_cells, ws=ws)
    flags = kvattn.kvattn_workspace_status(ws, clear=True)
    assert flags & kvattn.KVATTN_DEVICE_BAD_PLAN_ENTRY
    masked = bad.copy()
    masked[0, 3] = -1
    masked[1, 130] = -1
    wo, wl = oracle.decode_f16(q, k, v, lens.tolist(), plan=masked)
    assert_close(out, lse, wo, wl)
    assert kvattn.kvattn_workspace_status(ws) == 0


def test_split_sweep_agrees(kvattn):
    rng = np.random.default_rng(11)
    N, H, Hk, D = 5000, 32, 8, 128
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    wo, wl = oracle.decode_f16(q, k, v, [N])
    outs = []
    for split in (32, 64, 128, 256, 512, 5024):
        out, lse = run_contiguous(kvattn, q, k, v, [N], split)
        assert_close(out, lse, wo, wl)
        outs.append(out.cpu().numpy())
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= TOL_O


def test_deterministic_bits(kvattn):
    rng = np.random.default_rng(12)
    N, H, Hk, D = 3000, 32, 8, 128
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    a = [t.cpu().numpy() for t in run_contiguous(kvattn, q, k, v, [N], 128)]
    b = [t.cpu().numpy() for t in run_contiguous(kvattn, q, k, v, [N], 128)]
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_gqa_matches_mha_with_repeated_kv(kvattn):
    rng = np.random.default_rng(13)
    N, H, Hk, D = 700, 24, 4, 128
    G = H // Hk
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    go, gl = run_contiguous(kvattn, q, k, v, [N], 128)
    mo, ml = run_contiguous(kvattn, q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), [N], 128)
    assert np.max(np.abs(go.cpu().numpy() - mo.cpu().numpy())) <= 1e-5
    assert np.max(np.abs(gl.cpu().numpy() - ml.cpu().numpy())) <= 1e-6


def test_merge_kernel(kvattn):
    import torch
    rng = np.random.default_rng(14)
    P, R, D = 37, 40, 128
    parts = rng.standard_normal((P, R, D)).astype(np.float32)
    lses = (rng.standard_normal((P, R)) * 4).astype(np.float32)
    lses[3] = -np.inf
    parts[3] = np.nan            # an empty part's O is never read
    lses[:, 7] = -np.inf         # a row with no cells at all
    out, lse = kvattn.merge(dev(parts), dev(lses))
    torch.cuda.synchronize()
    wo, wl = oracle.merge(parts.astype(np.float64), lses.astype(np.float64))
    assert_close(out, lse, wo, wl, tol_o=1e-5, tol_l=1e-5)


def test_output_guard_regions_untouched(kvattn):
    import torch
    rng = np.random.default_rng(15)
    N, H, Hk, D = 900, 16, 4, 128
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    guard = 1024
    big_o = torch.full((H * D + 2 * guard,), 12345.0, device="cuda")
    big_l = torch.full((H + 2 * guard,), 12345.0, device="cuda")
    out = big_o[guard:guard + H * D].view(1, H, D)
    lse = big_l[guard:guard + H].view(1, H)
    kvattn.decode(dev(q), dev(k), dev(v), dev(np.array([N], np.int32)), split=128, out=out, lse=lse)
    torch.cuda.synchronize()
    bo, bl = big_o.cpu().numpy(), big_l.cpu().numpy()
    assert np.all(bo[:guard] == 12345.0) and np.all(bo[-guard:] == 12345.0)
    assert np.all(bl[:guard] == 12345.0) and np.all(bl[-guard:] == 12345.0)
    wo, wl = oracle.decode_f16(q, k, v, [N])
    assert_close(out, lse, wo, wl)


def test_bounded_wait_reports_timeout_and_context_survives(kvattn, monkeypatch):
    """A pipeline wait that can never complete gives up after its limit and reports it."""
    import torch
    rng = np.random.default_rng(16)
    N, H, Hk, D = 256, 8, 2, 128
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    ws = kvattn.decode_workspace(1, H, D, N, 128)
    monkeypatch.setenv("KVATTN_DEBUG_STALL_TX", "16")
    monkeypatch.setenv("KVATTN_DEBUG_WAIT_MS", "20")
    kvattn.decode(dev(q), dev(k), dev(v), dev(np.array([N], np.int32)), split=128, ws=ws)
    torch.cuda.synchronize()
    assert kvattn.kvattn_workspace_status(ws, clear=True) & kvattn.KVATTN_DEVICE_WAIT_TIMEOUT
    monkeypatch.delenv("KVATTN_DEBUG_STALL_TX")
    out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(np.array([N], np.int32)), split=128, ws=ws)
    torch.cuda.synchronize()
    assert kvattn.kvattn_workspace_status(ws) == 0
    wo, wl = oracle.decode_f16(q, k, v, [N])
    assert_close(out, lse, wo, wl)


def test_partials_then_merge_equals_decode(kvattn):
    import torch
    rng = np.random.default_rng(17)
    S, N, H, Hk, D, split = 2, 3000, 16, 4, 128, 256
    q = rand_f16(rng, (S, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    lens = np.array([3000, 900], np.int32)
    n_split = -(-N // split)
    part_o = torch.empty((S, n_split, H, D), dtype=torch.float32, device="cuda")
    part_l = torch.empty((S, n_split, H), dtype=torch.float32, device="cuda")
    ws = kvattn.decode_workspace(S, H, D, N, split)
    kvattn.kvattn_decode_partials(dev(q), dev(k), dev(v), None, None, 0, N, None, 0, dev(lens), S, N, H, Hk,
                                  D, split, 1 / np.sqrt(D), part_o, part_l, ws, ws.numel())
    torch.cuda.synchronize()
    pl = part_l.cpu().numpy()
    assert np.all(np.isneginf(pl[1, -(-900 // split):]))      # splits past the length
    assert np.all(np.isfinite(pl[1, :-(-900 // split)]))
    wo, wl = oracle.decode_f16(q, k, v, lens.tolist())
    for s in range(S):
        mo, ml = kvattn.merge(part_o[s].contiguous(), part_l[s].contiguous())
        torch.cuda.synchronize()
        assert_close(mo.view(1, H, D), ml.view(1, H), wo[s:s + 1], wl[s:s + 1])
    # kvattn_decode combines splits in clusters before its final merge: the same values up
    # to the order of the fp32 reductions
    do, dl = run_contiguous(kvattn, q, k, v, lens, split)
    for s in range(S):
        mo, ml = kvattn.merge(part_o[s].contiguous(), part_l[s].contiguous())
        torch.cuda.synchronize()
        assert np.max(np.abs(mo.cpu().numpy() - do.cpu().numpy()[s])) <= 1e-5
        assert np.max(np.abs(ml.cpu().numpy() - dl.cpu().numpy()[s])) <= 1e-5


@pytest.mark.parametrize("kv,D,S,N", [("f16", 128, 1, 16384), ("f16", 256, 3, 3000), ("q8", 128, 2, 9000)])
def test_split_zero_selects_a_split(kvattn, kv, D, S, N):
    """split 0: kvattn_decode picks the split with kvattn_select_split (one wave of units)."""
    import torch
    rng = np.random.default_rng(N + D)
    Hk, G = 4, 4
    H = Hk * G
    kind = kvattn.KVATTN_KV_F16 if kv == "f16" else kvattn.KVATTN_KV_Q8_0
    sp = kvattn.kvattn_select_split(kind, S, N, Hk, D)
    assert sp >= 64 and sp & (sp - 1) == 0
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    # the device rule agrees with the pure one for some resident count of whole CTAs per SM
    assert any(kvattn.kvattn_select_split_for(S, N, Hk, sm * b) == sp for b in range(1, 17))
    q = rand_f16(rng, (S, H, D))
    lens = np.array([N - 7 * s for s in range(S)], np.int32)
    if kv == "f16":
        k = rand_f16(rng, (S, N, Hk, D))
        v = rand_f16(rng, (S, N, Hk, D))
        out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(lens), split=0, n_cells=N, max_len=N)
        torch.cuda.synchronize()
        wo, wl = oracle.decode_f16(q, k, v, lens.tolist())
    else:
        kq = rng.integers(-127, 128, (S, N, Hk, D), dtype=np.int8)
        vq = rng.integers(-127, 128, (S, N, Hk, D), dtype=np.int8)
        kd = rng.uniform(0.001, 0.02, (S, N, Hk, D // 32)).astype(np.float16)
        vd = rng.uniform(0.001, 0.02, (S, N, Hk, D // 32)).astype(np.float16)
        out, lse = kvattn.decode(dev(q), dev(kq), dev(vq), dev(lens), split=0, n_cells=N, max_len=N,
                                 k_scales=dev(kd), v_scales=dev(vd))
        torch.cuda.synchronize()
        wo, wl = oracle.decode_q8_0(q, kq, kd, vq, vd, lens.tolist())
    assert_close(out, lse, wo, wl)


def test_calls_from_several_host_threads(kvattn):
    """Four host threads, each with its own stream and workspace, decode at once (the first
    calls on a fresh process race to fill the library's per-device caches)."""
    import threading

    import torch
    rng = np.random.default_rng(13)
    cases = []
    for t in range(4):
        N, D = 900 + 300 * t, (128, 256)[t % 2]
        q = rand_f16(rng, (1, 16, D))
        k = rand_f16(rng, (N, 4, D))
        v = rand_f16(rng, (N, 4, D))
        cases.append((q, k, v, N))
    results = [None] * 4
    errors = []

    def work(t):
        try:
            q, k, v, N = cases[t]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                qd, kd, vd = dev(q), dev(k), dev(v)
                lens = dev(np.array([N], np.int32))
                for _ in range(5):
                    out, lse = kvattn.decode(qd, kd, vd, lens, split=0, stream=s)
                s.synchronize()
                results[t] = (out.cpu().numpy(), lse.cpu().numpy())
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for (q, k, v, N), (o, l) in zip(cases, results):
        wo, wl = oracle.decode_f16(q, k, v, [N])
        assert np.max(np.abs(o - wo)) <= TOL_O and np.max(np.abs(l - wl)) <= 1e-4


def test_more_than_65535_sequences(kvattn):
    """70000 short sequences in one call (a batch far past the 16-bit grid limit of older
    designs): units and merge rows are numbered in 32 bits; a sample of rows against the
    oracle, the rest against the sequences' own properties (finite, empty where empty)."""
    import torch
    rng = np.random.default_rng(14)
    S, N, H, Hk, D = 70000, 24, 2, 1, 128
    lens = rng.integers(0, N + 1, S).astype(np.int32)
    lens[:3] = [N, 0, 1]
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    q = rand_f16(rng, (S, H, D))
    out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(lens), split=32, n_cells=N, max_len=N)
    torch.cuda.synchronize()
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert np.array_equal(np.isneginf(l), (lens == 0)[:, None].repeat(H, 1))
    assert np.all(np.isfinite(o)) and np.all(o[lens == 0] == 0)
    pick = np.concatenate([[0, 1, 2], rng.choice(S, 200, replace=False), [S - 1]])
    wo, wl = oracle.decode_f16(q[pick], k[pick], v[pick], lens[pick].tolist())
    assert_close(out[pick], lse[pick], wo, wl)


def test_launch_trace_only_on_request(kvattn, monkeypatch, capfd):
    """KVATTN_LOG=1: one stderr line per launching call with the decisions taken; silent
    otherwise."""
    import torch
    rng = np.random.default_rng(15)
    N, H, Hk, D = 4096, 32, 8, 128
    q, k, v = rand_f16(rng, (1, H, D)), rand_f16(rng, (N, Hk, D)), rand_f16(rng, (N, Hk, D))
    args = (dev(q), dev(k), dev(v), dev(np.array([N], np.int32)))
    capfd.readouterr()
    kvattn.decode(*args, split=256)
    torch.cuda.synchronize()
    assert capfd.readouterr().err == ""
    monkeypatch.setenv("KVATTN_LOG", "1")
    kvattn.decode(*args, split=0)
    torch.cuda.synchronize()
    err = capfd.readouterr().err
    monkeypatch.delenv("KVATTN_LOG")
    lines = [ln for ln in err.splitlines() if ln.startswith("kvattn: decode ")]
    assert len(lines) == 1, err
    sp = kvattn.kvattn_select_split(0, 1, N, Hk, D)
    assert f"split={sp} " in lines[0] and f"n_split={-(-N // sp)} " in lines[0] and "plan=0" in lines[0]
