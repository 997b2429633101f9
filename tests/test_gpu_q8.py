"""GPU parity of the Q8_0 decode kernels (self-loading warps, 16-cell chunks) against the
fp64 oracle: compact plans with holes (one-run chunks through TMA, scattered chunks through
per-row copies), several sequences with ragged and empty lengths, fully masked splits,
partial slots past a sequence's length, and the bounded pipeline wait.

Unselected cells carry NaN scales: a masked cell whose scale reached the arithmetic would
turn its row's output into NaN.
"""
import numpy as np
import pytest

import oracle
from oracle import plan_oracle as po
from tests.gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu


def q8_cache(rng, n_cells, Hk, D):
    kq = rng.integers(-127, 128, (n_cells, Hk, D), dtype=np.int8)
    vq = rng.integers(-127, 128, (n_cells, Hk, D), dtype=np.int8)
    kd = rng.uniform(0.001, 0.02, (n_cells, Hk, D // 32)).astype(np.float16)
    vd = rng.uniform(0.001, 0.02, (n_cells, Hk, D // 32)).astype(np.float16)
    return kq, vq, kd, vd


def run(K, q, kq, vq, kd, vd, lens, split, plan=None, n_cells=None, max_len=None):
    import torch
    out, lse = K.decode(dev(q), dev(kq), dev(vq), dev(np.asarray(lens, np.int32)), split=split,
                        k_scales=dev(kd), v_scales=dev(vd), cell_plan=None if plan is None else dev(plan),
                        n_cells=n_cells, max_len=max_len)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("D,G,split", [(128, 4, 128), (128, 6, 256), (256, 8, 128), (256, 1, 64)])
def test_q8_0_compact_plan_with_holes(kvattn, D, G, split):
    """Records of 128 cells with ~25 % holes: every 16-cell chunk is one physical run (TMA)."""
    rng = np.random.default_rng(100 + D + G)
    Hk, pool = 2, 24
    H = Hk * G
    n_cells = pool * 128
    kq, vq, kd, vd = q8_cache(rng, n_cells, Hk, D)
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
    out, lse = run(kvattn, q, kq, vq, kd, vd, lens, split, plan=plan, n_cells=n_cells, max_len=plan.shape[1])
    wo, wl = oracle.decode_q8_0(q, kq, kd, vq, vd, lens.tolist(), plan=plan)
    assert_close(out, lse, wo, wl)


@pytest.mark.parametrize("D", [128, 256])
def test_q8_0_scattered_plan(kvattn, D):
    """Plan entries in random order (most chunks are not one run: per-row copies), -1 holes,
    a fully masked split, and an empty sequence."""
    rng = np.random.default_rng(200 + D)
    Hk, G, split = 4, 4, 64
    H = Hk * G
    n_cells = 3000
    kq, vq, kd, vd = q8_cache(rng, n_cells, Hk, D)
    stride = 700
    lens = np.array([700, 0, 333, 64], np.int32)
    plan = np.full((4, stride), -1, np.int32)
    used = np.zeros(n_cells, bool)
    for s, L in enumerate(lens):
        cells = rng.choice(n_cells, size=L, replace=False).astype(np.int32)
        cells[rng.random(L) < 0.2] = -1
        plan[s, :L] = cells
        used[cells[cells >= 0]] = True
    plan[0, 128:192] = -1          # one split of sequence 0 holds no valid cell
    plan[2, 32:48] = np.arange(1000, 1016, dtype=np.int32)   # one chunk that is a run
    used[1000:1016] = True
    kd[~used] = np.nan
    vd[~used] = np.nan
    q = rng.standard_normal((4, H, D), dtype=np.float32).astype(np.float16)
    out, lse = run(kvattn, q, kq, vq, kd, vd, lens, split, plan=plan, n_cells=n_cells, max_len=stride)
    wo, wl = oracle.decode_q8_0(q, kq, kd, vq, vd, lens.tolist(), plan=plan)
    assert_close(out, lse, wo, wl)
    assert np.all(np.isneginf(lse.cpu().numpy()[1]))


@pytest.mark.parametrize("D", [128, 256])
def test_q8_0_multi_sequence_ragged(kvattn, D):
    rng = np.random.default_rng(300 + D)
    S, N, Hk, G, split = 3, 1100, 2, 5, 128
    H = Hk * G
    kq, vq, kd, vd = q8_cache(rng, S * N, Hk, D)
    kq, vq = kq.reshape(S, N, Hk, D), vq.reshape(S, N, Hk, D)
    kd, vd = kd.reshape(S, N, Hk, D // 32), vd.reshape(S, N, Hk, D // 32)
    lens = [1100, 0, 17]
    q = rng.standard_normal((S, H, D), dtype=np.float32).astype(np.float16)
    out, lse = run(kvattn, q, kq, vq, kd, vd, lens, split, n_cells=N, max_len=N)
    wo, wl = oracle.decode_q8_0(q, kq, kd, vq, vd, lens)
    assert_close(out, lse, wo, wl)


def test_q8_0_partials_past_length(kvattn):
    """kvattn_decode_partials writes (0, -inf) in every slot past a sequence's length, and
    the written partials merge to the decode result."""
    import torch
    rng = np.random.default_rng(400)
    S, N, Hk, G, D, split = 2, 2048, 2, 4, 128, 256
    H = Hk * G
    kq, vq, kd, vd = q8_cache(rng, S * N, Hk, D)
    kq, vq = kq.reshape(S, N, Hk, D), vq.reshape(S, N, Hk, D)
    kd, vd = kd.reshape(S, N, Hk, D // 32), vd.reshape(S, N, Hk, D // 32)
    lens = np.array([2048, 500], np.int32)
    q = rng.standard_normal((S, H, D), dtype=np.float32).astype(np.float16)
    n_split = N // split
    part_o = torch.full((S, n_split, H, D), float("nan"), dtype=torch.float32, device="cuda")
    part_l = torch.full((S, n_split, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = kvattn.decode_workspace(S, H, D, N, split)
    kvattn.kvattn_decode_partials(dev(q), dev(kq), dev(vq), dev(kd), dev(vd), kvattn.KVATTN_KV_Q8_0, N, None, 0,
                                  dev(lens), S, N, H, Hk, D, split, 1 / np.sqrt(D), part_o, part_l, ws, ws.numel())
    torch.cuda.synchronize()
    pl, po_ = part_l.cpu().numpy(), part_o.cpu().numpy()
    used = -(-500 // split)
    assert np.all(np.isneginf(pl[1, used:])) and np.all(po_[1, used:] == 0)
    assert np.all(np.isfinite(pl[:, :used])) and np.all(np.isfinite(pl[0]))
    wo, wl = oracle.decode_q8_0(q, kq, kd, vq, vd, lens.tolist())
    for s in range(S):
        mo, ml = oracle.merge(po_[s], pl[s])
        assert np.max(np.abs(mo - wo[s])) <= 2e-3 and np.max(np.abs(ml - wl[s])) <= 1e-4


def test_q8_0_bounded_wait_reports_timeout_and_context_survives(kvattn, monkeypatch):
    import torch
    rng = np.random.default_rng(500)
    N, Hk, G, D = 512, 2, 4, 128
    H = Hk * G
    kq, vq, kd, vd = q8_cache(rng, N, Hk, D)
    q = rng.standard_normal((1, H, D), dtype=np.float32).astype(np.float16)
    ws = kvattn.decode_workspace(1, H, D, N, 128)
    monkeypatch.setenv("KVATTN_DEBUG_STALL_TX", "16")
    monkeypatch.setenv("KVATTN_DEBUG_WAIT_MS", "20")
    kvattn.decode(dev(q), dev(kq), dev(vq), dev(np.array([N], np.int32)), split=128, k_scales=dev(kd),
                  v_scales=dev(vd), ws=ws)
    torch.cuda.synchronize()
    assert kvattn.kvattn_workspace_status(ws, clear=True) & kvattn.KVATTN_DEVICE_WAIT_TIMEOUT
    monkeypatch.delenv("KVATTN_DEBUG_STALL_TX")
    out, lse = kvattn.decode(dev(q), dev(kq), dev(vq), dev(np.array([N], np.int32)), split=128,
                             k_scales=dev(kd), v_scales=dev(vd), ws=ws)
    torch.cuda.synchronize()
    assert kvattn.kvattn_workspace_status(ws) == 0
    wo, wl = oracle.decode_q8_0(q, kq, kd, vq, vd, [N])
    assert_close(out, lse, wo, wl)


@pytest.mark.parametrize("kv", ["q8", "q8q4", "q4"])
@pytest.mark.parametrize("G,Hk", [(4, 8), (2, 2), (1, 4)])
def test_head_pairs_equal_single_heads(kvattn, monkeypatch, kv, G, Hk):
    """KV-head pairs (the default for head_dim 128, G <= 4, even KV-head counts) and one KV
    head per work unit (KVATTN_PAIR=0) both match the oracle and agree with each other to
    rounding; a compact plan with holes over NaN-scaled cells, ragged lengths."""
    import torch
    import oracle
    from oracle import plan_oracle as po
    rng = np.random.default_rng([37, G, Hk, len(kv)])
    D, pool = 128, 16
    H = G * Hk
    n_cells = pool * 128
    kq = (rng.integers(0, 256, (n_cells, Hk, D // 2), dtype=np.uint8) if kv == "q4"
          else rng.integers(-127, 128, (n_cells, Hk, D), dtype=np.int8))
    kd = rng.uniform(0.001, 0.3 if kv == "q4" else 0.02, (n_cells, Hk, D // 32)).astype(np.float16)
    vq = (rng.integers(-127, 128, (n_cells, Hk, D), dtype=np.int8) if kv == "q8"
          else rng.integers(0, 256, (n_cells, Hk, D // 2), dtype=np.uint8))
    vd = rng.uniform(0.001, 0.02 if kv == "q8" else 0.3, (n_cells, Hk, D // 32)).astype(np.float16)
    perm = rng.permutation(pool)
    encoded, selected = [], []
    for recs in (perm[:5], perm[5:6], perm[6:12]):
        cells = (recs[:, None] * 128 + np.arange(128)[None]).reshape(-1)
        sel = cells[rng.random(cells.size) >= 0.25]
        encoded.append(sel.astype(np.int64)[rng.permutation(sel.size)])
        selected.append(sel)
    unused = np.setdiff1d(np.arange(n_cells), np.concatenate(selected))
    kd[unused] = np.nan
    vd[unused] = np.nan
    plan, lens = kvattn.build_cell_plan(encoded, n_cells)
    q = rng.standard_normal((3, H, D), dtype=np.float32).astype(np.float16)
    kt = {"q8": kvattn.KVATTN_KV_Q8_0, "q8q4": kvattn.KVATTN_KV_Q8_0_Q4_0, "q4": kvattn.KVATTN_KV_Q4_0}[kv]
    res = []
    for pair in ("1", "0"):
        monkeypatch.setenv("KVATTN_PAIR", pair)
        out, lse = kvattn.decode(dev(q), dev(kq), dev(vq), dev(lens), split=128, k_scales=dev(kd), v_scales=dev(vd),
                                 cell_plan=dev(plan), n_cells=n_cells, kv_type=kt)
        torch.cuda.synchronize()
        res.append((out.cpu().numpy(), lse.cpu().numpy()))
    fn = {"q8": oracle.decode_q8_0, "q8q4": oracle.decode_q8_0_q4_0, "q4": oracle.decode_q4_0}[kv]
    wo, wl = fn(q, kq, kd, vq, vd, lens.tolist(), plan=plan)
    for o, l in res:
        assert_close(torch.from_numpy(o), torch.from_numpy(l), wo, wl)
    # the two geometries give a warp different cells (two warps per pair unit, four per
    # single-head unit), so their running maxima and the f16 roundings of P differ: the
    # results agree to rounding, not bit for bit
    assert np.max(np.abs(res[0][0] - res[1][0])) <= 1e-3
    assert np.max(np.abs(res[0][1] - res[1][1])) <= 1e-4
