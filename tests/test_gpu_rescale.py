"""GPU parity of the online-softmax rescale and of the ``scale`` argument, in every kernel
family, against the fp64 oracle.

Flash-decoding is exact only if every running maximum that moves rescales what was summed
before it ("KVARN KV Performance optimizations", item 9: a partial window keeps its maximum,
numerator and denominator; the merge of partials is the same step one level up).  The
kernels move their reference maximum lazily, only when a row's maximum grows by more than
2^8 (in exp2 units), so inputs drawn N(0, 1) at the default scale never reach that branch
after a unit's first tile.  The inputs here are shaped to reach it:

* ``ramp_split``    the scores climb a 16-step staircase through every split (about 3 natural
                    units per step, 45 per split): the reference moves every second step;
* ``ramp_global``   a steeper staircase over the whole sequence (6 units per step, more than
                    the slack): every step moves it, and early splits merge with weights of
                    e^-90;
* ``dominant_last`` one cell 30 units above the rest at the last valid position of every
                    split: the move comes on a unit's last tile, after all the others;
* ``dominant_mid``  the same cell in the second 16-cell half of a middle 32-cell tile (the
                    second consumer warp's cells, an odd 16-cell chunk of the quantised
                    kernels);
* ``q_x8``, ``q_x16``  queries scaled by 8 and 16 (peaked softmax, maxima that keep moving);
* ``scale_1``, ``scale_0p01``  a non-default softmax scale;
* ``offset_p200``, ``offset_m200``  every score shifted by +200 and -200 natural units.

Two control dimensions carry the shape: K[., 0] and K[., 1] hold multiples of 0.5 in
[-4, 3.5] (representable exactly in f16, in a Q8_0 block of scale 1/16 and in a Q4_0 block of
scale 1/2), and the query's dimensions 0 and 1 weight them.  Every query value is a multiple
of 1/16 and every key value a multiple of 2^-7 with power-of-two block scales, so each score
q.K is exact in fp32 whatever the order of summation: the comparison checks the softmax
arithmetic, not the rounding of a 128-term dot product around 2000.
"""
import numpy as np
import pytest

import oracle
from tests.gpu_util import TOL_LSE, TOL_O, TOL_RMSE_O, assert_close, dev

pytestmark = pytest.mark.gpu

CASES = ["ramp_split", "ramp_global", "dominant_last", "dominant_mid", "q_x8", "q_x16", "scale_1",
         "scale_0p01", "offset_p200", "offset_m200"]
# cases built so that the lazy reference maximum must move after a unit's first 16 cells
MOVING = {"ramp_split", "ramp_global", "dominant_last", "dominant_mid", "q_x16", "scale_1"}

KIND_ORACLE = {"f16": oracle.decode_f16, "q8": oracle.decode_q8_0, "q8q4": oracle.decode_q8_0_q4_0,
               "q4": oracle.decode_q4_0}


def grid16(x):
    """Round to a multiple of 1/16 and store as f16 (exact below 2048 in magnitude)."""
    return (np.round(np.asarray(x, np.float64) * 16.0) / 16.0).astype(np.float16)


def controls(case, lens, N, split):
    """Per (sequence, logical position) control values kc0, kc1 and the natural-log score
    each unit of them adds (a_nat, b_nat), the query multiplier and the softmax scale."""
    S = len(lens)
    kc0 = np.zeros((S, N))
    kc1 = np.zeros((S, N))
    a_nat = b_nat = 0.0
    qmul, scale = 1.0, None
    pos = np.arange(N)
    if case == "ramp_split":
        kc1[:] = 0.5 * np.floor(16 * (pos % split) / split) - 4.0
        b_nat = 6.0                      # 3 natural units per 0.5 step
    elif case == "ramp_global":
        for s, L in enumerate(lens):
            L = max(L, 1)
            kc1[s] = 0.5 * np.minimum(np.floor(16 * pos / L), 15) - 4.0
        b_nat = 12.0                     # 6 per step: more than 2^8 in exp2 units
    elif case in ("dominant_last", "dominant_mid"):
        for s, L in enumerate(lens):
            for s0 in range(0, L, split):
                n_here = min(split, L - s0)
                if case == "dominant_last":
                    c = s0 + n_here - 1
                else:
                    c = s0 + 32 * ((n_here // 32) // 2) + 21
                    if c >= s0 + n_here:
                        c = s0 + n_here - 1
                kc0[s, c] = 3.5
        a_nat = 30.0 / 3.5
    elif case == "q_x8":
        qmul = 8.0
    elif case == "q_x16":
        qmul = 16.0
    elif case == "scale_1":
        scale = 1.0
    elif case == "scale_0p01":
        scale = 0.01
    elif case in ("offset_p200", "offset_m200"):
        kc0[:] = 1.0
        a_nat = 200.0 if case == "offset_p200" else -200.0
    else:
        raise ValueError(case)
    return kc0, kc1, a_nat, b_nat, qmul, scale


def make_q(rng, lead, D, a_nat, b_nat, qmul, scale):
    """q [*lead][D]: N(0,1) x qmul on the 1/16 grid; dims 0 and 1 weight the controls."""
    q = grid16(rng.standard_normal(tuple(lead) + (D,)) * qmul).astype(np.float64)
    sc = scale if scale is not None else 1.0 / np.sqrt(D)
    q[..., 0] = float(grid16(a_nat / sc))
    q[..., 1] = float(grid16(b_nat / sc))
    return q.astype(np.float16)


def make_cache(rng, kind, lead, D, kc0, kc1):
    """K (with the control values in dims 0, 1) and V in the cache format ``kind``.
    lead: the cell-major leading shape ([S, N, Hk] or [N, Hk]); kc0/kc1 broadcast over the KV
    heads.  Returns the cache arguments in the order the oracle and ``kvattn.decode`` take."""
    lead = tuple(lead)
    nb = D // 32
    kc0 = np.broadcast_to(np.asarray(kc0)[..., None], lead)
    kc1 = np.broadcast_to(np.asarray(kc1)[..., None], lead)
    # block 0: multiples of 0.5 in [-2, 2] beside the two controls
    blk0 = 0.5 * rng.integers(-4, 5, lead + (32,)).astype(np.float64)
    blk0[..., 0] = kc0
    blk0[..., 1] = kc1
    if kind == "f16":
        k = grid16(np.clip(rng.standard_normal(lead + (D,)), -4, 4)).astype(np.float64)
        k[..., :32] = blk0
        v = rng.standard_normal(lead + (D,)).astype(np.float16)
        return (k.astype(np.float16), v)
    if kind in ("q8", "q8q4"):
        kq = rng.integers(-127, 128, lead + (D,)).astype(np.int8)
        kd = (2.0 ** -rng.integers(5, 8, lead + (nb,))).astype(np.float16)
        kq[..., :32] = (16 * blk0).astype(np.int8)
        kd[..., 0] = 1.0 / 16
    else:
        lo = rng.integers(0, 16, lead + (nb, 16))
        hi = rng.integers(0, 16, lead + (nb, 16))
        # block 0 holds element j in the low nibble of byte j, element 16 + j in the high one
        n0 = (2 * blk0 + 8).astype(np.int64)
        lo[..., 0, :] = n0[..., :16]
        hi[..., 0, :] = n0[..., 16:]
        kq = (lo | (hi << 4)).astype(np.uint8).reshape(lead + (D // 2,))
        kd = (2.0 ** -rng.integers(2, 4, lead + (nb,))).astype(np.float16)
        kd[..., 0] = 0.5
    if kind == "q8":
        vq = rng.integers(-127, 128, lead + (D,)).astype(np.int8)
        vd = rng.uniform(0.001, 0.02, lead + (nb,)).astype(np.float16)
    else:
        vq = rng.integers(0, 256, lead + (D // 2,)).astype(np.uint8)
        vd = rng.uniform(0.001, 0.3, lead + (nb,)).astype(np.float16)
    return (kq, kd, vq, vd)


def dequant_k(kind, cache):
    if kind == "f16":
        return cache[0].astype(np.float64)
    if kind in ("q8", "q8q4"):
        return oracle.dequant_q8_0(cache[0], cache[1])
    return oracle.dequant_q4_0(cache[0], cache[1])


def moves(q, kind, cache, lens, split, scale, n_q=1, strides=(1, 2, 4)):
    """How often the lazy reference maximum (slack 2^8 in exp2 units) would move after the
    first 16-cell chunk of a unit, when a warp walks every s-th chunk of each split (s = 1,
    2, 4 covers the kernels' cell-to-warp assignments).  A property of the inputs alone: the
    scores come from numpy on the exact dequantised values."""
    K = dequant_k(kind, cache)
    if K.ndim == 3:
        K = K[None]
    qq = q.astype(np.float64)
    if qq.ndim == 3:
        qq = qq[:, None]
    S, _, H, D = qq.shape
    Hk = K.shape[2]
    G = H // Hk
    sc = scale if scale is not None else 1.0 / np.sqrt(D)
    total = 0
    for s, L in enumerate(lens):
        for h in range(0, H, max(1, H // 4)):
            x = (K[s, :L, h // G] @ qq[s, n_q - 1, h]) * sc / np.log(2.0)
            for s0 in range(0, L, split):
                chunks = [x[c:c + 16].max() for c in range(s0, min(L, s0 + split), 16)]
                for st in strides:
                    for w in range(st):
                        mine = chunks[w::st]
                        if not mine:
                            continue
                        ref = mine[0]
                        for m in mine[1:]:
                            if m > ref + 8.0:
                                total += 1
                                ref = m
    return total


KV_TYPE = {"q8": "KVATTN_KV_Q8_0", "q8q4": "KVATTN_KV_Q8_0_Q4_0", "q4": "KVATTN_KV_Q4_0"}


def gpu_decode(K, kind, q, cache, lens, split, scale, n_cells, max_len, plan=None):
    import torch
    kw = dict(split=split, scale=scale, n_cells=n_cells, max_len=max_len,
              cell_plan=None if plan is None else dev(plan))
    if kind == "f16":
        out, lse = K.decode(dev(q), dev(cache[0]), dev(cache[1]), dev(np.asarray(lens, np.int32)), **kw)
    else:
        kq, kd, vq, vd = cache
        out, lse = K.decode(dev(q), dev(kq), dev(vq), dev(np.asarray(lens, np.int32)), k_scales=dev(kd),
                            v_scales=dev(vd), kv_type=getattr(K, KV_TYPE[kind]), **kw)
    torch.cuda.synchronize()
    return out, lse


def oracle_cache(kind, cache):
    # the oracle takes (k, v) for f16 and (k, k_scales, v, v_scales) for the quantised types
    return cache


# ---------------------------------------------------------------------------------------------
# single-query decode: f16, Q8_0, Q8_0 + Q4_0, Q4_0 at head_dim 128 and 256
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("kind,D", [("f16", 128), ("f16", 256), ("q8", 128), ("q8", 256), ("q8q4", 128),
                                    ("q8q4", 256), ("q4", 128), ("q4", 256)])
def test_rescale_single_query(kvattn, kind, D, case):
    rng = np.random.default_rng([31, D, CASES.index(case), list(KIND_ORACLE).index(kind)])
    S, N, Hk, G = 2, 2048, 2, 6 if D == 128 else 4
    H = Hk * G
    split = 512 if kind != "f16" else 256
    lens = [N, 1459]
    kc0, kc1, a_nat, b_nat, qmul, scale = controls(case, lens, N, split)
    q = make_q(rng, (S, H), D, a_nat, b_nat, qmul, scale)
    cache = make_cache(rng, kind, (S, N, Hk), D, kc0, kc1)
    if case in MOVING:
        assert moves(q, kind, cache, lens, split, scale) > 0
    out, lse = gpu_decode(kvattn, kind, q, cache, lens, split, scale, N, N)
    wo, wl = KIND_ORACLE[kind](q, *cache, lens, scale=scale)
    assert_close(out, lse, wo, wl)


@pytest.mark.parametrize("case", ["ramp_split", "dominant_mid", "q_x16", "offset_m200"])
@pytest.mark.parametrize("kind,D", [("f16", 128), ("f16", 256), ("q8", 128), ("q8q4", 256), ("q4", 128)])
def test_rescale_scattered_plan(kvattn, kind, D, case):
    """A plan in random physical order with -1 holes: most tiles are not one run and arrive as
    per-row copies into the plain layout.  The controls follow the logical position."""
    rng = np.random.default_rng([32, D, CASES.index(case), list(KIND_ORACLE).index(kind)])
    N, Hk, G, split = 1800, 2, 4, 256
    H = Hk * G
    L = N
    plan = rng.permutation(N).astype(np.int32)[None]
    plan[0, rng.random(N) < 0.1] = -1
    kc0l, kc1l, a_nat, b_nat, qmul, scale = controls(case, [L], L, split)
    kc0 = np.zeros(N)
    kc1 = np.zeros(N)
    ok = plan[0] >= 0
    kc0[plan[0, ok]] = kc0l[0, ok]
    kc1[plan[0, ok]] = kc1l[0, ok]
    q = make_q(rng, (1, H), D, a_nat, b_nat, qmul, scale)
    cache = make_cache(rng, kind, (N, Hk), D, kc0, kc1)
    out, lse = gpu_decode(kvattn, kind, q, cache, [L], split, scale, N, L, plan=plan)
    wo, wl = KIND_ORACLE[kind](q, *cache, [L], plan=plan, scale=scale)
    assert_close(out, lse, wo, wl)


# ---------------------------------------------------------------------------------------------
# multi-query decode: every row layout (8 rows on the single-query kernels, 16 rows, 32 rows,
# row groups) of every cache type
# ---------------------------------------------------------------------------------------------

MQ_CASES = ["ramp_split", "ramp_global", "dominant_last", "dominant_mid", "q_x16", "scale_1", "offset_p200",
            "offset_m200"]
# (n_q, G): 8 rows per KV head, 16, 32 and 48 (two or more row groups)
MQ_ROWS = [(2, 4), (4, 4), (8, 4), (8, 6)]


@pytest.mark.parametrize("case", MQ_CASES)
@pytest.mark.parametrize("n_q,G", MQ_ROWS)
@pytest.mark.parametrize("kind,D", [("f16", 128), ("f16_mma", 128), ("f16", 256), ("q8", 128), ("q8", 256),
                                    ("q8q4", 128), ("q4", 256)])
def test_rescale_multi_query(kvattn, monkeypatch, kind, D, n_q, G, case):
    """f16 head_dim 128 with more than 16 rows runs on the tcgen05 kernel; f16_mma is the
    same case on the mma.sync layouts (KVATTN_TC=0)."""
    import torch
    if kind == "f16_mma":
        monkeypatch.setenv("KVATTN_TC", "0")
        kind = "f16"
    rng = np.random.default_rng([33, D, n_q, G, MQ_CASES.index(case), list(KIND_ORACLE).index(kind)])
    S, N, Hk = 2, 1100, 2
    H = Hk * G
    split = 256
    lens = [N, 700]
    kc0, kc1, a_nat, b_nat, qmul, scale = controls(case, lens, N, split)
    q = make_q(rng, (S, n_q, H), D, a_nat, b_nat, qmul, scale)
    cache = make_cache(rng, kind, (S, N, Hk), D, kc0, kc1)
    if case in MOVING:
        assert moves(q, kind, cache, lens, split, scale, n_q=n_q) > 0
    kw = dict(split=split, scale=scale, n_cells=N, max_len=N)
    if kind == "f16":
        out, lse = kvattn.decode_multi(dev(q), dev(cache[0]), dev(cache[1]), dev(np.asarray(lens, np.int32)), **kw)
    else:
        kq, kd, vq, vd = cache
        out, lse = kvattn.decode_multi(dev(q), dev(kq), dev(vq), dev(np.asarray(lens, np.int32)),
                                       k_scales=dev(kd), v_scales=dev(vd), **kw)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_multi(KIND_ORACLE[kind], q, lens, *cache, scale=scale)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert np.array_equal(np.isneginf(l), np.isneginf(wl))
    fin = np.isfinite(wl)
    assert np.max(np.abs(l[fin] - wl[fin]), initial=0.0) <= TOL_LSE
    assert np.max(np.abs(o - wo)) <= TOL_O
    assert np.sqrt(np.mean((o.astype(np.float64) - wo) ** 2)) <= TOL_RMSE_O


# ---------------------------------------------------------------------------------------------
# window + host tail (staged tiles and the tail read in place), and the merge alone
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("mode", ["staged", "direct"])
def test_rescale_window_tail(kvattn, mode, case):
    import torch
    rng = np.random.default_rng([34, CASES.index(case), mode == "direct"])
    N, n_win, H, Hk, D = 5000, 1000, 40, 8, 128
    split, tail_split = 128, 64
    n_tail = N - n_win
    # one sequence; the staircase period follows the tail's split so every tail unit climbs
    kc0, kc1, a_nat, b_nat, qmul, scale = controls(case, [N], N, tail_split)
    q = make_q(rng, (1, H), D, a_nat, b_nat, qmul, scale)
    k, v = make_cache(rng, "f16", (N, Hk), D, kc0[0], kc1[0])
    k_tail = torch.from_numpy(k[:n_tail]).pin_memory()
    v_tail = torch.from_numpy(v[:n_tail]).pin_memory()
    if mode == "staged":
        wt = kvattn.WindowTail()
        out, lse = wt(dev(q[0]), dev(k[n_tail:]), dev(v[n_tail:]), k_tail, v_tail, split=split, tile_cells=512,
                      tail_split=tail_split, scale=scale, copy_stream=torch.cuda.Stream())
        kvattn.kvattn_tail_wait(wt.ctx, 30000)
    else:
        out, lse = kvattn.window_tail_direct(dev(q[0]), dev(k[n_tail:]), dev(v[n_tail:]), k_tail, v_tail,
                                             split=split, tail_split=tail_split, scale=scale)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_f16(q, k, v, [N], scale=scale)
    assert_close(out.view(1, H, D), lse.view(1, H), wo, wl)
    if mode == "staged":
        wt.close()


@pytest.mark.parametrize("spread", [1.0, 30.0, 120.0])
@pytest.mark.parametrize("centre", [0.0, 200.0, -200.0])
def test_merge_extreme_lses(kvattn, centre, spread):
    """kvattn_merge over parts whose LSEs sit around +-200 and spread by up to 120 natural
    units, a third of them empty (-inf, NaN O that must never be read)."""
    import torch
    rng = np.random.default_rng([35, int(centre) + 1000, int(spread)])
    P, R, D = 37, 24, 128
    parts = rng.standard_normal((P, R, D))
    lses = centre + spread * rng.uniform(-1.0, 1.0, (P, R))
    empty = rng.random((P, R)) < 0.33
    empty[:, 0] = True                        # row 0: every part empty
    empty[0, 1:] = False                      # the others keep at least one
    lses[empty] = -np.inf
    parts[empty] = np.nan
    out, lse = kvattn.merge(dev(parts.astype(np.float32)), dev(lses.astype(np.float32)))
    torch.cuda.synchronize()
    # the oracle merges the same fp32 values in fp64
    wo, wl = oracle.merge(parts.astype(np.float32), lses.astype(np.float32))
    assert_close(out, lse, wo, wl)


@pytest.mark.parametrize("case", ["ramp_split", "ramp_global", "dominant_last", "dominant_mid", "q_x16", "scale_1",
                                  "offset_p200", "offset_m200"])
@pytest.mark.parametrize("kind,G", [("q8", 4), ("q8q4", 3), ("q4", 2), ("q8", 1)])
def test_rescale_head_pairs(kvattn, kind, G, case):
    """Quantised head_dim-128 caches with at most four query heads per KV head and an even
    number of KV heads run as KV-head pairs on the head_dim-256 kernels (each query row
    keeps its own head's half of the 256 dimensions)."""
    rng = np.random.default_rng([36, G, CASES.index(case), list(KIND_ORACLE).index(kind)])
    S, N, Hk, D, split = 2, 2048, 4, 128, 512
    H = Hk * G
    lens = [N, 1459]
    kc0, kc1, a_nat, b_nat, qmul, scale = controls(case, lens, N, split)
    q = make_q(rng, (S, H), D, a_nat, b_nat, qmul, scale)
    cache = make_cache(rng, kind, (S, N, Hk), D, kc0, kc1)
    out, lse = gpu_decode(kvattn, kind, q, cache, lens, split, scale, N, N)
    wo, wl = KIND_ORACLE[kind](q, *cache, lens, scale=scale)
    assert_close(out, lse, wo, wl)
