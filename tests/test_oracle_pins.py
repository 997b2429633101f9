"""Pins for the fp64 CPU oracle: closed forms, identities, library routines, brute force.

Each check ties the oracle to something other than itself, so that a plausible slip
in it (a dropped term, a wrong sign or index, a transposed operand, log2 for ln, a
wrong GQA head mapping, a misplaced Q8_0 scale) fails at least one test here.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import brute


def rand_f16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def test_f16_conversion_exhaustive():
    """The oracle's binary16 decoder against numpy on all 65536 bit patterns."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("with_plan", [False, True])
def test_brute_force_tiny(with_plan):
    """Against the pure-Python fsum brute force, ragged lengths, GQA-2."""
    rng = np.random.default_rng(7)
    S, H, Hk, D = 2, 4, 2, 8
    q = rand_f16(rng, (S, H, D))
    if with_plan:
        Np = 16
        k = rand_f16(rng, (Np, Hk, D))
        v = rand_f16(rng, (Np, Hk, D))
        plan = np.array([[3, -1, 9, 0, 15, -1, 4], [12, 2, -1, -1, 7, 8, 1]], dtype=np.int32)
        lens = [7, 5]
        out, lse = oracle.decode_f16(q, k, v, lens, plan=plan)
        bo, bl = brute.decode(q.tolist(), k.tolist(), v.tolist(), lens, plan=plan.tolist())
    else:
        N = 6
        k = rand_f16(rng, (S, N, Hk, D))
        v = rand_f16(rng, (S, N, Hk, D))
        lens = [6, 3]
        out, lse = oracle.decode_f16(q, k, v, lens)
        bo, bl = brute.decode(q.tolist(), k.tolist(), v.tolist(), lens)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-13)


def test_library_softmax_and_logsumexp():
    """x = scale * K q with numpy matmul, then scipy softmax / logsumexp, per head."""
    rng = np.random.default_rng(11)
    N, H, Hk, D = 300, 8, 2, 64
    G = H // Hk
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    scale = 1 / math.sqrt(D)
    out, lse = oracle.decode_f16(q, k, v, [N])
    for h in range(H):
        kh = k[:, h // G, :].astype(np.float64)
        vh = v[:, h // G, :].astype(np.float64)
        x = scale * (kh @ q[0, h].astype(np.float64))
        np.testing.assert_allclose(out[0, h], scipy.special.softmax(x) @ vh, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], scipy.special.logsumexp(x), rtol=0, atol=1e-12)


def test_constant_v_returns_v():
    rng = np.random.default_rng(3)
    N, H, Hk, D = 257, 4, 1, 128
    q = rand_f16(rng, (1, H, D), 3.0)
    k = rand_f16(rng, (N, Hk, D), 3.0)
    row = rand_f16(rng, (D,))
    v = np.broadcast_to(row, (N, Hk, D)).copy()
    out, _ = oracle.decode_f16(q, k, v, [N])
    np.testing.assert_allclose(out[0], np.broadcast_to(row.astype(np.float64), (H, D)), rtol=0,
                               atol=1e-12)


def test_single_cell():
    rng = np.random.default_rng(4)
    H, Hk, D = 6, 3, 32
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (1, Hk, D))
    v = rand_f16(rng, (1, Hk, D))
    scale = 0.37
    out, lse = oracle.decode_f16(q, k, v, [1], scale=scale)
    for h in range(H):
        g = h // 2
        np.testing.assert_array_equal(out[0, h], v[0, g].astype(np.float64))
        x = scale * float(np.dot(q[0, h].astype(np.float64), k[0, g].astype(np.float64)))
        assert abs(lse[0, h] - x) < 1e-12


def test_zero_query_gives_mean_and_ln_n():
    """All scores 0: O is the mean of the valid V rows and LSE = ln(n) (natural log)."""
    rng = np.random.default_rng(5)
    N, H, Hk, D = 100, 2, 2, 16
    q = np.zeros((1, H, D), np.float16)
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    out, lse = oracle.decode_f16(q, k, v, [N])
    for h in range(H):
        np.testing.assert_allclose(out[0, h], v[:, h].astype(np.float64).mean(0), atol=1e-13)
        assert abs(lse[0, h] - math.log(N)) < 1e-13
    # a zero scale is the same special case
    q2 = rand_f16(rng, (1, H, D))
    out2, lse2 = oracle.decode_f16(q2, k, v, [N], scale=0.0)
    np.testing.assert_allclose(out2, out, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, atol=1e-13)


def test_two_cells_sigmoid_closed_form():
    rng = np.random.default_rng(6)
    H, Hk, D = 2, 1, 8
    q = rand_f16(rng, (1, H, D), 2.0)
    k = rand_f16(rng, (2, Hk, D), 2.0)
    v = rand_f16(rng, (2, Hk, D))
    scale = 0.5
    out, lse = oracle.decode_f16(q, k, v, [2], scale=scale)
    for h in range(H):
        x1 = scale * float(q[0, h].astype(np.float64) @ k[0, 0].astype(np.float64))
        x2 = scale * float(q[0, h].astype(np.float64) @ k[1, 0].astype(np.float64))
        sig = scipy.special.expit(x1 - x2)
        want = sig * v[0, 0].astype(np.float64) + (1 - sig) * v[1, 0].astype(np.float64)
        np.testing.assert_allclose(out[0, h], want, atol=1e-13)
        assert abs(lse[0, h] - np.logaddexp(x1, x2)) < 1e-13


def test_empty_sequence():
    rng = np.random.default_rng(8)
    q = rand_f16(rng, (2, 4, 8))
    k = rand_f16(rng, (2, 5, 2, 8))
    v = rand_f16(rng, (2, 5, 2, 8))
    out, lse = oracle.decode_f16(q, k, v, [0, 5])
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


@pytest.mark.parametrize("split", [1, 3, 64, 1000])
def test_split_then_merge_equals_unsplit(split):
    """Partials over disjoint cell ranges, LSE-merged, equal the unsplit definition."""
    rng = np.random.default_rng(9)
    N, H, Hk, D = 1000, 4, 2, 32
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    full_o, full_l = oracle.decode_f16(q, k, v, [N])
    parts, lses = [], []
    for lo in range(0, N, split):
        hi = min(N, lo + split)
        o, l = oracle.decode_f16(q, k[lo:hi], v[lo:hi], [hi - lo])
        parts.append(o[0])
        lses.append(l[0])
    mo, ml = oracle.merge(np.stack(parts), np.stack(lses))
    np.testing.assert_allclose(mo, full_o[0], atol=1e-12)
    np.testing.assert_allclose(ml, full_l[0], atol=1e-12)


def test_window_plus_tail_equals_resident():
    rng = np.random.default_rng(10)
    N, n_win, H, Hk, D = 3000, 512, 5, 1, 16
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    tail_o, tail_l = oracle.decode_f16(q, k[:N - n_win], v[:N - n_win], [N - n_win])
    win_o, win_l = oracle.decode_f16(q, k[N - n_win:], v[N - n_win:], [n_win])
    mo, ml = oracle.merge(np.stack([win_o[0], tail_o[0]]), np.stack([win_l[0], tail_l[0]]))
    full_o, full_l = oracle.decode_f16(q, k, v, [N])
    np.testing.assert_allclose(mo, full_o[0], atol=1e-12)
    np.testing.assert_allclose(ml, full_l[0], atol=1e-12)


def test_holes_and_nan_cells_contribute_nothing():
    """A plan with -1 holes over NaN-filled cells equals the same cells copied compactly."""
    rng = np.random.default_rng(12)
    Np, H, Hk, D = 512, 6, 1, 16
    k = rand_f16(rng, (Np, Hk, D))
    v = rand_f16(rng, (Np, Hk, D))
    q = rand_f16(rng, (1, H, D))
    row = np.arange(128, 384, dtype=np.int32)
    holes = rng.random(row.shape[0]) < 0.3
    row[holes] = -1
    unused = np.setdiff1d(np.arange(Np), row[row >= 0])
    k[unused] = np.nan
    v[unused] = np.nan
    out, lse = oracle.decode_f16(q, k, v, [row.shape[0]], plan=row[None, :])
    valid = row[row >= 0]
    co, cl = oracle.decode_f16(q, k[valid], v[valid], [valid.shape[0]])
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out, co, atol=1e-13)
    np.testing.assert_allclose(lse, cl, atol=1e-13)


def test_permutation_invariance():
    rng = np.random.default_rng(13)
    Np, H, Hk, D = 200, 4, 2, 16
    k = rand_f16(rng, (Np, Hk, D))
    v = rand_f16(rng, (Np, Hk, D))
    q = rand_f16(rng, (1, H, D))
    a = np.arange(Np, dtype=np.int32)[None]
    b = rng.permutation(Np).astype(np.int32)[None]
    oa, la = oracle.decode_f16(q, k, v, [Np], plan=a)
    ob, lb = oracle.decode_f16(q, k, v, [Np], plan=b)
    np.testing.assert_allclose(oa, ob, atol=1e-13)
    np.testing.assert_allclose(la, lb, atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv():
    """Head h reads KV head floor(h / G): repeating each KV head G times gives MHA."""
    rng = np.random.default_rng(14)
    N, H, Hk, D = 77, 12, 3, 32
    G = H // Hk
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    go, gl = oracle.decode_f16(q, k, v, [N])
    mo, ml = oracle.decode_f16(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), [N])
    np.testing.assert_array_equal(go, mo)
    np.testing.assert_array_equal(gl, ml)


@pytest.mark.parametrize("D", [128, 256])
def test_q8_0_front_end_equals_explicit_dequant(D):
    rng = np.random.default_rng(15)
    N, H, Hk = 90, 4, 2
    q = rand_f16(rng, (1, H, D))
    kq = rng.integers(-127, 128, (N, Hk, D), dtype=np.int8)
    vq = rng.integers(-127, 128, (N, Hk, D), dtype=np.int8)
    kd = rng.uniform(0.001, 0.02, (N, Hk, D // 32)).astype(np.float16)
    vd = rng.uniform(0.001, 0.02, (N, Hk, D // 32)).astype(np.float16)
    o8, l8 = oracle.decode_q8_0(q, kq, kd, vq, vd, [N])
    of, lf = oracle.decode_f64(q.astype(np.float64), oracle.dequant_q8_0(kq, kd),
                               oracle.dequant_q8_0(vq, vd), [N])
    np.testing.assert_array_equal(o8, of)
    np.testing.assert_array_equal(l8, lf)
    # the scale of block b multiplies head_dim elements 32b .. 32b+31 only
    kd2 = kd.copy()
    kd2[:, :, 1] *= 2
    o9, _ = oracle.decode_q8_0(q, kq, kd2, vq, vd, [N])
    assert not np.allclose(o9, o8)


def test_q4_0_block_worked_by_hand():
    """q4_0 as the llama.cpp block defines it: 32 elements, one f16 scale, byte j holding
    element j in its low nibble and element j + 16 in its high nibble, value d * (n - 8).
    Bytes j | (15 - j) << 4 with d = 0.5 give elements 0..15 = 0.5 (j - 8) and elements
    16..31 = 0.5 (7 - j), written out below.  A single cell reduces attention to O = V, so
    the C oracle's Q4_0 front end is pinned to the same literal row."""
    expected = [-4.0, -3.5, -3.0, -2.5, -2.0, -1.5, -1.0, -0.5, 0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 3.0, 3.5,
                3.5, 3.0, 2.5, 2.0, 1.5, 1.0, 0.5, 0.0, -0.5, -1.0, -1.5, -2.0, -2.5, -3.0, -3.5, -4.0]
    row = np.array([j | ((15 - j) << 4) for j in range(16)], dtype=np.uint8)
    d = np.array([0.5], dtype=np.float16)
    np.testing.assert_array_equal(oracle.dequant_q4_0(row, d), expected)
    # D = 128: four blocks with scales 0.5, 1, 2, -0.25 over the same bytes
    D = 128
    v4 = np.tile(row, 4).reshape(1, 1, D // 2)
    vd = np.array([[[0.5, 1.0, 2.0, -0.25]]], dtype=np.float16)
    kq = np.ones((1, 1, D), dtype=np.int8)
    kd = np.full((1, 1, D // 32), 0.01, dtype=np.float16)
    q = np.ones((1, 1, D), dtype=np.float16)
    out, lse = oracle.decode_q8_0_q4_0(q, kq, kd, v4, vd, [1])
    want = np.concatenate([np.array(expected) * f for f in (1.0, 2.0, 4.0, -0.5)])
    np.testing.assert_array_equal(out[0, 0], want)
    # x = scale * sum_d 1 * 0.01 (f16) = the single cell's logit = its LSE
    assert lse[0, 0] == pytest.approx(float(np.float16(0.01)) * D / math.sqrt(D), rel=1e-15)
    o4, _ = oracle.decode_q4_0(q, np.tile(row, 4).reshape(1, 1, D // 2), vd, v4, vd, [1])
    np.testing.assert_array_equal(o4[0, 0], want)


@pytest.mark.parametrize("D", [128, 256])
def test_q4_0_front_ends_equal_explicit_dequant(D):
    rng = np.random.default_rng(16)
    N, H, Hk = 90, 6, 2
    q = rand_f16(rng, (1, H, D))
    kq = rng.integers(-127, 128, (N, Hk, D), dtype=np.int8)
    k4 = rng.integers(0, 256, (N, Hk, D // 2), dtype=np.uint8)
    v4 = rng.integers(0, 256, (N, Hk, D // 2), dtype=np.uint8)
    kd = rng.uniform(0.001, 0.02, (N, Hk, D // 32)).astype(np.float16)
    vd = rng.uniform(0.001, 0.02, (N, Hk, D // 32)).astype(np.float16)
    om, lm = oracle.decode_q8_0_q4_0(q, kq, kd, v4, vd, [N])
    of, lf = oracle.decode_f64(q.astype(np.float64), oracle.dequant_q8_0(kq, kd), oracle.dequant_q4_0(v4, vd), [N])
    np.testing.assert_array_equal(om, of)
    np.testing.assert_array_equal(lm, lf)
    o4, l4 = oracle.decode_q4_0(q, k4, kd * 8, v4, vd, [N])
    of, lf = oracle.decode_f64(q.astype(np.float64), oracle.dequant_q4_0(k4, kd * 8), oracle.dequant_q4_0(v4, vd),
                               [N])
    np.testing.assert_array_equal(o4, of)
    np.testing.assert_array_equal(l4, lf)
    # nibble value 8 is zero: O = 0 and the LSE is that of the keys alone
    eights = np.full_like(v4, 0x88)
    oz, lz = oracle.decode_q8_0_q4_0(q, kq, kd, eights, vd, [N])
    assert np.all(oz == 0.0)
    np.testing.assert_array_equal(lz, lm)
    # a block's scale reaches its own 32 elements only
    vd2 = vd.copy()
    vd2[:, :, 1] *= 2
    o9, _ = oracle.decode_q8_0_q4_0(q, kq, kd, v4, vd2, [N])
    changed = np.any(o9 != om, axis=(0, 1))
    assert changed[32:64].all() and not changed[:32].any() and not changed[64:].any()


def test_merge_special_cases():
    rng = np.random.default_rng(16)
    R, D = 3, 8
    o1 = rng.standard_normal((1, R, D))
    l1 = rng.standard_normal((1, R))
    mo, ml = oracle.merge(o1, l1)
    np.testing.assert_array_equal(mo, o1[0])
    np.testing.assert_array_equal(ml, l1[0])
    # an -inf part is ignored even when its O is NaN
    o2 = np.concatenate([o1, np.full((1, R, D), np.nan)])
    l2 = np.concatenate([l1, np.full((1, R), -np.inf)])
    mo, ml = oracle.merge(o2, l2)
    np.testing.assert_array_equal(mo, o1[0])
    np.testing.assert_array_equal(ml, l1[0])
    # two parts of equal LSE: the average, LSE + ln 2
    o3 = rng.standard_normal((2, R, D))
    l3 = np.stack([l1[0], l1[0]])
    mo, ml = oracle.merge(o3, l3)
    np.testing.assert_allclose(mo, o3.mean(0), atol=1e-15)
    np.testing.assert_allclose(ml, l1[0] + math.log(2), atol=1e-15)
    # every part empty
    mo, ml = oracle.merge(np.zeros((2, R, D)), np.full((2, R), -np.inf))
    assert np.all(mo == 0) and np.all(np.isneginf(ml))


def test_rejects_plan_entries_outside_the_cache():
    rng = np.random.default_rng(17)
    k = rand_f16(rng, (10, 1, 8))
    q = rand_f16(rng, (1, 1, 8))
    with pytest.raises(ValueError):
        oracle.decode_f16(q, k, k, [2], plan=np.array([[3, -5]], np.int32))
    with pytest.raises(ValueError):
        oracle.decode_f16(q, k, k, [2], plan=np.array([[3, 10]], np.int32))


# ------------------------- multi-query decode (causal, n_q tokens) -------------------------

def _mq_case(rng, S, n_q, N, H, Hk, D):
    q = rng.standard_normal((S, n_q, H, D)).astype(np.float16)
    k = rng.standard_normal((S, N, Hk, D)).astype(np.float16)
    v = rng.standard_normal((S, N, Hk, D)).astype(np.float16)
    return q, k, v


def test_multi_query_matches_brute_force_contiguous():
    from oracle import brute
    rng = np.random.default_rng(71)
    q, k, v = _mq_case(rng, 2, 3, 6, 4, 2, 8)
    lens = [6, 2]                       # sequence 1: token 0 sees nothing
    wo, wl = oracle.decode_multi(oracle.decode_f16, q, lens, k, v)
    bo, bl = brute.decode_multi(q.tolist(), k.tolist(), v.tolist(), lens, n_head_kv=2)
    assert np.allclose(wo, np.array(bo), atol=1e-12, rtol=0)
    assert np.array_equal(np.isneginf(wl), np.isneginf(np.array(bl)))
    fin = np.isfinite(wl)
    assert np.allclose(wl[fin], np.array(bl)[fin], atol=1e-12, rtol=0)
    assert np.all(np.isneginf(wl[1, 0])) and np.all(wo[1, 0] == 0)


def test_multi_query_matches_brute_force_plan_with_holes():
    from oracle import brute
    rng = np.random.default_rng(72)
    Hk, D, H, n_q = 2, 8, 4, 2
    n_phys = 20
    k = rng.standard_normal((n_phys, Hk, D)).astype(np.float16)
    v = rng.standard_normal((n_phys, Hk, D)).astype(np.float16)
    q = rng.standard_normal((2, n_q, H, D)).astype(np.float16)
    plan = np.array([[3, -1, 7, 8, 11, -1, 2], [5, 6, -1, 0, -1, -1, -1]], np.int32)
    lens = [7, 5]                       # sequence 0's last token at a -1 entry
    wo, wl = oracle.decode_multi(oracle.decode_f16, q, lens, k, v, plan=plan)
    bo, bl = brute.decode_multi(q.tolist(), k.tolist(), v.tolist(), lens, plan=plan.tolist(), n_head_kv=2)
    assert np.allclose(wo, np.array(bo), atol=1e-12, rtol=0)
    assert np.allclose(wl, np.array(bl), atol=1e-12, rtol=0)


def test_multi_query_reductions():
    rng = np.random.default_rng(73)
    q, k, v = _mq_case(rng, 3, 4, 50, 8, 2, 16)
    lens = [50, 3, 0]
    wo, wl = oracle.decode_multi(oracle.decode_f16, q, lens, k, v)
    # the last token sees the whole sequence: single-query decode of the full length
    so, sl = oracle.decode_f16(q[:, -1], k, v, lens)
    assert np.array_equal(wo[:, -1], so) and np.array_equal(wl[:, -1], sl)
    # one token is single-query decode
    o1, l1 = oracle.decode_multi(oracle.decode_f16, q[:, :1], lens, k, v)
    so1, sl1 = oracle.decode_f16(q[:, 0], k, v, lens)
    assert np.array_equal(o1[:, 0], so1) and np.array_equal(l1[:, 0], sl1)
    # a sequence shorter than n_q: tokens 0 (and only 0) of [3] see nothing; [0] none do
    assert np.all(np.isneginf(wl[1, 0])) and np.all(np.isfinite(wl[1, 1:]))
    assert np.all(np.isneginf(wl[2])) and np.all(wo[2] == 0)
    # V constant over the cells of each (sequence, KV head): every token gets that row
    vc = np.repeat(v[:, :1], v.shape[1], axis=1)
    co, _ = oracle.decode_multi(oracle.decode_f16, q, [50, 50, 50], k, vc)
    for s_ in range(3):
        for h in range(8):
            assert np.allclose(co[s_, :, h], vc[s_, 0, h // 4].astype(np.float64)[None], atol=1e-12, rtol=0)
