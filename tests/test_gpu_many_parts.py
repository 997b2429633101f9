"""GPU parity against the fp64 oracle when a row has many partials.

The merge folds a row's partials in rounds of 64 (head_dim 128) or 32 (head_dim 256) per
CTA; these cases take several rounds, end ragged sequences inside a round, include empty
sequences, run over a workspace holding random bytes past its status word, and repeat
calls on one workspace.
"""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu


def rand_f16(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def garbage_ws(kvattn, nbytes, seed):
    """A workspace of random bytes past the (zeroed) status word."""
    import torch
    g = torch.Generator(device="cpu").manual_seed(seed)
    host = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g)
    host[:256] = 0
    return host.cuda()


@pytest.mark.parametrize("D,H,Hk,lens,split", [
    (128, 8, 2, [9000, 6149, 0], 32),     # 282 parts: 5 rounds of 64; 193 parts (the 4th round holds one)
    (128, 32, 8, [16384], 64),            # 256 parts, 4 full rounds
    (256, 8, 4, [3000, 1000], 32),        # head_dim 256: 94 parts in rounds of 32
    (128, 12, 2, [4133, 129, 1], 32),     # GQA-6, ragged lengths of one to three rounds
])
def test_many_parts_contiguous(kvattn, D, H, Hk, lens, split):
    rng = np.random.default_rng(sum(lens) + D)
    S, N = len(lens), max(lens)
    q = rand_f16(rng, (S, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(np.array(lens, np.int32)), split=split, n_cells=N,
                             max_len=N)
    wo, wl = oracle.decode_f16(q, k, v, lens)
    assert_close(out, lse, wo, wl)
    if 0 in lens:
        s = lens.index(0)
        assert np.all(np.isneginf(lse.cpu().numpy()[s])) and np.all(out.cpu().numpy()[s] == 0)


def test_workspace_garbage_and_repeated_calls(kvattn):
    """Only the status word of a workspace needs to start at zero: a workspace holding
    random bytes past it gives the oracle's result, three times, and the same bits each
    time."""
    import torch
    rng = np.random.default_rng(31)
    S, N, H, Hk, D, split = 2, 7000, 16, 4, 128, 32
    lens = [7000, 4500]
    q = rand_f16(rng, (S, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    ws = garbage_ws(kvattn, kvattn.kvattn_decode_workspace_bytes(S, H, D, N, split), 5)
    args = (dev(q), dev(k), dev(v), dev(np.array(lens, np.int32)))
    wo, wl = oracle.decode_f16(q, k, v, lens)
    prev = None
    for _ in range(3):
        out, lse = kvattn.decode(*args, split=split, n_cells=N, max_len=N, ws=ws)
        torch.cuda.synchronize()
        assert_close(out, lse, wo, wl)
        cur = (out.cpu().numpy().copy(), lse.cpu().numpy().copy())
        if prev is not None:
            assert np.array_equal(cur[0], prev[0]) and np.array_equal(cur[1], prev[1])
        prev = cur
    assert kvattn.kvattn_workspace_status(ws) == 0


def test_many_parts_q8_0(kvattn):
    rng = np.random.default_rng(32)
    S, N, H, Hk, D, split = 1, 9000, 8, 2, 128, 32
    kq = rng.integers(-127, 128, (S, N, Hk, D), dtype=np.int8)
    vq = rng.integers(-127, 128, (S, N, Hk, D), dtype=np.int8)
    kd = rng.uniform(0.001, 0.02, (S, N, Hk, D // 32)).astype(np.float16)
    vd = rng.uniform(0.001, 0.02, (S, N, Hk, D // 32)).astype(np.float16)
    q = rand_f16(rng, (S, H, D))
    out, lse = kvattn.decode(dev(q), dev(kq), dev(vq), dev(np.array([N], np.int32)), split=split, n_cells=N,
                             max_len=N, k_scales=dev(kd), v_scales=dev(vd))
    wo, wl = oracle.decode_q8_0(q, kq, kd, vq, vd, [N])
    assert_close(out, lse, wo, wl)


def test_many_parts_multi_query(kvattn):
    import torch
    rng = np.random.default_rng(33)
    S, N, H, Hk, D, n_q, split = 2, 6000, 16, 4, 128, 4, 32
    lens = [6000, 2500]
    q = rand_f16(rng, (S, n_q, H, D))
    k = rand_f16(rng, (S, N, Hk, D))
    v = rand_f16(rng, (S, N, Hk, D))
    out, lse = kvattn.decode_multi(dev(q), dev(k), dev(v), dev(np.array(lens, np.int32)), split=split, n_cells=N,
                                   max_len=N)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_multi(oracle.decode_f16, q, lens, k, v)
    assert_close(out, lse, wo, wl)


def test_many_parts_plan_with_holes(kvattn):
    """A plan of 40 shuffled records with holes over NaN-filled unused cells, split 32."""
    rng = np.random.default_rng(34)
    Hk, H, D = 2, 8, 128
    pool = 48
    n_cells = pool * 128
    k = rand_f16(rng, (n_cells, Hk, D))
    v = rand_f16(rng, (n_cells, Hk, D))
    perm = rng.permutation(pool)
    encoded, selected = [], []
    for recs in (perm[:40], perm[40:43]):
        cells = (recs[:, None] * 128 + np.arange(128)[None]).reshape(-1)
        sel = cells[rng.random(cells.size) >= 0.1]
        encoded.append(sel.astype(np.int64)[rng.permutation(sel.size)])
        selected.append(sel)
    unused = np.setdiff1d(np.arange(n_cells), np.concatenate(selected))
    k[unused] = np.nan
    v[unused] = np.nan
    plan, lens = kvattn.build_cell_plan(encoded, n_cells)
    q = rand_f16(rng, (2, H, D))
    out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(lens), split=32, cell_plan=dev(plan), n_cells=n_cells)
    wo, wl = oracle.decode_f16(q, k, v, lens.tolist(), plan=plan)
    assert_close(out, lse, wo, wl)
