"""kvattn_decode_noalloc: decode attention for callers that cannot allocate device memory.

Code that runs inside a fixed memory pool's budget, plugins that are handed only their
input and output buffers, or paths that must not wait on the driver's allocator cannot
call cudaMalloc to make a workspace.  kvattn_decode_noalloc takes the same inputs and
outputs as kvattn_decode and keeps its scratch in a fixed-size array inside the library.
These tests call it through the C ABI twice in a row (the second call reuses the array
the first one left behind) and compare each result with kvattn_decode's, within the
tolerances the other tests use.  This file is named so that pytest collects it last.
"""
import math

import numpy as np
import pytest

from tests.gpu_util import TOL_LSE, TOL_O

A = 0x7f0000000000  # fake, aligned addresses: the size check fails before any use


def test_oversized_call_is_refused_before_any_launch(kvattn):
    # 4 sequences x 65536 cells x 48 heads need ~50 MB of scratch, more than the array holds
    need = kvattn.kvattn_decode_workspace_bytes(4, 48, 128, 65536, 128)
    assert need > kvattn.KVATTN_NOALLOC_SCRATCH_BYTES
    rc = kvattn.lib.kvattn_decode_noalloc(A, A, A, None, None, 0, 65536, None, 0, A, 4, 65536, 48, 8, 128,
                                          128, 0.088, A, A, None)
    assert rc == kvattn.KVATTN_ERR_WORKSPACE


def test_argument_errors_come_before_the_size_refusal(kvattn):
    # the same oversized shape, with one argument wrong: the argument's own error, still
    # before the array is looked up or anything is enqueued (no GPU is needed to see it)
    f = kvattn.lib.kvattn_decode_noalloc
    # a split that is not a multiple of the 32-cell tile
    assert f(A, A, A, None, None, 0, 65536, None, 0, A, 4, 65536, 48, 8, 128, 48, 0.088, A, A,
             None) == kvattn.KVATTN_ERR_UNSUPPORTED
    # heads that do not divide into KV heads
    assert f(A, A, A, None, None, 0, 65536, None, 0, A, 4, 65536, 47, 8, 128, 128, 0.088, A, A,
             None) == kvattn.KVATTN_ERR_INVALID_ARG
    # an unknown cache type, a quantised type without scales, a missing output
    assert f(A, A, A, None, None, 9, 65536, None, 0, A, 4, 65536, 48, 8, 128, 128, 0.088, A, A,
             None) == kvattn.KVATTN_ERR_INVALID_ARG
    assert f(A, A, A, None, None, 1, 65536, None, 0, A, 4, 65536, 48, 8, 128, 128, 0.088, A, A,
             None) == kvattn.KVATTN_ERR_INVALID_ARG
    assert f(A, A, A, None, None, 0, 65536, None, 0, A, 4, 65536, 48, 8, 128, 128, 0.088, None, A,
             None) == kvattn.KVATTN_ERR_INVALID_ARG


def _case(rng, S, N, H, Hk, D):
    import torch
    q = torch.from_numpy(rng.standard_normal((S, H, D), dtype=np.float32).astype(np.float16)).cuda()
    k = torch.from_numpy(rng.standard_normal((S, N, Hk, D), dtype=np.float32).astype(np.float16)).cuda()
    v = torch.from_numpy(rng.standard_normal((S, N, Hk, D), dtype=np.float32).astype(np.float16)).cuda()
    lens = torch.tensor(rng.integers(N // 2, N + 1, size=S), dtype=torch.int32).cuda()
    return q, k, v, lens


@pytest.mark.gpu
def test_no_alloc_matches_decode_on_two_calls_in_a_row(kvattn):
    import torch
    rng = np.random.default_rng(2026)
    cases = [(1, 16384, 32, 8, 128, 256),   # the Qwen3-8B-shaped layer
             (3, 5000, 24, 4, 128, 128)]    # several sequences, ragged lengths
    for S, N, H, Hk, D, split in cases:
        q, k, v, lens = _case(rng, S, N, H, Hk, D)
        scale = 1.0 / math.sqrt(D)
        out_a = torch.full((S, H, D), float("nan"), device="cuda")
        lse_a = torch.full((S, H), float("nan"), device="cuda")
        kvattn.kvattn_decode_noalloc(q, k, v, None, None, kvattn.KVATTN_KV_F16, N, None, 0, lens, S, N, H, Hk,
                                     D, split, scale, out_a, lse_a)
        out_b, lse_b = kvattn.decode(q, k, v, lens, split=split, n_cells=N, max_len=N)
        torch.cuda.synchronize()
        oa, ob = out_a.cpu().numpy(), out_b.cpu().numpy()
        la, lb = lse_a.cpu().numpy(), lse_b.cpu().numpy()
        assert np.all(np.isfinite(oa)) and np.all(np.isfinite(la))
        assert np.max(np.abs(oa - ob)) <= TOL_O
        assert np.max(np.abs(la - lb)) <= TOL_LSE


def _plan(kvattn, rng, pool, hole_p):
    """A compact plan over `pool` 128-cell records: three sequences owning 5, 1 and 8 records,
    each cell kept with probability 1 - hole_p (the rest are -1 holes)."""
    n_cells = pool * 128
    perm = rng.permutation(pool)
    encoded = []
    for recs in (perm[:5], perm[5:6], perm[6:14]):
        cells = (recs[:, None] * 128 + np.arange(128)[None]).reshape(-1)
        encoded.append(cells[rng.random(cells.size) >= hole_p].astype(np.int64))
    return kvattn.build_cell_plan(encoded, n_cells), n_cells


@pytest.mark.gpu
def test_no_alloc_plans_after_a_larger_call(kvattn):
    """A large call leaves the array full of its descriptors and partials; smaller calls
    through compact plans with -1 holes follow -- f16 (descriptors built inside the decode)
    and Q8_0 (descriptors from their own launch) -- so any descriptor or partial a call
    failed to rewrite would be read stale.  Each result is compared with kvattn_decode's and
    with the oracle's."""
    import torch
    import oracle
    from tests.gpu_util import assert_close
    rng = np.random.default_rng(2027)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()

    # the large call first: 4 sequences x 8192 cells, 32/8 heads, split 128 (about 4 MB of
    # partials), its plan-free descriptors region then holding whatever it left
    q, k, v, lens = _case(rng, 4, 8192, 32, 8, 128)
    big_o = torch.empty((4, 32, 128), device="cuda")
    big_l = torch.empty((4, 32), device="cuda")
    kvattn.kvattn_decode_noalloc(q, k, v, None, None, kvattn.KVATTN_KV_F16, 8192, None, 0, lens, 4, 8192, 32, 8,
                                 128, 128, 1.0 / math.sqrt(128), big_o, big_l)

    for trial, kind in enumerate(["f16", "q8_0", "f16", "q8_0"]):
        (plan, plens), n_cells = _plan(kvattn, rng, 24, 0.2 + 0.1 * trial)
        S, stride = plan.shape
        D, Hk, G = (128, 2, 6) if kind == "f16" else (256, 2, 4)
        H = Hk * G
        qh = rng.standard_normal((S, H, D), dtype=np.float32).astype(np.float16)
        if kind == "f16":
            kc = rng.standard_normal((n_cells, Hk, D), dtype=np.float32).astype(np.float16)
            vc = rng.standard_normal((n_cells, Hk, D), dtype=np.float32).astype(np.float16)
            cache = (kc, vc)
            args = (dev(kc), dev(vc), None, None, kvattn.KVATTN_KV_F16)
            wo, wl = oracle.decode_f16(qh, kc, vc, plens.tolist(), plan=plan)
        else:
            kq = rng.integers(-127, 128, (n_cells, Hk, D), dtype=np.int8)
            vq = rng.integers(-127, 128, (n_cells, Hk, D), dtype=np.int8)
            kd = rng.uniform(0.001, 0.02, (n_cells, Hk, D // 32)).astype(np.float16)
            vd = rng.uniform(0.001, 0.02, (n_cells, Hk, D // 32)).astype(np.float16)
            args = (dev(kq), dev(vq), dev(kd), dev(vd), kvattn.KVATTN_KV_Q8_0)
            wo, wl = oracle.decode_q8_0(qh, kq, kd, vq, vd, plens.tolist(), plan=plan)
        split = 128
        scale = 1.0 / math.sqrt(D)
        out_a = torch.full((S, H, D), float("nan"), device="cuda")
        lse_a = torch.full((S, H), float("nan"), device="cuda")
        kvattn.kvattn_decode_noalloc(dev(qh), *args, n_cells, dev(plan), stride, dev(plens), S, stride, H, Hk, D,
                                     split, scale, out_a, lse_a)
        out_b, lse_b = kvattn.decode(dev(qh), args[0], args[1], dev(plens), split=split, cell_plan=dev(plan),
                                     k_scales=args[2], v_scales=args[3], n_cells=n_cells, max_len=stride,
                                     kv_type=args[4])
        torch.cuda.synchronize()
        assert np.max(np.abs(out_a.cpu().numpy() - out_b.cpu().numpy())) <= TOL_O
        assert np.max(np.abs(lse_a.cpu().numpy() - lse_b.cpu().numpy())) <= TOL_LSE
        assert_close(out_a, lse_a, wo, wl)
