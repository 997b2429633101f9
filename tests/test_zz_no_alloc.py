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
