"""Window + pinned-host tail on small cases: ragged last tile, no window, no tail,
repeated calls reusing the staging slots, host-side fault injection and the bounded
host wait.  Tail tiles move by the copy kernel (mapped pinned memory) by default; one
case forces the copy-engine path."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu


def make(rng, N, n_win, H, Hk, D):
    q = rng.standard_normal((1, H, D), dtype=np.float32).astype(np.float16)
    k = rng.standard_normal((N, Hk, D), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((N, Hk, D), dtype=np.float32).astype(np.float16)
    return q, k, v


def run(kvattn, wt, q, k, v, n_win, tile, split=128, tail_split=64, ws=None, copy_stream=None):
    import torch
    n_tail = k.shape[0] - n_win
    k_tail = torch.from_numpy(k[:n_tail]).pin_memory()
    v_tail = torch.from_numpy(v[:n_tail]).pin_memory()
    k_win = dev(k[n_tail:]) if n_win else None
    v_win = dev(v[n_tail:]) if n_win else None
    if copy_stream is None:
        copy_stream = torch.cuda.Stream()
    out, lse = wt(dev(q[0]), k_win, v_win, k_tail if n_tail else None, v_tail if n_tail else None,
                  split=split, tile_cells=tile, tail_split=tail_split, ws=ws, copy_stream=copy_stream)
    kvattn.kvattn_tail_wait(wt.ctx, 30000)
    torch.cuda.synchronize()
    return out.view(1, *out.shape), lse.view(1, -1)


@pytest.mark.parametrize("N,n_win,tile,H,Hk", [
    (5000, 1000, 512, 40, 8),     # ragged last tile (4000 = 7 x 512 + 416)
    (3000, 0, 256, 16, 4),        # everything in the tail
    (777, 777, 256, 16, 4),       # everything resident
    (4096, 64, 128, 24, 4),       # many small tiles, GQA-6
])
def test_window_tail_small(kvattn, N, n_win, tile, H, Hk):
    rng = np.random.default_rng(N + n_win)
    q, k, v = make(rng, N, n_win, H, Hk, 128)
    wt = kvattn.WindowTail()
    out, lse = run(kvattn, wt, q, k, v, n_win, tile)
    wo, wl = oracle.decode_f16(q, k, v, [N])
    assert_close(out, lse, wo, wl)
    wt.close()


@pytest.mark.parametrize("copy_kernel", ["0", "1"])
def test_tile_copy_paths(kvattn, monkeypatch, copy_kernel):
    """The copy engine (cudaMemcpyAsync per tile) and the copy kernel give the same result."""
    monkeypatch.setenv("KVATTN_TAIL_COPY", copy_kernel)
    rng = np.random.default_rng(21)
    N, n_win, H, Hk = 4500, 300, 32, 8
    q, k, v = make(rng, N, n_win, H, Hk, 128)
    wt = kvattn.WindowTail()
    out, lse = run(kvattn, wt, q, k, v, n_win, 512)
    wo, wl = oracle.decode_f16(q, k, v, [N])
    assert_close(out, lse, wo, wl)
    wt.close()


def test_repeated_calls_reuse_slots(kvattn):
    import torch
    rng = np.random.default_rng(3)
    N, n_win, H, Hk, D = 6000, 500, 16, 4, 128
    wt = kvattn.WindowTail()
    ws = wt.workspace(H, Hk, D, n_win, N - n_win, 128, 256, 64)
    cs = torch.cuda.Stream()
    for trial in range(3):
        q, k, v = make(rng, N, n_win, H, Hk, D)
        out, lse = run(kvattn, wt, q, k, v, n_win, 256, ws=ws, copy_stream=cs)
        wo, wl = oracle.decode_f16(q, k, v, [N])
        assert_close(out, lse, wo, wl)
    wt.close()


def test_fault_injection_then_recovery(kvattn, monkeypatch):
    """A failed tile copy (injected on the host) returns an error; the next call works."""
    rng = np.random.default_rng(4)
    N, n_win, H, Hk, D = 4000, 500, 16, 4, 128
    q, k, v = make(rng, N, n_win, H, Hk, D)
    wt = kvattn.WindowTail()
    monkeypatch.setenv("KVATTN_FAULT", "copy@3")
    with pytest.raises(kvattn.KvattnError) as e:
        run(kvattn, wt, q, k, v, n_win, 256)
    assert e.value.status == kvattn.KVATTN_ERR_CUDA
    monkeypatch.delenv("KVATTN_FAULT")
    out, lse = run(kvattn, wt, q, k, v, n_win, 256)
    wo, wl = oracle.decode_f16(q, k, v, [N])
    assert_close(out, lse, wo, wl)
    wt.close()


def test_host_wait_times_out_then_completes(kvattn):
    """kvattn_tail_wait gives up after its limit while the stream is still busy."""
    import torch
    rng = np.random.default_rng(5)
    N, n_win, H, Hk, D = 3000, 500, 16, 4, 128
    q, k, v = make(rng, N, n_win, H, Hk, D)
    n_tail = N - n_win
    k_tail = torch.from_numpy(k[:n_tail]).pin_memory()
    v_tail = torch.from_numpy(v[:n_tail]).pin_memory()
    wt = kvattn.WindowTail()
    qd, kw, vw = dev(q[0]), dev(k[n_tail:]), dev(v[n_tail:])
    ws = wt.workspace(H, Hk, D, n_win, n_tail, 128, 256, 64)
    out = torch.empty((H, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((H,), dtype=torch.float32, device="cuda")
    copy_stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    torch.cuda._sleep(400_000_000)   # a bounded busy kernel ahead of the decode on this stream
    wt(qd, kw, vw, k_tail, v_tail, split=128, tile_cells=256, tail_split=64, out=out, lse=lse, ws=ws,
       copy_stream=copy_stream)
    with pytest.raises(kvattn.KvattnError) as e:
        kvattn.kvattn_tail_wait(wt.ctx, 1)
    assert e.value.status == kvattn.KVATTN_ERR_TIMEOUT
    kvattn.kvattn_tail_wait(wt.ctx, 60000)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_f16(q, k, v, [N])
    assert_close(out.view(1, *out.shape), lse.view(1, -1), wo, wl)
    wt.close()


def test_replayed_graph_reads_new_host_data(kvattn):
    """Same buffers, new contents: the recorded pipeline must copy the new tail each call."""
    import torch
    rng = np.random.default_rng(6)
    N, n_win, H, Hk, D = 5000, 700, 16, 4, 128
    n_tail = N - n_win
    k_tail = torch.empty((n_tail, Hk, D), dtype=torch.float16).pin_memory()
    v_tail = torch.empty((n_tail, Hk, D), dtype=torch.float16).pin_memory()
    kw = torch.empty((n_win, Hk, D), dtype=torch.float16, device="cuda")
    vw = torch.empty((n_win, Hk, D), dtype=torch.float16, device="cuda")
    qd = torch.empty((H, D), dtype=torch.float16, device="cuda")
    wt = kvattn.WindowTail()
    ws = wt.workspace(H, Hk, D, n_win, n_tail, 128, 512, 128)
    out = torch.empty((H, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((H,), dtype=torch.float32, device="cuda")
    cs = torch.cuda.Stream()
    for trial in range(3):
        q, k, v = make(rng, N, n_win, H, Hk, D)
        torch.cuda.synchronize()
        k_tail.copy_(torch.from_numpy(k[:n_tail]))
        v_tail.copy_(torch.from_numpy(v[:n_tail]))
        kw.copy_(torch.from_numpy(k[n_tail:]))
        vw.copy_(torch.from_numpy(v[n_tail:]))
        qd.copy_(torch.from_numpy(q[0]))
        torch.cuda.synchronize()
        wt(qd, kw, vw, k_tail, v_tail, split=128, tile_cells=512, tail_split=128, out=out, lse=lse, ws=ws,
           copy_stream=cs)
        kvattn.kvattn_tail_wait(wt.ctx, 30000)
        torch.cuda.synchronize()
        wo, wl = oracle.decode_f16(q, k, v, [N])
        assert_close(out.view(1, H, D), lse.view(1, H), wo, wl)
    wt.close()


@pytest.mark.parametrize("N,n_win,H,Hk,tail_split", [
    (5000, 1000, 40, 8, 128),     # ragged tail
    (3000, 0, 16, 4, 64),         # everything in the tail
    (777, 777, 16, 4, 128),       # everything resident
    (4100, 64, 24, 4, 256),       # GQA-6
])
def test_direct_tail_reads(kvattn, N, n_win, H, Hk, tail_split):
    """The tail read in place from pinned host memory (no staging copies)."""
    import torch
    rng = np.random.default_rng(N + 7 * n_win)
    q, k, v = make(rng, N, n_win, H, Hk, 128)
    n_tail = N - n_win
    k_tail = torch.from_numpy(k[:n_tail]).pin_memory() if n_tail else None
    v_tail = torch.from_numpy(v[:n_tail]).pin_memory() if n_tail else None
    kw = dev(k[n_tail:]) if n_win else None
    vw = dev(v[n_tail:]) if n_win else None
    out, lse = kvattn.window_tail_direct(dev(q[0]), kw, vw, k_tail, v_tail, split=128, tail_split=tail_split)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_f16(q, k, v, [N])
    assert_close(out.view(1, H, 128), lse.view(1, H), wo, wl)


@pytest.mark.parametrize("mode", ["staged", "direct"])
def test_window_tail_head_dim_256(kvattn, mode):
    """head_dim 256 (512-byte rows): a ragged last tile, GQA-2."""
    import torch
    rng = np.random.default_rng(31)
    N, n_win, H, Hk, D = 3000, 500, 16, 8, 256
    q, k, v = make(rng, N, n_win, H, Hk, D)
    n_tail = N - n_win
    k_tail = torch.from_numpy(k[:n_tail]).pin_memory()
    v_tail = torch.from_numpy(v[:n_tail]).pin_memory()
    if mode == "staged":
        wt = kvattn.WindowTail()
        out, lse = wt(dev(q[0]), dev(k[n_tail:]), dev(v[n_tail:]), k_tail, v_tail, split=128, tile_cells=384,
                      tail_split=128, copy_stream=torch.cuda.Stream())
        kvattn.kvattn_tail_wait(wt.ctx, 30000)
        wt.close()
    else:
        out, lse = kvattn.window_tail_direct(dev(q[0]), dev(k[n_tail:]), dev(v[n_tail:]), k_tail, v_tail, split=128,
                                             tail_split=128)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_f16(q, k, v, [N])
    assert_close(out.view(1, H, D), lse.view(1, H), wo, wl)


def test_unpinned_tail(kvattn):
    """Pageable host memory: the staged path copies it with cudaMemcpyAsync (the copy kernel
    needs a device mapping) and records no graph.  The direct path needs a device address
    for the tail: where the platform gives pageable memory one (a coherent host such as
    Grace, through address translation) it reads the tail in place and must be right,
    elsewhere it refuses the call before any launch."""
    import torch
    rng = np.random.default_rng(41)
    N, n_win, H, Hk, D = 1500, 300, 16, 4, 128
    q, k, v = make(rng, N, n_win, H, Hk, D)
    n_tail = N - n_win
    k_tail = torch.from_numpy(k[:n_tail].copy())  # not pinned
    v_tail = torch.from_numpy(v[:n_tail].copy())
    wt = kvattn.WindowTail()
    out, lse = wt(dev(q[0]), dev(k[n_tail:]), dev(v[n_tail:]), k_tail, v_tail, split=128, tile_cells=256,
                  tail_split=64, copy_stream=torch.cuda.Stream())
    kvattn.kvattn_tail_wait(wt.ctx, 30000)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_f16(q, k, v, [N])
    assert_close(out.view(1, H, D), lse.view(1, H), wo, wl)
    wt.close()
    try:
        out, lse = kvattn.window_tail_direct(dev(q[0]), dev(k[n_tail:]), dev(v[n_tail:]), k_tail, v_tail,
                                             split=128, tail_split=64)
        torch.cuda.synchronize()
        assert_close(out.view(1, H, D), lse.view(1, H), wo, wl)
    except kvattn.KvattnError as e:
        assert e.status == kvattn.KVATTN_ERR_INVALID_ARG
    # the context is still usable
    out, lse = kvattn.window_tail_direct(dev(q[0]), dev(k[n_tail:]), dev(v[n_tail:]), k_tail.pin_memory(),
                                         v_tail.pin_memory(), split=128, tail_split=64)
    torch.cuda.synchronize()
    assert_close(out.view(1, H, D), lse.view(1, H), wo, wl)
