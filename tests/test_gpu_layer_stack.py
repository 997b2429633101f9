"""A stack of layers through one tail context, enqueued back to back with no host sync
between layers, each layer checked against the fp64 oracle: cross-layer prefetch mode
(copies wait only for their staging slot's last reader, the slot sequence continuing from
layer to layer), a switch between the modes in the middle of a stack, and more layers than
the context keeps recorded graphs for."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu

H, HK, D = 16, 4, 128


def make_layers(rng, shapes):
    """shapes: (n_win, n_tail) per layer.  Every layer has its own q, window and tail."""
    import torch
    layers = []
    for n_win, n_tail in shapes:
        N = n_win + n_tail
        q = rng.standard_normal((1, H, D), dtype=np.float32).astype(np.float16)
        k = rng.standard_normal((N, HK, D), dtype=np.float32).astype(np.float16)
        v = rng.standard_normal((N, HK, D), dtype=np.float32).astype(np.float16)
        layers.append(dict(
            q=q, k=k, v=v, n_win=n_win, n_tail=n_tail, qd=dev(q[0]),
            k_win=dev(k[n_tail:]) if n_win else None, v_win=dev(v[n_tail:]) if n_win else None,
            k_tail=torch.from_numpy(k[:n_tail]).pin_memory() if n_tail else None,
            v_tail=torch.from_numpy(v[:n_tail]).pin_memory() if n_tail else None))
    return layers


def run_stack(kvattn, wt, layers, tile, ws, cs, xs, split=128, tail_split=64, modes=None):
    import torch
    outs = []
    with torch.cuda.stream(cs):
        for i, ly in enumerate(layers):
            if modes is not None:
                kvattn.kvattn_tail_ctx_set_flags(wt.ctx, modes[i])
            out = torch.empty((H, D), dtype=torch.float32, device="cuda")
            lse = torch.empty((H,), dtype=torch.float32, device="cuda")
            wt(ly["qd"], ly["k_win"], ly["v_win"], ly["k_tail"], ly["v_tail"], split=split, tile_cells=tile,
               tail_split=tail_split, out=out, lse=lse, ws=ws, compute_stream=cs, copy_stream=xs)
            outs.append((out, lse))
    kvattn.kvattn_tail_wait(wt.ctx, 60000)
    torch.cuda.synchronize()
    return outs


def check(outs, layers):
    for (out, lse), ly in zip(outs, layers):
        wo, wl = oracle.decode_f16(ly["q"], ly["k"], ly["v"], [ly["n_win"] + ly["n_tail"]])
        assert_close(out.view(1, H, D), lse.view(1, H), wo, wl)


# odd and even tile counts per layer (so the staging slot a layer starts on alternates),
# a layer without tail, a layer without window, a ragged last tile
SHAPES = [(300, 1000), (64, 700), (500, 1300), (128, 256), (200, 0), (0, 900), (96, 513), (256, 1024)]


@pytest.mark.parametrize("copy_kernel", ["0", "1"])
def test_prefetch_stack_matches_oracle(kvattn, monkeypatch, copy_kernel):
    import torch
    monkeypatch.setenv("KVATTN_TAIL_COPY", copy_kernel)
    rng = np.random.default_rng(61 + int(copy_kernel))
    layers = make_layers(rng, SHAPES)
    tile = 256
    wt = kvattn.WindowTail(prefetch=True)
    max_win = max(s[0] for s in SHAPES)
    max_tail = max(s[1] for s in SHAPES)
    ws = wt.workspace(H, HK, D, max_win, max_tail, 128, tile, 64)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(2):  # a second pass carries the slot sequence over from the first
        outs = run_stack(kvattn, wt, layers, tile, ws, cs, xs)
        check(outs, layers)
    wt.close()


def test_whole_layer_tiles(kvattn):
    """One tile per layer: the two staging slots alternate between layers, so a layer's
    whole tail is copied while the layer before it computes."""
    import torch
    rng = np.random.default_rng(62)
    shapes = [(256, 1024)] * 5 + [(256, 700)]
    layers = make_layers(rng, shapes)
    wt = kvattn.WindowTail(prefetch=True)
    ws = wt.workspace(H, HK, D, 256, 1024, 128, 1024, 128)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    outs = run_stack(kvattn, wt, layers, 1024, ws, cs, xs, tail_split=128)
    check(outs, layers)
    wt.close()


def test_mode_switches_inside_a_stack(kvattn):
    """Recorded-graph calls, then prefetch calls, then graph calls again, all enqueued
    before any result is read: each switch keeps the staging slots ordered."""
    import torch
    rng = np.random.default_rng(63)
    layers = make_layers(rng, SHAPES)
    modes = [0, 0, kvattn.KVATTN_TAIL_PREFETCH, kvattn.KVATTN_TAIL_PREFETCH, kvattn.KVATTN_TAIL_PREFETCH, 0,
             kvattn.KVATTN_TAIL_PREFETCH, 0]
    wt = kvattn.WindowTail()
    ws = wt.workspace(H, HK, D, 500, 1300, 128, 256, 64)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(2):
        outs = run_stack(kvattn, wt, layers, 256, ws, cs, xs, modes=modes)
        check(outs, layers)
    wt.close()


def test_first_prefetch_call_with_one_tile(kvattn):
    """The first call of a carried sequence uses one staging slot only; the next call's copy
    into the other slot must still follow the recorded-graph call that read it before."""
    import torch
    rng = np.random.default_rng(66)
    shapes = [(64, 1300), (64, 200), (64, 900), (64, 700), (64, 1300), (64, 100), (64, 1000)]
    P = kvattn.KVATTN_TAIL_PREFETCH
    modes = [0, P, P, P, 0, P, P]
    layers = make_layers(rng, shapes)
    wt = kvattn.WindowTail()
    ws = wt.workspace(H, HK, D, 64, 1300, 128, 256, 64)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        outs = run_stack(kvattn, wt, layers, 256, ws, cs, xs, modes=modes)
        check(outs, layers)
    wt.close()


def test_more_layers_than_recorded_graphs(kvattn):
    """70 layers through one context that keeps 64 recorded pipelines: the least recently
    used ones are replaced, and every layer's result stays right over two passes (the
    second pass with new queries, read by the replayed or re-recorded graphs)."""
    import torch
    rng = np.random.default_rng(64)
    shapes = [(64, 200 + 7 * (i % 5)) for i in range(70)]
    layers = make_layers(rng, shapes)
    wt = kvattn.WindowTail()
    ws_list = [wt.workspace(H, HK, D, 64, 228, 128, 128, 64) for _ in range(2)]
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    for p in range(2):
        if p == 1:
            for ly in layers:
                ly["q"] = rng.standard_normal((1, H, D), dtype=np.float32).astype(np.float16)
                ly["qd"].copy_(torch.from_numpy(ly["q"][0]))
        outs = []
        with torch.cuda.stream(cs):
            for i, ly in enumerate(layers):
                out = torch.empty((H, D), dtype=torch.float32, device="cuda")
                lse = torch.empty((H,), dtype=torch.float32, device="cuda")
                wt(ly["qd"], ly["k_win"], ly["v_win"], ly["k_tail"], ly["v_tail"], split=128, tile_cells=128,
                   tail_split=64, out=out, lse=lse, ws=ws_list[i % 2], compute_stream=cs, copy_stream=xs)
                outs.append((out, lse))
        torch.cuda.synchronize()
        check(outs, layers)
    wt.close()


@pytest.mark.parametrize("copy_kernel", ["0", "1"])
def test_captured_prefetch_stack(kvattn, monkeypatch, copy_kernel):
    """A whole stack in prefetch mode recorded as one CUDA graph by the caller and replayed:
    the replay reads the queries and tails as they are at replay time."""
    import torch
    monkeypatch.setenv("KVATTN_TAIL_COPY", copy_kernel)
    rng = np.random.default_rng(65)
    layers = make_layers(rng, SHAPES)
    wt = kvattn.WindowTail(prefetch=True)
    ws = wt.workspace(H, HK, D, 500, 1300, 128, 256, 64)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    outs = [(torch.empty((H, D), dtype=torch.float32, device="cuda"),
             torch.empty((H,), dtype=torch.float32, device="cuda")) for _ in layers]
    run_stack(kvattn, wt, layers, 256, ws, cs, xs)  # an eager pass first: the capture must not carry it over
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        for ly, (out, lse) in zip(layers, outs):
            wt(ly["qd"], ly["k_win"], ly["v_win"], ly["k_tail"], ly["v_tail"], split=128, tile_cells=256,
               tail_split=64, out=out, lse=lse, ws=ws, compute_stream=cs, copy_stream=xs)
    for _ in range(2):
        for ly in layers:
            ly["q"] = rng.standard_normal((1, H, D), dtype=np.float32).astype(np.float16)
            ly["qd"].copy_(torch.from_numpy(ly["q"][0]))
            if ly["n_tail"]:
                n = ly["n_tail"]
                ly["k"][:n] = rng.standard_normal((n, HK, D), dtype=np.float32).astype(np.float16)
                ly["k_tail"].copy_(torch.from_numpy(ly["k"][:n]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        check(outs, layers)
    del g
    wt.close()


def test_captured_stack_one_tile_per_layer(kvattn):
    """Whole-layer tiles inside a capture: the first captured layer fills one staging slot,
    and the second layer's copy into the other slot must wait on a record made inside the
    capture, not on one from the eager calls before it."""
    import torch
    rng = np.random.default_rng(67)
    shapes = [(128, 1024), (128, 1000), (128, 700), (128, 1024)]
    layers = make_layers(rng, shapes)
    wt = kvattn.WindowTail(prefetch=True)
    ws = wt.workspace(H, HK, D, 128, 1024, 128, 1024, 128)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    outs = [(torch.empty((H, D), dtype=torch.float32, device="cuda"),
             torch.empty((H,), dtype=torch.float32, device="cuda")) for _ in layers]
    run_stack(kvattn, wt, layers, 1024, ws, cs, xs, tail_split=128)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        for ly, (out, lse) in zip(layers, outs):
            wt(ly["qd"], ly["k_win"], ly["v_win"], ly["k_tail"], ly["v_tail"], split=128, tile_cells=1024,
               tail_split=128, out=out, lse=lse, ws=ws, compute_stream=cs, copy_stream=xs)
    for _ in range(2):
        for ly in layers:
            ly["q"] = rng.standard_normal((1, H, D), dtype=np.float32).astype(np.float16)
            ly["qd"].copy_(torch.from_numpy(ly["q"][0]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        check(outs, layers)
    del g
    wt.close()
