"""Out-of-bounds guards for every kernel family: sentinel regions before and after every
buffer the library writes (out, lse, caller partials, the workspace) and inside the
workspace (the alignment gaps between the descriptor, partial-LSE, partial-O and staging
regions), checked byte for byte after each call.  A write past a buffer's end, or a padded
GQA row written as if it were a real head -- the out-of-bounds access the pages record
("KVARN KV Performance optimizations", item 2) -- lands in a sentinel.

Cases: every cache type at head_dim 128 and 256, ragged lengths and an empty sequence,
G = 5, 6 and 7 (query rows padded to eight), the quantised head_dim-128 caches as KV-head
pairs (G = 2, 3, 4: each query row keeps its own head's half), compact plans with holes, the partials entry
point, multi-query row layouts and row groups, window + tail (staged tiles with a ragged
last tile, and the tail read in place) and the merge.  Results are also checked against the
oracle so that a guard cannot pass on a call that did nothing.
"""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu

FSENT = 12345.0     # float sentinel around out / lse / partials
BSENT = 0xA5        # byte sentinel around and inside the workspace
GUARD = 4096        # sentinel bytes on each side (a multiple of the 256-byte workspace alignment)
WS_ALIGN = 256
STATUS_BYTES = 256


def align_up(x, a=WS_ALIGN):
    return (x + a - 1) // a * a


def decode_layout(n_seq, n_rows, D, n_split):
    """Byte ranges of the decode workspace: status word | descriptors | partial LSE |
    partial O, each region starting on a 256-byte boundary.  Returns (total, used ranges)."""
    off = STATUS_BYTES
    desc = (off, off + n_seq * n_split * 16)
    off = align_up(desc[1])
    lse = (off, off + n_seq * n_split * n_rows * 4)
    off = align_up(lse[1])
    o = (off, off + n_seq * n_split * n_rows * D * 4)
    total = align_up(o[1])
    return total, [(0, 4), desc, lse, o]


def tail_layout(H, Hk, D, n_win, n_tail, split, tile, tail_split):
    """Window + tail workspace: status | slot 0 K, V | slot 1 K, V | the partials of every
    window split and tail tile split (a decode layout of one sequence)."""
    tile_bytes = tile * Hk * D * 2
    off = STATUS_BYTES
    used = [(0, 4)]
    for _ in range(4):
        used.append((off, off + tile_bytes))
        off = align_up(off + tile_bytes)
    n_parts = -(-n_win // split) + (-(-n_tail // tile)) * (tile // tail_split)
    ptotal, pused = decode_layout(1, H, D, n_parts)
    used += [(off + a, off + b) for a, b in pused[1:]]
    return off + ptotal, used


class Guarded:
    """A device buffer of n elements between sentinel regions (floats, or bytes for a
    workspace); ``inner`` is the view handed to the library."""

    def __init__(self, shape, kind="f32", used=None):
        import torch
        n = int(np.prod(shape))
        self.n = n
        if kind == "f32":
            self.g = GUARD // 4
            self.big = torch.full((n + 2 * self.g,), FSENT, dtype=torch.float32, device="cuda")
            self.sent = FSENT
        else:
            self.g = GUARD
            self.big = torch.full((n + 2 * self.g,), BSENT, dtype=torch.uint8, device="cuda")
            self.big[self.g:self.g + 4] = 0           # the status word starts clear
            self.sent = BSENT
        self.inner = self.big[self.g:self.g + n].view(shape)
        self.used = used

    def check(self, what):
        b = self.big.cpu().numpy()
        before, after = b[:self.g], b[self.g + self.n:]
        assert np.all(before == self.sent), f"{what}: write before the buffer"
        assert np.all(after == self.sent), f"{what}: write past the end"
        if self.used is not None:
            body = b[self.g:self.g + self.n]
            free = np.ones(self.n, bool)
            for lo, hi in self.used:
                free[lo:hi] = False
            bad = np.nonzero(free & (body != self.sent))[0]
            assert bad.size == 0, f"{what}: write in a workspace gap at byte {bad[:4]}"
            assert int.from_bytes(body[:4].tobytes(), "little") == 0, f"{what}: status word set"


def rand_f16(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def quant_cache(rng, kind, lead, D):
    lead = tuple(lead)
    if kind == "q4":
        kq = rng.integers(0, 256, lead + (D // 2,), dtype=np.uint8)
        kd = rng.uniform(0.001, 0.3, lead + (D // 32,)).astype(np.float16)
    else:
        kq = rng.integers(-127, 128, lead + (D,), dtype=np.int8)
        kd = rng.uniform(0.001, 0.02, lead + (D // 32,)).astype(np.float16)
    if kind == "q8":
        vq = rng.integers(-127, 128, lead + (D,), dtype=np.int8)
        vd = rng.uniform(0.001, 0.02, lead + (D // 32,)).astype(np.float16)
    else:
        vq = rng.integers(0, 256, lead + (D // 2,), dtype=np.uint8)
        vd = rng.uniform(0.001, 0.3, lead + (D // 32,)).astype(np.float16)
    return kq, kd, vq, vd


KV_TYPE = {"f16": "KVATTN_KV_F16", "q8": "KVATTN_KV_Q8_0", "q8q4": "KVATTN_KV_Q8_0_Q4_0", "q4": "KVATTN_KV_Q4_0"}
ORACLE = {"f16": oracle.decode_f16, "q8": oracle.decode_q8_0, "q8q4": oracle.decode_q8_0_q4_0,
          "q4": oracle.decode_q4_0}


def make_cache(rng, kind, lead, D):
    if kind == "f16":
        return rand_f16(rng, tuple(lead) + (D,)), rand_f16(rng, tuple(lead) + (D,))
    return quant_cache(rng, kind, lead, D)


def device_args(kind, cache):
    """(k, v, k_scales, v_scales) device tensors for the C ABI."""
    if kind == "f16":
        return dev(cache[0]), dev(cache[1]), None, None
    kq, kd, vq, vd = cache
    return dev(kq), dev(vq), dev(kd), dev(vd)


SINGLE = [
    # kind, D, G, lens, split
    ("f16", 128, 5, [1000, 333, 0], 128),
    ("f16", 128, 7, [77, 1500], 64),
    ("f16", 256, 6, [999, 0, 250], 128),
    ("q8", 128, 7, [1100, 17, 0], 128),
    ("q8", 256, 5, [700, 1023], 64),
    ("q8q4", 128, 6, [1300, 0, 99], 256),
    ("q8q4", 256, 7, [515, 64], 128),
    ("q4", 128, 5, [2049, 3], 512),
    ("q4", 256, 6, [800, 0], 128),
    # head_dim 128 with G <= 4 and an even KV-head count: KV-head pairs on the 256 kernels
    ("q8", 128, 4, [1100, 17, 0], 128),
    ("q8q4", 128, 3, [515, 64], 64),
    ("q4", 128, 2, [2049, 3], 512),
    # more units than one wave of two-warp CTAs: one-warp CTAs, a unit per warp (782 KV-head
    # pair units; 628 units of head_dim 256)
    ("q8", 128, 4, [100000], 128),
    ("q4", 256, 6, [20000, 333], 128),
    # 125 parts a row at head_dim 128: each row's merge spread over several CTAs
    ("f16", 128, 4, [4000, 1000, 0], 32),
    ("q8", 128, 4, [4000, 77], 32),
]


@pytest.mark.parametrize("kind,D,G,lens,split", SINGLE)
def test_guards_single_query(kvattn, kind, D, G, lens, split):
    import torch
    rng = np.random.default_rng([41, D, G, len(lens)])
    S, Hk = len(lens), 2
    H = G * Hk
    N = max(lens)
    q = rand_f16(rng, (S, H, D))
    cache = make_cache(rng, kind, (S, N, Hk), D)
    k, v, ks, vs = device_args(kind, cache)
    n_split = -(-N // split)
    total, used = decode_layout(S, H, D, n_split)
    assert total == kvattn.kvattn_decode_workspace_bytes(S, H, D, N, split)
    out = Guarded((S, H, D))
    lse = Guarded((S, H))
    ws = Guarded((total,), "u8", used)
    kvattn.kvattn_decode(dev(q), k, v, ks, vs, getattr(kvattn, KV_TYPE[kind]), N, None, 0,
                         dev(np.asarray(lens, np.int32)), S, N, H, Hk, D, split, 1.0 / np.sqrt(D), out.inner,
                         lse.inner, ws.inner, total)
    torch.cuda.synchronize()
    out.check("out")
    lse.check("lse")
    ws.check("workspace")
    wo, wl = ORACLE[kind](q, *cache, lens)
    assert_close(out.inner, lse.inner, wo, wl)


@pytest.mark.parametrize("kind,D,G", [("f16", 128, 6), ("f16", 256, 5), ("q8", 128, 7), ("q4", 256, 6),
                                     ("q8q4", 128, 4)])
def test_guards_plan_and_partials(kvattn, kind, D, G):
    """A compact plan with holes (descriptors written into the workspace), decoded once
    through kvattn_decode and once through kvattn_decode_partials into guarded caller
    partials; the partials merged by kvattn_merge into guarded outputs."""
    import torch
    rng = np.random.default_rng([42, D, G])
    Hk, pool = 2, 20
    H = G * Hk
    n_cells = pool * 128
    cache = make_cache(rng, kind, (n_cells, Hk), D)
    perm = rng.permutation(pool)
    encoded = []
    for recs in (perm[:5], perm[5:6], perm[6:13]):
        cells = (recs[:, None] * 128 + np.arange(128)[None]).reshape(-1)
        sel = cells[rng.random(cells.size) >= 0.2]
        encoded.append(sel.astype(np.int64))
    plan, lens = kvattn.build_cell_plan(encoded, n_cells)
    S, stride = plan.shape
    split = 128
    q = rand_f16(rng, (S, H, D))
    k, v, ks, vs = device_args(kind, cache)
    n_split = -(-stride // split)
    total, used = decode_layout(S, H, D, n_split)
    scale = 1.0 / np.sqrt(D)
    kt = getattr(kvattn, KV_TYPE[kind])
    wo, wl = ORACLE[kind](q, *cache, lens.tolist(), plan=plan)

    out, lse, ws = Guarded((S, H, D)), Guarded((S, H)), Guarded((total,), "u8", used)
    kvattn.kvattn_decode(dev(q), k, v, ks, vs, kt, n_cells, dev(plan), stride, dev(lens), S, stride, H, Hk, D, split,
                         scale, out.inner, lse.inner, ws.inner, total)
    torch.cuda.synchronize()
    for g, what in ((out, "out"), (lse, "lse"), (ws, "workspace")):
        g.check(what)
    assert_close(out.inner, lse.inner, wo, wl)

    # partials: [S][n_split][H][D] and [S][n_split][H]; the workspace holds status + descriptors
    po, pl = Guarded((S, n_split, H, D)), Guarded((S, n_split, H))
    ws2 = Guarded((total,), "u8", used[:2])
    kvattn.kvattn_decode_partials(dev(q), k, v, ks, vs, kt, n_cells, dev(plan), stride, dev(lens), S, stride, H, Hk,
                                  D, split, scale, po.inner, pl.inner, ws2.inner, total)
    torch.cuda.synchronize()
    for g, what in ((po, "partial O"), (pl, "partial LSE"), (ws2, "workspace (partials)")):
        g.check(what)
    mo, ml = Guarded((S * H, D)), Guarded((S * H,))
    parts = po.inner.permute(1, 0, 2, 3).reshape(n_split, S * H, D).contiguous()
    lses = pl.inner.permute(1, 0, 2).reshape(n_split, S * H).contiguous()
    kvattn.kvattn_merge(parts, lses, n_split, S * H, D, mo.inner, ml.inner)
    torch.cuda.synchronize()
    mo.check("merged out")
    ml.check("merged lse")
    assert_close(mo.inner.view(S, H, D), ml.inner.view(S, H), wo, wl)


MULTI = [
    # kind, D, n_q, G, lens, split  (rows per KV head = n_q * G)
    ("f16", 128, 1, 7, [900, 5], 128),        # one token, 7 rows padded to 8
    ("f16", 128, 2, 5, [700, 1, 0], 64),      # 10 rows: one 16-row tile
    ("f16", 128, 4, 5, [1033, 4], 128),       # 20 rows (units in one wave: the tcgen05 kernel)
    ("f16", 128, 6, 7, [600, 6, 2], 64),      # 42 rows: the tcgen05 kernel, two row warps
    ("f16", 256, 1, 6, [500, 77], 128),
    ("f16", 256, 3, 5, [777, 0], 128),        # 15 rows: 8 per warp
    ("f16", 256, 5, 6, [400, 5], 64),         # 30 rows: row groups of 16
    ("q8", 128, 2, 7, [901, 2], 128),         # 14 rows: the 16-row quantised consumer
    ("q8", 128, 6, 5, [640, 3], 64),          # 30 rows: row groups of 16
    ("q8q4", 256, 2, 6, [513, 0], 128),       # 12 rows: row groups of 8
    ("q4", 128, 1, 5, [1000, 9], 256),
    ("q4", 256, 3, 7, [333, 3], 64),          # 21 rows: row groups of 8
]


@pytest.mark.parametrize("kind,D,n_q,G,lens,split", MULTI)
def test_guards_multi_query(kvattn, kind, D, n_q, G, lens, split):
    import torch
    rng = np.random.default_rng([43, D, n_q, G])
    S, Hk = len(lens), 2
    H = G * Hk
    N = max(lens)
    q = rand_f16(rng, (S, n_q, H, D))
    cache = make_cache(rng, kind, (S, N, Hk), D)
    k, v, ks, vs = device_args(kind, cache)
    n_split = -(-N // split)
    total, used = decode_layout(S, n_q * H, D, n_split)
    assert total == kvattn.kvattn_decode_multi_workspace_bytes(S, n_q, H, D, N, split)
    out, lse, ws = Guarded((S, n_q, H, D)), Guarded((S, n_q, H)), Guarded((total,), "u8", used)
    kvattn.kvattn_decode_multi(dev(q), k, v, ks, vs, getattr(kvattn, KV_TYPE[kind]), N, None, 0,
                               dev(np.asarray(lens, np.int32)), S, N, n_q, H, Hk, D, split, 1.0 / np.sqrt(D),
                               out.inner, lse.inner, ws.inner, total)
    torch.cuda.synchronize()
    for g, what in ((out, "out"), (lse, "lse"), (ws, "workspace")):
        g.check(what)
    wo, wl = oracle.decode_multi(ORACLE[kind], q, lens, *cache)
    o, l = out.inner.cpu().numpy(), lse.inner.cpu().numpy()
    fin = np.isfinite(wl)
    assert np.array_equal(np.isneginf(l), np.isneginf(wl))
    assert np.max(np.abs(o - wo)) <= 2e-3
    assert np.max(np.abs(l[fin] - wl[fin]), initial=0.0) <= 1e-4


@pytest.mark.parametrize("mode", ["staged", "direct"])
@pytest.mark.parametrize("N,n_win,tile,G,D", [(4500, 700, 512, 5, 128), (3001, 1, 256, 7, 128),
                                              (2100, 300, 256, 6, 256)])
def test_guards_window_tail(kvattn, mode, N, n_win, tile, G, D):
    """Ragged last tile (4500 - 700 = 7 x 512 + 216; 3000 = 11 x 256 + 184), a one-cell window,
    head_dim 256; the staging slots, partials and outputs all guarded."""
    import torch
    rng = np.random.default_rng([44, N, G, mode == "direct"])
    Hk = 2
    H = G * Hk
    split, tail_split = 128, 64
    n_tail = N - n_win
    q = rand_f16(rng, (1, H, D))
    k = rand_f16(rng, (N, Hk, D))
    v = rand_f16(rng, (N, Hk, D))
    k_tail = torch.from_numpy(k[:n_tail]).pin_memory()
    v_tail = torch.from_numpy(v[:n_tail]).pin_memory()
    scale = 1.0 / np.sqrt(D)
    out, lse = Guarded((H, D)), Guarded((H,))
    if mode == "staged":
        total, used = tail_layout(H, Hk, D, n_win, n_tail, split, tile, tail_split)
        assert total == kvattn.kvattn_window_tail_workspace_bytes(H, Hk, D, n_win, n_tail, split, tile, tail_split)
        ws = Guarded((total,), "u8", used)
        wt = kvattn.WindowTail()
        wt(dev(q[0]), dev(k[n_tail:]), dev(v[n_tail:]), k_tail, v_tail, split=split, tile_cells=tile,
           tail_split=tail_split, out=out.inner, lse=lse.inner, ws=ws.inner, copy_stream=torch.cuda.Stream())
        kvattn.kvattn_tail_wait(wt.ctx, 30000)
    else:
        n_parts = -(-n_win // split) + -(-n_tail // tail_split)
        total, used = decode_layout(1, H, D, n_parts)
        assert total == kvattn.kvattn_window_tail_direct_workspace_bytes(H, Hk, D, n_win, n_tail, split, tail_split)
        ws = Guarded((total,), "u8", used)
        kvattn.window_tail_direct(dev(q[0]), dev(k[n_tail:]), dev(v[n_tail:]), k_tail, v_tail, split=split,
                                  tail_split=tail_split, out=out.inner, lse=lse.inner, ws=ws.inner)
    torch.cuda.synchronize()
    for g, what in ((out, "out"), (lse, "lse"), (ws, "workspace")):
        g.check(what)
    if mode == "staged":
        wt.close()
    wo, wl = oracle.decode_f16(q, k, v, [N])
    assert_close(out.inner.view(1, H, D), lse.inner.view(1, H), wo, wl)


@pytest.mark.parametrize("P,R,D", [(1, 7, 128), (65, 13, 128), (33, 5, 256), (300, 3, 128)])
def test_guards_merge(kvattn, P, R, D):
    import torch
    rng = np.random.default_rng([45, P, R, D])
    parts = rng.standard_normal((P, R, D)).astype(np.float32)
    lses = (rng.standard_normal((P, R)) * 3).astype(np.float32)
    if P > 1:
        lses[1] = -np.inf
        parts[1] = np.nan
    out, lse = Guarded((R, D)), Guarded((R,))
    kvattn.kvattn_merge(dev(parts), dev(lses), P, R, D, out.inner, lse.inner)
    torch.cuda.synchronize()
    out.check("out")
    lse.check("lse")
    wo, wl = oracle.merge(parts, lses)
    assert_close(out.inner, lse.inner, wo, wl, tol_o=1e-5, tol_l=1e-5)
