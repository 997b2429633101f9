"""Seeded synthetic inputs for single-query decode attention.

This module only draws random numbers and lays them out in the cache formats the
library reads. It holds none of the attention arithmetic, builds no cell plan and
computes no expected value, so both the CUDA path and the CPU oracle may take
their inputs from it.

Layouts (all row-major, C order):

* q            f16  [n_seq][n_head][head_dim]
* K, V (f16)   f16  [n_cells][n_head_kv][head_dim]          (cell-major rows)
* K, V (Q8_0)  qs int8 [n_cells][n_head_kv][head_dim] plus
               d  f16  [n_cells][n_head_kv][head_dim // 32]  (value = d * qs)
* K, V (Q4_0)  packed uint8 [n_cells][n_head_kv][head_dim // 2] plus
               d  f16  [n_cells][n_head_kv][head_dim // 32]
               (byte j of block b: element 32b + j low nibble, 32b + 16 + j high;
               value = d * (nibble - 8))
* encoded cells for the plan builder: int64, low 32 bits = physical cell,
  high 32 bits = a stage-slot tag that the read plan ignores.

Workloads follow the five decode-attention shapes used throughout the tests and
the benchmark: a tiny GQA-4 case, a Qwen3-8B-shaped layer, a four-sequence GQA-6
unified cache read through a compact cell plan, a Q8_0 long-context cache, a
window + host-tail overflow cache, and 36-layer stacks of window + host tail.  Seeds: 1000+w for q, 2000+w for K, 3000+w
for V, 4000+w for the record layout and holes (w = workload number).
"""
from __future__ import annotations

import dataclasses

import numpy as np

RECORD_CELLS = 128  # physical record size of the unified cache


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    number: int
    n_seq: int
    n_cells: int            # cells per sequence (contiguous) or physical pool size (plan)
    n_head: int
    n_head_kv: int
    head_dim: int
    split: int
    kv_type: str = "f16"     # "f16", "q8_0", "q8_0_q4_0" or "q4_0"
    seq_lens: tuple = ()
    hole_prob: float = 0.0
    pool_records: int = 0
    n_window: int = 0        # window + tail only
    tile_cells: int = 0      # window + tail only
    tail_split: int = 0      # window + tail only
    layers: int = 1

    @property
    def group(self) -> int:
        return self.n_head // self.n_head_kv


TINY = Workload("tiny_gqa4_n512", 1, 1, 512, 8, 2, 128, 128, seq_lens=(512,))
QWEN3_8B_LAYER = Workload("qwen3_8b_layer_n16384", 2, 1, 16384, 32, 8, 128, 256,
                          seq_lens=(16384,), layers=36)
MULTISLOT_PLAN = Workload("multislot_gqa6_plan", 3, 4, 1152 * RECORD_CELLS, 48, 8, 128, 256,
                          seq_lens=(8192, 20480, 40960, 65536), hole_prob=0.1,
                          pool_records=1152)
Q8_LONG_D128 = Workload("q8_0_n131072_d128", 4, 1, 131072, 32, 8, 128, 512,
                        kv_type="q8_0", seq_lens=(131072,))
Q8_LONG_D256 = Workload("q8_0_n131072_d256", 4, 1, 131072, 32, 8, 256, 512,
                        kv_type="q8_0", seq_lens=(131072,))
WINDOW_TAIL = Workload("window_tail_n524288", 5, 1, 524288, 40, 8, 128, 256,
                       seq_lens=(524288,), n_window=16384, tile_cells=512, tail_split=128)

# Layer stacks of window + host tail at the two overflow operating points of the pages'
# Qwen3-8B table (36 layers that all stream a tail; ~13.1k-token prompt): 11008 resident
# cells and ~2.1k tail cells per layer (295 MiB of tail per token), and the 256-cell window
# floor with ~12.9k tail cells per layer (1815 MiB).  tile_cells holds a layer's whole tail.
STACK_TAIL_295MIB = Workload("qwen3_8b_x36_tail_295mib", 6, 1, 11008 + 2100, 32, 8, 128, 256,
                             seq_lens=(11008 + 2100,), n_window=11008, tile_cells=2176, tail_split=128,
                             layers=36)
STACK_TAIL_1815MIB = Workload("qwen3_8b_x36_tail_1815mib", 7, 1, 256 + 12900, 32, 8, 128, 256,
                              seq_lens=(256 + 12900,), n_window=256, tile_cells=12928, tail_split=128,
                              layers=36)

# The mixed cache of the pages' resident-compression anchors: Q8_0 keys, Q4_0 values, at the
# Q8_0 long-context shape.
Q8Q4_LONG_D128 = Workload("q8_0_q4_0_n131072_d128", 8, 1, 131072, 32, 8, 128, 512, kv_type="q8_0_q4_0",
                          seq_lens=(131072,))
Q8Q4_LONG_D256 = Workload("q8_0_q4_0_n131072_d256", 8, 1, 131072, 32, 8, 256, 512, kv_type="q8_0_q4_0",
                          seq_lens=(131072,))

# A serving batch: 64 sequences of 4096 cells each through one call (Qwen3-8B-shaped heads, a
# per-sequence cache), the automatic split.
BATCH64 = Workload("qwen3_8b_batch64_n4096", 11, 64, 4096, 32, 8, 128, 0, seq_lens=(4096,) * 64)

# head_dim 256 (as the global layers of the pages' Gemma-family model): 16/8 heads, 65536 cells,
# the automatic split.
F16_D256_LONG = Workload("f16_n65536_d256", 10, 1, 65536, 16, 8, 256, 0, seq_lens=(65536,))

# The pages' q4_0 cache (keys and values), same shape.
Q4_LONG_D128 = Workload("q4_0_n131072_d128", 9, 1, 131072, 32, 8, 128, 512, kv_type="q4_0", seq_lens=(131072,))
Q4_LONG_D256 = Workload("q4_0_n131072_d256", 9, 1, 131072, 32, 8, 256, 512, kv_type="q4_0", seq_lens=(131072,))

WORKLOADS = {w.name: w for w in
             (TINY, QWEN3_8B_LAYER, MULTISLOT_PLAN, Q8_LONG_D128, Q8_LONG_D256, WINDOW_TAIL,
              STACK_TAIL_295MIB, STACK_TAIL_1815MIB, Q8Q4_LONG_D128, Q8Q4_LONG_D256, Q4_LONG_D128,
              Q4_LONG_D256, F16_D256_LONG, BATCH64)}


def _rng(*seed) -> np.random.Generator:
    return np.random.default_rng(list(seed))


def normal_f16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """N(0, 1) draws rounded to f16, generated in chunks to bound temporaries."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float16)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = rng.standard_normal(hi - lo, dtype=np.float32)
    return out.reshape(shape)


def normal_f16_torch(seed, shape, device="cuda"):
    """N(0, 1) draws rounded to f16 from a seeded torch generator on ``device`` (used for
    benchmark-only buffers too large to draw quickly on the host)."""
    import torch
    g = torch.Generator(device=device)
    s = np.random.SeedSequence(list(seed) if isinstance(seed, (tuple, list)) else [seed])
    g.manual_seed(int(s.generate_state(1, dtype=np.uint64)[0] >> 1))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).half()


def q8_0_planes(rng: np.random.Generator, n_cells: int, n_head_kv: int, head_dim: int):
    """Q8_0 SoA planes: int8 values uniform in [-127, 127], f16 scales ~U(0.001, 0.02)."""
    assert head_dim % 32 == 0
    qs = rng.integers(-127, 128, size=(n_cells, n_head_kv, head_dim), dtype=np.int8)
    d = rng.uniform(0.001, 0.02, size=(n_cells, n_head_kv, head_dim // 32)).astype(np.float16)
    return qs, d


def q4_0_planes(rng: np.random.Generator, n_cells: int, n_head_kv: int, head_dim: int):
    """Q4_0 SoA planes: packed bytes uniform in [0, 255] (two 4-bit values each, so every
    value 0..15 is equally likely), f16 scales ~U(0.001, 0.3) (values up to ~2.4 in
    magnitude, as for Q8_0)."""
    assert head_dim % 32 == 0
    packed = rng.integers(0, 256, size=(n_cells, n_head_kv, head_dim // 2), dtype=np.uint8)
    d = rng.uniform(0.001, 0.3, size=(n_cells, n_head_kv, head_dim // 32)).astype(np.float16)
    return packed, d


def make_q(w: Workload, layer: int = 0, seed: int | None = None) -> np.ndarray:
    s = 1000 + w.number if seed is None else seed
    return normal_f16(_rng(s, layer), (w.n_seq, w.n_head, w.head_dim))


def make_kv_f16(w: Workload, layer: int = 0, n_cells: int | None = None, seed_k=None, seed_v=None):
    """Cell-major f16 K and V, one cache of ``n_cells`` rows per sequence."""
    n = w.n_cells if n_cells is None else n_cells
    sk = 2000 + w.number if seed_k is None else seed_k
    sv = 3000 + w.number if seed_v is None else seed_v
    shape = (w.n_seq, n, w.n_head_kv, w.head_dim) if w.n_seq > 1 else (n, w.n_head_kv, w.head_dim)
    return normal_f16(_rng(sk, layer), shape), normal_f16(_rng(sv, layer), shape)


def make_kv_q8(w: Workload, layer: int = 0):
    k = q8_0_planes(_rng(2000 + w.number, layer, w.head_dim), w.n_cells, w.n_head_kv, w.head_dim)
    v = q8_0_planes(_rng(3000 + w.number, layer, w.head_dim), w.n_cells, w.n_head_kv, w.head_dim)
    return k, v


def make_kv_q4(w: Workload, layer: int = 0):
    """Q4_0 key and value planes: ((k_packed, k_d), (v_packed, v_d))."""
    k = q4_0_planes(_rng(2000 + w.number, layer, w.head_dim), w.n_cells, w.n_head_kv, w.head_dim)
    v = q4_0_planes(_rng(3000 + w.number, layer, w.head_dim), w.n_cells, w.n_head_kv, w.head_dim)
    return k, v


def make_kv_q8q4(w: Workload, layer: int = 0):
    """Q8_0 key planes and Q4_0 value planes: ((k_qs, k_d), (v_packed, v_d))."""
    k = q8_0_planes(_rng(2000 + w.number, layer, w.head_dim), w.n_cells, w.n_head_kv, w.head_dim)
    v = q4_0_planes(_rng(3000 + w.number, layer, w.head_dim), w.n_cells, w.n_head_kv, w.head_dim)
    return k, v


@dataclasses.dataclass
class UnifiedCacheLayout:
    """Which physical cells each sequence owns in a unified, record-interleaved cache."""
    pool_records: int
    records_per_seq: list          # list of int arrays of physical record ids (unsorted)
    selected: list                 # list of int64 arrays of selected physical cells (sorted)
    encoded_cells: list            # list of int64 arrays in logical (shuffled) order,
                                   # with duplicates and stage-slot tags in the high bits


def make_unified_layout(w: Workload, seed: int | None = None, dup_frac: float = 0.02,
                        min_valid: int = 1) -> UnifiedCacheLayout:
    """Scatter each sequence's records over the physical pool and punch -1 holes.

    Sequence s owns ``seq_lens[s] / 128`` records chosen without replacement from a
    shuffled pool; inside each owned record every cell is selected with probability
    ``1 - hole_prob``.  The encoded list handed to the plan builder is the selected
    cells in a random logical order, with a few duplicates and a random stage-slot tag
    in the high 32 bits.
    """
    rng = _rng(4000 + w.number if seed is None else seed)
    need = [L // RECORD_CELLS for L in w.seq_lens]
    assert all(L % RECORD_CELLS == 0 for L in w.seq_lens)
    assert sum(need) <= w.pool_records
    perm = rng.permutation(w.pool_records)
    recs, sel, enc = [], [], []
    pos = 0
    for n_rec in need:
        r = perm[pos:pos + n_rec].astype(np.int64)
        pos += n_rec
        cells = (r[:, None] * RECORD_CELLS + np.arange(RECORD_CELLS)[None, :]).reshape(-1)
        keep = rng.random(cells.shape[0]) >= w.hole_prob
        if keep.sum() < min_valid:
            keep[0] = True
        chosen = np.sort(cells[keep])
        n_dup = int(dup_frac * chosen.shape[0])
        dups = rng.choice(chosen, size=n_dup, replace=True) if n_dup and chosen.size else \
            np.empty(0, np.int64)
        logical = np.concatenate([chosen, dups])
        rng.shuffle(logical)
        tags = rng.integers(0, 4, size=logical.shape[0], dtype=np.int64)
        encoded = (tags << 32) | logical
        recs.append(r)
        sel.append(chosen)
        enc.append(encoded.astype(np.int64))
    return UnifiedCacheLayout(w.pool_records, recs, sel, enc)


def nan_fill_unselected(k: np.ndarray, v: np.ndarray, selected_union: np.ndarray) -> None:
    """Write NaN into every physical cell no sequence selected (holes, unused records)."""
    mask = np.ones(k.shape[0], dtype=bool)
    mask[selected_union] = False
    k[mask] = np.float16(np.nan)
    v[mask] = np.float16(np.nan)


def flatten_encoded(encoded_cells: list):
    """Concatenate per-sequence encoded lists into (cells int64[], offsets int64[S+1])."""
    offsets = np.zeros(len(encoded_cells) + 1, dtype=np.int64)
    for i, e in enumerate(encoded_cells):
        offsets[i + 1] = offsets[i] + e.shape[0]
    cells = np.concatenate(encoded_cells) if encoded_cells else np.empty(0, np.int64)
    return np.ascontiguousarray(cells, dtype=np.int64), offsets
