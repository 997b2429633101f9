"""Independent Python builder of the compact cell plan and its per-split descriptors.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Written with sets and sorting,
sharing nothing with the library's C++ builder, so that the two can be compared bit
for bit.

Compact cell plan ("KVARN KV Performance optimizations", items 3 and 4):
* every requested cell is an encoded 64-bit index whose low 32 bits (unsigned) are the
  physical cell and whose high bits carry stage-slot metadata the read plan ignores
  (item 5: low-32-bit physical-cell extraction, stage slot preserved elsewhere);
* duplicates are dropped (first occurrence wins; the plan is positional, so which
  copy survives does not change it) and a cell at or beyond the cache capacity is an
  error (item 3: capacity checks);
* selected cells are grouped by their physical 128-cell record, the records are
  sorted by physical id, and each selected record gets one complete, monotonic
  128-entry segment whose entry j is ``record*128 + j`` when that cell was selected and
  -1 (a hole) otherwise (item 4);
* the sequence's length is 128 x its record count; the row is padded with -1.

Descriptors (item 5, "descriptor setup"): for each sequence s and split p covering plan
entries [p*split, min((p+1)*split, L_s)) with L_s = min(seq_len[s], max_len, plan_stride):
``[n_valid, lo, hi, flags]`` where an entry is valid when 0 <= e < n_cells_phys, lo/hi
are the smallest/largest valid physical cell (-1 when none), and flags has
bit 0 = no valid entry (the split is skipped), bit 1 = linear (every valid entry
satisfies e - i = constant, i.e. the split reads one physical run with positional
holes), bit 2 = an entry outside [-1, n_cells_phys) was seen (treated as masked),
bit 3 = the split starts at or beyond L_s.
"""
from __future__ import annotations

import numpy as np

RECORD = 128

FLAG_EMPTY = 1
FLAG_LINEAR = 2
FLAG_BAD = 4
FLAG_BEYOND = 8


class CapacityError(ValueError):
    pass


def physical_cell(encoded: int) -> int:
    return int(encoded) & 0xFFFFFFFF


def plan_rows(encoded_per_seq, capacity: int):
    """List of per-sequence plan rows (Python lists of ints, no padding)."""
    rows = []
    for seq in encoded_per_seq:
        selected = set()
        for e in seq:
            c = physical_cell(e)
            if c >= capacity:
                raise CapacityError(f"cell {c} >= capacity {capacity}")
            selected.add(c)  # a set keeps one copy of each cell
        row = []
        for r in sorted({c // RECORD for c in selected}):
            row.extend(r * RECORD + j if (r * RECORD + j) in selected else -1 for j in range(RECORD))
        rows.append(row)
    return rows


def build_cell_plan(encoded_per_seq, capacity: int, plan_stride: int | None = None):
    """Returns (plan int32 [S][plan_stride], seq_lens int32 [S])."""
    rows = plan_rows(encoded_per_seq, capacity)
    lens = np.array([len(r) for r in rows], dtype=np.int32)
    stride = int(lens.max(initial=0)) if plan_stride is None else plan_stride
    if lens.size and lens.max() > stride:
        raise CapacityError("plan row longer than plan_stride")
    plan = np.full((len(rows), stride), -1, dtype=np.int32)
    for s, r in enumerate(rows):
        plan[s, :len(r)] = r
    return plan, lens


def descriptors(plan, seq_lens, max_len: int, split: int, n_cells_phys: int):
    """Per-split descriptors, int32 [S][ceil(max_len/split)][4]."""
    plan = np.asarray(plan)
    S, stride = plan.shape
    n_split = -(-max_len // split) if max_len > 0 else 0
    out = np.zeros((S, n_split, 4), dtype=np.int32)
    for s in range(S):
        L = max(0, min(int(seq_lens[s]), max_len, stride))
        for p in range(n_split):
            i0 = p * split
            i1 = min(i0 + split, L)
            n_valid, lo, hi, bad = 0, -1, -1, False
            offsets = set()
            for i in range(i0, i1):
                e = int(plan[s, i])
                if 0 <= e < n_cells_phys:
                    n_valid += 1
                    lo = e if lo < 0 else min(lo, e)
                    hi = max(hi, e)
                    offsets.add(e - i)
                elif e != -1:
                    bad = True
            flags = 0
            if n_valid == 0:
                flags |= FLAG_EMPTY
            elif len(offsets) == 1:
                flags |= FLAG_LINEAR
            if bad:
                flags |= FLAG_BAD
            if i0 >= L:
                flags |= FLAG_BEYOND
            out[s, p] = (n_valid, lo, hi, flags)
    return out
