"""Pure-Python brute force of single-query decode attention -- TEST INFRASTRUCTURE ONLY.

For tiny inputs only (a handful of cells and dims).  Works on nested Python lists
of floats and uses ``math.fsum`` for every sum, so it has no dependence on numpy or
on the C oracle.  Definition as in the C oracle's header: scores x_c = scale * q.K_c,
O = sum softmax(x)_c V_c, LSE = ln sum exp(x_c).
"""
from __future__ import annotations

import math


def attend(q, keys, values, scale):
    """q: [D]; keys, values: [n][D] (n may be 0).  Returns (out [D], lse)."""
    D = len(q)
    if not keys:
        return [0.0] * D, -math.inf
    x = [scale * math.fsum(q[d] * k[d] for d in range(D)) for k in keys]
    m = max(x)
    w = [math.exp(xi - m) for xi in x]
    l = math.fsum(w)
    out = [math.fsum(w[j] * values[j][d] for j in range(len(keys))) / l for d in range(D)]
    return out, m + math.log(l)


def decode(q, k, v, seq_lens, plan=None, scale=None, n_head_kv=None):
    """q: [S][H][D]; k, v: [S][N][Hk][D] (contiguous) or [Nphys][Hk][D] (with plan)."""
    S, H, D = len(q), len(q[0]), len(q[0][0])
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    Hk = n_head_kv if n_head_kv is not None else (len(k[0][0]) if plan is None else len(k[0]))
    G = H // Hk
    outs, lses = [], []
    for s in range(S):
        if plan is None:
            cells = [(s, i) for i in range(seq_lens[s])]
            get = lambda arr, c, g: arr[c[0]][c[1]][g]
        else:
            cells = [plan[s][i] for i in range(seq_lens[s]) if plan[s][i] != -1]
            get = lambda arr, c, g: arr[c][g]
        o_s, l_s = [], []
        for h in range(H):
            g = h // G
            keys = [list(map(float, get(k, c, g))) for c in cells]
            vals = [list(map(float, get(v, c, g))) for c in cells]
            o, l = attend([float(x) for x in q[s][h]], keys, vals, scale)
            o_s.append(o)
            l_s.append(l)
        outs.append(o_s)
        lses.append(l_s)
    return outs, lses


def decode_multi(q, k, v, seq_lens, plan=None, scale=None, n_head_kv=None):
    """Causal multi-query decode, written out directly.  q: [S][n_q][H][D]; k, v as in
    decode().  Query token t of sequence s sits at logical position p = L - n_q + t and
    sees the entries at positions 0..p (inside the length, not -1)."""
    S, n_q, H, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    Hk = n_head_kv if n_head_kv is not None else (len(k[0][0]) if plan is None else len(k[0]))
    G = H // Hk
    outs, lses = [], []
    for s in range(S):
        L = seq_lens[s]
        o_s, l_s = [], []
        for t in range(n_q):
            p = L - n_q + t
            o_t, l_t = [], []
            for h in range(H):
                g = h // G
                keys, vals = [], []
                for i in range(L):
                    if i > p:
                        continue
                    if plan is None:
                        kc, vc = k[s][i][g], v[s][i][g]
                    else:
                        if plan[s][i] == -1:
                            continue
                        kc, vc = k[plan[s][i]][g], v[plan[s][i]][g]
                    keys.append([float(x) for x in kc])
                    vals.append([float(x) for x in vc])
                o, l = attend([float(x) for x in q[s][t][h]], keys, vals, scale)
                o_t.append(o)
                l_t.append(l)
            o_s.append(o_t)
            l_s.append(l_t)
        outs.append(o_s)
        lses.append(l_s)
    return outs, lses
