"""CPU oracle for decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The library never does: it shares no code with the CUDA
path, and the CUDA path fails loudly when its own extension is missing instead of
falling back to anything here.

Contents
* ``attn_oracle.c`` -- the fp64 attention definition and the LSE merge (plain C,
  OpenMP over independent (sequence, head) rows), loaded through ctypes.
* ``brute.py``      -- a pure-Python brute force for tiny inputs.
* ``plan_oracle.py``-- an independent Python builder of the compact cell plan and of
  the per-split descriptors.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c with gcc (OpenMP) into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if force or not fresh:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            common = [i64, i64, P, i64, P, i32, i32, i32, i32, dbl, P, P, i32]
            lib.oracle_decode_f16.argtypes = [P, P, P] + common
            lib.oracle_decode_q8_0.argtypes = [P, P, P, P, P] + common
            lib.oracle_decode_f64.argtypes = [P, P, P] + common
            lib.oracle_decode_q8_0_q4_0.argtypes = [P, P, P, P, P] + common
            lib.oracle_decode_q4_0.argtypes = [P, P, P, P, P] + common
            for f in (lib.oracle_decode_f16, lib.oracle_decode_q8_0, lib.oracle_decode_f64,
                      lib.oracle_decode_q8_0_q4_0, lib.oracle_decode_q4_0):
                f.restype = ctypes.c_int
            lib.oracle_merge.argtypes = [P, P, i32, i32, i32, P, P]
            lib.oracle_merge.restype = ctypes.c_int
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _geometry(k_shape, n_seq, plan):
    """(n_cells_phys, per_seq_cells) from the cache shape."""
    if plan is not None:
        return k_shape[0], 0
    if len(k_shape) == 4:
        assert k_shape[0] == n_seq
        return k_shape[0] * k_shape[1], k_shape[1]
    assert n_seq == 1, "a 3-D cache holds one sequence; pass [S][N][Hk][D] for several"
    return k_shape[0], k_shape[0]


def _common(q, k_shape, seq_lens, plan, scale, n_threads):
    S, H, D = q.shape
    Hk = k_shape[-2]
    assert k_shape[-1] == D
    n_phys, per_seq = _geometry(k_shape, S, plan)
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int64).reshape(S))
    plan_arr, stride = None, 0
    if plan is not None:
        plan_arr = np.ascontiguousarray(np.asarray(plan, dtype=np.int32).reshape(S, -1))
        stride = plan_arr.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((S, H, D), dtype=np.float64)
    lse = np.zeros((S, H), dtype=np.float64)
    nt = default_threads() if n_threads is None else n_threads
    args = [n_phys, per_seq, _ptr(plan_arr), stride, _ptr(lens), S, H, Hk, D, float(scale),
            _ptr(out), _ptr(lse), nt]
    return args, out, lse, (lens, plan_arr)


def decode_f16(q, k, v, seq_lens, plan=None, scale=None, n_threads=None):
    """fp64 decode attention over f16 inputs.  Returns (out [S][H][D], lse [S][H])."""
    q = np.ascontiguousarray(q, dtype=np.float16)
    k = np.ascontiguousarray(k, dtype=np.float16)
    v = np.ascontiguousarray(v, dtype=np.float16)
    assert k.shape == v.shape
    args, out, lse, keep = _common(q, k.shape, seq_lens, plan, scale, n_threads)
    rc = _load().oracle_decode_f16(_ptr(q), _ptr(k), _ptr(v), *args)
    if rc != 0:
        raise ValueError("oracle_decode_f16 rejected its arguments")
    return out, lse


def decode_q8_0(q, k_qs, k_d, v_qs, v_d, seq_lens, plan=None, scale=None, n_threads=None):
    """fp64 decode attention over Q8_0 (int8 values, f16 per-32 scales)."""
    q = np.ascontiguousarray(q, dtype=np.float16)
    k_qs = np.ascontiguousarray(k_qs, dtype=np.int8)
    v_qs = np.ascontiguousarray(v_qs, dtype=np.int8)
    k_d = np.ascontiguousarray(k_d, dtype=np.float16)
    v_d = np.ascontiguousarray(v_d, dtype=np.float16)
    args, out, lse, keep = _common(q, k_qs.shape, seq_lens, plan, scale, n_threads)
    rc = _load().oracle_decode_q8_0(_ptr(q), _ptr(k_qs), _ptr(k_d), _ptr(v_qs), _ptr(v_d), *args)
    if rc != 0:
        raise ValueError("oracle_decode_q8_0 rejected its arguments")
    return out, lse


def decode_q8_0_q4_0(q, k_qs, k_d, v_q4, v_d, seq_lens, plan=None, scale=None, n_threads=None):
    """fp64 decode attention over Q8_0 keys and Q4_0 values.  v_q4: uint8 [cells][Hk][D/2]
    (block b of a row = bytes 16b..16b+15; byte j: element j low nibble, j+16 high), v_d:
    f16 [cells][Hk][D/32]; element value d * (nibble - 8)."""
    q = np.ascontiguousarray(q, dtype=np.float16)
    k_qs = np.ascontiguousarray(k_qs, dtype=np.int8)
    v_q4 = np.ascontiguousarray(v_q4, dtype=np.uint8)
    k_d = np.ascontiguousarray(k_d, dtype=np.float16)
    v_d = np.ascontiguousarray(v_d, dtype=np.float16)
    assert v_q4.shape[:-1] == k_qs.shape[:-1] and 2 * v_q4.shape[-1] == k_qs.shape[-1]
    args, out, lse, keep = _common(q, k_qs.shape, seq_lens, plan, scale, n_threads)
    rc = _load().oracle_decode_q8_0_q4_0(_ptr(q), _ptr(k_qs), _ptr(k_d), _ptr(v_q4), _ptr(v_d), *args)
    if rc != 0:
        raise ValueError("oracle_decode_q8_0_q4_0 rejected its arguments")
    return out, lse


def decode_q4_0(q, k_q4, k_d, v_q4, v_d, seq_lens, plan=None, scale=None, n_threads=None):
    """fp64 decode attention over Q4_0 keys and values (layout as decode_q8_0_q4_0's V)."""
    q = np.ascontiguousarray(q, dtype=np.float16)
    k_q4 = np.ascontiguousarray(k_q4, dtype=np.uint8)
    v_q4 = np.ascontiguousarray(v_q4, dtype=np.uint8)
    k_d = np.ascontiguousarray(k_d, dtype=np.float16)
    v_d = np.ascontiguousarray(v_d, dtype=np.float16)
    assert k_q4.shape == v_q4.shape
    shape = k_q4.shape[:-1] + (2 * k_q4.shape[-1],)
    args, out, lse, keep = _common(q, shape, seq_lens, plan, scale, n_threads)
    rc = _load().oracle_decode_q4_0(_ptr(q), _ptr(k_q4), _ptr(k_d), _ptr(v_q4), _ptr(v_d), *args)
    if rc != 0:
        raise ValueError("oracle_decode_q4_0 rejected its arguments")
    return out, lse


def decode_f64(q, k, v, seq_lens, plan=None, scale=None, n_threads=None):
    """fp64 decode attention over fp64 inputs (no storage-format front end)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    args, out, lse, keep = _common(q, k.shape, seq_lens, plan, scale, n_threads)
    rc = _load().oracle_decode_f64(_ptr(q), _ptr(k), _ptr(v), *args)
    if rc != 0:
        raise ValueError("oracle_decode_f64 rejected its arguments")
    return out, lse


def decode_multi(decode_one, q, seq_lens, *cache, plan=None, scale=None, n_threads=None):
    """Multi-query decode: n_q new tokens per sequence, each attending causally.

    ``q`` is [S][n_q][H][D].  ``seq_lens[s]`` counts the sequence's cells including the n_q
    new tokens' own (already appended) cells, so token t sits at logical position
    L - n_q + t and attends to positions 0 .. L - n_q + t: exactly single-query decode of
    the first L - n_q + 1 + t positions (fewer than one: no cell, O = 0, LSE = -inf).
    ``decode_one`` is decode_f16 or decode_q8_0 and ``cache`` its cache arguments.
    Returns (out [S][n_q][H][D], lse [S][n_q][H])."""
    q = np.asarray(q)
    S, n_q, H, D = q.shape
    lens = np.asarray(seq_lens, dtype=np.int64).reshape(S)
    out = np.zeros((S, n_q, H, D), dtype=np.float64)
    lse = np.zeros((S, n_q, H), dtype=np.float64)
    for t in range(n_q):
        lens_t = np.maximum(lens - n_q + 1 + t, 0)
        o, l = decode_one(np.ascontiguousarray(q[:, t]), *cache, lens_t.tolist(), plan=plan, scale=scale,
                          n_threads=n_threads)
        out[:, t] = o
        lse[:, t] = l
    return out, lse


def merge(parts, lses):
    """LSE-weighted merge.  parts [P][R][D], lses [P][R] -> (out [R][D], lse [R])."""
    parts = np.ascontiguousarray(parts, dtype=np.float64)
    lses = np.ascontiguousarray(lses, dtype=np.float64)
    P, R, D = parts.shape
    assert lses.shape == (P, R)
    out = np.zeros((R, D), dtype=np.float64)
    lse = np.zeros(R, dtype=np.float64)
    rc = _load().oracle_merge(_ptr(parts), _ptr(lses), P, R, D, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_merge rejected its arguments")
    return out, lse


def f16_to_f64(bits: int) -> float:
    return _load().oracle_f16_to_f64(bits)


def dequant_q4_0(packed, d):
    """Explicit fp64 dequantisation of Q4_0 planes (used only to pin the oracle): packed
    uint8 [..., D/2], d f16 [..., D/32] -> float64 [..., D]."""
    packed = np.asarray(packed, dtype=np.uint8)
    d = np.asarray(d).astype(np.float64)
    blocks = packed.reshape(packed.shape[:-1] + (-1, 16))
    lo = (blocks & 0x0F).astype(np.float64) - 8.0    # elements 0..15 of each block
    hi = (blocks >> 4).astype(np.float64) - 8.0      # elements 16..31
    vals = np.concatenate([lo, hi], axis=-1)         # [..., D/32, 32]
    return (vals * d[..., None]).reshape(packed.shape[:-1] + (2 * packed.shape[-1],))


def dequant_q8_0(qs, d):
    """Explicit fp64 dequantisation value = d * qs (used only to pin the oracle)."""
    qs = np.asarray(qs)
    d = np.asarray(d).astype(np.float64)
    return np.repeat(d, 32, axis=-1) * qs.astype(np.float64)
