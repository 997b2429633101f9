"""Thin Python binding over the kvattn C ABI (argument marshalling only).

Every function with a ``kvattn_`` name calls the C entry point of the same name; torch
tensors are passed by ``data_ptr()``, streams by their ``cuda_stream`` handle, and a
non-OK status raises :class:`KvattnError`.  The convenience wrappers at the end
(``decode``, ``merge``, ``WindowTail``) only allocate outputs and workspaces with torch
and infer sizes from tensor shapes; all arithmetic runs in the library's kernels.

Importing this module loads ``_lib/libkvattn.so`` and raises if it has not been built
(``python -m kv_cache_decode_02_gb300._build``): there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libkvattn.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with "
                      "`python -m kv_cache_decode_02_gb300._build` (no fallback exists)")
lib = ctypes.CDLL(_LIB_PATH)

KVATTN_OK = 0
KVATTN_ERR_INVALID_ARG = -1
KVATTN_ERR_UNSUPPORTED = -2
KVATTN_ERR_WORKSPACE = -3
KVATTN_ERR_CAPACITY = -4
KVATTN_ERR_CUDA = -5
KVATTN_ERR_TIMEOUT = -6
KVATTN_KV_F16 = 0
KVATTN_KV_Q8_0 = 1
KVATTN_KV_Q8_0_Q4_0 = 2
KVATTN_KV_Q4_0 = 3
KVATTN_DEVICE_WAIT_TIMEOUT = 1
KVATTN_DEVICE_BAD_PLAN_ENTRY = 2
KVATTN_TAIL_PREFETCH = 1

EXPORTED = (
    "kvattn_status_string", "kvattn_version", "kvattn_build_cell_plan", "kvattn_build_descriptors",
    "kvattn_decode_workspace_bytes", "kvattn_decode", "kvattn_decode_partials", "kvattn_merge",
    "kvattn_tail_ctx_create",
    "kvattn_tail_ctx_destroy", "kvattn_window_tail_workspace_bytes", "kvattn_decode_window_tail",
    "kvattn_tail_wait", "kvattn_workspace_status", "kvattn_decode_noalloc",
    "kvattn_window_tail_direct_workspace_bytes", "kvattn_decode_window_tail_direct",
    "kvattn_select_split_for", "kvattn_select_split", "kvattn_decode_multi_workspace_bytes",
    "kvattn_decode_multi", "kvattn_tail_ctx_set_flags",
)

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float

lib.kvattn_status_string.argtypes = [_I]
lib.kvattn_status_string.restype = ctypes.c_char_p
lib.kvattn_version.argtypes = []
lib.kvattn_version.restype = _I
lib.kvattn_build_cell_plan.argtypes = [_P, _P, _I, _I64, _P, _I64, _P]
lib.kvattn_build_cell_plan.restype = _I
lib.kvattn_build_descriptors.argtypes = [_P, _I64, _P, _I, _I64, _I, _I64, _P, _P]
lib.kvattn_build_descriptors.restype = _I
lib.kvattn_decode_workspace_bytes.argtypes = [_I, _I, _I, _I64, _I]
lib.kvattn_decode_workspace_bytes.restype = _SZ
lib.kvattn_decode_multi_workspace_bytes.argtypes = [_I, _I, _I, _I, _I64, _I]
lib.kvattn_decode_multi_workspace_bytes.restype = _SZ
lib.kvattn_decode_multi.argtypes = [_P, _P, _P, _P, _P, _I, _I64, _P, _I64, _P, _I, _I64, _I, _I, _I, _I, _I, _F,
                                    _P, _P, _P, _SZ, _P]
lib.kvattn_decode_multi.restype = _I
lib.kvattn_select_split_for.argtypes = [_I, _I64, _I, _I64]
lib.kvattn_select_split_for.restype = _I
lib.kvattn_select_split.argtypes = [_I, _I, _I64, _I, _I]
lib.kvattn_select_split.restype = _I
lib.kvattn_decode.argtypes = [_P, _P, _P, _P, _P, _I, _I64, _P, _I64, _P, _I, _I64, _I, _I, _I, _I,
                              _F, _P, _P, _P, _SZ, _P]
lib.kvattn_decode.restype = _I
lib.kvattn_decode_partials.argtypes = lib.kvattn_decode.argtypes
lib.kvattn_decode_partials.restype = _I
lib.kvattn_decode_noalloc.argtypes = [_P, _P, _P, _P, _P, _I, _I64, _P, _I64, _P, _I, _I64, _I, _I, _I, _I,
                                      _F, _P, _P, _P]
lib.kvattn_decode_noalloc.restype = _I
KVATTN_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024
lib.kvattn_merge.argtypes = [_P, _P, _I, _I, _I, _P, _P, _P]
lib.kvattn_merge.restype = _I
lib.kvattn_tail_ctx_create.argtypes = [ctypes.POINTER(_P)]
lib.kvattn_tail_ctx_create.restype = _I
lib.kvattn_tail_ctx_destroy.argtypes = [_P]
lib.kvattn_tail_ctx_destroy.restype = _I
lib.kvattn_tail_ctx_set_flags.argtypes = [_P, ctypes.c_uint32]
lib.kvattn_tail_ctx_set_flags.restype = _I
lib.kvattn_window_tail_workspace_bytes.argtypes = [_I, _I, _I, _I64, _I64, _I, _I64, _I]
lib.kvattn_window_tail_workspace_bytes.restype = _SZ
lib.kvattn_decode_window_tail.argtypes = [_P, _P, _P, _P, _I64, _P, _P, _I64, _I64, _I, _I, _I, _I,
                                          _I, _F, _P, _P, _P, _SZ, _P, _P]
lib.kvattn_decode_window_tail.restype = _I
lib.kvattn_window_tail_direct_workspace_bytes.argtypes = [_I, _I, _I, _I64, _I64, _I, _I]
lib.kvattn_window_tail_direct_workspace_bytes.restype = _SZ
lib.kvattn_decode_window_tail_direct.argtypes = [_P, _P, _P, _I64, _P, _P, _I64, _I, _I, _I, _I, _I, _F, _P,
                                                 _P, _P, _SZ, _P]
lib.kvattn_decode_window_tail_direct.restype = _I
lib.kvattn_tail_wait.argtypes = [_P, _I]
lib.kvattn_tail_wait.restype = _I
lib.kvattn_workspace_status.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32), _I, _P]
lib.kvattn_workspace_status.restype = _I


class KvattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kvattn_status_string(status)} ({status})")


def _ptr(x):
    """Address of a torch tensor / numpy array / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, where: str) -> None:
    if rc != KVATTN_OK:
        raise KvattnError(rc, where)


# ----------------------------- same names as the C ABI -----------------------------

def kvattn_status_string(status: int) -> str:
    return lib.kvattn_status_string(status).decode()


def kvattn_version() -> int:
    return lib.kvattn_version()


def kvattn_build_cell_plan(cells, offsets, n_seq, capacity_cells, plan, plan_stride, seq_lens):
    """Host arrays (numpy int64 / int32).  ``plan`` may be None to only size the rows."""
    rc = lib.kvattn_build_cell_plan(_ptr(cells), _ptr(offsets), n_seq, capacity_cells, _ptr(plan),
                                    plan_stride, _ptr(seq_lens))
    _check(rc, "kvattn_build_cell_plan")


def kvattn_build_descriptors(cell_plan, plan_stride, seq_lens, n_seq, max_len, split, n_cells, desc,
                             stream=None):
    rc = lib.kvattn_build_descriptors(_ptr(cell_plan), plan_stride, _ptr(seq_lens), n_seq, max_len,
                                      split, n_cells, _ptr(desc), _stream(stream))
    _check(rc, "kvattn_build_descriptors")


def kvattn_decode_workspace_bytes(n_seq, n_head, head_dim, max_len, split) -> int:
    return lib.kvattn_decode_workspace_bytes(n_seq, n_head, head_dim, max_len, split)


def kvattn_decode_multi_workspace_bytes(n_seq, n_q, n_head, head_dim, max_len, split) -> int:
    return lib.kvattn_decode_multi_workspace_bytes(n_seq, n_q, n_head, head_dim, max_len, split)


def kvattn_decode_multi(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan, plan_stride, seq_lens,
                        n_seq, max_len, n_q, n_head, n_head_kv, head_dim, split, scale, out, lse, ws, ws_bytes,
                        stream=None):
    rc = lib.kvattn_decode_multi(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales), kv_type,
                                 n_cells, _ptr(cell_plan), plan_stride, _ptr(seq_lens), n_seq, max_len, n_q, n_head,
                                 n_head_kv, head_dim, split, scale, _ptr(out), _ptr(lse), _ptr(ws), ws_bytes,
                                 _stream(stream))
    _check(rc, "kvattn_decode_multi")


def kvattn_select_split_for(n_seq, max_len, n_head_kv, resident_ctas) -> int:
    rc = lib.kvattn_select_split_for(n_seq, max_len, n_head_kv, resident_ctas)
    if rc < 0:
        raise KvattnError(rc, "kvattn_select_split_for")
    return rc


def kvattn_select_split(kv_type, n_seq, max_len, n_head_kv, head_dim) -> int:
    rc = lib.kvattn_select_split(kv_type, n_seq, max_len, n_head_kv, head_dim)
    if rc < 0:
        raise KvattnError(rc, "kvattn_select_split")
    return rc


def kvattn_decode(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan, plan_stride,
                  seq_lens, n_seq, max_len, n_head, n_head_kv, head_dim, split, scale, out, lse, ws,
                  ws_bytes, stream=None):
    rc = lib.kvattn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
                           kv_type, n_cells, _ptr(cell_plan), plan_stride, _ptr(seq_lens), n_seq,
                           max_len, n_head, n_head_kv, head_dim, split, scale, _ptr(out), _ptr(lse),
                           _ptr(ws), ws_bytes, _stream(stream))
    _check(rc, "kvattn_decode")


def kvattn_decode_partials(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan,
                           plan_stride, seq_lens, n_seq, max_len, n_head, n_head_kv, head_dim, split,
                           scale, part_o, part_lse, ws, ws_bytes, stream=None):
    rc = lib.kvattn_decode_partials(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales),
                                    _ptr(v_scales), kv_type, n_cells, _ptr(cell_plan), plan_stride,
                                    _ptr(seq_lens), n_seq, max_len, n_head, n_head_kv, head_dim, split,
                                    scale, _ptr(part_o), _ptr(part_lse), _ptr(ws), ws_bytes,
                                    _stream(stream))
    _check(rc, "kvattn_decode_partials")


def kvattn_decode_noalloc(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan,
                          plan_stride, seq_lens, n_seq, max_len, n_head, n_head_kv, head_dim, split, scale,
                          out, lse, stream=None):
    """kvattn_decode without a workspace, for callers that cannot allocate device memory:
    the library keeps the scratch in its own fixed-size device array (see kvattn.h)."""
    rc = lib.kvattn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales),
                                   _ptr(v_scales), kv_type, n_cells, _ptr(cell_plan), plan_stride,
                                   _ptr(seq_lens), n_seq, max_len, n_head, n_head_kv, head_dim, split,
                                   scale, _ptr(out), _ptr(lse), _stream(stream))
    _check(rc, "kvattn_decode_noalloc")


def kvattn_merge(partials, lses, n_parts, n_rows, head_dim, out, lse, stream=None):
    rc = lib.kvattn_merge(_ptr(partials), _ptr(lses), n_parts, n_rows, head_dim, _ptr(out),
                          _ptr(lse), _stream(stream))
    _check(rc, "kvattn_merge")


def kvattn_tail_ctx_create() -> int:
    h = _P()
    _check(lib.kvattn_tail_ctx_create(ctypes.byref(h)), "kvattn_tail_ctx_create")
    return h.value


def kvattn_tail_ctx_destroy(ctx: int) -> None:
    _check(lib.kvattn_tail_ctx_destroy(ctx), "kvattn_tail_ctx_destroy")


def kvattn_tail_ctx_set_flags(ctx: int, flags: int) -> None:
    _check(lib.kvattn_tail_ctx_set_flags(ctx, flags), "kvattn_tail_ctx_set_flags")


def kvattn_window_tail_workspace_bytes(n_head, n_head_kv, head_dim, n_win, n_tail, split, tile_cells,
                                       tail_split) -> int:
    return lib.kvattn_window_tail_workspace_bytes(n_head, n_head_kv, head_dim, n_win, n_tail, split,
                                                  tile_cells, tail_split)


def kvattn_decode_window_tail(ctx, q, k_win, v_win, n_win, k_tail_host, v_tail_host, n_tail,
                              tile_cells, n_head, n_head_kv, head_dim, split, tail_split, scale,
                              out, lse, ws, ws_bytes, compute_stream=None, copy_stream=None):
    rc = lib.kvattn_decode_window_tail(ctx, _ptr(q), _ptr(k_win), _ptr(v_win), n_win,
                                       _ptr(k_tail_host), _ptr(v_tail_host), n_tail, tile_cells,
                                       n_head, n_head_kv, head_dim, split, tail_split, scale,
                                       _ptr(out), _ptr(lse), _ptr(ws), ws_bytes,
                                       _stream(compute_stream), _stream(copy_stream))
    _check(rc, "kvattn_decode_window_tail")


def kvattn_window_tail_direct_workspace_bytes(n_head, n_head_kv, head_dim, n_win, n_tail, split,
                                              tail_split) -> int:
    return lib.kvattn_window_tail_direct_workspace_bytes(n_head, n_head_kv, head_dim, n_win, n_tail, split,
                                                         tail_split)


def kvattn_decode_window_tail_direct(q, k_win, v_win, n_win, k_tail_host, v_tail_host, n_tail, n_head,
                                     n_head_kv, head_dim, split, tail_split, scale, out, lse, ws, ws_bytes,
                                     stream=None):
    rc = lib.kvattn_decode_window_tail_direct(_ptr(q), _ptr(k_win), _ptr(v_win), n_win, _ptr(k_tail_host),
                                              _ptr(v_tail_host), n_tail, n_head, n_head_kv, head_dim, split,
                                              tail_split, scale, _ptr(out), _ptr(lse), _ptr(ws), ws_bytes,
                                              _stream(stream))
    _check(rc, "kvattn_decode_window_tail_direct")


def window_tail_direct(q, k_win, v_win, k_tail_host, v_tail_host, *, split, tail_split, scale=None,
                       out=None, lse=None, ws=None, stream=None):
    """Window in HBM + tail read in place from pinned host memory.  q: half [H][D]."""
    import torch
    H, D = q.shape[-2], q.shape[-1]
    Hk = k_win.shape[-2] if k_win is not None else k_tail_host.shape[-2]
    n_win = k_win.shape[0] if k_win is not None else 0
    n_tail = k_tail_host.shape[0] if k_tail_host is not None else 0
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((H, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((H,), dtype=torch.float32, device=q.device)
    if ws is None:
        nbytes = kvattn_window_tail_direct_workspace_bytes(H, Hk, D, n_win, n_tail, split, tail_split)
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    kvattn_decode_window_tail_direct(q, k_win, v_win, n_win, k_tail_host, v_tail_host, n_tail, H, Hk, D, split,
                                     tail_split, scale, out, lse, ws, ws.numel(), stream)
    return out, lse


def kvattn_tail_wait(ctx: int, timeout_ms: int) -> None:
    _check(lib.kvattn_tail_wait(ctx, timeout_ms), "kvattn_tail_wait")


def kvattn_workspace_status(ws, clear: bool = False, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check(lib.kvattn_workspace_status(_ptr(ws), ctypes.byref(flags), int(clear), _stream(stream)),
           "kvattn_workspace_status")
    return flags.value


# ----------------------------- torch conveniences -----------------------------

def decode_workspace(n_seq, n_head, head_dim, max_len, split, device="cuda"):
    import torch
    nbytes = kvattn_decode_workspace_bytes(n_seq, n_head, head_dim, max_len, split)
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


def decode(q, k_cache, v_cache, seq_lens, *, split, max_len=None, cell_plan=None, k_scales=None,
           v_scales=None, scale=None, n_cells=None, out=None, lse=None, ws=None, stream=None, kv_type=None):
    """q: half [S][H][D] (cuda); K/V as the C ABI describes; seq_lens int32 [S] (cuda).

    ``kv_type`` defaults to f16 without scales, to Q4_0 when K's rows hold head_dim / 2 bytes,
    to Q8_0_Q4_0 when only V's do, and to Q8_0 otherwise.  ``n_cells`` defaults to K's cell dimension (dim 0 for a
    unified cache or a single sequence, dim 1 for a per-sequence [S][N][Hk][D] cache).
    Returns (out, lse).
    """
    import torch
    S, H, D = q.shape
    if kv_type is None:
        if k_scales is None:
            kv_type = KVATTN_KV_F16
        else:
            if k_cache.shape[-1] * 2 == D:
                kv_type = KVATTN_KV_Q4_0
            else:
                kv_type = KVATTN_KV_Q8_0_Q4_0 if v_cache.shape[-1] * 2 == D else KVATTN_KV_Q8_0
    Hk = k_cache.shape[-2]
    if n_cells is None:
        n_cells = k_cache.shape[1] if (k_cache.dim() == 4) else k_cache.shape[0]
    plan_stride = 0
    if cell_plan is not None:
        plan_stride = cell_plan.shape[-1]
    if max_len is None:
        max_len = plan_stride if cell_plan is not None else n_cells
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((S, H, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((S, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = decode_workspace(S, H, D, max_len, split, device=q.device)
    kvattn_decode(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan, plan_stride,
                  seq_lens, S, max_len, H, Hk, D, split, scale, out, lse, ws, ws.numel(), stream)
    return out, lse


def decode_multi(q, k_cache, v_cache, seq_lens, *, split, max_len=None, cell_plan=None, scale=None, n_cells=None,
                 out=None, lse=None, ws=None, stream=None, k_scales=None, v_scales=None):
    """q: half [S][n_q][H][D] (cuda); f16 K/V, or a quantised cache with k_scales / v_scales
    (the type inferred from the row widths as in decode), as the C ABI describes.  Returns
    (out, lse)."""
    import torch
    S, n_q, H, D = q.shape
    Hk = k_cache.shape[-2]
    if n_cells is None:
        n_cells = k_cache.shape[1] if (k_cache.dim() == 4) else k_cache.shape[0]
    plan_stride = cell_plan.shape[-1] if cell_plan is not None else 0
    if max_len is None:
        max_len = plan_stride if cell_plan is not None else n_cells
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((S, n_q, H, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((S, n_q, H), dtype=torch.float32, device=q.device)
    if ws is None:
        nbytes = kvattn_decode_multi_workspace_bytes(S, n_q, H, D, max_len, split)
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    if k_scales is None:
        kv_type = KVATTN_KV_F16
    elif k_cache.shape[-1] * 2 == D:
        kv_type = KVATTN_KV_Q4_0
    else:
        kv_type = KVATTN_KV_Q8_0_Q4_0 if v_cache.shape[-1] * 2 == D else KVATTN_KV_Q8_0
    kvattn_decode_multi(q, k_cache, v_cache, k_scales, v_scales, kv_type, n_cells, cell_plan, plan_stride, seq_lens,
                        S, max_len, n_q, H, Hk, D, split, scale, out, lse, ws, ws.numel(), stream)
    return out, lse


def merge(partials, lses, out=None, lse=None, stream=None):
    """partials float [P][R][D], lses float [P][R] (cuda) -> (out [R][D], lse [R])."""
    import torch
    P, R, D = partials.shape
    if out is None:
        out = torch.empty((R, D), dtype=torch.float32, device=partials.device)
    if lse is None:
        lse = torch.empty((R,), dtype=torch.float32, device=partials.device)
    kvattn_merge(partials, lses, P, R, D, out, lse, stream)
    return out, lse


def build_cell_plan(encoded_per_seq, capacity_cells, plan_stride=None):
    """Host helper: list of int64 arrays -> (plan int32 [S][stride], seq_lens int32 [S])."""
    n_seq = len(encoded_per_seq)
    offsets = np.zeros(n_seq + 1, dtype=np.int64)
    for i, e in enumerate(encoded_per_seq):
        offsets[i + 1] = offsets[i] + len(e)
    cells = (np.concatenate([np.asarray(e, dtype=np.int64) for e in encoded_per_seq])
             if n_seq and offsets[-1] else np.zeros(1, dtype=np.int64))
    lens = np.zeros(max(n_seq, 1), dtype=np.int32)
    if plan_stride is None:
        kvattn_build_cell_plan(cells, offsets, n_seq, capacity_cells, None, 0, lens)
        plan_stride = int(lens[:n_seq].max(initial=0))
    plan = np.full((max(n_seq, 1), max(plan_stride, 1)), -1, dtype=np.int32)
    kvattn_build_cell_plan(cells, offsets, n_seq, capacity_cells, plan, plan_stride, lens)
    return plan[:n_seq, :plan_stride], lens[:n_seq]


class WindowTail:
    """Owns a tail context (events only) and runs kvattn_decode_window_tail.

    ``prefetch=True`` sets KVATTN_TAIL_PREFETCH: one context serves every layer of a model,
    and a layer's tail copies wait only for the decode that last read their staging slot,
    not for the layers before it."""

    def __init__(self, prefetch=False):
        self.ctx = kvattn_tail_ctx_create()
        if prefetch:
            kvattn_tail_ctx_set_flags(self.ctx, KVATTN_TAIL_PREFETCH)

    def close(self):
        if self.ctx:
            kvattn_tail_ctx_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def workspace(n_head, n_head_kv, head_dim, n_win, n_tail, split, tile_cells, tail_split,
                  device="cuda"):
        import torch
        nbytes = kvattn_window_tail_workspace_bytes(n_head, n_head_kv, head_dim, n_win, n_tail,
                                                    split, tile_cells, tail_split)
        if nbytes == 0:
            raise KvattnError(KVATTN_ERR_INVALID_ARG, "kvattn_window_tail_workspace_bytes")
        return torch.zeros(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, q, k_win, v_win, k_tail_host, v_tail_host, *, split, tile_cells, tail_split,
                 scale=None, out=None, lse=None, ws=None, compute_stream=None, copy_stream=None):
        import torch
        H, D = q.shape[-2], q.shape[-1]
        Hk = k_win.shape[-2] if k_win is not None else k_tail_host.shape[-2]
        n_win = k_win.shape[0] if k_win is not None else 0
        n_tail = k_tail_host.shape[0] if k_tail_host is not None else 0
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        if out is None:
            out = torch.empty((H, D), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((H,), dtype=torch.float32, device=q.device)
        if ws is None:
            ws = self.workspace(H, Hk, D, n_win, n_tail, split, tile_cells, tail_split, q.device)
        kvattn_decode_window_tail(self.ctx, q, k_win, v_win, n_win, k_tail_host, v_tail_host, n_tail,
                                  tile_cells, H, Hk, D, split, tail_split, scale, out, lse, ws,
                                  ws.numel(), compute_stream, copy_stream)
        return out, lse
