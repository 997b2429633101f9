"""The C-ABI library loads, exports what include/kvattn.h declares, and rejects bad
arguments on the host before touching CUDA (so these run without a GPU)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Fake, suitably aligned device addresses: validation must fail before any dereference.
A = 0x7f0000000000
B = 0x7f0000100000
C = 0x7f0000200000


def declared_symbols():
    with open(os.path.join(ROOT, "include", "kvattn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvattn_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(kvattn):
    names = declared_symbols()
    assert len(names) >= 13
    for n in names:
        assert hasattr(kvattn.lib, n), n
    assert sorted(kvattn.EXPORTED) == names


def test_status_strings_and_version(kvattn):
    for code, name in [(0, "KVATTN_OK"), (-1, "KVATTN_ERR_INVALID_ARG"), (-2, "KVATTN_ERR_UNSUPPORTED"),
                       (-3, "KVATTN_ERR_WORKSPACE"), (-4, "KVATTN_ERR_CAPACITY"), (-5, "KVATTN_ERR_CUDA"),
                       (-6, "KVATTN_ERR_TIMEOUT")]:
        assert kvattn.kvattn_status_string(code) == name
    assert kvattn.kvattn_status_string(-99) == "KVATTN_ERR_UNKNOWN"
    assert kvattn.kvattn_version() >> 16 == 1


def decode_args(**over):
    a = dict(q=A, k=B, v=C, ks=None, vs=None, kv_type=0, n_cells=1024, plan=None, plan_stride=0,
             seq_lens=A + 4096, n_seq=1, max_len=1024, n_head=32, n_head_kv=8, head_dim=128, split=256,
             scale=0.0884, out=A + 8192, lse=A + 16384, ws=A + 65536, ws_bytes=1 << 30, stream=None)
    a.update(over)
    return a


def call_decode(kvattn, a):
    return kvattn.lib.kvattn_decode(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["kv_type"], a["n_cells"],
                                    a["plan"], a["plan_stride"], a["seq_lens"], a["n_seq"], a["max_len"],
                                    a["n_head"], a["n_head_kv"], a["head_dim"], a["split"], a["scale"],
                                    a["out"], a["lse"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,want", [
    (dict(n_head=30), -1),                 # n_head % n_head_kv
    (dict(n_head=72, n_head_kv=8), -2),    # G = 9 > 8
    (dict(head_dim=64), -2),
    (dict(head_dim=96), -2),
    (dict(split=48), -2),                  # not a multiple of the 32-cell tile
    (dict(n_seq=70_000_000), -2),          # (sequence, head) rows and work units beyond 32 bits
    (dict(split=-32), -1),                 # (split 0 selects the split: needs a device)
    (dict(q=None), -1),
    (dict(out=None), -1),
    (dict(ws=None), -1),
    (dict(seq_lens=None), -1),
    (dict(k=B + 8), -1),                   # K not 16-byte aligned
    (dict(out=A + 8196), -1),              # out not 16-byte aligned
    (dict(ws=A + 65536 + 128), -1),        # workspace not 256-byte aligned
    (dict(kv_type=1), -1),                 # Q8_0 without scales
    (dict(kv_type=2), -1),                 # Q8_0 K + Q4_0 V without scales
    (dict(kv_type=2, ks=A, vs=A + 4), -1),  # scale planes not 8-byte aligned
    (dict(kv_type=3), -1),                 # Q4_0 without scales
    (dict(kv_type=4, ks=A, vs=A), -1),     # no such type
    (dict(ks=A, vs=A), -1),                # f16 with scales
    (dict(kv_type=7), -1),
    (dict(n_cells=0), -1),
    (dict(max_len=-1), -1),
    (dict(n_seq=-1), -1),
    (dict(plan=A, plan_stride=0), -1),
    (dict(scale=float("nan")), -1),
    (dict(ws_bytes=1000), -3),             # workspace too small
])
def test_decode_validation(kvattn, over, want):
    assert call_decode(kvattn, decode_args(**over)) == want


def test_decode_partials_validation(kvattn):
    a = decode_args()
    f = kvattn.lib.kvattn_decode_partials
    args = [a["q"], a["k"], a["v"], None, None, 0, 1024, None, 0, a["seq_lens"], 1, 1024, 32, 8, 128, 256,
            0.0884, A + 8192, A + 1048576, a["ws"], a["ws_bytes"], None]
    bad = list(args); bad[17] = None
    assert f(*bad) == -1
    bad = list(args); bad[17] = A + 8200          # part_o not 16-byte aligned
    assert f(*bad) == -1
    bad = list(args); bad[14] = 64
    assert f(*bad) == -2
    bad = list(args); bad[20] = 100
    assert f(*bad) == -3


def test_decode_workspace_query(kvattn):
    n = kvattn.kvattn_decode_workspace_bytes(1, 32, 128, 16384, 256)
    # status word, descriptors, LSE partials and O partials of 64 splits x 32 heads
    assert n >= 64 * 32 * 128 * 4 + 64 * 32 * 4
    assert n % 256 == 0
    assert kvattn.kvattn_decode_workspace_bytes(1, 32, 128, 16384, -32) == 0
    assert call_decode(kvattn, decode_args(max_len=16384, n_cells=16384, ws_bytes=n - 1)) == -3


def test_merge_validation(kvattn):
    m = kvattn.lib.kvattn_merge
    assert m(A, B, 4, 8, 130, C, C + 8192, None) == -1       # head_dim % 4
    assert m(A, B, 4, 8, 2048, C, C + 8192, None) == -1      # head_dim > 1024
    assert m(None, B, 4, 8, 128, C, C + 8192, None) == -1
    assert m(A, B, 4, 8, 128, C + 4, C + 8192, None) == -1   # out alignment
    assert m(A, B, -1, 8, 128, C, C + 8192, None) == -1
    assert m(A, B, 4, 0, 128, C, C + 8192, None) == 0        # nothing to do


def test_descriptor_validation(kvattn):
    f = kvattn.lib.kvattn_build_descriptors
    assert f(A, 0, B, 1, 128, 128, 1024, C, None) == -1      # plan_stride
    assert f(A, 128, B, 1, 128, 0, 1024, C, None) == -1      # split
    assert f(A, 128, B, 1, 128, 128, 0, C, None) == -1       # n_cells
    assert f(None, 128, B, 1, 128, 128, 1024, C, None) == -1
    assert f(A, 128, B, 1, 128, 128, 1024, C + 4, None) == -1  # desc alignment
    assert f(A, 128, B, 0, 128, 128, 1024, C, None) == 0     # nothing to do


def test_window_tail_validation(kvattn):
    assert kvattn.kvattn_window_tail_workspace_bytes(40, 8, 128, 16384, 507904, 256, 500, 128) == 0
    n = kvattn.kvattn_window_tail_workspace_bytes(40, 8, 128, 16384, 507904, 256, 512, 128)
    assert n > 4 * 512 * 8 * 128 * 2
    f = kvattn.lib.kvattn_decode_window_tail
    ctx = A  # never dereferenced: validation fails first
    base = [ctx, A, B, C, 16384, A, B, 507904, 512, 40, 8, 128, 256, 128, 0.0884, C + 8192, C + 16384,
            A + (1 << 20), n, 1, 2]
    bad = list(base); bad[-1] = bad[-2]           # same stream twice
    assert f(*bad) == -1
    bad = list(base); bad[8] = 500                # tile not a multiple of tail_split
    assert f(*bad) == -1
    bad = list(base); bad[18] = n - 1             # workspace too small
    assert f(*bad) == -3
    bad = list(base); bad[10] = 3                 # 40 % 3
    assert f(*bad) == -1
    bad = list(base); bad[0] = None               # no context
    assert f(*bad) == -1
    assert kvattn.lib.kvattn_tail_ctx_destroy(None) == -1
    assert kvattn.lib.kvattn_tail_ctx_set_flags(None, kvattn.KVATTN_TAIL_PREFETCH) == -1
    assert kvattn.lib.kvattn_tail_wait(None, 10) == -1


def test_window_tail_direct_validation(kvattn):
    f = kvattn.lib.kvattn_decode_window_tail_direct
    n = kvattn.kvattn_window_tail_direct_workspace_bytes(40, 8, 128, 16384, 507904, 256, 128)
    assert n > (64 + 3968) * 40 * 128 * 4
    base = [A, B, C, 16384, A + 4096, B + 4096, 507904, 40, 8, 128, 256, 128, 0.0884, C + 8192, C + 16384,
            A + (1 << 20), n, None]
    bad = list(base); bad[0] = None
    assert f(*bad) == -1
    bad = list(base); bad[9] = 64                 # head_dim
    assert f(*bad) == -2
    bad = list(base); bad[11] = 48                # tail split not a multiple of 32
    assert f(*bad) == -2
    bad = list(base); bad[16] = n - 1             # workspace
    assert f(*bad) == -3
    bad = list(base); bad[4] = A + 4100           # tail not 16-byte aligned
    assert f(*bad) == -1


def test_multi_query_limits(kvattn, monkeypatch):
    """Checked on the host before any device work."""
    def call(**over):
        a = dict(q=A, k=B, v=C, ks=None, vs=None, kv_type=0, n_cells=1024, plan=None, plan_stride=0,
                 seq_lens=A + 4096, n_seq=1, max_len=1024, n_q=4, n_head=32, n_head_kv=8, head_dim=128, split=256,
                 scale=0.0884, out=A + 8192, lse=A + 16384, ws=A + 65536, ws_bytes=1 << 30, stream=None)
        a.update(over)
        return kvattn.lib.kvattn_decode_multi(*a.values())
    assert call(n_q=33) == kvattn.KVATTN_ERR_UNSUPPORTED           # 4 x 33 = 132 rows > 128
    assert call(head_dim=256, n_q=33) == kvattn.KVATTN_ERR_UNSUPPORTED  # head_dim 256: 132 rows > 128
    assert call(head_dim=256, kv_type=1, ks=A, vs=A, n_q=33) == kvattn.KVATTN_ERR_UNSUPPORTED  # 132 rows
    assert call(head_dim=64) == kvattn.KVATTN_ERR_UNSUPPORTED
    assert call(kv_type=1, ks=A, vs=A, n_q=33) == kvattn.KVATTN_ERR_UNSUPPORTED  # Q8_0: 132 rows > 128
    assert call(kv_type=3, ks=A, vs=A, n_q=33) == kvattn.KVATTN_ERR_UNSUPPORTED  # Q4_0: 132 rows > 128
    assert call(n_q=17, n_head=64) == kvattn.KVATTN_ERR_UNSUPPORTED  # 8 x 17 = 136 rows > 128
    assert call(n_q=32, ws_bytes=1000) == kvattn.KVATTN_ERR_WORKSPACE  # 128 rows pass the limits
    # 100000 sequences x 2048 splits x 8 KV heads fit 32 bits, x 4 row groups (64 rows of a
    # Q8_0 cache, 16 a group) do not; f16 head_dim 128 takes 64 rows in one tcgen05 unit
    big = dict(n_seq=100000, max_len=65536, n_cells=65536, split=32)
    assert call(n_q=16, kv_type=1, ks=A, vs=A, **big) == kvattn.KVATTN_ERR_UNSUPPORTED
    assert call(n_q=16, **big) == kvattn.KVATTN_ERR_WORKSPACE                 # one unit: only the workspace
    assert call(n_q=8, **big) == kvattn.KVATTN_ERR_WORKSPACE                  # one group: only the workspace
    monkeypatch.setenv("KVATTN_TC", "0")                                     # the mma.sync row groups (2 x 32)
    assert call(n_q=16, **big) == kvattn.KVATTN_ERR_UNSUPPORTED
    monkeypatch.delenv("KVATTN_TC")
    assert call(kv_type=1) == kvattn.KVATTN_ERR_INVALID_ARG                   # Q8_0 without scales
    assert call(n_q=0) == kvattn.KVATTN_ERR_INVALID_ARG
    assert call(q=None) == kvattn.KVATTN_ERR_INVALID_ARG
    assert call(ws_bytes=1000) == kvattn.KVATTN_ERR_WORKSPACE
    one = kvattn.kvattn_decode_workspace_bytes(2, 4 * 32, 128, 4096, 128)
    assert kvattn.kvattn_decode_multi_workspace_bytes(2, 4, 32, 128, 4096, 128) == one
    assert kvattn.kvattn_decode_multi_workspace_bytes(2, 0, 32, 128, 4096, 128) == 0
