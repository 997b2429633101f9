"""The split selector (kvattn_select_split_for): the smallest power of two >= 64 whose work
units (sequences x splits x KV heads) fit in one wave of resident CTAs.  The expected
values are the fastest splits measured on GB300 for the Qwen3-8B-shaped decode (32/8
heads, head_dim 128; 608 resident CTAs = 152 SMs x 4) over splits 64-4096; where two
splits tied within 1 %, the selector's is one of them."""
import pytest

RESIDENT = 608


@pytest.mark.parametrize("n_seq,max_len,want", [
    (1, 1024, 64),       # measured: 64 best (6.7 us)
    (1, 4096, 64),       # 64 best (8.1 us)
    (1, 16384, 256),     # 256 best (14.9 us; 128: 18.7, 512: 17.8)
    (1, 65536, 1024),    # 1024 best (44.5 us; 512: 49.2)
    (1, 262144, 4096),   # 4096 best (156.8 us; 1024: 161.2)
    (4, 1024, 64),       # 64 best
    (4, 4096, 256),      # 256 best (14.8 us; 128: 18.5)
    (4, 16384, 1024),    # 1024 best (44.0 us; 256: 46.2)
    (4, 65536, 4096),    # 4096: 159.3 us, 1024: 158.3 us (tie)
])
def test_matches_measured_best_splits(kvattn, n_seq, max_len, want):
    assert kvattn.kvattn_select_split_for(n_seq, max_len, 8, RESIDENT) == want


def test_rule_and_edges(kvattn):
    sel = kvattn.kvattn_select_split_for
    for n_seq in (1, 3, 16):
        for max_len in (0, 1, 31, 100, 5000, 123457, 1 << 22):
            for hk in (1, 2, 8):
                for res in (1, 100, 608, 4096):
                    sp = sel(n_seq, max_len, hk, res)
                    assert sp >= 64 and sp & (sp - 1) == 0 and sp % 32 == 0
                    units = n_seq * (-(-max_len // sp)) * hk
                    if units > res:
                        # only when one split per sequence (or the 2^30 cap) is reached
                        assert sp >= max_len or sp == 1 << 30
                    if sp > 64:
                        half = sp // 2
                        assert n_seq * (-(-max_len // half)) * hk > res and half < max_len
    assert sel(0, 1000, 8, 608) == 64
    assert sel(1, 0, 8, 608) == 64
    from kv_cache_decode_02_gb300.kvattn import KvattnError
    for bad in ((-1, 10, 8, 608), (1, -1, 8, 608), (1, 10, 0, 608), (1, 10, 8, 0)):
        with pytest.raises(KvattnError):
            sel(*bad)


def test_workspace_for_split_zero_covers_every_selection(kvattn):
    for n_seq, max_len in ((1, 16384), (4, 65536), (2, 1000)):
        auto = kvattn.kvattn_decode_workspace_bytes(n_seq, 32, 128, max_len, 0)
        assert auto == kvattn.kvattn_decode_workspace_bytes(n_seq, 32, 128, max_len, 64)
        for sp in (64, 128, 256, 1024, 4096):
            assert kvattn.kvattn_decode_workspace_bytes(n_seq, 32, 128, max_len, sp) <= auto
    assert kvattn.kvattn_decode_workspace_bytes(1, 32, 128, 100, -1) == 0
