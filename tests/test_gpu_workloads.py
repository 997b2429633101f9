"""GPU parity at the full sizes of the five decode-attention workloads, in the launch
configuration the benchmark times, against the fp64 oracle over every output row."""
import numpy as np
import pytest

import oracle
from oracle import plan_oracle as po
from kv_cache_decode_02_gb300 import inputs
from tests.gpu_util import assert_close, dev, rmse

pytestmark = pytest.mark.gpu


def test_qwen3_8b_layer(kvattn):
    import torch
    w = inputs.QWEN3_8B_LAYER
    q = inputs.make_q(w, layer=0)
    k, v = inputs.make_kv_f16(w, layer=0)
    out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(np.array(w.seq_lens, np.int32)), split=w.split)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_f16(q, k, v, list(w.seq_lens))
    assert_close(out, lse, wo, wl)
    assert rmse(out, wo) < 3e-4


def test_multislot_plan_gqa6(kvattn):
    import torch
    w = inputs.MULTISLOT_PLAN
    lay = inputs.make_unified_layout(w)
    plan, lens = kvattn.build_cell_plan(lay.encoded_cells, w.n_cells)
    wplan, wlens = po.build_cell_plan(lay.encoded_cells, w.n_cells)
    assert np.array_equal(plan, wplan) and np.array_equal(lens, wlens)
    q = inputs.make_q(w)
    k = inputs.normal_f16(np.random.default_rng([2000 + w.number, 0]), (w.n_cells, w.n_head_kv, w.head_dim))
    v = inputs.normal_f16(np.random.default_rng([3000 + w.number, 0]), (w.n_cells, w.n_head_kv, w.head_dim))
    inputs.nan_fill_unselected(k, v, np.concatenate(lay.selected))
    out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(lens), split=w.split, cell_plan=dev(plan),
                             n_cells=w.n_cells)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_f16(q, k, v, lens.tolist(), plan=plan)
    assert_close(out, lse, wo, wl)
    # descriptors of this plan, bit for bit
    n_split = -(-plan.shape[1] // w.split)
    desc = torch.zeros((w.n_seq, n_split, 4), dtype=torch.int32, device="cuda")
    kvattn.kvattn_build_descriptors(dev(plan), plan.shape[1], dev(lens), w.n_seq, plan.shape[1], w.split,
                                    w.n_cells, desc)
    torch.cuda.synchronize()
    assert np.array_equal(desc.cpu().numpy(), po.descriptors(plan, lens, plan.shape[1], w.split, w.n_cells))


def test_serving_batch_of_64_sequences(kvattn):
    """64 sequences x 4096 cells in one call with the automatic split (the bench's
    configuration): a sample of sequences against the oracle."""
    import torch
    w = inputs.BATCH64
    q = inputs.make_q(w)
    rng = np.random.default_rng(2000 + w.number)
    k = rng.standard_normal((w.n_seq, w.n_cells, w.n_head_kv, w.head_dim), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((w.n_seq, w.n_cells, w.n_head_kv, w.head_dim), dtype=np.float32).astype(np.float16)
    lens = np.array(w.seq_lens, np.int32)
    out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(lens), split=0, n_cells=w.n_cells, max_len=w.n_cells)
    torch.cuda.synchronize()
    pick = np.array([0, 1, 17, 40, 63])
    wo, wl = oracle.decode_f16(q[pick], k[pick], v[pick], lens[pick].tolist())
    assert_close(out[pick], lse[pick], wo, wl)


def test_f16_head_dim_256_long_context(kvattn):
    """65536 cells at head_dim 256 with the automatic split (the bench's configuration)."""
    import torch
    w = inputs.F16_D256_LONG
    q = inputs.make_q(w)
    k, v = inputs.make_kv_f16(w)
    out, lse = kvattn.decode(dev(q), dev(k), dev(v), dev(np.array(w.seq_lens, np.int32)), split=0)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_f16(q, k, v, list(w.seq_lens))
    assert_close(out, lse, wo, wl)


@pytest.mark.parametrize("w", [inputs.Q8_LONG_D128, inputs.Q8_LONG_D256], ids=lambda w: w.name)
def test_q8_0_long_context(kvattn, w):
    import torch
    q = inputs.make_q(w)
    (kq, kd), (vq, vd) = inputs.make_kv_q8(w)
    out, lse = kvattn.decode(dev(q), dev(kq), dev(vq), dev(np.array(w.seq_lens, np.int32)), split=w.split,
                             k_scales=dev(kd), v_scales=dev(vd))
    torch.cuda.synchronize()
    wo, wl = oracle.decode_q8_0(q, kq, kd, vq, vd, list(w.seq_lens))
    assert_close(out, lse, wo, wl)


def test_window_tail_equals_resident_and_oracle(kvattn):
    import torch
    w = inputs.WINDOW_TAIL
    q = inputs.make_q(w)
    k, v = inputs.make_kv_f16(w)
    n_tail = w.n_cells - w.n_window
    # tail = the older cells in pinned host memory; window = the most recent cells in HBM
    k_tail = torch.from_numpy(k[:n_tail]).pin_memory()
    v_tail = torch.from_numpy(v[:n_tail]).pin_memory()
    k_win, v_win = dev(k[n_tail:]), dev(v[n_tail:])
    qd = dev(q[0])
    wt = kvattn.WindowTail()
    copy_stream = torch.cuda.Stream()
    out, lse = wt(qd, k_win, v_win, k_tail, v_tail, split=w.split, tile_cells=w.tile_cells,
                  tail_split=w.tail_split, copy_stream=copy_stream)
    kvattn.kvattn_tail_wait(wt.ctx, 60000)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_f16(q, k, v, list(w.seq_lens))
    assert_close(out.view(1, *out.shape), lse.view(1, -1), wo, wl)
    # the same cache fully resident, through the plain decode entry point
    ro, rl = kvattn.decode(qd.view(1, *qd.shape), dev(k), dev(v), dev(np.array(w.seq_lens, np.int32)),
                           split=w.split)
    torch.cuda.synchronize()
    assert np.max(np.abs(ro.cpu().numpy()[0] - out.cpu().numpy())) <= 2e-3
    assert np.max(np.abs(rl.cpu().numpy()[0] - lse.cpu().numpy())) <= 1e-4
    wt.close()


def test_window_tail_direct_full(kvattn):
    import torch
    w = inputs.WINDOW_TAIL
    q = inputs.make_q(w)
    k, v = inputs.make_kv_f16(w)
    n_tail = w.n_cells - w.n_window
    k_tail = torch.from_numpy(k[:n_tail]).pin_memory()
    v_tail = torch.from_numpy(v[:n_tail]).pin_memory()
    out, lse = kvattn.window_tail_direct(dev(q[0]), dev(k[n_tail:]), dev(v[n_tail:]), k_tail, v_tail,
                                         split=w.split, tail_split=w.tail_split)
    torch.cuda.synchronize()
    wo, wl = oracle.decode_f16(q, k, v, list(w.seq_lens))
    assert_close(out.view(1, *out.shape), lse.view(1, -1), wo, wl)
