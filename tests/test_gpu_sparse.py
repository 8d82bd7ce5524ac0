"""GPU parity of the index-driven (sparse) decode against the float64 oracle.

The oracle (sparse_decode_ref) attends each query token to exactly its listed
rows; it is pinned on the CPU by its reduction to the dense oracle when the list
is a whole sequence.  Tolerances as everywhere (tests/_tol.py).
"""
import numpy as np
import pytest

from oracle import mla_oracle as O
from mla_latent_cache_gb300 import workloads as W
from tests._tol import parity

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _run(mla, sw, cuda, num_slots=0, override=0, checked=False, expect=None):
    import torch
    from mla_latent_cache_gb300.runtime import SparseStep
    st = SparseStep(sw, device=cuda, num_slots=num_slots, num_splits_override=override, checked=checked)
    st.decode()
    torch.cuda.synchronize()
    status, info = mla.mla_read_device_status(st.workspace)
    assert status == (mla.MLA_OK if expect is None else expect), (mla.mla_status_string(status), info)
    return st


def _oracle(sw):
    w = sw.ctx
    pool = W.bf16_bits_to_f64(w.full_pool())
    return O.sparse_decode_ref(W.bf16_bits_to_f64(w.q_lat), W.bf16_bits_to_f64(w.q_pe), pool, sw.indices,
                               sw.topk_length)


def _check(st, sw, name):
    ro, rl = _oracle(sw)
    parity(_np(st.o_lat), ro, f"{name} o_lat")
    parity(st.lse.cpu().numpy().astype(np.float64), rl, f"{name} lse")


@pytest.mark.parametrize("sharp", [False, True])
def test_sparse_v32_topk2048(mla, cuda, sharp):
    # V3 heads, two query tokens per sequence (S_q = 2), top-2048 lists over
    # contexts of 3000 .. 9000 rows, one list shorter than topk and not a
    # multiple of 64, one of a single row
    sw = W.sparse_workload(128, [3000, 9000, 4100, 2500], 2, 2048, lengths=[2048, 1000, 1, 2048], sharp=sharp,
                           name="v32_sparse")
    st = _run(mla, sw, cuda)
    _check(st, sw, f"sparse topk2048 sharp={sharp}")


def test_sparse_in_order_equals_dense(mla, cuda):
    # a list of a whole sequence's rows, in order, is the dense decode of that sequence
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    lens = [1000, 4096, 130, 2048]
    sw = W.sparse_workload(128, lens, 1, 4096, lengths=lens, in_order=True, name="in_order")
    st = _run(mla, sw, cuda, num_slots=8)
    dn = DecodeStep(sw.ctx, device=cuda, num_slots=8, with_absorb=False)
    dn.plan()
    dn.decode()
    torch.cuda.synchronize()
    assert torch.equal(st.o_lat, dn.o_lat)
    assert torch.equal(st.lse, dn.lse)
    _check(st, sw, "in order")


@pytest.mark.parametrize("override,slots", [(0, 3), (4, 0), (0, 0)])
def test_sparse_splits_and_merge(mla, cuda, override, slots):
    # few work ranges (or a forced split) cut each list into partial segments merged in the kernel
    sw = W.sparse_workload(128, [8192, 6000, 300], 1, 4096, lengths=[4096, 2900, 300], name="split")
    st = _run(mla, sw, cuda, num_slots=slots, override=override)
    _check(st, sw, f"split override={override} slots={slots}")


def test_sparse_repeats_and_small_heads(mla, cuda):
    # rows drawn with replacement (a repeated row counts once per listing), H = 16, topk 100
    sw = W.sparse_workload(16, [500, 70, 2000], 3, 100, replace=True, name="repeats")
    assert any(len(np.unique(sw.indices[b, t, :sw.topk_length[b]])) < sw.topk_length[b]
               for b in range(sw.B) for t in range(sw.S_q))
    st = _run(mla, sw, cuda)
    _check(st, sw, "repeats H=16")


@pytest.mark.parametrize("H", [1, 8, 64])
def test_sparse_head_counts(mla, cuda, H):
    sw = W.sparse_workload(H, [700, 3000], 2, 640, lengths=[640, 333], name=f"h{H}")
    st = _run(mla, sw, cuda)
    _check(st, sw, f"H={H}")


def test_sparse_empty_lists(mla, cuda):
    # an empty list gives o = 0 and lse = -inf; its neighbours are unaffected
    sw = W.sparse_workload(128, [1000, 1000, 1000], 1, 256, lengths=[0, 256, 0], name="empty")
    st = _run(mla, sw, cuda)
    o, lse = _np(st.o_lat), st.lse.cpu().numpy()
    assert np.all(o[0] == 0) and np.all(o[2] == 0)
    assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
    _check(st, sw, "empty lists")


def test_sparse_lengths_past_topk_clamp(mla, cuda):
    # a length above topk counts as topk, and is reported (checked or not)
    import torch
    sw = W.sparse_workload(128, [3000, 3000], 1, 512, lengths=[512, 512], name="clamp")
    st = _run(mla, sw, cuda)
    sw_long = W.SparseWorkload(ctx=sw.ctx, topk=512, indices=sw.indices,
                               topk_length=np.array([900, 512], dtype=np.int32))
    st2 = _run(mla, sw_long, cuda, expect=mla.MLA_ERR_DEVICE_CHECK)
    assert torch.equal(st.o_lat, st2.o_lat)
    assert torch.equal(st.lse, st2.lse)


def test_sparse_checked_reports_rows_outside_the_pool(mla, cuda):
    sw = W.sparse_workload(128, [2000, 2000], 1, 256, name="bad_row")
    bad = sw.indices.copy()
    bad[1, 0, 17] = sw.ctx.num_blocks * 64      # one past the pool's last row
    sw_bad = W.SparseWorkload(ctx=sw.ctx, topk=256, indices=bad, topk_length=sw.topk_length)
    st = _run(mla, sw_bad, cuda, checked=True, expect=mla.MLA_ERR_DEVICE_CHECK)
    # sequence 0 is untouched by the bad entry
    ro, rl = _oracle(sw)
    parity(_np(st.o_lat)[:1], ro[:1], "bad row neighbour o_lat")
    # unchecked, the row reads as zeros (score 0, value 0): compare with the oracle over
    # the same list with that row replaced by an all-zero row
    st2 = _run(mla, sw_bad, cuda)
    w = sw.ctx
    pool = W.bf16_bits_to_f64(w.full_pool())
    pool = np.concatenate([pool, np.zeros((1, 64, 576))], axis=0)
    ro2, rl2 = O.sparse_decode_ref(W.bf16_bits_to_f64(w.q_lat), W.bf16_bits_to_f64(w.q_pe), pool, bad,
                                   sw.topk_length)
    parity(_np(st2.o_lat), ro2, "bad row as zeros o_lat")
    parity(st2.lse.cpu().numpy().astype(np.float64), rl2, "bad row as zeros lse")
