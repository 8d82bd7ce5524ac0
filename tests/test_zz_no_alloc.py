"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (code inside an allocator or memory-pool callback, or a serving
loop whose device memory must stay fixed once it starts) hand the library only
their inputs and outputs; the library plans and decodes in a fixed scratch
array of its own.  These tests call that entry point through the C ABI twice in
a row, on two different batches, and check each result against the regular
entry points (mla_plan + mla_decode with a caller-allocated workspace) and the
float64 oracle, within the parity tolerance used by the other GPU tests; that
the default range count (num_slots = 0) is shrunk to fit the scratch at V3
geometry; that device-side errors come back through mla_read_device_status
without a workspace; and that a batch needing more than the fixed scratch is
refused before anything runs.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

from oracle import mla_oracle as O
from mla_latent_cache_gb300 import workloads as W
from tests._tol import parity

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


def _regular(mla, torch, st):
    """Output of the existing entry points (caller-allocated workspace)."""
    st.plan()
    st.decode()
    torch.cuda.synchronize()
    return st.o_lat.float().cpu().numpy(), st.lse.cpu().numpy()


def _noalloc(mla, torch, st, batch=None):
    o_lat = torch.full_like(st.o_lat, float("nan"))
    lse = torch.full_like(st.lse, float("nan"))
    status = mla.mla_decode_noalloc(st.geom, st.batch if batch is None else batch, st.q_lat, st.q_pe, st.cache,
                                    st.block_table, st.block_table.shape[1], st.seq_lens, o_lat, lse)
    assert status == mla.MLA_OK, mla.mla_status_string(status)
    torch.cuda.synchronize()
    status, info = mla.mla_read_device_status(None)
    assert status == mla.MLA_OK, (mla.mla_status_string(status), info)
    return o_lat.float().cpu().numpy(), lse.cpu().numpy()


def _oracle(w):
    pool, bt = w.compact_view()
    o, l = O.decode_ref(W.bf16_bits_to_f64(w.q_lat), W.bf16_bits_to_f64(w.q_pe), W.bf16_bits_to_f64(pool), bt,
                        w.seq_lens, w.causal)
    return o, l


def test_noalloc_matches_regular_entry_point_twice(mla, cuda):
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    cases = [
        (W.config_workload(1), 8, 0),                                                  # V2-Lite tiny, split 8 ways
        (W.custom_workload(128, [300, 1000, 64, 4096, 0, 129], T=1, seed=23), 0, 0),  # V3 heads, ragged, default ranges
    ]
    for w, slots, ov in cases:
        st = DecodeStep(w, device=cuda, num_slots=slots, num_splits_override=ov, with_absorb=False)
        ref_o, ref_l = _regular(mla, torch, st)
        got_o, got_l = _noalloc(mla, torch, st)
        parity(got_o, ref_o, f"{w.name} o_lat vs mla_decode")
        parity(got_l, ref_l, f"{w.name} lse vs mla_decode")
        or_o, or_l = _oracle(w)
        parity(got_o, or_o, f"{w.name} o_lat vs oracle")
        parity(got_l, or_l, f"{w.name} lse vs oracle")


def test_noalloc_default_ranges_fit_the_scratch_at_v3_geometry(mla, cuda):
    """With num_slots = 0 the default range count (one per CTA pair) would need more
    partial space than the scratch holds; the call shrinks it and still decodes."""
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    w = W.custom_workload(128, [4096] * 8 + [700, 5000, 64, 1], T=1, seed=29, sharp=True)
    st = DecodeStep(w, device=cuda, with_absorb=False)
    assert mla.mla_workspace_size(st.geom, st.batch) > mla.NOALLOC_SCRATCH_BYTES
    got_o, got_l = _noalloc(mla, torch, st)
    or_o, or_l = _oracle(w)
    parity(got_o, or_o, "o_lat vs oracle")
    parity(got_l, or_l, "lse vs oracle")


def test_noalloc_reports_device_errors_without_a_workspace(mla, cuda):
    """A length beyond the block table is caught by the planner on the device; the
    status comes back through mla_read_device_status(NULL) and is cleared there."""
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    w = W.custom_workload(16, [200, 100], T=1, seed=31)
    st = DecodeStep(w, device=cuda, num_slots=4, with_absorb=False)
    st.seq_lens[1] = w.max_pages * 64 + 1
    o_lat = torch.empty_like(st.o_lat)
    lse = torch.empty_like(st.lse)
    assert mla.mla_decode_noalloc(st.geom, st.batch, st.q_lat, st.q_pe, st.cache, st.block_table,
                                  st.block_table.shape[1], st.seq_lens, o_lat, lse) == mla.MLA_OK
    status, info = mla.mla_read_device_status(None)
    assert status == mla.MLA_ERR_DEVICE_CHECK and info == 1
    assert mla.mla_read_device_status(None)[0] == mla.MLA_OK


def test_noalloc_refuses_batches_beyond_its_scratch(mla, cuda):
    import torch
    g = mla.make_geom(128)
    b = mla.make_batch(64, 1, False, 64, num_slots=152)   # needs ~80 MB of partial slots
    assert mla.mla_workspace_size(g, b) > mla.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(64, dtype=torch.uint8, device=cuda)
    cache = mla.mla_cache(dummy.data_ptr(), dummy.data_ptr(), 576, 64 * 576, 576, 64 * 576, 1)
    p = dummy.data_ptr()
    assert mla.mla_decode_noalloc(g, b, p, p, cache, p, 64, p, p, p) == mla.MLA_ERR_WORKSPACE
