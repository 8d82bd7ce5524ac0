"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (code inside an allocator or memory-pool callback, or a serving
loop whose device memory must stay fixed once it starts) hand the library only
their inputs and outputs; the library plans and decodes in a fixed scratch
array of its own.  This test calls that entry point through the C ABI twice in
a row, on two different batches, and checks each result against the regular
entry points (mla_plan + mla_decode with a caller-allocated workspace) within
the parity tolerance used by the other GPU tests.  It also checks that a batch
needing more than the fixed scratch is refused before anything runs.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import pytest

from mla_latent_cache_gb300 import workloads as W
from tests._tol import parity

pytestmark = pytest.mark.gpu


def _regular(mla, torch, st):
    """Output of the existing entry points (caller-allocated workspace)."""
    st.plan()
    st.decode()
    torch.cuda.synchronize()
    return st.o_lat.float().cpu().numpy(), st.lse.cpu().numpy()


def _noalloc(mla, torch, st):
    o_lat = torch.full_like(st.o_lat, float("nan"))
    lse = torch.full_like(st.lse, float("nan"))
    status = mla.mla_decode_noalloc(st.geom, st.batch, st.q_lat, st.q_pe, st.cache, st.block_table,
                                    st.block_table.shape[1], st.seq_lens, o_lat, lse)
    assert status == mla.MLA_OK, mla.mla_status_string(status)
    torch.cuda.synchronize()
    return o_lat.float().cpu().numpy(), lse.cpu().numpy()


def test_noalloc_matches_regular_entry_point_twice(mla, cuda):
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    cases = [
        (W.config_workload(1), 8, 0),                                            # V2-Lite tiny, split 8 ways
        (W.custom_workload(128, [300, 1000, 64, 4096, 0, 129], T=1, seed=23), 16, 0),  # V3 heads, ragged
    ]
    for w, slots, ov in cases:
        st = DecodeStep(w, device=cuda, num_slots=slots, num_splits_override=ov, with_absorb=False)
        assert mla.mla_workspace_size(st.geom, st.batch) <= mla.NOALLOC_SCRATCH_BYTES
        ref_o, ref_l = _regular(mla, torch, st)
        got_o, got_l = _noalloc(mla, torch, st)
        parity(got_o, ref_o, f"{w.name} o_lat")
        parity(got_l, ref_l, f"{w.name} lse")


def test_noalloc_refuses_batches_beyond_its_scratch(mla, cuda):
    import torch
    g = mla.make_geom(128)
    b = mla.make_batch(64, 1, False, 64, num_slots=152)   # needs ~80 MB of partial slots
    assert mla.mla_workspace_size(g, b) > mla.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.uint8, device=cuda)
    cache = mla.mla_cache(dummy.data_ptr(), dummy.data_ptr(), 576, 64 * 576, 576, 64 * 576, 1)
    p = dummy.data_ptr()
    assert mla.mla_decode_noalloc(g, b, p, p, cache, p, 64, p, p, p) == mla.MLA_ERR_WORKSPACE
