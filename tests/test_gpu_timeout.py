"""The failure detector: a bounded pipeline wait that runs out is reported as
MLA_ERR_TIMEOUT through the workspace status word, the launch returns (its
copies and MMAs drained, tensor memory freed), and the context stays usable.

The wait is made to run out by shortening the pipeline waits' limit to a few
cycles (mla_debug_set_wait_limit): a page cannot land that fast.  Nothing here
faults or traps the GPU; the drains keep their full limit.
"""
import numpy as np
import pytest

from mla_latent_cache_gb300 import workloads as W
from oracle import mla_oracle as O
from tests._tol import parity

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


def test_pipeline_timeout_is_reported_and_recoverable(mla, cuda):
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    # four sequences of 16 pages on four work ranges: one segment per range, no merge records
    w = W.custom_workload(128, [1024, 1000, 1024, 990], seed=5)
    st = DecodeStep(w, device=cuda, num_slots=4, with_absorb=False)
    st.plan()
    torch.cuda.synchronize()
    assert int(st.plan_header()[mla.HDR["NUM_MERGE"]]) == 0
    try:
        mla.check(mla.mla_debug_set_wait_limit(16), "set wait limit")
        for _ in range(2):
            st.plan()
            st.decode()
            torch.cuda.synchronize()
            status, info = mla.mla_read_device_status(st.workspace)
            assert status == mla.MLA_ERR_TIMEOUT, (mla.mla_status_string(status), info)
            assert info > 0          # the role and wait that gave up
    finally:
        mla.check(mla.mla_debug_set_wait_limit(0), "reset wait limit")
    # the same workspace, re-planned, decodes normally afterwards
    st.plan()
    st.decode()
    torch.cuda.synchronize()
    status, info = mla.mla_read_device_status(st.workspace)
    assert status == mla.MLA_OK, (mla.mla_status_string(status), info)
    pool, bt = w.compact_view()
    q_lat, q_pe = W.bf16_bits_to_f64(w.q_lat), W.bf16_bits_to_f64(w.q_pe)
    for b in range(w.B):
        rows = W.bf16_bits_to_f64(O.gather_rows(pool, bt[b], int(w.seq_lens[b])))
        ro, rl = O.attend_latent(q_lat[b], q_pe[b], rows, O.causal_mask(int(w.seq_lens[b]), 1, False))
        parity(st.o_lat[b].float().cpu().numpy().astype(np.float64), ro, f"after timeout o_lat b={b}")
        parity(st.lse[b].cpu().numpy().astype(np.float64), rl, f"after timeout lse b={b}")
