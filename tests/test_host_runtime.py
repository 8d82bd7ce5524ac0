"""Host-side runtime and bench bookkeeping (no GPU needed)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_bytes_ledger_uniform_v3():
    """The roofline numerator of the V3 uniform batch (B=64, S=4096, H=128, T=1),
    term by term: cache rows once (576 bf16), q_lat + q_pe, o_lat, lse, block
    table, lengths."""
    sys.path.insert(0, ROOT)
    import bench
    from mla_latent_cache_gb300 import workloads as W
    w = W.config_workload(2)
    rows = 64 * 4096 * 576 * 2
    q = 64 * 128 * (512 + 64) * 2
    o = 64 * 128 * 512 * 2
    lse = 64 * 128 * 4
    bt = 64 * 64 * 4
    sl = 64 * 4
    assert rows + q + o + lse + bt + sl == 319_865_088
    assert bench.algorithmic_bytes(w)["decode"] == 319_865_088


def test_step_inputs_share_one_buffer(mla):
    """q_nope, q_pe, seq_lens and the block table are views of one buffer at
    256-byte-aligned offsets (one host-to-device copy per step), holding the
    workload's values."""
    import torch
    from mla_latent_cache_gb300 import workloads as W
    from mla_latent_cache_gb300.runtime import DecodeStep
    w = W.custom_workload(16, [300, 77, 5, 0], T=1, seed=3)
    st = DecodeStep(w, device="cpu")
    base, end = st.inputs.data_ptr(), st.inputs.data_ptr() + st.inputs.numel()
    for name in ("q_nope", "q_pe", "seq_lens", "block_table"):
        t = getattr(st, name)
        off = t.data_ptr() - base
        assert off % 256 == 0 and t.data_ptr() + t.numel() * t.element_size() <= end, name
        assert t.is_contiguous()
    assert np.array_equal(st.seq_lens.numpy(), w.seq_lens)
    assert np.array_equal(st.block_table.numpy(), w.block_table)
    assert np.array_equal(st.q_pe.view(torch.int16).numpy().view(np.uint16), w.q_pe)
    assert np.array_equal(st.q_nope.view(torch.int16).numpy().view(np.uint16), w.q_nope)
    # writing through the buffer is seen by the views (they alias it)
    st.inputs.zero_()
    assert int(st.seq_lens.abs().sum()) == 0


def test_profiled_traffic_only_for_the_profiled_sources(tmp_path, monkeypatch):
    """bench.py reports ncu DRAM traffic only while the decode sources hash to
    the value recorded beside it (a capture of an older kernel reads as null)."""
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    h = hashlib.sha256()
    for f in bench.DECODE_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    sha = h.hexdigest()[:16]
    prof = tmp_path / "p.md"
    monkeypatch.setattr(bench, "PROFILE", str(prof))
    assert bench.profiled_traffic() is None                      # no summary
    prof.write_text(f"kernel_source_sha256: {sha}\n| dram_bytes_per_launch | 123456 |\n")
    assert bench.profiled_traffic() == 123456
    prof.write_text("kernel_source_sha256: 0000000000000000\n| dram_bytes_per_launch | 123456 |\n")
    assert bench.profiled_traffic() is None                      # stale capture


def test_peaks_measured_else_fallback(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    hbm, tc, kind = bench._peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert kind == "measured" and hbm > 1000 and tc > 100
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._peaks() == (6800.0, 1900.0, "fallback")
