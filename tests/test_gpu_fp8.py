"""GPU parity of the decode over FP8 cache rows against the float64 oracle.

The pool is packed on the GPU into 656-byte rows (mla_fp8_pack_cache, itself
bit-exact against the oracle's quantiser) and decoded by mla_decode_fp8.  The
oracle quantises the same bf16 rows with its own fp8_row_quantize, widens them
with fp8_row_dequantize (value = E4M3 code * its tile's scale, exactly) and
runs the plain latent attention on those values.  The kernel rounds each
dequantised value to bf16 (its tensor-core operand); the tolerance covers that
the same way it covers the bf16 rounding of q_lat and P.
"""
import numpy as np
import pytest

from mla_latent_cache_gb300 import workloads as W
from oracle import mla_oracle as O
from tests._tol import parity

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _fp8_rows(bits):
    """Oracle: bf16 rows [S, 576] (bit patterns) -> dequantised float64 rows [S, 576]."""
    packed = O.fp8_row_quantize(W.bf16_bits_to_f64(bits[:, :512]), bits[:, 512:])
    lat, _, rope_bits = O.fp8_row_dequantize(packed)
    return np.concatenate([lat, W.bf16_bits_to_f64(rope_bits)], axis=-1)


def _oracle_fp8(w, batches):
    pool, bt = w.compact_view()
    q_lat, q_pe = W.bf16_bits_to_f64(w.q_lat), W.bf16_bits_to_f64(w.q_pe)
    out = {}
    for b in batches:
        S = int(w.seq_lens[b])
        if S == 0:
            out[b] = (np.zeros((w.T, w.H, 512)), np.full((w.T, w.H), -np.inf))
            continue
        rows = _fp8_rows(O.gather_rows(pool, bt[b], S))
        out[b] = O.attend_latent(q_lat[b], q_pe[b], rows, O.causal_mask(S, w.T, w.causal))
    return out


def _run(mla, w, cuda, num_slots=0, override=0, checked=False, expect=None):
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    st = DecodeStep(w, device=cuda, num_slots=num_slots, num_splits_override=override, checked=checked,
                    with_absorb=False, cache_format="fp8")
    st.plan()
    st.decode()
    torch.cuda.synchronize()
    status, info = mla.mla_read_device_status(st.workspace)
    assert status == (mla.MLA_OK if expect is None else expect), (mla.mla_status_string(status), info)
    return st


def _check(st, w, batches, name):
    ref = _oracle_fp8(w, batches)
    o, lse = _np(st.o_lat), st.lse.cpu().numpy().astype(np.float64)
    parity(np.stack([o[b] for b in batches]), np.stack([ref[b][0] for b in batches]), f"{name} o_lat")
    parity(np.stack([lse[b] for b in batches]), np.stack([ref[b][1] for b in batches]), f"{name} lse")


@pytest.mark.parametrize("H,seq_lens,T,causal", [
    (16, [300, 77, 1, 64, 65, 129, 0, 1000], 1, False),   # page boundaries, ragged tails, an empty sequence
    (128, [700, 90, 2048], 3, True),                     # extend rows, causal
    (64, [513, 4000], 1, False),
])
def test_fp8_decode_small(mla, cuda, H, seq_lens, T, causal):
    w = W.custom_workload(H, seq_lens, T=T, causal=causal, seed=17)
    st = _run(mla, w, cuda)
    _check(st, w, range(w.B), f"fp8 H={H} T={T}")


@pytest.mark.parametrize("sharp", [False, True])
@pytest.mark.parametrize("override", [0, 8])
def test_fp8_decode_splits(mla, cuda, sharp, override):
    # few work ranges or a forced split: partial states merged in the kernel; sharp
    # logits make a wrong merge weight visible
    w = W.custom_workload(128, [5000, 3000, 200, 6100], seed=19, sharp=sharp)
    st = _run(mla, w, cuda, num_slots=3 if override == 0 else 0, override=override)
    _check(st, w, range(w.B), f"fp8 splits override={override} sharp={sharp}")


def test_fp8_decode_v3_uniform_sampled(mla, cuda):
    # the uniform V3 batch at full size (B=64, S=4096) in its default launch; the
    # oracle quantises only the sampled sequences' rows (the quantiser is row-local)
    w = W.config_workload(2)
    st = _run(mla, w, cuda)
    _check(st, w, [0, 17, 40, 63], "fp8 v3 uniform")


def test_fp8_decode_v3_ragged_sampled(mla, cuda):
    # the ragged V3 batch (B=128, S from 256 to 32768, balanced ranges merged in the
    # kernel) at full size; sampled sequences include the shortest and the longest
    w = W.config_workload(3)
    st = _run(mla, w, cuda)
    lens = w.seq_lens
    bs = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 5, 100})
    _check(st, w, bs, "fp8 v3 ragged")


def test_fp8_decode_matches_bf16_within_quantisation(mla, cuda):
    # the FP8 rows change every latent value by at most half an E4M3 step of its
    # tile's scale: the outputs move accordingly, and nothing else differs
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    w = W.custom_workload(128, [1500, 640], seed=23)
    f8 = _run(mla, w, cuda)
    bf = DecodeStep(w, device=cuda, with_absorb=False)
    bf.plan()
    bf.decode()
    torch.cuda.synchronize()
    d = np.abs(_np(f8.o_lat) - _np(bf.o_lat)).max()
    assert 0 < d < 0.1 * np.abs(_np(bf.o_lat)).max()


def test_fp8_checked_mode_flags_bad_block(mla, cuda):
    w = W.custom_workload(16, [300, 200], seed=29)
    w.block_table[1, 1] = -7                        # outside the pool: read as zeros and reported
    st = _run(mla, w, cuda, checked=True, expect=mla.MLA_ERR_DEVICE_CHECK)
    # the other sequence is unaffected
    ref = _oracle_fp8(w, [0])
    parity(_np(st.o_lat)[:1], ref[0][0][None], "fp8 neighbour of a bad block")
