"""The Normal (decompressed) arm on the GPU against the float64 oracle.

mla_normal_expand must give k_nope = W_UK c and v = W_UV c for every visible
cache row (exact zeros for the padding rows of the last 128-row tile), and
mla_normal_attention the oracle's causal MHA output and LSE, within the
parity tolerance.  Ragged tails, rows past T in the last query tile, empty
sequences and invalid block ids of unused pages are covered; the full-size
extend workload is checked on sampled heads (heads are independent in MHA, so
the oracle on one head's slice is the exact reference for that head).
"""
import numpy as np
import pytest

from mla_latent_cache_gb300 import workloads as W
from oracle import mla_oracle as O
from tests._tol import parity

pytestmark = pytest.mark.gpu


def _f64(a):
    return W.bf16_bits_to_f64(a)


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _oracle_normal(w, batches=None, heads=None):
    pool, bt = w.compact_view()
    qn, qp, wuk, wuv = _f64(w.q_nope), _f64(w.q_pe), _f64(w.w_uk), _f64(w.w_uv)
    if heads is not None:
        qn, qp, wuk, wuv = qn[:, :, heads], qp[:, :, heads], wuk[heads], wuv[heads]
    return O.normal_ref(qn, qp, _f64(pool), bt, w.seq_lens, wuk, wuv, w.causal, batches=batches)


@pytest.mark.parametrize("H,seq_lens", [(16, [100, 300, 64, 1, 129]), (128, [200, 65])])
def test_normal_expand(mla, cuda, H, seq_lens):
    import torch
    from mla_latent_cache_gb300.runtime import NormalStep
    w = W.custom_workload(H, seq_lens, T=1, seed=31)
    st = NormalStep(w, device=cuda)
    st.expanded().fill_(float("nan"))
    st.expand()
    torch.cuda.synchronize()
    status, _ = mla.mla_read_device_status(None)
    assert status == mla.MLA_OK, mla.mla_status_string(status)
    exp = st.expanded()
    pool, bt = w.compact_view()
    for b, S in enumerate(seq_lens):
        rows = O.gather_rows(_f64(pool), bt[b], S)
        k_ref, v_ref = O.decompress_ref(rows[:, :512], _f64(w.w_uk), _f64(w.w_uv))
        r0 = b * st.rows_per_seq
        got = _np(exp[:, r0:r0 + S])                       # [H, S, 256]
        parity(np.transpose(got[:, :, :128], (1, 0, 2)), k_ref, f"k_nope b={b}")
        parity(np.transpose(got[:, :, 128:], (1, 0, 2)), v_ref, f"v b={b}")
        pad = -(-S // 128) * 128
        assert torch.all(exp[:, r0 + S:r0 + pad] == 0), f"padding rows of sequence {b} are not zero"


@pytest.mark.parametrize("H,seq_lens,T,causal", [
    (16, [300, 64, 1000, 0], 1, False),      # decode, ragged tails, an empty sequence
    (128, [200, 129], 16, True),             # extend, causal within the new rows
    (16, [600], 170, True),                  # two query tiles, the second ragged
    (128, [257], 1, False),                  # a tile whose second page is absent
])
def test_normal_attention(mla, cuda, H, seq_lens, T, causal):
    import torch
    from mla_latent_cache_gb300.runtime import NormalStep
    w = W.custom_workload(H, seq_lens, T=T, causal=causal, seed=37)
    st = NormalStep(w, device=cuda)
    st.o.fill_(float("nan"))
    st.lse.fill_(float("nan"))
    st.step()
    torch.cuda.synchronize()
    status, _ = mla.mla_read_device_status(None)
    assert status == mla.MLA_OK, mla.mla_status_string(status)
    o_ref, lse_ref = _oracle_normal(w)
    parity(_np(st.o), o_ref, "o")
    parity(st.lse.cpu().numpy(), lse_ref, "lse")


def test_normal_matches_absorbed_path(mla, cuda):
    """Both arms on the GPU give the same o (the identity the oracle is pinned to)."""
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep, NormalStep
    w = W.custom_workload(128, [700, 90], T=4, causal=True, seed=41)
    n = NormalStep(w, device=cuda)
    n.step()
    a = DecodeStep(w, device=cuda)
    a.step()
    torch.cuda.synchronize()
    o_ref, _ = _oracle_normal(w)
    parity(_np(n.o), o_ref, "normal o")
    parity(_np(a.o), o_ref, "absorbed o")
    parity(_np(n.lse), _np(a.lse), "lse normal vs absorbed")


@pytest.mark.parametrize("T", [16, 170])
def test_normal_extend_full_size_sampled_heads(mla, cuda, T):
    """The extend workload (B=8, prefix 8192 + T new rows) at full size, checked on
    sampled heads of two sequences."""
    import torch
    from mla_latent_cache_gb300.runtime import NormalStep
    w = W.config_workload(5, T=T)
    st = NormalStep(w, device=cuda)
    st.step()
    torch.cuda.synchronize()
    status, _ = mla.mla_read_device_status(None)
    assert status == mla.MLA_OK, mla.mla_status_string(status)
    heads = [0, 77, 127]
    bs = [0, 7]
    o_ref, lse_ref = _oracle_normal(w, batches=bs, heads=heads)
    o_got = _np(st.o)[:, :, heads]
    lse_got = st.lse.cpu().numpy()[:, :, heads]
    parity(o_got[bs], o_ref[bs], "o (sampled heads)")
    parity(lse_got[bs], lse_ref[bs], "lse (sampled heads)")


def _oracle_chunked(w, chunk, batches=None, heads=None):
    pool, bt = w.compact_view()
    qn, qp, wuk, wuv = _f64(w.q_nope), _f64(w.q_pe), _f64(w.w_uk), _f64(w.w_uv)
    if heads is not None:
        qn, qp, wuk, wuv = qn[:, :, heads], qp[:, :, heads], wuk[heads], wuv[heads]
    return O.normal_chunked_ref(qn, qp, _f64(pool), bt, w.seq_lens, wuk, wuv, w.causal, chunk, batches=batches)


@pytest.mark.parametrize("H,seq_lens,T,causal,chunk", [
    (16, [700, 1500, 0, 64], 3, True, 256),    # several windows, a ragged last window, an empty sequence
    (128, [1000, 300], 16, True, 128),         # the smallest window; the new rows span two windows
    (16, [600], 170, True, 512),               # two query tiles; the new rows span both windows
    (128, [257], 1, False, 1024),              # one window longer than the sequence
    (16, [4000, 130], 1, False, 384),          # a window not a power of two
])
def test_normal_chunked(mla, cuda, H, seq_lens, T, causal, chunk):
    """The chunked-prefix Normal path against the oracle's chunked restatement (and,
    through it, the one-shot Normal path)."""
    import torch
    from mla_latent_cache_gb300.runtime import NormalStep
    w = W.custom_workload(H, seq_lens, T=T, causal=causal, seed=43)
    st = NormalStep(w, device=cuda, chunk_rows=chunk)
    st.o.fill_(float("nan"))
    st.lse.fill_(float("nan"))
    st.step()
    torch.cuda.synchronize()
    status, _ = mla.mla_read_device_status(None)
    assert status == mla.MLA_OK, mla.mla_status_string(status)
    o_ref, lse_ref = _oracle_chunked(w, chunk)
    parity(_np(st.o), o_ref, f"chunked o (chunk {chunk})")
    parity(st.lse.cpu().numpy(), lse_ref, f"chunked lse (chunk {chunk})")
    one = NormalStep(w, device=cuda)
    one.step()
    torch.cuda.synchronize()
    parity(_np(st.o), _np(one.o), "chunked vs one-shot o")


@pytest.mark.parametrize("T", [16, 512])
def test_normal_chunked_extend_full_size_sampled_heads(mla, cuda, T):
    """The extend workload at full size through 2048-row windows (the expanded rows held
    at once drop from the whole prefix to one window), checked on sampled heads."""
    import torch
    from mla_latent_cache_gb300.runtime import NormalStep
    w = W.config_workload(5, T=T)
    st = NormalStep(w, device=cuda, chunk_rows=2048)
    assert st.kv_exp.numel() * 2 == w.H * w.B * 2048 * 512
    st.step()
    torch.cuda.synchronize()
    status, _ = mla.mla_read_device_status(None)
    assert status == mla.MLA_OK, mla.mla_status_string(status)
    heads = [3, 64]
    bs = [0, 5]
    o_ref, lse_ref = _oracle_chunked(w, 2048, batches=bs, heads=heads)
    o_got = _np(st.o)[:, :, heads]
    lse_got = st.lse.cpu().numpy()[:, :, heads]
    parity(o_got[bs], o_ref[bs], "chunked o (sampled heads)")
    parity(lse_got[bs], lse_ref[bs], "chunked lse (sampled heads)")
