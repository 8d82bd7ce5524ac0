"""Pins of the oracle's references for two "next" rows: sparse index-driven
decode ("M5.8" 0x0B physical indices with a valid-prefix length) and the
chunked-prefix Normal path (zdszero "路径选择", MHA_CHUNKED_KV)."""
import numpy as np

from oracle import mla_oracle as O


def _setup(seed, H=4, lens=(70, 129, 1), T=1, nb=12):
    rng = np.random.default_rng(seed)
    B = len(lens)
    pool = rng.standard_normal((nb, 64, 576)) * 0.1
    pages = [(s + 63) // 64 for s in lens]
    perm = rng.permutation(nb)
    bt = np.full((B, max(pages)), -1, dtype=np.int64)
    k = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[k:k + n]
        k += n
    q_lat = rng.standard_normal((B, T, H, 512)) * 0.3
    q_pe = rng.standard_normal((B, T, H, 64)) * 0.3
    return rng, pool, bt, np.array(lens), q_lat, q_pe


def _phys(bt_row, S):
    return np.array([O.physical_row(bt_row, j) for j in range(S)], dtype=np.int64)


def test_sparse_listing_every_row_equals_dense():
    rng, pool, bt, lens, q_lat, q_pe = _setup(1)
    topk = int(lens.max())
    idx = np.zeros((len(lens), 1, topk), dtype=np.int64)
    for b, S in enumerate(lens):
        idx[b, 0, :S] = rng.permutation(_phys(bt[b], S))          # any order
    o, l = O.sparse_decode_ref(q_lat, q_pe, pool, idx, topk_length=lens)
    od, ld = O.decode_ref(q_lat, q_pe, pool, bt, lens, causal=False)
    np.testing.assert_allclose(o, od, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l, ld, rtol=1e-12)


def test_sparse_prefix_duplicates_and_empty():
    rng, pool, bt, lens, q_lat, q_pe = _setup(2, lens=(100, 100))
    rows = _phys(bt[0], 100)
    idx = np.stack([rows[:10], rows[:10]])[:, None, :]            # [2, 1, 10]
    # entries past topk_length are ignored, whatever they hold
    idx_junk = idx.copy()
    idx_junk[:, :, 6:] = 10 ** 9
    o1, l1 = O.sparse_decode_ref(q_lat, q_pe, pool, idx, topk_length=np.array([6, 0]))
    o2, l2 = O.sparse_decode_ref(q_lat, q_pe, pool, idx_junk, topk_length=np.array([6, 0]))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # an empty list: o = 0, lse = -inf
    assert np.all(o1[1] == 0) and np.all(l1[1] == -np.inf)
    # a row listed twice counts twice: same output, lse + ln 2
    one = np.array([[[rows[3]]]] * 2)
    two = np.array([[[rows[3], rows[3]]]] * 2)
    oa, la = O.sparse_decode_ref(q_lat, q_pe, pool, one)
    ob, lb = O.sparse_decode_ref(q_lat, q_pe, pool, two)
    np.testing.assert_allclose(oa, ob, rtol=1e-13)
    np.testing.assert_allclose(lb, la + np.log(2.0), rtol=1e-13)
    # a single listed row is returned exactly (its latent), lse = its score
    c = pool[rows[3] // 64, rows[3] % 64]
    assert np.allclose(oa[0, 0], np.broadcast_to(c[:512], oa[0, 0].shape), rtol=0, atol=1e-15)
    s = (q_lat[0, 0] @ c[:512] + q_pe[0, 0] @ c[512:]) * O.SCALE
    np.testing.assert_allclose(la[0, 0], s, rtol=1e-13)


def test_chunked_normal_equals_one_shot():
    rng = np.random.default_rng(3)
    H, T = 3, 5
    _, pool, bt, lens, _, _ = _setup(3, H=H, lens=(70, 140, 0, 5), T=T)
    lens = np.maximum(lens, np.where(lens > 0, T, 0))
    q_nope = rng.standard_normal((len(lens), T, H, 128)) * 0.3
    q_pe = rng.standard_normal((len(lens), T, H, 64)) * 0.3
    w_uk = rng.standard_normal((H, 128, 512)) / np.sqrt(512)
    w_uv = rng.standard_normal((H, 128, 512)) / np.sqrt(512)
    for causal in (False, True):
        ref_o, ref_l = O.normal_ref(q_nope, q_pe, pool, bt, lens, w_uk, w_uv, causal)
        for chunk in (1, 7, 64, 100, 1000):
            o, l = O.normal_chunked_ref(q_nope, q_pe, pool, bt, lens, w_uk, w_uv, causal, chunk)
            np.testing.assert_allclose(o, ref_o, rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(l, ref_l, rtol=1e-12)
    # and the chunked Normal path equals the absorbed path (the identity the pages rest on)
    ab_o, _, ab_l, _ = O.absorbed_layer_ref(q_nope, q_pe, pool, bt, lens, w_uk, w_uv, True)
    o, l = O.normal_chunked_ref(q_nope, q_pe, pool, bt, lens, w_uk, w_uv, True, 33)
    np.testing.assert_allclose(o, ab_o, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(l, ab_l, rtol=1e-12)
