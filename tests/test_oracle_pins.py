"""Pins for the float64 oracle: what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: printed
values (tests/golden), the Normal (decompressed) path as an independent
closed-form identity, a textbook library routine (torch SDPA in float64),
special cases with known answers, invariants of the exact split merge, and
brute force on tiny inputs.  Mutation tests plant each of the three bugs the
M5.8 page names (0x04 "Batched absorption trace") into oracle-built variants
and check that the identity pin catches them.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import mla_oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _rand_case(rng, H, S, T, d_c=O.D_C, d_r=O.D_R, d_n=O.D_N, d_v=O.D_V, page=O.PAGE, spare=2, qs=1.0):
    """Random float64 case with a shuffled block table over a slightly larger pool."""
    n_pages = max(1, -(-S // page))
    num_blocks = n_pages + spare
    pool = rng.normal(size=(num_blocks, page, d_c + d_r))
    perm = rng.permutation(num_blocks)[:n_pages]
    bt = perm.reshape(1, n_pages).astype(np.int64)
    q_nope = rng.normal(size=(1, T, H, d_n)) * qs
    q_pe = rng.normal(size=(1, T, H, d_r)) * qs
    w_uk = rng.normal(size=(H, d_n, d_c)) / math.sqrt(d_c)
    w_uv = rng.normal(size=(H, d_v, d_c)) / math.sqrt(d_c)
    return dict(pool=pool, bt=bt, seq_lens=np.array([S]), q_nope=q_nope, q_pe=q_pe, w_uk=w_uk, w_uv=w_uv,
                scale=1.0 / math.sqrt(d_n + d_r))


# ---------------------------------------------------------------------------
# printed values
# ---------------------------------------------------------------------------
def test_ledger_printed_values(golden_dir):
    g = _load(golden_dir, "ledger.json")
    assert O.latent_bytes_per_token() == g["latent_bytes_per_token_layer_f16"]["value"]
    assert O.decompressed_bytes_per_token(128) == g["decompressed_bytes_per_token_layer_v3_h128"]["value"]
    assert O.decompressed_bytes_per_token(16) == g["decompressed_bytes_per_token_layer_v2lite_h16"]["value"]
    assert round(O.decompressed_bytes_per_token(128) / O.latent_bytes_per_token(), 1) == g["ratio_v3"]["value"]
    assert round(O.decompressed_bytes_per_token(16) / O.latent_bytes_per_token(), 1) == g["ratio_v2lite"]["value"]
    assert 61 * O.latent_bytes_per_token() == g["latent_bytes_per_token_61_layers"]["value"]
    assert 61 * O.decompressed_bytes_per_token(128) / 2**20 == g["expanded_mib_per_token_61_layers"]["value"]
    assert 60 * O.decompressed_bytes_per_token(128) / 2**20 == g["v2_naive_mib_per_token_60_layers"]["value"]
    assert 60 * O.latent_bytes_per_token() / 2**10 == g["v2_latent_kib_per_token_60_layers"]["value"]
    assert 4096 * 60 * O.decompressed_bytes_per_token(128) / 2**30 == g["v2_naive_gib_at_4096"]["value"]
    assert 4096 * 60 * O.latent_bytes_per_token() / 2**20 == g["v2_latent_mib_at_4096"]["value"]
    assert 2 * O.normal_upproj_macs(1) == g["naive_expansion_flops_per_context_token"]["value"]


def test_mac_formulas_printed(golden_dir):
    g = _load(golden_dir, "ledger.json")
    coef = g["upproj_mac_coefficient_per_row"]["value"]
    # Normal expands S rows, Absorb folds T rows; both coefficients are the same ~16.8M
    assert O.normal_upproj_macs(1) == coef
    assert O.absorb_upproj_macs(1) == coef
    assert O.normal_upproj_macs(4096) == 4096 * 512 * 128 * 256
    assert O.absorb_upproj_macs(7) == 7 * 2 * 128 * 128 * 512
    # attention inflation 1088/320 and the two per-pair constants in the crossover denominator
    assert O.absorb_attention_macs(1, 1) == 139264 and O.normal_attention_macs(1, 1) == 40960
    assert round(O.absorb_attention_macs(1, 1) / O.normal_attention_macs(1, 1), 1) == g["attention_inflation"]["value"]
    # crossover T ~ 16.8M / (139264 - 40960) ~ 170.67 as S grows; below 171 for every S
    t_inf = coef / (139264 - 40960)
    assert round(t_inf, 2) == g["crossover_T"]["formula_value"]
    assert int(t_inf) == g["crossover_T"]["value"]
    for S in (8192, 65536, 1 << 22):
        t = O.crossover_T(S)
        assert t < t_inf and t_inf - t < t_inf * 170.0 / S * 1.01
    assert abs(O.crossover_T(1 << 30) - t_inf) < 1e-3


def test_core_flops_and_intensity_printed(golden_dir):
    g = _load(golden_dir, "ledger.json")
    pairs = O.visible_pairs(4096, 1, causal=False)
    core = O.decode_core_flops(128, pairs)
    assert core == 2 * 128 * 4096 * 1088 == 1_140_850_688
    assert round(core / 1e9, 2) == g["core_gflop_v3_s4096_t1"]["value"]
    bmm = 2 * O.absorb_upproj_macs(1)
    assert round(bmm / 1e6, 2) == g["absorb_bmm_mflop_v3_t1"]["value"]
    assert bmm / core < 0.03
    assert round(61 * core / 1e9, 1) == g["v3_61_layers_s4096_gflop"]["value"]
    assert round(61 * 4096 * O.latent_bytes_per_token() / 1e6, 1) == g["v3_61_layers_s4096_cache_mb"]["value"]
    assert round(O.decode_intensity(128)) == g["decode_intensity_v3"]["value"]
    assert abs(O.decode_intensity(128) / 128 - 1088 / 576) < 1e-12


def test_causal_pair_count_printed(golden_dir):
    g = _load(golden_dir, "ledger.json")
    P, Q = 5, 3
    assert O.visible_pairs(P + Q, Q, causal=True) == g["causal_pairs_prefix5_q3"]["value"]
    for P, Q in [(0, 1), (0, 4), (7, 1), (64, 17), (8192, 64)]:
        assert O.visible_pairs(P + Q, Q, causal=True) == P * Q + Q * (Q + 1) // 2
        assert O.visible_pairs(P + Q, Q, causal=False) == (P + Q) * Q


# ---------------------------------------------------------------------------
# paged address translation
# ---------------------------------------------------------------------------
def test_paged_gather_golden(golden_dir):
    g = _load(golden_dir, "paged_gather.json")
    c0 = g["cases"][0]
    page = c0["page"]
    bt = np.array(c0["block_table"])
    pool = np.arange(len(bt) * page * 2, dtype=np.float64).reshape(len(bt), page, 2)  # row id in column 0
    pool[..., 0] = np.arange(len(bt) * page).reshape(len(bt), page)
    rows = O.gather_rows(pool, bt, c0["seq_len"])
    assert rows[:, 0].astype(int).tolist() == c0["physical_rows"]
    c1 = g["cases"][1]
    bt1 = np.array(c1["block_table"])
    for j, phys in c1["probe"].items():
        assert O.physical_row(bt1, int(j), c1["page"]) == phys
    with pytest.raises(IndexError):
        O.physical_row(np.array([3, -1]), 64, 64)


def test_paged_gather_brute_force():
    rng = np.random.default_rng(5)
    for page in (1, 3, 64):
        nb = 9
        pool = rng.normal(size=(nb, page, 4))
        bt = rng.permutation(nb)[:5]
        S = 5 * page - (page // 2)
        rows = O.gather_rows(pool, bt, S)
        flat = pool.reshape(-1, 4)
        for j in range(S):
            assert np.array_equal(rows[j], flat[bt[j // page] * page + j % page])


def test_decompress_brute_force_and_absorption_identity():
    """decompress_ref against explicit loops on tiny ranks, and the absorption
    identity q_nope . (W_UK c) == (q_nope W_UK) . c that ties W_UK's orientation."""
    rng = np.random.default_rng(12)
    H, dn, dv, dc, S = 2, 3, 2, 5, 4
    c = rng.normal(size=(S, dc))
    w_uk = rng.normal(size=(H, dn, dc))
    w_uv = rng.normal(size=(H, dv, dc))
    k, v = O.decompress_ref(c, w_uk, w_uv)
    assert k.shape == (S, H, dn) and v.shape == (S, H, dv)
    for j in range(S):
        for h in range(H):
            for n in range(dn):
                assert abs(k[j, h, n] - sum(w_uk[h, n, x] * c[j, x] for x in range(dc))) < 1e-12
            for m in range(dv):
                assert abs(v[j, h, m] - sum(w_uv[h, m, x] * c[j, x] for x in range(dc))) < 1e-12
    q = rng.normal(size=(1, 1, H, dn))
    q_lat = O.absorb_ref(q, w_uk)[0, 0]                  # [H, dc]
    lhs = np.einsum("hn,jhn->jh", q[0, 0], k)
    rhs = np.einsum("hc,jc->jh", q_lat, c)
    assert np.max(np.abs(lhs - rhs)) < 1e-12


# ---------------------------------------------------------------------------
# closed-form identity: absorbed == Normal (decompressed) path
# ---------------------------------------------------------------------------
def _identity_err(c, T, causal, absorbed_fn=None):
    if absorbed_fn is None:
        o_a, _, lse_a, _ = O.absorbed_layer_ref(c["q_nope"], c["q_pe"], c["pool"], c["bt"], c["seq_lens"],
                                                 c["w_uk"], c["w_uv"], causal, c["scale"])
    else:
        o_a, lse_a = absorbed_fn(c, causal)
    o_n, lse_n = O.normal_ref(c["q_nope"], c["q_pe"], c["pool"], c["bt"], c["seq_lens"], c["w_uk"], c["w_uv"],
                              causal, c["scale"])
    err_o = np.max(np.abs(o_a - o_n)) / np.max(np.abs(o_n))
    fin = np.isfinite(lse_n)
    err_l = np.max(np.abs(lse_a[fin] - lse_n[fin])) if fin.any() else 0.0
    return err_o, err_l


@pytest.mark.parametrize("H", [1, 2, 16])
@pytest.mark.parametrize("S", [1, 2, 5, 63, 64, 65])
@pytest.mark.parametrize("T", [1, 3])
def test_absorbed_equals_normal_small_ranks(H, S, T):
    if T > S:
        pytest.skip("T new rows must fit in S")
    rng = np.random.default_rng(1000 * H + 10 * S + T)
    c = _rand_case(rng, H, S, T, d_c=8, d_r=4, d_n=3, d_v=5, page=4)
    for causal in (False, True):
        e_o, e_l = _identity_err(c, T, causal)
        assert e_o < 1e-12 and e_l < 1e-12


@pytest.mark.parametrize("H,S,T", [(1, 65, 1), (2, 64, 3), (16, 129, 3)])
def test_absorbed_equals_normal_full_width(H, S, T):
    rng = np.random.default_rng(H + S + T)
    c = _rand_case(rng, H, S, T)
    for causal in (False, True):
        e_o, e_l = _identity_err(c, T, causal)
        assert e_o < 1e-12 and e_l < 1e-12


# Mutation tests: each of the three bugs named in M5.8 0x04 must break the identity.
def _mut_softmax_over_heads(c, causal):
    q_lat = O.absorb_ref(c["q_nope"], c["w_uk"])
    S = int(c["seq_lens"][0])
    T = q_lat.shape[1]
    rows = O.gather_rows(c["pool"], c["bt"][0], S)
    d_c = q_lat.shape[-1]
    s = (np.einsum("thc,jc->thj", q_lat[0], rows[:, :d_c]) + np.einsum("thr,jr->thj", c["q_pe"][0], rows[:, d_c:])) * c["scale"]
    s = np.where(O.causal_mask(S, T, causal)[:, None, :], s, -np.inf)
    p, lse = O.softmax_rows(np.swapaxes(s, 1, 2))   # planted: normalise over heads
    p = np.swapaxes(p, 1, 2)
    o_lat = np.einsum("thj,jc->thc", p, rows[:, :d_c])[None]
    return O.unabsorb_ref(o_lat, c["w_uv"]), O.decode_ref(q_lat, c["q_pe"], c["pool"], c["bt"], c["seq_lens"], causal, c["scale"])[1]


def _mut_shared_latent_out(c, causal):
    q_lat = O.absorb_ref(c["q_nope"], c["w_uk"])
    o_lat, lse = O.decode_ref(q_lat, c["q_pe"], c["pool"], c["bt"], c["seq_lens"], causal, c["scale"])
    o_lat = np.broadcast_to(o_lat[:, :, :1, :], o_lat.shape)   # planted: head 0's latent output for all heads
    return O.unabsorb_ref(o_lat, c["w_uv"]), lse


def _mut_dc_transposed(c, causal):
    q_lat = O.absorb_ref(c["q_nope"], c["w_uk"])
    o_lat, lse = O.decode_ref(q_lat, c["q_pe"], c["pool"], c["bt"], c["seq_lens"], causal, c["scale"])
    return O.unabsorb_ref(o_lat, c["w_uv"][..., ::-1]), lse   # planted: d_c order differs in W_UV


@pytest.mark.parametrize("mutant", [_mut_softmax_over_heads, _mut_shared_latent_out, _mut_dc_transposed])
def test_named_bugs_break_identity(mutant):
    rng = np.random.default_rng(77)
    c = _rand_case(rng, 4, 37, 2, d_c=16, d_r=4, d_n=6, d_v=5, page=8, qs=3.0)
    e_o, _ = _identity_err(c, 2, False, absorbed_fn=mutant)
    assert e_o > 1e-3


# ---------------------------------------------------------------------------
# special cases and a textbook routine
# ---------------------------------------------------------------------------
def test_single_row_and_zero_query():
    rng = np.random.default_rng(3)
    c = _rand_case(rng, 4, 1, 1)
    q_lat = rng.normal(size=(1, 1, 4, O.D_C))
    o, lse = O.decode_ref(q_lat, c["q_pe"], c["pool"], c["bt"], c["seq_lens"], False)
    row = c["pool"].reshape(-1, O.D_K)[c["bt"][0, 0] * O.PAGE]
    assert np.array_equal(o[0, 0], np.broadcast_to(row[:O.D_C], (4, O.D_C)))
    s = (q_lat[0, 0] @ row[:O.D_C] + c["q_pe"][0, 0] @ row[O.D_C:]) * O.SCALE
    assert np.allclose(lse[0, 0], s, rtol=0, atol=1e-12)
    # zero query: uniform weights -> mean of the latent rows, lse = ln S
    for S in (5, 64, 130):
        c = _rand_case(rng, 3, S, 1)
        z_lat = np.zeros((1, 1, 3, O.D_C))
        z_pe = np.zeros((1, 1, 3, O.D_R))
        o, lse = O.decode_ref(z_lat, z_pe, c["pool"], c["bt"], c["seq_lens"], False)
        rows = O.gather_rows(c["pool"], c["bt"][0], S)
        assert np.allclose(o[0, 0], rows[:, :O.D_C].mean(axis=0), rtol=0, atol=1e-13)
        assert np.allclose(lse, math.log(S), rtol=0, atol=1e-13)


def test_textbook_sdpa_float64():
    """Absorbed decode is MQA with d_k = 576, d_v = 512: compare with torch's SDPA in float64."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(11)
    for H, S, T, causal in [(1, 70, 1, False), (16, 200, 1, False), (8, 131, 5, True)]:
        c = _rand_case(rng, H, S, T)
        q_lat = rng.normal(size=(1, T, H, O.D_C)) * 0.2
        o, _ = O.decode_ref(q_lat, c["q_pe"], c["pool"], c["bt"], c["seq_lens"], causal)
        rows = O.gather_rows(c["pool"], c["bt"][0], S)
        q = torch.from_numpy(np.concatenate([q_lat[0], c["q_pe"][0]], -1)).permute(1, 0, 2)  # [H,T,576]
        k = torch.from_numpy(rows)[None].expand(H, S, O.D_K)
        v = torch.from_numpy(rows[:, :O.D_C])[None].expand(H, S, O.D_C)
        mask = torch.from_numpy(O.causal_mask(S, T, causal))[None].expand(H, T, S) if causal else None
        ref = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=O.SCALE)
        assert np.allclose(o[0], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# exact split merge
# ---------------------------------------------------------------------------
def test_split_invariance_and_negative_controls():
    rng = np.random.default_rng(21)
    H, S, T = 8, 1000, 3
    c = _rand_case(rng, H, S, T, qs=3.0)
    q_lat = rng.normal(size=(1, T, H, O.D_C))
    for causal in (False, True):
        full_o, full_l = O.decode_ref(q_lat, c["q_pe"], c["pool"], c["bt"], c["seq_lens"], causal)
        n = -(-S // O.PAGE)
        for trial in range(5):
            cuts = sorted(set([0, n] + list(rng.integers(1, n, size=trial + 1))))
            parts = [O.partial_ref(q_lat[0], c["q_pe"][0], c["pool"], c["bt"][0], S, T, causal, a, b)
                     for a, b in zip(cuts[:-1], cuts[1:])]
            po = np.stack([p[0] for p in parts])
            pl = np.stack([p[1] for p in parts])
            mo, ml = O.merge_ref(po, pl)
            assert np.max(np.abs(mo - full_o[0])) < 1e-12 * max(1.0, np.max(np.abs(full_o)))
            assert np.max(np.abs(ml - full_l[0])) < 1e-12 * 100
            if len(parts) > 1:
                # averaging partial outputs is wrong
                assert np.max(np.abs(po.mean(0) - full_o[0])) > 1e-3
                # natural-log lse merged as if it were log2 must fail (the mlxcel negative control)
                m = pl.max(0)
                w = np.exp2(pl - m)
                bad = (w[..., None] * po).sum(0) / w.sum(0)[..., None]
                assert np.max(np.abs(bad - full_o[0])) > 1e-4


def test_merge_empty_partials():
    o, l = O.merge_ref(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(l))
    o, l = O.merge_ref(np.zeros((0, 2, 4)), np.zeros((0, 2)))
    assert np.all(o == 0) and np.all(np.isneginf(l))
    po = np.stack([np.ones((2, 4)), np.zeros((2, 4))])
    pl = np.stack([np.full(2, 0.5), np.full(2, -np.inf)])
    o, l = O.merge_ref(po, pl)
    assert np.allclose(o, 1.0) and np.allclose(l, 0.5)


# ---------------------------------------------------------------------------
# split planner: brute-force properties of the stated rule
# ---------------------------------------------------------------------------
def _check_plan(seq_lens, T, H, causal, G, N):
    plan = O.plan_ref(seq_lens, T, H, causal, G, N)
    groups = O.group_pages(seq_lens, T, H, causal)
    segs = plan["segments"]
    # every group's pages covered exactly once, in order, by its segments
    for (b, rb, n) in groups:
        mine = [s for s in segs if s[0] == b and s[1] == rb]
        covered = []
        for s in mine:
            assert s[2] < s[3]
            covered.extend(range(s[2], s[3]))
        assert covered == list(range(n))
        if len(mine) == 1:
            assert mine[0][5] == -1
        else:
            assert all(s[5] >= 0 for s in mine)
    # slots numbered in segment order
    slots = [s[5] for s in segs if s[5] >= 0]
    assert slots == list(range(plan["num_partials"]))
    # range pointers
    rp = plan["range_ptr"]
    assert rp[0] == 0 and rp[-1] == len(segs) and len(rp) == plan["num_ranges"] + 1
    for r in range(plan["num_ranges"]):
        assert all(segs[i][4] == r for i in range(rp[r], rp[r + 1]))
    # merge list: exactly the groups without a single final segment
    for (b, rb, n) in groups:
        entry = [m for m in plan["merge"] if m[0] == b and m[1] == rb]
        nseg = len([s for s in segs if s[0] == b and s[1] == rb])
        if n == 0:
            assert entry == [(b, rb, 0, 0)]
        elif nseg == 1:
            assert entry == []
        else:
            assert len(entry) == 1 and entry[0][3] == nseg
    if N > 0:
        for (b, rb, n) in groups:
            assert len([s for s in segs if s[0] == b and s[1] == rb]) == min(n, N) if n else True
    else:
        W = sum(n for (_, _, n) in groups)
        q = max(O.MIN_SPLIT_PAGES, -(-W // G))
        nonempty = [g for g in groups if g[2] > 0]
        loads = [0] * max(1, plan["num_ranges"])
        starts = [0] * max(1, plan["num_ranges"])
        for s in segs:
            loads[s[4]] += s[3] - s[2]
            starts[s[4]] += s[2] == 0
        assert plan["num_ranges"] <= G
        if len(nonempty) <= G and max((g[2] for g in nonempty), default=0) <= -(-5 * q // 4):
            # one whole group per range
            assert all(s[2] == 0 and s[5] == -1 for s in segs) and len(segs) == len(nonempty)
        else:
            # a range's work (pages + c per group starting in it, the first group's
            # start free) fits in q' line positions plus the one gap it may begin with
            c = O.SEGMENT_COST_PAGES
            qw = max(O.MIN_SPLIT_PAGES, -(-(W + c * (len(nonempty) - 1)) // G))
            for r in range(plan["num_ranges"]):
                assert loads[r] <= qw
                assert loads[r] + c * starts[r] <= qw + c
    return plan


def test_plan_gap_rule_worked_examples():
    """The balanced rule's line of pages and gaps, worked by hand (T=1, H=128: one
    group of ceil(S/64) pages per sequence; c = 8)."""
    assert O.SEGMENT_COST_PAGES == 8
    # pages [10, 2, 2, 10], G=3: W=24, q=8; 4 groups > 3 -> balanced.  U = 24 + 3*8 =
    # 48, q' = 16.  Line: g0 [0,10) gap g1 [18,20) gap g2 [28,30) gap g3 [38,48);
    # ranges [0,16) [16,32) [32,48) -> g0 | g1 g2 | g3, nothing cut (the old rule,
    # ranges of 8 pages, cut g0 and g3 and put four groups in the middle range).
    p = O.plan_ref([640, 128, 128, 640], 1, 128, False, 3)
    assert p["segments"] == [(0, 0, 0, 10, 0, -1), (1, 0, 0, 2, 1, -1), (2, 0, 0, 2, 1, -1), (3, 0, 0, 10, 2, -1)]
    assert p["range_ptr"] == [0, 1, 3, 4] and p["merge"] == []
    # pages [1, 6], G=10: W=7, q=4, 6 > ceil(5*4/4)=5 -> balanced.  U = 7 + 8 = 15,
    # q' = max(4, 2) = 4.  Line: g0 [0,1) gap [1,9) g1 [9,15); ranges [0,4) [4,8)
    # [8,12) [12,16): g0 | (inside the gap: empty) | g1 pages 0-3 | g1 pages 3-6.
    p = O.plan_ref([64, 384], 1, 128, False, 10)
    assert p["segments"] == [(0, 0, 0, 1, 0, -1), (1, 0, 0, 3, 2, 0), (1, 0, 3, 6, 3, 1)]
    assert p["num_ranges"] == 4 and p["range_ptr"] == [0, 1, 1, 2, 3] and p["merge"] == [(1, 0, 0, 2)]
    # five one-page groups, G=4: W=5, 5 groups > 4 -> balanced.  U = 5 + 4*8 = 37,
    # q' = 10.  Pages at 0, 9, 18, 27, 36 -> ranges g0 g1 | g2 | g3 | g4.
    p = O.plan_ref([64] * 5, 1, 128, False, 4)
    assert [s[4] for s in p["segments"]] == [0, 0, 1, 2, 3] and p["range_ptr"] == [0, 2, 3, 4, 5]


def test_plan_properties_random():
    rng = np.random.default_rng(8)
    for trial in range(60):
        B = int(rng.integers(1, 40))
        lens = rng.integers(0, 5000, size=B)
        T = int(rng.choice([1, 1, 2, 16]))
        lens = np.maximum(lens, T) if trial % 3 else lens
        H = int(rng.choice([16, 128]))
        G = int(rng.choice([1, 7, 76, 148, 152]))
        N = int(rng.choice([0, 0, 0, 3, 64]))
        _check_plan(lens, T, H, bool(trial % 2) and T > 1, G, N)


def test_plan_named_workloads():
    # uniform V3 batch on 152 slots: 4096 pages -> q = 27 (64 > ceil(5*27/4): split);
    # with the 63 gaps of 8 between sequences, 4600 positions in ranges of q' = 31
    p = _check_plan([4096] * 64, 1, 128, False, 152, 0)
    assert p["num_ranges"] == 149 and p["num_partials"] > 64
    # one long sequence: no gap, 2048 pages in 76 ranges of 27 (the last 23)
    p = _check_plan([131072], 1, 128, False, 76, 0)
    assert p["num_ranges"] == 76 and [s[3] - s[2] for s in p["segments"]] == [27] * 75 + [23]
    # on 76 slots it fits without splitting (64 <= ceil(5*54/4))
    p = _check_plan([4096] * 64, 1, 128, False, 76, 0)
    assert p["num_partials"] == 0 and p["num_ranges"] == 64
    # long context with explicit split counts: 2048 pages in N chunks of 2048/N
    for N in (64, 128, 256):
        p = _check_plan([131072], 1, 128, False, 152, N)
        assert p["num_partials"] == N and all(s[3] - s[2] == 2048 // N for s in p["segments"])
    # extend: T=16 new rows, H=128 -> 16 row blocks per sequence, causal page counts
    g = O.group_pages([8192 + 16], 16, 128, True)
    assert len(g) == 16 and g[0][2] == -(-(8192 + 1) // 64) and g[-1][2] == -(-(8192 + 16) // 64)
