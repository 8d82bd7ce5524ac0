"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Floating-point outputs (q_lat, o_lat, lse, o) must satisfy
max|err| <= 2e-2 max|ref| and sum|err|/sum|ref| <= 5e-3 (tests/_tol.py);
the split plan and the paged gather must be bit-exact.
"""
import numpy as np
import pytest

from oracle import mla_oracle as O
from mla_latent_cache_gb300 import workloads as W
from tests._tol import parity

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


def _f64(u16):
    return W.bf16_bits_to_f64(u16)


def _to_np(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def _oracle_decode(w, batches=None, tokens=None):
    """Oracle o_lat/lse for the listed sequences (and tokens) of a workload, from its own bf16 inputs.
    Each sequence's rows are gathered as bf16 bit patterns and widened after the gather
    (the same values as widening the whole pool first)."""
    pool, bt = w.compact_view()
    q_lat = _f64(w.q_lat)
    q_pe = _f64(w.q_pe)
    out = {}
    for b in (range(w.B) if batches is None else batches):
        S = int(w.seq_lens[b])
        ts = list(range(w.T)) if tokens is None else list(tokens)
        if S == 0:
            out[b] = (np.zeros((len(ts), w.H, 512)), np.full((len(ts), w.H), -np.inf))
            continue
        rows = _f64(O.gather_rows(pool, bt[b], S))
        mask = O.causal_mask(S, w.T, w.causal)[ts]
        out[b] = O.attend_latent(q_lat[b, ts], q_pe[b, ts], rows, mask)
    return out


def _oracle_partials(w, b, segments):
    """The oracle's partial states (o_r normalised, lse_r) of sequence b over the given page ranges."""
    pool, bt = w.compact_view()
    S = int(w.seq_lens[b])
    rows = _f64(O.gather_rows(pool, bt[b], S))
    q_lat, q_pe = _f64(w.q_lat)[b], _f64(w.q_pe)[b]
    mask = O.causal_mask(S, w.T, w.causal)
    parts_o, parts_l = [], []
    for p0, p1 in segments:
        j0, j1 = 64 * p0, min(S, 64 * p1)
        o, l = O.attend_latent(q_lat, q_pe, rows[j0:j1], mask[:, j0:j1])
        parts_o.append(o)
        parts_l.append(l)
    return np.stack(parts_o), np.stack(parts_l)


def _run_decode(mla, w, cuda, num_slots=0, override=0, checked=False):
    from mla_latent_cache_gb300.runtime import DecodeStep
    st = DecodeStep(w, device=cuda, num_slots=num_slots, num_splits_override=override, checked=checked,
                    with_absorb=False)
    st.plan()
    st.decode()
    import torch
    torch.cuda.synchronize()
    status, info = mla.mla_read_device_status(st.workspace)
    assert status == mla.MLA_OK, (mla.mla_status_string(status), info)
    return st


def _compare(st, w, batches=None, tokens=None, name=""):
    ref = _oracle_decode(w, batches, tokens)
    o_lat = _to_np(st.o_lat)
    lse = _to_np(st.lse)
    ts = slice(None) if tokens is None else list(tokens)
    bs = sorted(ref)
    ro = np.stack([ref[b][0] for b in bs])
    rl = np.stack([ref[b][1] for b in bs])
    go = np.stack([o_lat[b][ts] for b in bs])
    gl = np.stack([lse[b][ts] for b in bs])
    parity(go, ro, f"{name} o_lat")
    parity(gl, rl, f"{name} lse")


# ---------------------------------------------------------------------------
# planner and gather: bit-exact
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["c1", "c2", "c2_76", "c3", "c4_auto", "c4_64", "c4_256", "c5_16", "c5_170", "rand",
                                  "gap", "gap5"])
def test_plan_bit_exact(mla, cuda, case):
    import torch
    from mla_latent_cache_gb300.runtime import read_plan_header, read_plan_tables
    rng = np.random.default_rng(4)
    spec = {
        "c1": (W.config_workload(1), 0, 0), "c2": (W.config_workload(2), 0, 0),
        "c2_76": (W.config_workload(2), 76, 0), "c3": (W.config_workload(3), 0, 0),
        "c4_auto": (W.config_workload(4), 0, 0), "c4_64": (W.config_workload(4), 0, 64),
        "c4_256": (W.config_workload(4), 0, 256), "c5_16": (W.config_workload(5, T=16), 0, 0),
        "c5_170": (W.config_workload(5, T=170), 0, 0),
        "rand": (W.custom_workload(16, list(rng.integers(0, 3000, size=37)) + [0, 1, 64, 65], T=2, causal=True),
                 13, 0),
        # a work range inside a gap of the balanced rule (no segment), and one-page groups
        "gap": (W.custom_workload(128, [64, 384]), 10, 0), "gap5": (W.custom_workload(128, [64] * 5), 4, 0),
    }[case]
    w, slots, ov = spec
    geom = mla.make_geom(w.H)
    batch = mla.make_batch(w.B, w.T, w.causal, w.max_pages, slots, ov)
    ws_bytes = mla.mla_workspace_size(geom, batch)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=cuda)
    seq = torch.from_numpy(w.seq_lens).to(cuda)
    mla.check(mla.mla_plan(geom, batch, seq, ws, ws_bytes))
    torch.cuda.synchronize()
    G = slots if slots > 0 else mla.mla_device_sm_count() // 2
    ref = O.plan_ref(w.seq_lens, w.T, w.H, w.causal, G, ov)

    seg, rp, mg = read_plan_tables(torch, ws)
    assert seg.shape[0] == len(ref["segments"])
    assert [tuple(int(x) for x in r[:6]) for r in seg] == [tuple(r) for r in ref["segments"]]
    assert rp.tolist() == ref["range_ptr"]
    assert [tuple(int(x) for x in r) for r in mg] == [tuple(r) for r in ref["merge"]]
    hdr = read_plan_header(torch, ws)
    assert hdr[mla.HDR["NUM_PARTIALS"]] == ref["num_partials"]
    assert hdr[mla.HDR["ERROR"]] == 0 or case == "rand"


def test_decode_plan_with_empty_range(mla, cuda):
    """The balanced rule can leave a work range inside a gap (its CTA pair has no
    segment): the decode over that plan against the oracle, sharp logits."""
    w = W.custom_workload(128, [64, 384, 200, 3000], seed=31, sharp=True)
    st = _run_decode(mla, w, cuda, num_slots=40)
    _compare(st, w, name="plan with an empty range")


@pytest.mark.parametrize("slots,ov", [(0, 0), (19, 0), (0, 5)])
def test_plan_bit_exact_many_groups(mla, cuda, slots, ov):
    """More row groups (70 sequences x 64 row blocks) than the planner keeps in
    shared memory: the per-group segment path, compared bit for bit."""
    import torch
    from mla_latent_cache_gb300.runtime import read_plan_header, read_plan_tables
    rng = np.random.default_rng(11)
    B, T, H = 70, 64, 128
    seq_lens = rng.integers(T, 3000, size=B).astype(np.int32)
    max_pages = (3000 + 63) // 64
    geom = mla.make_geom(H)
    batch = mla.make_batch(B, T, True, max_pages, slots, ov)
    ws_bytes = mla.mla_workspace_size(geom, batch)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=cuda)
    seq = torch.from_numpy(seq_lens).to(cuda)
    mla.check(mla.mla_plan(geom, batch, seq, ws, ws_bytes))
    torch.cuda.synchronize()
    G = slots if slots > 0 else mla.mla_device_sm_count() // 2
    ref = O.plan_ref(seq_lens, T, H, True, G, ov)
    assert len(O.group_pages(seq_lens, T, H, True)) == B * 64 > 4096
    seg, rp, mg = read_plan_tables(torch, ws)
    assert [tuple(int(x) for x in r[:6]) for r in seg] == [tuple(r) for r in ref["segments"]]
    assert rp.tolist() == ref["range_ptr"]
    assert [tuple(int(x) for x in r) for r in mg] == [tuple(r) for r in ref["merge"]]
    hdr = read_plan_header(torch, ws)
    assert hdr[mla.HDR["NUM_PARTIALS"]] == ref["num_partials"] and hdr[mla.HDR["ERROR"]] == 0


def _gather_expected(w, cpool, cbt, b, S, bad_pages=()):
    """The oracle's gather of sequence b; pages whose block id is outside the pool read as zeros."""
    ref = O.gather_rows(cpool, np.where(cbt[b] >= 0, cbt[b], 0), S).copy()
    for p in bad_pages:
        ref[64 * p: 64 * (p + 1)] = 0
    return ref


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_gather_bit_exact(mla, cuda, cfg, split):
    """The decode kernel's own page loads (tensor maps, box coordinates from the block
    table, both the page-half boxes and the reload boxes) copy exactly the rows the
    oracle's paged gather names ("M5.8" 0x05), on combined and split pools."""
    import torch
    from mla_latent_cache_gb300.runtime import pool_to_device
    w = W.config_workload(cfg)
    pool = pool_to_device(torch, w, cuda)
    if split:
        ckv, kpe = pool[..., :512].contiguous(), pool[..., 512:].contiguous()   # kept alive for the raw pointers
        cache = mla.cache_from_split(ckv, kpe)
    else:
        cache = mla.cache_from_pool(pool)
    bt = torch.from_numpy(w.block_table).to(cuda)
    seq = torch.from_numpy(w.seq_lens).to(cuda)
    cpool, cbt = w.compact_view()
    picks = range(w.B) if w.B <= 64 else sorted({0, 1, w.B // 2, w.B - 1} | set(range(0, w.B, 9)))
    for b in picks:
        S = int(w.seq_lens[b])
        ref = _gather_expected(w, cpool, cbt, b, S)
        for path in (0, 1):
            out = torch.zeros((S, 576), dtype=torch.bfloat16, device=cuda)
            mla.check(mla.mla_debug_gather(cache, bt, bt.shape[1], seq, b, path, out))
            got = out.view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, ref), (b, path)
    status, _ = mla.mla_read_device_status(None)
    assert status == mla.MLA_OK


def test_gather_out_of_pool_ids_read_zeros(mla, cuda):
    """A block id outside [0, num_blocks) reads as zeros through the decode's maps; the
    other pages, including a ragged last page, are untouched."""
    import torch
    from mla_latent_cache_gb300.runtime import pool_to_device
    w = W.custom_workload(16, [700, 130], T=1, seed=19)
    pool = pool_to_device(torch, w, cuda)
    cache = mla.cache_from_pool(pool)
    bt_np = w.block_table.copy()
    bt_np[0, 2] = w.num_blocks + 7
    bt_np[0, 5] = -3
    bt = torch.from_numpy(bt_np).to(cuda)
    seq = torch.from_numpy(w.seq_lens).to(cuda)
    cpool, cbt = w.compact_view()
    for b, bad in [(0, (2, 5)), (1, ())]:
        S = int(w.seq_lens[b])
        ref = _gather_expected(w, cpool, cbt, b, S, bad)
        for path in (0, 1):
            out = torch.full((S, 576), float("nan"), dtype=torch.bfloat16, device=cuda)
            mla.check(mla.mla_debug_gather(cache, bt, bt.shape[1], seq, b, path, out))
            got = out.view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, ref), (b, path)


# ---------------------------------------------------------------------------
# decode against the oracle
# ---------------------------------------------------------------------------
def test_decode_tiny_config(mla, cuda):
    w = W.config_workload(1)
    st = _run_decode(mla, w, cuda)
    _compare(st, w, name="tiny")


@pytest.mark.parametrize("sharp", [False, True])
def test_decode_v3_uniform_all(mla, cuda, sharp):
    """Every one of the 64 sequences (one CTA pair each) compared element by element."""
    w = W.config_workload(2, sharp=sharp)
    st = _run_decode(mla, w, cuda)
    _compare(st, w, name=f"v3 uniform sharp={sharp}")


@pytest.mark.parametrize("sharp", [False, True])
def test_decode_v3_ragged_all(mla, cuda, sharp):
    """Every one of the 128 sequences: balanced page ranges that cut sequences at
    arbitrary pages, partial states merged by log-sum-exp."""
    w = W.config_workload(3, sharp=sharp)
    st = _run_decode(mla, w, cuda)
    hdr = st.plan_header()
    assert hdr[mla.HDR["NUM_PARTIALS"]] > 0        # the plan does split sequences
    _compare(st, w, name=f"v3 ragged sharp={sharp}")


@pytest.mark.parametrize("sharp", [False, True])
@pytest.mark.parametrize("override", [0, 64, 128, 256])
def test_decode_v3_long(mla, cuda, override, sharp):
    w = W.config_workload(4, sharp=sharp)
    st = _run_decode(mla, w, cuda, override=override)
    _compare(st, w, name=f"v3 long N={override} sharp={sharp}")


@pytest.mark.parametrize("override", [0, 64])
def test_long_sharp_merge_negative_controls(mla, cuda, override):
    """With peaked logits the partials' LSEs differ widely, so the tolerance separates
    the exact merge from the wrong ones the pages warn about ("M5.8" 0x0C: averaging
    per-split outputs is wrong; mlxcel Stage 2: weights are e^x of natural-log LSEs,
    not 2^x).  The wrong merges are built from the oracle's own partials for the
    device plan's segments (planted on the CPU); the device result, merged by the
    same plan, must pass where they fail."""
    from mla_latent_cache_gb300.runtime import read_plan_tables
    import torch
    w = W.config_workload(4, sharp=True)
    st = _run_decode(mla, w, cuda, override=override)
    seg, _, _ = read_plan_tables(torch, st.workspace)
    segments = [(int(r[2]), int(r[3])) for r in seg]
    assert len(segments) > 1
    po, pl = _oracle_partials(w, 0, segments)
    ref_o, ref_l = O.merge_ref(po, pl)
    parity(_to_np(st.o_lat)[0], ref_o, "device o_lat")
    parity(_to_np(st.lse)[0], ref_l, "device lse")
    avg = po.mean(axis=0)
    m = pl.max(axis=0)
    w2 = np.exp2(pl - m)
    log2_o = (w2[..., None] * po).sum(axis=0) / w2.sum(axis=0)[..., None]
    for name, bad in [("average", avg), ("2^x weights", log2_o)]:
        with pytest.raises(AssertionError):
            parity(bad, ref_o, name)


@pytest.mark.parametrize("T", [1, 16, 64, 170, 512])
def test_decode_v3_extend_sampled(mla, cuda, T):
    w = W.config_workload(5, T=T)
    st = _run_decode(mla, w, cuda)
    toks = sorted({0, T // 2, T - 1})
    _compare(st, w, batches=[0, 7], tokens=toks, name=f"extend T={T}")


@pytest.mark.parametrize("H", [16, 128])
@pytest.mark.parametrize("T,causal", [(1, False), (3, True), (3, False)])
def test_decode_page_boundaries(mla, cuda, H, T, causal):
    lens = [1, 63, 64, 65, 127, 128, 129, 4096, 0, 3]
    lens = [s for s in lens if s == 0 or s >= T]
    w = W.custom_workload(H, lens, T=T, causal=causal, seed=31 + H + T)
    for slots, ov in [(0, 0), (5, 0), (0, 3)]:
        st = _run_decode(mla, w, cuda, num_slots=slots, override=ov)
        _compare(st, w, name=f"edges H={H} T={T} slots={slots} ov={ov}")


def test_decode_sharp_softmax_tiny(mla, cuda):
    w = W.config_workload(1, sharp=True)
    st = _run_decode(mla, w, cuda)
    _compare(st, w, name="sharp tiny")


@pytest.mark.parametrize("H", [1, 2, 4, 8, 32, 64])
@pytest.mark.parametrize("T,causal", [(1, False), (3, True)])
def test_decode_head_counts(mla, cuda, H, T, causal):
    """Every head count the boundary accepts (128 % H == 0) besides 16 and 128: a
    128-row group then spans 128 / H tokens, or a token's rows split across groups."""
    lens = [1, 64, 65, 300, 1000, 3]
    lens = [s for s in lens if s >= T]
    w = W.custom_workload(H, lens, T=T, causal=causal, seed=41 + H + T, sharp=(H % 2 == 0))
    for slots, ov in [(0, 0), (3, 0), (0, 4)]:
        st = _run_decode(mla, w, cuda, num_slots=slots, override=ov)
        _compare(st, w, name=f"H={H} T={T} slots={slots} ov={ov}")


def test_decode_split_cache_layout(mla, cuda):
    """Separate latent and RoPE pools (FlashInfer-style ckv/kpe) give the same result."""
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    w = W.custom_workload(16, [300, 77], T=1, seed=5)
    st = DecodeStep(w, device=cuda, with_absorb=False, num_splits_override=2)
    ckv = st.pool[..., :512].contiguous()
    kpe = st.pool[..., 512:].contiguous()
    st.cache = mla.cache_from_split(ckv, kpe)
    st.plan()
    st.decode()
    torch.cuda.synchronize()
    _compare(st, w, name="split cache")


@pytest.mark.parametrize("split", [False, True])
def test_fp8_pack_cache_bit_exact(mla, cuda, split):
    """The 656-byte FP8 rows the CUDA writer packs ("M5.8" 0x0B) equal the
    oracle's byte for byte (codes, fp32 scales, RoPE), combined and split pools."""
    import torch
    rng = np.random.default_rng(21)
    nb = 24
    vals = (rng.standard_normal((nb, 64, 576)) * 0.1).astype(np.float32)
    vals[3, 5, 128:256] = 0.0                       # an all-zero tile: scale 1
    vals[7, :, :512] *= 1e-3                        # small tiles
    vals[9, 1, :512] = np.where(rng.random(512) < 0.5, -0.0, 0.0)   # signed zeros only
    vals[11, 2, 0] = 3.0                            # one dominant value: the rest of its tile goes subnormal
    bits = W.f32_to_bf16_bits(vals)
    pool = torch.from_numpy(bits.view(np.int16)).to(cuda).view(torch.bfloat16)
    if split:
        ckv, kpe = pool[..., :512].contiguous(), pool[..., 512:].contiguous()   # kept alive: the cache holds raw pointers
        cache = mla.cache_from_split(ckv, kpe)
    else:
        cache = mla.cache_from_pool(pool)
    out = torch.zeros((nb, 64, 656), dtype=torch.uint8, device=cuda)
    mla.check(mla.mla_fp8_pack_cache(cache, out))
    torch.cuda.synchronize()
    ref = O.fp8_row_quantize(W.bf16_bits_to_f32(bits[..., :512]), bits[..., 512:])
    got = out.cpu().numpy()
    assert np.array_equal(got[..., 512:], ref[..., 512:])     # scales and RoPE
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# absorption GEMMs and the whole chain
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", [1, 2])
def test_absorb_unabsorb(mla, cuda, cfg):
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    w = W.config_workload(cfg)
    st = DecodeStep(w, device=cuda)
    st.absorb()
    # un-absorb a drawn o_lat (the q_lat draw has the right shape and scale)
    o_lat_in = st.o_lat
    o_lat_in.copy_(torch.from_numpy(w.q_lat.view(np.int16)).to(cuda).view(torch.bfloat16))
    st.unabsorb()
    torch.cuda.synchronize()
    parity(_to_np(st.q_lat), O.absorb_ref(_f64(w.q_nope), _f64(w.w_uk)), "q_lat")
    parity(_to_np(st.o), O.unabsorb_ref(_f64(w.q_lat), _f64(w.w_uv)), "o")


@pytest.mark.parametrize("H,lens,T", [(1, [5, 200], 3), (2, [70], 1), (8, [300] * 3, 2), (32, [64] * 5, 1),
                                      (64, [129, 1, 1000], 3)])
def test_absorb_unabsorb_head_counts(mla, cuda, H, lens, T):
    """Every head count the boundary accepts (128 % H == 0), with token counts that
    leave the GEMMs' 128-token tiles ragged (B*T = 3 .. 15)."""
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    w = W.custom_workload(H, lens, T=T, causal=True, seed=57 + H)
    st = DecodeStep(w, device=cuda)
    st.absorb()
    st.o_lat.copy_(torch.from_numpy(w.q_lat.view(np.int16)).to(cuda).view(torch.bfloat16))
    st.unabsorb()
    torch.cuda.synchronize()
    parity(_to_np(st.q_lat), O.absorb_ref(_f64(w.q_nope), _f64(w.w_uk)), f"q_lat H={H}")
    parity(_to_np(st.o), O.unabsorb_ref(_f64(w.q_lat), _f64(w.w_uv)), f"o H={H}")


@pytest.mark.parametrize("cfg", [1, 2])
def test_full_chain(mla, cuda, cfg):
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    w = W.config_workload(cfg)
    st = DecodeStep(w, device=cuda)
    st.step()
    torch.cuda.synchronize()
    pool, bt = w.compact_view()
    bs = [0] if cfg == 1 else [0, 40]
    o, o_lat, lse, q_lat = O.absorbed_layer_ref(_f64(w.q_nope)[bs], _f64(w.q_pe)[bs], _f64(pool), bt[bs],
                                                w.seq_lens[bs], _f64(w.w_uk), _f64(w.w_uv), w.causal)
    parity(_to_np(st.q_lat)[bs], q_lat, "q_lat")
    parity(_to_np(st.o_lat)[bs], o_lat, "o_lat")
    parity(_to_np(st.lse)[bs], lse, "lse")
    parity(_to_np(st.o)[bs], o, "o")
    # and the decompressed Normal path gives the same o (the identity the oracle is pinned to)
    o_n, _ = O.normal_ref(_f64(w.q_nope)[bs], _f64(w.q_pe)[bs], _f64(pool), bt[bs], w.seq_lens[bs], _f64(w.w_uk),
                          _f64(w.w_uv), w.causal)
    parity(_to_np(st.o)[bs], o_n, "o vs normal")


# ---------------------------------------------------------------------------
# public merge, device checks
# ---------------------------------------------------------------------------
def test_split_merge_public(mla, cuda):
    import torch
    rng = np.random.default_rng(9)
    rows, D = 40, 512
    counts = [3, 1, 0, 5, 2]
    N = sum(counts)
    part_o = rng.normal(size=(N, rows, D)).astype(np.float32)
    part_lse = (rng.normal(size=(N, rows)) * 3).astype(np.float32)
    part_lse[1, :7] = -np.inf   # some empty partials
    part_lse[3] = -np.inf       # output 1's only partial is empty
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    d = lambda a: torch.from_numpy(a).to(cuda)
    o = torch.empty((len(counts), rows, D), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((len(counts), rows), dtype=torch.float32, device=cuda)
    mla.check(mla.mla_split_merge(d(part_o), d(part_lse), d(indptr), len(counts), rows, D, o, lse))
    torch.cuda.synchronize()
    for m in range(len(counts)):
        a, b = indptr[m], indptr[m + 1]
        ro, rl = O.merge_ref(part_o[a:b].astype(np.float64), part_lse[a:b].astype(np.float64))
        parity(_to_np(o[m]), ro, f"merge o[{m}]")
        parity(_to_np(lse[m]), rl, f"merge lse[{m}]")


def test_checked_mode_flags_bad_block_and_stale_plan(mla, cuda):
    import torch
    from mla_latent_cache_gb300.runtime import DecodeStep
    w = W.custom_workload(16, [200, 100], T=1, seed=12)
    st = DecodeStep(w, device=cuda, with_absorb=False, checked=True)
    st.plan()
    st.block_table[1, 0] = w.num_blocks + 5   # out of the pool
    st.decode()
    status, info = mla.mla_read_device_status(st.workspace)
    assert status == mla.MLA_ERR_DEVICE_CHECK and (info >> 16) == 1
    # a plan built for other lengths is flagged
    st.block_table.copy_(torch.from_numpy(w.block_table).to(cuda))
    st.plan()
    st.seq_lens[0] = 150
    st.decode()
    status, _ = mla.mla_read_device_status(st.workspace)
    assert status == mla.MLA_ERR_PLAN_STALE
    # a length beyond the block table is reported by the planner
    st.seq_lens[0] = w.max_pages * 64 + 1
    st.plan()
    status, info = mla.mla_read_device_status(st.workspace)
    assert status == mla.MLA_ERR_DEVICE_CHECK and info == 0
