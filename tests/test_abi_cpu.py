"""The C ABI loads and exports every symbol include/mla.h declares; host-side validation (no GPU needed)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "mla.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(mla):
    names = _declared()
    assert "mla_decode" in names and "mla_absorb_q" in names and "mla_split_merge" in names
    lib = ctypes.CDLL(mla.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"libmla.so does not export {n}"
    assert set(mla.EXPORTED) >= set(names)


def test_status_strings(mla):
    for code in range(-8, 1):
        s = mla.mla_status_string(code)
        assert s and s != "unknown status"
    assert mla.mla_status_string(17) == "unknown status"


def test_workspace_size_host_only(mla):
    g = mla.make_geom(128)
    b = mla.make_batch(64, 1, False, 64, num_slots=152)
    ws = mla.mla_workspace_size(g, b)
    # 2*G partial slots of 128 x 512 fp32 dominate
    assert ws >= 2 * 152 * 128 * 512 * 4
    assert ws % 256 == 0
    b2 = mla.make_batch(1, 1, False, 2048, num_slots=152, num_splits_override=256)
    assert mla.mla_workspace_size(g, b2) >= 256 * 128 * 512 * 4
    # invalid geometry / batch -> 0
    assert mla.mla_workspace_size(mla.make_geom(96), b) == 0
    bad = mla.make_batch(4, 0, False, 8, num_slots=4)
    assert mla.mla_workspace_size(g, bad) == 0


def test_host_validation_rejects_before_launch(mla):
    g = mla.make_geom(16)
    # null pointers are rejected on the host before any CUDA call
    assert mla.mla_absorb_q(g, None, None, None, 4, 0) == mla.MLA_ERR_ARG
    assert mla.mla_unabsorb_o(g, None, None, None, 4, 0) == mla.MLA_ERR_ARG
    assert mla.mla_absorb_q(g, 0x1000, 0x2000, 0x3008, 4, 0) == mla.MLA_ERR_ALIGN
    # outputs written with 32-byte stores must be 32-byte aligned (16 is not enough)
    assert mla.mla_absorb_q(g, 0x1000, 0x2000, 0x3010, 4, 0) == mla.MLA_ERR_ALIGN
    assert mla.mla_unabsorb_o(g, 0x1000, 0x2000, 0x3010, 4, 0) == mla.MLA_ERR_ALIGN
    assert mla.mla_absorb_q(mla.make_geom(24), 0x1000, 0x2000, 0x3000, 4, 0) == mla.MLA_ERR_SHAPE
    assert mla.mla_absorb_q(g, 0x1000, 0x2000, 0x3000, 0, 0) == mla.MLA_OK  # nothing to do
    b = mla.make_batch(2, 1, False, 8, num_slots=4)
    assert mla.mla_plan(g, b, None, None, 0, 0) == mla.MLA_ERR_ARG
    assert mla.mla_plan(g, b, 0x1000, 0x2000, 16, 0) == mla.MLA_ERR_WORKSPACE
    cache = mla.mla_cache(0x1000, 0x1400, 576, 64 * 576, 576, 64 * 576, 8)
    assert mla.mla_decode(g, b, None, None, cache, None, 8, None, 0, None, None, None, 0, 0) == mla.MLA_ERR_ARG
    bad_cache = mla.mla_cache(0x1000, 0x1402, 576, 64 * 576, 576, 64 * 576, 8)
    assert mla.mla_decode(g, b, 0x1000, 0x2000, bad_cache, 0x3000, 8, 0x4000, 0, 0x5000, 0x6000, 0x7000,
                          1 << 30, 0) == mla.MLA_ERR_ALIGN
    assert mla.mla_split_merge(None, None, None, 2, 4, 12, None, None, 0) == mla.MLA_ERR_ARG
    assert mla.mla_split_merge(0x1000, 0x2000, 0x3000, 0, 4, 16, 0x4000, 0x5000, 0) == mla.MLA_OK
    # every pointer of the merge is checked, the LSE arrays included
    assert mla.mla_split_merge(0x1000, 0x2004, 0x3000, 2, 4, 16, 0x4000, 0x5000, 0) == mla.MLA_ERR_ALIGN
    assert mla.mla_split_merge(0x1000, 0x2000, 0x3000, 2, 4, 16, 0x4000, 0x5004, 0) == mla.MLA_ERR_ALIGN
    # the gather export: a path other than 0 or 1, or a misaligned output, is refused
    assert mla.mla_debug_gather(cache, 0x1000, 8, 0x2000, 0, 2, 0x3000, 0) == mla.MLA_ERR_ARG
    assert mla.mla_debug_gather(cache, 0x1000, 8, 0x2000, 0, 0, 0x3008, 0) == mla.MLA_ERR_ALIGN
    # the no-alloc decode runs every decode argument check before launching anything
    assert mla.mla_decode_noalloc(g, b, None, None, cache, None, 8, None, None, None, 0) == mla.MLA_ERR_ARG
    assert mla.mla_decode_noalloc(g, b, 0x1000, 0x2000, bad_cache, 0x3000, 8, 0x4000, 0x5000, 0x6000,
                                  0) == mla.MLA_ERR_ALIGN
    assert mla.mla_decode_noalloc(g, b, 0x1000, 0x2000, cache, 0x3000, 4, 0x4000, 0x5000, 0x6000,
                                  0) == mla.MLA_ERR_ARG     # block-table row narrower than max_pages
    assert mla.mla_decode_noalloc(g, b, 0x1000, 0x2000, cache, 0x3000, 8, 0x4000, 0x5010, 0x6000,
                                  0) == mla.MLA_ERR_ALIGN   # o_lat is written with 32-byte stores
    # FP8 cache rows: output present and 16-byte aligned, cache valid
    assert mla.mla_fp8_pack_cache(cache, None, 0) == mla.MLA_ERR_ARG
    assert mla.mla_fp8_pack_cache(cache, 0x3008, 0) == mla.MLA_ERR_ALIGN
    assert mla.mla_fp8_pack_cache(bad_cache, 0x3000, 0) == mla.MLA_ERR_ALIGN
    empty = mla.mla_cache(0x1000, 0x1400, 576, 64 * 576, 576, 64 * 576, 0)
    assert mla.mla_fp8_pack_cache(empty, 0x3000, 0) == mla.MLA_ERR_ARG


def test_fp8_decode_host_side(mla):
    g = mla.make_geom(128)
    b = mla.make_batch(2, 1, False, 8, num_slots=4)
    ws = mla.mla_workspace_size(g, b)
    ok = [0x10000, 0x20000, 0x30000, 16, 0x40000, 8, 0x50000, 0, 0x60000, 0x70000, 0x80000, ws]

    def call(i=None, v=None, batch=b):
        a = list(ok)
        if i is not None:
            a[i] = v
        return mla.mla_decode_fp8(g, batch, *a, 0)

    assert call(2, None) == mla.MLA_ERR_ARG          # no FP8 cache
    assert call(3, 0) == mla.MLA_ERR_ARG             # no blocks
    assert call(5, 4) == mla.MLA_ERR_ARG             # block-table row narrower than max_pages
    assert call(2, 0x30008) == mla.MLA_ERR_ALIGN     # the cache rows are read by TMA
    assert call(8, 0x60010) == mla.MLA_ERR_ALIGN     # o_lat is written with 32-byte stores
    assert call(11, ws - 1) == mla.MLA_ERR_WORKSPACE
    assert call(batch=mla.make_batch(0, 1, False, 8, num_slots=4)) == mla.MLA_OK


def test_sparse_decode_host_side(mla):
    g = mla.make_geom(128)
    b = mla.make_batch(4, 2, False, 1, num_slots=8)
    # the workspace is that of a dense decode over B * S_q one-token sequences of ceil(topk / 64) pages
    vb = mla.make_batch(8, 1, False, 32, num_slots=8)
    assert mla.mla_sparse_workspace_size(g, b, 2048) == mla.mla_workspace_size(g, vb)
    assert mla.mla_sparse_workspace_size(g, b, 2047) == mla.mla_workspace_size(g, vb)
    assert mla.mla_sparse_workspace_size(g, b, 0) == 0
    assert mla.mla_sparse_workspace_size(g, mla.make_batch(4, 2, True, 1, num_slots=8), 64) == 0  # causal refused
    cache = mla.mla_cache(0x1000, 0x1400, 576, 64 * 576, 576, 64 * 576, 8)
    ws = mla.mla_sparse_workspace_size(g, b, 2048)
    ok = dict(q_lat=0x10000, q_pe=0x20000, indices=0x30000, topk_length=0x40000, o_lat=0x50000, lse=0x60000,
              workspace=0x70000)

    def call(cache=cache, batch=b, topk=2048, ws_bytes=ws, **kw):
        a = {**ok, **kw}
        return mla.mla_decode_sparse(g, batch, a["q_lat"], a["q_pe"], cache, a["indices"], topk, a["topk_length"], 0,
                                     a["o_lat"], a["lse"], a["workspace"], ws_bytes, 0)

    assert call(indices=None) == mla.MLA_ERR_ARG
    assert call(topk_length=None) == mla.MLA_ERR_ARG
    assert call(topk=0) == mla.MLA_ERR_ARG
    assert call(batch=mla.make_batch(4, 2, True, 1, num_slots=8)) == mla.MLA_ERR_ARG
    assert call(indices=0x30004) == mla.MLA_ERR_ALIGN
    assert call(o_lat=0x50010) == mla.MLA_ERR_ALIGN
    assert call(ws_bytes=ws - 1) == mla.MLA_ERR_WORKSPACE
    # blocks that are not evenly spaced rows cannot be indexed as one row array
    gapped = mla.mla_cache(0x1000, 0x1400, 576, 64 * 576 + 8, 576, 64 * 576 + 8, 8)
    assert call(cache=gapped) == mla.MLA_ERR_ARG
    assert call(cache=mla.mla_cache(0x1000, 0x1402, 576, 64 * 576, 576, 64 * 576, 8)) == mla.MLA_ERR_ALIGN
    assert call(batch=mla.make_batch(0, 2, False, 1, num_slots=8)) == mla.MLA_OK  # nothing to do


def test_normal_arm_host_side(mla):
    g = mla.make_geom(128)
    assert mla.mla_normal_rows_per_seq(1) == 128 and mla.mla_normal_rows_per_seq(2) == 128
    assert mla.mla_normal_rows_per_seq(137) == 69 * 128 and mla.mla_normal_rows_per_seq(0) == 0
    assert mla.mla_normal_expanded_bytes(g, 8, 136) == 128 * 8 * 68 * 128 * 256 * 2
    assert mla.mla_normal_expanded_bytes(mla.make_geom(96), 8, 136) == 0
    cache = mla.mla_cache(0x1000, 0x1400, 576, 64 * 576, 576, 64 * 576, 8)
    # null pointers and misalignment are rejected on the host before any CUDA call
    assert mla.mla_normal_expand(g, cache, None, 8, None, 2, 8, None, None, None, 0) == mla.MLA_ERR_ARG
    assert mla.mla_normal_expand(g, cache, 0x1000, 4, 0x2000, 2, 8, 0x3000, 0x4000, 0x5000, 0) == mla.MLA_ERR_ARG
    assert mla.mla_normal_expand(g, cache, 0x1000, 8, 0x2000, 2, 8, 0x3000, 0x4000, 0x5008, 0) == mla.MLA_ERR_ALIGN
    assert mla.mla_normal_expand(g, cache, 0x1000, 8, 0x2000, 0, 8, 0x3000, 0x4000, 0x5000, 0) == mla.MLA_OK
    b = mla.make_batch(2, 16, True, 8)
    assert mla.mla_normal_attention(g, b, None, None, cache, None, 8, None, None, None, None, 0) == mla.MLA_ERR_ARG
    assert mla.mla_normal_attention(g, b, 0x1000, 0x2000, cache, 0x3000, 8, 0x4000, 0x5000, 0x6000, 0x7004,
                                    0) == mla.MLA_ERR_ALIGN
    assert mla.mla_normal_attention(mla.make_geom(24), b, 0x1000, 0x2000, cache, 0x3000, 8, 0x4000, 0x5000, 0x6000,
                                    0x7000, 0) == mla.MLA_ERR_SHAPE


def test_normal_chunked_host_side(mla):
    g = mla.make_geom(128)
    # one window of expanded rows per sequence, and the fp32 running state
    assert mla.mla_normal_chunk_bytes(g, 8, 2048) == 128 * 8 * 2048 * 256 * 2
    assert mla.mla_normal_chunk_bytes(g, 8, 200) == 0 and mla.mla_normal_chunk_bytes(g, 8, 0) == 0
    b = mla.make_batch(2, 16, True, 8)
    assert mla.mla_normal_chunk_state_bytes(g, b) >= 2 * 16 * 128 * (128 + 1) * 4
    cache = mla.mla_cache(0x1000, 0x1400, 576, 64 * 576, 576, 64 * 576, 8)
    ok = [0x10000, 0x20000, cache, 0x30000, 8, 0x40000, 0x50000, 0x60000, 256, 0x70000, 0x80000, 0x90000, 0xA0000]

    def call(i=None, v=None, batch=b):
        a = list(ok)
        if i is not None:
            a[i] = v
        return mla.mla_normal_chunked(g, batch, *a, 0)

    assert call(8, 200) == mla.MLA_ERR_ARG     # window not a multiple of 128
    assert call(8, 0) == mla.MLA_ERR_ARG
    assert call(0, None) == mla.MLA_ERR_ARG
    assert call(10, None) == mla.MLA_ERR_ARG   # no state buffer
    assert call(4, 4) == mla.MLA_ERR_ARG       # block-table row narrower than max_pages
    assert call(10, 0x80010) == mla.MLA_ERR_ALIGN
    assert call(9, 0x70010) == mla.MLA_ERR_ALIGN
    assert call(batch=mla.make_batch(0, 16, True, 8)) == mla.MLA_OK
