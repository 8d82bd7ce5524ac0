"""ctypes binding of libmla.so (include/mla.h): argument marshalling only.

Every step of the hot path runs in the library's CUDA kernels.  Functions keep
the C names and return the C status code; ``check`` turns a status into an
exception.  Tensors are passed as raw device pointers; PyTorch is used only
for device memory and streams.  If libmla.so is missing this module raises at
import time: there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla.so")

MLA_OK = 0
MLA_ERR_ARG = -1
MLA_ERR_SHAPE = -2
MLA_ERR_ALIGN = -3
MLA_ERR_WORKSPACE = -4
MLA_ERR_PLAN_STALE = -5
MLA_ERR_CUDA = -6
MLA_ERR_DEVICE_CHECK = -7
MLA_ERR_TIMEOUT = -8

# plan header word indices (include/mla.h)
HDR = dict(MAGIC=0, B=1, T=2, H=3, CAUSAL=4, NUM_GROUPS=5, NUM_SEGMENTS=6, NUM_RANGES=7, NUM_PARTIALS=8,
           NUM_MERGE=9, SEQ_HASH=10, ERROR=11, ERROR_INFO=12, PAGES_PER_RANGE=13, NUM_SLOTS=14, OVERRIDE=15,
           MAX_PAGES=16, OFF_SEGMENTS=17, OFF_RANGE_PTR=18, OFF_MERGE=19, OFF_PART_LSE=20, OFF_PART_O=21,
           CAP_SEGMENTS=22, CAP_PARTIALS=23, CAP_RANGES=24, CAP_GROUPS=25)
HDR_WORDS = 64
PLAN_MAGIC = 0x4D4C4131


class mla_geom(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("d_lat", ctypes.c_int), ("d_rope", ctypes.c_int), ("d_nope", ctypes.c_int),
                ("d_v", ctypes.c_int), ("block_size", ctypes.c_int), ("softmax_scale", ctypes.c_float)]


class mla_cache(ctypes.Structure):
    _fields_ = [("ckv", ctypes.c_void_p), ("kpe", ctypes.c_void_p), ("ckv_row_stride", ctypes.c_int64),
                ("ckv_block_stride", ctypes.c_int64), ("kpe_row_stride", ctypes.c_int64),
                ("kpe_block_stride", ctypes.c_int64), ("num_blocks", ctypes.c_int)]


class mla_batch(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("causal", ctypes.c_int), ("max_pages", ctypes.c_int),
                ("num_slots", ctypes.c_int), ("num_splits_override", ctypes.c_int)]


class MlaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {mla_status_string(status)} ({status})" if what else mla_status_string(status))


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmla.so is not built ({LIB_PATH}); run mla_latent_cache_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    I = ctypes.c_int
    G = ctypes.POINTER(mla_geom)
    C = ctypes.POINTER(mla_cache)
    Bt = ctypes.POINTER(mla_batch)
    sig = {
        "mla_workspace_size": (ctypes.c_size_t, [G, Bt]),
        "mla_plan": (I, [G, Bt, P, P, ctypes.c_size_t, P]),
        "mla_absorb_q": (I, [G, P, P, P, I, P]),
        "mla_unabsorb_o": (I, [G, P, P, P, I, P]),
        "mla_decode": (I, [G, Bt, P, P, C, P, I, P, I, P, P, P, ctypes.c_size_t, P]),
        "mla_decode_noalloc": (I, [G, Bt, P, P, C, P, I, P, P, P, P]),
        "mla_sparse_workspace_size": (ctypes.c_size_t, [G, Bt, I]),
        "mla_decode_fp8": (I, [G, Bt, P, P, P, I, P, I, P, I, P, P, P, ctypes.c_size_t, P]),
        "mla_decode_sparse": (I, [G, Bt, P, P, C, P, I, P, I, P, P, P, ctypes.c_size_t, P]),
        "mla_split_merge": (I, [P, P, P, I, I, I, P, P, P]),
        "mla_debug_gather": (I, [C, P, I, P, I, I, P, P]),
        "mla_debug_set_wait_limit": (I, [ctypes.c_longlong]),
        "mla_fp8_pack_cache": (I, [C, P, P]),
        "mla_normal_rows_per_seq": (ctypes.c_int64, [I]),
        "mla_normal_expanded_bytes": (ctypes.c_size_t, [G, I, I]),
        "mla_normal_expand": (I, [G, C, P, I, P, I, I, P, P, P, P]),
        "mla_normal_attention": (I, [G, Bt, P, P, C, P, I, P, P, P, P, P]),
        "mla_normal_chunk_bytes": (ctypes.c_size_t, [G, I, I]),
        "mla_normal_chunk_state_bytes": (ctypes.c_size_t, [G, Bt]),
        "mla_normal_chunked": (I, [G, Bt, P, P, C, P, I, P, P, P, I, P, P, P, P, P]),
        "mla_read_device_status": (I, [P, ctypes.POINTER(ctypes.c_int), P]),
        "mla_status_string": (ctypes.c_char_p, [I]),
        "mla_device_sm_count": (I, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
EXPORTED = ("mla_workspace_size", "mla_plan", "mla_absorb_q", "mla_unabsorb_o", "mla_decode", "mla_decode_noalloc",
            "mla_sparse_workspace_size", "mla_decode_sparse", "mla_decode_fp8",
            "mla_split_merge", "mla_normal_rows_per_seq", "mla_normal_expanded_bytes", "mla_normal_expand",
            "mla_normal_attention", "mla_normal_chunk_bytes", "mla_normal_chunk_state_bytes", "mla_normal_chunked",
            "mla_fp8_pack_cache", "mla_debug_gather", "mla_debug_set_wait_limit", "mla_read_device_status",
            "mla_status_string",
            "mla_device_sm_count")


def lib() -> ctypes.CDLL:
    return _lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_geom(H: int, softmax_scale: float | None = None) -> mla_geom:
    return mla_geom(H, 512, 64, 128, 128, 64, 1.0 / math.sqrt(192.0) if softmax_scale is None else softmax_scale)


def make_batch(B: int, T: int, causal: bool, max_pages: int, num_slots: int = 0, num_splits_override: int = 0) -> mla_batch:
    return mla_batch(B, T, 1 if causal else 0, max_pages, num_slots, num_splits_override)


def cache_from_pool(pool) -> mla_cache:
    """A combined [num_blocks, 64, 576] bf16 pool (contiguous)."""
    nb, page, width = pool.shape
    base = pool.data_ptr()
    return mla_cache(base, base + 512 * 2, width, page * width, width, page * width, nb)


def cache_from_split(ckv, kpe) -> mla_cache:
    """Separate latent [num_blocks, 64, 512] and RoPE [num_blocks, 64, 64] pools."""
    nb = ckv.shape[0]
    return mla_cache(ckv.data_ptr(), kpe.data_ptr(), ckv.stride(1), ckv.stride(0), kpe.stride(1), kpe.stride(0), nb)


def check(status: int, what: str = "") -> None:
    if status != MLA_OK:
        raise MlaError(status, what)


# ---------------------------------------------------------------------------
# the C entry points, same names
# ---------------------------------------------------------------------------
def mla_status_string(status: int) -> str:
    return _lib.mla_status_string(int(status)).decode()


def mla_device_sm_count() -> int:
    return int(_lib.mla_device_sm_count())


def mla_workspace_size(geom: mla_geom, batch: mla_batch) -> int:
    return int(_lib.mla_workspace_size(ctypes.byref(geom), ctypes.byref(batch)))


def mla_plan(geom, batch, seq_lens, workspace, ws_bytes: int, stream=None) -> int:
    return _lib.mla_plan(ctypes.byref(geom), ctypes.byref(batch), _ptr(seq_lens), _ptr(workspace), ws_bytes,
                         _stream(stream))


def mla_absorb_q(geom, q_nope, w_uk, q_lat, BT: int, stream=None) -> int:
    return _lib.mla_absorb_q(ctypes.byref(geom), _ptr(q_nope), _ptr(w_uk), _ptr(q_lat), BT, _stream(stream))


def mla_unabsorb_o(geom, o_lat, w_uv, o, BT: int, stream=None) -> int:
    return _lib.mla_unabsorb_o(ctypes.byref(geom), _ptr(o_lat), _ptr(w_uv), _ptr(o), BT, _stream(stream))


def mla_decode(geom, batch, q_lat, q_pe, cache: mla_cache, block_table, bt_stride: int, seq_lens, checked: int,
               o_lat, lse, workspace, ws_bytes: int, stream=None) -> int:
    return _lib.mla_decode(ctypes.byref(geom), ctypes.byref(batch), _ptr(q_lat), _ptr(q_pe), ctypes.byref(cache),
                           _ptr(block_table), bt_stride, _ptr(seq_lens), int(checked), _ptr(o_lat), _ptr(lse),
                           _ptr(workspace), ws_bytes, _stream(stream))


def mla_decode_noalloc(geom, batch, q_lat, q_pe, cache: mla_cache, block_table, bt_stride: int, seq_lens, o_lat, lse,
                       stream=None) -> int:
    """Plan + decode in the library's fixed device scratch (for callers that cannot allocate)."""
    return _lib.mla_decode_noalloc(ctypes.byref(geom), ctypes.byref(batch), _ptr(q_lat), _ptr(q_pe),
                                   ctypes.byref(cache), _ptr(block_table), bt_stride, _ptr(seq_lens), _ptr(o_lat),
                                   _ptr(lse), _stream(stream))


NOALLOC_SCRATCH_BYTES = 32 << 20


def mla_decode_fp8(geom, batch, q_lat, q_pe, cache_fp8, num_blocks: int, block_table, bt_stride: int, seq_lens,
                   checked: int, o_lat, lse, workspace, ws_bytes: int, stream=None) -> int:
    """Decode over the FP8 cache rows (uint8 [num_blocks, 64, 656]); plan with mla_plan first."""
    return _lib.mla_decode_fp8(ctypes.byref(geom), ctypes.byref(batch), _ptr(q_lat), _ptr(q_pe), _ptr(cache_fp8),
                               int(num_blocks), _ptr(block_table), bt_stride, _ptr(seq_lens), int(checked),
                               _ptr(o_lat), _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream))


def mla_sparse_workspace_size(geom, batch, topk: int) -> int:
    return _lib.mla_sparse_workspace_size(ctypes.byref(geom), ctypes.byref(batch), int(topk))


def mla_decode_sparse(geom, batch, q_lat, q_pe, cache: mla_cache, indices, topk: int, topk_length, checked: int,
                      o_lat, lse, workspace, ws_bytes: int, stream=None) -> int:
    """Plan + decode over listed physical rows indices [B, S_q, topk] (lengths topk_length [B])."""
    return _lib.mla_decode_sparse(ctypes.byref(geom), ctypes.byref(batch), _ptr(q_lat), _ptr(q_pe),
                                  ctypes.byref(cache), _ptr(indices), int(topk), _ptr(topk_length), int(checked),
                                  _ptr(o_lat), _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream))


def mla_split_merge(part_o, part_lse, indptr, M: int, rows: int, D: int, o, lse, stream=None) -> int:
    return _lib.mla_split_merge(_ptr(part_o), _ptr(part_lse), _ptr(indptr), M, rows, D, _ptr(o), _ptr(lse),
                                _stream(stream))


def mla_fp8_pack_cache(cache: mla_cache, out, stream=None) -> int:
    return _lib.mla_fp8_pack_cache(ctypes.byref(cache), _ptr(out), _stream(stream))


def mla_debug_gather(cache: mla_cache, block_table, bt_stride: int, seq_lens, b: int, path: int, out,
                     stream=None) -> int:
    """Copy sequence b's logical rows through the decode kernel's own page loads
    (path 0: page-half boxes; path 1: latent columns through the reload boxes)."""
    return _lib.mla_debug_gather(ctypes.byref(cache), _ptr(block_table), bt_stride, _ptr(seq_lens), b, int(path),
                                 _ptr(out), _stream(stream))


def mla_debug_set_wait_limit(cycles: int) -> int:
    """Limit of the decode kernel's pipeline waits on the current device (<= 0: the default)."""
    return _lib.mla_debug_set_wait_limit(int(cycles))


def mla_normal_rows_per_seq(max_pages: int) -> int:
    return int(_lib.mla_normal_rows_per_seq(max_pages))


def mla_normal_expanded_bytes(geom: mla_geom, B: int, max_pages: int) -> int:
    return int(_lib.mla_normal_expanded_bytes(ctypes.byref(geom), B, max_pages))


def mla_normal_expand(geom, cache: mla_cache, block_table, bt_stride: int, seq_lens, B: int, max_pages: int, w_uk,
                      w_uv, kv_exp, stream=None) -> int:
    return _lib.mla_normal_expand(ctypes.byref(geom), ctypes.byref(cache), _ptr(block_table), bt_stride,
                                  _ptr(seq_lens), B, max_pages, _ptr(w_uk), _ptr(w_uv), _ptr(kv_exp), _stream(stream))


def mla_normal_attention(geom, batch, q_nope, q_pe, cache: mla_cache, block_table, bt_stride: int, seq_lens, kv_exp,
                         o, lse, stream=None) -> int:
    return _lib.mla_normal_attention(ctypes.byref(geom), ctypes.byref(batch), _ptr(q_nope), _ptr(q_pe),
                                     ctypes.byref(cache), _ptr(block_table), bt_stride, _ptr(seq_lens), _ptr(kv_exp),
                                     _ptr(o), _ptr(lse), _stream(stream))


def mla_normal_chunk_bytes(geom, B: int, chunk_rows: int) -> int:
    return _lib.mla_normal_chunk_bytes(ctypes.byref(geom), B, chunk_rows)


def mla_normal_chunk_state_bytes(geom, batch) -> int:
    return _lib.mla_normal_chunk_state_bytes(ctypes.byref(geom), ctypes.byref(batch))


def mla_normal_chunked(geom, batch, q_nope, q_pe, cache: mla_cache, block_table, bt_stride: int, seq_lens, w_uk,
                       w_uv, chunk_rows: int, kv_chunk, state, o, lse, stream=None) -> int:
    """The Normal path with the prefix expanded and attended chunk_rows rows at a time (LSE-merged)."""
    return _lib.mla_normal_chunked(ctypes.byref(geom), ctypes.byref(batch), _ptr(q_nope), _ptr(q_pe),
                                   ctypes.byref(cache), _ptr(block_table), bt_stride, _ptr(seq_lens), _ptr(w_uk),
                                   _ptr(w_uv), int(chunk_rows), _ptr(kv_chunk), _ptr(state), _ptr(o), _ptr(lse),
                                   _stream(stream))


def mla_read_device_status(workspace, stream=None) -> tuple[int, int]:
    info = ctypes.c_int(0)
    st = _lib.mla_read_device_status(_ptr(workspace), ctypes.byref(info), _stream(stream))
    return int(st), int(info.value)
