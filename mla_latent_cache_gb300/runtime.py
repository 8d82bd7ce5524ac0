"""Device-side state for one decode step, built on the C ABI.

``DecodeStep`` owns the device buffers (PyTorch allocations) for one batch
shape and runs the hot path through libmla.so:
plan -> absorb (q_nope @ W_UK) -> split-KV latent attention (+ merge) ->
un-absorb (o_lat @ W_UV).  Nothing here computes: it allocates and marshals.
"""
from __future__ import annotations

import numpy as np

from . import binding as L
from .workloads import Workload


def _u16_to_bf16(torch, a: np.ndarray, device):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def pool_to_device(torch, w: Workload, device):
    """Materialise the [num_blocks, 64, 576] pool on the device (NaN outside the referenced blocks)."""
    pool = torch.full((w.num_blocks, 64, 576), float("nan"), dtype=torch.bfloat16, device=device)
    data = _u16_to_bf16(torch, w.pool_data, device)
    ids = torch.from_numpy(w.pool_ids).to(device)
    pool.index_copy_(0, ids, data)
    return pool


class DecodeStep:
    """cache_format "fp8": the bf16 pool is packed once into 656-byte FP8 rows
    (mla_fp8_pack_cache) and the decode reads those (mla_decode_fp8)."""

    def __init__(self, w: Workload, device="cuda", num_slots: int = 0, num_splits_override: int = 0,
                 checked: bool = False, with_absorb: bool = True, cache_format: str = "bf16"):
        import torch
        self.torch = torch
        self.w = w
        self.device = torch.device(device)
        self.geom = L.make_geom(w.H)
        self.batch = L.make_batch(w.B, w.T, w.causal, w.max_pages, num_slots, num_splits_override)
        self.checked = 1 if checked else 0
        dev = self.device
        self.pool = pool_to_device(torch, w, dev)
        self.cache = L.cache_from_pool(self.pool)
        self.cache_format = cache_format
        if cache_format == "fp8":
            self.pool_fp8 = torch.empty((w.num_blocks, 64, 656), dtype=torch.uint8, device=dev)
            L.check(L.mla_fp8_pack_cache(self.cache, self.pool_fp8), "mla_fp8_pack_cache")
        elif cache_format != "bf16":
            raise ValueError(f"cache_format {cache_format!r}")
        self.block_table = torch.from_numpy(w.block_table).to(dev)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(dev)
        self.q_pe = _u16_to_bf16(torch, w.q_pe, dev)
        if with_absorb:
            self.q_nope = _u16_to_bf16(torch, w.q_nope, dev)
            self.w_uk = _u16_to_bf16(torch, w.w_uk, dev)
            self.w_uv = _u16_to_bf16(torch, w.w_uv, dev)
            self.q_lat = torch.empty((w.B, w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
            self.o = torch.empty((w.B, w.T, w.H, 128), dtype=torch.bfloat16, device=dev)
        else:
            self.q_lat = _u16_to_bf16(torch, w.q_lat, dev)
        # The per-step inputs (query halves, lengths, block table) become views of one
        # device buffer, so that a step's host-to-device traffic can be one copy.
        parts = [n for n in ("q_nope", "q_pe", "seq_lens", "block_table") if hasattr(self, n)]
        offs, off = [], 0
        for n in parts:
            off = (off + 255) // 256 * 256
            offs.append(off)
            off += getattr(self, n).numel() * getattr(self, n).element_size()
        self.inputs = torch.empty(off, dtype=torch.uint8, device=dev)
        for n, o in zip(parts, offs):
            src = getattr(self, n)
            view = self.inputs[o: o + src.numel() * src.element_size()].view(src.dtype).view(src.shape)
            view.copy_(src)
            setattr(self, n, view)
        self._input_parts = list(zip(parts, offs))
        self.o_lat = torch.empty((w.B, w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.B, w.T, w.H), dtype=torch.float32, device=dev)
        self.ws_bytes = L.mla_workspace_size(self.geom, self.batch)
        if self.ws_bytes == 0:
            raise L.MlaError(L.MLA_ERR_ARG, "mla_workspace_size")
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)

    @property
    def BT(self) -> int:
        return self.w.B * self.w.T

    def io_set(self) -> dict:
        """The per-step input buffer (with its views) and output o of this step."""
        return {"inputs": self.inputs, "o": getattr(self, "o", None),
                **{n: getattr(self, n) for n, _ in self._input_parts}}

    def new_io_set(self) -> dict:
        """A second input buffer (same contents) and output, for double-buffered steps."""
        torch = self.torch
        inputs = self.inputs.clone()
        io = {"inputs": inputs, "o": torch.empty_like(self.o) if hasattr(self, "o") else None}
        for n, off in self._input_parts:
            src = getattr(self, n)
            io[n] = inputs[off: off + src.numel() * src.element_size()].view(src.dtype).view(src.shape)
        return io

    def bind(self, io: dict):
        """Point the step at an input/output set (the next calls use its buffers)."""
        self.inputs = io["inputs"]
        if io.get("o") is not None:
            self.o = io["o"]
        for n, _ in self._input_parts:
            setattr(self, n, io[n])

    def plan(self, stream=None):
        L.check(L.mla_plan(self.geom, self.batch, self.seq_lens, self.workspace, self.ws_bytes, stream), "mla_plan")

    def absorb(self, stream=None):
        L.check(L.mla_absorb_q(self.geom, self.q_nope, self.w_uk, self.q_lat, self.BT, stream), "mla_absorb_q")

    def decode(self, stream=None):
        if self.cache_format == "fp8":
            L.check(L.mla_decode_fp8(self.geom, self.batch, self.q_lat, self.q_pe, self.pool_fp8, self.w.num_blocks,
                                     self.block_table, self.block_table.shape[1], self.seq_lens, self.checked,
                                     self.o_lat, self.lse, self.workspace, self.ws_bytes, stream), "mla_decode_fp8")
            return
        L.check(L.mla_decode(self.geom, self.batch, self.q_lat, self.q_pe, self.cache, self.block_table,
                             self.block_table.shape[1], self.seq_lens, self.checked, self.o_lat, self.lse,
                             self.workspace, self.ws_bytes, stream), "mla_decode")

    def unabsorb(self, stream=None):
        L.check(L.mla_unabsorb_o(self.geom, self.o_lat, self.w_uv, self.o, self.BT, stream), "mla_unabsorb_o")

    def step(self, stream=None):
        """One pass of the whole hot path (plan, absorb, decode + merge, un-absorb)."""
        self.plan(stream)
        self.absorb(stream)
        self.decode(stream)
        self.unabsorb(stream)

    def plan_header(self):
        return read_plan_header(self.torch, self.workspace)

    def plan_tables(self):
        return read_plan_tables(self.torch, self.workspace)


def read_plan_header(torch, workspace):
    """The plan header words (include/mla.h) copied to the host."""
    return workspace[: L.HDR_WORDS * 4].view(torch.int32).cpu().numpy()


def read_plan_tables(torch, workspace):
    """(segments [n,8], range_ptr [n_ranges+1], merge [m,4]) copied from the workspace."""
    hdr = read_plan_header(torch, workspace)

    def words(off, n):
        return workspace[off: off + 4 * n].view(torch.int32).cpu().numpy()

    nseg = int(hdr[L.HDR["NUM_SEGMENTS"]])
    nr = int(hdr[L.HDR["NUM_RANGES"]])
    nm = int(hdr[L.HDR["NUM_MERGE"]])
    seg = words(int(hdr[L.HDR["OFF_SEGMENTS"]]), nseg * 8).reshape(nseg, 8)
    rp = words(int(hdr[L.HDR["OFF_RANGE_PTR"]]), nr + 1)
    mg = words(int(hdr[L.HDR["OFF_MERGE"]]), nm * 4).reshape(nm, 4)
    return seg, rp, mg


class SparseStep:
    """The index-driven decode (mla_decode_sparse) on one SparseWorkload: the
    absorbed query attends to the listed physical rows of the pool."""

    def __init__(self, sw, device="cuda", num_slots: int = 0, num_splits_override: int = 0, checked: bool = False):
        import torch
        self.torch = torch
        self.sw = sw
        w = sw.ctx
        dev = self.device = torch.device(device)
        self.geom = L.make_geom(w.H)
        self.batch = L.make_batch(w.B, w.T, False, 1, num_slots, num_splits_override)
        self.checked = 1 if checked else 0
        self.pool = pool_to_device(torch, w, dev)
        self.cache = L.cache_from_pool(self.pool)
        self.q_lat = _u16_to_bf16(torch, w.q_lat, dev)
        self.q_pe = _u16_to_bf16(torch, w.q_pe, dev)
        self.indices = torch.from_numpy(np.ascontiguousarray(sw.indices)).to(dev)
        self.topk_length = torch.from_numpy(np.ascontiguousarray(sw.topk_length)).to(dev)
        self.o_lat = torch.empty((w.B, w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.B, w.T, w.H), dtype=torch.float32, device=dev)
        self.ws_bytes = L.mla_sparse_workspace_size(self.geom, self.batch, sw.topk)
        if self.ws_bytes == 0:
            raise L.MlaError(L.MLA_ERR_ARG, "mla_sparse_workspace_size")
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)

    def decode(self, stream=None):
        L.check(L.mla_decode_sparse(self.geom, self.batch, self.q_lat, self.q_pe, self.cache, self.indices,
                                    self.sw.topk, self.topk_length, self.checked, self.o_lat, self.lse,
                                    self.workspace, self.ws_bytes, stream), "mla_decode_sparse")


class NormalStep:
    """The Normal (decompressed) arm on one workload: expand the latent cache into
    per-head keys and values (mla_normal_expand), then causal MHA over them
    (mla_normal_attention).  Inputs are q_nope / q_pe directly; no absorption."""

    def __init__(self, w: Workload, device="cuda", chunk_rows: int = 0):
        import torch
        self.torch = torch
        self.w = w
        self.device = torch.device(device)
        dev = self.device
        self.chunk_rows = int(chunk_rows)
        self.geom = L.make_geom(w.H)
        self.batch = L.make_batch(w.B, w.T, w.causal, w.max_pages)
        self.pool = pool_to_device(torch, w, dev)
        self.cache = L.cache_from_pool(self.pool)
        self.block_table = torch.from_numpy(w.block_table).to(dev)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(dev)
        self.q_nope = _u16_to_bf16(torch, w.q_nope, dev)
        self.q_pe = _u16_to_bf16(torch, w.q_pe, dev)
        self.w_uk = _u16_to_bf16(torch, w.w_uk, dev)
        self.w_uv = _u16_to_bf16(torch, w.w_uv, dev)
        if self.chunk_rows > 0:
            # chunked prefix: one window of expanded rows plus the running fp32 state
            self.rows_per_seq = self.chunk_rows
            nbytes = L.mla_normal_chunk_bytes(self.geom, w.B, self.chunk_rows)
            sbytes = L.mla_normal_chunk_state_bytes(self.geom, self.batch)
            if nbytes == 0 or sbytes == 0:
                raise L.MlaError(L.MLA_ERR_ARG, "mla_normal_chunk_bytes")
            self.state = torch.empty(sbytes, dtype=torch.uint8, device=dev)
        else:
            self.rows_per_seq = L.mla_normal_rows_per_seq(w.max_pages)
            nbytes = L.mla_normal_expanded_bytes(self.geom, w.B, w.max_pages)
            if nbytes == 0 and w.B > 0:
                raise L.MlaError(L.MLA_ERR_ARG, "mla_normal_expanded_bytes")
        self.kv_exp = torch.empty(max(1, nbytes // 2), dtype=torch.bfloat16, device=dev)
        self.o = torch.empty((w.B, w.T, w.H, 128), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.B, w.T, w.H), dtype=torch.float32, device=dev)

    def expand(self, stream=None):
        L.check(L.mla_normal_expand(self.geom, self.cache, self.block_table, self.block_table.shape[1], self.seq_lens,
                                    self.w.B, self.w.max_pages, self.w_uk, self.w_uv, self.kv_exp, stream),
                "mla_normal_expand")

    def attention(self, stream=None):
        L.check(L.mla_normal_attention(self.geom, self.batch, self.q_nope, self.q_pe, self.cache, self.block_table,
                                       self.block_table.shape[1], self.seq_lens, self.kv_exp, self.o, self.lse,
                                       stream), "mla_normal_attention")

    def chunked(self, stream=None):
        L.check(L.mla_normal_chunked(self.geom, self.batch, self.q_nope, self.q_pe, self.cache, self.block_table,
                                     self.block_table.shape[1], self.seq_lens, self.w_uk, self.w_uv, self.chunk_rows,
                                     self.kv_exp, self.state, self.o, self.lse, stream), "mla_normal_chunked")

    def step(self, stream=None):
        if self.chunk_rows > 0:
            self.chunked(stream)
            return
        self.expand(stream)
        self.attention(stream)

    def expanded(self):
        """kv_exp viewed as [H, B * rows_per_seq, 256] (k_nope | v)."""
        return self.kv_exp[: self.w.H * self.w.B * self.rows_per_seq * 256].view(
            self.w.H, self.w.B * self.rows_per_seq, 256)
