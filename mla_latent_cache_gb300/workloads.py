"""Seeded synthetic inputs for absorbed MLA decode over a paged latent cache.

This module draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path (through the tests and the bench) and
the float64 oracle consume the exact bf16 bit patterns produced here, so the two
sides see identical inputs.

Input recipe (shared by every workload):
  * values of q_nope, q_pe, q_lat and of every cached latent/RoPE element are
    drawn as float32 N(0, 1) times a per-tensor scale and rounded to bf16 with
    round-to-nearest-even (0.1 for q_nope, q_pe and the cache; 0.05 for a
    directly drawn q_lat, the spread that q_nope @ W_UK has under this recipe);
  * W_UK and W_UV are N(0, 1/512) (variance 1/512, i.e. std 1/sqrt(512));
  * the "sharp" variant multiplies the query scales (q_nope, q_pe by 300,
    q_lat by 300) so that the softmax is far from uniform;
  * every tensor has its own generator, ``numpy.random.default_rng([seed, k])``,
    so adding or resizing one tensor never changes another;
  * pool blocks that no block table references, and the rows of a sequence's
    last page that lie past its length, hold bf16 NaN: a kernel that reads them
    poisons its output.

Geometry (DeepSeek-V2-Lite / V3): kv_lora_rank d_c = 512, RoPE width d_R = 64,
nope width d_N = 128, value width d_V = 128, page (block) size 64, one cached
row = 576 bf16 values = [c_KV (512) | k_pe (64)].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

D_C = 512
D_R = 64
D_N = 128
D_V = 128
D_K = D_C + D_R  # 576
PAGE = 64

BF16_NAN = np.uint16(0x7FC0)

# Per-tensor generator streams.
_S_LAYOUT, _S_CACHE, _S_QNOPE, _S_QPE, _S_WUK, _S_WUV, _S_QLAT, _S_SPARSE = range(8)


def f32_to_bf16_bits(x: np.ndarray, scale: float | None = None) -> np.ndarray:
    """Round float32 values (times ``scale`` in float32, when given) to bf16
    (nearest, ties to even); return uint16 bits.  Works in cache-sized chunks."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.size, dtype=np.uint16)
    step = 1 << 22
    for i in range(0, flat.size, step):
        c = flat[i:i + step]
        if scale is not None:
            c = c * np.float32(scale)
        b = c.view(np.uint32)
        r = (b >> np.uint32(16)) & np.uint32(1)
        r += np.uint32(0x7FFF)
        r += b
        r >>= np.uint32(16)
        out[i:i + step] = r
    return out.reshape(x.shape)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(u: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float64 (exact)."""
    return bf16_bits_to_f32(u).astype(np.float64)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def _normal_bf16(seed: int, stream: int, shape, scale: float) -> np.ndarray:
    g = _rng(seed, stream)
    x = g.standard_normal(size=int(np.prod(shape)), dtype=np.float32)
    return f32_to_bf16_bits(x, scale).reshape(shape)


@dataclass
class Workload:
    """One batch of synthetic decode/extend input, all bf16 as uint16 bits.

    Shapes: q_nope [B,T,H,128], q_pe [B,T,H,64], q_lat [B,T,H,512],
    w_uk / w_uv [H,128,512], block_table int32 [B, max_pages] (-1 past a
    sequence's pages), seq_lens int32 [B] (visible rows, the T new rows
    included).  The pool is stored compactly: ``pool_ids[i]`` is the physical
    block whose 64x576 rows are ``pool_data[i]``; every other block of the
    ``num_blocks`` pool is NaN.
    """

    name: str
    seed: int
    H: int
    B: int
    T: int
    causal: bool
    seq_lens: np.ndarray
    block_table: np.ndarray
    num_blocks: int
    pool_ids: np.ndarray
    q_scale: float = 0.1
    qlat_scale: float = 0.05
    _cache: dict = field(default_factory=dict, repr=False)

    # -- tensors are drawn on first use ---------------------------------------
    @property
    def pool_data(self) -> np.ndarray:
        """[n_used_blocks, 64, 576] rows of the referenced blocks (NaN past each sequence's end)."""
        if "pool_data" not in self._cache:
            data = _normal_bf16(self.seed, _S_CACHE, (len(self.pool_ids), PAGE, D_K), 0.1)
            pos = 0
            for b in range(self.B):
                n = (int(self.seq_lens[b]) + PAGE - 1) // PAGE
                if n:
                    tail = int(self.seq_lens[b]) - (n - 1) * PAGE
                    if tail < PAGE:
                        data[pos + n - 1, tail:, :] = BF16_NAN
                pos += n
            self._cache["pool_data"] = data
        return self._cache["pool_data"]

    @property
    def q_nope(self) -> np.ndarray:
        if "q_nope" not in self._cache:
            self._cache["q_nope"] = _normal_bf16(self.seed, _S_QNOPE, (self.B, self.T, self.H, D_N), self.q_scale)
        return self._cache["q_nope"]

    @property
    def q_pe(self) -> np.ndarray:
        if "q_pe" not in self._cache:
            self._cache["q_pe"] = _normal_bf16(self.seed, _S_QPE, (self.B, self.T, self.H, D_R), self.q_scale)
        return self._cache["q_pe"]

    @property
    def q_lat(self) -> np.ndarray:
        """A directly drawn absorbed query, for testing decode on its own."""
        if "q_lat" not in self._cache:
            self._cache["q_lat"] = _normal_bf16(self.seed, _S_QLAT, (self.B, self.T, self.H, D_C), self.qlat_scale)
        return self._cache["q_lat"]

    @property
    def w_uk(self) -> np.ndarray:
        if "w_uk" not in self._cache:
            self._cache["w_uk"] = _normal_bf16(self.seed, _S_WUK, (self.H, D_N, D_C), 1.0 / math.sqrt(512.0))
        return self._cache["w_uk"]

    @property
    def w_uv(self) -> np.ndarray:
        if "w_uv" not in self._cache:
            self._cache["w_uv"] = _normal_bf16(self.seed, _S_WUV, (self.H, D_V, D_C), 1.0 / math.sqrt(512.0))
        return self._cache["w_uv"]

    # -- cache views ----------------------------------------------------------
    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def full_pool(self) -> np.ndarray:
        """The whole [num_blocks, 64, 576] pool (NaN where nothing is stored)."""
        pool = np.full((self.num_blocks, PAGE, D_K), BF16_NAN, dtype=np.uint16)
        pool[self.pool_ids] = self.pool_data
        return pool

    def compact_view(self):
        """(pool, block_table) with blocks renumbered to index ``pool_data``.

        The renumbering is a relabelling of physical block ids only: every
        logical row resolves to the same 576 values as through the full pool.
        """
        remap = np.full(self.num_blocks, -1, dtype=np.int64)
        remap[self.pool_ids] = np.arange(len(self.pool_ids))
        bt = self.block_table.astype(np.int64)
        out = np.where(bt >= 0, remap[np.clip(bt, 0, None)], -1).astype(np.int32)
        return self.pool_data, out

    def total_rows(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())


def _build(name, seed, H, T, seq_lens, num_blocks, causal, q_scale, qlat_scale, assign="perm") -> Workload:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = len(seq_lens)
    pages = [(int(s) + PAGE - 1) // PAGE for s in seq_lens]
    total_pages = sum(pages)
    if total_pages > num_blocks:
        raise ValueError(f"{name}: {total_pages} pages do not fit a pool of {num_blocks} blocks")
    g = _rng(seed, _S_LAYOUT)
    if assign == "perm":
        order = g.permutation(num_blocks)[:total_pages]
    else:  # sampled without replacement from the pool
        order = g.choice(num_blocks, size=total_pages, replace=False)
    max_pages = max(1, max(pages) if pages else 1)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(pages):
        bt[b, :n] = order[pos:pos + n]
        pos += n
    pool_ids = np.asarray(order[:total_pages], dtype=np.int64)
    return Workload(name=name, seed=seed, H=H, B=B, T=T, causal=causal, seq_lens=seq_lens,
                    block_table=bt, num_blocks=num_blocks, pool_ids=pool_ids,
                    q_scale=q_scale, qlat_scale=qlat_scale)


SHARP_Q = 300.0


def config_workload(index: int, T: int | None = None, sharp: bool = False) -> Workload:
    """The five named workloads (index 1..5); seed = 1000 + index.

    1 tiny  : DeepSeek-V2-Lite geometry, H=16, B=1, T=1, S=512, pool of 8 blocks.
    2 uniform: V3 geometry, H=128, B=64, T=1, S=4096, pool of 4096 blocks.
    3 ragged: V3, B=128, S_b = floor(exp(U(ln 256, ln 32768))), pool 65536,
              block ids sampled without replacement.
    4 long  : V3, B=1, T=1, S=131072, pool of 2048 blocks.
    5 extend: V3, B=8, prefix 8192 plus T new rows (T in {1,16,64,170,512}),
              causal within the new rows, pool 8*ceil((8192+512)/64) blocks.
    """
    seed = 1000 + index
    qs, ql = (0.1, 0.05) if not sharp else (0.1 * SHARP_Q, 0.05 * SHARP_Q)
    if index == 1:
        return _build("tiny_v2lite_h16_b1_s512", seed, 16, 1, [512], 8, False, qs, ql)
    if index == 2:
        return _build("v3_uniform_b64_s4096", seed, 128, 1, [4096] * 64, 4096, False, qs, ql)
    if index == 3:
        g = _rng(seed, 100)
        u = g.uniform(math.log(256.0), math.log(32768.0), size=128)
        lens = np.floor(np.exp(u)).astype(np.int64)
        return _build("v3_ragged_b128_s256to32768", seed, 128, 1, lens, 65536, False, qs, ql, assign="choice")
    if index == 4:
        return _build("v3_long_b1_s131072", seed, 128, 1, [131072], 2048, False, qs, ql)
    if index == 5:
        T = 1 if T is None else int(T)
        if T not in (1, 16, 64, 170, 512):
            raise ValueError("extend workload takes T in {1, 16, 64, 170, 512}")
        pool = 8 * ((8192 + 512 + PAGE - 1) // PAGE)
        return _build(f"v3_extend_b8_p8192_t{T}", seed, 128, T, [8192 + T] * 8, pool, True, qs, ql)
    raise ValueError(f"no workload {index}")


def custom_workload(H: int, seq_lens, T: int = 1, causal: bool = False, seed: int = 7,
                    num_blocks: int | None = None, sharp: bool = False, name: str = "custom") -> Workload:
    """A small workload with the same recipe, for edge cases and ragged tails."""
    pages = sum((int(s) + PAGE - 1) // PAGE for s in seq_lens)
    if num_blocks is None:
        num_blocks = max(1, pages + 3)
    qs, ql = (0.1, 0.05) if not sharp else (0.1 * SHARP_Q, 0.05 * SHARP_Q)
    return _build(name, seed, H, T, list(seq_lens), num_blocks, causal, qs, ql)


@dataclass
class SparseWorkload:
    """Input of the index-driven decode: a context workload ``ctx`` (its T is the
    S_q query tokens per sequence, its block table places each sequence's rows)
    and, per query token, a list of physical rows (block * 64 + offset) of that
    sequence's context, as an indexer's top-k would give.

    indices int32 [B, S_q, topk]; topk_length int32 [B] (entries at or past a
    sequence's length point at a NaN row of an unreferenced block, or are -1 when
    the pool has none: a kernel that reads them poisons its output).
    """

    ctx: Workload
    topk: int
    indices: np.ndarray
    topk_length: np.ndarray
    name: str = "sparse"

    @property
    def B(self) -> int:
        return self.ctx.B

    @property
    def S_q(self) -> int:
        return self.ctx.T

    @property
    def H(self) -> int:
        return self.ctx.H


def sparse_workload(H: int, ctx_lens, S_q: int, topk: int, lengths=None, replace: bool = False, seed: int = 11,
                    num_blocks: int | None = None, sharp: bool = False, in_order: bool = False,
                    name: str = "sparse") -> SparseWorkload:
    """Per token, ``lengths[b]`` (default min(topk, context length)) positions of
    sequence b's context drawn uniformly (distinct unless ``replace``; all of them
    in order when ``in_order``), mapped through the block table to physical rows,
    in the drawn order."""
    w = custom_workload(H, ctx_lens, T=S_q, causal=False, seed=seed, num_blocks=num_blocks, sharp=sharp, name=name)
    B = w.B
    if lengths is None:
        lengths = [min(topk, int(s)) for s in w.seq_lens]
    lengths = np.asarray(lengths, dtype=np.int32)
    free = np.setdiff1d(np.arange(w.num_blocks), w.pool_ids)
    poison = int(free[0]) * PAGE if len(free) else -1
    g = _rng(seed, _S_SPARSE)
    idx = np.full((B, S_q, topk), poison, dtype=np.int32)
    for b in range(B):
        S = int(w.seq_lens[b])
        n = min(int(lengths[b]), topk)
        if n <= 0:
            continue
        for t in range(S_q):
            if in_order:
                pos = np.arange(n)
            else:
                pos = g.choice(S, size=n, replace=replace)
            idx[b, t, :n] = w.block_table[b, pos // PAGE].astype(np.int64) * PAGE + pos % PAGE
    return SparseWorkload(ctx=w, topk=topk, indices=idx, topk_length=lengths, name=name)
