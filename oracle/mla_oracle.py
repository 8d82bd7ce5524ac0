"""Float64 CPU oracle for absorbed MLA decode over a paged latent cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this module: only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference arm use it.  It shares no code with the CUDA
path.  Every function is the plain definition (or, for the split planner, the
rule written out step by step) in float64 NumPy, with no blocking, fusion or
reordering beyond what the definition states.  Each contraction is written as
one ``np.einsum`` over the definition's indices; ``optimize=True`` lets NumPy
evaluate it through BLAS (the same sums, in another float64 summation order).

Sources (web pages, cited by title and section):
  [MLA-in-depth]  "MLA in full detail" (mlinterviewnotes, ch. 7.2): Step 2 "fold
                  W_UK into the query", Step 3 "attend against the latent
                  directly", Step 4 "fold W_UV into the output", "What it costs",
                  and the closing float64 single-head parity reference.
  [zdszero]       "MLA" (zdszero.github.io): "Normal 与 Absorb" (the Normal and
                  Absorb forms), "计算量分析" (the MAC table), "谁更省" (the T~170
                  crossover), the decoupled-RoPE note that the scale stays sqrt(192),
                  "路径选择" (per-batch path choice: the MHA_CHUNKED_KV variant).
  [mlxcel]        "mlxcel: MLA absorbed decode": the bytes/token table and the
                  Stage-2 split-KV merge contract (partials normalised by their own
                  denominator, grouped by an indptr).
  [M5.8]          "M5.8 - Multi-Head Latent Attention: Latent KV State, Weight
                  Absorption, and FlashMLA": 0x04 "Batched absorption trace"
                  (canonical einsum shapes), 0x05 "Paged and ragged address
                  translation", 0x06 "Numeric Cache Ledger", 0x09 (decode
                  intensity), 0x0B "FP8 Cache Format And Sparse Selection" (the
                  656-byte FP8 row, sparse physical indices), 0x0C (exact merge
                  of sequence-split state).

Parity status: every function below is pinned by a CPU test (closed forms,
printed values, brute force, a library routine or an invariant) except
``plan_ref``, whose rule the pages leave open; it is pinned by brute-force
coverage/balance properties and is bit-exact-compared with the device planner.
"""
from __future__ import annotations

import math

import numpy as np

D_C = 512      # kv_lora_rank
D_R = 64       # qk_rope_head_dim
D_N = 128      # qk_nope_head_dim
D_V = 128      # v_head_dim
D_K = D_C + D_R
PAGE = 64
ROWS_PER_BLOCK = 128   # flattened (t, h) query rows handled together
MIN_SPLIT_PAGES = 4
# Plan rule: the fixed cost of starting a group's work in a range, in pages (a query
# staging and an output write per segment; the pages fix no split rule, see plan_ref).
SEGMENT_COST_PAGES = 8

SCALE = 1.0 / math.sqrt(D_N + D_R)   # 1/sqrt(192): [zdszero] decoupled-RoPE note; [MLA-in-depth] parity reference


# ---------------------------------------------------------------------------
# Paged address translation  ([M5.8] 0x05 "Paged and ragged address translation")
# ---------------------------------------------------------------------------
def physical_row(block_table_row: np.ndarray, j: int, page: int = PAGE) -> int:
    """physical(j) = block_table[page(j)] * P + offset(j), page(j) = j // P, offset(j) = j mod P."""
    logical_page, offset = divmod(int(j), page)
    phys_page = int(block_table_row[logical_page])
    if phys_page < 0:
        raise IndexError(f"logical row {j} maps to an unassigned page")
    return phys_page * page + offset


def gather_rows(pool: np.ndarray, block_table_row: np.ndarray, n_rows: int) -> np.ndarray:
    """Logical rows 0..n_rows-1 of one sequence, in order, as [n_rows, 576] (same dtype as pool).

    ``pool`` is [num_blocks, P, 576]; rows are resolved one logical page at a time.
    """
    page = pool.shape[1]
    flat = pool.reshape(-1, pool.shape[-1])
    out = np.empty((n_rows, pool.shape[-1]), dtype=pool.dtype)
    for j in range(n_rows):
        out[j] = flat[physical_row(block_table_row, j, page)]
    return out


# ---------------------------------------------------------------------------
# Absorption GEMMs  ([M5.8] 0x04 "Batched absorption trace"; [MLA-in-depth] Steps 2 and 4)
# ---------------------------------------------------------------------------
def absorb_ref(q_nope: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """q_lat[b,t,h,c] = sum_n q_nope[b,t,h,n] * W_UK[h,n,c]   (W_UK is [H, d_N, d_c])."""
    return np.einsum("bthn,hnc->bthc", q_nope, w_uk, optimize=True)


def unabsorb_ref(o_lat: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """o[b,t,h,v] = sum_c o_lat[b,t,h,c] * W_UV[h,v,c]   (W_UV is [H, d_V, d_c])."""
    return np.einsum("bthc,hvc->bthv", o_lat, w_uv, optimize=True)


# ---------------------------------------------------------------------------
# Causal visibility for T new rows already in the cache
# ---------------------------------------------------------------------------
def visible_limit(S: int, T: int, t: int, causal: bool) -> int:
    """Number of cache rows query token t (0..T-1) attends to.

    The T new rows are the last T of the S visible rows (they were appended
    before the step); with causal masking token t sees rows 0..S-T+t, i.e. the
    prefix plus new rows up to and including itself (bottom-right alignment;
    [MLA-in-depth] "prefix P=5, Q=3" gives P*Q + Q(Q+1)/2 visible pairs).
    """
    if not causal:
        return S
    return max(0, min(S, S - T + t + 1))


def causal_mask(S: int, T: int, causal: bool) -> np.ndarray:
    """Boolean [T, S]: True where token t may attend to cache row j."""
    m = np.zeros((T, S), dtype=bool)
    for t in range(T):
        m[t, :visible_limit(S, T, t, causal)] = True
    return m


# ---------------------------------------------------------------------------
# Absorbed decode  ([M5.8] 0x04 absorbed reference; [MLA-in-depth] Step 3)
# ---------------------------------------------------------------------------
def softmax_rows(s: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Softmax over the last (key) axis with max subtraction; returns (p, lse).

    Rows whose entries are all -inf give p = 0 and lse = -inf.
    """
    m = np.max(s, axis=-1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe)
    l = np.sum(e, axis=-1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
        lse = np.where(l[..., 0] > 0, m_safe[..., 0] + np.log(np.where(l[..., 0] > 0, l[..., 0], 1.0)), -np.inf)
    return p, lse


def attend_latent(q_lat: np.ndarray, q_pe: np.ndarray, rows: np.ndarray, mask: np.ndarray,
                  scale: float = SCALE) -> tuple[np.ndarray, np.ndarray]:
    """One sequence: q_lat [T,H,512], q_pe [T,H,64], rows [S,576], mask [T,S].

    s[t,h,j] = (q_lat[t,h] . c_j + q_pe[t,h] . k_pe_j) * scale, softmax over j
    (the key axis only), o_lat[t,h] = sum_j p[t,h,j] c_j, lse = log sum_j e^{s}.
    Returns (o_lat [T,H,512], lse [T,H]).
    """
    d_c = q_lat.shape[-1]
    c = rows[:, :d_c]
    kpe = rows[:, d_c:]
    s = (np.einsum("thc,jc->thj", q_lat, c, optimize=True) + np.einsum("thr,jr->thj", q_pe, kpe, optimize=True)) * scale
    s = np.where(mask[:, None, :], s, -np.inf)
    p, lse = softmax_rows(s)
    o = np.einsum("thj,jc->thc", p, c, optimize=True)
    return o, lse


def decode_ref(q_lat: np.ndarray, q_pe: np.ndarray, pool: np.ndarray, block_table: np.ndarray,
               seq_lens: np.ndarray, causal: bool, scale: float = SCALE, batches=None):
    """Absorbed attention over the paged latent cache for every (or the listed) sequence.

    q_lat [B,T,H,512], q_pe [B,T,H,64] (float64), pool [num_blocks,64,576] (float64),
    block_table [B,max_pages], seq_lens [B] (visible rows including the T new ones).
    Returns o_lat [B,T,H,512] and lse [B,T,H] (natural log; -inf, o=0 for S_b=0).
    """
    B, T, H, d_c = q_lat.shape
    o_lat = np.zeros((B, T, H, d_c))
    lse = np.full((B, T, H), -np.inf)
    for b in (range(B) if batches is None else batches):
        S = int(seq_lens[b])
        if S == 0:
            continue
        rows = gather_rows(pool, block_table[b], S)
        o_lat[b], lse[b] = attend_latent(q_lat[b], q_pe[b], rows, causal_mask(S, T, causal), scale)
    return o_lat, lse


def absorbed_layer_ref(q_nope, q_pe, pool, block_table, seq_lens, w_uk, w_uv, causal, scale=SCALE):
    """The whole absorbed chain: absorb, latent attention, un-absorb.  Returns (o, o_lat, lse, q_lat)."""
    q_lat = absorb_ref(q_nope, w_uk)
    o_lat, lse = decode_ref(q_lat, q_pe, pool, block_table, seq_lens, causal, scale)
    return unabsorb_ref(o_lat, w_uv), o_lat, lse, q_lat


# ---------------------------------------------------------------------------
# Normal (decompressed) path  ([zdszero] Normal mode; [MLA-in-depth] Step 1 "what the naive path does")
# ---------------------------------------------------------------------------
def decompress_ref(c, w_uk, w_uv):
    """Per-head keys and values of cached latents c [S, d_c] ([MLA-in-depth] naive path):
    k_nope[j,h,n] = sum_c W_UK[h,n,c] c_j[c],  v[j,h,v] = sum_c W_UV[h,v,c] c_j[c]."""
    return np.einsum("hnc,jc->jhn", w_uk, c, optimize=True), np.einsum("hvc,jc->jhv", w_uv, c, optimize=True)


def normal_ref(q_nope, q_pe, pool, block_table, seq_lens, w_uk, w_uv, causal, scale=SCALE, batches=None):
    """Up-project every cached latent into per-head keys/values, then ordinary MHA.

    k_nope[j,h,n] = sum_c W_UK[h,n,c] c_j[c];  v[j,h,v] = sum_c W_UV[h,v,c] c_j[c];
    k[j,h] = [k_nope[j,h] ; k_pe_j] (192 wide, k_pe broadcast over heads);
    q[t,h] = [q_nope ; q_pe];  o = softmax(q k^T * scale) v.
    Returns o [B,T,H,128] and lse [B,T,H].
    """
    B, T, H, _ = q_nope.shape
    d_c = w_uk.shape[-1]
    d_r = q_pe.shape[-1]
    o = np.zeros((B, T, H, w_uv.shape[1]))
    lse = np.full((B, T, H), -np.inf)
    for b in (range(B) if batches is None else batches):
        S = int(seq_lens[b])
        if S == 0:
            continue
        rows = gather_rows(pool, block_table[b], S)
        c = rows[:, :d_c]
        kpe = rows[:, d_c:]
        k_nope, v = decompress_ref(c, w_uk, w_uv)
        k = np.concatenate([k_nope, np.broadcast_to(kpe[:, None, :], (S, H, d_r))], axis=-1)
        q = np.concatenate([q_nope[b], q_pe[b]], axis=-1)
        s = np.einsum("thd,jhd->thj", q, k, optimize=True) * scale
        s = np.where(causal_mask(S, T, causal)[:, None, :], s, -np.inf)
        p, lse[b] = softmax_rows(s)
        o[b] = np.einsum("thj,jhv->thv", p, v, optimize=True)
    return o, lse


# ---------------------------------------------------------------------------
# Split-KV partial state and its exact merge
# ([M5.8] 0x0C exact merge; [mlxcel] Stage 2 merge contract)
# ---------------------------------------------------------------------------
def partial_ref(q_lat_b, q_pe_b, pool, block_table_row, S, T, causal, page_begin, page_end, scale=SCALE):
    """Attention of one sequence restricted to the keys in logical pages [page_begin, page_end).

    Returns the partial output normalised by its own denominator, o_r [T,H,512],
    and its log-sum-exp lse_r [T,H] (natural log; -inf where no key is visible).
    """
    T_, H, d_c = q_lat_b.shape
    page = pool.shape[1]
    j0 = page_begin * page
    j1 = min(S, page_end * page)
    if j1 <= j0:
        return np.zeros((T_, H, d_c)), np.full((T_, H), -np.inf)
    rows_all = gather_rows(pool, block_table_row, j1)
    mask = causal_mask(S, T, causal)[:, j0:j1]
    return attend_latent(q_lat_b, q_pe_b, rows_all[j0:j1], mask, scale)


def merge_ref(part_o: np.ndarray, part_lse: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Exact merge of R partial states: part_o [R,...,D] (each normalised), part_lse [R,...].

    m = max_r lse_r; w_r = e^{lse_r - m}; o = sum_r w_r o_r / sum_r w_r; lse = m + ln sum_r w_r.
    (Equivalent to m = max m_r, l = sum e^{m_r-m} l_r, o = sum e^{m_r-m} o_r, O = o/l.)
    If every partial is empty (lse = -inf) the result is o = 0, lse = -inf.
    """
    part_o = np.asarray(part_o, dtype=np.float64)
    part_lse = np.asarray(part_lse, dtype=np.float64)
    if part_o.shape[0] == 0:
        return np.zeros(part_o.shape[1:]), np.full(part_lse.shape[1:], -np.inf)
    m = np.max(part_lse, axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(part_lse - m_safe)
    w = np.where(np.isfinite(part_lse), w, 0.0)
    l = np.sum(w, axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        o = np.where(l[..., None] > 0, np.sum(w[..., None] * part_o, axis=0) / np.where(l > 0, l, 1.0)[..., None], 0.0)
        lse = np.where(l > 0, m_safe + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse


# ---------------------------------------------------------------------------
# Sparse index-driven decode  ([M5.8] 0x0B "Sparse indices are physical execution
# metadata"; 0x08 dense vs sparse ABI).  indices [B, S_q, topk] name physical
# cache rows; topk_length [B] bounds the valid left prefix of every index row of
# sequence b; causal = False in this ABI.  Reading where the pages are silent: an
# entry encodes row (block * 64 + offset); a row listed twice counts twice (the
# softmax runs over the list); an empty list gives o = 0, lse = -inf.
# ---------------------------------------------------------------------------
def sparse_decode_ref(q_lat, q_pe, pool, indices, topk_length=None, scale=SCALE):
    """q_lat [B,S_q,H,512], q_pe [B,S_q,H,64], pool [num_blocks,64,576] (float64
    row values; FP8 rows pass their dequantized values), indices [B,S_q,topk].
    Returns o_lat [B,S_q,H,512] and lse [B,S_q,H]."""
    B, Sq, H, d_c = q_lat.shape
    page = pool.shape[1]
    topk = indices.shape[-1]
    o = np.zeros((B, Sq, H, d_c))
    lse = np.full((B, Sq, H), -np.inf)
    for b in range(B):
        n = topk if topk_length is None else int(topk_length[b])
        if n <= 0:
            continue
        for t in range(Sq):
            idx = np.asarray(indices[b, t, :n], dtype=np.int64)
            rows = pool[idx // page, idx % page]
            ob, lb = attend_latent(q_lat[b, t:t + 1], q_pe[b, t:t + 1], rows, np.ones((1, n), dtype=bool), scale)
            o[b, t], lse[b, t] = ob[0], lb[0]
    return o, lse


# ---------------------------------------------------------------------------
# Chunked-prefix Normal path  ([zdszero] "路径选择" (path choice), the
# MHA_CHUNKED_KV variant): the prefix is read in chunks, each chunk is expanded
# with kv_b and attended, and the chunks' states are merged by LSE, so the
# expanded prefix held at once is bounded by one chunk.
# ---------------------------------------------------------------------------
def normal_chunked_ref(q_nope, q_pe, pool, block_table, seq_lens, w_uk, w_uv, causal, chunk_rows: int,
                       scale=SCALE, batches=None):
    """The Normal path over the visible rows in chunks of chunk_rows rows: per
    chunk, k_nope/v = kv_b expansion of its latents, attention restricted to its
    keys (partial o normalised by its own sum, partial lse), then merge_ref over
    the chunks.  Returns o [B,T,H,128] and lse [B,T,H]."""
    B, T, H, _ = q_nope.shape
    d_c = w_uk.shape[-1]
    d_r = q_pe.shape[-1]
    o = np.zeros((B, T, H, w_uv.shape[1]))
    lse = np.full((B, T, H), -np.inf)
    for b in (range(B) if batches is None else batches):
        S = int(seq_lens[b])
        if S == 0:
            continue
        rows = gather_rows(pool, block_table[b], S)
        mask = causal_mask(S, T, causal)
        q = np.concatenate([q_nope[b], q_pe[b]], axis=-1)
        parts_o, parts_l = [], []
        for j0 in range(0, S, chunk_rows):
            j1 = min(S, j0 + chunk_rows)
            c = rows[j0:j1, :d_c]
            kpe = rows[j0:j1, d_c:]
            k_nope, v = decompress_ref(c, w_uk, w_uv)
            k = np.concatenate([k_nope, np.broadcast_to(kpe[:, None, :], (j1 - j0, H, d_r))], axis=-1)
            s = np.einsum("thd,jhd->thj", q, k, optimize=True) * scale
            s = np.where(mask[:, None, j0:j1], s, -np.inf)
            p, l_part = softmax_rows(s)
            parts_o.append(np.einsum("thj,jhv->thv", p, v, optimize=True))
            parts_l.append(l_part)
        o[b], lse[b] = merge_ref(np.stack(parts_o), np.stack(parts_l))
    return o, lse


# ---------------------------------------------------------------------------
# Split planner.  The pages leave the rule open (FlashMLA's scheduler metadata
# is opaque; [M5.8] 0x08 only says it must be rebuilt when geometry or lengths
# change).  This is the rule both the device planner and this restatement follow.
# ---------------------------------------------------------------------------
def group_pages(seq_lens, T: int, H: int, causal: bool) -> list[tuple[int, int, int]]:
    """Work groups (b, rb, n_pages) in b-major order.

    Query rows of a sequence are flattened as r = t*H + h and cut into row
    blocks of 128; row block rb needs the pages visible to its last token.
    """
    R = T * H
    RB = (R + ROWS_PER_BLOCK - 1) // ROWS_PER_BLOCK
    out = []
    for b, S in enumerate(seq_lens):
        S = int(S)
        for rb in range(RB):
            r_last = min(R, (rb + 1) * ROWS_PER_BLOCK) - 1
            t_last = r_last // H
            vis = visible_limit(S, T, t_last, causal)
            out.append((b, rb, (vis + PAGE - 1) // PAGE))
    return out


def plan_ref(seq_lens, T: int, H: int, causal: bool, num_slots: int, num_splits_override: int = 0):
    """Deterministic split plan.

    Returns dict with
      segments : list of (b, rb, page_begin, page_end, range_id, slot)  slot=-1 => final output
      num_ranges, num_partials,
      range_ptr: [num_ranges+1] segment offsets of each work range,
      merge    : list of (b, rb, slot_begin, count) for every group not finished by a
                 single final segment (count 0 => the group is empty: o=0, lse=-inf).
    Rule:
      1. groups (b, rb, n) as in group_pages; W = sum n.
      2. override N>0: a group with n>0 is cut into k=min(n,N) segments,
         segment s = [floor(s n/k), floor((s+1) n/k)); each segment is its own range.
      3. auto: q = max(4, ceil(W/G)).  If the non-empty groups number at most G
         and none has more than ceil(5q/4) pages, every non-empty group is one
         segment and one range.  Otherwise the non-empty groups are laid out on
         a line, in order, each after a gap of c = SEGMENT_COST_PAGES positions
         from the previous one (none before the first): group g's pages occupy
         [u_g, u_g + n_g) with u_g = (pages of the groups before g) + c x (non-empty
         groups before g); with U = W + c x (non-empty groups - 1) and
         q' = max(4, ceil(U/G)), range r covers positions [r q', (r+1) q') and
         each group is cut where the range boundaries fall.  (A range's work is
         then its pages plus c for every group that starts in it; a range that
         lies inside a gap holds no segment.)
      4. a segment that covers its whole group is final (slot -1); the other
         segments get partial slots numbered in segment order.
    """
    groups = group_pages(seq_lens, T, H, causal)
    G = max(1, int(num_slots))
    raw = []  # (b, rb, p0, p1, range)
    n_ranges = 0
    if num_splits_override > 0:
        for (b, rb, n) in groups:
            if n == 0:
                continue
            k = min(n, int(num_splits_override))
            for s in range(k):
                raw.append((b, rb, (s * n) // k, ((s + 1) * n) // k, n_ranges))
                n_ranges += 1
    else:
        W = sum(n for (_, _, n) in groups)
        q = max(MIN_SPLIT_PAGES, -(-W // G)) if W > 0 else MIN_SPLIT_PAGES
        nonempty = [g for g in groups if g[2] > 0]
        max_n = max((g[2] for g in nonempty), default=0)
        if len(nonempty) <= G and max_n <= -(-5 * q // 4):
            for (b, rb, n) in nonempty:
                raw.append((b, rb, 0, n, n_ranges))
                n_ranges += 1
        else:
            c = SEGMENT_COST_PAGES
            U = W + c * (len(nonempty) - 1) if nonempty else 0
            qw = max(MIN_SPLIT_PAGES, -(-U // G)) if U > 0 else MIN_SPLIT_PAGES
            u = 0          # line position of the next group's first page
            started = False
            for (b, rb, n) in groups:
                if n == 0:
                    continue
                if started:
                    u += c
                started = True
                p = 0
                while p < n:
                    r = (u + p) // qw
                    end_in_group = min(n, (r + 1) * qw - u)
                    raw.append((b, rb, p, end_in_group, r))
                    p = end_in_group
                u += n
            n_ranges = -(-U // qw) if U > 0 else 0
    n_of = {(b, rb): n for (b, rb, n) in groups}
    segments = []
    slot = 0
    for (b, rb, p0, p1, r) in raw:
        if p0 == 0 and p1 == n_of[(b, rb)]:
            segments.append((b, rb, p0, p1, r, -1))
        else:
            segments.append((b, rb, p0, p1, r, slot))
            slot += 1
    range_ptr = [0] * (n_ranges + 1)
    for s in segments:
        range_ptr[s[4] + 1] += 1
    for r in range(n_ranges):
        range_ptr[r + 1] += range_ptr[r]
    merge = []
    for (b, rb, n) in groups:
        segs = [s for s in segments if s[0] == b and s[1] == rb]
        if n == 0:
            merge.append((b, rb, 0, 0))
        elif segs[0][5] >= 0:
            merge.append((b, rb, segs[0][5], len(segs)))
    return {"segments": segments, "num_ranges": n_ranges, "num_partials": slot,
            "range_ptr": range_ptr, "merge": merge}


# ---------------------------------------------------------------------------
# Byte and operation ledgers
# ([mlxcel] bytes/token table; [M5.8] 0x02 and 0x06 ledgers; [zdszero] 计算量分析;
#  [MLA-in-depth] "What it costs")
# ---------------------------------------------------------------------------
def latent_bytes_per_token(d_c=D_C, d_r=D_R, elem=2) -> int:
    """One cached row per token per layer: (d_c + d_R) values."""
    return (d_c + d_r) * elem


def decompressed_bytes_per_token(H, d_n=D_N, d_r=D_R, d_v=D_V, elem=2) -> int:
    """Per-head keys (d_N + d_R wide) and values (d_V wide) for every head."""
    return H * ((d_n + d_r) + d_v) * elem


def normal_upproj_macs(S, d_c=D_C, H=128, d_n=D_N, d_v=D_V) -> int:
    """kv_b up-projection of S cached latents into keys and values: S*d_c*H*d_N + S*d_c*H*d_V."""
    return S * d_c * H * d_n + S * d_c * H * d_v


def absorb_upproj_macs(T, d_c=D_C, H=128, d_n=D_N, d_v=D_V) -> int:
    """Absorbing W_UK into T queries and applying W_UV to T outputs."""
    return T * H * d_n * d_c + T * H * d_c * d_v


def normal_attention_macs(T, S, H=128, d_n=D_N, d_r=D_R, d_v=D_V) -> int:
    return H * (T * S * (d_n + d_r) + T * S * d_v)


def absorb_attention_macs(T, S, H=128, d_c=D_C, d_r=D_R) -> int:
    return H * (T * S * (d_c + d_r) + T * S * d_c)


def visible_pairs(S, T, causal) -> int:
    """Number of (query token, cache row) pairs that attend (from the mask)."""
    return int(causal_mask(S, T, causal).sum())


def decode_core_flops(H, pairs, d_c=D_C, d_r=D_R) -> int:
    """2 flops per MAC of q.k (d_c+d_R wide) and p.v (d_c wide) per head per visible pair."""
    return 2 * H * pairs * ((d_c + d_r) + d_c)


def crossover_T(S, H=128) -> float:
    """Query-block length T at which Absorb and Normal cost the same MACs for context S.

    Solves absorb_upproj(T) + absorb_attention(T,S) = normal_upproj(S) + normal_attention(T,S)
    for T (both sides linear in T).
    """
    a = absorb_upproj_macs(1, H=H) + absorb_attention_macs(1, S, H=H) - normal_attention_macs(1, S, H=H)
    return normal_upproj_macs(S, H=H) / a


def decode_intensity(H, d_c=D_C, d_r=D_R, elem=2) -> float:
    """Core FLOPs per cache byte at T=1 (query/output traffic excluded)."""
    return decode_core_flops(H, 1, d_c, d_r) / ((d_c + d_r) * elem)


# ---------------------------------------------------------------------------
# FP8 latent row  ([M5.8] 0x0B "FP8 Cache Format And Sparse Selection", "Exact
# 656-byte FP8 row"): 512 E4M3 latent values + 4 fp32 scales + 64 bf16 RoPE
# values; storage format only, attention runs on the dequantized bf16 values.
# The pages give the three segments and their sizes; the readings taken where
# they are silent: one scale per 128 consecutive latent values, scale = the
# tile's largest magnitude / 448 rounded to fp32 (1 for an all-zero tile), the
# segments stored in the order the pages sum them (codes, scales, RoPE), all
# multi-byte words little-endian.  The stored scale is fp32 (the segment the
# pages give), so it is the exact quotient amax / 448 rounded once to fp32; each
# code is then the E4M3 value nearest to the exact quotient value / scale (ties
# to the even mantissa), decided exactly: |value| is compared with the
# midpoints between neighbouring E4M3 values times the scale, products that
# float64 holds exactly (at most 5 + 24 significant bits).  E4M3 is the OFP8 format: sign, 4 exponent
# bits (bias 7), 3 mantissa bits, subnormals at exponent 0, S.1111.111 = NaN,
# no infinities, largest finite value 448.
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0
FP8_TILE = 128
FP8_ROW_BYTES = D_C * 1 + (D_C // FP8_TILE) * 4 + D_R * 2   # 656


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 byte (float64; NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 byte to each value, ties to the even mantissa; magnitudes
    beyond 448 saturate to +-448 (the quantizer's scale keeps them within it)."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.int64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    out = np.empty(a.shape, dtype=np.int64)
    flat_a, flat_o = a.reshape(-1), out.reshape(-1)
    for i, v in enumerate(flat_a):
        if v < 2.0 ** -6:                       # subnormal range: steps of 2^-9
            m = int(np.rint(v / 2.0 ** -9))      # rint rounds half to even
            flat_o[i] = m                        # m == 8 is the smallest normal, code 0x08
            continue
        e = int(math.floor(math.log2(v)))
        frac = v / 2.0 ** e                      # in [1, 2)
        if frac >= 2.0:                          # log2 rounding at a power of two
            e, frac = e + 1, frac / 2.0
        elif frac < 1.0:
            e, frac = e - 1, frac * 2.0
        m = int(np.rint((frac - 1.0) * 8.0))
        if m == 8:
            e, m = e + 1, 0
        code = ((e + 7) << 3) | m
        flat_o[i] = min(code, 0x7E)              # 1.875 * 2^8 would be the NaN code: saturate
    return (out | sign).astype(np.uint8)


def f32_nearest_quotient(num: float, den: float) -> np.float32:
    """The fp32 value nearest to the exact quotient num / den (ties to the even
    significand), for finite float64 num and den > 0."""
    from fractions import Fraction
    exact = Fraction(num) / Fraction(den)
    x = np.float32(float(exact))
    # the nearest fp32 value is x or one of its neighbours: compare all three exactly
    cands = [np.nextafter(x, np.float32(-np.inf)), x, np.nextafter(x, np.float32(np.inf))]
    dist = [abs(exact - Fraction(float(v))) for v in cands]
    best = min(dist)
    near = [v for v, d in zip(cands, dist) if d == best]
    if len(near) == 1:
        return near[0]
    return [v for v in near if (int(np.asarray(v).view(np.uint32)) & 1) == 0][0]


def e4m3_encode_scaled(values: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """E4M3 byte nearest to the exact quotient values / scale (ties to the even
    mantissa; magnitudes beyond 448 saturate to +-448): values [..., n] float64,
    scale [...] positive.  The decision compares |value| with each midpoint
    between neighbouring E4M3 values times the scale; a midpoint has at most 5
    significant bits and the fp32 scale 24, so every product is exact in
    float64 and so is every comparison."""
    values = np.asarray(values, dtype=np.float64)
    pos = e4m3_decode(np.arange(0x7F))                       # 0 .. 448, ascending
    mids = (pos[:-1] + pos[1:]) / 2.0                        # 126 midpoints, exact
    thr = mids * np.asarray(scale, dtype=np.float64)[..., None]     # [..., 126], exact products
    a = np.abs(values)
    lead, n = values.shape[:-1], values.shape[-1]
    thr_f = thr.reshape(-1, mids.size)
    a_f = a.reshape(-1, n)
    codes = np.empty(a_f.shape, dtype=np.int64)
    for i in range(a_f.shape[0]):
        k = np.searchsorted(thr_f[i], a_f[i], side="left")   # thresholds strictly below |value|
        tie = (k < mids.size) & (thr_f[i][np.minimum(k, mids.size - 1)] == a_f[i])
        codes[i] = np.where(tie & (k % 2 == 1), k + 1, k)    # a tie between codes k and k+1: the even one
    sign = np.where(np.signbit(values), 0x80, 0).reshape(codes.shape)
    return (codes | sign).astype(np.uint8).reshape(lead + (n,))


def fp8_row_quantize(c: np.ndarray, k_pe_bits: np.ndarray) -> np.ndarray:
    """Pack latent rows c [..., 512] (float64 values) and RoPE bf16 bit patterns
    k_pe_bits [..., 64] (uint16) into 656-byte rows [..., 656] (uint8)."""
    c = np.asarray(c, dtype=np.float64)
    lead = c.shape[:-1]
    tiles = c.reshape(lead + (D_C // FP8_TILE, FP8_TILE))
    amax = np.abs(tiles).max(axis=-1)
    scale = np.ones(amax.shape, dtype=np.float32)
    for idx in zip(*np.nonzero(amax > 0)):
        scale[idx] = f32_nearest_quotient(float(amax[idx]), E4M3_MAX)
    codes = e4m3_encode_scaled(tiles, scale).reshape(lead + (D_C,))
    out = np.empty(lead + (FP8_ROW_BYTES,), dtype=np.uint8)
    out[..., :D_C] = codes
    out[..., D_C:D_C + 16] = scale.astype("<f4").view(np.uint8).reshape(lead + (16,))
    out[..., D_C + 16:] = np.asarray(k_pe_bits, dtype="<u2").view(np.uint8).reshape(lead + (2 * D_R,))
    return out


def fp8_row_dequantize(rows: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(latent values [..., 512] float64, fp32 scales [..., 4], RoPE bf16 bits
    [..., 64]) of 656-byte rows: value = E4M3 code value * its tile's scale."""
    rows = np.asarray(rows, dtype=np.uint8)
    lead = rows.shape[:-1]
    scale = np.ascontiguousarray(rows[..., D_C:D_C + 16]).view("<f4").reshape(lead + (D_C // FP8_TILE,))
    vals = e4m3_decode(rows[..., :D_C]).reshape(lead + (D_C // FP8_TILE, FP8_TILE))
    c_hat = (vals * scale.astype(np.float64)[..., None]).reshape(lead + (D_C,))
    k_pe_bits = np.ascontiguousarray(rows[..., D_C + 16:]).view("<u2").reshape(lead + (D_R,))
    return c_hat, scale, k_pe_bits
