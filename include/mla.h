/*
 * mla.h — C ABI of libmla.so: absorbed Multi-head Latent Attention (MLA) decode
 * over a paged latent KV cache, for GB300 (sm_103a).
 *
 * The operation (sources cited by page title and section):
 *   - "MLA in full detail" (mlinterviewnotes ch. 7.2), Step 2 "fold W_UK into
 *     the query", Step 3 "attend against the latent directly", Step 4 "fold
 *     W_UV into the output";
 *   - "M5.8 - Multi-Head Latent Attention ..." 0x04 "Batched absorption trace"
 *     (canonical shapes), 0x05 "Paged and ragged address translation", 0x08
 *     "FlashMLA Runtime ABI" (scheduler metadata that must be rebuilt when the
 *     batch geometry or the lengths change; a returned LSE), 0x0C (exact merge
 *     of split softmax state);
 *   - "mlxcel: MLA absorbed decode", Stage 2 (split-KV partials normalised by
 *     their own denominator, merged by log-sum-exp through an indptr).
 *
 * Geometry: kv_lora_rank d_c = 512, RoPE width d_R = 64, nope width d_N = 128,
 * value width d_V = 128, page (block) size P = 64, softmax scale 1/sqrt(192).
 * One cached row is 576 bf16 values: [c_KV (512) | k_pe (64)], shared by all
 * H query heads (one latent KV head).
 *
 * Tensor layouts (row-major, contiguous unless a stride is given; bf16 unless noted):
 *   q_nope [B,T,H,128]   q_pe [B,T,H,64]   q_lat [B,T,H,512]
 *   W_UK, W_UV [H,128,512]   (W_UK[h,n,c] contracted over n with q_nope;
 *                             W_UV[h,v,c] contracted over c with o_lat)
 *   cache: latent row j of block k at ckv + k*ckv_block_stride + j*ckv_row_stride
 *          (elements), its RoPE values at kpe + k*kpe_block_stride + j*kpe_row_stride;
 *          one combined [num_blocks, 64, 576] buffer or two separate ones
 *   block_table int32 [B, bt_stride]; seq_lens int32 [B] (visible rows,
 *          including the T new rows, which are the last T of them)
 *   o_lat [B,T,H,512]   lse float32 [B,T,H] (natural log)   o [B,T,H,128]
 *
 * Conventions.
 *   Ownership: the caller allocates every device buffer, the workspace
 *     included.  The library never allocates or frees device memory and never
 *     synchronises, except mla_read_device_status.
 *   Asynchrony: every call enqueues work on `stream` and returns at once.  The
 *     returned status covers host-side validation and launch errors only;
 *     errors seen by kernels are recorded in the workspace's status word and
 *     read back with mla_read_device_status.
 *   Programmatic dependent launch: every kernel is launched so that it may
 *     start while the previous kernel in the stream finishes, and waits for that
 *     kernel before reading anything a previous kernel may produce or writing
 *     anything it may read.  The weights (w_uk, w_uv), which no call of this
 *     library writes, may be read before that wait: a caller's kernel that
 *     writes them must not trigger programmatic launch before it has written
 *     them (a kernel that never triggers is safe).
 *   Alignment: every device pointer must be 16-byte aligned, and strides must
 *     keep rows 16-byte aligned (MLA_ERR_ALIGN otherwise); the outputs written
 *     with 32-byte stores (q_lat of mla_absorb_q, o of mla_unabsorb_o, o_lat
 *     and the workspace of mla_plan / mla_decode, kv_exp of mla_normal_expand,
 *     o of mla_normal_attention) must be 32-byte aligned.
 *   Causality: with causal != 0, query token t of sequence b sees cache rows
 *     0 .. S_b - T + t (bottom-right aligned); otherwise all S_b rows.
 *   Empty sequences: S_b = 0 gives o_lat = 0 and lse = -inf.
 *   Errors never trap: a kernel that meets a bad block id, a length beyond the
 *     block table, a stale plan or a wait that runs out records an error code
 *     in the workspace and skips the access.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* mla_stream_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_ARG = -1,          /* null pointer, negative size, unsupported flag */
  MLA_ERR_SHAPE = -2,        /* geometry not supported (d_* must be 512/64/128/128, P = 64, 1 <= H <= 128, 128 % H == 0) */
  MLA_ERR_ALIGN = -3,        /* pointer or stride not 16-byte (outputs: 32-byte) aligned */
  MLA_ERR_WORKSPACE = -4,    /* workspace smaller than mla_workspace_size() */
  MLA_ERR_PLAN_STALE = -5,   /* (device) plan built for other lengths/geometry */
  MLA_ERR_CUDA = -6,         /* a CUDA runtime call or launch failed */
  MLA_ERR_DEVICE_CHECK = -7, /* (device) bad block id, or seq_len beyond the block table, or T > seq_len */
  MLA_ERR_TIMEOUT = -8       /* (device) a bounded wait ran out */
} mla_status;

typedef struct {
  int H;               /* query heads (DeepSeek-V2-Lite 16, V3 128) */
  int d_lat;           /* kv_lora_rank, must be 512 */
  int d_rope;          /* qk_rope_head_dim, must be 64 */
  int d_nope;          /* qk_nope_head_dim, must be 128 */
  int d_v;             /* v_head_dim, must be 128 */
  int block_size;      /* rows per cache page, must be 64 */
  float softmax_scale; /* 1/sqrt(d_nope + d_rope) = 1/sqrt(192) */
} mla_geom;

typedef struct {
  const void* ckv;          /* bf16 latent part of the pool (512 values per row) */
  const void* kpe;          /* bf16 RoPE part (64 values per row); for the combined 576-wide row, (bf16*)ckv + 512 */
  int64_t ckv_row_stride;   /* elements between consecutive latent rows of a block (576 combined, 512 split) */
  int64_t ckv_block_stride; /* elements between consecutive latent blocks (64*576 combined) */
  int64_t kpe_row_stride;   /* elements between consecutive RoPE rows (576 combined, 64 split) */
  int64_t kpe_block_stride; /* elements between consecutive RoPE blocks */
  int num_blocks;           /* blocks in the pool; valid block ids are 0 .. num_blocks-1 */
} mla_cache;

typedef struct {
  int B;                   /* sequences in the batch (>= 0) */
  int T;                   /* new query tokens per sequence (>= 1) */
  int causal;              /* 1: causal within the new tokens */
  int max_pages;           /* width of a block-table row, in pages (>= 1) */
  int num_slots;           /* work ranges run concurrently (one per CTA pair); 0 = half the device's SM count */
  int num_splits_override; /* 0: automatic split rule; N > 0: every query-row group is cut into min(pages, N) chunks */
} mla_batch;

/*
 * Scheduler plan stored at the start of the workspace (all int32; written by
 * mla_plan, read by mla_decode).  Offsets are in bytes from the workspace base.
 * The split rule (the pages leave it open; FlashMLA's metadata is opaque):
 *   query rows of a sequence are flattened r = t*H + h and cut into row blocks
 *   of 128 (a "group" (b, rb)); a group needs the pages visible to its last
 *   token.  Let W be the total pages over all groups and q = max(4, ceil(W/G)),
 *   G = num_slots.  With an override N, each group is cut into min(n, N) even
 *   chunks, one range each.  Otherwise, if at most G groups are non-empty and
 *   none exceeds ceil(5q/4) pages, each group is one segment and one range;
 *   else the non-empty groups' pages are laid out in order on a line with a gap
 *   of c = 8 positions before each group but the first (a segment's fixed cost
 *   in pages), U = W + c (non-empty groups - 1), q' = max(4, ceil(U/G)), and
 *   range r covers line positions [r q', (r+1) q'), each group cut where the
 *   range boundaries fall (a range inside a gap holds no segment).
 *   A segment covering its whole group writes final outputs; the others write
 *   partial state to numbered slots, merged afterwards.
 */
enum {
  MLA_HDR_MAGIC = 0, MLA_HDR_B, MLA_HDR_T, MLA_HDR_H, MLA_HDR_CAUSAL, MLA_HDR_NUM_GROUPS,
  MLA_HDR_NUM_SEGMENTS, MLA_HDR_NUM_RANGES, MLA_HDR_NUM_PARTIALS, MLA_HDR_NUM_MERGE,
  MLA_HDR_SEQ_HASH, MLA_HDR_ERROR, MLA_HDR_ERROR_INFO, MLA_HDR_PAGES_PER_RANGE,
  MLA_HDR_NUM_SLOTS, MLA_HDR_OVERRIDE, MLA_HDR_MAX_PAGES,
  MLA_HDR_OFF_SEGMENTS, MLA_HDR_OFF_RANGE_PTR, MLA_HDR_OFF_MERGE, MLA_HDR_OFF_PART_LSE, MLA_HDR_OFF_PART_O,
  MLA_HDR_CAP_SEGMENTS, MLA_HDR_CAP_PARTIALS, MLA_HDR_CAP_RANGES, MLA_HDR_CAP_GROUPS,
  MLA_HDR_WORDS = 64
};
#define MLA_PLAN_MAGIC 0x4d4c4131 /* "MLA1" */
/* range pointers: int32 [cap_ranges + 1]; the segments of range r are
 *   rptr[r] .. rptr[r+1]-1; entries past num_ranges equal the segment count
 * segment record: int32[8] = {b, rb, page_begin, page_end, range, slot (-1 = final),
 *   merge record of its group (-1 = final), 0}
 * merge record:   int32[4] = {b, rb, slot_begin, count} (count 0 = empty group), and two
 *   int32 counters per record (partial rows stored, rows merged; zero between decodes)
 * part_lse float32 [cap_partials, 128]; part_o float32 [cap_partials, 128, 512] (normalised) */

/* Bytes of workspace needed for this geometry and batch shape. 0 on invalid arguments. */
size_t mla_workspace_size(const mla_geom* geom, const mla_batch* batch);

/*
 * Split plan ("M5.8" 0x08 "FlashMLA Runtime ABI": scheduler metadata rebuilt
 * whenever the batch geometry or the lengths change).
 * Build the split plan on the device from seq_lens (device int32 [B]) into the
 * workspace.  Must be re-run whenever B, T, causal, the lengths or num_slots
 * change (the plan is stamped with them; mla_decode with checked != 0 flags a
 * stale plan).  Also clears the workspace status word.
 */
mla_status mla_plan(const mla_geom* geom, const mla_batch* batch, const int32_t* seq_lens,
                    void* workspace, size_t ws_bytes, mla_stream_t stream);

/*
 * Key absorption ("MLA in full detail", Step 2 "fold W_UK into the query";
 * "M5.8" 0x04 "Batched absorption trace", the q_nope x W_UK einsum):
 * q_lat[b,t,h,:] = q_nope[b,t,h,:] @ W_UK[h]   over BT = B*T query tokens.
 * q_nope [BT,H,128], w_uk [H,128,512], q_lat [BT,H,512] (all bf16, device).
 * fp32 accumulation, bf16 output (round to nearest even).
 */
mla_status mla_absorb_q(const mla_geom* geom, const void* q_nope, const void* w_uk, void* q_lat,
                        int BT, mla_stream_t stream);

/*
 * Value un-absorption ("MLA in full detail", Step 4 "fold W_UV into the
 * output"; "M5.8" 0x04, the o_lat x W_UV einsum):
 * o[b,t,h,v] = sum_c o_lat[b,t,h,c] * W_UV[h,v,c]   over BT query tokens.
 * o_lat [BT,H,512], w_uv [H,128,512], o [BT,H,128] (bf16, device); fp32 accumulation.
 */
mla_status mla_unabsorb_o(const mla_geom* geom, const void* o_lat, const void* w_uv, void* o,
                          int BT, mla_stream_t stream);

/*
 * Absorbed attention over the paged latent cache ("MLA in full detail", Step 3
 * "attend against the latent directly"; "M5.8" 0x05 "Paged and ragged address
 * translation" for the pages; 0x0C and "mlxcel" Stage 2 for the merge of split
 * states), using the plan in the workspace: scores s = (q_lat . c_j + q_pe . k_pe_j) * scale, softmax over the
 * visible rows j, o_lat = sum_j p_j c_j, lse = log sum_j e^{s_j}.  One kernel
 * launch: the split-KV decode, whose CTAs also merge the plan's partial segments.
 * q_lat [B,T,H,512], q_pe [B,T,H,64] bf16; o_lat [B,T,H,512] bf16; lse [B,T,H] float32.
 * checked != 0 validates every block id read, the plan stamp and T <= S_b on the
 * device (errors go to the status word; invalid pages are skipped).
 */
mla_status mla_decode(const mla_geom* geom, const mla_batch* batch, const void* q_lat, const void* q_pe,
                      const mla_cache* cache, const int32_t* block_table, int bt_stride,
                      const int32_t* seq_lens, int checked, void* o_lat, float* lse,
                      void* workspace, size_t ws_bytes, mla_stream_t stream);

/*
 * Absorbed decode over FP8 cache rows ("M5.8" 0x0B "Exact 656-byte FP8 row";
 * the row as mla_fp8_pack_cache writes it: 512 E4M3 latent codes, 4 fp32
 * scales, 64 bf16 RoPE values).  The same computation and plan as mla_decode
 * (mla_plan on the same workspace first), with cache row j's latent value c
 * = E4M3(code_c) * scale_{c / 128}, rounded to bf16 as the tensor-core operand,
 * and its RoPE values as stored.  cache_fp8: uint8 [num_blocks, 64, 656]
 * (contiguous, 16-byte aligned, device); every other argument as for
 * mla_decode.  The page's raw rows are read from HBM once (656 bytes per row,
 * 0.57 of the bf16 row) and converted to bf16 in shared memory.
 */
mla_status mla_decode_fp8(const mla_geom* geom, const mla_batch* batch, const void* q_lat, const void* q_pe,
                          const void* cache_fp8, int num_blocks, const int32_t* block_table, int bt_stride,
                          const int32_t* seq_lens, int checked, void* o_lat, float* lse, void* workspace,
                          size_t ws_bytes, mla_stream_t stream);

/*
 * Index-driven (sparse) decode ("M5.8" 0x0B "FP8 Cache Format And Sparse
 * Selection", the sparse-indices passage: indices [B, S_q, topk] of physical
 * rows, block * 64 + offset, with topk_length [B] bounding each list's valid
 * prefix; "MLA in full detail", the DeepSeek-V3.2 passage: an indexer picks the rows
 * of the latent cache the absorbed decode attends to).  Same arithmetic as
 * mla_decode, but token t of sequence b attends to exactly the rows
 * indices[b, t, 0 .. topk_length[b]) (repeats count once per listing), in any
 * order, instead of a block-table prefix; no causal mask.
 *   batch: B, T (= S_q), num_slots and num_splits_override as for mla_decode;
 *     causal must be 0; max_pages is ignored (taken as ceil(topk / 64)).
 *   q_lat [B,T,H,512], q_pe [B,T,H,64] bf16; o_lat [B,T,H,512] bf16, lse
 *     [B,T,H] float32 (-inf, o = 0 for an empty list); indices int32 [B,T,topk]
 *     and topk_length int32 [B] on the device, 16-byte aligned; a length above
 *     topk counts as topk, a negative one as 0, and either is reported in the
 *     workspace status word (MLA_ERR_DEVICE_CHECK, info = b * S_q + t of the
 *     first token affected), checked or not.
 *   cache: its blocks must be evenly spaced (block stride = 64 x row stride, for
 *     both parts), so that the pool is one array of num_blocks * 64 rows.
 *   checked != 0 reports, in the same word, a listed row outside
 *     [0, num_blocks * 64) (MLA_ERR_DEVICE_CHECK); without it such a row reads
 *     as zeros (it still takes part in the softmax, with score 0).
 * Plans and decodes in one call (no separate mla_plan): the workspace needs
 * mla_sparse_workspace_size(geom, batch, topk) bytes (0 on invalid arguments).
 */
size_t mla_sparse_workspace_size(const mla_geom* geom, const mla_batch* batch, int topk);
mla_status mla_decode_sparse(const mla_geom* geom, const mla_batch* batch, const void* q_lat, const void* q_pe,
                             const mla_cache* cache, const int32_t* indices, int topk, const int32_t* topk_length,
                             int checked, void* o_lat, float* lse, void* workspace, size_t ws_bytes,
                             mla_stream_t stream);

/*
 * Exact merge of split partial states ("M5.8" 0x0C; "mlxcel" Stage-2
 * contract, here with natural-log LSE):
 * part_o float32 [N, rows, D] (each normalised by its own denominator),
 * part_lse float32 [N, rows] (natural log, -inf = empty), indptr int32 [M+1]
 * (partials indptr[m] .. indptr[m+1]-1 form output m).  Writes o bf16 [M, rows, D]
 * and lse float32 [M, rows]: m* = max lse_r, w_r = e^{lse_r - m*},
 * o = sum w_r o_r / sum w_r, lse = m* + ln sum w_r; an output with no
 * non-empty partial gets o = 0, lse = -inf.  D must be a multiple of 8.
 */
mla_status mla_split_merge(const float* part_o, const float* part_lse, const int32_t* indptr, int M,
                           int rows, int D, void* o, float* lse, mla_stream_t stream);

/*
 * FP8 cache rows ("M5.8" 0x0B "Exact 656-byte FP8 row": 512 E4M3 latent values,
 * 4 fp32 scales, 64 bf16 RoPE values).  Packs every row of the bf16 pool in
 * `cache` into out uint8 [num_blocks, 64, 656] (device, 16-byte aligned), row
 * layout: bytes [0,512) E4M3 codes of latent values 0..511; [512,528) fp32
 * scales, scale t for latent values [128t, 128t+128); [528,656) the RoPE values,
 * bf16 (all little-endian).  Scale t = (largest |value| of its tile) / 448 in
 * fp32, 1 for an all-zero tile; code = E4M3 (round to nearest even, saturating
 * at +-448) of value / scale in fp32; the row decodes as value = E4M3 * scale.
 * The pages give the three segments and their sizes; the tile size, scale rule
 * and order are readings.  NaN inputs are not supported.
 */
mla_status mla_fp8_pack_cache(const mla_cache* cache, void* out, mla_stream_t stream);

/*
 * Test export of the paged gather ("M5.8" 0x05 "Paged and ragged address
 * translation": logical row j of sequence b is row j % 64 of block
 * block_table[b, j / 64]): copies the S_b logical rows of sequence b, in order,
 * into out bf16 [S_b, 576] (latent | RoPE), fetching every page with the decode
 * kernel's own tensor maps and load functions.  path 0: the page-half boxes the
 * producer issues (rows [0, 32) and [32, 64), all 576 columns); path 1: the
 * latent columns through the two-column-block boxes of the P V reloads, issued
 * for every column pair of both halves, the RoPE columns as in path 0.  A block
 * id outside [0, num_blocks) reads as zeros, as in the decode.  block_table,
 * seq_lens and out must be 16-byte aligned; S_b is clamped to bt_stride * 64.
 */
mla_status mla_debug_gather(const mla_cache* cache, const int32_t* block_table, int bt_stride,
                            const int32_t* seq_lens, int b, int path, void* out, mla_stream_t stream);

/*
 * Test export of the failure detector: sets, on the current device, the limit in
 * clock cycles of the decode kernel's pipeline waits (a page to land, scores to
 * be written, a merge record to fill); cycles <= 0 restores the default (about
 * one second).  A wait that runs past the limit abandons the launch: the kernel
 * records MLA_ERR_TIMEOUT in the workspace status word (mla_read_device_status),
 * lets every copy and MMA it issued land (those waits keep the full limit),
 * frees its tensor memory and returns, leaving the context usable; the next
 * mla_plan + mla_decode on the workspace run normally.  Synchronous; affects
 * every later decode launch on the device, from any thread, until reset.
 */
mla_status mla_debug_set_wait_limit(long long cycles);

/*
 * Decode for callers that cannot allocate device memory (no counterpart on the
 * source pages; this is a deployment convenience).  Code running inside an
 * allocator or memory-pool callback, or a serving loop that must keep device
 * memory fixed once it starts, can still run a step: this call plans and
 * decodes (plus the split merge) using a fixed scratch array of
 * MLA_NOALLOC_SCRATCH_BYTES held in the library's device image, so the caller
 * passes only inputs and outputs (same meaning as mla_plan + mla_decode with
 * checked = 0).  It calls no allocator.
 *   Checks: every host-side check of mla_decode runs before anything is
 *     launched (the same MLA_ERR_* codes).
 *   Limit: returns MLA_ERR_WORKSPACE, before launching anything, when
 *     mla_workspace_size(geom, batch) exceeds MLA_NOALLOC_SCRATCH_BYTES; a
 *     smaller num_slots (or num_splits_override) shrinks the need.  With
 *     num_slots = 0 and no override the call takes the largest range count, up
 *     to the default, whose workspace fits (the default of one range per CTA
 *     pair needs about 40 MB on a 152-SM GPU).
 *   Errors seen on the device (a length beyond the block table, T > S_b, a
 *     wait that ran out) are recorded in the scratch; mla_read_device_status
 *     called with workspace = NULL returns that status (and clears it).
 *   Set-up: the first call on a device looks up the scratch address with that
 *     device current; make that first call before any stream capture.
 *   Sharing: all calls on a device share the one array (every GPU that loads
 *     the library holds it until exit).  Calls that overlap on the GPU race;
 *     order them on one stream.  Nothing in the array needs clearing between
 *     calls: the planning step rewrites all the state the kernels read.
 */
#define MLA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
mla_status mla_decode_noalloc(const mla_geom* geom, const mla_batch* batch, const void* q_lat, const void* q_pe,
                              const mla_cache* cache, const int32_t* block_table, int bt_stride,
                              const int32_t* seq_lens, void* o_lat, float* lse, mla_stream_t stream);

/*
 * The Normal (decompressed) arm, the baseline the absorbed path is compared
 * with ("MLA in full detail", the naive path of Step 1; "M5.8" 0x02 and
 * 0x06): every cached latent is up-projected into per-head keys and values,
 * then ordinary multi-head attention runs with 192-wide keys [k_nope | k_pe]
 * (k_pe shared by the heads) and 128-wide values, scale geom->softmax_scale.
 *
 * Expanded rows: kv_exp bf16 [H][B * rows_per_seq][256]; row b * rows_per_seq + j
 * of head h holds [W_UK[h] c_j (128) | W_UV[h] c_j (128)] for cache row j of
 * sequence b, rows_per_seq = mla_normal_rows_per_seq(max_pages) (max_pages
 * rounded up to an even count, times 64).  The caller allocates kv_exp
 * (mla_normal_expanded_bytes).
 *
 * mla_normal_expand: writes the rows j < S_b of every sequence, and zeros up
 *   to the next multiple of 128; later rows are not touched.  w_uk, w_uv bf16
 *   [H, 128, 512].  Uses block_table[b, 0 .. ceil(S_b/64)); an id outside
 *   [0, num_blocks) reads as zeros.
 * mla_normal_attention: o bf16 [B, T, H, 128] and lse fp32 [B, T, H] (natural
 *   log) for q_nope bf16 [B, T, H, 128], q_pe bf16 [B, T, H, 64], keys and
 *   values from kv_exp (as written by mla_normal_expand for the same
 *   batch->max_pages and seq_lens) and k_pe from the cache; token t of
 *   sequence b sees cache rows j < S_b - T + t + 1 when batch->causal, else all
 *   S_b.  A row that sees no key gets o = 0, lse = -inf.  batch->num_slots and
 *   num_splits_override are ignored.
 * Both validate on the host (MLA_ERR_ARG / SHAPE / ALIGN as elsewhere) and run
 * asynchronously; a bounded wait that ran out in either is reported by
 * mla_read_device_status (with or without a workspace).
 */
int64_t mla_normal_rows_per_seq(int max_pages);
size_t mla_normal_expanded_bytes(const mla_geom* geom, int B, int max_pages);
mla_status mla_normal_expand(const mla_geom* geom, const mla_cache* cache, const int32_t* block_table, int bt_stride,
                             const int32_t* seq_lens, int B, int max_pages, const void* w_uk, const void* w_uv,
                             void* kv_exp, mla_stream_t stream);
mla_status mla_normal_attention(const mla_geom* geom, const mla_batch* batch, const void* q_nope, const void* q_pe,
                                const mla_cache* cache, const int32_t* block_table, int bt_stride,
                                const int32_t* seq_lens, const void* kv_exp, void* o, float* lse,
                                mla_stream_t stream);

/*
 * Chunked-prefix Normal path (zdszero "MLA", "路径选择" (path choice), the
 * MHA_CHUNKED_KV variant: the prefix is read, expanded and attended one chunk
 * at a time and the chunks' states are merged by LSE, so the expanded prefix
 * held at once is one chunk): the same o and lse as mla_normal_expand +
 * mla_normal_attention, with the expanded rows bounded by chunk_rows rows per
 * sequence.  Window c covers cache rows [c * chunk_rows, (c + 1) * chunk_rows)
 * for c < ceil(max_pages * 64 / chunk_rows); per window the call expands the
 * window's rows into kv_chunk (bf16 [H][B * chunk_rows][256], layout as
 * kv_exp), attends to the window's visible keys, and merges the window's
 * state into a running one ("M5.8" 0x0C merge: m = max lse, weights
 * e^{lse - m}); the last window writes o bf16 [B,T,H,128] and lse fp32 [B,T,H].
 * chunk_rows: a positive multiple of 128.  kv_chunk: mla_normal_chunk_bytes
 * bytes; state: mla_normal_chunk_state_bytes bytes (fp32 running o and lse,
 * overwritten); both 32-byte aligned, owned by the caller.  Two launches per
 * window on the stream; validation and errors as for mla_normal_attention.
 */
size_t mla_normal_chunk_bytes(const mla_geom* geom, int B, int chunk_rows);
size_t mla_normal_chunk_state_bytes(const mla_geom* geom, const mla_batch* batch);
mla_status mla_normal_chunked(const mla_geom* geom, const mla_batch* batch, const void* q_nope, const void* q_pe,
                              const mla_cache* cache, const int32_t* block_table, int bt_stride,
                              const int32_t* seq_lens, const void* w_uk, const void* w_uv, int chunk_rows,
                              void* kv_chunk, void* state, void* o, float* lse, mla_stream_t stream);

/* Synchronise `stream`, then return the status word a kernel recorded in the
 * workspace (MLA_OK if none) and, if info != NULL, its detail word.  The
 * workspace-free kernels (absorption, un-absorption, the Normal arm, the gather
 * export) keep one status word per device, also returned (and cleared) here.
 * With workspace = NULL the call reads that word and then the status and
 * detail words of mla_decode_noalloc's scratch on the current device, returns
 * the first that is set and clears it. */
mla_status mla_read_device_status(const void* workspace, int* info, mla_stream_t stream);

/* Static description of a status code. */
const char* mla_status_string(mla_status status);

/* SMs of the current device (the default for num_slots). */
int mla_device_sm_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H_ */
