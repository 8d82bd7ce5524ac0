// The C ABI of libmla.so (declared in include/mla.h): host-side validation,
// workspace layout and kernel launches.  No allocation, no synchronisation
// (except mla_read_device_status).
#include <string.h>

#include <atomic>

#include "mla_internal.cuh"

namespace mla {

cudaError_t launch_fp8_pack(const CacheView& cv, unsigned char* out, cudaStream_t st);  // mla_fp8.cu

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

mla_status check_geom(const mla_geom* g) {
  if (!g) return MLA_ERR_ARG;
  if (g->d_lat != kDLat || g->d_rope != kDRope || g->d_nope != kDNope || g->d_v != kDV || g->block_size != kPage)
    return MLA_ERR_SHAPE;
  if (g->H < 1 || g->H > kRowsPerBlock || (kRowsPerBlock % g->H) != 0) return MLA_ERR_SHAPE;
  if (!(g->softmax_scale > 0.f)) return MLA_ERR_ARG;
  return MLA_OK;
}

mla_status check_batch(const mla_batch* b) {
  if (!b) return MLA_ERR_ARG;
  if (b->B < 0 || b->T < 1 || b->max_pages < 1 || b->num_slots < 0 || b->num_splits_override < 0)
    return MLA_ERR_ARG;
  if ((long long)b->T * kRowsPerBlock > (1LL << 24)) return MLA_ERR_SHAPE;
  return MLA_OK;
}

mla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

}  // namespace

// Default work-range count: one per CTA pair of the decode kernel (half the SMs).
int resolve_slots(const mla_batch* b) {
  if (b->num_slots > 0) return b->num_slots;
  return decode_sm103_pairs_per_device();
}

bool compute_layout(const mla_geom* g, const mla_batch* b, WsLayout* L) {
  const long long RB = ((long long)b->T * g->H + kRowsPerBlock - 1) / kRowsPerBlock;
  const long long groups = (long long)b->B * RB;
  const int G = resolve_slots(b);
  long long cap_ranges, cap_segments, cap_partials;
  if (b->num_splits_override > 0) {
    const long long k = b->num_splits_override < b->max_pages ? b->num_splits_override : b->max_pages;
    cap_ranges = cap_segments = cap_partials = groups * k;
  } else {
    cap_ranges = G;
    cap_segments = groups + G;
    cap_partials = 2LL * G;
  }
  if (groups > (1 << 26) || cap_segments > (1 << 26)) return false;
  size_t off = align_up(MLA_HDR_WORDS * sizeof(int));
  L->off_groups = off;     off = align_up(off + (size_t)groups * kGroupWords * sizeof(int));
  L->off_segments = off;   off = align_up(off + (size_t)cap_segments * kSegWords * sizeof(int));
  L->off_range_ptr = off;  off = align_up(off + (size_t)(cap_ranges + 1) * sizeof(int));
  L->off_merge = off;      off = align_up(off + (size_t)groups * kMergeWords * sizeof(int));
  L->off_merge_sync = off; off = align_up(off + (size_t)groups * 2 * sizeof(int));
  L->off_part_lse = off;   off = align_up(off + (size_t)cap_partials * kRowsPerBlock * sizeof(float));
  L->off_part_o = off;     off = align_up(off + (size_t)cap_partials * kRowsPerBlock * kDLat * sizeof(float));
  L->total = off;
  L->cap_groups = (int)groups;
  L->cap_segments = (int)cap_segments;
  L->cap_ranges = (int)cap_ranges;
  L->cap_partials = (int)cap_partials;
  L->num_slots = G;
  return true;
}

}  // namespace mla

using namespace mla;

extern "C" {

int mla_device_sm_count(void) {
  // Filled on first use per device; concurrent first calls store the same value.
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_acquire);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_release);
  }
  return n;
}

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_ARG: return "invalid argument";
    case MLA_ERR_SHAPE: return "unsupported geometry or shape";
    case MLA_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case MLA_ERR_WORKSPACE: return "workspace too small";
    case MLA_ERR_PLAN_STALE: return "plan built for other lengths or geometry";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_DEVICE_CHECK: return "device check failed (block id, length or T)";
    case MLA_ERR_TIMEOUT: return "bounded wait ran out";
  }
  return "unknown status";
}

size_t mla_workspace_size(const mla_geom* geom, const mla_batch* batch) {
  if (check_geom(geom) != MLA_OK || check_batch(batch) != MLA_OK) return 0;
  WsLayout L;
  if (!compute_layout(geom, batch, &L)) return 0;
  return L.total;
}

mla_status mla_plan(const mla_geom* geom, const mla_batch* batch, const int32_t* seq_lens, void* workspace,
                    size_t ws_bytes, mla_stream_t stream) {
  mla_status s = check_geom(geom);
  if (s != MLA_OK) return s;
  if ((s = check_batch(batch)) != MLA_OK) return s;
  if (!workspace || (batch->B > 0 && !seq_lens)) return MLA_ERR_ARG;
  if (!aligned32(workspace) || !aligned16(seq_lens)) return MLA_ERR_ALIGN;
  WsLayout L;
  if (!compute_layout(geom, batch, &L)) return MLA_ERR_SHAPE;
  if (ws_bytes < L.total) return MLA_ERR_WORKSPACE;
  return cuda_status(launch_plan(seq_lens, geom, batch, L, workspace, (cudaStream_t)stream));
}

mla_status mla_absorb_q(const mla_geom* geom, const void* q_nope, const void* w_uk, void* q_lat, int BT,
                        mla_stream_t stream) {
  mla_status s = check_geom(geom);
  if (s != MLA_OK) return s;
  if (BT < 0) return MLA_ERR_ARG;
  if (BT == 0) return MLA_OK;
  if (!q_nope || !w_uk || !q_lat) return MLA_ERR_ARG;
  if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned32(q_lat)) return MLA_ERR_ALIGN;
  return cuda_status(launch_absorb_sm103(static_cast<const __nv_bfloat16*>(q_nope), static_cast<const __nv_bfloat16*>(w_uk),
                                   static_cast<__nv_bfloat16*>(q_lat), BT, geom->H, (cudaStream_t)stream));
}

mla_status mla_unabsorb_o(const mla_geom* geom, const void* o_lat, const void* w_uv, void* o, int BT,
                          mla_stream_t stream) {
  mla_status s = check_geom(geom);
  if (s != MLA_OK) return s;
  if (BT < 0) return MLA_ERR_ARG;
  if (BT == 0) return MLA_OK;
  if (!o_lat || !w_uv || !o) return MLA_ERR_ARG;
  if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned32(o)) return MLA_ERR_ALIGN;
  return cuda_status(launch_unabsorb_sm103(static_cast<const __nv_bfloat16*>(o_lat), static_cast<const __nv_bfloat16*>(w_uv),
                                     static_cast<__nv_bfloat16*>(o), BT, geom->H, (cudaStream_t)stream));
}

static mla_status check_cache(const mla_cache* cache, CacheView* cv);

}  // extern "C"

// Host validation of mla_decode's arguments other than the workspace.
mla_status mla::check_decode_args(const mla_geom* geom, const mla_batch* batch, const void* q_lat, const void* q_pe,
                                  const mla_cache* cache, const int32_t* block_table, int bt_stride,
                                  const int32_t* seq_lens, const void* o_lat, const float* lse, CacheView* cv) {
  mla_status s = check_geom(geom);
  if (s != MLA_OK) return s;
  if ((s = check_batch(batch)) != MLA_OK) return s;
  if (batch->B == 0) return MLA_OK;
  if (!q_lat || !q_pe || !block_table || !seq_lens || !o_lat || !lse) return MLA_ERR_ARG;
  if (bt_stride < batch->max_pages) return MLA_ERR_ARG;
  if (!aligned16(q_lat) || !aligned16(q_pe) || !aligned32(o_lat) || !aligned16(lse) || !aligned16(block_table) ||
      !aligned16(seq_lens))
    return MLA_ERR_ALIGN;
  return check_cache(cache, cv);
}

extern "C" {

static mla_status check_cache(const mla_cache* cache, CacheView* cv) {
  if (!cache || !cache->ckv || !cache->kpe || cache->num_blocks < 1) return MLA_ERR_ARG;
  if (cache->ckv_row_stride < 1 || cache->kpe_row_stride < 1 || cache->ckv_block_stride < 1 ||
      cache->kpe_block_stride < 1)
    return MLA_ERR_ARG;
  if (!aligned16(cache->ckv) || !aligned16(cache->kpe)) return MLA_ERR_ALIGN;
  if ((cache->ckv_row_stride * 2) % 16 != 0 || (cache->ckv_block_stride * 2) % 16 != 0 ||
      (cache->kpe_row_stride * 2) % 16 != 0 || (cache->kpe_block_stride * 2) % 16 != 0)
    return MLA_ERR_ALIGN;
  cv->ckv = static_cast<const __nv_bfloat16*>(cache->ckv);
  cv->kpe = static_cast<const __nv_bfloat16*>(cache->kpe);
  cv->ckv_row = cache->ckv_row_stride;
  cv->ckv_block = cache->ckv_block_stride;
  cv->kpe_row = cache->kpe_row_stride;
  cv->kpe_block = cache->kpe_block_stride;
  cv->num_blocks = cache->num_blocks;
  return MLA_OK;
}

mla_status mla_decode(const mla_geom* geom, const mla_batch* batch, const void* q_lat, const void* q_pe,
                      const mla_cache* cache, const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                      int checked, void* o_lat, float* lse, void* workspace, size_t ws_bytes, mla_stream_t stream) {
  CacheView cv;
  mla_status s = check_decode_args(geom, batch, q_lat, q_pe, cache, block_table, bt_stride, seq_lens, o_lat, lse, &cv);
  if (s != MLA_OK) return s;
  if (batch->B == 0) return MLA_OK;
  if (!workspace) return MLA_ERR_ARG;
  if (!aligned32(workspace)) return MLA_ERR_ALIGN;
  WsLayout L;
  if (!compute_layout(geom, batch, &L)) return MLA_ERR_SHAPE;
  if (ws_bytes < L.total) return MLA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  // One kernel: the split-KV decode, and (when the plan has merge records) the
  // LSE merge of each split group by the CTAs that finish its partial states last.
  return cuda_status(launch_decode_sm103(geom, batch, L, static_cast<const __nv_bfloat16*>(q_lat),
                                         static_cast<const __nv_bfloat16*>(q_pe), cv, block_table, bt_stride,
                                         seq_lens, checked, static_cast<__nv_bfloat16*>(o_lat), lse, workspace, st));
}

mla_status mla_decode_fp8(const mla_geom* geom, const mla_batch* batch, const void* q_lat, const void* q_pe,
                          const void* cache_fp8, int num_blocks, const int32_t* block_table, int bt_stride,
                          const int32_t* seq_lens, int checked, void* o_lat, float* lse, void* workspace,
                          size_t ws_bytes, mla_stream_t stream) {
  mla_status s = check_geom(geom);
  if (s != MLA_OK) return s;
  if ((s = check_batch(batch)) != MLA_OK) return s;
  if (batch->B == 0) return MLA_OK;
  if (!q_lat || !q_pe || !cache_fp8 || !block_table || !seq_lens || !o_lat || !lse || !workspace) return MLA_ERR_ARG;
  if (num_blocks < 1 || bt_stride < batch->max_pages) return MLA_ERR_ARG;
  if ((long long)num_blocks * kPage >= (1LL << 31)) return MLA_ERR_SHAPE;
  if (!aligned16(q_lat) || !aligned16(q_pe) || !aligned16(cache_fp8) || !aligned16(block_table) ||
      !aligned16(seq_lens) || !aligned32(o_lat) || !aligned16(lse) || !aligned32(workspace))
    return MLA_ERR_ALIGN;
  WsLayout L;
  if (!compute_layout(geom, batch, &L)) return MLA_ERR_SHAPE;
  if (ws_bytes < L.total) return MLA_ERR_WORKSPACE;
  CacheView cv{};
  cv.num_blocks = num_blocks;
  const Fp8Pool pool{static_cast<const unsigned char*>(cache_fp8), num_blocks};
  return cuda_status(launch_decode_sm103(geom, batch, L, static_cast<const __nv_bfloat16*>(q_lat),
                                         static_cast<const __nv_bfloat16*>(q_pe), cv, block_table, bt_stride,
                                         seq_lens, checked, static_cast<__nv_bfloat16*>(o_lat), lse, workspace,
                                         (cudaStream_t)stream, nullptr, &pool));
}

// The sparse decode as a dense one over B * S_q one-token sequences of up to topk
// listed rows (non-causal), lengths topk_length[b] shared by sequence b's tokens.
static bool sparse_batch(const mla_batch* batch, int topk, mla_batch* vb) {
  if (!batch || topk < 1 || batch->B < 0 || batch->T < 1 || batch->causal) return false;
  if ((long long)batch->B * batch->T > (1LL << 26)) return false;
  *vb = *batch;
  vb->B = batch->B * batch->T;
  vb->T = 1;
  vb->causal = 0;
  vb->max_pages = (topk + kPage - 1) / kPage;
  return true;
}

size_t mla_sparse_workspace_size(const mla_geom* geom, const mla_batch* batch, int topk) {
  mla_batch vb;
  if (!sparse_batch(batch, topk, &vb)) return 0;
  return mla_workspace_size(geom, &vb);
}

mla_status mla_decode_sparse(const mla_geom* geom, const mla_batch* batch, const void* q_lat, const void* q_pe,
                             const mla_cache* cache, const int32_t* indices, int topk, const int32_t* topk_length,
                             int checked, void* o_lat, float* lse, void* workspace, size_t ws_bytes,
                             mla_stream_t stream) {
  mla_status s = check_geom(geom);
  if (s != MLA_OK) return s;
  mla_batch vb;
  if (!sparse_batch(batch, topk, &vb)) return MLA_ERR_ARG;
  if ((s = check_batch(&vb)) != MLA_OK) return s;
  if (vb.B == 0) return MLA_OK;
  if (!q_lat || !q_pe || !indices || !topk_length || !o_lat || !lse || !workspace) return MLA_ERR_ARG;
  if (!aligned16(q_lat) || !aligned16(q_pe) || !aligned16(indices) || !aligned16(topk_length) || !aligned32(o_lat) ||
      !aligned16(lse) || !aligned32(workspace))
    return MLA_ERR_ALIGN;
  CacheView cv;
  if ((s = check_cache(cache, &cv)) != MLA_OK) return s;
  // The pool's rows must be evenly spaced across blocks (one 2-D array of rows).
  if (cv.ckv_block != (int64_t)kPage * cv.ckv_row || cv.kpe_block != (int64_t)kPage * cv.kpe_row) return MLA_ERR_ARG;
  if ((long long)cv.num_blocks * kPage >= (1LL << 31)) return MLA_ERR_SHAPE;
  WsLayout L;
  if (!compute_layout(geom, &vb, &L)) return MLA_ERR_SHAPE;
  if (ws_bytes < L.total) return MLA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  if (launch_plan(topk_length, geom, &vb, L, workspace, st, batch->T, topk) != cudaSuccess) return MLA_ERR_CUDA;
  const SparseList list{indices, topk, batch->T};
  return cuda_status(launch_decode_sm103(geom, &vb, L, static_cast<const __nv_bfloat16*>(q_lat),
                                         static_cast<const __nv_bfloat16*>(q_pe), cv, nullptr, 0, topk_length,
                                         checked, static_cast<__nv_bfloat16*>(o_lat), lse, workspace, st, &list));
}

mla_status mla_split_merge(const float* part_o, const float* part_lse, const int32_t* indptr, int M, int rows, int D,
                           void* o, float* lse, mla_stream_t stream) {
  if (M < 0 || rows < 0 || D <= 0 || (D % 8) != 0) return MLA_ERR_ARG;
  if (M == 0 || rows == 0) return MLA_OK;
  if (!part_o || !part_lse || !indptr || !o || !lse) return MLA_ERR_ARG;
  if (!aligned16(part_o) || !aligned16(part_lse) || !aligned16(o) || !aligned16(lse) || !aligned16(indptr))
    return MLA_ERR_ALIGN;
  if (((size_t)rows * D * sizeof(float)) % 16 != 0) return MLA_ERR_ALIGN;
  return cuda_status(launch_split_merge(part_o, part_lse, indptr, M, rows, D, static_cast<__nv_bfloat16*>(o), lse,
                                        (cudaStream_t)stream));
}

mla_status mla_fp8_pack_cache(const mla_cache* cache, void* out, mla_stream_t stream) {
  if (!out) return MLA_ERR_ARG;
  if (!aligned16(out)) return MLA_ERR_ALIGN;
  CacheView cv;
  mla_status s = check_cache(cache, &cv);
  if (s != MLA_OK) return s;
  return cuda_status(launch_fp8_pack(cv, static_cast<unsigned char*>(out), (cudaStream_t)stream));
}

mla_status mla_debug_gather(const mla_cache* cache, const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                            int b, int path, void* out, mla_stream_t stream) {
  if (!block_table || !seq_lens || !out || b < 0 || bt_stride < 1 || (path != 0 && path != 1)) return MLA_ERR_ARG;
  if (!aligned16(out) || !aligned16(block_table) || !aligned16(seq_lens)) return MLA_ERR_ALIGN;
  CacheView cv;
  mla_status s = check_cache(cache, &cv);
  if (s != MLA_OK) return s;
  return cuda_status(launch_debug_gather(cv, block_table, bt_stride, seq_lens, b, path,
                                         static_cast<__nv_bfloat16*>(out), (cudaStream_t)stream));
}

mla_status mla_debug_set_wait_limit(long long cycles) {
  return cuda_status(set_pipeline_wait_limit(cycles));
}

int64_t mla_normal_rows_per_seq(int max_pages) { return max_pages < 1 ? 0 : normal_rows_per_seq(max_pages); }

size_t mla_normal_expanded_bytes(const mla_geom* geom, int B, int max_pages) {
  if (check_geom(geom) != MLA_OK || B < 0 || max_pages < 1) return 0;
  return (size_t)geom->H * (size_t)B * (size_t)normal_rows_per_seq(max_pages) * 256 * 2;
}

mla_status mla_normal_expand(const mla_geom* geom, const mla_cache* cache, const int32_t* block_table, int bt_stride,
                             const int32_t* seq_lens, int B, int max_pages, const void* w_uk, const void* w_uv,
                             void* kv_exp, mla_stream_t stream) {
  mla_status s = check_geom(geom);
  if (s != MLA_OK) return s;
  if (B < 0 || max_pages < 1) return MLA_ERR_ARG;
  if (B == 0) return MLA_OK;
  if (!block_table || !seq_lens || !w_uk || !w_uv || !kv_exp || bt_stride < max_pages) return MLA_ERR_ARG;
  if ((long long)B * normal_rows_per_seq(max_pages) >= (1LL << 31)) return MLA_ERR_SHAPE;
  if (!aligned16(block_table) || !aligned16(seq_lens) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned32(kv_exp))
    return MLA_ERR_ALIGN;
  CacheView cv;
  if ((s = check_cache(cache, &cv)) != MLA_OK) return s;
  return cuda_status(launch_normal_expand(geom, cv, block_table, bt_stride, seq_lens, B, max_pages,
                                          static_cast<const __nv_bfloat16*>(w_uk),
                                          static_cast<const __nv_bfloat16*>(w_uv),
                                          static_cast<__nv_bfloat16*>(kv_exp), (cudaStream_t)stream));
}

mla_status mla_normal_attention(const mla_geom* geom, const mla_batch* batch, const void* q_nope, const void* q_pe,
                                const mla_cache* cache, const int32_t* block_table, int bt_stride,
                                const int32_t* seq_lens, const void* kv_exp, void* o, float* lse,
                                mla_stream_t stream) {
  mla_status s = check_geom(geom);
  if (s != MLA_OK) return s;
  if ((s = check_batch(batch)) != MLA_OK) return s;
  if (batch->B == 0) return MLA_OK;
  if (!q_nope || !q_pe || !block_table || !seq_lens || !kv_exp || !o || !lse) return MLA_ERR_ARG;
  if (bt_stride < batch->max_pages) return MLA_ERR_ARG;
  if ((long long)batch->B * normal_rows_per_seq(batch->max_pages) >= (1LL << 31) || batch->B > 65535 ||
      (batch->T + 127) / 128 > 65535)
    return MLA_ERR_SHAPE;
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(block_table) || !aligned16(seq_lens) ||
      !aligned16(kv_exp) || !aligned32(o) || !aligned16(lse))
    return MLA_ERR_ALIGN;
  CacheView cv;
  if ((s = check_cache(cache, &cv)) != MLA_OK) return s;
  return cuda_status(launch_normal_attention(geom, batch, static_cast<const __nv_bfloat16*>(q_nope),
                                             static_cast<const __nv_bfloat16*>(q_pe), cv, block_table, bt_stride,
                                             seq_lens, static_cast<const __nv_bfloat16*>(kv_exp),
                                             static_cast<__nv_bfloat16*>(o), lse, (cudaStream_t)stream));
}

size_t mla_normal_chunk_bytes(const mla_geom* geom, int B, int chunk_rows) {
  if (check_geom(geom) != MLA_OK || B < 0 || chunk_rows < 128 || chunk_rows % 128 != 0) return 0;
  return (size_t)geom->H * (size_t)B * (size_t)chunk_rows * 256 * 2;
}

size_t mla_normal_chunk_state_bytes(const mla_geom* geom, const mla_batch* batch) {
  if (check_geom(geom) != MLA_OK || check_batch(batch) != MLA_OK) return 0;
  const size_t rows = (size_t)batch->B * batch->T * geom->H;
  return align_up(rows * kDV * 4) + align_up(rows * 4);
}

mla_status mla_normal_chunked(const mla_geom* geom, const mla_batch* batch, const void* q_nope, const void* q_pe,
                              const mla_cache* cache, const int32_t* block_table, int bt_stride,
                              const int32_t* seq_lens, const void* w_uk, const void* w_uv, int chunk_rows,
                              void* kv_chunk, void* state, void* o, float* lse, mla_stream_t stream) {
  mla_status s = check_geom(geom);
  if (s != MLA_OK) return s;
  if ((s = check_batch(batch)) != MLA_OK) return s;
  if (chunk_rows < 128 || chunk_rows % 128 != 0) return MLA_ERR_ARG;
  if (batch->B == 0) return MLA_OK;
  if (!q_nope || !q_pe || !block_table || !seq_lens || !w_uk || !w_uv || !kv_chunk || !state || !o || !lse)
    return MLA_ERR_ARG;
  if (bt_stride < batch->max_pages) return MLA_ERR_ARG;
  if ((long long)batch->B * chunk_rows >= (1LL << 31) || batch->B > 65535 || (batch->T + 127) / 128 > 65535)
    return MLA_ERR_SHAPE;
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(block_table) || !aligned16(seq_lens) ||
      !aligned16(w_uk) || !aligned16(w_uv) || !aligned32(kv_chunk) || !aligned32(state) || !aligned32(o) ||
      !aligned16(lse))
    return MLA_ERR_ALIGN;
  CacheView cv;
  if ((s = check_cache(cache, &cv)) != MLA_OK) return s;
  const size_t rows = (size_t)batch->B * batch->T * geom->H;
  float* st_o = static_cast<float*>(state);
  float* st_lse = reinterpret_cast<float*>(static_cast<char*>(state) + align_up(rows * kDV * 4));
  return cuda_status(launch_normal_chunked(geom, batch, static_cast<const __nv_bfloat16*>(q_nope),
                                           static_cast<const __nv_bfloat16*>(q_pe), cv, block_table, bt_stride,
                                           seq_lens, static_cast<const __nv_bfloat16*>(w_uk),
                                           static_cast<const __nv_bfloat16*>(w_uv), chunk_rows,
                                           static_cast<__nv_bfloat16*>(kv_chunk), st_o, st_lse,
                                           static_cast<__nv_bfloat16*>(o), lse, (cudaStream_t)stream));
}

mla_status mla_read_device_status(const void* workspace, int* info, mla_stream_t stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (info) *info = 0;
  if (workspace) {
    int words[2] = {0, 0};
    const char* base = static_cast<const char*>(workspace) + MLA_HDR_ERROR * sizeof(int);
    if (cudaMemcpy(words, base, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
    if (info) *info = words[1];
    if (words[0] != 0) return (mla_status)words[0];
  }
  // Kernels without a workspace keep their (rare) timeout in one word per device.
  int* bmm = bmm_status_ptr();
  if (bmm) {
    int v = 0;
    if (cudaMemcpy(&v, bmm, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
    if (v != 0) {
      const int zero = 0;
      cudaMemcpy(bmm, &zero, sizeof(int), cudaMemcpyHostToDevice);
      if (info) *info = -1;
      return (mla_status)v;
    }
  }
  // mla_decode_noalloc plans and decodes in the library's own scratch: its status
  // word (and detail) is read here, without a workspace, and cleared.
  if (!workspace) {
    int* na = noalloc_status_words();
    if (na) {
      int words[2] = {0, 0};
      if (cudaMemcpy(words, na, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
      if (words[0] != 0) {
        const int zero[2] = {0, 0};
        cudaMemcpy(na, zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (info) *info = words[1];
        return (mla_status)words[0];
      }
    }
  }
  return MLA_OK;
}

}  // extern "C"
