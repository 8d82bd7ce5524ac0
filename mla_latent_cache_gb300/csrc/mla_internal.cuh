// Internal declarations shared by the libmla translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

constexpr int kDLat = 512;
constexpr int kDRope = 64;
constexpr int kDK = kDLat + kDRope;  // 576
constexpr int kDNope = 128;
constexpr int kDV = 128;
constexpr int kPage = 64;
constexpr int kRowsPerBlock = 128;   // flattened (t, h) query rows per group
constexpr int kMinSplitPages = 4;
constexpr int kSegWords = 8;
constexpr int kMergeWords = 4;
constexpr int kGroupWords = 8;

// Workspace layout, computed on the host from (geometry, batch shape, slots).
struct WsLayout {
  size_t off_groups, off_segments, off_range_ptr, off_merge, off_merge_sync, off_part_lse, off_part_o, total;
  int cap_groups, cap_segments, cap_ranges, cap_partials;
  int num_slots;
};

bool compute_layout(const mla_geom* g, const mla_batch* b, WsLayout* L);
int resolve_slots(const mla_batch* b);
struct CacheView;
// Host validation of mla_decode's arguments other than the workspace (fills cv).
mla_status check_decode_args(const mla_geom* geom, const mla_batch* batch, const void* q_lat, const void* q_pe,
                             const mla_cache* cache, const int32_t* block_table, int bt_stride,
                             const int32_t* seq_lens, const void* o_lat, const float* lse, CacheView* cv);
// Status and detail words of mla_decode_noalloc's scratch on the current device,
// or nullptr before that entry point's first call there.
int* noalloc_status_words();

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation and waits for the grid before it in the
// stream (pdl_wait) before its first global-memory access, so its set-up
// (barriers, TMEM, tensor-map prefetch) overlaps the tail of that grid; it
// lets the next grid start its own set-up (pdl_trigger) once all of its CTAs
// are running.  Without a programmatic predecessor the wait returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Status word helpers (device): first error wins.
__device__ __forceinline__ void record_error(int* hdr, int code, int info) {
  if (atomicCAS(&hdr[MLA_HDR_ERROR], 0, code) == 0) {
    atomicExch(&hdr[MLA_HDR_ERROR_INFO], info);
  }
}

// Paged address translation ("M5.8", 0x05): physical row of logical row j of
// sequence b is block_table[b, j / 64] * 64 + j % 64; the element offset of
// that row is block * block_stride + (j % 64) * row_stride.
struct CacheView {
  const __nv_bfloat16* ckv;
  const __nv_bfloat16* kpe;
  int64_t ckv_row, ckv_block, kpe_row, kpe_block;
  int num_blocks;
};

__device__ __forceinline__ const __nv_bfloat16* ckv_row_ptr(const CacheView& c, int block, int j_in_page) {
  return c.ckv + (int64_t)block * c.ckv_block + (int64_t)j_in_page * c.ckv_row;
}
__device__ __forceinline__ const __nv_bfloat16* kpe_row_ptr(const CacheView& c, int block, int j_in_page) {
  return c.kpe + (int64_t)block * c.kpe_block + (int64_t)j_in_page * c.kpe_row;
}

// Visible rows of query token t (bottom-right causal alignment).
__host__ __device__ __forceinline__ int visible_limit(int S, int T, int t, int causal) {
  if (!causal) return S;
  int v = S - T + t + 1;
  return v < 0 ? 0 : (v > S ? S : v);
}

// Launchers (one per translation unit); all return cudaError_t of the launch.
cudaError_t launch_plan(const int32_t* seq_lens, const mla_geom* g, const mla_batch* b,
                        const WsLayout& L, void* ws, cudaStream_t st, int seq_div = 1, int max_rows = 0);
// The sparse decode's index lists: physical rows indices [B', topk] for the
// B' = B * seq_div (sequence, query token) pairs, lengths seq_lens[b' / seq_div].
struct SparseList {
  const int32_t* indices;
  int topk, seq_div;
};
// The FP8 decode's cache: num_blocks x 64 rows of 656 bytes, contiguous.
struct Fp8Pool {
  const unsigned char* rows;
  int num_blocks;
};
cudaError_t launch_decode_sm103(const mla_geom* g, const mla_batch* b, const WsLayout& L,
                                const __nv_bfloat16* q_lat, const __nv_bfloat16* q_pe, const CacheView& cv,
                                const int32_t* block_table, int bt_stride, const int32_t* seq_lens, int checked,
                                __nv_bfloat16* o_lat, float* lse, void* ws, cudaStream_t st,
                                const SparseList* sparse = nullptr, const Fp8Pool* fp8 = nullptr);
int decode_sm103_pairs_per_device();
cudaError_t launch_split_merge(const float* part_o, const float* part_lse, const int32_t* indptr, int M,
                               int rows, int D, __nv_bfloat16* o, float* lse, cudaStream_t st);
cudaError_t launch_absorb_sm103(const __nv_bfloat16* q_nope, const __nv_bfloat16* w_uk, __nv_bfloat16* q_lat,
                                int BT, int H, cudaStream_t st);
cudaError_t launch_unabsorb_sm103(const __nv_bfloat16* o_lat, const __nv_bfloat16* w_uv, __nv_bfloat16* o,
                                  int BT, int H, cudaStream_t st);
int* bmm_status_ptr();
int64_t normal_rows_per_seq(int max_pages);
cudaError_t launch_normal_expand(const mla_geom* g, const CacheView& cv, const int32_t* block_table, int bt_stride,
                                 const int32_t* seq_lens, int B, int max_pages, const __nv_bfloat16* w_uk,
                                 const __nv_bfloat16* w_uv, __nv_bfloat16* kv_exp, cudaStream_t st);
cudaError_t launch_normal_attention(const mla_geom* g, const mla_batch* b, const __nv_bfloat16* q_nope,
                                    const __nv_bfloat16* q_pe, const CacheView& cv, const int32_t* block_table,
                                    int bt_stride, const int32_t* seq_lens, const __nv_bfloat16* kv_exp,
                                    __nv_bfloat16* o, float* lse, cudaStream_t st);
// The chunked-prefix Normal path over windows of chunk_rows (a multiple of 128)
// cache rows; kv_chunk holds one window ([H][B * chunk_rows][256]), st_o / st_lse
// the running state (fp32 [B,T,H,128] and [B,T,H]).
cudaError_t launch_normal_chunked(const mla_geom* g, const mla_batch* bt, const __nv_bfloat16* q_nope,
                                  const __nv_bfloat16* q_pe, const CacheView& cv, const int32_t* block_table,
                                  int bt_stride, const int32_t* seq_lens, const __nv_bfloat16* w_uk,
                                  const __nv_bfloat16* w_uv, int chunk_rows, __nv_bfloat16* kv_chunk, float* st_o,
                                  float* st_lse, __nv_bfloat16* o, float* lse, cudaStream_t st);
cudaError_t launch_debug_gather(const CacheView& cv, const int32_t* block_table, int bt_stride,
                                const int32_t* seq_lens, int b, int path, __nv_bfloat16* out, cudaStream_t st);
// Limit (clock cycles) of the decode kernel's pipeline waits on the current device; <= 0: the default.
cudaError_t set_pipeline_wait_limit(long long cycles);

}  // namespace mla
