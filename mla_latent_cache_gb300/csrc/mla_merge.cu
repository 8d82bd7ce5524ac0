// Exact log-sum-exp merge of split-KV partial states.
//
// "M5.8" 0x0C: for partial states (m_r, l_r, o_r) the merged state is
// m = max m_r, l = sum e^{m_r - m} l_r, o = sum e^{m_r - m} o_r, O = o / l.
// With partials stored normalised (o_r / l_r) together with
// lse_r = m_r + ln l_r (the "mlxcel" Stage-2 contract, natural-log units here),
// the weight of partial r is w_r = e^{lse_r - max lse}, and
// O = sum w_r (o_r / l_r) / sum w_r, lse = max lse + ln sum w_r.
#include <math.h>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMaxCached = 64;  // partial weights kept in shared memory per row chunk

// Merge `count` partials for `nrows` rows of width D starting at partial `first`.
// part_o rows are addressed as part_o[(first + r) * row_pitch + row * D + c].
__device__ void merge_rows(const float* part_o, const float* part_lse, size_t o_pitch, size_t lse_pitch,
                           int first, int count, int nrows, int D, __nv_bfloat16* o_out, float* lse_out) {
  __shared__ float s_w[kMaxCached];
  __shared__ float s_inv;
  __shared__ float s_lse;
  for (int row = 0; row < nrows; ++row) {
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = -INFINITY;
      for (int r = 0; r < count; ++r) m = fmaxf(m, part_lse[(size_t)(first + r) * lse_pitch + row]);
      float l = 0.f;
      const float m_use = (m == -INFINITY) ? 0.f : m;
      for (int r = 0; r < count; ++r) {
        const float x = part_lse[(size_t)(first + r) * lse_pitch + row];
        const float w = (x == -INFINITY) ? 0.f : __expf(x - m_use);
        if (r < kMaxCached) s_w[r] = w;
        l += w;
      }
      s_inv = l > 0.f ? 1.f / l : 0.f;
      s_lse = l > 0.f ? m_use + logf(l) : -INFINITY;
    }
    __syncthreads();
    const float inv = s_inv;
    float m_use = 0.f;
    if (count > kMaxCached) {  // recompute the max for weights past the cache
      m_use = -INFINITY;
      for (int r = 0; r < count; ++r) m_use = fmaxf(m_use, part_lse[(size_t)(first + r) * lse_pitch + row]);
      if (m_use == -INFINITY) m_use = 0.f;
    }
    for (int c2 = threadIdx.x * 2; c2 < D; c2 += blockDim.x * 2) {
      float a0 = 0.f, a1 = 0.f;
      for (int r = 0; r < count; ++r) {
        float w;
        if (r < kMaxCached) {
          w = s_w[r];
        } else {
          const float x = part_lse[(size_t)(first + r) * lse_pitch + row];
          w = (x == -INFINITY) ? 0.f : __expf(x - m_use);
        }
        if (w != 0.f) {
          const float2 v = *reinterpret_cast<const float2*>(part_o + (size_t)(first + r) * o_pitch + (size_t)row * D + c2);
          a0 = fmaf(w, v.x, a0);
          a1 = fmaf(w, v.y, a1);
        }
      }
      *reinterpret_cast<__nv_bfloat162*>(o_out + (size_t)row * D + c2) = __floats2bfloat162_rn(a0 * inv, a1 * inv);
    }
    if (threadIdx.x == 0) lse_out[row] = s_lse;
  }
}

struct PlanMergeArgs {
  int T, H;
  __nv_bfloat16* o_lat;
  float* lse;
  WsLayout L;
};

// One CTA per merge record of the plan (groups that were split, or are empty).
__global__ void __launch_bounds__(kMergeThreads) plan_merge_kernel(PlanMergeArgs a, const char* ws) {
  const int* hdr = reinterpret_cast<const int*>(ws);
  const int* mrg = reinterpret_cast<const int*>(ws + a.L.off_merge);
  const float* part_lse = reinterpret_cast<const float*>(ws + a.L.off_part_lse);
  const float* part_o = reinterpret_cast<const float*>(ws + a.L.off_part_o);
  const int num_merge = hdr[MLA_HDR_NUM_MERGE];
  const int R = a.T * a.H;
  for (int i = blockIdx.x; i < num_merge; i += gridDim.x) {
    const int b = mrg[i * kMergeWords + 0], rb = mrg[i * kMergeWords + 1];
    const int first = mrg[i * kMergeWords + 2], count = mrg[i * kMergeWords + 3];
    const int row0 = rb * kRowsPerBlock;
    const int nrows = min(kRowsPerBlock, R - row0);
    const size_t grow = (size_t)b * R + row0;
    merge_rows(part_o, part_lse, (size_t)kRowsPerBlock * kDLat, kRowsPerBlock, first, count, nrows, kDLat,
               a.o_lat + grow * kDLat, a.lse + grow);
  }
}

struct SplitMergeArgs {
  const float* part_o;
  const float* part_lse;
  const int32_t* indptr;
  int M, rows, D;
  __nv_bfloat16* o;
  float* lse;
};

// Public contract: one CTA per (output m, chunk of 32 rows).
__global__ void __launch_bounds__(kMergeThreads) split_merge_kernel(SplitMergeArgs a) {
  const int m = blockIdx.x;
  const int row0 = blockIdx.y * 32;
  const int nrows = min(32, a.rows - row0);
  if (m >= a.M || nrows <= 0) return;
  const int first = a.indptr[m], count = a.indptr[m + 1] - a.indptr[m];
  merge_rows(a.part_o + (size_t)row0 * a.D, a.part_lse + row0, (size_t)a.rows * a.D, a.rows, first,
             count < 0 ? 0 : count, nrows, a.D, a.o + ((size_t)m * a.rows + row0) * a.D,
             a.lse + (size_t)m * a.rows + row0);
}

}  // namespace

cudaError_t launch_plan_merge(const mla_geom* g, const mla_batch* b, const WsLayout& L, __nv_bfloat16* o_lat,
                              float* lse, void* ws, cudaStream_t st) {
  PlanMergeArgs a;
  a.T = b->T; a.H = g->H; a.o_lat = o_lat; a.lse = lse; a.L = L;
  int grid = L.cap_groups;
  if (grid <= 0) return cudaSuccess;
  if (grid > 4096) grid = 4096;
  plan_merge_kernel<<<grid, kMergeThreads, 0, st>>>(a, reinterpret_cast<const char*>(ws));
  return cudaGetLastError();
}

cudaError_t launch_split_merge(const float* part_o, const float* part_lse, const int32_t* indptr, int M, int rows,
                               int D, __nv_bfloat16* o, float* lse, cudaStream_t st) {
  if (M <= 0 || rows <= 0) return cudaSuccess;
  SplitMergeArgs a{part_o, part_lse, indptr, M, rows, D, o, lse};
  dim3 grid(M, (rows + 31) / 32);
  split_merge_kernel<<<grid, kMergeThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
