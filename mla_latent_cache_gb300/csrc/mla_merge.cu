// Exact log-sum-exp merge of split-KV partial states: the public merge entry
// point (the split plan's own merge runs inside the decode kernel, with the
// helpers of mla_plan_merge.cuh).
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
constexpr int kBatch = 8;  // partial loads kept in flight per thread

// Merge four adjacent columns of one row from `count` partials: partial r of
// those columns starts at part_o[r * o_pitch], its LSE is part_lse[r * lse_pitch].
// Every thread of a row recomputes the (few) weights from the LSEs (broadcast
// loads); the loads of kBatch partials are issued before any is used so that
// the merge is bound by bandwidth, not by one load latency per partial.  The
// sums run over r in increasing order, and a partial of weight 0 is skipped
// (select, so that whatever its slot holds cannot reach the result).
__device__ __forceinline__ void merge4(const float* part_o, const float* part_lse, size_t o_pitch, size_t lse_pitch,
                                       int count, __nv_bfloat16* o_out, float* lse_out) {
  float m = -INFINITY;
  for (int r = 0; r < count; ++r) m = fmaxf(m, part_lse[(size_t)r * lse_pitch]);
  const float m_use = (m == -INFINITY) ? 0.f : m;
  float l = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  for (int r0 = 0; r0 < count; r0 += kBatch) {
    float w[kBatch];
    float4 v[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int r = r0 + k < count ? r0 + k : count - 1;
      const float x = part_lse[(size_t)r * lse_pitch];
      w[k] = (r0 + k < count && x != -INFINITY) ? __expf(x - m_use) : 0.f;
      v[k] = *reinterpret_cast<const float4*>(part_o + (size_t)r * o_pitch);
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const bool use = w[k] != 0.f;
      l += w[k];
      a0 = use ? fmaf(w[k], v[k].x, a0) : a0;
      a1 = use ? fmaf(w[k], v[k].y, a1) : a1;
      a2 = use ? fmaf(w[k], v[k].z, a2) : a2;
      a3 = use ? fmaf(w[k], v[k].w, a3) : a3;
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(a0 * inv, a1 * inv);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(a2 * inv, a3 * inv);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&h0);
  u.y = *reinterpret_cast<const uint32_t*>(&h1);
  *reinterpret_cast<uint2*>(o_out) = u;
  if (lse_out) *lse_out = l > 0.f ? m_use + logf(l) : -INFINITY;
}

struct SplitMergeArgs {
  const float* part_o;
  const float* part_lse;
  const int32_t* indptr;
  int M, rows, D;
  __nv_bfloat16* o;
  float* lse;
};

// Public contract: CTAs (m, *) merge output m; work item k (stepping by the
// y-grid) owns columns 4 (k % (D/4)) .. +3 of row k / (D/4).
__global__ void __launch_bounds__(kMergeThreads) split_merge_kernel(SplitMergeArgs a) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x;
  if (m >= a.M) return;
  const int chunks = a.D / 4;
  const long long items = (long long)a.rows * chunks;
  const int first = a.indptr[m], count = a.indptr[m + 1] - a.indptr[m];
  for (long long k = (long long)blockIdx.y * blockDim.x + threadIdx.x; k < items;
       k += (long long)gridDim.y * blockDim.x) {
    const int row = (int)(k / chunks), c = 4 * (int)(k % chunks);
    merge4(a.part_o + ((size_t)first * a.rows + row) * a.D + c, a.part_lse + (size_t)first * a.rows + row,
           (size_t)a.rows * a.D, a.rows, count < 0 ? 0 : count, a.o + ((size_t)m * a.rows + row) * a.D + c,
           c == 0 ? a.lse + (size_t)m * a.rows + row : nullptr);
  }
}

}  // namespace

cudaError_t launch_split_merge(const float* part_o, const float* part_lse, const int32_t* indptr, int M, int rows,
                               int D, __nv_bfloat16* o, float* lse, cudaStream_t st) {
  if (M <= 0 || rows <= 0) return cudaSuccess;
  SplitMergeArgs a{part_o, part_lse, indptr, M, rows, D, o, lse};
  const long long blocks = ((long long)rows * (D / 4) + kMergeThreads - 1) / kMergeThreads;
  const dim3 grid(M, (unsigned)(blocks < 65535 ? blocks : 65535));
  return launch_pdl(split_merge_kernel, grid, dim3(kMergeThreads), 0, st, a);
}

}  // namespace mla
