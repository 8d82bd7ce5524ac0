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

struct PlanMergeArgs {
  int T, H;
  __nv_bfloat16* o_lat;
  float* lse;
  WsLayout L;
};

constexpr int kPlanMergeThreads = 1024;            // eight groups of 128 threads, one float4 column chunk each
constexpr int kGroups = kPlanMergeThreads / (kDLat / 4);
constexpr int kPartBatch = 8;                      // partial loads a thread keeps in flight

// Running merge state of one thread: m = max LSE seen, l = sum of e^{lse - m},
// acc = sum of e^{lse - m} o (four columns).  Folding in a batch whose maximum
// raises m rescales what is already there by e^{m_old - m_new}.
struct MergeState {
  float m, l, a0, a1, a2, a3;
};

// Fold partials r = r0, r0 + step, ... (< count) of one row into st, in batches
// whose loads are all issued before any is used.  A partial of LSE -inf has
// weight 0 and is skipped (select), whatever its slot holds.
__device__ __forceinline__ void fold_partials(MergeState& st, const float* po, const float* pl, size_t o_pitch,
                                              size_t l_pitch, int r0, int step, int count) {
  for (int rb = r0; rb < count; rb += kPartBatch * step) {
    float x[kPartBatch];
    float4 v[kPartBatch];
#pragma unroll
    for (int k = 0; k < kPartBatch; ++k) {
      const int r = rb + k * step;
      const int rr = r < count ? r : r0;
      x[k] = r < count ? __ldcg(pl + (size_t)rr * l_pitch) : -INFINITY;
      v[k] = __ldcg(reinterpret_cast<const float4*>(po + (size_t)rr * o_pitch));
    }
    float mb = -INFINITY;
#pragma unroll
    for (int k = 0; k < kPartBatch; ++k) mb = fmaxf(mb, x[k]);
    const float mn = fmaxf(st.m, mb);
    if (mn == -INFINITY) continue;                 // nothing with weight yet
    const float sc = st.m == -INFINITY ? 0.f : __expf(st.m - mn);
    st.l *= sc; st.a0 *= sc; st.a1 *= sc; st.a2 *= sc; st.a3 *= sc;
#pragma unroll
    for (int k = 0; k < kPartBatch; ++k) {
      const float w = x[k] == -INFINITY ? 0.f : __expf(x[k] - mn);
      const bool use = w != 0.f;
      st.l += w;
      st.a0 = use ? fmaf(w, v[k].x, st.a0) : st.a0;
      st.a1 = use ? fmaf(w, v[k].y, st.a1) : st.a1;
      st.a2 = use ? fmaf(w, v[k].z, st.a2) : st.a2;
      st.a3 = use ? fmaf(w, v[k].w, st.a3) : st.a3;
    }
    st.m = mn;
  }
}

// Store four merged columns of one row (and, from the thread of column 0, its LSE).
__device__ __forceinline__ void store_row(const PlanMergeArgs& a, size_t grow, int c, const MergeState& st) {
  const float inv = st.l > 0.f ? 1.f / st.l : 0.f;
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(st.a0 * inv, st.a1 * inv);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(st.a2 * inv, st.a3 * inv);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&h0);
  u.y = *reinterpret_cast<const uint32_t*>(&h1);
  *reinterpret_cast<uint2*>(a.o_lat + grow * kDLat + c) = u;
  if (c == 0) a.lse[grow] = st.l > 0.f ? st.m + logf(st.l) : -INFINITY;
}

// A record of at most kPartBatch partials, padded to CP (2, 4 or 8): each
// thread merges kPartBatch / CP rows at once (rows rl = grp + kGroups j of the
// nrows starting at row0), so that every thread has kPartBatch loads in flight
// whatever the count.
template <int CP>
__device__ __forceinline__ void merge_rows(const PlanMergeArgs& a, const float* part_o, const float* part_lse,
                                           int first, int count, int b, int rb, int R, int row0, int nrows, int grp,
                                           int c) {
  constexpr int RG = kPartBatch / CP;
  float x[kPartBatch];
  float4 v[kPartBatch];
#pragma unroll
  for (int k = 0; k < kPartBatch; ++k) {
    const int j = k / CP, r = k % CP;
    const int rl = grp + kGroups * j;
    const bool ok = rl < nrows && rb * kRowsPerBlock + row0 + rl < R && r < count;
    const size_t pr = (size_t)(first + r) * kRowsPerBlock + row0 + rl;
    x[k] = ok ? __ldcg(part_lse + pr) : -INFINITY;
    v[k] = ok ? __ldcg(reinterpret_cast<const float4*>(part_o + pr * kDLat + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int j = 0; j < RG; ++j) {
    const int rl = grp + kGroups * j;
    const int fr = rb * kRowsPerBlock + row0 + rl;
    if (rl >= nrows || fr >= R) continue;
    float mx = -INFINITY;
#pragma unroll
    for (int r = 0; r < CP; ++r) mx = fmaxf(mx, x[j * CP + r]);
    MergeState st{mx, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (mx != -INFINITY) {
#pragma unroll
      for (int r = 0; r < CP; ++r) {
        const float xr = x[j * CP + r];
        const float w = xr == -INFINITY ? 0.f : __expf(xr - mx);
        const bool use = w != 0.f;
        st.l += w;
        st.a0 = use ? fmaf(w, v[j * CP + r].x, st.a0) : st.a0;
        st.a1 = use ? fmaf(w, v[j * CP + r].y, st.a1) : st.a1;
        st.a2 = use ? fmaf(w, v[j * CP + r].z, st.a2) : st.a2;
        st.a3 = use ? fmaf(w, v[j * CP + r].w, st.a3) : st.a3;
      }
    }
    store_row(a, (size_t)b * R + fr, c, st);
  }
}

// Merge records of the plan (groups that were split, or are empty).  The work
// is the rows of all records (record-major); CTA k takes a contiguous share, so
// it reads each record it touches once.  A record of `count` partials is
// merged by one thread per column chunk when count <= 8 (merge_rows: several
// rows per thread for small counts), else S = 2, 4 or 8 ways (count <= 16, <= 32,
// more): the CTA's eight groups of 128 threads take 8/S rows at a time, each row
// split over S groups that fold every S-th partial and then combine their
// states through shared memory in group order.  Each thread owns four columns.
__global__ void __launch_bounds__(kPlanMergeThreads) plan_merge_kernel(PlanMergeArgs a, const char* ws) {
  __shared__ float s_st[kGroups][6][kDLat / 4];
  pdl_wait();
  pdl_trigger();
  const int* hdr = reinterpret_cast<const int*>(ws);
  const int* mrg = reinterpret_cast<const int*>(ws + a.L.off_merge);
  const float* part_lse = reinterpret_cast<const float*>(ws + a.L.off_part_lse);
  const float* part_o = reinterpret_cast<const float*>(ws + a.L.off_part_o);
  const int R = a.T * a.H;
  const long long V = (long long)hdr[MLA_HDR_NUM_MERGE] * kRowsPerBlock;
  const long long per = (V + gridDim.x - 1) / gridDim.x;
  const long long v_end = min(V, (blockIdx.x + 1) * per);
  const int grp = threadIdx.x / (kDLat / 4);
  const int c = 4 * (threadIdx.x % (kDLat / 4));
  int cur = -1, b = 0, rb = 0, first = 0, count = 0, S = 1;
  for (long long v = blockIdx.x * per; v < v_end;) {
    const int i = (int)(v / kRowsPerBlock);
    const int row0 = (int)(v % kRowsPerBlock);
    if (i != cur) {
      cur = i;
      b = mrg[i * kMergeWords + 0];
      rb = mrg[i * kMergeWords + 1];
      first = mrg[i * kMergeWords + 2];
      count = mrg[i * kMergeWords + 3];
      S = count <= kPartBatch ? 1 : count <= 2 * kPartBatch ? 2 : count <= 4 * kPartBatch ? 4 : 8;
    }
    if (S == 1) {
      const int cp = count <= 2 ? 2 : count <= 4 ? 4 : 8;   // an empty group (count 0) takes 2
      const int nrows = (int)min((long long)min(kGroups * (kPartBatch / cp), kRowsPerBlock - row0), v_end - v);
      if (cp == 2) merge_rows<2>(a, part_o, part_lse, first, count, b, rb, R, row0, nrows, grp, c);
      else if (cp == 4) merge_rows<4>(a, part_o, part_lse, first, count, b, rb, R, row0, nrows, grp, c);
      else merge_rows<8>(a, part_o, part_lse, first, count, b, rb, R, row0, nrows, grp, c);
      v += nrows;
      continue;
    }
    const int nrows = (int)min((long long)min(kGroups / S, kRowsPerBlock - row0), v_end - v);
    const int rl = grp / S, s = grp % S;
    const int row = row0 + rl;
    const int fr = rb * kRowsPerBlock + row;
    const bool valid = rl < nrows && fr < R;
    MergeState st{-INFINITY, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (valid)
      fold_partials(st, part_o + ((size_t)first * kRowsPerBlock + row) * kDLat + c,
                    part_lse + (size_t)first * kRowsPerBlock + row, (size_t)kRowsPerBlock * kDLat, kRowsPerBlock, s,
                    S, count);
    {
      const int t = threadIdx.x % (kDLat / 4);
      s_st[grp][0][t] = st.m; s_st[grp][1][t] = st.l;
      s_st[grp][2][t] = st.a0; s_st[grp][3][t] = st.a1; s_st[grp][4][t] = st.a2; s_st[grp][5][t] = st.a3;
      __syncthreads();
      if (s == 0) {
        float mx = -INFINITY;
        for (int j = 0; j < S; ++j) mx = fmaxf(mx, s_st[grp + j][0][t]);
        MergeState m{mx, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (mx != -INFINITY) {
          for (int j = 0; j < S; ++j) {
            const float mj = s_st[grp + j][0][t];
            const float f = mj == -INFINITY ? 0.f : __expf(mj - mx);
            m.l = fmaf(f, s_st[grp + j][1][t], m.l);
            m.a0 = fmaf(f, s_st[grp + j][2][t], m.a0);
            m.a1 = fmaf(f, s_st[grp + j][3][t], m.a1);
            m.a2 = fmaf(f, s_st[grp + j][4][t], m.a2);
            m.a3 = fmaf(f, s_st[grp + j][5][t], m.a3);
          }
        }
        st = m;
      }
      __syncthreads();
    }
    if (valid && s == 0) store_row(a, (size_t)b * R + fr, c, st);
    v += nrows;
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

cudaError_t launch_plan_merge(const mla_geom* g, const mla_batch* b, const WsLayout& L, __nv_bfloat16* o_lat,
                              float* lse, void* ws, cudaStream_t st) {
  PlanMergeArgs a;
  a.T = b->T; a.H = g->H; a.o_lat = o_lat; a.lse = lse; a.L = L;
  if (L.cap_groups <= 0) return cudaSuccess;
  // One 1024-thread CTA per SM; never more CTAs than the possible rows.
  const long long cap_rows = (long long)L.cap_groups * kRowsPerBlock;
  const int sms = mla_device_sm_count();
  long long nctas = sms > 0 ? sms : 148;
  if (nctas > cap_rows) nctas = cap_rows;
  const dim3 grid((unsigned)nctas);
  return launch_pdl(plan_merge_kernel, grid, dim3(kPlanMergeThreads), 0, st, a, reinterpret_cast<const char*>(ws));
}

cudaError_t launch_split_merge(const float* part_o, const float* part_lse, const int32_t* indptr, int M, int rows,
                               int D, __nv_bfloat16* o, float* lse, cudaStream_t st) {
  if (M <= 0 || rows <= 0) return cudaSuccess;
  SplitMergeArgs a{part_o, part_lse, indptr, M, rows, D, o, lse};
  const long long blocks = ((long long)rows * (D / 4) + kMergeThreads - 1) / kMergeThreads;
  const dim3 grid(M, (unsigned)(blocks < 65535 ? blocks : 65535));
  return launch_pdl(split_merge_kernel, grid, dim3(kMergeThreads), 0, st, a);
}

}  // namespace mla
