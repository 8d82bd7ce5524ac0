// Exact log-sum-exp merge of the split plan's partial states, run by the decode
// kernel's own CTAs after all of them have written their partials.
//
// "M5.8" 0x0C: for partial states (m_r, l_r, o_r) the merged state is
// m = max m_r, l = sum e^{m_r - m} l_r, o = sum e^{m_r - m} o_r, O = o / l.
// With partials stored normalised (o_r / l_r) together with
// lse_r = m_r + ln l_r (the "mlxcel" Stage-2 contract, natural-log units here),
// the weight of partial r is w_r = e^{lse_r - max lse}, and
// O = sum w_r (o_r / l_r) / sum w_r, lse = max lse + ln sum w_r.
//
// Work: the rows of all merge records, record-major; CTA k of n takes a
// contiguous share, so it reads each record it touches once.  There is no
// grid-wide barrier: every softmax warp that stored partial rows of a split
// group counts them into the group's record (16 counts per segment: eight
// warps in each CTA of the pair), and a CTA merges a record once its count is
// complete, so CTAs that finish early merge while others still decode.  The
// CTA that merges a record's last rows zeroes its counters for the next decode.  The CTA's
// threads form kGroups groups of 128, each thread owning four columns of a
// row.  A record of at most kPartBatch partials is merged by one thread per
// column chunk, several rows per thread for small counts (every thread keeps
// kPartBatch loads in flight); a larger record is split over all kGroups
// groups, which fold every kGroups-th partial and combine their states through
// shared memory in group order.  An empty record (a group with no visible row)
// gets o = 0, lse = -inf.
#pragma once

#include <math.h>

#include "mla_internal.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace merge {

constexpr int kPartBatch = 16;  // partial loads a thread keeps in flight

struct Out {
  int T, H;
  __nv_bfloat16* o_lat;
  float* lse;
};

// Running merge state of one thread: m = max LSE seen, l = sum of e^{lse - m},
// acc = sum of e^{lse - m} o (four columns).  Folding in a batch whose maximum
// raises m rescales what is already there by e^{m_old - m_new}.
struct State {
  float m, l, a0, a1, a2, a3;
};

// Fold partials r = r0, r0 + step, ... (< count) of one row into st, in batches
// whose loads are all issued before any is used.  A partial of LSE -inf has
// weight 0 and is skipped (select), whatever its slot holds.
__device__ __forceinline__ void fold_partials(State& st, const float* po, const float* pl, size_t o_pitch,
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
__device__ __forceinline__ void store_row(const Out& a, size_t grow, int c, const State& st) {
  const float inv = st.l > 0.f ? 1.f / st.l : 0.f;
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(st.a0 * inv, st.a1 * inv);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(st.a2 * inv, st.a3 * inv);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&h0);
  u.y = *reinterpret_cast<const uint32_t*>(&h1);
  *reinterpret_cast<uint2*>(a.o_lat + grow * kDLat + c) = u;
  if (c == 0) a.lse[grow] = st.l > 0.f ? st.m + logf(st.l) : -INFINITY;
}

// A record of at most kPartBatch partials, padded to CP (2, 4, 8 or 16): each
// thread merges kPartBatch / CP rows at once (rows rl = grp + G j of the nrows
// starting at row0), so that every thread has kPartBatch loads in flight
// whatever the count.
template <int G, int CP>
__device__ __forceinline__ void merge_rows(const Out& a, const float* part_o, const float* part_lse, int first,
                                           int count, int b, int rb, int R, int row0, int nrows, int grp, int c) {
  constexpr int RG = kPartBatch / CP;
  float x[kPartBatch];
  float4 v[kPartBatch];
#pragma unroll
  for (int k = 0; k < kPartBatch; ++k) {
    const int j = k / CP, r = k % CP;
    const int rl = grp + G * j;
    const bool ok = rl < nrows && rb * kRowsPerBlock + row0 + rl < R && r < count;
    const size_t pr = (size_t)(first + r) * kRowsPerBlock + row0 + rl;
    x[k] = ok ? __ldcg(part_lse + pr) : -INFINITY;
    v[k] = ok ? __ldcg(reinterpret_cast<const float4*>(part_o + pr * kDLat + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int j = 0; j < RG; ++j) {
    const int rl = grp + G * j;
    const int fr = rb * kRowsPerBlock + row0 + rl;
    if (rl >= nrows || fr >= R) continue;
    float mx = -INFINITY;
#pragma unroll
    for (int r = 0; r < CP; ++r) mx = fmaxf(mx, x[j * CP + r]);
    State st{mx, 0.f, 0.f, 0.f, 0.f, 0.f};
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

constexpr int kCountsPerSegment = 16;   // softmax warps of a CTA pair that store a segment's partial rows

// Bounded wait (thread 0) until record i's partial rows are all stored, then the
// whole CTA proceeds.  Returns false (after recording MLA_ERR_TIMEOUT) if the
// count never completes.
__device__ __forceinline__ bool wait_record(int* hdr, int* stored, int need, volatile int* flag) {
  if (threadIdx.x == 0) {
    bool ok = true;
    const long long t0 = clock64();
    while (true) {
      int v;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(stored) : "memory");
      if (v >= need) break;
      if (clock64() - t0 > MLA_PIPELINE_WAIT_LIMIT) { ok = false; record_error(hdr, MLA_ERR_TIMEOUT, 60); break; }
      __nanosleep(64);
    }
    *flag = ok ? 1 : 0;
  }
  __syncthreads();
  return *flag != 0;
}

// Rows [r0, r1) of record i merged by this CTA: add them to the record's merged
// count; the CTA completing the record zeroes both counters.
__device__ __forceinline__ void finish_rows(int* msync, int i, int n) {
  __syncthreads();   // this CTA's stores of those rows are issued
  if (threadIdx.x == 0 && n > 0) {
    if (atomicAdd(msync + 2 * i + 1, n) + n == kRowsPerBlock) {
      atomicExch(msync + 2 * i, 0);
      atomicExch(msync + 2 * i + 1, 0);
    }
  }
}

// CTA `cta` of `nctas` merges its share of the plan's merge records with its
// first 128 * G threads (threadIdx.x < 128 G; every one of them must call).
// s_st: shared memory of G * 6 * 128 floats; flag: one shared int.
template <int G>
__device__ __forceinline__ void merge_plan_share(const Out& a, char* ws, const WsLayout& L, int num_merge,
                                                 int cta, int nctas, float* s_st, volatile int* flag) {
  int* hdr = reinterpret_cast<int*>(ws);
  int* msync = reinterpret_cast<int*>(ws + L.off_merge_sync);
  const int* mrg = reinterpret_cast<const int*>(ws + L.off_merge);
  const float* part_lse = reinterpret_cast<const float*>(ws + L.off_part_lse);
  const float* part_o = reinterpret_cast<const float*>(ws + L.off_part_o);
  const int R = a.T * a.H;
  const long long V = (long long)num_merge * kRowsPerBlock;
  const long long per = (V + nctas - 1) / nctas;
  const long long v_end = min(V, (cta + 1) * per);
  const int grp = threadIdx.x / (kDLat / 4);
  const int t = threadIdx.x % (kDLat / 4);
  const int c = 4 * t;
  int cur = -1, b = 0, rb = 0, first = 0, count = 0, done = 0;
  for (long long v = cta * per; v < v_end;) {
    const int i = (int)(v / kRowsPerBlock);
    const int row0 = (int)(v % kRowsPerBlock);
    if (i != cur) {
      if (cur >= 0) finish_rows(msync, cur, done);
      cur = i;
      done = 0;
      b = __ldcg(mrg + i * kMergeWords + 0);
      rb = __ldcg(mrg + i * kMergeWords + 1);
      first = __ldcg(mrg + i * kMergeWords + 2);
      count = __ldcg(mrg + i * kMergeWords + 3);
      if (!wait_record(hdr, msync + 2 * i, kCountsPerSegment * count, flag)) return;
    }
    if (count <= kPartBatch) {
      const int cp = count <= 2 ? 2 : count <= 4 ? 4 : count <= 8 ? 8 : 16;   // an empty group (count 0) takes 2
      const int nrows = (int)min((long long)min(G * (kPartBatch / cp), kRowsPerBlock - row0), v_end - v);
      if (cp == 2) merge_rows<G, 2>(a, part_o, part_lse, first, count, b, rb, R, row0, nrows, grp, c);
      else if (cp == 4) merge_rows<G, 4>(a, part_o, part_lse, first, count, b, rb, R, row0, nrows, grp, c);
      else if (cp == 8) merge_rows<G, 8>(a, part_o, part_lse, first, count, b, rb, R, row0, nrows, grp, c);
      else merge_rows<G, 16>(a, part_o, part_lse, first, count, b, rb, R, row0, nrows, grp, c);
      v += nrows;
      done += nrows;
      continue;
    }
    // One row at a time, its partials split over the G groups.
    const int row = row0;
    const int fr = rb * kRowsPerBlock + row;
    const bool valid = fr < R;
    State st{-INFINITY, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (valid)
      fold_partials(st, part_o + ((size_t)first * kRowsPerBlock + row) * kDLat + c,
                    part_lse + (size_t)first * kRowsPerBlock + row, (size_t)kRowsPerBlock * kDLat, kRowsPerBlock, grp,
                    G, count);
    float* my = s_st + (grp * 6) * 128 + t;
    my[0] = st.m; my[128] = st.l; my[256] = st.a0; my[384] = st.a1; my[512] = st.a2; my[640] = st.a3;
    __syncthreads();
    if (grp == 0 && valid) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < G; ++j) mx = fmaxf(mx, s_st[(j * 6) * 128 + t]);
      State m{mx, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (mx != -INFINITY) {
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float* sj = s_st + (j * 6) * 128 + t;
          const float f = sj[0] == -INFINITY ? 0.f : __expf(sj[0] - mx);
          m.l = fmaf(f, sj[128], m.l);
          m.a0 = fmaf(f, sj[256], m.a0);
          m.a1 = fmaf(f, sj[384], m.a1);
          m.a2 = fmaf(f, sj[512], m.a2);
          m.a3 = fmaf(f, sj[640], m.a3);
        }
      }
      store_row(a, (size_t)b * R + fr, c, m);
    }
    __syncthreads();
    v += 1;
    done += 1;
  }
  if (cur >= 0) finish_rows(msync, cur, done);
}

}  // namespace merge
}  // namespace mla
