// Device split planner: builds the work plan (segments, ranges, merge list) in
// the workspace from the device-resident sequence lengths, with no host sync.
// The rule is stated in include/mla.h next to the plan layout.
#include <climits>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kPlanThreads = 1024;

constexpr int kSmemGroups = 4096;   // groups whose segment bases the planner keeps in shared memory

// Block-wide exclusive scans of three ints per thread at once; tot[] gets the
// block sums.  sh holds 3 x 32 ints.
__device__ void block_excl_scan3(int (&v)[3], int (&tot)[3], int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int x[3] = {v[0], v[1], v[2]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int y = __shfl_up_sync(0xffffffffu, x[j], o);
      if (lane >= o) x[j] += y;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int j = 0; j < 3; ++j) sh[32 * j + warp] = x[j];
  }
  __syncthreads();
  if (warp < 3) {
    int w = lane < nwarps ? sh[32 * warp + lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh[32 * warp + lane] = w;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int pre = warp ? sh[32 * j + warp - 1] : 0;
    tot[j] = sh[32 * j + nwarps - 1];
    v[j] = pre + x[j] - v[j];
  }
  __syncthreads();
}

// Block-wide (sum, max) of two ints and (wrapping sum, min) of an unsigned and
// an int: warp shuffles, then one value per warp through shared memory.
__device__ void block_reduce(unsigned& usum, int& imin, int& isum, int& imax, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    usum += __shfl_xor_sync(0xffffffffu, usum, o);
    imin = min(imin, __shfl_xor_sync(0xffffffffu, imin, o));
    isum += __shfl_xor_sync(0xffffffffu, isum, o);
    imax = max(imax, __shfl_xor_sync(0xffffffffu, imax, o));
  }
  if (lane == 0) {
    sh[warp] = (int)usum; sh[32 + warp] = imin; sh[64 + warp] = isum; sh[96 + warp] = imax;
  }
  __syncthreads();
  if (warp == 0) {
    usum = lane < nwarps ? (unsigned)sh[lane] : 0u;
    imin = lane < nwarps ? sh[32 + lane] : INT_MAX;
    isum = lane < nwarps ? sh[64 + lane] : 0;
    imax = lane < nwarps ? sh[96 + lane] : INT_MIN;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      usum += __shfl_xor_sync(0xffffffffu, usum, o);
      imin = min(imin, __shfl_xor_sync(0xffffffffu, imin, o));
      isum += __shfl_xor_sync(0xffffffffu, isum, o);
      imax = max(imax, __shfl_xor_sync(0xffffffffu, imax, o));
    }
    // (the shuffles follow every lane's reads, so lane 0 may overwrite the slots)
    if (lane == 0) {
      sh[0] = (int)usum; sh[1] = imin; sh[2] = isum; sh[3] = imax;
    }
  }
  __syncthreads();
  usum = (unsigned)sh[0]; imin = sh[1]; isum = sh[2]; imax = sh[3];
  __syncthreads();
}

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  x ^= x >> 16; x *= 0x7feb352dU; x ^= x >> 15; x *= 0x846ca68bU; x ^= x >> 16;
  return x;
}

struct PlanArgs {
  const int32_t* seq_lens;   // length of sequence b is seq_lens[b / seq_div]
  int seq_div;               // 1; the sparse decode's S_q (one length per sequence, shared by its tokens)
  int B, T, H, causal, G, N, max_pages;
  int max_rows;              // longest allowed length: max_pages * 64, or the sparse decode's topk
  int RB, num_groups;
  WsLayout L;
};

// Fixed cost of starting a group's work in a range, in pages (query staging and
// an output write per segment: measured ~8 us per segment change on the ragged
// V3 batch against ~0.8 us per page): the balanced ranges leave that many line
// positions between consecutive non-empty groups.
constexpr int kSegmentCostPages = 8;

// Segment s of a group with n pages whose first page sits at line position u
// (mode 1) and whose first segment is sb, in the given mode; writes the record
// and the range pointer of every range whose first segment it is (in mode 1
// also of the ranges inside the gap before it, which hold no segment).  ne:
// non-empty groups before this one.
__device__ __forceinline__ void write_segment(int* seg, int* rptr, int mode, int q, int b, int rb, int n, int u,
                                              int k, int sb, int pb, int mi, int s, int ne) {
  int p0, p1, r;
  if (mode == 2) {
    p0 = (int)(((long long)s * n) / k);
    p1 = (int)(((long long)(s + 1) * n) / k);
    r = sb + s;
  } else if (mode == 0) {
    p0 = 0; p1 = n; r = sb;
  } else {
    r = u / q + s;
    const int gs = max(u, r * q), ge = min(u + n, (r + 1) * q);
    p0 = gs - u; p1 = ge - u;
  }
  int* rec = seg + (size_t)(sb + s) * kSegWords;
  rec[0] = b; rec[1] = rb; rec[2] = p0; rec[3] = p1; rec[4] = r;
  rec[5] = (k > 1) ? pb + s : -1; rec[6] = (k > 1) ? mi : -1; rec[7] = 0;
  if (mode != 1 || s > 0) {
    rptr[r] = sb + s;     // a cut: the segment starts its range
  } else {
    // the previous non-empty group's last page sits just before this group's gap
    const int r_prev = ne > 0 ? (u - kSegmentCostPages - 1) / q : -1;
    for (int rr = r_prev + 1; rr <= r; ++rr) rptr[rr] = sb;
  }
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a, char* ws) {
  int* hdr = reinterpret_cast<int*>(ws);
  int* grp = reinterpret_cast<int*>(ws + a.L.off_groups);
  int* seg = reinterpret_cast<int*>(ws + a.L.off_segments);
  int* rptr = reinterpret_cast<int*>(ws + a.L.off_range_ptr);
  int* mrg = reinterpret_cast<int*>(ws + a.L.off_merge);
  int* msync = reinterpret_cast<int*>(ws + a.L.off_merge_sync);
  __shared__ int sh[128];
  __shared__ int s_sb[kSmemGroups];
  __shared__ int s_q, s_mode, s_U;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();

  // Sequence-length stamp (a wrapping sum, so order-free) and validation (the
  // smallest offending sequence is reported).
  unsigned hsum = 0;
  int errb = INT_MAX;
  for (int b = tid; b < a.B; b += blockDim.x) {
    const int S = a.seq_lens[b / a.seq_div];
    hsum += mix32((uint32_t)S * 0x9E3779B1u + mix32((uint32_t)b + 0x632BE5ABu));
    if (S < 0 || S > a.max_rows || (S > 0 && S < a.T)) errb = min(errb, b);
  }

  // Pass A: pages per group and their exclusive prefix.
  int carry = 0, nonempty = 0, maxn = 0, nonempty_carry = 0;
  const int R = a.T * a.H;
  for (int base = 0; base < a.num_groups; base += blockDim.x) {
    const int g = base + tid;
    int n = 0;
    if (g < a.num_groups) {
      const int b = g / a.RB, rb = g % a.RB;
      int S = a.seq_lens[b / a.seq_div];
      S = S < 0 ? 0 : (S > a.max_rows ? a.max_rows : S);
      const int r_last = min(R, (rb + 1) * kRowsPerBlock) - 1;
      const int vis = visible_limit(S, a.T, r_last / a.H, a.causal);
      n = (vis + kPage - 1) / kPage;
    }
    int v[3] = {n, n > 0 ? 1 : 0, 0}, tot[3];
    block_excl_scan3(v, tot, sh);
    if (g < a.num_groups) {
      const int ne = nonempty_carry + v[1];     // non-empty groups before g
      grp[g * kGroupWords + 0] = n;
      grp[g * kGroupWords + 1] = carry + v[0];
      grp[g * kGroupWords + 6] = carry + v[0] + kSegmentCostPages * ne;   // line position of its first page
      grp[g * kGroupWords + 7] = ne;
      nonempty += n > 0;
      maxn = max(maxn, n);
    }
    carry += tot[0];
    nonempty_carry += tot[1];
  }
  block_reduce(hsum, errb, nonempty, maxn, sh);
  const int W = carry;
  if (tid == 0) {
    int q = (W + a.G - 1) / a.G;
    q = q < kMinSplitPages ? kMinSplitPages : q;
    s_q = q;
    if (a.N > 0) s_mode = 2;
    else if (nonempty <= a.G && maxn <= (5 * q + 3) / 4) s_mode = 0;
    else s_mode = 1;
    if (s_mode == 1) {
      // balanced ranges over the line of pages and gaps
      const int U = W + kSegmentCostPages * (nonempty - 1);
      const int qw = (U + a.G - 1) / a.G;
      s_q = qw < kMinSplitPages ? kMinSplitPages : qw;
      s_U = U;
    }
  }
  __syncthreads();
  const int q = s_q, mode = s_mode;

  // Pass B: segments per group, segment/slot/merge bases; merge records.
  int cseg = 0, cpart = 0, cmrg = 0;
  for (int base = 0; base < a.num_groups; base += blockDim.x) {
    const int g = base + tid;
    int k = 0, n = 0;
    if (g < a.num_groups) {
      n = grp[g * kGroupWords + 0];
      const int u = grp[g * kGroupWords + 6];
      if (n > 0) {
        if (mode == 2) k = min(n, a.N);
        else if (mode == 0) k = 1;
        else k = (u + n - 1) / q - u / q + 1;
      }
    }
    const int part = k > 1 ? k : 0;
    const int mflag = (g < a.num_groups && k != 1) ? 1 : 0;
    int v[3] = {k, part, mflag}, tot[3];
    block_excl_scan3(v, tot, sh);
    if (g < a.num_groups) {
      const int sb = cseg + v[0];
      const int pb = part ? cpart + v[1] : -1;
      grp[g * kGroupWords + 2] = k;
      grp[g * kGroupWords + 3] = sb;
      grp[g * kGroupWords + 4] = pb;
      grp[g * kGroupWords + 5] = mflag ? cmrg + v[2] : -1;
      if (g < kSmemGroups) s_sb[g] = sb;
      msync[2 * g] = 0;       // merge record g's stored-partial count and merged-row count
      msync[2 * g + 1] = 0;
      if (mflag) {
        int* m = mrg + (size_t)(cmrg + v[2]) * kMergeWords;
        m[0] = g / a.RB; m[1] = g % a.RB; m[2] = (k > 1) ? pb : 0; m[3] = (k > 1) ? k : 0;
      }
    }
    cseg += tot[0]; cpart += tot[1]; cmrg += tot[2];
  }
  __syncthreads();
  const int total_seg = cseg;
  const int num_ranges = (mode == 1) ? (s_U + q - 1) / q : total_seg;

  // Pass C: segment records and range pointers, one segment per thread (its
  // group found by binary search over the segment bases), or one group per
  // thread when there are more groups than shared memory holds.
  if (a.num_groups <= kSmemGroups) {
    for (int i = tid; i < total_seg; i += blockDim.x) {
      int lo = 0, hi = a.num_groups;        // last group whose first segment is <= i
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_sb[mid] <= i) lo = mid; else hi = mid;
      }
      const int g = lo;
      const int* gr = grp + g * kGroupWords;
      write_segment(seg, rptr, mode, q, g / a.RB, g % a.RB, gr[0], gr[6], gr[2], gr[3], gr[4], gr[5], i - gr[3], gr[7]);
    }
  } else {
    for (int g = tid; g < a.num_groups; g += blockDim.x) {
      const int* gr = grp + g * kGroupWords;
      const int k = gr[2];
      for (int s = 0; s < k; ++s)
        write_segment(seg, rptr, mode, q, g / a.RB, g % a.RB, gr[0], gr[6], k, gr[3], gr[4], gr[5], s, gr[7]);
    }
  }
  // Range pointers past the last range repeat the segment count, up to the
  // table's capacity: a decode CTA pair then reads its ranges' pointers
  // directly, without first reading the range count.
  for (int r = num_ranges + 1 + tid; r <= a.L.cap_ranges; r += blockDim.x) rptr[r] = total_seg;
  if (tid == 0) {
    rptr[num_ranges] = total_seg;
    hdr[MLA_HDR_B] = a.B; hdr[MLA_HDR_T] = a.T; hdr[MLA_HDR_H] = a.H; hdr[MLA_HDR_CAUSAL] = a.causal;
    hdr[MLA_HDR_NUM_GROUPS] = a.num_groups;
    hdr[MLA_HDR_NUM_SEGMENTS] = total_seg;
    hdr[MLA_HDR_NUM_RANGES] = num_ranges;
    hdr[MLA_HDR_NUM_PARTIALS] = cpart;
    hdr[MLA_HDR_NUM_MERGE] = cmrg;
    hdr[MLA_HDR_SEQ_HASH] = (int)hsum;
    hdr[MLA_HDR_ERROR] = errb == INT_MAX ? 0 : MLA_ERR_DEVICE_CHECK;
    hdr[MLA_HDR_ERROR_INFO] = errb == INT_MAX ? 0 : errb;
    hdr[MLA_HDR_PAGES_PER_RANGE] = q;
    hdr[MLA_HDR_NUM_SLOTS] = a.G;
    hdr[MLA_HDR_OVERRIDE] = a.N;
    hdr[MLA_HDR_MAX_PAGES] = a.max_pages;
    hdr[MLA_HDR_OFF_SEGMENTS] = (int)a.L.off_segments;
    hdr[MLA_HDR_OFF_RANGE_PTR] = (int)a.L.off_range_ptr;
    hdr[MLA_HDR_OFF_MERGE] = (int)a.L.off_merge;
    hdr[MLA_HDR_OFF_PART_LSE] = (int)a.L.off_part_lse;
    hdr[MLA_HDR_OFF_PART_O] = (int)a.L.off_part_o;
    hdr[MLA_HDR_CAP_SEGMENTS] = a.L.cap_segments;
    hdr[MLA_HDR_CAP_PARTIALS] = a.L.cap_partials;
    hdr[MLA_HDR_CAP_RANGES] = a.L.cap_ranges;
    hdr[MLA_HDR_CAP_GROUPS] = a.L.cap_groups;
    __threadfence();
    hdr[MLA_HDR_MAGIC] = MLA_PLAN_MAGIC;
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* seq_lens, const mla_geom* g, const mla_batch* b, const WsLayout& L,
                        void* ws, cudaStream_t st, int seq_div, int max_rows) {
  PlanArgs a;
  a.seq_lens = seq_lens;
  a.seq_div = seq_div;
  a.B = b->B; a.T = b->T; a.H = g->H; a.causal = b->causal ? 1 : 0;
  a.G = L.num_slots; a.N = b->num_splits_override; a.max_pages = b->max_pages;
  a.max_rows = max_rows > 0 ? max_rows : b->max_pages * kPage;
  a.RB = (b->T * g->H + kRowsPerBlock - 1) / kRowsPerBlock;
  a.num_groups = b->B * a.RB;
  a.L = L;
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, a, reinterpret_cast<char*>(ws));
}

}  // namespace mla
