// Device split planner: builds the work plan (segments, ranges, merge list) in
// the workspace from the device-resident sequence lengths, with no host sync.
// The rule is stated in include/mla.h next to the plan layout.
#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kPlanThreads = 1024;

// Block-wide exclusive scan of one int per thread; *total gets the block sum.
__device__ int block_excl_scan(int v, int* total, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;
  }
  __syncthreads();
  int pre = warp ? sh[warp - 1] : 0;
  *total = sh[nwarps - 1];
  __syncthreads();
  return pre + x - v;
}

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  x ^= x >> 16; x *= 0x7feb352dU; x ^= x >> 15; x *= 0x846ca68bU; x ^= x >> 16;
  return x;
}

struct PlanArgs {
  const int32_t* seq_lens;
  int B, T, H, causal, G, N, max_pages;
  int RB, num_groups;
  WsLayout L;
};

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a, char* ws) {
  int* hdr = reinterpret_cast<int*>(ws);
  int* grp = reinterpret_cast<int*>(ws + a.L.off_groups);
  int* seg = reinterpret_cast<int*>(ws + a.L.off_segments);
  int* rptr = reinterpret_cast<int*>(ws + a.L.off_range_ptr);
  int* mrg = reinterpret_cast<int*>(ws + a.L.off_merge);
  __shared__ int sh[32];
  __shared__ int s_W, s_nonempty, s_maxn, s_err, s_errinfo;
  __shared__ unsigned s_hash;
  __shared__ int s_q, s_mode, s_total_seg, s_total_part, s_total_merge;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_W = 0; s_nonempty = 0; s_maxn = 0; s_err = 0; s_errinfo = 0; s_hash = 0;
  }
  pdl_wait();
  pdl_trigger();
  __syncthreads();

  // Sequence-length stamp and validation.
  for (int b = tid; b < a.B; b += blockDim.x) {
    int S = a.seq_lens[b];
    atomicAdd(&s_hash, mix32((uint32_t)S * 0x9E3779B1u + mix32((uint32_t)b + 0x632BE5ABu)));
    if (S < 0 || S > a.max_pages * kPage || (S > 0 && S < a.T)) {
      if (atomicCAS(&s_err, 0, MLA_ERR_DEVICE_CHECK) == 0) s_errinfo = b;
    }
  }

  // Pass A: pages per group and their exclusive prefix.
  int carry = 0;
  const int R = a.T * a.H;
  for (int base = 0; base < a.num_groups; base += blockDim.x) {
    const int g = base + tid;
    int n = 0;
    if (g < a.num_groups) {
      const int b = g / a.RB, rb = g % a.RB;
      int S = a.seq_lens[b];
      S = S < 0 ? 0 : (S > a.max_pages * kPage ? a.max_pages * kPage : S);
      const int r_last = min(R, (rb + 1) * kRowsPerBlock) - 1;
      const int vis = visible_limit(S, a.T, r_last / a.H, a.causal);
      n = (vis + kPage - 1) / kPage;
    }
    int tot;
    int off = block_excl_scan(n, &tot, sh);
    if (g < a.num_groups) {
      grp[g * kGroupWords + 0] = n;
      grp[g * kGroupWords + 1] = carry + off;
      if (n > 0) {
        atomicAdd(&s_nonempty, 1);
        atomicMax(&s_maxn, n);
      }
    }
    carry += tot;
  }
  if (tid == 0) {
    s_W = carry;
    int q = (carry + a.G - 1) / a.G;
    q = q < kMinSplitPages ? kMinSplitPages : q;
    s_q = q;
    if (a.N > 0) s_mode = 2;
    else if (s_nonempty <= a.G && s_maxn <= (5 * q + 3) / 4) s_mode = 0;
    else s_mode = 1;
  }
  __syncthreads();
  const int q = s_q, mode = s_mode;

  // Pass B: segments per group, segment/slot/merge bases.
  int cseg = 0, cpart = 0, cmrg = 0;
  for (int base = 0; base < a.num_groups; base += blockDim.x) {
    const int g = base + tid;
    int k = 0, n = 0;
    if (g < a.num_groups) {
      n = grp[g * kGroupWords + 0];
      const int off = grp[g * kGroupWords + 1];
      if (n > 0) {
        if (mode == 2) k = min(n, a.N);
        else if (mode == 0) k = 1;
        else k = (off + n - 1) / q - off / q + 1;
      }
    }
    const int part = k > 1 ? k : 0;
    const int mflag = (g < a.num_groups && k != 1) ? 1 : 0;
    int t1, t2, t3;
    int sb = block_excl_scan(k, &t1, sh);
    int pb = block_excl_scan(part, &t2, sh);
    int mb = block_excl_scan(mflag, &t3, sh);
    if (g < a.num_groups) {
      grp[g * kGroupWords + 2] = k;
      grp[g * kGroupWords + 3] = cseg + sb;
      grp[g * kGroupWords + 4] = part ? cpart + pb : -1;
      grp[g * kGroupWords + 5] = mflag ? cmrg + mb : -1;
    }
    cseg += t1; cpart += t2; cmrg += t3;
  }
  if (tid == 0) {
    s_total_seg = cseg; s_total_part = cpart; s_total_merge = cmrg;
  }
  __syncthreads();
  const int num_ranges = (mode == 1) ? (s_W + q - 1) / q : s_total_seg;

  // Pass C: segment records, merge records and range pointers.
  for (int g = tid; g < a.num_groups; g += blockDim.x) {
    const int n = grp[g * kGroupWords + 0];
    const int off = grp[g * kGroupWords + 1];
    const int k = grp[g * kGroupWords + 2];
    const int sb = grp[g * kGroupWords + 3];
    const int pb = grp[g * kGroupWords + 4];
    const int mi = grp[g * kGroupWords + 5];
    const int b = g / a.RB, rb = g % a.RB;
    for (int s = 0; s < k; ++s) {
      int p0, p1, r;
      if (mode == 2) {
        p0 = (int)(((long long)s * n) / k);
        p1 = (int)(((long long)(s + 1) * n) / k);
        r = sb + s;
      } else if (mode == 0) {
        p0 = 0; p1 = n; r = sb;
      } else {
        const int r0 = off / q;
        r = r0 + s;
        const int gs = max(off, r * q), ge = min(off + n, (r + 1) * q);
        p0 = gs - off; p1 = ge - off;
      }
      int* rec = seg + (size_t)(sb + s) * kSegWords;
      rec[0] = b; rec[1] = rb; rec[2] = p0; rec[3] = p1; rec[4] = r;
      rec[5] = (k > 1) ? pb + s : -1; rec[6] = 0; rec[7] = 0;
    }
    if (mi >= 0) {
      int* m = mrg + (size_t)mi * kMergeWords;
      m[0] = b; m[1] = rb; m[2] = (k > 1) ? pb : 0; m[3] = (k > 1) ? k : 0;
    }
  }
  __syncthreads();
  // First segment of each range (segments are in nondecreasing range order).
  for (int i = tid; i < s_total_seg; i += blockDim.x) {
    const int r = seg[(size_t)i * kSegWords + 4];
    const int rprev = i ? seg[(size_t)(i - 1) * kSegWords + 4] : -1;
    for (int rr = rprev + 1; rr <= r; ++rr) rptr[rr] = i;
  }
  if (tid == 0) {
    rptr[num_ranges] = s_total_seg;
    hdr[MLA_HDR_B] = a.B; hdr[MLA_HDR_T] = a.T; hdr[MLA_HDR_H] = a.H; hdr[MLA_HDR_CAUSAL] = a.causal;
    hdr[MLA_HDR_NUM_GROUPS] = a.num_groups;
    hdr[MLA_HDR_NUM_SEGMENTS] = s_total_seg;
    hdr[MLA_HDR_NUM_RANGES] = num_ranges;
    hdr[MLA_HDR_NUM_PARTIALS] = s_total_part;
    hdr[MLA_HDR_NUM_MERGE] = s_total_merge;
    hdr[MLA_HDR_SEQ_HASH] = (int)s_hash;
    hdr[MLA_HDR_ERROR] = s_err;
    hdr[MLA_HDR_ERROR_INFO] = s_errinfo;
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
                        void* ws, cudaStream_t st) {
  PlanArgs a;
  a.seq_lens = seq_lens;
  a.B = b->B; a.T = b->T; a.H = g->H; a.causal = b->causal ? 1 : 0;
  a.G = L.num_slots; a.N = b->num_splits_override; a.max_pages = b->max_pages;
  a.RB = (b->T * g->H + kRowsPerBlock - 1) / kRowsPerBlock;
  a.num_groups = b->B * a.RB;
  a.L = L;
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, a, reinterpret_cast<char*>(ws));
}

}  // namespace mla
