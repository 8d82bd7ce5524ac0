// Split-KV absorbed-MLA decode on the sm_103a tensor cores (TMA + tcgen05/TMEM,
// 2-CTA clusters).
//
// What it computes ("MLA in full detail", Step 3; "M5.8" 0x04 absorbed
// reference): for every query row (b, t, h) of a plan segment,
//   s_j = (q_lat . c_j + q_pe . k_pe_j) * scale   over the visible cache rows j,
//   o_lat = sum_j softmax(s)_j c_j,  lse = log sum_j e^{s_j},
// where row j of the paged cache is [c_j (512) | k_pe_j (64)] and page
// j / 64 is found through the block table ("M5.8" 0x05).
//
// Work decomposition.  A query-row group is 128 flattened (t, h) rows of one
// sequence (one token's 128 heads at V3 geometry).  Its fp32 accumulator,
// 128 x 512, would take all 512 TMEM columns of an SM, so each group is
// handled by a CLUSTER of two CTAs: CTA h accumulates the output columns
// [256 h, 256 h + 256).  For each 64-row cache page both CTAs form the full
// 128 x 64 score tile S = Q K^T over all 576 columns (the second read of a
// page usually hits L2; the pair is co-scheduled as a cluster), run the same
// softmax, and each accumulates O[:, cols_h] += P V[:, cols_h], V being the
// leading 512 columns of the cached rows.  Swapping partial score tiles
// between the two CTAs instead of computing S twice was measured to cost more
// than it saves: the exchange moves as many bytes as the cache itself through
// distributed shared memory.
// Tensor-core shapes: Q K^T is M=128 x N=64 per K=16 step (36 steps per page);
// P V is M=128 x N=256 x K=16 (four steps per page), P read from TMEM.
//
// TMEM per CTA (512 columns): O half at 0..255; two 64-column score tiles at
// 256..383 (page t uses tile t % 2, so Q K^T of page t+1 runs while the
// softmax of page t reads its tile); the softmax writes P (bf16 pairs) over
// the first 32 columns of the tile it has read, which is where P V takes its
// A operand; query columns 0..255 (bf16 pairs, the TMEM A operand of Q K^T)
// at 384..511.  The rest of the query tile (latent 256..511 and RoPE) stays in
// shared memory next to a 2-stage page ring.
//
// Roles per CTA (384 threads): warp 0 lane 0 issues TMA loads (each page as
// two groups of 64 x 64 boxes, block-table entries read a few pages ahead);
// warp 1 issues Q K^T and warp 2 P V, each as a converged warp whose elected
// lane issues the MMAs (warp-uniform descriptors); warps 4..11 run the
// online softmax with two threads per query row (TMEM lane), write P and the
// epilogue.  At a segment boundary the softmax stages the next segment's
// query columns before it writes the finished segment out, so Q K^T of the
// next segment overlaps that epilogue.  The softmax keeps a per-row
// reference max and rescales the TMEM accumulator only when the running max
// grows past it by more than 2^8 (exact for any reference; only rounding
// differs), with scores in log2 units.  Cache rows past the sequence end
// (last page only) are zeroed in shared memory before P V so stale or NaN
// contents never reach the accumulator.
//
// Every wait is bounded; a wait that runs out records MLA_ERR_TIMEOUT in the
// workspace and raises a CTA-wide abort flag.  Loads and MMAs already issued
// are drained, TMEM is freed and both CTAs meet at a final cluster barrier.
#include <math.h>

#include "mla_internal.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kThreads = 384;                  // TMA, Q K^T and P V issue warps, 1 idle, 8 softmax warps
constexpr int kSoftmaxThreads = 256;
constexpr int kBoxBytes = 64 * 64 * 2;         // 8 KB: one 64-row page x 64 bf16 columns
constexpr int kQBoxBytes = 128 * 64 * 2;       // 16 KB: 128 query rows x 64 bf16
constexpr int kBoxes = 9;                      // 8 latent boxes + 1 RoPE box per row
constexpr int kOwnBoxes = 4;                   // latent boxes whose columns this CTA accumulates
constexpr int kQTmemBoxes = 4;                 // query boxes 0..3 live in TMEM
constexpr int kQSmemBoxes = kBoxes - kQTmemBoxes;
constexpr int kStages = 2;                     // page stages in the ring
constexpr int kGroupABoxes = 5;                // boxes only Q K^T needs (released after it)
constexpr int kStageBytes = kBoxes * kBoxBytes;  // group A (5 boxes) then group B (4 value boxes)
constexpr int kSmemQ = 0;
constexpr int kSmemRing = kSmemQ + kQSmemBoxes * kQBoxBytes;  // 81920
constexpr int kSmemBar = kSmemRing + kStages * kStageBytes;   // 229376
constexpr int kSmemXchg = kSmemBar + 256;                     // float [2 buffers][2 halves][128 rows]
constexpr int kSmemBytes = kSmemXchg + 2048;
constexpr int kSmemAlloc = kSmemBytes + 768;                  // slack to align the base to 1024 B (checked)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;   // tile t % 2 at kTmemS + 64 (t % 2)
constexpr uint32_t kTmemQ = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum {
  BAR_FULL_A = 0,                      // kStages: group A of a page landed
  BAR_EMPTY_A = BAR_FULL_A + kStages,  // kStages: Q K^T done with group A
  BAR_FULL_B = BAR_EMPTY_A + kStages,  // kStages: group B (value boxes) landed
  BAR_EMPTY_B = BAR_FULL_B + kStages,  // kStages: P V done with group B
  BAR_Q_FULL = BAR_EMPTY_B + kStages,  // query boxes in shared memory landed
  BAR_Q_EMPTY,                         // Q K^T done with the segment's query
  BAR_QT_FULL,                         // query columns staged in TMEM (256 arrivals)
  BAR_S_FULL,                          // 2: score tile written
  BAR_P_FULL = BAR_S_FULL + 2,         // 2: P written over the score tile (256 arrivals)
  BAR_P_EMPTY = BAR_P_FULL + 2,        // 2: P V done with the tile (it may be overwritten)
  BAR_O_EMPTY = BAR_P_EMPTY + 2,       // epilogue done with the accumulator (256 arrivals)
  BAR_FINAL,
  BAR_FINAL_PV,
  BAR_XCH,                             // 4: the two softmax warps of a TMEM lane quadrant
  kNumBars = BAR_XCH + 4
};
static_assert(kNumBars * 8 + 8 <= 256, "barrier area");
static_assert(kSmemAlloc <= 232448, "shared memory per CTA");

// A page is staged as two groups of 64 x 64 boxes: group A holds the five
// boxes this CTA needs only for Q K^T (the other CTA's four latent boxes and
// the RoPE box), released as soon as those MMAs complete; group B holds the
// four latent boxes whose columns this CTA accumulates, contiguous so that one
// N=256 MMA per K step covers them in P V, and released after P V.  Box order
// (by 64-column box index of the cached row; 8 = RoPE):
template <int HALF> struct Boxes {
  static constexpr int a(int j) { return j == 4 ? 8 : (HALF == 0 ? 4 + j : j); }
  static constexpr int b(int c) { return 4 * HALF + c; }
};

struct FastArgs {
  const __nv_bfloat16* q_lat;
  const int32_t* block_table;
  int bt_stride;
  const int32_t* seq_lens;
  int B, T, H, causal, checked, max_pages, num_blocks;
  float scale_log2;          // softmax scale times log2(e)
  __nv_bfloat16* o_lat;
  float* lse;
  WsLayout L;
};

struct Shared {
  uint32_t base;
  __device__ uint32_t q(int box) const { return base + kSmemQ + (box - kQTmemBoxes) * kQBoxBytes; }
  __device__ uint32_t stage_a(int st) const { return base + kSmemRing + st * kStageBytes; }
  __device__ uint32_t stage_b(int st) const { return stage_a(st) + kGroupABoxes * kBoxBytes; }
  __device__ uint32_t bar(int i) const { return base + kSmemBar + i * 8; }
};

// The segments of this pair's work ranges, in order: ranges pair,
// pair + num_pairs, ...; segment indices of range r are rptr[r] .. rptr[r+1).
struct SegWalk {
  const int* rptr;
  int r, si, end, step, num_ranges;
  __device__ SegWalk(const int* rp, int pair, int num_pairs, int nr)
      : rptr(rp), r(pair), si(0), end(0), step(num_pairs), num_ranges(nr) {
    if (r < nr) { si = rp[r]; end = rp[r + 1]; }
  }
  // Index of the current segment, or -1 once the walk is over.
  __device__ int cur() {
    while (r < num_ranges && si >= end) {
      r += step;
      if (r < num_ranges) { si = rptr[r]; end = rptr[r + 1]; }
    }
    return r < num_ranges ? si : -1;
  }
  __device__ void advance() { ++si; }
};

// Issue the Q K^T MMAs of one group of boxes into score tile d: A from TMEM
// (query boxes 0..3) or shared memory (4..8), B from consecutive 8 KB boxes
// starting at b0 (descriptor).  Called by the whole warp; one lane issues.
template <int HALF, bool GROUP_B>
__device__ __forceinline__ void issue_qk_group(uint32_t d, uint32_t tmem, const uint64_t (&qdesc)[kQSmemBoxes],
                                               uint64_t b0, uint32_t idesc) {
  constexpr int n = GROUP_B ? kOwnBoxes : kGroupABoxes;
#pragma unroll
  for (int j = 0; j < n; ++j) {
    const int box = GROUP_B ? Boxes<HALF>::b(j) : Boxes<HALF>::a(j);
    const uint64_t bd = b0 + (uint64_t)(j * (kBoxBytes >> 4));
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t acc = (GROUP_B || j || kk) ? 1u : 0u;
      if (box < kQTmemBoxes)
        mma_bf16_tmem_a_e(d, tmem + kTmemQ + 32 * box + 8 * kk, bd + 2 * kk, idesc, acc);
      else
        mma_bf16_e(d, qdesc[box - kQTmemBoxes] + 2 * kk, bd + 2 * kk, idesc, acc);
    }
  }
}

__device__ __forceinline__ void fail(int* hdr, volatile int* abort_flag, int where) {
  *abort_flag = 1;
  record_error(hdr, MLA_ERR_TIMEOUT, where);
}

// A bounded wait taken by every lane of a warp; true only if all lanes saw the
// phase complete (on a timeout lane 0 records it and raises the abort flag).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* hdr,
                                          int where) {
  const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
  if (!ok && (threadIdx.x & 31) == 0) fail(hdr, abort_flag, where);
  return ok;
}

// Q K^T issuer of one CTA (HALF = its rank in the pair), one converged warp.
// Page t goes to score tile t % 2 once P V of page t-2 has released it: Q K^T
// over group A, release A, Q K^T over group B -> S_FULL.
template <int HALF>
__device__ __forceinline__ void qk_role(const Shared& sh, uint32_t tmem, int* hdr, volatile int* abort_flag,
                                        const int* seg, SegWalk walk) {
  const uint32_t id_qk = idesc_bf16_f32(128, 64, 0);
  // Descriptors are built once; steps only move the start-address field (16-byte
  // units): +2 per 32-byte K step of a K-major tile, +kBoxBytes/16 per box,
  // +kStageBytes/16 per stage.
  uint64_t qdesc[kQSmemBoxes];
#pragma unroll
  for (int bx = 0; bx < kQSmemBoxes; ++bx) qdesc[bx] = sw128_desc(sh.q(kQTmemBoxes + bx), 16, 1024);
  const uint64_t adesc0 = sw128_desc(sh.stage_a(0), 16, 1024);
  const uint64_t bdesc0 = sw128_desc(sh.stage_b(0), 16, 1024);
  constexpr uint32_t kStageStep = kStageBytes >> 4;
  int ti = 0, sc = 0;
  bool ok = true;
  for (int si = walk.cur(); ok && si >= 0; walk.advance(), si = walk.cur()) {
    const int* rec = seg + (size_t)si * kSegWords;
    const int n_tiles = rec[3] - rec[2];
    if (!warp_wait(sh.bar(BAR_Q_FULL), sc & 1, abort_flag, hdr, 22) ||
        !warp_wait(sh.bar(BAR_QT_FULL), sc & 1, abort_flag, hdr, 22)) {
      ok = false; break;
    }
    tc_fence_after();
    for (int i = 0; ok && i < n_tiles; ++i, ++ti) {
      const int st = ti % kStages, sb = ti & 1;
      const uint32_t par = (ti / kStages) & 1;
      if ((ti >= 2 && !warp_wait(sh.bar(BAR_P_EMPTY + sb), ((ti >> 1) - 1) & 1, abort_flag, hdr, 23)) ||
          !warp_wait(sh.bar(BAR_FULL_A + st), par, abort_flag, hdr, 23)) {
        ok = false; break;
      }
      tc_fence_after();
      const uint32_t d = tmem + kTmemS + 64 * sb;
      issue_qk_group<HALF, false>(d, tmem, qdesc, adesc0 + st * kStageStep, id_qk);
      mma_commit_e(sh.bar(BAR_EMPTY_A + st));
      if (!warp_wait(sh.bar(BAR_FULL_B + st), par, abort_flag, hdr, 24)) { ok = false; break; }
      tc_fence_after();
      issue_qk_group<HALF, true>(d, tmem, qdesc, bdesc0 + st * kStageStep, id_qk);
      mma_commit_e(sh.bar(BAR_S_FULL + sb));
      if (i == n_tiles - 1) mma_commit_e(sh.bar(BAR_Q_EMPTY));
    }
    ++sc;
  }
  // Wait for every MMA issued by this warp before TMEM is released.
  mma_commit_e(sh.bar(BAR_FINAL));
  volatile int never = 0;
  mbar_wait(sh.bar(BAR_FINAL), 0, &never);
  __syncwarp();
}

// P V issuer, one converged warp: as soon as P of page t is written, O[:, own] +=
// P V over the page's group B (one N=256 MMA per K step, A = P from TMEM), then
// release group B and the score tile.
__device__ __forceinline__ void pv_role(const Shared& sh, uint32_t tmem, int* hdr, volatile int* abort_flag,
                                        const int* seg, SegWalk walk) {
  const uint32_t id_pv = idesc_bf16_f32(128, 256, 1);
  const uint64_t vdesc0 = sw128_desc(sh.stage_b(0), kBoxBytes, 1024);
  constexpr uint32_t kStageStep = kStageBytes >> 4;
  int ti = 0, sc = 0;
  bool ok = true;
  for (int si = walk.cur(); ok && si >= 0; walk.advance(), si = walk.cur()) {
    const int* rec = seg + (size_t)si * kSegWords;
    const int n_tiles = rec[3] - rec[2];
    for (int i = 0; i < n_tiles; ++i, ++ti) {
      if (i == 0 && sc > 0 && !warp_wait(sh.bar(BAR_O_EMPTY), (sc - 1) & 1, abort_flag, hdr, 20)) {
        ok = false; break;
      }
      const int sb = ti & 1, st = ti % kStages;
      if (!warp_wait(sh.bar(BAR_P_FULL + sb), (ti >> 1) & 1, abort_flag, hdr, 21)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16_tmem_a_e(tmem + kTmemO, tmem + kTmemS + 64 * sb + 8 * kk, vdesc0 + st * kStageStep + 128 * kk, id_pv,
                          (i == 0 && kk == 0) ? 0u : 1u);
      mma_commit_e(sh.bar(BAR_EMPTY_B + st));
      mma_commit_e(sh.bar(BAR_P_EMPTY + sb));
    }
    ++sc;
  }
  mma_commit_e(sh.bar(BAR_FINAL_PV));
  volatile int never = 0;
  mbar_wait(sh.bar(BAR_FINAL_PV), 0, &never);
  __syncwarp();
}

// What a softmax thread needs to know about one segment.
struct SegRows {
  int b, p0, p1, slot_out, S, fr, limit;
  bool row_valid;
};

__device__ __forceinline__ SegRows seg_rows(const int* rec, const FastArgs& a, int R, int row) {
  SegRows s;
  s.b = rec[0];
  s.p0 = rec[2];
  s.p1 = rec[3];
  s.slot_out = rec[5];
  int S = a.seq_lens[s.b];
  s.S = S < 0 ? 0 : min(S, a.max_pages * kPage);
  s.fr = rec[1] * kRowsPerBlock + row;
  s.row_valid = s.fr < R;
  s.limit = s.row_valid ? visible_limit(s.S, a.T, s.fr / a.H, a.causal) : 0;
  return s;
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_sm103_kernel(const __grid_constant__ CUtensorMap tm_qlat, const __grid_constant__ CUtensorMap tm_qpe,
                        const __grid_constant__ CUtensorMap tm_ckv, const __grid_constant__ CUtensorMap tm_kpe,
                        FastArgs a, char* ws) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* hdr = reinterpret_cast<int*>(ws);
  // The 128-byte-swizzled tiles need a 1024-byte-aligned base; the allocation
  // carries kSmemAlloc - kSmemBytes bytes of slack for that.  Refuse (uniformly,
  // before anything is set up) if the slack does not cover the misalignment.
  if ((uintptr_t)(smem - smem_raw) + kSmemBytes > (uintptr_t)kSmemAlloc) {
    pdl_wait();
    if (threadIdx.x == 0) record_error(hdr, MLA_ERR_DEVICE_CHECK, -2);
    return;
  }
  Shared sh{smem_addr(smem)};
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + kSmemBar + kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemBar + kNumBars * 8 + 4);

  const int* seg = reinterpret_cast<const int*>(ws + a.L.off_segments);
  const int* rptr = reinterpret_cast<const int*>(ws + a.L.off_range_ptr);
  float* part_lse = reinterpret_cast<float*>(ws + a.L.off_part_lse);
  float* part_o = reinterpret_cast<float*>(ws + a.L.off_part_o);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = (int)cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  const int R = a.T * a.H;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(sh.bar(BAR_FULL_A + i), 1);
      mbar_init(sh.bar(BAR_EMPTY_A + i), 1);
      mbar_init(sh.bar(BAR_FULL_B + i), 1);
      mbar_init(sh.bar(BAR_EMPTY_B + i), 1);
    }
    mbar_init(sh.bar(BAR_Q_FULL), 1);
    mbar_init(sh.bar(BAR_Q_EMPTY), 1);
    mbar_init(sh.bar(BAR_QT_FULL), kSoftmaxThreads);
    for (int i = 0; i < 2; ++i) {
      mbar_init(sh.bar(BAR_S_FULL + i), 1);
      mbar_init(sh.bar(BAR_P_FULL + i), kSoftmaxThreads);
      mbar_init(sh.bar(BAR_P_EMPTY + i), 1);
    }
    mbar_init(sh.bar(BAR_O_EMPTY), kSoftmaxThreads);
    mbar_init(sh.bar(BAR_FINAL), 1);
    mbar_init(sh.bar(BAR_FINAL_PV), 1);
    for (int i = 0; i < 4; ++i) mbar_init(sh.bar(BAR_XCH + i), 64);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_qlat);
    prefetch_tmap(&tm_qpe);
    prefetch_tmap(&tm_ckv);
    prefetch_tmap(&tm_kpe);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_base_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  // No early trigger: the merge that follows should be placed on the SMs as they
  // free up together, not packed onto the first few that do.
  pdl_wait();
  const int num_ranges = hdr[MLA_HDR_NUM_RANGES];
  const SegWalk walk0(rptr, pair, num_pairs, num_ranges);

  if (a.checked && blockIdx.x == 0 && tid == 0) {
    if (hdr[MLA_HDR_MAGIC] != MLA_PLAN_MAGIC || hdr[MLA_HDR_B] != a.B || hdr[MLA_HDR_T] != a.T ||
        hdr[MLA_HDR_H] != a.H || hdr[MLA_HDR_CAUSAL] != a.causal) {
      record_error(hdr, MLA_ERR_PLAN_STALE, 0);
    } else {
      unsigned h = 0;
      for (int b = 0; b < a.B; ++b) {
        unsigned S = (unsigned)a.seq_lens[b];
        unsigned x = (unsigned)b + 0x632BE5ABu;
        x ^= x >> 16; x *= 0x7feb352dU; x ^= x >> 15; x *= 0x846ca68bU; x ^= x >> 16;
        unsigned y = S * 0x9E3779B1u + x;
        y ^= y >> 16; y *= 0x7feb352dU; y ^= y >> 15; y *= 0x846ca68bU; y ^= y >> 16;
        h += y;
      }
      if ((int)h != hdr[MLA_HDR_SEQ_HASH]) record_error(hdr, MLA_ERR_PLAN_STALE, 1);
    }
  }

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      SegWalk walk = walk0;
      int gt = 0, sc = 0;
      bool q_in_flight = false, ok = true, a_only = false;
      for (int si = walk.cur(); ok && si >= 0; walk.advance(), si = walk.cur()) {
        const int* rec = seg + (size_t)si * kSegWords;
        const int b = rec[0], rb = rec[1], p0 = rec[2], p1 = rec[3];
        if (sc > 0 && !mbar_wait(sh.bar(BAR_Q_EMPTY), (sc - 1) & 1, abort_flag)) { fail(hdr, abort_flag, 10); ok = false; break; }
        const int row0 = b * R + rb * kRowsPerBlock;
        mbar_arrive_expect_tx(sh.bar(BAR_Q_FULL), kQSmemBoxes * kQBoxBytes);
        for (int box = kQTmemBoxes; box < 8; ++box) tma_load_2d(sh.q(box), &tm_qlat, sh.bar(BAR_Q_FULL), 64 * box, row0);
        tma_load_2d(sh.q(8), &tm_qpe, sh.bar(BAR_Q_FULL), 0, row0);
        q_in_flight = true;
        // Block ids are read a few pages ahead of their use (independent loads in flight).
        const int32_t* btrow = a.block_table + (size_t)b * a.bt_stride;
        int bq0 = p0 < p1 ? btrow[p0] : 0;
        int bq1 = p0 + 1 < p1 ? btrow[p0 + 1] : 0;
        int bq2 = p0 + 2 < p1 ? btrow[p0 + 2] : 0;
        int bq3 = p0 + 3 < p1 ? btrow[p0 + 3] : 0;
        for (int p = p0; ok && p < p1; ++p) {
          int blk = bq0;
          bq0 = bq1; bq1 = bq2; bq2 = bq3;
          bq3 = p + 4 < p1 ? btrow[p + 4] : 0;
          if (blk < 0 || blk >= a.num_blocks) {
            // An out-of-pool id reads as zeros through the tensor map; report it when checking.
            if (a.checked) record_error(hdr, MLA_ERR_DEVICE_CHECK, (b << 16) | p);
            blk = -1;
          }
          const int st = gt % kStages;
          const uint32_t par = ((gt / kStages) & 1) ^ 1;
          if (!mbar_wait_backoff(sh.bar(BAR_EMPTY_A + st), par, abort_flag)) { fail(hdr, abort_flag, 11); ok = false; break; }
          mbar_arrive_expect_tx(sh.bar(BAR_FULL_A + st), kGroupABoxes * kBoxBytes);
          for (int j = 0; j < kGroupABoxes; ++j) {
            const int box = half == 0 ? Boxes<0>::a(j) : Boxes<1>::a(j);
            const uint32_t dst = sh.stage_a(st) + j * kBoxBytes;
            if (box < 8) tma_load_3d(dst, &tm_ckv, sh.bar(BAR_FULL_A + st), 64 * box, 0, blk);
            else tma_load_3d(dst, &tm_kpe, sh.bar(BAR_FULL_A + st), 0, 0, blk);
          }
          if (!mbar_wait_backoff(sh.bar(BAR_EMPTY_B + st), par, abort_flag)) {
            fail(hdr, abort_flag, 12); ok = false; a_only = true; break;
          }
          mbar_arrive_expect_tx(sh.bar(BAR_FULL_B + st), kOwnBoxes * kBoxBytes);
          for (int c = 0; c < kOwnBoxes; ++c)
            tma_load_3d(sh.stage_b(st) + c * kBoxBytes, &tm_ckv, sh.bar(BAR_FULL_B + st), 64 * (4 * half + c), 0, blk);
          ++gt;
        }
        ++sc;
      }
      // Drain: every load issued must have landed before the CTA may exit (a page
      // whose group B was not issued after a failure is covered by its group A wait).
      const int first = gt > kStages ? gt - kStages : 0;
      for (int g = first; g < gt + (a_only ? 1 : 0); ++g) {
        volatile int never = 0;
        mbar_wait(sh.bar(BAR_FULL_A + g % kStages), (g / kStages) & 1, &never);
        if (g < gt) mbar_wait(sh.bar(BAR_FULL_B + g % kStages), (g / kStages) & 1, &never);
      }
      if (q_in_flight) {
        volatile int never = 0;
        mbar_wait(sh.bar(BAR_Q_FULL), (sc - 1) & 1, &never);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ Q K^T issuer (whole warp)
    if (half == 0) qk_role<0>(sh, tmem, hdr, abort_flag, seg, walk0);
    else qk_role<1>(sh, tmem, hdr, abort_flag, seg, walk0);
  } else if (warp == 2) {
    // ------------------------------------------------------------ P V issuer (whole warp)
    pv_role(sh, tmem, hdr, abort_flag, seg, walk0);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    // Two threads per query row: warps 4..7 take score columns 0..31 of their
    // TMEM lane quadrant, warps 8..11 columns 32..63 (a warp may only touch the
    // 32 TMEM lanes of quadrant warp % 4).  The row maximum is combined through
    // shared memory; each thread owns half of the row's P and O columns.
    const int q4 = warp & 3;
    const int ch = (warp - 4) >> 2;           // column half
    const int row = 32 * q4 + lane;           // query row within the group == TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q4) << 16);
    float* xrow = reinterpret_cast<float*>(smem + kSmemXchg);  // [buffer][half][row] partner exchange
    // Exchange a value with the partner thread of the same row (bounded wait on the
    // quadrant's mbarrier; double-buffered by exchange parity).  It also orders this
    // thread's earlier TMEM reads before the partner's later TMEM writes.
    int xc = 0;
    auto swap_with_partner = [&](float v, float* out) -> bool {
      float* slot = xrow + (xc & 1) * 256;
      slot[ch * 128 + row] = v;
      tc_fence_before();
      mbar_arrive(sh.bar(BAR_XCH + q4));
      const bool w = mbar_wait(sh.bar(BAR_XCH + q4), xc & 1, abort_flag);
      tc_fence_after();
      *out = slot[(ch ^ 1) * 128 + row];
      ++xc;
      return __all_sync(0xffffffffu, w);
    };
    // Query columns 0..255 of this row go to TMEM (A operand of Q K^T for boxes
    // 0..3; this thread stages boxes 2 ch and 2 ch + 1) once the previous
    // segment's Q K^T MMAs are done with them.
    auto stage_q = [&](const SegRows& s, int sc_of) -> bool {
      const bool w_ok = sc_of == 0 || mbar_wait(sh.bar(BAR_Q_EMPTY), (sc_of - 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, w_ok)) return false;
      tc_fence_after();
      const uint4* src = reinterpret_cast<const uint4*>(a.q_lat + ((size_t)s.b * R + (s.row_valid ? s.fr : 0)) * kDLat) +
                         16 * ch;
      uint32_t q0[32], q1[32];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint4 v0 = s.row_valid ? __ldg(src + e) : make_uint4(0, 0, 0, 0);
        const uint4 v1 = s.row_valid ? __ldg(src + 8 + e) : make_uint4(0, 0, 0, 0);
        q0[4 * e] = v0.x; q0[4 * e + 1] = v0.y; q0[4 * e + 2] = v0.z; q0[4 * e + 3] = v0.w;
        q1[4 * e] = v1.x; q1[4 * e + 1] = v1.y; q1[4 * e + 2] = v1.z; q1[4 * e + 3] = v1.w;
      }
      tmem_st32(t_lane + kTmemQ + 32 * (2 * ch), q0);
      tmem_st32(t_lane + kTmemQ + 32 * (2 * ch + 1), q1);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(sh.bar(BAR_QT_FULL));
      return true;
    };

    SegWalk walk = walk0;
    int si = walk.cur();
    int ti = 0, sc = 0;
    bool ok = true;
    SegRows cur;
    if (si >= 0) {
      cur = seg_rows(seg + (size_t)si * kSegWords, a, R, row);
      if (!stage_q(cur, 0)) { fail(hdr, abort_flag, 33); ok = false; }
    }
    while (ok && si >= 0) {
      float m_ref = -INFINITY, l = 0.f;   // l: this thread's half of the row sum
      const int n_tiles = cur.p1 - cur.p0;
      for (int i = 0; i < n_tiles; ++i, ++ti) {
        const int sb = ti & 1;
        const uint32_t s_col = kTmemS + 64 * sb;
        const int jbase = (cur.p0 + i) * kPage + 32 * ch;   // first cache row of this thread's columns
        bool w_ok = mbar_wait(sh.bar(BAR_S_FULL + sb), (ti >> 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) { fail(hdr, abort_flag, 30); ok = false; break; }
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld32(t_lane + s_col + 32 * ch, sr);
        tmem_wait_ld();
        // Raw-score maximum over the visible columns (the scale is positive).
        const bool full = jbase + 32 <= cur.limit;
        float tmax = -INFINITY;
        if (full) {
#pragma unroll
          for (int j = 0; j < 32; ++j) tmax = fmaxf(tmax, __uint_as_float(sr[j]));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (jbase + j < cur.limit) tmax = fmaxf(tmax, __uint_as_float(sr[j]));
        }
        {
          float other;
          if (!swap_with_partner(tmax, &other)) { fail(hdr, abort_flag, 37); ok = false; break; }
          tmax = fmaxf(tmax, other) * a.scale_log2;
        }
        // Lazy rescale of the running state: needs the accumulator up to date (P V of
        // the previous page complete); rare once the reference max has settled.
        const bool grow = tmax > m_ref + kRescaleThreshold;
        const float new_ref = grow ? tmax : m_ref;
        const float factor = (grow && m_ref != -INFINITY) ? ex2(m_ref - new_ref) : 1.f;
        if (i > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
          const int t1 = ti - 1;
          w_ok = mbar_wait(sh.bar(BAR_P_EMPTY + (t1 & 1)), (t1 >> 1) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, w_ok)) { fail(hdr, abort_flag, 31); ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 4 * ch; c < 4 * ch + 4; ++c) {
            uint32_t o[32];
            tmem_ld32(t_lane + kTmemO + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
            tmem_st32(t_lane + kTmemO + 32 * c, o);
          }
          tmem_wait_st();
        }
        l *= factor;
        m_ref = new_ref;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        // This thread's 32 P values, p = 2^(s * scale * log2 e - m), as bf16 pairs over
        // columns 16 ch .. 16 ch + 15 of the score tile it has read (the partner has
        // read its scores too: the exchange above came after both reads).
        float psum = 0.f;
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = 2 * e;
          float x0 = ex2(fmaf(__uint_as_float(sr[j]), a.scale_log2, -m_use));
          float x1 = ex2(fmaf(__uint_as_float(sr[j + 1]), a.scale_log2, -m_use));
          if (!full) {
            x0 = (jbase + j < cur.limit) ? x0 : 0.f;
            x1 = (jbase + j + 1 < cur.limit) ? x1 : 0.f;
          }
          psum += x0 + x1;
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
          pw[e] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        tmem_st16(t_lane + s_col + 16 * ch, pw);
        l += psum;
        // Rows of the last page past the sequence end are zeroed in the four value
        // boxes of this page (its group B) before P V reads them.
        const int valid = cur.S - (cur.p0 + i) * kPage;
        if (valid < kPage) {
          const int t256 = tid - 128;   // 0..255 over the two warpgroups
          for (int idx = t256; idx < kOwnBoxes * kPage; idx += 256) {
            const int c = idx / kPage, rr = idx % kPage;
            if (rr >= valid) {
              const uint32_t dst = sh.stage_b(ti % kStages) + c * kBoxBytes + rr * 128;
#pragma unroll
              for (int z = 0; z < 8; ++z)
                asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(dst + 16 * z), "r"(0) : "memory");
            }
          }
          fence_proxy_async_smem();
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(sh.bar(BAR_P_FULL + sb));
      }
      if (!ok) break;
      // The next segment's query goes to TMEM now, so that its Q K^T can run while
      // this segment is written out.
      walk.advance();
      const int si_next = walk.cur();
      SegRows nxt = cur;
      if (si_next >= 0) {
        nxt = seg_rows(seg + (size_t)si_next * kSegWords, a, R, row);
        if (!stage_q(nxt, sc + 1)) { fail(hdr, abort_flag, 33); ok = false; break; }
      }
      // Epilogue: wait for the last P V, combine the two halves of the row sum,
      // then normalise and store this thread's 128 output columns.
      {
        const int tl = ti - 1;
        const bool w_ok = mbar_wait(sh.bar(BAR_P_EMPTY + (tl & 1)), (tl >> 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) { fail(hdr, abort_flag, 32); ok = false; break; }
        tc_fence_after();
      }
      float l_other;
      if (!swap_with_partner(l, &l_other)) { fail(hdr, abort_flag, 38); ok = false; break; }
      const float l_row = ch == 0 ? l + l_other : l_other + l;
      const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      const float lse_v = l_row > 0.f ? (m_use + __log2f(l_row)) * 0.69314718055994531f : -INFINITY;
      const int b = cur.b, fr = cur.fr, slot_out = cur.slot_out;
#pragma unroll 1
      for (int c = 4 * ch; c < 4 * ch + 4; ++c) {
        uint32_t o[32];
        tmem_ld32(t_lane + kTmemO + 32 * c, o);
        tmem_wait_ld();
        if (cur.row_valid) {
          // 32-byte stores: each thread writes whole sectors of its row.
          if (slot_out < 0) {
            __nv_bfloat16* dst = a.o_lat + ((size_t)b * R + fr) * kDLat + 256 * half + 32 * c;
#pragma unroll
            for (int e = 0; e < 32; e += 16) {
              uint32_t w[8];
              pack_bf16x8(o + e, inv, w);
              pack_bf16x8(o + e + 8, inv, w + 4);
              st_global_v8(dst + e, w);
            }
          } else {
            float* dst = part_o + ((size_t)slot_out * kRowsPerBlock + row) * kDLat + 256 * half + 32 * c;
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint32_t w[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(__uint_as_float(o[e + k]) * inv);
              st_global_v8(dst + e, w);
            }
          }
        }
      }
      if (cur.row_valid && half == 0 && ch == 0) {
        if (slot_out < 0) a.lse[(size_t)b * R + fr] = lse_v;
        else part_lse[(size_t)slot_out * kRowsPerBlock + row] = lse_v;
      }
      tc_fence_before();
      mbar_arrive(sh.bar(BAR_O_EMPTY));
      ++sc;
      si = si_next;
      cur = nxt;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// --------------------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
              const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides_bytes, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool set_kernel_attributes() {
  static bool done = false;
  if (!done) {
    if (cudaFuncSetAttribute(decode_sm103_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) !=
        cudaSuccess)
      return false;
    done = true;
  }
  return true;
}

// Launch configuration: clusters of two CTAs; with `pdl`, also programmatic
// stream serialisation (the kernel waits for its predecessor in pdl_wait).
void cluster_launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int pairs, cudaStream_t st,
                           bool pdl) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = dim3(2 * pairs, 1, 1);
  cfg->blockDim = dim3(kThreads, 1, 1);
  cfg->dynamicSmemBytes = kSmemAlloc;
  cfg->stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attr;
  cfg->numAttrs = pdl ? 2 : 1;
}

}  // namespace

// Clusters (CTA pairs) of the decode kernel that can be resident at once on the current device.
int decode_sm103_pairs_per_device() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    if (set_kernel_attributes()) {
      cudaLaunchConfig_t cfg;
      cudaLaunchAttribute attr[2];
      cluster_launch_config(&cfg, attr, 256, 0, false);
      if (cudaOccupancyMaxActiveClusters(&n, decode_sm103_kernel, &cfg) != cudaSuccess) n = 0;
    }
    if (n <= 0) {
      const int sms = mla_device_sm_count();
      n = sms >= 2 ? sms / 2 : 1;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

cudaError_t launch_decode_sm103(const mla_geom* g, const mla_batch* b, const WsLayout& L,
                                const __nv_bfloat16* q_lat, const __nv_bfloat16* q_pe, const CacheView& cv,
                                const int32_t* block_table, int bt_stride, const int32_t* seq_lens, int checked,
                                __nv_bfloat16* o_lat, float* lse, void* ws, cudaStream_t st) {
  const long long rows_total = (long long)b->B * b->T * g->H;
  CUtensorMap m_qlat, m_qpe, m_ckv, m_kpe;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kDLat, (cuuint64_t)rows_total};
    const cuuint64_t str[1] = {(cuuint64_t)kDLat * 2};
    const cuuint32_t box[2] = {64, 128};
    if (!make_map(&m_qlat, q_lat, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kDRope, (cuuint64_t)rows_total};
    const cuuint64_t str[1] = {(cuuint64_t)kDRope * 2};
    const cuuint32_t box[2] = {64, 128};
    if (!make_map(&m_qpe, q_pe, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kDLat, (cuuint64_t)kPage, (cuuint64_t)cv.num_blocks};
    const cuuint64_t str[2] = {(cuuint64_t)cv.ckv_row * 2, (cuuint64_t)cv.ckv_block * 2};
    const cuuint32_t box[3] = {64, 64, 1};
    if (!make_map(&m_ckv, cv.ckv, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kDRope, (cuuint64_t)kPage, (cuuint64_t)cv.num_blocks};
    const cuuint64_t str[2] = {(cuuint64_t)cv.kpe_row * 2, (cuuint64_t)cv.kpe_block * 2};
    const cuuint32_t box[3] = {64, 64, 1};
    if (!make_map(&m_kpe, cv.kpe, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  FastArgs a;
  a.q_lat = q_lat;
  a.block_table = block_table; a.bt_stride = bt_stride; a.seq_lens = seq_lens;
  a.B = b->B; a.T = b->T; a.H = g->H; a.causal = b->causal ? 1 : 0; a.checked = checked;
  a.max_pages = b->max_pages; a.num_blocks = cv.num_blocks;
  a.scale_log2 = g->softmax_scale * 1.4426950408889634f;
  a.o_lat = o_lat; a.lse = lse; a.L = L;
  if (!set_kernel_attributes()) return cudaErrorInvalidValue;
  int pairs = L.cap_ranges;
  const int max_pairs = decode_sm103_pairs_per_device();
  if (pairs > max_pairs) pairs = max_pairs;
  if (pairs <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cluster_launch_config(&cfg, attr, pairs, st, true);
  return cudaLaunchKernelEx(&cfg, decode_sm103_kernel, m_qlat, m_qpe, m_ckv, m_kpe, a, reinterpret_cast<char*>(ws));
}

}  // namespace mla
