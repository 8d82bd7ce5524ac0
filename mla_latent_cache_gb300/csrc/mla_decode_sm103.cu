// Split-KV absorbed-MLA decode on the sm_103a tensor cores: TMA, tcgen05 pair
// MMAs (cta_group::2) with tensor-memory accumulators, 2-CTA clusters.
//
// What it computes ("MLA in full detail", Step 3; "M5.8" 0x04 absorbed
// reference): for every query row (b, t, h) of a plan segment,
//   s_j = (q_lat . c_j + q_pe . k_pe_j) * scale   over the visible cache rows j,
//   o_lat = sum_j softmax(s)_j c_j,  lse = log sum_j e^{s_j},
// where row j of the paged cache is [c_j (512) | k_pe_j (64)] and page
// j / 64 is found through the block table ("M5.8" 0x05).
//
// Work decomposition.  A query-row group is 128 flattened (t, h) rows of one
// sequence (one token's 128 heads at V3 geometry), handled by a CLUSTER of two
// CTAs: CTA r owns rows [64 r, 64 r + 64) and everything per row (softmax
// state, accumulator, outputs).  Every product is a pair MMA issued by CTA 0:
//   S = Q K^T   M=128 (64 rows per CTA), N=64 (one page), K=576: each CTA
//               holds half of the page's cache rows (rows [32 r, 32 r + 32))
//               as its half of B, so the page is read once per pair and no
//               score is computed twice;
//   O += P V    M=128, N=256 per MMA (two MMAs cover the 512 latent columns),
//               K=64 page rows: A = P of the CTA's own rows (shared memory),
//               B = V split along N: CTA r supplies latent columns
//               [256 m + 128 r, +128) of MMA m for all 64 rows of the page.
// For P V each CTA therefore also needs the other half's rows of its latent
// columns; once Q K^T is done with a page, the four slots that held this
// CTA's Q K^T-only latent boxes are reloaded with exactly those rows (an L2 hit:
// the partner CTA fetched them from HBM), which puts every P V operand at the
// same shared-memory offset in both CTAs.
//
// Tensor memory per CTA (512 columns, allocated for the pair):
//   O:  columns 0..255: 64 rows x 512 latent columns, packed two rows per TMEM
//       lane: lane i < 64 holds row i, latent [256 m, +128) of MMA m at columns
//       128 m ..; lane 64 + i holds row i, latent [256 m + 128, +128);
//   S:  two 32-column score tiles (page t uses tile t % 2): lane i < 64 holds
//       row i's scores for page rows 0..31, lane 64 + i for rows 32..63;
//   Q:  query columns 0..383 (bf16 pairs), the TMEM A operand of the first 24
//       K steps; query columns 384..575 stay in shared memory.  Row i sits in
//       lane i AND lane 64 + i: with the packed M=128 pair layout, the lanes
//       that produce the second half of N read their A rows from lanes 64..127
//       (measured on this part: the lower copy alone leaves that half without
//       those K steps).
// Shared memory per CTA: a ring of page stages (nine 32-row x 64-column boxes,
// 36 KB), the P tiles (64 rows x 64 page rows, bf16, K-major) and the shared
// part of the query.
//
// Roles (384 threads per CTA): warp 0's lane 0 issues the page loads and its
// lane 1 the reloads; in CTA 0 warp 1 issues the Q K^T MMAs and warp 2 the P V MMAs (two
// issuers, so that Q K^T of the next pages keeps the tensor pipe busy while
// P V waits for the softmax); in CTA 1 warps 2 and 1 forward the arrival of
// its page halves and of its reloads to CTA 0; warps 4..11 run the online
// softmax (two threads per TMEM lane: row i % 64, page half i / 64, half of
// the lane's columns each), write P, stage the query and write the outputs.  The softmax keeps a per-row reference max and rescales its accumulator rows only
// when the running max grows past it by more than 2^8 (exact for any
// reference; only rounding differs), with scores in log2 units.  Cache rows
// past the sequence end (last page only) are zeroed in shared memory before
// P V so stale or NaN contents never reach the accumulator.
//
// Segments that are splits of their group write normalised partial states;
// after freeing tensor memory the CTAs merge the plan's records (exact LSE
// merge), each record once its partial rows are counted in.
//
// Load modes (template kMode): bf16 pages through the block table; the sparse
// decode's listed rows (copied by whole warps with cp.async); FP8 656-byte
// rows, converted to bf16 in shared memory by four more warps (512 threads).
//
// Every wait is bounded; a wait that runs out records MLA_ERR_TIMEOUT in the
// workspace and raises a CTA-wide abort flag.  Loads and MMAs already issued
// are drained, and both CTAs meet at a final cluster barrier before the
// tensor memory is freed.
#include <math.h>

#include <atomic>

// The decode's pipeline waits read their limit from here (a test can shorten it
// through mla_debug_set_wait_limit; the drains keep the full limit).
namespace mla {
namespace wait_override {
__constant__ long long c_pipeline_wait_limit = 2000000000LL;
}
}  // namespace mla
#define MLA_PIPELINE_WAIT_LIMIT (::mla::wait_override::c_pipeline_wait_limit)

#include "mla_internal.cuh"
#include "mla_plan_merge.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

// Load modes of the decode kernel: bf16 pages through the block table, listed
// rows (the sparse decode), or 656-byte FP8 rows through the block table.
constexpr int kModeDense = 0, kModeSparse = 1, kModeFp8 = 2;
constexpr int kThreads = 384;   // a multiple of 128 (the merge's thread groups)
constexpr int kFp8Threads = 512;  // plus four converter warps (12..15) in the FP8 mode
template <int kMode>
__host__ __device__ constexpr int threads_of() { return kMode == kModeFp8 ? kFp8Threads : kThreads; }
constexpr int kCtaRows = 64;                   // query rows per CTA
constexpr int kHalfRows = 32;                  // page rows loaded by each CTA
constexpr int kBoxes = 9;                      // 8 latent boxes + 1 RoPE box per cached row
constexpr int kSlotBytes = kHalfRows * 128;    // 4 KB: 32 rows x 64 bf16, 128-byte swizzled
constexpr int kStageBytes = kBoxes * kSlotBytes;
constexpr int kStages = 5;
constexpr int kQTmemBoxes = 6;                 // query boxes 0..5 in TMEM
constexpr int kQSmemBoxes = kBoxes - kQTmemBoxes;
constexpr int kQBoxBytes = kCtaRows * 128;     // 8 KB
constexpr int kPBufs = 2;
// The first segment's query boxes 0..5 land in ring stages 3 and 4 (before their
// first page) and are copied from there into tensor memory.
constexpr int kQStageFirst = 3;
constexpr int kPBytes = kCtaRows * 128;        // 8 KB: 64 rows x 64 page rows bf16
constexpr int kSmemQ = 0;
constexpr int kSmemP = kSmemQ + kQSmemBoxes * kQBoxBytes;
constexpr int kSmemRing = kSmemP + kPBufs * kPBytes;
constexpr int kSmemBar = kSmemRing + kStages * kStageBytes;
constexpr int kSmemXchg = kSmemBar + 512;                     // float [2 buffers][4 quarters][64 rows]
constexpr int kSmemScales = kSmemXchg + 2048;                 // FP8 mode: a stage's 32 rows x 4 fp32 scales
constexpr int kSmemBytes = kSmemScales + kStages * 512;
constexpr int kSmemAlloc = kSmemBytes + 1024;                 // slack to align the base to 1024 B (checked)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;   // tile t % 2 at kTmemS + 32 (t % 2)
constexpr uint32_t kTmemQ = 320;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

static_assert(kTmemQ + 32 * kQTmemBoxes <= kTmemCols, "tensor memory");
static_assert(kQStageFirst + 2 == kStages && kQTmemBoxes * 8192 <= 2 * kBoxes * 4096, "query staging in the ring");
static_assert(kSmemAlloc <= 232448, "shared memory per CTA");
static_assert(kSmemRing % 1024 == 0 && kSmemP % 1024 == 0 && kSlotBytes % 1024 == 0, "swizzle atoms");
static_assert(kSlotBytes == 4096 && kQBoxBytes == 8192 && kQTmemBoxes == 6 && kBoxes == 9,
              "the immediate operand offsets of qk_page_e and pv_page_e");

enum {
  BAR_FULL = 0,                        // kStages: this CTA's half-page landed (TMA); at CTA 0 also CTA 1's (relayed)
  BAR_RELOAD = BAR_FULL + kStages,     // kStages: the reloaded rows landed (TMA); at CTA 0 also CTA 1's (relayed)
  BAR_QK_DONE = BAR_RELOAD + kStages,  // kStages: Q K^T of the page done (both CTAs)
  BAR_PV_DONE = BAR_QK_DONE + kStages, // kStages: P V of the page done (both CTAs)
  BAR_S_FULL = BAR_PV_DONE + kStages,  // 2: score tile written (both CTAs)
  BAR_S_FREE = BAR_S_FULL + 2,         // 2: (CTA 0) both CTAs' softmax read the tile (16 warp arrivals)
  BAR_P_FULL = BAR_S_FREE + 2,         // kPBufs: (CTA 0) both CTAs wrote P (16 warp arrivals)
  BAR_Q_TMA = BAR_P_FULL + kPBufs,     // query boxes in shared memory landed (TMA)
  BAR_Q_READY = BAR_Q_TMA + 1,         // (CTA 0) both CTAs staged the query (16 warp arrivals)
  BAR_Q_COPIED = BAR_Q_READY + 1,      // the first query's boxes 0..5 left ring stages 3, 4 (8 local warp arrivals)
  BAR_Q_FREE = BAR_Q_COPIED + 1,        // Q K^T of the segment done with the query (both CTAs)
  BAR_O_FREE = BAR_Q_FREE + 1,         // (CTA 0) both CTAs' epilogues read the accumulator (16 warp arrivals)
  BAR_XCH = BAR_O_FREE + 1,            // 2: the four softmax warps sharing a row range (4 warp arrivals)
  BAR_FINAL_QK = BAR_XCH + 2,
  BAR_FINAL_PV,
  // FP8 mode: the raw rows landed (TMA), for the converter warps; then BAR_FULL and
  // BAR_RELOAD count the four converter warps' arrivals (at CTA 0 also CTA 1's, relayed).
  BAR_RAW,                             // kStages: the page half's raw rows
  BAR_RLRAW = BAR_RAW + kStages,       // kStages: the other half's raw codes and scales of this CTA's P V boxes
  kNumBars = BAR_RLRAW + kStages
};
static_assert(kNumBars * 8 + 16 <= 512, "barrier area");

// Slots: box b of a page half is slot b.  CTA r accumulates latent boxes
// {2r, 2r+1, 4+2r, 5+2r}; after Q K^T the slots of the other four latent boxes
// receive those boxes' rows of the other page half.
__device__ __forceinline__ int own_pv_box(int r, int i) { return (i < 2 ? 0 : 4) + 2 * r + (i & 1); }
__device__ __forceinline__ int reload_slot(int r, int i) { return (i < 2 ? 0 : 4) + 2 * (1 - r) + (i & 1); }

// The paged address translation of a load ("M5.8" 0x05): page rows are tensor-map
// coordinates (64 columns, 64 rows of a block, column block, block id), so a
// block id selects the page and a row offset selects the half; a block id of -1
// (outside the pool) reads zeros.  These two functions are the only places that
// form those coordinates; the debug gather export issues them too.
//
// Half `half` of a page (rows [32 half, 32 half + 32), all 576 columns) into the
// nine 32-row slots of a stage, arriving on `bar` with the stage's byte count.
__device__ __forceinline__ void load_page_half(uint32_t stage, const CUtensorMap* tm_page, const CUtensorMap* tm_kpe,
                                               uint32_t bar, int half, int blk, int kpe_separate) {
  mbar_arrive_expect_tx(bar, kStageBytes);
  tma_load_4d(stage, tm_page, bar, 0, kHalfRows * half, 0, blk);
  if (kpe_separate) tma_load_3d(stage + 8 * kSlotBytes, tm_kpe, bar, 0, kHalfRows * half, blk);
}
// Latent column blocks {box, box + 1} of rows [32 half, 32 half + 32) into two
// adjacent slots at dst (8 KB; the caller accounts for the bytes on `bar`).
__device__ __forceinline__ void load_pair_box(uint32_t dst, const CUtensorMap* tm_pair, uint32_t bar, int half,
                                              int box, int blk) {
  tma_load_4d(dst, tm_pair, bar, 0, kHalfRows * half, box, blk);
}

struct FastArgs {
  const __nv_bfloat16* q_lat;
  const int32_t* block_table;
  int bt_stride;
  const int32_t* seq_lens;   // length of sequence b: seq_lens[b / seq_div]
  int seq_div;
  int B, T, H, causal, checked, max_pages, num_blocks;
  int max_rows;              // longest length: max_pages * 64, or the sparse decode's topk
  const int32_t* indices;    // sparse decode: physical cache rows [B, topk] (B = sequences x query tokens)
  int topk;
  const __nv_bfloat16* ckv;  // sparse decode: the pool's rows (latent part), row stride ckv_row elements
  const __nv_bfloat16* kpe;  // and their RoPE values, row stride kpe_row
  long long ckv_row, kpe_row;
  int kpe_separate;          // RoPE values not at latent + 512 in the same rows: loaded by their own box
  float scale_log2;          // softmax scale times log2(e)
  __nv_bfloat16* o_lat;
  float* lse;
  WsLayout L;
};

struct Shared {
  uint32_t base;
  __device__ uint32_t q(int box) const { return base + kSmemQ + (box - kQTmemBoxes) * kQBoxBytes; }
  // Where the first segment's query box 0..5 lands (inside ring stages 3, 4).
  __device__ uint32_t q_first(int box) const { return base + kSmemRing + kQStageFirst * kStageBytes + box * kQBoxBytes; }
  __device__ uint32_t p(int buf) const { return base + kSmemP + buf * kPBytes; }
  __device__ uint32_t stage(int st) const { return base + kSmemRing + st * kStageBytes; }
  __device__ uint32_t slot(int st, int s) const { return stage(st) + s * kSlotBytes; }
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

__device__ __forceinline__ void fail(int* hdr, volatile int* abort_flag, int where) {
  *abort_flag = 1;
  record_error(hdr, MLA_ERR_TIMEOUT, where);
}

// A bounded wait taken by every lane of a warp; true only if all lanes saw the
// phase complete (on a timeout lane 0 records it and raises the abort flag).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* hdr,
                                          int where) {
  const bool ok = __all_sync(0xffffffffu, mbar_wait_sleep(bar, parity, abort_flag));
  if (!ok && (threadIdx.x & 31) == 0) fail(hdr, abort_flag, where);
  return ok;
}

// One arrival per warp on a barrier of CTA 0 (local for CTA 0, through the
// cluster window for CTA 1).  What these arrivals order is either in the
// arriving CTA's own shared or tensor memory, read by its own SM's half of the
// pair MMA (P and the query after fence.proxy.async / tcgen05 fences), or a
// read the arriving CTA has finished (score and accumulator loads), so the
// default CTA-scope release suffices; a cluster-scope release was measured to
// cost ~1000 cycles per arrival.
__device__ __forceinline__ void warp_arrive_leader(uint32_t bar, int rank) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    if (rank == 0) mbar_arrive(bar);
    else asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(map_to_cta(bar, 0)) : "memory");
  }
  __syncwarp();
}

// Descriptors.  K-major 128-byte-swizzled tiles: rows of 128 bytes, 8-row atoms
// 1024 bytes apart; a 16-element K step moves the start address by 32 bytes.
// V (B of P V) is N-major: 64-column blocks one slot (LBO) apart, 8-row atoms
// 1024 bytes apart; a 16-row K step moves the start by 2048 bytes.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr) { return sw128_desc(saddr, 16, 1024); }
__device__ __forceinline__ uint64_t vdesc(uint32_t saddr) { return sw128_desc(saddr, kSlotBytes, 1024); }

// What a softmax thread needs to know about one segment.
struct SegRows {
  int b, p0, p1, slot_out, merge_rec, S, fr, limit;
  bool row_valid;
};

__device__ __forceinline__ SegRows seg_rows(const int* rec, const FastArgs& a, int R, int row) {
  SegRows s;
  s.b = rec[0];
  s.p0 = rec[2];
  s.p1 = rec[3];
  s.slot_out = rec[5];
  s.merge_rec = rec[6];
  int S = a.seq_lens[s.b / a.seq_div];
  s.S = S < 0 ? 0 : min(S, a.max_rows);
  s.fr = rec[1] * kRowsPerBlock + row;
  s.row_valid = s.fr < R;
  s.limit = s.row_valid ? visible_limit(s.S, a.T, s.fr / a.H, a.causal) : 0;
  return s;
}

// Block id `blk` of page p of sequence b (read from the table by the caller)
// validated: -1 = outside the pool, reads as zeros.
__device__ __forceinline__ int checked_block(const FastArgs& a, int blk, int b, int p, int* hdr, bool report) {
  if (blk < 0 || blk >= a.num_blocks) {
    if (report && a.checked) record_error(hdr, MLA_ERR_DEVICE_CHECK, (b << 16) | p);
    blk = -1;
  }
  return blk;
}
// Block id of page p of sequence b (-1 = outside the pool, reads as zeros).
__device__ __forceinline__ int page_block(const FastArgs& a, int b, int p, int* hdr, bool report) {
  int blk = a.block_table[(size_t)b * a.bt_stride + p];
  if (blk < 0 || blk >= a.num_blocks) {
    if (report && a.checked) record_error(hdr, MLA_ERR_DEVICE_CHECK, (b << 16) | p);
    blk = -1;
  }
  return blk;
}

// One page of Q K^T as a single issue sequence from one elected lane (36 pair
// MMAs, K = 576 in steps of 16): issuing the 36 MMAs from one asm block, with the
// operand addresses advanced by immediate offsets, was measured to raise the
// page rate over one elect.sync per MMA.  A operand: query boxes 0..5 in tensor
// memory (32 columns per box, 8 per K step), boxes 6..8 in shared memory
// (8 KB apart, 32 bytes per K step); B operand: the stage's nine 4 KB slots
// (descriptor units of 16 bytes: 256 per slot, 2 per K step).  The first MMA
// overwrites the score tile.
#define QK_TS(AOFF, BOFF)                                                  \
  "add.u32 aq, %1, " #AOFF ";\n\tadd.u64 bq, %2, " #BOFF ";\n\t"        \
  "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [aq], bq, %3, t;\n\t"
#define QK_SS(AOFF, BOFF)                                                  \
  "add.u64 as, %4, " #AOFF ";\n\tadd.u64 bq, %2, " #BOFF ";\n\t"        \
  "@e tcgen05.mma.cta_group::2.kind::f16 [%0], as, bq, %3, t;\n\t"
__device__ __forceinline__ void qk_page_e(uint32_t d_tmem, uint32_t q_tmem, uint64_t b_desc0, uint32_t idesc,
                                          uint64_t q_smem_desc0) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t.reg .b64 bq, as;\n\t.reg .b32 aq;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.eq.b32 p, 1, 0;\n\t"
      "setp.eq.b32 t, 1, 1;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      QK_TS(8, 2)
      QK_TS(16, 4)
      QK_TS(24, 6)
      QK_TS(32, 256)
      QK_TS(40, 258)
      QK_TS(48, 260)
      QK_TS(56, 262)
      QK_TS(64, 512)
      QK_TS(72, 514)
      QK_TS(80, 516)
      QK_TS(88, 518)
      QK_TS(96, 768)
      QK_TS(104, 770)
      QK_TS(112, 772)
      QK_TS(120, 774)
      QK_TS(128, 1024)
      QK_TS(136, 1026)
      QK_TS(144, 1028)
      QK_TS(152, 1030)
      QK_TS(160, 1280)
      QK_TS(168, 1282)
      QK_TS(176, 1284)
      QK_TS(184, 1286)
      QK_SS(0, 1536)
      QK_SS(2, 1538)
      QK_SS(4, 1540)
      QK_SS(6, 1542)
      QK_SS(512, 1792)
      QK_SS(514, 1794)
      QK_SS(516, 1796)
      QK_SS(518, 1798)
      QK_SS(1024, 2048)
      QK_SS(1026, 2050)
      QK_SS(1028, 2052)
      QK_SS(1030, 2054)
      "}" ::"r"(d_tmem), "r"(q_tmem), "l"(b_desc0), "r"(idesc), "l"(q_smem_desc0)
      : "memory");
}
#undef QK_TS
#undef QK_SS

// One page of P V the same way (8 pair MMAs, N = 256: two 256-column halves of
// the accumulator, K = 64 page rows in steps of 16).  A: P (K-major, 32 bytes
// per K step); B: V, N-major, latent column block pairs {4m, 4m+1} for rows
// 0..31 (steps 0, 1: 2 KB apart) and {4m+2, 4m+3} for rows 32..63.  The first
// MMA of each half accumulates only when `accumulate` != 0.
#define PV_SS(D, AOFF, BOFF, PRED)                                          \
  "add.u64 ap, %1, " #AOFF ";\n\tadd.u64 bv, %2, " #BOFF ";\n\t"         \
  "@e tcgen05.mma.cta_group::2.kind::f16 [" #D "], ap, bv, %3, " #PRED ";\n\t"
__device__ __forceinline__ void pv_page_e(uint32_t o_tmem, uint64_t p_desc0, uint64_t v_desc0, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t.reg .b64 ap, bv;\n\t.reg .b32 d1;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 1, 1;\n\t"
      "add.u32 d1, %0, 128;\n\t"
      PV_SS(%0, 0, 0, p)
      PV_SS(%0, 2, 128, t)
      PV_SS(%0, 4, 512, t)
      PV_SS(%0, 6, 640, t)
      PV_SS(d1, 0, 1024, p)
      PV_SS(d1, 2, 1152, t)
      PV_SS(d1, 4, 1536, t)
      PV_SS(d1, 6, 1664, t)
      "}" ::"r"(o_tmem), "l"(p_desc0), "l"(v_desc0), "r"(idesc), "r"(accumulate)
      : "memory");
}
#undef PV_SS

// ---------------------------------------------------------------- sparse (index-driven) loads
// "M5.8" 0x0B: sparse indices are physical cache rows (block * 64 + offset).  A
// sparse decode's "page" p of a (sequence, query token) is listed rows
// 64 p .. 64 p + 63; its half for CTA r is rows 64 p + 32 r .. + 31.  A whole
// warp copies them with cp.async, 16 bytes per lane per copy, straight into the
// 128-byte-swizzled slots a page half fills (eight lanes cover one 128-byte
// piece of a row, so every copy instruction reads four rows' contiguous
// pieces); list entries at or past the list's length, and rows outside the
// pool, are zero-filled (and masked like the rows past a sequence's end).  The
// writing warp waits for its own copies, makes them visible to the tensor
// cores (fence.proxy.async) and then arrives on the stage's barrier.

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory"); }

// The physical row of list entry e of (virtual) sequence b whose list holds S
// valid entries, or -1 (past the length, or outside the pool: reported in
// checked mode when `report`).
__device__ __forceinline__ int sparse_row(const FastArgs& a, int b, int e, int S, int* hdr, bool report) {
  if (e >= S) return -1;
  const int v = __ldg(a.indices + (size_t)b * a.topk + e);
  if (v < 0 || v >= a.num_blocks * kPage) {
    if (report && a.checked) record_error(hdr, MLA_ERR_DEVICE_CHECK, (b << 16) | (e & 0xFFFF));
    return -1;
  }
  return v;
}

// Warp-wide: the 32 rows whose physical rows the lanes hold (lane i: row i of the
// page half, v = -1 for a zero row), latent column block box[k] (8 = the RoPE
// values) into slot slot[k] of the stage, k < kN.
template <int kN>
__device__ __forceinline__ void sparse_copy(uint32_t stage, const FastArgs& a, int v, int lane, const int (&box)[kN],
                                            const int (&slot)[kN]) {
  const int c = lane & 7;
#pragma unroll 1   // (unrolled, the copy code measured ~2 % slower: instruction fetch)
  for (int q = 0; q < 8; ++q) {
    const int r = (lane >> 3) + 4 * q;
    const int rv = __shfl_sync(0xffffffffu, v, r);
    const bool valid = rv >= 0;
    const __nv_bfloat16* lat = a.ckv + (valid ? (long long)rv * a.ckv_row : 0);
    const __nv_bfloat16* rope = a.kpe + (valid ? (long long)rv * a.kpe_row : 0);
    const uint32_t dst_row = stage + r * 128 + 16 * (c ^ (r & 7));
#pragma unroll
    for (int k = 0; k < kN; ++k) {
      const __nv_bfloat16* src = (box[k] < 8 ? lat + 64 * box[k] : rope) + 8 * c;
      cp_async16(dst_row + slot[k] * kSlotBytes, src, valid);
    }
  }
}

// Completion of the oldest pages a warp copied: each lane waits for its copy
// groups but the kKeep most recent, makes them visible to the async proxy, and
// lane 0 arrives on the barriers of the pages that completed.
template <int kKeep>
__device__ __forceinline__ void sparse_complete(const Shared& sh, int bar0, int& done, int issued, int lane) {
  if (issued - done <= kKeep) return;
  if (kKeep == 0) cp_async_wait<0>();
  else cp_async_wait<kKeep>();
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0)
    for (int g = done; g < issued - kKeep; ++g) mbar_arrive(sh.bar(bar0 + g % kStages));
  __syncwarp();
  done = issued - kKeep;
}

// Sparse mode, warp 3: the query loads (lane 0) and the page halves (all lanes).
// A page's barrier is signalled once two later pages are in flight; at a
// segment's end every page is completed first (the next segment's query waits
// for the last Q K^T of this one, which needs those pages).
__device__ __forceinline__ void sparse_gather_role(const Shared& sh, const CUtensorMap* tm_qlat,
                                                   const CUtensorMap* tm_qpe, const FastArgs& a, int* hdr,
                                                   volatile int* abort_flag, const int* seg, SegWalk walk, int rank,
                                                   int R, int lane) {
  // A page's barrier is signalled once kInFlight later pages are issued.  Issuing
  // page g waits for P V of page g - kStages, which needs the reload of that page,
  // which the reload warp signals after Q K^T of the next page, which needs page
  // g - kStages + 1's barrier: so kInFlight <= kStages - 2.
  constexpr int kInFlight = 2;
  static_assert(kInFlight <= kStages - 2, "the gather must signal a page before it waits for that page's P V");
  const int box[9] = {0, 1, 2, 3, 4, 5, 6, 7, 8};
  int gt = 0, done = 0, sc = 0;
  bool ok = true, q_in_flight = false;
  for (int si = walk.cur(); ok && si >= 0; walk.advance(), si = walk.cur()) {
    const int* rec = seg + (size_t)si * kSegWords;
    const int b = rec[0], rb = rec[1], p0 = rec[2], p1 = rec[3];
    sparse_complete<0>(sh, BAR_FULL, done, gt, lane);
    if (sc > 0 && !warp_wait(sh.bar(BAR_Q_FREE), (sc - 1) & 1, abort_flag, hdr, 10)) { ok = false; break; }
    if (lane == 0) {
      const int row0 = b * R + rb * kRowsPerBlock + kCtaRows * rank;
      mbar_arrive_expect_tx(sh.bar(BAR_Q_TMA), (sc == 0 ? kBoxes : kQSmemBoxes) * kQBoxBytes);
      if (sc == 0)
        for (int qb = 0; qb < kQTmemBoxes; ++qb) tma_load_2d(sh.q_first(qb), tm_qlat, sh.bar(BAR_Q_TMA), 64 * qb, row0);
      for (int qb = kQTmemBoxes; qb < 8; ++qb) tma_load_2d(sh.q(qb), tm_qlat, sh.bar(BAR_Q_TMA), 64 * qb, row0);
      tma_load_2d(sh.q(8), tm_qpe, sh.bar(BAR_Q_TMA), 0, row0);
    }
    __syncwarp();
    q_in_flight = true;
    int S = a.seq_lens[b / a.seq_div];
    S = S < 0 ? 0 : min(S, a.max_rows);
    // the list entries of the next two pages are loaded ahead (a dependent load
    // at the head of every page otherwise paces the warp)
    int v_next[2];
#pragma unroll
    for (int k = 0; k < 2; ++k)
      v_next[k] = p0 + k < p1 ? sparse_row(a, b, (p0 + k) * kPage + kHalfRows * rank + lane, S, hdr, true) : -1;
    for (int p = p0; ok && p < p1; ++p, ++gt) {
      const int v = v_next[0];
      v_next[0] = v_next[1];
      v_next[1] = p + 2 < p1 ? sparse_row(a, b, (p + 2) * kPage + kHalfRows * rank + lane, S, hdr, true) : -1;
      const int st = gt % kStages;
      if (gt >= kStages && !warp_wait(sh.bar(BAR_PV_DONE + st), ((gt / kStages) - 1) & 1, abort_flag, hdr, 11)) {
        ok = false; break;
      }
      if (gt >= kQStageFirst && gt < kStages && !warp_wait(sh.bar(BAR_Q_COPIED), 0, abort_flag, hdr, 15)) {
        ok = false; break;
      }
      sparse_copy<9>(sh.stage(st), a, v, lane, box, box);
      cp_async_commit();
      sparse_complete<kInFlight>(sh, BAR_FULL, done, gt + 1, lane);
    }
    ++sc;
  }
  // Drain: every copy must have landed before the CTA may exit (signalled too
  // when nothing failed), and the last query load.
  if (ok) sparse_complete<0>(sh, BAR_FULL, done, gt, lane);
  else cp_async_wait<0>();
  if (q_in_flight && lane == 0) mbar_wait_drain(sh.bar(BAR_Q_TMA), (sc - 1) & 1);
  __syncwarp();
}

// Sparse mode, warp 0: the other half's rows of this CTA's P V boxes, once Q K^T
// is done with the page; a page's reload is signalled once the next one is in
// flight, and at a segment's end at once (the softmax waits for it there).
__device__ __forceinline__ void sparse_reload_role(const Shared& sh, const FastArgs& a, int* hdr,
                                                   volatile int* abort_flag, const int* seg, SegWalk walk, int rank,
                                                   int lane) {
  const int box[4] = {own_pv_box(rank, 0), own_pv_box(rank, 1), own_pv_box(rank, 2), own_pv_box(rank, 3)};
  const int slot[4] = {reload_slot(rank, 0), reload_slot(rank, 1), reload_slot(rank, 2), reload_slot(rank, 3)};
  int gt = 0, done = 0;
  bool ok = true;
  for (int si = walk.cur(); ok && si >= 0; walk.advance(), si = walk.cur()) {
    const int* rec = seg + (size_t)si * kSegWords;
    const int b = rec[0];
    int S = a.seq_lens[b / a.seq_div];
    S = S < 0 ? 0 : min(S, a.max_rows);
    const int p1 = rec[3];
    int v_next = rec[2] < p1 ? sparse_row(a, b, rec[2] * kPage + kHalfRows * (1 - rank) + lane, S, hdr, false) : -1;
    for (int p = rec[2]; ok && p < p1; ++p, ++gt) {
      const int v = v_next;
      v_next = p + 1 < p1 ? sparse_row(a, b, (p + 1) * kPage + kHalfRows * (1 - rank) + lane, S, hdr, false) : -1;
      const int st = gt % kStages;
      if (!warp_wait(sh.bar(BAR_QK_DONE + st), (gt / kStages) & 1, abort_flag, hdr, 13)) { ok = false; break; }
      sparse_copy<4>(sh.stage(st), a, v, lane, box, slot);
      cp_async_commit();
      sparse_complete<1>(sh, BAR_RELOAD, done, gt + 1, lane);
    }
    if (ok) sparse_complete<0>(sh, BAR_RELOAD, done, gt, lane);
  }
  if (!ok) cp_async_wait<0>();
  __syncwarp();
}

// ---------------------------------------------------------------- FP8 656-byte rows
// "M5.8" 0x0B "Exact 656-byte FP8 row": a cached row is 512 E4M3 latent codes,
// 4 fp32 scales (scale t for latent values [128 t, 128 t + 128)) and 64 bf16
// RoPE values; value = E4M3(code) * scale.  The pool is one 2-D byte array of
// rows (block * 64 + offset, 656 bytes each).  A page half lands by TMA as:
// codes [128 t, 128 t + 128) of the 32 rows (128 bytes per row) in slot 2 t + 1;
// the RoPE values straight into slot 8 (a bf16 map over the rows' last 128
// bytes, 128-byte swizzled like a bf16 page); the scales into a small ring of
// their own.  Converter thread (row rho, tile t) reads its 128 codes from row
// rho of slot 2 t + 1 and writes them as bf16 (the dequantised value rounded
// to nearest, the MMA operand type) to row rho of slots 2 t and 2 t + 1: no
// thread overwrites another's input, so no barrier is needed between them.
// After Q K^T the other half's codes of this CTA's P V boxes land in Q K^T-only
// slot reload_slot(rank, 2 m + 1) (m = 0, 1) and their scales in slot 8 (no
// longer read), and are converted into reload_slot(rank, 2 m), +1 the same way.
constexpr int kFp8Row = 656;
constexpr int kRawHalfBytes = kHalfRows * kFp8Row;                         // 20992
constexpr int kRawReloadBytes = 2 * kHalfRows * 128 + kHalfRows * 16;    // 8704
// The reload of page g - kReloadLag is converted after page g's own rows: the
// reload's L2 round trip then overlaps a page's conversion (1 measured faster
// than 2 or 3; any lag up to kStages - 1 keeps the ring free of a wait cycle).
constexpr int kReloadLag = 1;

// Rows [y, y + 32) of the FP8 pool (y < 0: a block outside the pool, read as
// zeros) into a stage and its scale entry.
__device__ __forceinline__ void fp8_load_half(uint32_t stage, uint32_t scales, const CUtensorMap* tm128,
                                              const CUtensorMap* tm_rope, const CUtensorMap* tm16, uint32_t bar,
                                              int y) {
  mbar_arrive_expect_tx(bar, kRawHalfBytes);
  for (int t = 0; t < 4; ++t) tma_load_2d(stage + (2 * t + 1) * kSlotBytes, tm128, bar, 128 * t, y);
  tma_load_2d(stage + 8 * kSlotBytes, tm_rope, bar, 0, y);
  tma_load_2d(scales, tm16, bar, 512, y);
}
// The other half's rows [y, y + 32): codes of this CTA's P V latent columns
// [256 m + 128 rank, +128) into slot reload_slot(rank, 2 m + 1), scales into slot 8.
__device__ __forceinline__ void fp8_load_reload(uint32_t stage, const CUtensorMap* tm128, const CUtensorMap* tm16,
                                                uint32_t bar, int y, int rank) {
  mbar_arrive_expect_tx(bar, kRawReloadBytes);
  for (int m = 0; m < 2; ++m)
    tma_load_2d(stage + reload_slot(rank, 2 * m + 1) * kSlotBytes, tm128, bar, 256 * m + 128 * rank, y);
  tma_load_2d(stage + 8 * kSlotBytes, tm16, bar, 512, y);
}

// Four E4M3 codes (the lowest byte first) times the tile's scale, as two bf16
// pairs: each code is widened exactly (to f16 by the E4M3 conversion, two codes
// per instruction, to fp32 by a mixed-precision multiply-add with 1), each pair
// multiplied by the fp32 scale in one packed multiply (each lane rounded to
// nearest, as two scalar multiplies), and the products rounded to bf16
// (measured faster than building the fp32 bits with integer operations).
// scale2: the scale in both halves.
__device__ __forceinline__ uint2 dequant4(uint32_t four, uint64_t scale2) {
  uint2 r;
  asm("{\n\t.reg .b16 c0, c1, l0, u0, l1, u1, one;\n\t.reg .b32 h0, h1;\n\t.reg .f32 a0, b0, a1, b1;\n\t"
      ".reg .b64 p0, p1;\n\t"
      "mov.b16 one, 0x3C00;\n\t"
      "mov.b32 {c0, c1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 h0, c0;\n\t"
      "cvt.rn.f16x2.e4m3x2 h1, c1;\n\t"
      "mov.b32 {l0, u0}, h0;\n\t"
      "mov.b32 {l1, u1}, h1;\n\t"
      "fma.rn.f32.f16 a0, l0, one, 0f00000000;\n\t"
      "fma.rn.f32.f16 b0, u0, one, 0f00000000;\n\t"
      "fma.rn.f32.f16 a1, l1, one, 0f00000000;\n\t"
      "fma.rn.f32.f16 b1, u1, one, 0f00000000;\n\t"
      "mov.b64 p0, {a0, b0};\n\t"
      "mov.b64 p1, {a1, b1};\n\t"
      "mul.rn.f32x2 p0, p0, %3;\n\t"
      "mul.rn.f32x2 p1, p1, %3;\n\t"
      "mov.b64 {a0, b0}, p0;\n\t"
      "mov.b64 {a1, b1}, p1;\n\t"
      "cvt.rn.bf16x2.f32 %0, b0, a0;\n\t"
      "cvt.rn.bf16x2.f32 %1, b1, a1;\n\t}"
      : "=r"(r.x), "=r"(r.y)
      : "r"(four), "l"(scale2));
  return r;
}
__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// 16 codes times the tile's scale, as bf16: output chunks oc and oc + 1 (8 values
// each; oc even) of the 128-byte-swizzled slot row at row_base (row `row`).
__device__ __forceinline__ void dequant_store16(uint4 code, float scale_f, uint32_t row_base, int oc, int row) {
  const uint64_t scale = ((uint64_t)__float_as_uint(scale_f) << 32) | __float_as_uint(scale_f);
  const int sw = row & 7;
  const uint2 x = dequant4(code.x, scale), y = dequant4(code.y, scale);
  const uint2 z = dequant4(code.z, scale), w = dequant4(code.w, scale);
  st_shared_u4(row_base + 16 * (oc ^ sw), make_uint4(x.x, x.y, y.x, y.y));
  st_shared_u4(row_base + 16 * ((oc + 1) ^ sw), make_uint4(z.x, z.y, w.x, w.y));
}

// Converter warps (warps 12..15; t = 0..127): page g's own half as soon as its raw
// rows land, then the reload of page g - kReloadLag.
__device__ __forceinline__ void fp8_convert_role(const Shared& sh, int* hdr, volatile int* abort_flag, const int* seg,
                                                 SegWalk walk, int rank, int t) {
  const int lane = t & 31, rho = t >> 2, q = t & 3;
  // own half: thread (rho, tile q); reload: thread (rho, m = q >> 1, half h = q & 1)
  const int m = q >> 1, h = q & 1;
  const int tile_rl = own_pv_box(rank, 2 * m) >> 1;
  // Shared-memory access order: lane L takes its 16-byte chunks in a rotated order
  // (own: chunk c ^ (L % 8); reload: (c + rot) % 4), so that any eight consecutive
  // lanes touch eight different 16-byte bank groups in every load and store.
  const int own_k = lane & 7;
  const int rl_rot = (m + 2 * h + 2 * (rho & 1)) & 3;
  auto own = [&](int g) -> bool {
    const int st = g % kStages;
    if (!__all_sync(0xffffffffu, mbar_wait(sh.bar(BAR_RAW + st), (g / kStages) & 1, abort_flag))) return false;
    const uint32_t stage = sh.stage(st);
    const uint32_t src = stage + (2 * q + 1) * kSlotBytes + rho * 128;
    uint4 code[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) code[c] = ld_shared_u4(src + 16 * (c ^ own_k));
    const float ts = ld_shared_f32(sh.base + kSmemScales + st * 512 + rho * 16 + 4 * q);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int ci = c ^ own_k;   // codes [16 ci, 16 ci + 16) of the tile: slot 2 q + ci / 4, chunks 2 ci % 8, +1
      dequant_store16(code[c], ts, stage + (2 * q + (ci >> 2)) * kSlotBytes + rho * 128, (2 * ci) & 7, rho);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(sh.bar(BAR_FULL + st));
    return true;
  };
  auto reload = [&](int g) -> bool {
    const int st = g % kStages;
    if (!__all_sync(0xffffffffu, mbar_wait(sh.bar(BAR_RLRAW + st), (g / kStages) & 1, abort_flag))) return false;
    const uint32_t stage = sh.stage(st);
    const uint32_t src = stage + reload_slot(rank, 2 * m + 1) * kSlotBytes + rho * 128 + 64 * h;
    uint4 code[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) code[c] = ld_shared_u4(src + 16 * ((c + rl_rot) & 3));
    const float ts = ld_shared_f32(stage + 8 * kSlotBytes + rho * 16 + 4 * tile_rl);
    __syncwarp();   // the lane of half 1 overwrites the raw row its half-0 neighbour reads
    const uint32_t dst = stage + reload_slot(rank, 2 * m + h) * kSlotBytes + rho * 128;
#pragma unroll
    for (int c = 0; c < 4; ++c) dequant_store16(code[c], ts, dst, 2 * ((c + rl_rot) & 3), rho);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(sh.bar(BAR_RELOAD + st));
    return true;
  };
  int g = 0;
  bool ok = true;
  for (int si = walk.cur(); ok && si >= 0; walk.advance(), si = walk.cur()) {
    const int* rec = seg + (size_t)si * kSegWords;
    for (int p = rec[2]; p < rec[3]; ++p, ++g) {
      if (!own(g) || (g >= kReloadLag && !reload(g - kReloadLag))) { ok = false; break; }
    }
  }
  for (int r = g > kReloadLag ? g - kReloadLag : 0; ok && r < g; ++r) ok = reload(r);
  if (!ok && lane == 0) fail(hdr, abort_flag, 40);
}

// Q K^T issuer (CTA 0, one converged warp): page t goes to score tile t % 2
// once both CTAs' halves of the page have landed (CTA 0's load barrier also
// counts CTA 1's, relayed) and both softmaxes have read the tile's previous
// scores (page t - 2).
__device__ __forceinline__ void qk_role(const Shared& sh, uint32_t tmem, int* hdr, volatile int* abort_flag,
                                        const int* seg, SegWalk walk) {
  const uint32_t id_qk = idesc_bf16_f32(128, 64, 0);
  const uint64_t qdesc0 = kmajor_desc(sh.q(kQTmemBoxes));
  int gt = 0, sc = 0;
  bool ok = true;
  for (int si = walk.cur(); ok && si >= 0; walk.advance(), si = walk.cur()) {
    const int* rec = seg + (size_t)si * kSegWords;
    const int n_tiles = rec[3] - rec[2];
    if (!warp_wait(sh.bar(BAR_Q_READY), sc & 1, abort_flag, hdr, 22)) { ok = false; break; }
    tc_fence_after();
    for (int i = 0; ok && i < n_tiles; ++i, ++gt) {
      const int st = gt % kStages, sb = gt & 1;
      const uint32_t par = (gt / kStages) & 1;
      if (!warp_wait(sh.bar(BAR_FULL + st), par, abort_flag, hdr, 23) ||
          (gt >= 2 && !warp_wait(sh.bar(BAR_S_FREE + sb), ((gt >> 1) - 1) & 1, abort_flag, hdr, 25))) {
        ok = false; break;
      }
      tc_fence_after();
      qk_page_e(tmem + kTmemS + 32 * sb, tmem + kTmemQ, kmajor_desc(sh.slot(st, 0)), id_qk, qdesc0);
      commit2_both_e(sh.bar(BAR_S_FULL + sb));
      commit2_both_e(sh.bar(BAR_QK_DONE + st));
      if (i == n_tiles - 1) commit2_both_e(sh.bar(BAR_Q_FREE));
    }
    ++sc;
  }
  // Every MMA issued by this warp must be complete before the CTAs may leave.
  commit2_both_e(sh.bar(BAR_FINAL_QK));
  mbar_wait_drain(sh.bar(BAR_FINAL_QK), 0);
  __syncwarp();
}

// P V issuer (CTA 0, one converged warp): O += P V for page t once both CTAs
// wrote P and both CTAs' reloads of the other half's rows landed (CTA 0's
// reload barrier also counts CTA 1's, relayed); the first
// page of a segment overwrites O, after the previous segment's epilogue.
__device__ __forceinline__ void pv_role(const Shared& sh, uint32_t tmem, int* hdr, volatile int* abort_flag,
                                        const int* seg, SegWalk walk) {
  const uint32_t id_pv = idesc_bf16_f32(128, 256, 1);
  int gv = 0, sc = 0;
  bool ok = true;
  for (int si = walk.cur(); ok && si >= 0; walk.advance(), si = walk.cur()) {
    const int* rec = seg + (size_t)si * kSegWords;
    const int n_tiles = rec[3] - rec[2];
    for (int i = 0; ok && i < n_tiles; ++i, ++gv) {
      const int st = gv % kStages, pb = gv % kPBufs;
      const uint32_t par = (gv / kStages) & 1;
      if ((i == 0 && sc > 0 && !warp_wait(sh.bar(BAR_O_FREE), (sc - 1) & 1, abort_flag, hdr, 20)) ||
          !warp_wait(sh.bar(BAR_RELOAD + st), par, abort_flag, hdr, 26) ||
          !warp_wait(sh.bar(BAR_P_FULL + pb), (gv / kPBufs) & 1, abort_flag, hdr, 21)) {
        ok = false; break;
      }
      tc_fence_after();
      pv_page_e(tmem + kTmemO, kmajor_desc(sh.p(pb)), vdesc(sh.slot(st, 0)), id_pv, i == 0 ? 0u : 1u);
      commit2_both_e(sh.bar(BAR_PV_DONE + st));
    }
    ++sc;
  }
  commit2_both_e(sh.bar(BAR_FINAL_PV));
  mbar_wait_drain(sh.bar(BAR_FINAL_PV), 0);
  __syncwarp();
}

// CTA 1: forward the completion of a per-page local barrier (its page half or
// its reload) to the matching barrier of CTA 0, page by page.
__device__ __forceinline__ void relay_role(const Shared& sh, int* hdr, volatile int* abort_flag, const int* seg,
                                           SegWalk walk, int from, int to, int where) {
  const uint32_t dst0 = map_to_cta(sh.bar(to), 0);
  int gt = 0;
  bool ok = true;
  for (int si = walk.cur(); ok && si >= 0; walk.advance(), si = walk.cur()) {
    const int* rec = seg + (size_t)si * kSegWords;
    for (int p = rec[2]; p < rec[3]; ++p, ++gt) {
      const int st = gt % kStages;
      if (!mbar_wait_sleep(sh.bar(from + st), (gt / kStages) & 1, abort_flag)) {
        fail(hdr, abort_flag, where); ok = false; break;
      }
      asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(dst0 + 8 * st) : "memory");
    }
  }
}

// Reloads of the other half's rows (one thread): once Q K^T is done with a page,
// the slots that held this CTA's Q K^T-only latent boxes receive the other page
// half's rows of the boxes this CTA accumulates (two 2-block boxes, L2 hits:
// the partner CTA fetched them from HBM).
// (FP8 rows: the raw codes and scales, by tm_pair and tm_aux, for the converter
// warps.  The sparse decode reloads with a whole warp: sparse_reload_role.)
template <int kMode>
__device__ __forceinline__ void reload_role(const Shared& sh, const CUtensorMap* tm_pair, const CUtensorMap* tm_aux,
                                            const FastArgs& a, int* hdr, volatile int* abort_flag, const int* seg,
                                            SegWalk walk, int rank) {
  const int landed = kMode == kModeFp8 ? BAR_RLRAW : BAR_RELOAD;
  int gt = 0;
  bool ok = true;
  for (int si = walk.cur(); ok && si >= 0; walk.advance(), si = walk.cur()) {
    const int* rec = seg + (size_t)si * kSegWords;
    const int b = rec[0];
    for (int p = rec[2]; ok && p < rec[3]; ++p, ++gt) {
      const int st = gt % kStages;
      if constexpr (kMode == kModeFp8) {
        const int blk = page_block(a, b, p, hdr, false);
        if (!mbar_wait_sleep(sh.bar(BAR_QK_DONE + st), (gt / kStages) & 1, abort_flag)) {
          fail(hdr, abort_flag, 13); ok = false; break;
        }
        fp8_load_reload(sh.stage(st), tm_pair, tm_aux, sh.bar(BAR_RLRAW + st),
                        blk >= 0 ? blk * kPage + kHalfRows * (1 - rank) : -kPage, rank);
      } else {
        const int blk = page_block(a, b, p, hdr, false);
        if (!mbar_wait_sleep(sh.bar(BAR_QK_DONE + st), (gt / kStages) & 1, abort_flag)) {
          fail(hdr, abort_flag, 13); ok = false; break;
        }
        // Two 2-block boxes: latent boxes {2r, 2r+1} and {4+2r, 5+2r} of the other half.
        mbar_arrive_expect_tx(sh.bar(BAR_RELOAD + st), 4 * kSlotBytes);
        for (int i = 0; i < 4; i += 2)
          load_pair_box(sh.slot(st, reload_slot(rank, i)), tm_pair, sh.bar(BAR_RELOAD + st), 1 - rank,
                        own_pv_box(rank, i), blk);
      }
    }
  }
  // Drain: every reload issued must have landed before the CTA may exit.
  const int first = gt > kStages ? gt - kStages : 0;
  for (int g = first; g < gt; ++g) {
    mbar_wait_drain(sh.bar(landed + g % kStages), (g / kStages) & 1);
  }
}

// kMode == kModeSparse: the sparse (index-driven) decode; tm_page is then the
// pool as a 2-D array of rows (the latent part when the RoPE values are
// separate, tm_kpe the RoPE part), tm_pair unused.  kMode == kModeFp8: the FP8
// pool as a 2-D byte array of 656-byte rows, through boxes 128 (tm_pair) and 16
// (tm_aux) bytes wide, 32 rows high, and tm_kpe the rows' RoPE values as bf16
// (64 x 32 boxes, 128-byte swizzled); tm_page unused.  tm_aux is unused by the
// other modes.
template <int kMode>
__global__ void __launch_bounds__(threads_of<kMode>(), 1)
    decode_sm103_kernel(const __grid_constant__ CUtensorMap tm_qlat, const __grid_constant__ CUtensorMap tm_qpe,
                        const __grid_constant__ CUtensorMap tm_page, const __grid_constant__ CUtensorMap tm_pair,
                        const __grid_constant__ CUtensorMap tm_kpe, const __grid_constant__ CUtensorMap tm_aux,
                        FastArgs a, char* ws) {
  constexpr bool kSparse = kMode == kModeSparse;
  constexpr bool kFp8 = kMode == kModeFp8;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* hdr = reinterpret_cast<int*>(ws);
  // The 128-byte-swizzled tiles need a 1024-byte-aligned base, at the same offset
  // in both CTAs (pair MMAs address both with one descriptor).  Refuse (uniformly,
  // before anything is set up) if the slack does not cover the misalignment.
  if ((uintptr_t)(smem - smem_raw) + kSmemBytes > (uintptr_t)kSmemAlloc) {
    pdl_wait();
    if (threadIdx.x == 0) record_error(hdr, MLA_ERR_DEVICE_CHECK, -2);
    return;
  }
  Shared sh{smem_addr(smem)};
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + kSmemBar + kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemBar + kNumBars * 8 + 4);
  volatile int* s_num_merge = reinterpret_cast<volatile int*>(smem + kSmemBar + kNumBars * 8 + 8);
  volatile int* s_merge_ok = reinterpret_cast<volatile int*>(smem + kSmemBar + kNumBars * 8 + 12);

  const int* seg = reinterpret_cast<const int*>(ws + a.L.off_segments);
  const int* rptr = reinterpret_cast<const int*>(ws + a.L.off_range_ptr);
  float* part_lse = reinterpret_cast<float*>(ws + a.L.off_part_lse);
  float* part_o = reinterpret_cast<float*>(ws + a.L.off_part_o);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  const int R = a.T * a.H;

  // The plan lines this pair reads first (its range pointers, the record of its
  // first segment when that is segment `pair`, as in plans of one segment per
  // range, and the header) go to the L2 while the previous grid finishes: after
  // a launch that streamed the cache through the L2 they are usually cold.
  if (tid == 96 && pair < a.L.cap_ranges) {
    prefetch_l2_line(rptr + pair);
    prefetch_l2_line(seg + (size_t)min(pair, a.L.cap_segments - 1) * kSegWords);
    prefetch_l2_line(hdr);
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      // CTA 0's load barriers also count the arrival relayed from CTA 1; in the FP8
      // mode the local arrivals are the converter warps' (one each).
      const int local = kFp8 ? 4 : 1;
      mbar_init(sh.bar(BAR_FULL + i), local + (rank == 0 ? 1 : 0));
      mbar_init(sh.bar(BAR_RELOAD + i), local + (rank == 0 ? 1 : 0));
      mbar_init(sh.bar(BAR_RAW + i), 1);
      mbar_init(sh.bar(BAR_RLRAW + i), 1);
      mbar_init(sh.bar(BAR_QK_DONE + i), 1);
      mbar_init(sh.bar(BAR_PV_DONE + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sh.bar(BAR_S_FULL + i), 1);
      mbar_init(sh.bar(BAR_S_FREE + i), 16);
      mbar_init(sh.bar(BAR_XCH + i), 4);
    }
    for (int i = 0; i < kPBufs; ++i) mbar_init(sh.bar(BAR_P_FULL + i), 16);
    mbar_init(sh.bar(BAR_Q_TMA), 1);
    mbar_init(sh.bar(BAR_Q_COPIED), 8);
    mbar_init(sh.bar(BAR_Q_READY), 16);
    mbar_init(sh.bar(BAR_Q_FREE), 1);
    mbar_init(sh.bar(BAR_O_FREE), 16);
    mbar_init(sh.bar(BAR_FINAL_QK), 1);
    mbar_init(sh.bar(BAR_FINAL_PV), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_qlat);
    prefetch_tmap(&tm_qpe);
    prefetch_tmap(&tm_page);
    prefetch_tmap(&tm_pair);
    if (a.kpe_separate || kFp8) prefetch_tmap(&tm_kpe);
    if (kFp8) prefetch_tmap(&tm_aux);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_base_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  pdl_wait();
  // Let the merge pass launch now: its CTAs cannot share an SM with this kernel's
  // (shared memory), so they take idle SMs and those this grid frees, and wait
  // there for this grid to finish instead of paying their launch after it.
  pdl_trigger();
  // The merge count is needed only after the roles: thread 0 (a loader) keeps the
  // load in flight and stores it at the end, off its first page's critical path.
  int num_merge_ld = 0;
  if (tid == 0) asm volatile("ld.global.b32 %0, [%1];" : "=r"(num_merge_ld) : "l"(hdr + MLA_HDR_NUM_MERGE) : "memory");
  // The planner fills the range pointers up to the capacity (empty ranges past the
  // last), so the walk needs no range count from the header.
  const SegWalk walk0(rptr, pair, num_pairs, a.L.cap_ranges);

  if (a.checked && blockIdx.x == 0 && tid == 0) {
    if (hdr[MLA_HDR_MAGIC] != MLA_PLAN_MAGIC || hdr[MLA_HDR_B] != a.B || hdr[MLA_HDR_T] != a.T ||
        hdr[MLA_HDR_H] != a.H || hdr[MLA_HDR_CAUSAL] != a.causal) {
      record_error(hdr, MLA_ERR_PLAN_STALE, 0);
    } else {
      unsigned h = 0;
      for (int b = 0; b < a.B; ++b) {
        unsigned S = (unsigned)a.seq_lens[b / a.seq_div];
        unsigned x = (unsigned)b + 0x632BE5ABu;
        x ^= x >> 16; x *= 0x7feb352dU; x ^= x >> 15; x *= 0x846ca68bU; x ^= x >> 16;
        unsigned y = S * 0x9E3779B1u + x;
        y ^= y >> 16; y *= 0x7feb352dU; y ^= y >> 15; y *= 0x846ca68bU; y ^= y >> 16;
        h += y;
      }
      if ((int)h != hdr[MLA_HDR_SEQ_HASH]) record_error(hdr, MLA_ERR_PLAN_STALE, 1);
    }
  }

  if (kSparse && warp == 0) {
    // ------------------------------------------------------------ sparse: the other half's rows (whole warp)
    sparse_reload_role(sh, a, hdr, abort_flag, seg, walk0, rank, lane);
  } else if (kSparse && warp == 3) {
    // ------------------------------------------------------------ sparse: query and listed rows (whole warp)
    sparse_gather_role(sh, &tm_qlat, &tm_qpe, a, hdr, abort_flag, seg, walk0, rank, R, lane);
  } else if (warp == 0) {
    // ------------------------------------------------------------ page-half and query loads
    if (lane == 0) {
      SegWalk walk = walk0;
      int gt = 0, sc = 0;
      bool ok = true, q_in_flight = false;
      // Page p of sequence b (block id blk) into stage gt % kStages, once P V of the
      // page that stage held is done.
      auto load_page = [&](int b, int p, int blk) -> bool {
        const int st = gt % kStages;
        if (gt >= kStages && !mbar_wait_sleep(sh.bar(BAR_PV_DONE + st), ((gt / kStages) - 1) & 1, abort_flag)) {
          fail(hdr, abort_flag, 11);
          return false;
        }
        if (gt >= kQStageFirst && gt < kStages && !mbar_wait_sleep(sh.bar(BAR_Q_COPIED), 0, abort_flag)) {
          fail(hdr, abort_flag, 15);
          return false;
        }
        // One 4-D box per page half: 32 rows x all column blocks, landing as the nine
        // 32-row x 64-column slots (streams ~8 % faster than nine 3-D boxes).
        if constexpr (kFp8)
          fp8_load_half(sh.stage(st), sh.base + kSmemScales + st * 512, &tm_pair, &tm_kpe, &tm_aux,
                        sh.bar(BAR_RAW + st), blk >= 0 ? blk * kPage + kHalfRows * rank : -kPage);
        else load_page_half(sh.stage(st), &tm_page, &tm_kpe, sh.bar(BAR_FULL + st), rank, blk, a.kpe_separate);
        ++gt;
        return true;
      };
      for (int si = walk.cur(); ok && si >= 0; walk.advance(), si = walk.cur()) {
        const int* rec = seg + (size_t)si * kSegWords;
        const int b = rec[0], rb = rec[1], p0 = rec[2], p1 = rec[3];
        const int row0 = b * R + rb * kRowsPerBlock + kCtaRows * rank;
        // The first page's block id is requested before the query copies are issued
        // (their issue covers its latency).
        int blk_first = 0;
        if (p0 < p1)
          asm volatile("ld.global.b32 %0, [%1];" : "=r"(blk_first) : "l"(a.block_table + (size_t)b * a.bt_stride + p0) : "memory");
        int p = p0;
        if (sc > 0) {
          // A later segment's first pages are requested before its query, which has to
          // wait until Q K^T is done with the previous one: at most kStages of them, so
          // that every stage they reuse held a page of an earlier segment (whose P V
          // does not wait for this segment's query).  Its query rows go to the L2 for
          // the softmax warps' staging.  (Measured on the ragged batch: ~8 us per
          // segment change when the pages waited for the query.)
          const int rows_valid = min(kCtaRows, R - (rb * kRowsPerBlock + kCtaRows * rank));
          if (rows_valid > 0) prefetch_l2_bulk(a.q_lat + (size_t)row0 * kDLat, (uint32_t)rows_valid * kDLat * 2);
          const int early = min(p1 - p0, kStages);
          for (; ok && p < p0 + early; ++p)
            ok = load_page(b, p, p == p0 ? checked_block(a, blk_first, b, p, hdr, true) : page_block(a, b, p, hdr, true));
          if (!ok) break;
          if (!mbar_wait(sh.bar(BAR_Q_FREE), (sc - 1) & 1, abort_flag)) { fail(hdr, abort_flag, 10); ok = false; break; }
        }
        // The first segment's whole query comes by TMA ahead of the pages (boxes 0..5
        // into ring stages 3, 4, copied to tensor memory by the softmax warps); later
        // segments' boxes 0..5 are read by those warps while the ring is in use.
        mbar_arrive_expect_tx(sh.bar(BAR_Q_TMA), (sc == 0 ? kBoxes : kQSmemBoxes) * kQBoxBytes);
        if (sc == 0)
          for (int box = 0; box < kQTmemBoxes; ++box)
            tma_load_2d(sh.q_first(box), &tm_qlat, sh.bar(BAR_Q_TMA), 64 * box, row0);
        for (int box = kQTmemBoxes; box < 8; ++box) tma_load_2d(sh.q(box), &tm_qlat, sh.bar(BAR_Q_TMA), 64 * box, row0);
        tma_load_2d(sh.q(8), &tm_qpe, sh.bar(BAR_Q_TMA), 0, row0);
        q_in_flight = true;
        for (; ok && p < p1; ++p)
          ok = load_page(b, p, p == p0 ? checked_block(a, blk_first, b, p, hdr, true) : page_block(a, b, p, hdr, true));
        ++sc;
      }
      // Drain: every load issued must have landed before the CTA may exit.
      const int first = gt > kStages ? gt - kStages : 0;
      for (int g = first; g < gt; ++g) {
        mbar_wait_drain(sh.bar((kFp8 ? BAR_RAW : BAR_FULL) + g % kStages), (g / kStages) & 1);
      }
      if (q_in_flight) {
        mbar_wait_drain(sh.bar(BAR_Q_TMA), (sc - 1) & 1);
      }
    } else if (lane == 1) {
      // ------------------------------------------------------------ reloads of the other half's rows
      reload_role<kMode>(sh, &tm_pair, &tm_aux, a, hdr, abort_flag, seg, walk0, rank);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ CTA 0: Q K^T issuer; CTA 1: reload relay
    if (rank == 0) qk_role(sh, tmem, hdr, abort_flag, seg, walk0);
    else if (lane == 0) relay_role(sh, hdr, abort_flag, seg, walk0, BAR_RELOAD, BAR_RELOAD, 14);
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ CTA 0: P V issuer; CTA 1: page-half relay
    if (rank == 0) pv_role(sh, tmem, hdr, abort_flag, seg, walk0);
    else if (lane == 0) relay_role(sh, hdr, abort_flag, seg, walk0, BAR_FULL, BAR_FULL, 12);
    __syncwarp();
  } else if (warp == 3) {
    // idle: a warp issuing next to two softmax warps slows them (measured)
    __syncwarp();
  } else if (kFp8 && warp >= 12) {
    // ------------------------------------------------------------ FP8 row conversion (warps 12..15)
    fp8_convert_role(sh, hdr, abort_flag, seg, walk0, rank, tid - 384);
  } else {
    // ------------------------------------------------------------ softmax + epilogue (warps 4..11)
    // TMEM lane ln holds query row hr = ln % 64 of this CTA and page half kh = ln / 64;
    // two threads share a lane (warps w and w + 4): thread half cw takes score
    // columns [16 cw, 16 cw + 16) of the lane, and accumulator columns
    // [128 cw, 128 cw + 128), i.e. latent block m = cw.
    const int q4 = warp & 3;
    const int cw = (warp - 4) >> 2;
    const int ln = 32 * q4 + lane;
    const int hr = ln & 63, kh = ln >> 6;
    const int part = 2 * kh + cw;                  // this thread's quarter of its row
    const int row = kCtaRows * rank + hr;          // row within the 128-row group
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q4) << 16);
    float* xrow = reinterpret_cast<float*>(smem + kSmemXchg);  // [buffer][quarter][row]
    const uint32_t xbar = sh.bar(BAR_XCH + (q4 & 1));
    // Combine a value over the four threads of a row (bounded wait on the mbarrier
    // of the four warps holding rows 32 (q4 & 1) .. + 31; double-buffered by parity).
    int xc = 0;
    auto row_exchange = [&](float v, float* out) -> bool {
      float* slot = xrow + (xc & 1) * 256;
      slot[part * 64 + hr] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);   // one arrival per warp, after the warp's stores
      const bool w = mbar_wait(xbar, xc & 1, abort_flag);
      out[0] = slot[hr];
      out[1] = slot[64 + hr];
      out[2] = slot[128 + hr];
      out[3] = slot[192 + hr];
      ++xc;
      return __all_sync(0xffffffffu, w);
    };
    // Query columns 0..383 of this row go to this thread's TMEM lane (A operand of
    // the first 24 K steps; both lanes of the row hold a copy, each thread three of
    // the six boxes) once the previous segment's Q K^T is done with them; then each
    // warp reports (with the query TMA) to CTA 0.
    auto stage_q = [&](const SegRows& s, int sc_of) -> bool {
      const bool w_ok = sc_of == 0 || mbar_wait(sh.bar(BAR_Q_FREE), (sc_of - 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, w_ok)) return false;
      tc_fence_after();
      uint4 v[24];
      if (sc_of == 0) {
        // From the TMA copy in ring stages 3, 4: row hr of box k, 16-byte chunk c
        // at k * 8 KB + 128 hr + 16 (c ^ (hr % 8)) (128-byte swizzle).
        const bool t_ok = mbar_wait(sh.bar(BAR_Q_TMA), 0, abort_flag);
        if (!__all_sync(0xffffffffu, t_ok)) return false;
#pragma unroll
        for (int bb = 0; bb < 3; ++bb) {
          const unsigned char* box = smem + kSmemRing + kQStageFirst * kStageBytes + (3 * cw + bb) * kQBoxBytes + hr * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) v[8 * bb + c] = *reinterpret_cast<const uint4*>(box + 16 * (c ^ (hr & 7)));
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(a.q_lat + ((size_t)s.b * R + (s.row_valid ? s.fr : 0)) * kDLat) +
                           8 * 3 * cw;
#pragma unroll
        for (int e = 0; e < 24; ++e) v[e] = s.row_valid ? __ldg(src + e) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int bb = 0; bb < 3; ++bb) {
        uint32_t q[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          q[4 * e] = v[8 * bb + e].x; q[4 * e + 1] = v[8 * bb + e].y;
          q[4 * e + 2] = v[8 * bb + e].z; q[4 * e + 3] = v[8 * bb + e].w;
        }
        tmem_st32(t_lane + kTmemQ + 32 * (3 * cw + bb), q);
      }
      tmem_wait_st();
      if (sc_of == 0) {
        // the staging area goes back to the page ring (its reads precede the page loads' writes)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(sh.bar(BAR_Q_COPIED));
      }
      const bool t_ok = mbar_wait(sh.bar(BAR_Q_TMA), sc_of & 1, abort_flag);
      if (!__all_sync(0xffffffffu, t_ok)) return false;
      tc_fence_before();
      warp_arrive_leader(sh.bar(BAR_Q_READY), rank);
      return true;
    };

    SegWalk walk = walk0;
    int si = walk.cur();
    int g = 0, sc = 0;
    bool ok = true;
    SegRows cur;
    if (si >= 0) {
      cur = seg_rows(seg + (size_t)si * kSegWords, a, R, row);
      if (!stage_q(cur, 0)) { fail(hdr, abort_flag, 33); ok = false; }
    }
    while (ok && si >= 0) {
      float m_ref = -INFINITY, l = 0.f;   // l: this thread's quarter of the row sum
      const int n_tiles = cur.p1 - cur.p0;
      for (int i = 0; i < n_tiles; ++i, ++g) {
        const int sb = g & 1, st = g % kStages, pb = g % kPBufs;
        const int page = cur.p0 + i;
        const int jbase = page * kPage + kHalfRows * kh + 16 * cw;   // first cache row of this thread's columns
        bool w_ok = mbar_wait(sh.bar(BAR_S_FULL + sb), (g >> 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) { fail(hdr, abort_flag, 30); ok = false; break; }
        tc_fence_after();
        uint32_t sr[16];
        tmem_ld16(t_lane + kTmemS + 32 * sb + 16 * cw, sr);
        tmem_wait_ld();
        tc_fence_before();
        warp_arrive_leader(sh.bar(BAR_S_FREE + sb), rank);
        // Raw-score maximum over the visible columns (the scale is positive).
        const bool full = jbase + 16 <= cur.limit;
        float mx[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) mx[k] = -INFINITY;
        if (full) {
#pragma unroll
          for (int j = 0; j < 16; ++j) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(sr[j]));
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (jbase + j < cur.limit) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(sr[j]));
        }
        float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        {
          float o4[4];
          if (!row_exchange(tmax, o4)) { fail(hdr, abort_flag, 37); ok = false; break; }
          tmax = fmaxf(fmaxf(o4[0], o4[1]), fmaxf(o4[2], o4[3])) * a.scale_log2;
        }
        // Lazy rescale of the running state: needs the accumulator up to date (P V of
        // the previous page complete); rare once the reference max has settled.
        const bool grow = tmax > m_ref + kRescaleThreshold;
        const float new_ref = grow ? tmax : m_ref;
        const float factor = (grow && m_ref != -INFINITY) ? ex2(m_ref - new_ref) : 1.f;
        if (i > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
          const int g1 = g - 1;
          w_ok = mbar_wait(sh.bar(BAR_PV_DONE + g1 % kStages), (g1 / kStages) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, w_ok)) { fail(hdr, abort_flag, 31); ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 4 * cw; c < 4 * cw + 4; ++c) {
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
        // This thread's 16 P values, p = 2^(s * scale * log2 e - m), as bf16 pairs.
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = ex2(fmaf(__uint_as_float(sr[j]), a.scale_log2, -m_use));
        if (!full) {
#pragma unroll
          for (int j = 0; j < 16; ++j) x[j] = (jbase + j < cur.limit) ? x[j] : 0.f;
        }
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pw[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          ps[e & 3] += x[2 * e] + x[2 * e + 1];
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
          pw[e] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        // P tile pb is free once P V of page g - kPBufs is done.
        if (g >= kPBufs) {
          const int g2 = g - kPBufs;
          w_ok = mbar_wait(sh.bar(BAR_PV_DONE + g2 % kStages), (g2 / kStages) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, w_ok)) { fail(hdr, abort_flag, 34); ok = false; break; }
        }
        {
          // Row hr of P (128 bytes, K-major, 128-byte swizzle): this thread's two 16-byte chunks.
          const uint32_t prow = sh.p(pb) + hr * 128;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint32_t chunk = (uint32_t)((4 * kh + 2 * cw + c) ^ (hr & 7));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + 16 * chunk), "r"(pw[4 * c]),
                         "r"(pw[4 * c + 1]), "r"(pw[4 * c + 2]), "r"(pw[4 * c + 3])
                         : "memory");
          }
        }
        // Rows of the last page past the sequence end are zeroed in the eight latent
        // slots P V reads, once the other half's rows (reloaded after Q K^T) landed.
        const int valid = cur.S - page * kPage;
        if (valid < kPage) {
          w_ok = mbar_wait(sh.bar(BAR_RELOAD + st), (g / kStages) & 1, abort_flag);
          if (!__all_sync(0xffffffffu, w_ok)) { fail(hdr, abort_flag, 35); ok = false; break; }
          // After the reload, latent slot s holds rows of page half (s >> 1) & 1 in both CTAs.
          const int idx = tid - 128;   // 0..255: slot idx / 32, row idx % 32
          const int s_ = idx / kHalfRows, rr = idx % kHalfRows;
          if (((s_ >> 1) & 1) * kHalfRows + rr >= valid) {
            const uint32_t dst = sh.slot(st, s_) + rr * 128;
#pragma unroll
            for (int z = 0; z < 8; ++z)
              asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(dst + 16 * z), "r"(0) : "memory");
          }
        }
        fence_proxy_async_smem();
        warp_arrive_leader(sh.bar(BAR_P_FULL + pb), rank);
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
      // Epilogue: wait for the last P V, combine the four quarters of the row sum,
      // then normalise and store this thread's 128 output columns.
      {
        const int gl = g - 1;
        const bool w_ok = mbar_wait(sh.bar(BAR_PV_DONE + gl % kStages), (gl / kStages) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) { fail(hdr, abort_flag, 32); ok = false; break; }
        tc_fence_after();
      }
      float l4[4];
      if (!row_exchange(l, l4)) { fail(hdr, abort_flag, 38); ok = false; break; }
      const float l_row = (l4[0] + l4[1]) + (l4[2] + l4[3]);
      const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      const float lse_v = l_row > 0.f ? (m_use + __log2f(l_row)) * 0.69314718055994531f : -INFINITY;
      const int b = cur.b, fr = cur.fr, slot_out = cur.slot_out;
      // Two 32-column chunks per tensor-memory wait (the stores of one pair overlap
      // the loads of the next; measured ~0.5 us per launch on the uniform batch).
#pragma unroll 1
      for (int c2 = 4 * cw; c2 < 4 * cw + 4; c2 += 2) {
        uint32_t o2[2][32];
        tmem_ld32(t_lane + kTmemO + 32 * c2, o2[0]);
        tmem_ld32(t_lane + kTmemO + 32 * c2 + 32, o2[1]);
        tmem_wait_ld();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
        const int c = c2 + hh;
        const uint32_t* o = o2[hh];
        // TMEM column 128 m + cc of this lane = latent column 256 m + 128 kh + cc.
        const int col0 = 256 * (c >> 2) + 128 * kh + 32 * (c & 3);
        if (cur.row_valid) {
          // 32-byte stores: each thread writes whole sectors of its row.
          if (slot_out < 0) {
            __nv_bfloat16* dst = a.o_lat + ((size_t)b * R + fr) * kDLat + col0;
#pragma unroll
            for (int e = 0; e < 32; e += 16) {
              uint32_t w[8];
              pack_bf16x8(o + e, inv, w);
              pack_bf16x8(o + e + 8, inv, w + 4);
              st_global_v8(dst + e, w);
            }
          } else {
            float* dst = part_o + ((size_t)slot_out * kRowsPerBlock + row) * kDLat + col0;
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
      }
      if (cur.row_valid && part == 0) {
        if (slot_out < 0) a.lse[(size_t)b * R + fr] = lse_v;
        else part_lse[(size_t)slot_out * kRowsPerBlock + row] = lse_v;
      }
      if (slot_out >= 0) {
        // this warp's partial rows of the group are stored: count them into its merge record
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          atomicAdd(reinterpret_cast<int*>(ws + a.L.off_merge_sync) + 2 * cur.merge_rec, 1);
        }
      }
      tc_fence_before();
      warp_arrive_leader(sh.bar(BAR_O_FREE), rank);
      ++sc;
      si = si_next;
      cur = nxt;
    }
  }

  if (tid == 0) *s_num_merge = num_merge_ld;
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);

  // The plan's merge records (split groups and empty groups): each CTA merges a
  // contiguous share of their rows, each record once all its partial rows are
  // stored (by any CTA of the grid).
  const int num_merge = *s_num_merge;
  if (num_merge > 0) {
    const merge::Out out{a.T, a.H, a.o_lat, a.lse};
    merge::merge_plan_share<threads_of<kMode>() / 128>(out, ws, a.L, num_merge, blockIdx.x, gridDim.x,
                                            reinterpret_cast<float*>(smem + kSmemRing), s_merge_ok);
  }
}

// Test export of the decode kernel's gather: page p of sequence b is fetched by
// load_page_half (path 0: all 576 columns of both halves) or, after that, by
// load_pair_box over every latent column pair of both halves (path 1: the
// latent columns come through the reload map, the RoPE columns through the page
// map), with the block id taken from the block table as the producer takes it,
// then copied out of the 128-byte-swizzled slots as rows j = 64 p + r < S_b of
// out [S_b, 576].  One CTA per page of the table row; a page past S_b returns.
constexpr int kGatherThreads = 128;

__global__ void __launch_bounds__(kGatherThreads)
    debug_gather_sm103_kernel(const __grid_constant__ CUtensorMap tm_page, const __grid_constant__ CUtensorMap tm_pair,
                              const __grid_constant__ CUtensorMap tm_kpe, const int32_t* block_table, int bt_stride,
                              const int32_t* seq_lens, int b, int num_blocks, int kpe_separate, int path,
                              __nv_bfloat16* out, int* status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t stage = smem_addr(smem);
  const uint32_t bar = stage + kStageBytes;
  __shared__ int s_ok;
  int S = seq_lens[b];
  S = S < 0 ? 0 : min(S, bt_stride * kPage);
  const int p = blockIdx.x;
  if (p * kPage >= S) return;
  int blk = block_table[(size_t)b * bt_stride + p];
  if (blk < 0 || blk >= num_blocks) blk = -1;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    s_ok = 1;
  }
  __syncthreads();
  uint32_t phase = 0;
  for (int half = 0; half < 2; ++half) {
    for (int pass = 0; pass < (path == 0 ? 1 : 2); ++pass) {
      if (threadIdx.x == 0) {
        if (pass == 0) {
          load_page_half(stage, &tm_page, &tm_kpe, bar, half, blk, kpe_separate);
        } else {
          mbar_arrive_expect_tx(bar, 8 * kSlotBytes);
          for (int box = 0; box < 8; box += 2) load_pair_box(stage + box * kSlotBytes, &tm_pair, bar, half, box, blk);
        }
        if (!mbar_wait_drain(bar, phase)) {
          s_ok = 0;
          atomicCAS(status, 0, MLA_ERR_TIMEOUT);
        }
      }
      phase ^= 1;
      __syncthreads();
    }
    if (s_ok) {
      // slot s, row r, 16-byte chunk c sits at s * 4 KB + r * 128 + 16 (c ^ (r % 8))
      for (int idx = threadIdx.x; idx < kHalfRows * kBoxes * 8; idx += kGatherThreads) {
        const int r = idx / (kBoxes * 8), sb = (idx / 8) % kBoxes, c = idx % 8;
        const int j = p * kPage + half * kHalfRows + r;
        if (j < S) {
          const uint4 v = *reinterpret_cast<const uint4*>(smem + sb * kSlotBytes + r * 128 + 16 * (c ^ (r & 7)));
          *reinterpret_cast<uint4*>(out + (size_t)j * kDK + 64 * sb + 8 * c) = v;
        }
      }
    }
    fence_proxy_async_smem();   // the reads above precede the next half's TMA writes
    __syncthreads();
  }
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
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};  // one per dimension (rank <= 5)
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides_bytes, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A 2-D byte tensor map over the FP8 pool's rows (656 bytes each): boxes
// box_w bytes wide and 32 rows high, no swizzle (the converters read them as rows).
bool make_fp8_map(CUtensorMap* m, const void* base, long long rows, uint32_t box_w) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kFp8Row, (cuuint64_t)rows};
  const cuuint64_t str[1] = {(cuuint64_t)kFp8Row};
  const cuuint32_t box[2] = {box_w, (cuuint32_t)kHalfRows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, str, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of the paged cache.  Page halves are 4-D boxes (64 columns, 32
// rows, column blocks, 1 block): with the RoPE values at latent + 512 of the same
// rows (the combined 576-wide row) the nine column blocks are one box; otherwise
// the eight latent blocks, plus a 3-D RoPE box.  m_pair loads two adjacent latent
// blocks (the reloads).
bool make_cache_maps(const CacheView& cv, CUtensorMap* m_page, CUtensorMap* m_pair, CUtensorMap* m_kpe,
                     bool* combined) {
  *combined = cv.kpe == cv.ckv + kDLat && cv.kpe_row == cv.ckv_row && cv.kpe_block == cv.ckv_block;
  const cuuint32_t ncb = *combined ? 9 : 8;
  {
    const cuuint64_t dims[4] = {64, (cuuint64_t)kPage, ncb, (cuuint64_t)cv.num_blocks};
    const cuuint64_t str[3] = {(cuuint64_t)cv.ckv_row * 2, 128, (cuuint64_t)cv.ckv_block * 2};
    const cuuint32_t box[4] = {64, kHalfRows, ncb, 1};
    if (!make_map(m_page, cv.ckv, 4, dims, str, box)) return false;
    const cuuint32_t box2[4] = {64, kHalfRows, 2, 1};
    if (!make_map(m_pair, cv.ckv, 4, dims, str, box2)) return false;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kDRope, (cuuint64_t)kPage, (cuuint64_t)cv.num_blocks};
    const cuuint64_t str[2] = {(cuuint64_t)cv.kpe_row * 2, (cuuint64_t)cv.kpe_block * 2};
    const cuuint32_t box[3] = {64, kHalfRows, 1};
    if (!make_map(m_kpe, cv.kpe, 3, dims, str, box)) return false;
  }
  return true;
}

// The shared-memory opt-in, once per device (setting it twice is harmless).
bool set_kernel_attributes() {
  static std::atomic<bool> done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (!done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(decode_sm103_kernel<kModeDense>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemAlloc) != cudaSuccess ||
        cudaFuncSetAttribute(decode_sm103_kernel<kModeSparse>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemAlloc) != cudaSuccess ||
        cudaFuncSetAttribute(decode_sm103_kernel<kModeFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemAlloc) != cudaSuccess)
      return false;
    done[dev].store(true, std::memory_order_release);
  }
  return true;
}

// Launch configuration: clusters of two CTAs; with `pdl`, also programmatic
// stream serialisation (the kernel waits for its predecessor in pdl_wait).
void cluster_launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int pairs, cudaStream_t st,
                           bool pdl, int threads = kThreads) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = dim3(2 * pairs, 1, 1);
  cfg->blockDim = dim3(threads, 1, 1);
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
  // Filled on first use per device; concurrent first calls compute and store the same value.
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int got = cached[dev].load(std::memory_order_acquire);
  if (got == 0) {
    int n = 0;
    if (set_kernel_attributes()) {
      cudaLaunchConfig_t cfg;
      cudaLaunchAttribute attr[2];
      cluster_launch_config(&cfg, attr, 256, 0, false);
      if (cudaOccupancyMaxActiveClusters(&n, decode_sm103_kernel<kModeDense>, &cfg) != cudaSuccess) n = 0;
    }
    if (n <= 0) {
      const int sms = mla_device_sm_count();
      n = sms >= 2 ? sms / 2 : 1;
    }
    cached[dev].store(n, std::memory_order_release);
    got = n;
  }
  return got;
}

cudaError_t launch_decode_sm103(const mla_geom* g, const mla_batch* b, const WsLayout& L,
                                const __nv_bfloat16* q_lat, const __nv_bfloat16* q_pe, const CacheView& cv,
                                const int32_t* block_table, int bt_stride, const int32_t* seq_lens, int checked,
                                __nv_bfloat16* o_lat, float* lse, void* ws, cudaStream_t st, const SparseList* sparse,
                                const Fp8Pool* fp8) {
  const long long rows_total = (long long)b->B * b->T * g->H;
  CUtensorMap m_qlat, m_qpe, m_page, m_pair, m_kpe, m_aux;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kDLat, (cuuint64_t)rows_total};
    const cuuint64_t str[1] = {(cuuint64_t)kDLat * 2};
    const cuuint32_t box[2] = {64, kCtaRows};
    if (!make_map(&m_qlat, q_lat, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)kDRope, (cuuint64_t)rows_total};
    const cuuint64_t str[1] = {(cuuint64_t)kDRope * 2};
    const cuuint32_t box[2] = {64, kCtaRows};
    if (!make_map(&m_qpe, q_pe, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  bool combined = false;
  int num_blocks = cv.num_blocks;
  if (fp8 != nullptr) {
    const long long rows = (long long)fp8->num_blocks * kPage;
    num_blocks = fp8->num_blocks;
    combined = true;
    if (!make_fp8_map(&m_pair, fp8->rows, rows, 128) || !make_fp8_map(&m_aux, fp8->rows, rows, 16))
      return cudaErrorInvalidValue;
    m_page = m_pair;
    // the RoPE values: bytes 528..655 of every row, as 64 bf16 (16-byte aligned: 528 = 33 x 16)
    const cuuint64_t dims[2] = {(cuuint64_t)kDRope, (cuuint64_t)rows};
    const cuuint64_t str[1] = {(cuuint64_t)kFp8Row};
    const cuuint32_t box[2] = {64, (cuuint32_t)kHalfRows};
    if (!make_map(&m_kpe, fp8->rows + 528, 2, dims, str, box)) return cudaErrorInvalidValue;
  } else if (sparse == nullptr) {
    if (!make_cache_maps(cv, &m_page, &m_pair, &m_kpe, &combined)) return cudaErrorInvalidValue;
    m_aux = m_pair;
  } else {
    // The sparse decode copies the listed rows with plain (cp.async) copies: no
    // cache maps (the kernel prefetches and never uses these).
    m_page = m_pair = m_kpe = m_aux = m_qlat;
  }
  FastArgs a;
  a.q_lat = q_lat;
  a.block_table = block_table; a.bt_stride = bt_stride; a.seq_lens = seq_lens;
  a.seq_div = sparse ? sparse->seq_div : 1;
  a.B = b->B; a.T = b->T; a.H = g->H; a.causal = b->causal ? 1 : 0; a.checked = checked;
  a.max_pages = b->max_pages; a.num_blocks = num_blocks;
  a.max_rows = sparse ? sparse->topk : b->max_pages * kPage;
  a.indices = sparse ? sparse->indices : nullptr;
  a.topk = sparse ? sparse->topk : 0;
  a.kpe_separate = combined ? 0 : 1;
  a.ckv = cv.ckv; a.kpe = cv.kpe; a.ckv_row = cv.ckv_row; a.kpe_row = cv.kpe_row;
  a.scale_log2 = g->softmax_scale * 1.4426950408889634f;
  a.o_lat = o_lat; a.lse = lse; a.L = L;
  if (!set_kernel_attributes()) return cudaErrorInvalidValue;
  int pairs = L.cap_ranges;
  const int max_pairs = decode_sm103_pairs_per_device();
  if (pairs > max_pairs) pairs = max_pairs;
  if (pairs <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cluster_launch_config(&cfg, attr, pairs, st, true, fp8 ? kFp8Threads : kThreads);
  char* w = reinterpret_cast<char*>(ws);
  if (fp8)
    return cudaLaunchKernelEx(&cfg, decode_sm103_kernel<kModeFp8>, m_qlat, m_qpe, m_page, m_pair, m_kpe, m_aux, a, w);
  if (sparse)
    return cudaLaunchKernelEx(&cfg, decode_sm103_kernel<kModeSparse>, m_qlat, m_qpe, m_page, m_pair, m_kpe, m_aux, a,
                              w);
  return cudaLaunchKernelEx(&cfg, decode_sm103_kernel<kModeDense>, m_qlat, m_qpe, m_page, m_pair, m_kpe, m_aux, a, w);
}

cudaError_t set_pipeline_wait_limit(long long cycles) {
  const long long v = cycles > 0 ? cycles : ptx::kWaitLimitCycles;
  return cudaMemcpyToSymbol(wait_override::c_pipeline_wait_limit, &v, sizeof(v));
}

cudaError_t launch_debug_gather(const CacheView& cv, const int32_t* block_table, int bt_stride,
                                const int32_t* seq_lens, int b, int path, __nv_bfloat16* out, cudaStream_t st) {
  int* status = bmm_status_ptr();
  if (!status) return cudaErrorInvalidValue;
  CUtensorMap m_page, m_pair, m_kpe;
  bool combined = false;
  if (!make_cache_maps(cv, &m_page, &m_pair, &m_kpe, &combined)) return cudaErrorInvalidValue;
  const size_t smem = kStageBytes + 1024 + 64;
  debug_gather_sm103_kernel<<<bt_stride, kGatherThreads, smem, st>>>(m_page, m_pair, m_kpe, block_table, bt_stride,
                                                                    seq_lens, b, cv.num_blocks, combined ? 0 : 1,
                                                                    path, out, status);
  return cudaGetLastError();
}

}  // namespace mla
