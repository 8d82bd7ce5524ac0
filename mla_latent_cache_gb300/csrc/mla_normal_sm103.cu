// The Normal (decompressed) arm on the sm_103a tensor cores: the cached
// latents are up-projected into per-head keys and values, then ordinary
// causal multi-head attention runs over them ("MLA in full detail", the naive
// path of Step 1; "M5.8" 0x02 and 0x06, the decompressed reference):
//   k_nope[j,h,:] = W_UK[h] c_j,   v[j,h,:] = W_UV[h] c_j          (128 each)
//   k[j,h] = [k_nope[j,h] | k_pe_j]   (192 wide; k_pe is shared by all heads)
//   o[t,h] = sum_j softmax_j((q_nope[t,h] . k_nope[j,h] + q_pe[t,h] . k_pe_j) * scale) v[j,h]
// over the cache rows visible to query token t (bottom-right causal alignment).
//
// Expansion kernel.  Expanded rows live in kv_exp bf16 [H][B * rows_per_seq][256]:
// row b * rows_per_seq + j of head h holds [k_nope (128) | v (128)] of cache
// row j of sequence b.  A CTA takes 128 cache rows (two pages) of one
// sequence, keeps them in shared memory (the A operand, 128 x 512) and loops
// over a group of heads: per head one M=128 x N=256 x K=512 product whose B
// operand is [W_UK[h]; W_UV[h]] (256 rows of 512, K-major) streamed through a
// 3-slot ring.  The fp32 accumulator is double-buffered in TMEM (2 x 256
// columns) so the epilogue of head i overlaps the MMAs of head i+1.  Rows past
// the sequence end inside the tile are zeroed in shared memory first, so the
// expanded tile holds exact zeros there.  k_pe is not copied per head: the
// attention kernel reads it from the latent cache.
//
// Attention kernel.  A CTA takes up to 128 query tokens of one (sequence,
// head) and walks the visible keys 128 at a time: S = Q K^T (M=128 tokens,
// N=128 keys, K=192: two k_nope boxes from kv_exp and the two pages' k_pe
// from the cache), online softmax with two threads per token row (each half
// of the tile's keys and of the value columns; the row maximum and sum combined
// through shared memory), lazy rescale of the TMEM accumulator when the row
// maximum grows by more than 2^8, P written over the score tile in TMEM (bf16
// pairs), then O += P V
// (M=128, N=128, K=128 keys, A from TMEM).  Score tiles are double-buffered
// so Q K^T of the next key tile runs while the softmax reads the current one.
//
// Every wait is bounded; a wait that runs out records MLA_ERR_TIMEOUT in the
// status word of the workspace-free kernels, the CTA drains what it issued,
// frees TMEM and exits.
#include <limits.h>
#include <math.h>

#include "mla_internal.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

// ----------------------------------------------------------------------------- expansion
constexpr int kExpThreads = 192;       // warp 0 TMA, warp 1 MMA, warps 2..5 zero-fill + epilogue
constexpr int kExpHeads = 32;          // heads per CTA
constexpr int kABoxBytes = 128 * 64 * 2;   // 128 rows x 64 latent columns
constexpr int kWBytes = 256 * 64 * 2;      // [W_UK[h]; W_UV[h]] rows x 64 latent columns
constexpr int kWSlots = 3;
constexpr int kExpSmemA = 0;
constexpr int kExpSmemW = kExpSmemA + 8 * kABoxBytes;          // 131072
constexpr int kExpSmemBar = kExpSmemW + kWSlots * kWBytes;     // 229376
constexpr int kExpSmemBytes = kExpSmemBar + 256;
constexpr int kExpSmemAlloc = kExpSmemBytes + 1024;
static_assert(kExpSmemAlloc <= 232448, "shared memory per CTA");

enum {
  EB_A_FULL = 0,
  EB_A_READY,
  EB_W_FULL,                       // kWSlots
  EB_W_EMPTY = EB_W_FULL + kWSlots,  // kWSlots
  EB_ACC_FULL = EB_W_EMPTY + kWSlots,  // 2
  EB_ACC_EMPTY = EB_ACC_FULL + 2,      // 2 (128 arrivals)
  EB_FINAL = EB_ACC_EMPTY + 2,
  kExpBars
};

struct ExpArgs {
  const int32_t* block_table;
  int bt_stride;
  const int32_t* seq_lens;
  int B, H, max_pages, num_blocks;
  int row_begin;                    // first cache row expanded (a multiple of 128)
  int rows_per_seq, tiles_per_seq;  // expanded rows held per sequence (from row_begin), in 128-row tiles
  __nv_bfloat16* kv_exp;
  int* status;
};

__device__ __forceinline__ void fail_status(int* status, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(status, 0, MLA_ERR_TIMEOUT);
}

__global__ void __launch_bounds__(kExpThreads, 1)
    normal_expand_kernel(const __grid_constant__ CUtensorMap tm_ckv, const __grid_constant__ CUtensorMap tm_wuk,
                         const __grid_constant__ CUtensorMap tm_wuv, ExpArgs a) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x / a.tiles_per_seq, tile = blockIdx.x % a.tiles_per_seq;
  int S = a.seq_lens[b];
  S = S < 0 ? 0 : min(S, a.max_pages * kPage);
  const int r0 = a.row_begin + tile * 128;
  if (r0 >= S) return;  // nothing of this sequence lives in the tile (uniform over the CTA)
  const int valid = min(128, S - r0);
  const int h0 = blockIdx.y * kExpHeads;
  const int nh = min(kExpHeads, a.H - h0);
  if (nh <= 0) return;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if ((uintptr_t)(smem - smem_raw) + kExpSmemBytes > (uintptr_t)kExpSmemAlloc) {
    if (threadIdx.x == 0) atomicCAS(a.status, 0, MLA_ERR_DEVICE_CHECK);
    return;
  }
  const uint32_t base = smem_addr(smem);
  auto bar = [&](int i) { return base + kExpSmemBar + 8 * i; };
  auto wslot = [&](int s) { return base + kExpSmemW + s * kWBytes; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kExpSmemBar + 8 * kExpBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kExpSmemBar + 8 * kExpBars + 4);
  int* page_loaded = reinterpret_cast<int*>(smem + kExpSmemBar + 8 * kExpBars + 8);  // [2]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(bar(EB_A_FULL), 1);
    mbar_init(bar(EB_A_READY), 128);
    for (int s = 0; s < kWSlots; ++s) {
      mbar_init(bar(EB_W_FULL + s), 1);
      mbar_init(bar(EB_W_EMPTY + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(EB_ACC_FULL + i), 1);
      mbar_init(bar(EB_ACC_EMPTY + i), 128);
    }
    mbar_init(bar(EB_FINAL), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_ckv);
    prefetch_tmap(&tm_wuk);
    prefetch_tmap(&tm_wuv);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_steps = nh * 8;  // (head, 64-column K slice) steps through the weight ring

  if (warp == 0) {
    if (lane == 0) {
      // The tile's two pages: all eight 64-column boxes of each present page.
      int blk[2], bytes = 0;
      for (int pg = 0; pg < 2; ++pg) {
        const int p = r0 / kPage + pg;
        blk[pg] = -1;
        if (p * kPage < S) {
          const int id = a.block_table[(size_t)b * a.bt_stride + p];
          if (id >= 0 && id < a.num_blocks) { blk[pg] = id; bytes += 8 * kPage * 128; }
        }
        page_loaded[pg] = blk[pg] >= 0 ? 1 : 0;
      }
      mbar_arrive_expect_tx(bar(EB_A_FULL), bytes);
      for (int pg = 0; pg < 2; ++pg) {
        if (blk[pg] < 0) continue;
        for (int bx = 0; bx < 8; ++bx)
          tma_load_3d(base + kExpSmemA + bx * kABoxBytes + pg * (kPage * 128), &tm_ckv, bar(EB_A_FULL), 64 * bx, 0,
                      blk[pg]);
      }
      int g = 0;
      bool ok = true;
      for (; g < n_steps; ++g) {
        const int s = g % kWSlots, hi = g >> 3, kb = g & 7;
        if (!mbar_wait(bar(EB_W_EMPTY + s), ((g / kWSlots) & 1) ^ 1, abort_flag)) { fail_status(a.status, abort_flag); ok = false; break; }
        mbar_arrive_expect_tx(bar(EB_W_FULL + s), kWBytes);
        tma_load_3d(wslot(s), &tm_wuk, bar(EB_W_FULL + s), 64 * kb, 0, h0 + hi);
        tma_load_3d(wslot(s) + kWBytes / 2, &tm_wuv, bar(EB_W_FULL + s), 64 * kb, 0, h0 + hi);
      }
      (void)ok;
      // Drain the loads still in flight before the CTA may exit.
      volatile int never = 0;
      mbar_wait(bar(EB_A_FULL), 0, &never);
      for (int d = g > kWSlots ? g - kWSlots : 0; d < g; ++d) mbar_wait(bar(EB_W_FULL + d % kWSlots), (d / kWSlots) & 1, &never);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 256, 0);
      const uint64_t adesc0 = sw128_desc(base + kExpSmemA, 16, 1024);
      const uint64_t wdesc0 = sw128_desc(wslot(0), 16, 1024);
      bool ok = mbar_wait(bar(EB_A_READY), 0, abort_flag);
      if (!ok) fail_status(a.status, abort_flag);
      tc_fence_after();
      for (int i = 0; ok && i < nh; ++i) {
        const int acc = i & 1;
        if (i >= 2 && !mbar_wait(bar(EB_ACC_EMPTY + acc), ((i >> 1) - 1) & 1, abort_flag)) {
          fail_status(a.status, abort_flag); ok = false; break;
        }
        tc_fence_after();
        for (int kb = 0; kb < 8; ++kb) {
          const int g = i * 8 + kb, s = g % kWSlots;
          if (!mbar_wait(bar(EB_W_FULL + s), (g / kWSlots) & 1, abort_flag)) { fail_status(a.status, abort_flag); ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem + 256 * acc, adesc0 + (uint64_t)(kb * (kABoxBytes >> 4)) + 2 * kk,
                     wdesc0 + (uint64_t)(s * (kWBytes >> 4)) + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
          mma_commit(bar(EB_W_EMPTY + s));
        }
        if (ok) mma_commit(bar(EB_ACC_FULL + acc));
      }
      mma_commit(bar(EB_FINAL));
      volatile int never = 0;
      mbar_wait(bar(EB_FINAL), 0, &never);
    }
    __syncwarp();
  } else {
    // warps 2..5: TMEM lane quadrant warp % 4, one tile row per thread
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q4) << 16);
    bool ok = __all_sync(0xffffffffu, mbar_wait(bar(EB_A_FULL), 0, abort_flag));
    if (!ok) fail_status(a.status, abort_flag);
    // Rows past the sequence end, or of a page that was not loaded, become zeros.
    if (row >= valid || !page_loaded[row >> 6]) {
#pragma unroll 1
      for (int bx = 0; bx < 8; ++bx) {
        const uint32_t dst = base + kExpSmemA + bx * kABoxBytes + row * 128;
#pragma unroll
        for (int z = 0; z < 8; ++z)
          asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(dst + 16 * z), "r"(0) : "memory");
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(bar(EB_A_READY));
    const size_t rows_cap = (size_t)a.B * a.rows_per_seq;
    const size_t grow = (size_t)b * a.rows_per_seq + (r0 - a.row_begin) + row;
    for (int i = 0; ok && i < nh; ++i) {
      const int acc = i & 1;
      const bool w_ok = mbar_wait(bar(EB_ACC_FULL + acc), (i >> 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, w_ok)) { fail_status(a.status, abort_flag); ok = false; break; }
      tc_fence_after();
      __nv_bfloat16* dst = a.kv_exp + ((size_t)(h0 + i) * rows_cap + grow) * 256;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t v[32];
        tmem_ld32(t_lane + 256 * acc + 32 * c, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 16) {
          uint32_t w[8];
          pack_bf16x8(v + e, 1.f, w);
          pack_bf16x8(v + e + 8, 1.f, w + 4);
          st_global_v8(dst + 32 * c + e, w);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(EB_ACC_EMPTY + acc));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ----------------------------------------------------------------------------- attention
constexpr int kAttThreads = 384;       // warp 0 TMA, 1 Q K^T, 2 P V, 3 idle, 4..11 softmax (two per row)
constexpr int kAttBox = 128 * 64 * 2;  // 16 KB: 128 rows x 64 bf16
constexpr int kAttStageK = 3 * kAttBox;  // k_nope (2 boxes) + k_pe (2 pages)
constexpr int kAttStage = kAttStageK + 2 * kAttBox;  // + v (2 boxes)
constexpr int kAttSmemQ = 0;                         // q_nope (2 boxes) + q_pe
constexpr int kAttSmemRing = 3 * kAttBox;            // 49152
constexpr int kAttSmemBar = kAttSmemRing + 2 * kAttStage;  // 212992
constexpr int kAttSmemXch = kAttSmemBar + 256;            // float [2 buffers][2 halves][128 rows]
constexpr int kAttSmemBytes = kAttSmemXch + 2048;
constexpr int kAttSmemAlloc = kAttSmemBytes + 1024;
static_assert(kAttSmemAlloc <= 232448, "shared memory per CTA");
constexpr uint32_t kAttTmemO = 0;    // 128 columns
constexpr uint32_t kAttTmemS = 128;  // 2 x 128 columns; P (bf16 pairs) over the first 64 of a tile
constexpr float kAttRescale = 8.0f;

enum {
  AB_Q_FULL = 0,
  AB_FULL_K,                  // 2
  AB_EMPTY_K = AB_FULL_K + 2,  // 2
  AB_FULL_V = AB_EMPTY_K + 2,  // 2
  AB_EMPTY_V = AB_FULL_V + 2,  // 2
  AB_S_FULL = AB_EMPTY_V + 2,  // 2
  AB_P_FULL = AB_S_FULL + 2,   // 2 (128 arrivals)
  AB_P_EMPTY = AB_P_FULL + 2,  // 2
  AB_FINAL = AB_P_EMPTY + 2,
  AB_FINAL_PV,
  AB_XCH,                     // the softmax warps exchanged a row value (8 warp arrivals)
  kAttBars
};

struct AttArgs {
  const int32_t* block_table;
  int bt_stride;
  const int32_t* seq_lens;
  int B, T, H, causal, max_pages, num_blocks, rows_per_seq;
  // Key window [key_begin, key_end): the expanded rows of a sequence start at
  // key_begin (a multiple of 128); keys outside the window are not attended.
  int key_begin, key_end;
  // Chunked prefix: merge this window's state with the running one (st_o fp32
  // [B,T,H,128] normalised, st_lse [B,T,H]) when has_prev; write the final bf16
  // o and lse when final_out, else the merged running state.
  int has_prev, final_out;
  float* st_o;
  float* st_lse;
  float scale_log2;
  __nv_bfloat16* o;
  float* lse;
  int* status;
};

__global__ void __launch_bounds__(kAttThreads, 1)
    normal_attention_kernel(const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qp,
                            const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_kpe,
                            AttArgs a) {
  pdl_wait();
  pdl_trigger();
  const int t0 = blockIdx.x * 128, h = blockIdx.y, b = blockIdx.z;
  int S = a.seq_lens[b];
  S = S < 0 ? 0 : min(S, a.max_pages * kPage);
  const int t_last = min(a.T, t0 + 128) - 1;
  const int lim_max = min(visible_limit(S, a.T, t_last, a.causal), a.key_end);
  const int n_tiles = lim_max > a.key_begin ? (lim_max - a.key_begin + 127) / 128 : 0;
  const int n_pages = (S + kPage - 1) / kPage;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if ((uintptr_t)(smem - smem_raw) + kAttSmemBytes > (uintptr_t)kAttSmemAlloc) {
    if (threadIdx.x == 0) atomicCAS(a.status, 0, MLA_ERR_DEVICE_CHECK);
    return;
  }
  const uint32_t base = smem_addr(smem);
  auto bar = [&](int i) { return base + kAttSmemBar + 8 * i; };
  auto stage = [&](int st) { return base + kAttSmemRing + st * kAttStage; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kAttSmemBar + 8 * kAttBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAttSmemBar + 8 * kAttBars + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(bar(AB_Q_FULL), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(AB_FULL_K + i), 1);
      mbar_init(bar(AB_EMPTY_K + i), 1);
      mbar_init(bar(AB_FULL_V + i), 1);
      mbar_init(bar(AB_EMPTY_V + i), 1);
      mbar_init(bar(AB_S_FULL + i), 1);
      mbar_init(bar(AB_P_FULL + i), 256);
      mbar_init(bar(AB_P_EMPTY + i), 1);
    }
    mbar_init(bar(AB_FINAL), 1);
    mbar_init(bar(AB_FINAL_PV), 1);
    mbar_init(bar(AB_XCH), 8);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_qn);
    prefetch_tmap(&tm_qp);
    prefetch_tmap(&tm_kv);
    prefetch_tmap(&tm_kpe);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int row0 = b * a.rows_per_seq;  // first expanded row of this sequence

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(AB_Q_FULL), 3 * kAttBox);
      tma_load_4d(base + kAttSmemQ, &tm_qn, bar(AB_Q_FULL), 0, h, t0, b);
      tma_load_4d(base + kAttSmemQ + kAttBox, &tm_qn, bar(AB_Q_FULL), 64, h, t0, b);
      tma_load_4d(base + kAttSmemQ + 2 * kAttBox, &tm_qp, bar(AB_Q_FULL), 0, h, t0, b);
      int kt = 0;
      bool a_only = false;
      for (; kt < n_tiles; ++kt) {
        const int st = kt & 1;
        const uint32_t par = ((kt >> 1) & 1) ^ 1;
        if (!mbar_wait(bar(AB_EMPTY_K + st), par, abort_flag)) { fail_status(a.status, abort_flag); break; }
        int blk[2], bytes = 2 * kAttBox;
        for (int pg = 0; pg < 2; ++pg) {
          const int p = a.key_begin / kPage + 2 * kt + pg;
          blk[pg] = -1;
          if (p < n_pages) {
            const int id = a.block_table[(size_t)b * a.bt_stride + p];
            if (id >= 0 && id < a.num_blocks) { blk[pg] = id; bytes += kPage * 128; }
          }
        }
        mbar_arrive_expect_tx(bar(AB_FULL_K + st), bytes);
        tma_load_3d(stage(st), &tm_kv, bar(AB_FULL_K + st), 0, row0 + 128 * kt, h);
        tma_load_3d(stage(st) + kAttBox, &tm_kv, bar(AB_FULL_K + st), 64, row0 + 128 * kt, h);
        for (int pg = 0; pg < 2; ++pg)
          if (blk[pg] >= 0)
            tma_load_3d(stage(st) + 2 * kAttBox + pg * (kPage * 128), &tm_kpe, bar(AB_FULL_K + st), 0, 0, blk[pg]);
        if (!mbar_wait(bar(AB_EMPTY_V + st), par, abort_flag)) { fail_status(a.status, abort_flag); a_only = true; break; }
        mbar_arrive_expect_tx(bar(AB_FULL_V + st), 2 * kAttBox);
        tma_load_3d(stage(st) + kAttStageK, &tm_kv, bar(AB_FULL_V + st), 128, row0 + 128 * kt, h);
        tma_load_3d(stage(st) + kAttStageK + kAttBox, &tm_kv, bar(AB_FULL_V + st), 192, row0 + 128 * kt, h);
      }
      volatile int never = 0;
      mbar_wait(bar(AB_Q_FULL), 0, &never);
      const int issued = kt + (a_only ? 1 : 0);
      for (int d = issued > 2 ? issued - 2 : 0; d < issued; ++d) {
        mbar_wait(bar(AB_FULL_K + (d & 1)), (d >> 1) & 1, &never);
        if (d < kt) mbar_wait(bar(AB_FULL_V + (d & 1)), (d >> 1) & 1, &never);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // Q K^T issuer: key tile kt into score tile kt % 2 once P V of tile kt-2 released it.
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 128, 0);
      bool ok = mbar_wait(bar(AB_Q_FULL), 0, abort_flag);
      if (!ok) fail_status(a.status, abort_flag);
      tc_fence_after();
      for (int kt = 0; ok && kt < n_tiles; ++kt) {
        const int st = kt & 1;
        if ((kt >= 2 && !mbar_wait(bar(AB_P_EMPTY + st), ((kt >> 1) - 1) & 1, abort_flag)) ||
            !mbar_wait(bar(AB_FULL_K + st), (kt >> 1) & 1, abort_flag)) {
          fail_status(a.status, abort_flag); ok = false; break;
        }
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const uint64_t qd = sw128_desc(base + kAttSmemQ + j * kAttBox, 16, 1024);
          const uint64_t kd = sw128_desc(stage(st) + j * kAttBox, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem + kAttTmemS + 128 * st, qd + 2 * kk, kd + 2 * kk, idesc, (j | kk) ? 1u : 0u);
        }
        mma_commit(bar(AB_EMPTY_K + st));
        mma_commit(bar(AB_S_FULL + st));
      }
      mma_commit(bar(AB_FINAL));
      volatile int never = 0;
      mbar_wait(bar(AB_FINAL), 0, &never);
    }
    __syncwarp();
  } else if (warp == 2) {
    // P V issuer: O += P (TMEM, bf16 pairs) x V (two 64-column boxes, N-major).
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 128, 1);
      bool ok = true;
      for (int kt = 0; ok && kt < n_tiles; ++kt) {
        const int st = kt & 1;
        if (!mbar_wait(bar(AB_P_FULL + st), (kt >> 1) & 1, abort_flag) ||
            !mbar_wait(bar(AB_FULL_V + st), (kt >> 1) & 1, abort_flag)) {
          fail_status(a.status, abort_flag); ok = false; break;
        }
        tc_fence_after();
        const uint64_t vd = sw128_desc(stage(st) + kAttStageK, kAttBox, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_tmem_a(tmem + kAttTmemO, tmem + kAttTmemS + 128 * st + 8 * kk, vd + 128 * kk, idesc,
                          (kt | kk) ? 1u : 0u);
        mma_commit(bar(AB_EMPTY_V + st));
        mma_commit(bar(AB_P_EMPTY + st));
      }
      mma_commit(bar(AB_FINAL_PV));
      volatile int never = 0;
      mbar_wait(bar(AB_FINAL_PV), 0, &never);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // Softmax + epilogue: two threads per query token (TMEM lane): warps w and w + 4
    // share lanes 32 (w % 4) .. + 31; half hf takes key columns [64 hf, +64) of
    // each score tile and value columns [64 hf, +64) of the accumulator.  The two
    // halves of a row combine their maximum (per tile) and sum (at the end)
    // through shared memory.
    const int q4 = warp & 3, hf = (warp - 4) >> 2;
    const int row = 32 * q4 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q4) << 16);
    const int t = t0 + row;
    const bool row_valid = t < a.T;
    const int limit = row_valid ? min(visible_limit(S, a.T, t, a.causal), a.key_end) : 0;
    float* xch = reinterpret_cast<float*>(smem + kAttSmemXch);
    int xc = 0;
    // Both halves' value of this row (double-buffered by phase parity: a half can
    // refill a buffer only after the other passed the next exchange).
    auto exchange = [&](float v, float* other) -> bool {
      float* buf = xch + (xc & 1) * 256;
      buf[hf * 128 + row] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(AB_XCH));
      const bool w = mbar_wait(bar(AB_XCH), xc & 1, abort_flag);
      *other = buf[(1 - hf) * 128 + row];
      ++xc;
      return __all_sync(0xffffffffu, w);
    };
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int kt = 0; kt < n_tiles; ++kt) {
      const int st = kt & 1;
      const uint32_t s_col = kAttTmemS + 128 * st;
      bool w_ok = mbar_wait(bar(AB_S_FULL + st), (kt >> 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, w_ok)) { fail_status(a.status, abort_flag); ok = false; break; }
      tc_fence_after();
      uint32_t s2[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld32(t_lane + s_col + 64 * hf + 32 * c, s2[c]);
      tmem_wait_ld();
      const int jbase = a.key_begin + 128 * kt + 64 * hf;
      const bool full = jbase + 64 <= limit;
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (full || jbase + 32 * c + j < limit) tmax = fmaxf(tmax, __uint_as_float(s2[c][j]));
      {
        // (both halves have read their scores once this returns: P may overwrite them)
        float other;
        if (!exchange(tmax, &other)) { fail_status(a.status, abort_flag); ok = false; break; }
        tmax = fmaxf(tmax, other) * a.scale_log2;
      }
      const bool grow = tmax > m_ref + kAttRescale;
      const float new_ref = grow ? tmax : m_ref;
      const float factor = (grow && m_ref != -INFINITY) ? ex2(m_ref - new_ref) : 1.f;
      if (kt > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
        // The accumulator must be up to date: P V of the previous tile complete.
        const int t1 = kt - 1;
        w_ok = mbar_wait(bar(AB_P_EMPTY + (t1 & 1)), (t1 >> 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) { fail_status(a.status, abort_flag); ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tmem_ld32(t_lane + kAttTmemO + 64 * hf + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
          tmem_st32(t_lane + kAttTmemO + 64 * hf + 32 * c, o);
        }
        tmem_wait_st();
      }
      l *= factor;
      m_ref = new_ref;
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      float psum = 0.f;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = jbase + 32 * c + 2 * e;
          float x0 = ex2(fmaf(__uint_as_float(s2[c][2 * e]), a.scale_log2, -m_use));
          float x1 = ex2(fmaf(__uint_as_float(s2[c][2 * e + 1]), a.scale_log2, -m_use));
          if (!full) {
            x0 = j < limit ? x0 : 0.f;
            x1 = j + 1 < limit ? x1 : 0.f;
          }
          psum += x0 + x1;
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
          pw[e] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        // keys [64 hf + 32 c, +32) as bf16 pairs: columns 32 hf + 16 c .. of the tile
        tmem_st16(t_lane + s_col + 32 * hf + 16 * c, pw);
      }
      l += psum;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(AB_P_FULL + st));
    }
    if (ok) {
      float other;
      if (!exchange(l, &other)) { fail_status(a.status, abort_flag); ok = false; }
      l += other;
    }
    // Epilogue: o = O / l (bf16), lse = m + ln l (natural log).
    if (ok && n_tiles > 0) {
      const int tl = n_tiles - 1;
      const bool w_ok = mbar_wait(bar(AB_P_EMPTY + (tl & 1)), (tl >> 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, w_ok)) { fail_status(a.status, abort_flag); ok = false; }
      tc_fence_after();
    }
    if (ok) {
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      const size_t ri = ((size_t)b * a.T + (row_valid ? t : 0)) * a.H + h;   // output row (t, h) of sequence b
      // This window's state (o_w = O / l, natural-log lse_w), merged with the running
      // one: m = max(lse_p, lse_w), weights e^{lse - m} normalised to sum 1.
      float lse_out = l > 0.f ? (m_use + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      float w_cur = l > 0.f ? 1.f / l : 0.f, w_prev = 0.f;
      if (a.has_prev && row_valid) {
        const float lp = a.st_lse[ri];
        const float m = fmaxf(lp, lse_out);
        if (m == -INFINITY) {
          w_cur = 0.f;
        } else {
          const float ep = expf(lp - m), ec = expf(lse_out - m), sum = ep + ec;
          w_prev = ep / sum;
          w_cur *= ec / sum;
          lse_out = m + logf(sum);
        }
      }
#pragma unroll 1
      for (int c = 2 * hf; c < 2 * hf + 2; ++c) {
        uint32_t o[32];
        if (n_tiles > 0) {
          tmem_ld32(t_lane + kAttTmemO + 32 * c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (!row_valid) continue;
        if (w_prev != 0.f) {
          const float4* prev = reinterpret_cast<const float4*>(a.st_o + ri * kDV + 32 * c);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 p = prev[e];
            o[4 * e] = __float_as_uint(fmaf(__uint_as_float(o[4 * e]), w_cur, p.x * w_prev));
            o[4 * e + 1] = __float_as_uint(fmaf(__uint_as_float(o[4 * e + 1]), w_cur, p.y * w_prev));
            o[4 * e + 2] = __float_as_uint(fmaf(__uint_as_float(o[4 * e + 2]), w_cur, p.z * w_prev));
            o[4 * e + 3] = __float_as_uint(fmaf(__uint_as_float(o[4 * e + 3]), w_cur, p.w * w_prev));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * w_cur);
        }
        if (a.final_out) {
          __nv_bfloat16* dst = a.o + ri * kDV + 32 * c;
#pragma unroll
          for (int e = 0; e < 32; e += 16) {
            uint32_t w[8];
            pack_bf16x8(o + e, 1.f, w);
            pack_bf16x8(o + e + 8, 1.f, w + 4);
            st_global_v8(dst + e, w);
          }
        } else {
          float* dst = a.st_o + ri * kDV + 32 * c;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = o[e + k];
            st_global_v8(dst + e, w);
          }
        }
      }
      if (row_valid && hf == 0) {
        if (a.final_out) a.lse[ri] = lse_out;
        else a.st_lse[ri] = lse_out;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ----------------------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A bf16 tensor map of rank 2..4 with 128-byte swizzle; strides in bytes for dims 1..rank-1.
bool make_map_n(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                const cuuint32_t* box) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int64_t normal_rows_per_seq(int max_pages) { return (int64_t)((max_pages + 1) / 2) * 128; }

cudaError_t launch_normal_expand_rows(const mla_geom* g, const CacheView& cv, const int32_t* block_table,
                                      int bt_stride, const int32_t* seq_lens, int B, int max_pages, int row_begin,
                                      int rows_per_seq, const __nv_bfloat16* w_uk, const __nv_bfloat16* w_uv,
                                      __nv_bfloat16* kv_exp, cudaStream_t st) {
  int* status = bmm_status_ptr();
  if (!status) return cudaErrorInvalidValue;
  CUtensorMap m_ckv, m_wuk, m_wuv;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kDLat, (cuuint64_t)kPage, (cuuint64_t)cv.num_blocks};
    const cuuint64_t str[2] = {(cuuint64_t)cv.ckv_row * 2, (cuuint64_t)cv.ckv_block * 2};
    const cuuint32_t box[3] = {64, 64, 1};
    if (!make_map_n(&m_ckv, cv.ckv, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kDLat, (cuuint64_t)kDNope, (cuuint64_t)g->H};
    const cuuint64_t str[2] = {(cuuint64_t)kDLat * 2, (cuuint64_t)kDNope * kDLat * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    if (!make_map_n(&m_wuk, w_uk, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (!make_map_n(&m_wuv, w_uv, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(normal_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kExpSmemAlloc) !=
        cudaSuccess)
      return cudaErrorInvalidValue;
    attr = true;
  }
  ExpArgs a;
  a.block_table = block_table; a.bt_stride = bt_stride; a.seq_lens = seq_lens;
  a.B = B; a.H = g->H; a.max_pages = max_pages; a.num_blocks = cv.num_blocks;
  a.row_begin = row_begin;
  a.rows_per_seq = rows_per_seq;
  a.tiles_per_seq = rows_per_seq / 128;
  a.kv_exp = kv_exp;
  a.status = status;
  const dim3 grid((unsigned)(B * a.tiles_per_seq), (unsigned)((g->H + kExpHeads - 1) / kExpHeads));
  return launch_pdl(normal_expand_kernel, grid, dim3(kExpThreads), kExpSmemAlloc, st, m_ckv, m_wuk, m_wuv, a);
}

cudaError_t launch_normal_expand(const mla_geom* g, const CacheView& cv, const int32_t* block_table, int bt_stride,
                                 const int32_t* seq_lens, int B, int max_pages, const __nv_bfloat16* w_uk,
                                 const __nv_bfloat16* w_uv, __nv_bfloat16* kv_exp, cudaStream_t st) {
  return launch_normal_expand_rows(g, cv, block_table, bt_stride, seq_lens, B, max_pages, 0,
                                   (int)normal_rows_per_seq(max_pages), w_uk, w_uv, kv_exp, st);
}

cudaError_t launch_normal_attention_window(const mla_geom* g, const mla_batch* bt, const __nv_bfloat16* q_nope,
                                           const __nv_bfloat16* q_pe, const CacheView& cv, const int32_t* block_table,
                                           int bt_stride, const int32_t* seq_lens, const __nv_bfloat16* kv_exp,
                                           int64_t rows_per_seq, int key_begin, int key_end, int has_prev,
                                           int final_out, float* st_o, float* st_lse, __nv_bfloat16* o, float* lse,
                                           cudaStream_t st) {
  int* status = bmm_status_ptr();
  if (!status) return cudaErrorInvalidValue;
  const int B = bt->B, T = bt->T, H = g->H;
  CUtensorMap m_qn, m_qp, m_kv, m_kpe;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kDNope, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t str[3] = {(cuuint64_t)kDNope * 2, (cuuint64_t)H * kDNope * 2, (cuuint64_t)T * H * kDNope * 2};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    if (!make_map_n(&m_qn, q_nope, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {(cuuint64_t)kDRope, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t str[3] = {(cuuint64_t)kDRope * 2, (cuuint64_t)H * kDRope * 2, (cuuint64_t)T * H * kDRope * 2};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    if (!make_map_n(&m_qp, q_pe, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t rows_cap = (cuuint64_t)B * rows_per_seq;
    const cuuint64_t dims[3] = {256, rows_cap, (cuuint64_t)H};
    const cuuint64_t str[2] = {256 * 2, rows_cap * 256 * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    if (!make_map_n(&m_kv, kv_exp, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kDRope, (cuuint64_t)kPage, (cuuint64_t)cv.num_blocks};
    const cuuint64_t str[2] = {(cuuint64_t)cv.kpe_row * 2, (cuuint64_t)cv.kpe_block * 2};
    const cuuint32_t box[3] = {64, 64, 1};
    if (!make_map_n(&m_kpe, cv.kpe, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(normal_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttSmemAlloc) !=
        cudaSuccess)
      return cudaErrorInvalidValue;
    attr = true;
  }
  AttArgs a;
  a.block_table = block_table; a.bt_stride = bt_stride; a.seq_lens = seq_lens;
  a.B = B; a.T = T; a.H = H; a.causal = bt->causal ? 1 : 0; a.max_pages = bt->max_pages;
  a.num_blocks = cv.num_blocks; a.rows_per_seq = (int)rows_per_seq;
  a.key_begin = key_begin; a.key_end = key_end;
  a.has_prev = has_prev; a.final_out = final_out; a.st_o = st_o; a.st_lse = st_lse;
  a.scale_log2 = g->softmax_scale * 1.4426950408889634f;
  a.o = o; a.lse = lse; a.status = status;
  const dim3 grid((unsigned)((T + 127) / 128), (unsigned)H, (unsigned)B);
  return launch_pdl(normal_attention_kernel, grid, dim3(kAttThreads), kAttSmemAlloc, st, m_qn, m_qp, m_kv, m_kpe, a);
}

cudaError_t launch_normal_attention(const mla_geom* g, const mla_batch* bt, const __nv_bfloat16* q_nope,
                                    const __nv_bfloat16* q_pe, const CacheView& cv, const int32_t* block_table,
                                    int bt_stride, const int32_t* seq_lens, const __nv_bfloat16* kv_exp,
                                    __nv_bfloat16* o, float* lse, cudaStream_t st) {
  return launch_normal_attention_window(g, bt, q_nope, q_pe, cv, block_table, bt_stride, seq_lens, kv_exp,
                                        normal_rows_per_seq(bt->max_pages), 0, INT_MAX, 0, 1, nullptr, nullptr, o,
                                        lse, st);
}

// The chunked-prefix Normal path: per window of chunk_rows cache rows, expand the
// window's latents (into kv_chunk, chunk_rows rows per sequence), then attend to
// the window's keys, merging into the running state; the last window writes o, lse.
cudaError_t launch_normal_chunked(const mla_geom* g, const mla_batch* bt, const __nv_bfloat16* q_nope,
                                  const __nv_bfloat16* q_pe, const CacheView& cv, const int32_t* block_table,
                                  int bt_stride, const int32_t* seq_lens, const __nv_bfloat16* w_uk,
                                  const __nv_bfloat16* w_uv, int chunk_rows, __nv_bfloat16* kv_chunk, float* st_o,
                                  float* st_lse, __nv_bfloat16* o, float* lse, cudaStream_t st) {
  const int64_t total = (int64_t)bt->max_pages * kPage;
  const int n_chunks = (int)((total + chunk_rows - 1) / chunk_rows);
  for (int c = 0; c < n_chunks; ++c) {
    const int j0 = c * chunk_rows;
    cudaError_t e = launch_normal_expand_rows(g, cv, block_table, bt_stride, seq_lens, bt->B, bt->max_pages, j0,
                                              chunk_rows, w_uk, w_uv, kv_chunk, st);
    if (e != cudaSuccess) return e;
    e = launch_normal_attention_window(g, bt, q_nope, q_pe, cv, block_table, bt_stride, seq_lens, kv_chunk,
                                       chunk_rows, j0, j0 + chunk_rows, c > 0 ? 1 : 0, c == n_chunks - 1 ? 1 : 0,
                                       st_o, st_lse, o, lse, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace mla
