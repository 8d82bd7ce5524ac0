// Absorption GEMMs on the sm_103a tensor cores ("M5.8" 0x04 batched
// absorption trace; "MLA in full detail" Steps 2 and 4):
//   absorb   : q_lat[r,h,c] = sum_n q_nope[r,h,n] W_UK[h,n,c]   (K = 128, N = 512)
//   un-absorb: o[r,h,v]     = sum_c o_lat[r,h,c] W_UV[h,v,c]    (K = 512, N = 128)
// Per head these are [BT x K] x [K x N] products, batched over the H heads.
// They are bound by reading the weights (16.8 MB each at V3 geometry) when
// the token count BT is small, so each CTA streams one head's weight slice
// once through TMA and accumulates a 128-token x N-tile block in TMEM.
//
// CTA = 128 threads: warp 0 lane 0 issues TMA loads through a ring of k-step
// slots (one 64-wide slice of K per slot), warp 1 lane 0 issues the MMAs
// (M = 128 tokens, N = the CTA's N tile, K = 16 per instruction), then all
// four warps read the accumulator (one token row per TMEM lane) and store
// bf16.  Token rows past BT read as zeros through the tensor map and are not
// stored.  W_UK is [H, n, c] with c contiguous, i.e. MN-major for this
// product; W_UV is [H, v, c], K-major.
#include "mla_internal.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kThreads = 128;
constexpr int kRing = 4;
constexpr int kABox = 128 * 64 * 2;  // 128 token rows x 64 K values

template <int KB, int NT, int BMN>
struct Cfg {
  static constexpr int kBBytes = NT * 64 * 2;          // one 64-wide K slice of the B tile
  static constexpr int kSlot = kABox + kBBytes;
  static constexpr int kSlots = KB < kRing ? KB : kRing;
  static constexpr int kSmemBar = kSlots * kSlot;
  static constexpr int kSmemAlloc = kSmemBar + 256 + 1024;
};

template <int KB, int NT, int BMN>
__global__ void __launch_bounds__(kThreads, 1)
    bmm_sm103_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     __nv_bfloat16* out, int BT, int H, int n_total, int* status) {
  using C = Cfg<KB, NT, BMN>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_addr(smem);
  auto slot_a = [&](int s) { return base + s * C::kSlot; };
  auto slot_b = [&](int s) { return base + s * C::kSlot + kABox; };
  auto bar = [&](int i) { return base + C::kSmemBar + 8 * i; };  // 0..S-1 full, S..2S-1 empty, 2S done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kSmemBar + 8 * (2 * C::kSlots + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kSmemBar + 8 * (2 * C::kSlots + 1) + 4);

  const int h = blockIdx.x, n0 = blockIdx.y * NT, m0 = blockIdx.z * 128;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(s), 1);
      mbar_init(bar(C::kSlots + s), 1);
    }
    mbar_init(bar(2 * C::kSlots), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), NT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  // The weights are no kernel's output, so the first ring's worth of weight
  // k-steps is requested before waiting on the previous kernel in the stream
  // (in a decode step, the planner): their streaming overlaps that kernel.
  if (warp == 0 && lane == 0) {
    for (int kb = 0; kb < C::kSlots; ++kb) {
      mbar_arrive_expect_tx(bar(kb), C::kSlot);
      if (BMN) {
        for (int j = 0; j < NT / 64; ++j) tma_load_3d(slot_b(kb) + j * 8192, &tm_b, bar(kb), n0 + 64 * j, 64 * kb, h);
      } else {
        tma_load_3d(slot_b(kb), &tm_b, bar(kb), 64 * kb, n0, h);
      }
    }
  }
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % C::kSlots;
        if (kb < C::kSlots) {  // weight slice already requested
          tma_load_3d(slot_a(s), &tm_a, bar(s), 64 * kb, h, m0);
          ++issued;
          continue;
        }
        if (!mbar_wait(bar(C::kSlots + s), ((kb / C::kSlots) & 1) ^ 1, abort_flag)) {
          *abort_flag = 1;
          atomicCAS(status, 0, MLA_ERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(bar(s), C::kSlot);
        tma_load_3d(slot_a(s), &tm_a, bar(s), 64 * kb, h, m0);
        if (BMN) {
          // W_UK[h]: K rows 64kb.., N columns n0..n0+NT in 64-wide boxes of 64 K rows
          for (int j = 0; j < NT / 64; ++j) tma_load_3d(slot_b(s) + j * 8192, &tm_b, bar(s), n0 + 64 * j, 64 * kb, h);
        } else {
          // W_UV[h]: N rows n0..n0+NT (<= 256 per box) of the 64-wide K slice
          tma_load_3d(slot_b(s), &tm_b, bar(s), 64 * kb, n0, h);
        }
        ++issued;
      }
      const int first = issued > C::kSlots ? issued - C::kSlots : 0;
      for (int g = first; g < issued; ++g) {
        volatile int never = 0;
        mbar_wait(bar(g % C::kSlots), (g / C::kSlots) & 1, &never);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, NT, BMN);
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % C::kSlots;
        if (!mbar_wait(bar(s), (kb / C::kSlots) & 1, abort_flag)) {
          *abort_flag = 1;
          atomicCAS(status, 0, MLA_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sw128_desc(slot_a(s) + 32 * kk, 16, 1024);
          const uint64_t bd = BMN ? sw128_desc(slot_b(s) + 2048 * kk, 8192, 1024) : sw128_desc(slot_b(s) + 32 * kk, 16, 1024);
          mma_bf16(tmem, ad, bd, idesc, (kb | kk) ? 1u : 0u);
        }
        mma_commit(bar(C::kSlots + s));
      }
      mma_commit(bar(2 * C::kSlots));
    }
    __syncwarp();
  }
  // Epilogue: all four warps, one token row per TMEM lane.
  {
    const bool w_ok = mbar_wait(bar(2 * C::kSlots), 0, abort_flag);
    ok = __all_sync(0xffffffffu, w_ok) && ok;
    tc_fence_after();
    if (ok) {
      const int row = 32 * warp + lane;
      const int tok = m0 + row;
      const uint32_t t_lane = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
      for (int c = 0; c < NT / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(t_lane + 32 * c, v);
        tmem_wait_ld();
        if (tok < BT) {
          __nv_bfloat16* dst = out + ((size_t)tok * H + h) * n_total + n0 + 32 * c;
#pragma unroll
          for (int e = 0; e < 32; e += 16) {
            uint32_t w[8];
            pack_bf16x8(v + e, 1.f, w);
            pack_bf16x8(v + e + 8, 1.f, w + 4);
            st_global_v8(dst + e, w);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, NT);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_map3(CUtensorMap* m, const void* base, cuuint64_t d0, cuuint64_t d1, cuuint64_t d2, cuuint64_t s1_bytes,
               cuuint64_t s2_bytes, cuuint32_t b0, cuuint32_t b1, cuuint32_t b2) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t str[2] = {s1_bytes, s2_bytes};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, str, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KB, int NT, int BMN>
cudaError_t launch_bmm(const CUtensorMap& ma, const CUtensorMap& mb, __nv_bfloat16* out, int BT, int H, int n_total,
                       int* status, cudaStream_t st) {
  using C = Cfg<KB, NT, BMN>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(bmm_sm103_kernel<KB, NT, BMN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(H, n_total / NT, (BT + 127) / 128);
  return launch_pdl(bmm_sm103_kernel<KB, NT, BMN>, grid, dim3(kThreads), C::kSmemAlloc, st, ma, mb, out, BT, H,
                    n_total, status);
}

__device__ int g_bmm_status;  // timeouts of these kernels (they have no workspace)

}  // namespace

// Device address of the absorption kernels' status word on the current device.
int* bmm_status_ptr() {
  static int* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bmm_status) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(p);
  }
  return cached[dev];
}

cudaError_t launch_absorb_sm103(const __nv_bfloat16* q_nope, const __nv_bfloat16* w_uk, __nv_bfloat16* q_lat, int BT,
                                int H, cudaStream_t st) {
  int* status = bmm_status_ptr();
  if (!status) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  // A = q_nope viewed as (n: 128, h: H, token: BT), box 64 x 1 x 128 tokens
  if (!make_map3(&ma, q_nope, kDNope, H, BT, (cuuint64_t)kDNope * 2, (cuuint64_t)H * kDNope * 2, 64, 1, 128))
    return cudaErrorInvalidValue;
  // B = W_UK viewed as (c: 512, n: 128, h: H), box 64 c x 64 n x 1
  if (!make_map3(&mb, w_uk, kDLat, kDNope, H, (cuuint64_t)kDLat * 2, (cuuint64_t)kDNope * kDLat * 2, 64, 64, 1))
    return cudaErrorInvalidValue;
  return launch_bmm<kDNope / 64, 256, 1>(ma, mb, q_lat, BT, H, kDLat, status, st);
}

cudaError_t launch_unabsorb_sm103(const __nv_bfloat16* o_lat, const __nv_bfloat16* w_uv, __nv_bfloat16* o, int BT,
                                  int H, cudaStream_t st) {
  int* status = bmm_status_ptr();
  if (!status) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  // A = o_lat viewed as (c: 512, h: H, token: BT), box 64 x 1 x 128
  if (!make_map3(&ma, o_lat, kDLat, H, BT, (cuuint64_t)kDLat * 2, (cuuint64_t)H * kDLat * 2, 64, 1, 128))
    return cudaErrorInvalidValue;
  // B = W_UV viewed as (c: 512, v: 128, h: H), box 64 c x 128 v x 1 (K-major rows of v)
  if (!make_map3(&mb, w_uv, kDLat, kDV, H, (cuuint64_t)kDLat * 2, (cuuint64_t)kDV * kDLat * 2, 64, 128, 1))
    return cudaErrorInvalidValue;
  return launch_bmm<kDLat / 64, 128, 0>(ma, mb, o, BT, H, kDV, status, st);
}

}  // namespace mla
