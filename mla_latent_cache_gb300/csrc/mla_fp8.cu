// FP8 latent cache rows ("M5.8" 0x0B "FP8 Cache Format And Sparse Selection",
// "Exact 656-byte FP8 row"): 512 E4M3 latent codes, 4 fp32 scales and the 64
// bf16 RoPE values, 656 bytes per token (against 1152 for bf16 rows).
//
// Row layout (bytes): [0, 512) codes, latent value i in byte i; [512, 528) the
// four scales, scale t covering latent values [128 t, 128 t + 128); [528, 656)
// the RoPE values, bf16 little-endian.  Scale t = (largest |value| of its
// tile) / 448 rounded once to fp32 (1 for an all-zero tile); code = the E4M3
// value nearest to the exact quotient value / scale, ties to the even mantissa,
// saturated at +-448.  A row decodes as latent value i = E4M3(code i) * scale.
// The code is decided exactly: the fp32 quotient (one rounding) gives a
// candidate that is the exact answer or a neighbour of it, and the sign of
// fma(midpoint, scale, -|value|) (one rounding of an exact product minus
// |value|, so its sign is exact) says on which side of each neighbouring
// midpoint |value| lies.
//
// This kernel packs a bf16 pool (combined or split) into such rows, HBM-bound:
// 1152 bytes read and 656 written per row.  One warp per row: lane l owns
// latent values [16 l, 16 l + 16) (tile l / 8, its amax reduced over the 8
// lanes of the tile); lanes 0..7 also move 8 RoPE values each.
#include <cuda_fp8.h>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kFp8RowBytes = 656;
constexpr int kFp8Threads = 256;

// Magnitude of the non-negative E4M3 code c (0 .. 0x7E): exact in fp32.
__device__ __forceinline__ float e4m3_magnitude(uint32_t c) {
  const uint32_t e = c >> 3, m = c & 7u;
  // subnormal: m * 2^-9; normal: (8 + m) * 2^(e - 10)
  const float p2 = __uint_as_float((uint32_t)(127 + (e ? (int)e - 10 : -9)) << 23);
  return (float)(e ? 8u + m : m) * p2;
}

// E4M3 byte nearest to the exact quotient x / scale (scale > 0, finite), ties to
// the even mantissa, saturating at +-448.
__device__ __forceinline__ uint32_t e4m3_nearest(float x, float scale) {
  const __nv_fp8_storage_t c0 = __nv_cvt_float_to_fp8(__fdiv_rn(x, scale), __NV_SATFINITE, __NV_E4M3);
  const uint32_t sign = (uint32_t)c0 & 0x80u;
  uint32_t c = (uint32_t)c0 & 0x7Fu;
  const float a = fabsf(x);
  const float y = e4m3_magnitude(c);
  if (c < 0x7Eu) {
    const float mid = 0.5f * (y + e4m3_magnitude(c + 1));
    const float r = fmaf(mid, scale, -a);           // > 0: below the midpoint; 0: on it
    if (r < 0.f || (r == 0.f && (c & 1u))) c += 1;
  }
  if (c > 0u && c == ((uint32_t)c0 & 0x7Fu)) {
    const float mid = 0.5f * (e4m3_magnitude(c - 1) + y);
    const float r = fmaf(mid, scale, -a);
    if (r > 0.f || (r == 0.f && (c & 1u))) c -= 1;
  }
  return sign | c;
}

__global__ void __launch_bounds__(kFp8Threads) fp8_pack_kernel(CacheView cv, unsigned char* out) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)cv.num_blocks * kPage;
  const long long warps = (long long)gridDim.x * (kFp8Threads / 32);
  for (long long r = (long long)blockIdx.x * (kFp8Threads / 32) + (threadIdx.x >> 5); r < rows; r += warps) {
    const int blk = (int)(r / kPage), j = (int)(r % kPage);
    const __nv_bfloat16* src = ckv_row_ptr(cv, blk, j) + 16 * lane;
    const uint4 u0 = *reinterpret_cast<const uint4*>(src);
    const uint4 u1 = *reinterpret_cast<const uint4*>(src + 8);
    float x[16];
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint32_t packed[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t v = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v |= e4m3_nearest(x[4 * k + e], scale) << (8 * e);
      }
      packed[k] = v;
    }
    unsigned char* dst = out + r * kFp8RowBytes;
    *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if ((lane & 7) == 0) *reinterpret_cast<float*>(dst + kDLat + 4 * (lane >> 3)) = scale;
    if (lane < 8) {
      const __nv_bfloat16* kp = cv.kpe + (int64_t)blk * cv.kpe_block + (int64_t)j * cv.kpe_row + 8 * lane;
      *reinterpret_cast<uint4*>(dst + kDLat + 16 + 16 * lane) = *reinterpret_cast<const uint4*>(kp);
    }
  }
}

}  // namespace

cudaError_t launch_fp8_pack(const CacheView& cv, unsigned char* out, cudaStream_t st) {
  const long long rows = (long long)cv.num_blocks * kPage;
  const int sms = mla_device_sm_count();
  long long ctas = (rows + (kFp8Threads / 32) - 1) / (kFp8Threads / 32);
  const long long cap = 8LL * (sms > 0 ? sms : 148);
  if (ctas > cap) ctas = cap;
  return launch_pdl(fp8_pack_kernel, dim3((unsigned)ctas), dim3(kFp8Threads), 0, st, cv, out);
}

}  // namespace mla
