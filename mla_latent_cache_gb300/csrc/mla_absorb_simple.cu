// Plain CUDA-core absorption GEMMs ("M5.8" 0x04 batched absorption trace):
//   q_lat[r,h,c] = sum_n q_nope[r,h,n] W_UK[h,n,c]      (absorb, K = 128, N = 512)
//   o[r,h,v]     = sum_c o_lat[r,h,c] W_UV[h,v,c]       (un-absorb, K = 512, N = 128)
// fp32 accumulation from bf16 operands, bf16 output.
#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kRT = 32;   // token rows per CTA
constexpr int kCT = 128;  // output columns per CTA

// grid (H, N/kCT, ceil(BT/kRT)); out[r, h, c] = sum_k x[r, h, k] * w(h, k, c)
// with w(h,k,c) = W[h, k, c] (absorb: W_UK [H,128,512]) or W[h, c, k] (un-absorb: W_UV [H,128,512]).
template <int K, int N, bool kTransW>
__global__ void __launch_bounds__(kThreads) bmm_kernel(const __nv_bfloat16* x, const __nv_bfloat16* w,
                                                       __nv_bfloat16* out, int BT, int H) {
  __shared__ __nv_bfloat16 xs[kRT][K + 2];
  __shared__ __nv_bfloat16 ws[32][kCT + 8];
  const int h = blockIdx.x, c0 = blockIdx.y * kCT, r0 = blockIdx.z * kRT;
  const int tid = threadIdx.x;
  for (int i = tid; i < kRT * K; i += kThreads) {
    const int rr = i / K, k = i % K;
    xs[rr][k] = (r0 + rr < BT) ? x[((size_t)(r0 + rr) * H + h) * K + k] : __float2bfloat16(0.f);
  }
  // thread -> (row rr = tid / 8, 16 columns starting at (tid % 8) * 16)
  const int rr = tid / 8, cc = (tid % 8) * 16;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int k0 = 0; k0 < K; k0 += 32) {
    __syncthreads();
    for (int i = tid; i < 32 * kCT; i += kThreads) {
      const int kk = i / kCT, c = i % kCT;
      const size_t idx = kTransW ? ((size_t)h * N + (c0 + c)) * K + (k0 + kk) : ((size_t)h * K + (k0 + kk)) * N + (c0 + c);
      ws[kk][c] = w[idx];
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < 32; ++kk) {
      const float xv = __bfloat162float(xs[rr][k0 + kk]);
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = fmaf(xv, __bfloat162float(ws[kk][cc + i]), acc[i]);
    }
  }
  if (r0 + rr < BT) {
    __nv_bfloat16* dst = out + ((size_t)(r0 + rr) * H + h) * N + c0 + cc;
#pragma unroll
    for (int i = 0; i < 16; i += 2)
      *reinterpret_cast<__nv_bfloat162*>(dst + i) = __floats2bfloat162_rn(acc[i], acc[i + 1]);
  }
}

}  // namespace

cudaError_t launch_absorb(const __nv_bfloat16* q_nope, const __nv_bfloat16* w_uk, __nv_bfloat16* q_lat, int BT,
                          int H, cudaStream_t st) {
  if (BT <= 0) return cudaSuccess;
  dim3 grid(H, kDLat / kCT, (BT + kRT - 1) / kRT);
  bmm_kernel<kDNope, kDLat, false><<<grid, kThreads, 0, st>>>(q_nope, w_uk, q_lat, BT, H);
  return cudaGetLastError();
}

cudaError_t launch_unabsorb(const __nv_bfloat16* o_lat, const __nv_bfloat16* w_uv, __nv_bfloat16* o, int BT, int H,
                            cudaStream_t st) {
  if (BT <= 0) return cudaSuccess;
  dim3 grid(H, kDV / kCT, (BT + kRT - 1) / kRT);
  bmm_kernel<kDLat, kDV, true><<<grid, kThreads, 0, st>>>(o_lat, w_uv, o, BT, H);
  return cudaGetLastError();
}

}  // namespace mla
