// Test export: copy a sequence's logical rows, in order, through the paged
// address translation the decode kernels use ("M5.8" 0x05).
#include "mla_internal.cuh"

namespace mla {
namespace {

__global__ void debug_gather_kernel(CacheView cv, const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                                    int b, __nv_bfloat16* out) {
  const int S = seq_lens[b];
  for (int j = blockIdx.x; j < S; j += gridDim.x) {
    if (j / kPage >= bt_stride) break;
    const int blk = block_table[(size_t)b * bt_stride + j / kPage];
    if (blk < 0 || blk >= cv.num_blocks) continue;
    const int jp = j % kPage;
    for (int c8 = threadIdx.x * 8; c8 < kDK; c8 += blockDim.x * 8) {
      const uint4 v = c8 < kDLat ? *reinterpret_cast<const uint4*>(ckv_row_ptr(cv, blk, jp) + c8)
                                 : *reinterpret_cast<const uint4*>(kpe_row_ptr(cv, blk, jp) + (c8 - kDLat));
      *reinterpret_cast<uint4*>(out + (size_t)j * kDK + c8) = v;
    }
  }
}

}  // namespace

cudaError_t launch_debug_gather(const CacheView& cv, const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                                int b, __nv_bfloat16* out, cudaStream_t st) {
  debug_gather_kernel<<<1024, 96, 0, st>>>(cv, block_table, bt_stride, seq_lens, b, out);
  return cudaGetLastError();
}

}  // namespace mla
