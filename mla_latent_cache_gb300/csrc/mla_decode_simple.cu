// Plain CUDA-core split-KV decode: one CTA per (work range, 16-row slice of a
// 128-row group).  It is the first correct path and the arithmetic baseline
// the tensor-core kernel is checked against on the GPU; it reads each key
// tile once per 16-row slice.
//
// Per segment (b, rb, pages [p0, p1)): for each 32-key tile, scores
// s = (q_lat . c_j + q_pe . k_pe_j) * scale are formed in fp32 from bf16
// operands, masked by the causal limit, folded into a running (m, l) online
// softmax ("M5.8" 0x0A/0x0C: rescale prior state when the running max changes),
// and p_j * c_j is accumulated into fp32 registers.
#include <math.h>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kSR = 16;        // query rows per CTA
constexpr int kKT = 32;        // keys per tile
constexpr int kThreads = 256;
constexpr int kKStride = kDK + 8;  // padded smem row (bf16) to spread banks

struct DecodeArgs {
  const __nv_bfloat16* q_lat;
  const __nv_bfloat16* q_pe;
  CacheView cv;
  const int32_t* block_table;
  int bt_stride;
  const int32_t* seq_lens;
  int B, T, H, causal, checked, max_pages;
  float scale;
  __nv_bfloat16* o_lat;
  float* lse;
  WsLayout L;
};

struct __align__(16) Smem {
  float q[kSR][kDK];                 // 36 KB
  __nv_bfloat16 k[kKT][kKStride];    // 36.5 KB
  float p[kSR][kKT];
  float alpha[kSR];
  int limit[kSR];
  int blk[kKT];
};

__global__ void __launch_bounds__(kThreads) decode_simple_kernel(DecodeArgs a, char* ws) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  int* hdr = reinterpret_cast<int*>(ws);
  const int* seg = reinterpret_cast<const int*>(ws + a.L.off_segments);
  const int* rptr = reinterpret_cast<const int*>(ws + a.L.off_range_ptr);
  float* part_lse = reinterpret_cast<float*>(ws + a.L.off_part_lse);
  float* part_o = reinterpret_cast<float*>(ws + a.L.off_part_o);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = blockIdx.y;
  const int num_ranges = hdr[MLA_HDR_NUM_RANGES];
  const int R = a.T * a.H;

  if (a.checked && blockIdx.x == 0 && sub == 0 && tid == 0) {
    if (hdr[MLA_HDR_MAGIC] != MLA_PLAN_MAGIC || hdr[MLA_HDR_B] != a.B || hdr[MLA_HDR_T] != a.T ||
        hdr[MLA_HDR_H] != a.H || hdr[MLA_HDR_CAUSAL] != a.causal) {
      record_error(hdr, MLA_ERR_PLAN_STALE, 0);
    } else {
      // Re-derive the length stamp and compare.
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

  for (int r = blockIdx.x; r < num_ranges; r += gridDim.x) {
    for (int si = rptr[r]; si < rptr[r + 1]; ++si) {
      const int* rec = seg + (size_t)si * kSegWords;
      const int b = rec[0], rb = rec[1], p0 = rec[2], p1 = rec[3], slot = rec[5];
      const int row0 = rb * kRowsPerBlock + sub * kSR;   // flat row within the sequence
      const int nrows = min(kSR, R - row0);
      if (nrows <= 0) continue;
      int S = a.seq_lens[b];
      S = S < 0 ? 0 : min(S, a.max_pages * kPage);
      __syncthreads();
      // Stage the 16 query rows as fp32: [q_lat (512) | q_pe (64)].
      for (int i = tid; i < kSR * kDK; i += kThreads) {
        const int rr = i / kDK, c = i % kDK;
        float v = 0.f;
        if (rr < nrows) {
          const size_t grow = (size_t)b * R + row0 + rr;
          v = c < kDLat ? __bfloat162float(a.q_lat[grow * kDLat + c])
                        : __bfloat162float(a.q_pe[grow * kDRope + (c - kDLat)]);
        }
        sm.q[rr][c] = v;
      }
      if (tid < kSR) {
        const int t = (row0 + tid) / a.H;
        sm.limit[tid] = tid < nrows ? visible_limit(S, a.T, t, a.causal) : 0;
      }
      // Running state: warp w owns rows 2w, 2w+1 for the softmax; for the
      // accumulation thread owns row tid/16 and 32 columns.
      const int my_row = tid / 16;
      const int my_col0 = (tid % 16) * 32;
      float acc[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) acc[c] = 0.f;
      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
      const int j_begin = p0 * kPage, j_end = min(S, p1 * kPage);
      __syncthreads();
      for (int j0 = j_begin; j0 < j_end; j0 += kKT) {
        // Resolve block ids for this tile (a 32-key tile lies inside one page).
        if (tid < kKT) {
          const int j = j0 + tid;
          int blk = -1;
          if (j < j_end) {
            blk = a.block_table[(size_t)b * a.bt_stride + j / kPage];
            if (a.checked && (blk < 0 || blk >= a.cv.num_blocks)) {
              record_error(hdr, MLA_ERR_DEVICE_CHECK, (b << 16) | (j / kPage));
              blk = -1;
            }
          }
          sm.blk[tid] = blk;
        }
        __syncthreads();
        for (int i = tid; i < kKT * (kDK / 8); i += kThreads) {
          const int kk = i / (kDK / 8), c8 = (i % (kDK / 8)) * 8;
          const int blk = sm.blk[kk];
          uint4 v = make_uint4(0, 0, 0, 0);
          if (blk >= 0) {
            const int jp = (j0 + kk) % kPage;
            v = c8 < kDLat ? *reinterpret_cast<const uint4*>(ckv_row_ptr(a.cv, blk, jp) + c8)
                           : *reinterpret_cast<const uint4*>(kpe_row_ptr(a.cv, blk, jp) + (c8 - kDLat));
          }
          *reinterpret_cast<uint4*>(&sm.k[kk][c8]) = v;
        }
        __syncthreads();
        // Scores and online softmax: warp w handles rows 2w and 2w+1, lane = key.
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int rr = warp * 2 + h2;
          const int j = j0 + lane;
          float s = -INFINITY;
          if (rr < nrows && j < j_end && j < sm.limit[rr] && sm.blk[lane] >= 0) {
            float dot = 0.f;
            const float* qv = sm.q[rr];
            const __nv_bfloat16* kv = sm.k[lane];
            for (int c = 0; c < kDK; c += 2) {
              const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(kv + c));
              dot = fmaf(qv[c], kf.x, dot);
              dot = fmaf(qv[c + 1], kf.y, dot);
            }
            s = dot * a.scale;
          }
          float tmax = s;
#pragma unroll
          for (int o = 16; o; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
          const float m_new = fmaxf(m_run[h2], tmax);
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          const float p = (s == -INFINITY) ? 0.f : __expf(s - m_use);
          const float alpha = (m_run[h2] == -INFINITY) ? 0.f : __expf(m_run[h2] - m_use);
          float psum = p;
#pragma unroll
          for (int o = 16; o; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
          l_run[h2] = l_run[h2] * alpha + psum;
          m_run[h2] = m_new;
          sm.p[rr][lane] = p;
          if (lane == 0) sm.alpha[rr] = alpha;
        }
        __syncthreads();
        // Accumulate p . c for this thread's row and 32 latent columns.
        {
          const float al = sm.alpha[my_row];
#pragma unroll
          for (int c = 0; c < 32; ++c) acc[c] *= al;
          for (int kk = 0; kk < kKT; ++kk) {
            const float p = sm.p[my_row][kk];
            if (p != 0.f) {
              const __nv_bfloat16* kv = &sm.k[kk][my_col0];
#pragma unroll
              for (int c = 0; c < 32; c += 2) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(kv + c));
                acc[c] = fmaf(p, f.x, acc[c]);
                acc[c + 1] = fmaf(p, f.y, acc[c + 1]);
              }
            }
          }
        }
        __syncthreads();
      }
      // Publish (m, l) per row, then normalise and write.
      __shared__ float s_l[kSR], s_m[kSR];
      if (lane == 0) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          s_l[warp * 2 + h2] = l_run[h2];
          s_m[warp * 2 + h2] = m_run[h2];
        }
      }
      __syncthreads();
      if (my_row < nrows) {
        const float l = s_l[my_row];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float lse_v = l > 0.f ? s_m[my_row] + logf(l) : -INFINITY;
        const int local_row = sub * kSR + my_row;
        if (slot < 0) {
          const size_t grow = (size_t)b * R + rb * kRowsPerBlock + local_row;
          __nv_bfloat16* dst = a.o_lat + grow * kDLat + my_col0;
#pragma unroll
          for (int c = 0; c < 32; c += 2)
            *reinterpret_cast<__nv_bfloat162*>(dst + c) = __floats2bfloat162_rn(acc[c] * inv, acc[c + 1] * inv);
          if (my_col0 == 0) a.lse[grow] = lse_v;
        } else {
          float* dst = part_o + ((size_t)slot * kRowsPerBlock + local_row) * kDLat + my_col0;
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4*>(dst + c) = make_float4(acc[c] * inv, acc[c + 1] * inv, acc[c + 2] * inv, acc[c + 3] * inv);
          if (my_col0 == 0) part_lse[(size_t)slot * kRowsPerBlock + local_row] = lse_v;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_decode_simple(const mla_geom* g, const mla_batch* b, const WsLayout& L,
                                 const __nv_bfloat16* q_lat, const __nv_bfloat16* q_pe, const CacheView& cv,
                                 const int32_t* block_table, int bt_stride, const int32_t* seq_lens, int checked,
                                 __nv_bfloat16* o_lat, float* lse, void* ws, cudaStream_t st) {
  DecodeArgs a;
  a.q_lat = q_lat; a.q_pe = q_pe; a.cv = cv; a.block_table = block_table; a.bt_stride = bt_stride;
  a.seq_lens = seq_lens; a.B = b->B; a.T = b->T; a.H = g->H; a.causal = b->causal ? 1 : 0;
  a.checked = checked; a.max_pages = b->max_pages; a.scale = g->softmax_scale;
  a.o_lat = o_lat; a.lse = lse; a.L = L;
  const size_t smem = sizeof(Smem);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_simple_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int rows_per_group = min(kRowsPerBlock, b->T * g->H);
  const int subs = (rows_per_group + kSR - 1) / kSR;
  dim3 grid(L.cap_ranges, subs);
  if (L.cap_ranges <= 0) return cudaSuccess;
  decode_simple_kernel<<<grid, kThreads, smem, st>>>(a, reinterpret_cast<char*>(ws));
  return cudaGetLastError();
}

}  // namespace mla
