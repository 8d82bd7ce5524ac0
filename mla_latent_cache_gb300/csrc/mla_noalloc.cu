// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run a
// decode step: code inside a custom allocator or a memory-pool callback, a
// runtime that forbids allocation once a serving loop has started (so that
// memory use stays fixed), or a host environment whose only device buffers are
// the inputs and outputs it was handed.  For them, mla_decode_noalloc plans and
// runs the split-KV decode (and its merge) in a fixed scratch array that lives
// in this library's device image instead of in a caller-allocated workspace.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes; every
// GPU that loads the library holds it until the process exits.  Host code may
// not pass the array's name to a kernel (on the host it is only a stand-in
// symbol), so the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device.  Make that first call before any stream capture begins.
//
// Every call on a device shares the one array and leaves its contents behind.
// Nothing in it needs to start at zero: the planning step rewrites every word
// of the plan and the status word that the decode and merge kernels read, and
// the decode kernel writes each partial slot before the merge reads it.  Calls
// whose work overlaps on the GPU (different streams, or different host threads
// without ordering) race on the array; callers must order them.
//
// Errors the kernels see (a length beyond the block table, T > S_b, a wait that
// ran out) land in the scratch's status word, which mla_read_device_status
// returns, and clears, when it is called without a workspace.
#include <mutex>

#include "mla_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = MLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array for the current device (looked up once per device).
mla_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MLA_OK;
}

}  // namespace

namespace mla {

int* noalloc_status_words() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) return nullptr;
  return static_cast<int*>(g_scratch_ptr[dev]) + MLA_HDR_ERROR;   // {status, detail}
}

}  // namespace mla

extern "C" mla_status mla_decode_noalloc(const mla_geom* geom, const mla_batch* batch, const void* q_lat,
                                         const void* q_pe, const mla_cache* cache, const int32_t* block_table,
                                         int bt_stride, const int32_t* seq_lens, void* o_lat, float* lse,
                                         mla_stream_t stream) {
  // Every host-side check of the decode runs before anything is launched.
  mla::CacheView cv;
  mla_status s = mla::check_decode_args(geom, batch, q_lat, q_pe, cache, block_table, bt_stride, seq_lens, o_lat,
                                        lse, &cv);
  if (s != MLA_OK) return s;
  mla_batch local = *batch;
  if (local.num_slots == 0 && local.num_splits_override == 0) {
    // The default (one work range per CTA pair) needs 2 x 128 x 512 fp32 partial
    // rows per range, more than the scratch holds on a large GPU: take the largest
    // range count whose workspace fits.
    int G = mla::resolve_slots(&local);
    for (; G > 1; --G) {
      local.num_slots = G;
      const size_t n = mla_workspace_size(geom, &local);
      if (n != 0 && n <= kNoAllocScratchBytes) break;
    }
    local.num_slots = G;
  }
  const size_t need = mla_workspace_size(geom, &local);
  if (need == 0) return MLA_ERR_ARG;
  if (need > kNoAllocScratchBytes) return MLA_ERR_WORKSPACE;  // batch needs more than the fixed scratch
  if (local.B == 0) return MLA_OK;
  void* scratch = nullptr;
  s = scratch_for_current_device(&scratch);
  if (s != MLA_OK) return s;
  s = mla_plan(geom, &local, seq_lens, scratch, kNoAllocScratchBytes, stream);
  if (s != MLA_OK) return s;
  return mla_decode(geom, &local, q_lat, q_pe, cache, block_table, bt_stride, seq_lens, /*checked=*/0, o_lat, lse,
                    scratch, kNoAllocScratchBytes, stream);
}
