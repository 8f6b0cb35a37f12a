// no_alloc.cu -- paged_decode_attention_static: decode attention whose scratch
// space lives in a fixed array inside the library instead of a caller buffer.
//
// Why it exists: some callers cannot allocate device memory at the point where
// they run decode attention -- for example code that runs under an allocator
// that is frozen while a CUDA graph is being recorded, a plugin that is handed
// only input and output buffers by its host framework, or a real-time loop
// that forbids any allocation after start-up.  paged_decode_attention needs a
// workspace for the partial results of split sequences; this entry point takes
// that workspace from the array below, so the caller passes only inputs and
// outputs.  It calls no allocating routine at all.
//
// Costs and limits:
//   - The array is kPkvStaticScratchBytes (16 MiB) and every GPU that loads
//     this library holds it until the process exits.
//   - A call whose workspace would not fit is rejected with PKV_ENOMEM before
//     anything is launched (paged_decode_workspace_bytes gives an upper bound
//     of the need).
//   - Every call on a device shares the one array and it keeps whatever the
//     last call left in it.  Nothing in it has to start at zero: every partial
//     result and every per-sequence record the merge reads is written earlier
//     in the same call.  Calls whose kernels can overlap on the GPU (different
//     streams without ordering between them) race on the array; serialise them.
//   - The first call on each device looks the array's device address up with
//     cudaGetSymbolAddress, with that device current.  Make that first call
//     before any stream capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv.h"

namespace {

constexpr size_t kPkvStaticScratchBytes = PKV_STATIC_SCRATCH_BYTES;
static_assert(kPkvStaticScratchBytes == (size_t)16 << 20, "header and array disagree");

// The scratch array.  In host code this name is only a stand-in for the
// device symbol, never a device address: kernels get the address looked up
// below.
static __device__ __align__(256) unsigned char g_pkv_static_scratch[kPkvStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the array on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ECUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_static_scratch) != cudaSuccess || !p) return PKV_ECUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" int paged_decode_attention_static(void* d_out, pkv_dtype out_dtype, const void* d_q,
                                             pkv_dtype q_dtype, const pkv_pool* pool, int layer,
                                             const int32_t* d_block_tables,
                                             int max_blocks_per_seq, const int32_t* d_seq_lens,
                                             int batch, int max_seq_len, float scale,
                                             float k_scale, float v_scale, int num_splits,
                                             cudaStream_t stream) {
  if (!pool) return PKV_EINVAL;
  void* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc != PKV_OK) return rc;
  // paged_decode_attention checks the workspace its launch plan needs against
  // the array's size and returns PKV_ENOMEM before launching anything if it is short.
  return paged_decode_attention(d_out, out_dtype, d_q, q_dtype, pool, layer, d_block_tables,
                                max_blocks_per_seq, d_seq_lens, batch, max_seq_len, scale,
                                k_scale, v_scale, num_splits, ws, kPkvStaticScratchBytes, stream);
}
