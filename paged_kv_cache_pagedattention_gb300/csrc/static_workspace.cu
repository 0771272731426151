// pa_decode_static_workspace: PagedAttention decode whose split-K scratch lives in
// a fixed array inside the library instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the point where they
// run attention -- for example an inference runtime whose memory planner hands out
// only the tensors it planned for (inputs, outputs, KV cache) and has no slot for
// an operator's scratch, or a plug-in that must not call cudaMalloc (or a caching
// allocator) on the serving path because that can synchronise the device or fail
// when the pool is exhausted.  Such a caller passes only inputs and outputs.
//
// The scratch is PA_STATIC_WORKSPACE_BYTES (include/pa.h) of device memory that
// every GPU which loads this library holds until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_ptr[kMaxDevices] = {};

// Device address of the array on the current device; looked up once per device
// (the first call on a device does it, with that device current).
void* static_workspace_ptr(int dev) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || ptr == nullptr) {
      (void)cudaGetLastError();  // consume it: a later launch check must not see it
      return nullptr;
    }
    g_ptr[dev] = ptr;
  }
  return g_ptr[dev];
}

}  // namespace

extern "C" pa_status pa_decode_static_workspace(
    void* out, const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
    int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
    float scale, pa_dtype q_dtype, pa_dtype kv_dtype, const float* k_scale, const float* v_scale,
    int32_t partition_size, pa_stream_t stream) {
  if (num_seqs < 0) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  // the same argument checks, in the same order, as pa_decode: an invalid argument is
  // reported as such, never as a workspace that is too small
  const pa_status st = pa::check_decode_args(out, q, k_cache, v_cache, num_blocks, block_tables,
                                             max_blocks_per_seq, seq_lens, max_seq_len, num_q_heads, num_kv_heads,
                                             head_size, block_size, scale, q_dtype, kv_dtype, k_scale, v_scale,
                                             partition_size);
  if (st != PA_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return PA_ERR_CUDA;
  }
  void* ws = static_workspace_ptr(dev);
  if (!ws) return PA_ERR_CUDA;
  const size_t cap = PA_STATIC_WORKSPACE_BYTES;
  int32_t part = partition_size;
  if (part == 0) {
    // the default partitioning, coarsened (doubled) until its partial states fit the
    // array; the doubling stops at one partition per sequence, and in 64 bits
    long long coarse = pa_default_partition_size(num_seqs, num_kv_heads, max_seq_len, block_size);
    while (coarse < max_seq_len &&
           pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size, max_seq_len, block_size,
                                    static_cast<int32_t>(coarse)) > cap)
      coarse *= 2;
    if (coarse > INT32_MAX) return PA_ERR_WORKSPACE;
    part = static_cast<int32_t>(coarse);
  }
  if (pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size, max_seq_len, block_size, part) >
      cap)
    return PA_ERR_WORKSPACE;  // the problem's partial states do not fit the fixed array
  return pa_decode(out, q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                   max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, scale, q_dtype, kv_dtype,
                   k_scale, v_scale, part, ws, cap, stream);
}
