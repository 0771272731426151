// copy_blocks: copy whole physical blocks of the paged cache (K and V, every KV
// head) from a source to a destination block.  [AGENTIC] "統一分頁 + 共用池"
// (reference counting + copy-on-write): forks share physical blocks until one of
// them must change shared content; [LINEAGE] "Prefix reuse": a shared block that is
// not yet full is copied before a branch writes its next token into it.
//
// Grid: x = pair, y = slice of the block.  A (block) of one cache tensor is
// contiguous (num_kv_heads x block_size x head_size elements), so each thread moves
// consecutive 16-byte pieces of K and V: coalesced, four pieces of each tensor in
// flight per thread.
#include "pa_common.cuh"

namespace pa {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kPiecesPerThread = 4;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyParams p) {
  const long long src = p.block_mapping[2 * (long long)blockIdx.x];
  const long long dst = p.block_mapping[2 * (long long)blockIdx.x + 1];
  if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
    if (blockIdx.y == 0 && threadIdx.x == 0) flag_error(p.err, PA_ERRFLAG_BLOCK_TABLE);
    return;
  }
  if (src == dst) return;
  const long long n16 = p.block_bytes / 16;
  const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.k_cache) + src * p.block_bytes);
  const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.v_cache) + src * p.block_bytes);
  uint4* kd = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.k_cache) + dst * p.block_bytes);
  uint4* vd = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.v_cache) + dst * p.block_bytes);
  const long long step = (long long)gridDim.y * kCopyThreads;
  long long i = (long long)blockIdx.y * kCopyThreads + threadIdx.x;
  for (; i + (kPiecesPerThread - 1) * step < n16; i += kPiecesPerThread * step) {
    uint4 a[kPiecesPerThread], b[kPiecesPerThread];
#pragma unroll
    for (int u = 0; u < kPiecesPerThread; ++u) {
      a[u] = ks[i + u * step];
      b[u] = vs[i + u * step];
    }
#pragma unroll
    for (int u = 0; u < kPiecesPerThread; ++u) {
      kd[i + u * step] = a[u];
      vd[i + u * step] = b[u];
    }
  }
  for (; i < n16; i += step) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream) {
  const long long n16 = p.block_bytes / 16;
  const long long per_cta = (long long)kCopyThreads * kPiecesPerThread;
  const unsigned slices = static_cast<unsigned>((n16 + per_cta - 1) / per_cta);
  dim3 grid(static_cast<unsigned>(p.num_pairs), slices > 0 ? slices : 1u);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
