// Internal interfaces between the C-ABI layer (api.cu) and the kernel translation
// units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// Bytes of one (block, KV head) tile of an NVFP4 cache: block_size rows of head/2
// bytes of E2M1 codes, then block_size rows of head/16 E4M3 block scales.
__host__ __device__ constexpr int nvfp4_tile_bytes(int block_size, int head) {
  return block_size * head / 2 + block_size * head / 16;
}

// Everything an attention kernel needs.  "Rows" are query rows: one per sequence
// in decode mode (query_start_loc == nullptr), one per flattened query token in
// varlen mode.
struct AttnParams {
  void* out;                       // [num_rows][Hq][d], q dtype
  const void* q;                   // [num_rows][Hq][d], q dtype
  const void* k_cache;             // [num_blocks][Hkv][bs][d] (NVFP4: [num_blocks][Hkv][tile bytes])
  const void* v_cache;
  const int32_t* block_tables;     // [num_seqs][max_blocks_per_seq]
  const int32_t* seq_lens;         // [num_seqs]
  const int32_t* query_start_loc;  // [num_seqs+1] in varlen mode, nullptr in decode mode
  const int32_t* part_off;         // varlen: first partial row of each request (plan kernel)
  const int4* work;                // varlen: prefill tile work list (plan kernel)
  const int32_t* work_count;       // varlen: number of entries in `work`
  const int32_t* plan_ok;          // varlen: 1 when query_start_loc passed the plan kernel's checks
  int32_t* work_claim;             // varlen: prefill tiles claimed so far (zeroed by the plan kernel)
  int32_t* work_full;              // varlen: leading entries of `work` that span a whole partition
  const int32_t* group_start;      // shared-prefix decode: [num_groups+1] runs of consecutive sequences
  const int32_t* group_shared_blocks;  // shared-prefix decode: [num_groups] leading blocks shared in a group
  float* ws_acc;                   // [partial rows][Hq][d]  un-normalised weighted sums
  float2* ws_ml;                   // [partial rows][Hq]     (running max in log2 units, weight sum)
  const float* k_scale;            // FP8 / NVFP4: scale of KV head h at k_scale[h * scale_stride]
  const float* v_scale;
  int scale_stride;                // 0: one scale per tensor, 1: one per KV head
  unsigned* err;                   // device error word
  int num_seqs;
  int num_rows;
  int num_blocks;
  int max_blocks_per_seq;
  int num_q_heads;
  int num_kv_heads;
  int head_size;
  int block_size;
  int group;            // Hq / Hkv
  int num_head_groups;  // ceil(group / 8) for the tensor-core kernels
  int max_seq_len;
  int max_query_len;
  int part;             // partition tokens for rows of single-token requests
  int part_pf;          // partition tokens for rows of multi-token requests
  int part_shared;      // partition tokens of a group's shared prefix (shared-prefix decode)
  int max_partitions;   // decode mode: partial rows reserved per query row
  int causal;
  int window;           // sliding window: a query at position p attends keys > p - window (0 = all)
  int num_groups;       // shared-prefix decode: number of groups (0 = no sharing)
  int max_group_size;   // shared-prefix decode: host bound on sequences per group (<= 8)
  int force_partials;   // every row writes partial states and goes through the merge
  float scale;          // softmax scale
};

struct ScatterParams {
  const void* key;
  const void* value;
  void* k_cache;
  void* v_cache;
  const int64_t* slot_mapping;
  const float* k_scale;  // FP8 / NVFP4: scale of KV head h at k_scale[h * scale_stride]
  const float* v_scale;
  int scale_stride;
  unsigned* err;
  int num_tokens;
  int num_blocks;
  int num_kv_heads;
  int head_size;
  int block_size;
};

struct CopyParams {
  void* k_cache;
  void* v_cache;
  const int64_t* block_mapping;  // [num_pairs][2] (src, dst)
  unsigned* err;
  int num_pairs;
  int num_blocks;
  long long block_bytes;         // bytes of one block of one cache tensor
};

cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream);

// pa_decode's argument checks on everything but the workspace (api.cu).
pa_status check_decode_args(const void* out, const void* q, const void* k_cache, const void* v_cache,
                            int32_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, int32_t max_seq_len, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_size, int32_t block_size, float scale,
                            pa_dtype q_dtype, pa_dtype kv_dtype, const float* k_scale, const float* v_scale,
                            int32_t partition_size);

// Query tokens handled by one CTA of the tcgen05 prefill kernel.
int prefill_tile_tokens(int group);

cudaError_t launch_reshape_and_cache(const ScatterParams& p, int src_dtype, int cache_dtype,
                                     cudaStream_t stream);
cudaError_t launch_attn_generic(const AttnParams& p, int q_dtype, int kv_dtype, int grid_z,
                                int only_multi_token, cudaStream_t stream);
cudaError_t launch_merge(const AttnParams& p, int q_dtype, cudaStream_t stream);
cudaError_t launch_varlen_plan(const AttnParams& p, int32_t* part_off, int4* work,
                               int32_t* work_count, int max_work, cudaStream_t stream);

bool decode_mma_supported(int q_dtype, int kv_dtype, int head_size, int block_size, int group);
cudaError_t launch_decode_mma(const AttnParams& p, int q_dtype, int kv_dtype, int grid_z,
                              const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                              cudaStream_t stream);

cudaError_t launch_shared_prefix(const AttnParams& p, int q_dtype, int kv_dtype, int grid_z,
                                 const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                 cudaStream_t stream);

cudaError_t launch_shared_prefix_tiles(const AttnParams& p, int q_dtype, int grid_z,
                                       const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                       cudaStream_t stream);

// tcgen05 prefill tiles (TMEM accumulators); tmap_k has one-piece boxes, tmap_v
// whole (block, head) tiles.  A persistent grid of at most max_ctas CTAs (one per SM)
// claims (work item, KV head group) tiles through p.work_claim; several launches may
// share one plan's list, each tile going to whichever CTA claims it first.
bool prefill_tc_supported(int q_dtype, int kv_dtype, int head_size, int block_size);
cudaError_t launch_prefill_tc(const AttnParams& p, int q_dtype, int kv_dtype, int num_items, int max_ctas,
                              const CUtensorMap* tmap_k, const CUtensorMap* tmap_v, cudaStream_t stream);

}  // namespace pa
