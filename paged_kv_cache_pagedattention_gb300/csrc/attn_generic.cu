// Portable kernels of the attention path:
//  * attn_generic_kernel -- one warp per (query row, query head, partition), plain
//    fp32 FMAs; serves fp32 caches and every shape the tensor-core kernels do not;
//  * merge_kernel -- combines the split-K partial states of a row into its output
//    (rescale each partial by exp2(m_j - m) to the common maximum, add, divide);
//  * varlen_plan_kernel -- validates query_start_loc and lays out, per request,
//    where its partial rows live and which prefill tiles exist.
// Sources: [AGENTIC] "Online softmax 到底在幹嘛" (weighted sum / weight sum per part,
// local maxima brought to the global maximum before adding); [LINEAGE]
// "PagedAttention" (K/V read through the block table).
#include "pa_common.cuh"

namespace pa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kGenericMaxPerLane = 8;  // head_size <= 256

template <int QDT, int KVDT>
__global__ void __launch_bounds__(128)
    attn_generic_kernel(const AttnParams p, int only_multi_token) {
  using QE = Elem<QDT>;
  using KE = Elem<KVDT>;
  const int lane = threadIdx.x & 31;
  const int head = blockIdx.y * 4 + (threadIdx.x >> 5);
  const int row = blockIdx.x;
  const int z = blockIdx.z;
  if (head >= p.num_q_heads || plan_rejected(p)) return;
  const RowInfo ri = row_info(p, row);
  const int d = p.head_size;
  typename QE::T* out = reinterpret_cast<typename QE::T*>(p.out) + ((long long)row * p.num_q_heads + head) * d;
  if (!ri.ok) {
    if (z == 0) {
      for (int i = lane; i < d; i += 32) out[i] = QE::from_float(0.f);
      if (lane == 0 && p.query_start_loc == nullptr) flag_error(p.err, PA_ERRFLAG_SEQ_LEN);
    }
    return;
  }
  if (p.query_start_loc != nullptr && only_multi_token >= 0 && (ri.q_len > 1) != (only_multi_token != 0)) return;
  if (z >= ri.parts_row) return;

  const int kvh = head / p.group;
  const int t0 = z * ri.part;
  const int t1 = min(t0 + ri.part, ri.kv_len);
  float kscale = 1.f, vscale = 1.f;
  if (KVDT == PA_FP8_E4M3) {
    kscale = *p.k_scale;
    vscale = *p.v_scale;
  }
  const float c = p.scale * kscale * kLog2e;

  const typename QE::T* qrow =
      reinterpret_cast<const typename QE::T*>(p.q) + ((long long)row * p.num_q_heads + head) * d;
  float qv[kGenericMaxPerLane], acc[kGenericMaxPerLane];
#pragma unroll
  for (int i = 0; i < kGenericMaxPerLane; ++i) {
    const int dd = lane + 32 * i;
    qv[i] = dd < d ? QE::load(qrow + dd) : 0.f;
    acc[i] = 0.f;
  }
  const typename KE::T* kc = reinterpret_cast<const typename KE::T*>(p.k_cache);
  const typename KE::T* vc = reinterpret_cast<const typename KE::T*>(p.v_cache);
  const int32_t* table = p.block_tables + (long long)ri.request * p.max_blocks_per_seq;
  float m = -INFINITY, l = 0.f;
  for (int t = t0; t < t1; ++t) {
    const int phys = table[t / p.block_size];
    if (phys < 0 || phys >= p.num_blocks) {
      if (lane == 0) flag_error(p.err, PA_ERRFLAG_BLOCK_TABLE);
      continue;
    }
    const long long base =
        (((long long)phys * p.num_kv_heads + kvh) * p.block_size + (t % p.block_size)) * d;
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < kGenericMaxPerLane; ++i) {
      const int dd = lane + 32 * i;
      if (dd < d) dot = fmaf(qv[i], KE::load(kc + base + dd), dot);
    }
    dot = warp_sum_xor(dot, 1, 16);
    const float s = dot * c;
    const float m_new = fmaxf(m, s);
    const float alpha = exp2f(m - m_new);  // m == -inf on the first key -> 0
    const float w = exp2f(s - m_new);
    l = l * alpha + w;
#pragma unroll
    for (int i = 0; i < kGenericMaxPerLane; ++i) {
      const int dd = lane + 32 * i;
      if (dd < d) acc[i] = fmaf(w, KE::load(vc + base + dd), acc[i] * alpha);
    }
    m = m_new;
  }
  if (ri.parts_row == 1) {
    const float inv = l > 0.f ? vscale / l : 0.f;
#pragma unroll
    for (int i = 0; i < kGenericMaxPerLane; ++i) {
      const int dd = lane + 32 * i;
      if (dd < d) out[dd] = QE::from_float(acc[i] * inv);
    }
  } else {
    const long long pi = row_partial_base(p, ri, row) + z;
    float* wa = p.ws_acc + (pi * p.num_q_heads + head) * d;
#pragma unroll
    for (int i = 0; i < kGenericMaxPerLane; ++i) {
      const int dd = lane + 32 * i;
      if (dd < d) wa[dd] = acc[i] * vscale;
    }
    if (lane == 0) p.ws_ml[pi * p.num_q_heads + head] = make_float2(m, l);
  }
}

// One CTA per (row, head): out = sum_j acc_j * 2^(m_j - M) / sum_j l_j * 2^(m_j - M)
// with M = max_j m_j.  The per-partition factors are computed once into shared
// memory; then each thread owns output dimensions and streams the partials with
// independent, coalesced loads.
constexpr int kMergeThreads = 128;
constexpr int kMergeChunk = 512;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
  v = is_max ? warp_max_xor(v, 1, 16) : warp_sum_xor(v, 1, 16);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float r = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  __syncthreads();
  return r;
}

template <int QDT>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const AttnParams p) {
  using QE = Elem<QDT>;
  __shared__ float wts[kMergeChunk];
  __shared__ float red[kMergeThreads / 32];
  const long long gid = blockIdx.x;
  const int row = static_cast<int>(gid / p.num_q_heads);
  const int head = static_cast<int>(gid % p.num_q_heads);
  if (row >= p.num_rows || plan_rejected(p)) return;
  const RowInfo ri = row_info(p, row);
  if (!ri.ok) return;
  int np = ri.parts_row;
  if (p.force_partials) {
    // shared-prefix decode: partials of the shared prefix, then of the private rest
    const int start = shared_prefix_tokens(p, row);
    np = (start > 0 ? (start + p.part_shared - 1) / p.part_shared : 0) +
         (ri.seq_len - start + ri.part - 1) / ri.part;
  } else if (np <= 1) {
    return;  // written directly by the attention kernel
  }
  const long long base = row_partial_base(p, ri, row);
  const int hq = p.num_q_heads, d = p.head_size;
  float M = -INFINITY;
  for (int j = threadIdx.x; j < np; j += blockDim.x) {
    const float2 ml = p.ws_ml[(base + j) * hq + head];
    if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
  M = block_reduce(M, true, red);
  float L = 0.f;
  for (int j = threadIdx.x; j < np; j += blockDim.x) {
    const float2 ml = p.ws_ml[(base + j) * hq + head];
    if (ml.y > 0.f) L += ml.y * exp2f(ml.x - M);
  }
  L = block_reduce(L, false, red);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  typename QE::T* out = reinterpret_cast<typename QE::T*>(p.out) + ((long long)row * hq + head) * d;
  for (int d0 = 0; d0 < d; d0 += blockDim.x) {
    const int dd = d0 + threadIdx.x;
    float o0 = 0.f, o1 = 0.f;
    for (int c0 = 0; c0 < np; c0 += kMergeChunk) {
      const int n = min(kMergeChunk, np - c0);
      __syncthreads();
      for (int j = threadIdx.x; j < n; j += blockDim.x) {
        const float2 ml = p.ws_ml[(base + c0 + j) * hq + head];
        wts[j] = ml.y > 0.f ? exp2f(ml.x - M) : 0.f;
      }
      __syncthreads();
      if (dd < d) {
        const float* src = p.ws_acc + ((base + c0) * hq + head) * d + dd;
        const long long stride = (long long)hq * d;
        int j = 0;
        for (; j + 1 < n; j += 2) {
          o0 = fmaf(src[j * stride], wts[j], o0);
          o1 = fmaf(src[(j + 1) * stride], wts[j + 1], o1);
        }
        if (j < n) o0 = fmaf(src[j * stride], wts[j], o0);
      }
    }
    if (dd < d) out[dd] = QE::from_float((o0 + o1) * inv);
  }
}

// Single CTA.  For each request: validates its query range and computes
//   part_off[r] = sum over earlier requests of q_len * ceil(seq_len / part_r),
// the index of its first partial row, and appends its prefill tiles (requests
// with q_len > 1) to the work list as (request, first query row, partition, 0).
__global__ void __launch_bounds__(1024)
    varlen_plan_kernel(const AttnParams p, int32_t* part_off, int4* work, int32_t* work_count,
                       int32_t* plan_ok, int max_work, int tile_tokens) {
  __shared__ int warp_tot[2][32];
  __shared__ int carry[2];
  __shared__ int bad;
  const int tid = threadIdx.x;
  const int lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  if (tid == 0) {
    carry[0] = 0;
    carry[1] = 0;
    const int q0 = p.query_start_loc[0], qn = p.query_start_loc[p.num_seqs];
    bad = (q0 != 0 || qn != p.num_rows) ? 1 : 0;
  }
  __syncthreads();
  for (int base = 0; base < p.num_seqs; base += blockDim.x) {
    const int r = base + tid;
    int parts = 0, items = 0;
    int q_len = 0, seq_len = 0, part = p.part;
    if (r < p.num_seqs) {
      q_len = p.query_start_loc[r + 1] - p.query_start_loc[r];
      if (q_len < 0) atomicOr(&bad, 1);
      seq_len = p.seq_lens[r];
      const bool ok = q_len >= 0 && q_len <= p.max_query_len && q_len <= seq_len &&
                      seq_len <= p.max_seq_len &&
                      (long long)seq_len <= (long long)p.max_blocks_per_seq * p.block_size;
      if (!ok && q_len != 0) flag_error(p.err, q_len < 0 || q_len > p.max_query_len || q_len > seq_len
                                                   ? PA_ERRFLAG_QUERY : PA_ERRFLAG_SEQ_LEN);
      if (ok && q_len > 0 && seq_len >= 1) {
        part = q_len == 1 ? p.part : p.part_pf;
        parts = ceil_div_dev(seq_len, part);
        if (q_len > 1) {
          // tiles of tile_tokens query tokens; a tile needs the partitions up to its last key
          for (int t0 = 0; t0 < q_len; t0 += tile_tokens) {
            const int last = min(t0 + tile_tokens, q_len) - 1;
            const int kv = p.causal ? seq_len - q_len + last + 1 : seq_len;
            items += ceil_div_dev(kv, part);
          }
        }
      }
    }
    int v0 = q_len > 0 ? q_len * parts : 0;
    int v1 = items;
    // block-wide exclusive scans of v0 and v1
    int s0 = v0, s1 = v1;
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, s0, o), b = __shfl_up_sync(0xffffffffu, s1, o);
      if (lane >= o) { s0 += a; s1 += b; }
    }
    if (lane == 31) { warp_tot[0][wid] = s0; warp_tot[1][wid] = s1; }
    __syncthreads();
    if (wid == 0) {
      int a = lane < nw ? warp_tot[0][lane] : 0, b = lane < nw ? warp_tot[1][lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, a, o), y = __shfl_up_sync(0xffffffffu, b, o);
        if (lane >= o) { a += x; b += y; }
      }
      warp_tot[0][lane] = a;
      warp_tot[1][lane] = b;
    }
    __syncthreads();
    const int ex0 = carry[0] + (wid ? warp_tot[0][wid - 1] : 0) + s0 - v0;
    const int ex1 = carry[1] + (wid ? warp_tot[1][wid - 1] : 0) + s1 - v1;
    if (r < p.num_seqs) {
      part_off[r] = ex0;
      if (items) {
        int k = ex1;
        const int row0 = p.query_start_loc[r];
        for (int t0 = 0; t0 < q_len; t0 += tile_tokens) {
          const int last = min(t0 + tile_tokens, q_len) - 1;
          const int kv = p.causal ? seq_len - q_len + last + 1 : seq_len;
          const int np = ceil_div_dev(kv, part);
          for (int z = 0; z < np; ++z, ++k)
            if (k < max_work) work[k] = make_int4(r, row0 + t0, z, 0);
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      carry[0] += warp_tot[0][nw - 1];
      carry[1] += warp_tot[1][nw - 1];
    }
    __syncthreads();
  }
  if (tid == 0) {
    *work_count = bad ? 0 : min(carry[1], max_work);
    *plan_ok = bad ? 0 : 1;
    if (bad) flag_error(p.err, PA_ERRFLAG_QUERY);
  }
}

template <int QDT, int KVDT>
cudaError_t launch_generic_t(const AttnParams& p, int grid_z, int only_multi, cudaStream_t s) {
  dim3 grid(p.num_rows, (p.num_q_heads + 3) / 4, grid_z);
  attn_generic_kernel<QDT, KVDT><<<grid, 128, 0, s>>>(p, only_multi);
  return cudaGetLastError();
}

template <int QDT>
cudaError_t launch_merge_t(const AttnParams& p, cudaStream_t s) {
  const long long ctas = (long long)p.num_rows * p.num_q_heads;
  merge_kernel<QDT><<<(unsigned)ctas, kMergeThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_generic(const AttnParams& p, int q_dtype, int kv_dtype, int grid_z,
                                int only_multi_token, cudaStream_t stream) {
  if (p.head_size > 32 * kGenericMaxPerLane) return cudaErrorInvalidValue;
#define PA_GEN(Q, KV) \
  if (q_dtype == Q && kv_dtype == KV) return launch_generic_t<Q, KV>(p, grid_z, only_multi_token, stream);
  PA_GEN(PA_F32, PA_F32)
  PA_GEN(PA_F16, PA_F16)
  PA_GEN(PA_BF16, PA_BF16)
  PA_GEN(PA_F16, PA_FP8_E4M3)
  PA_GEN(PA_BF16, PA_FP8_E4M3)
  PA_GEN(PA_F32, PA_FP8_E4M3)
#undef PA_GEN
  return cudaErrorInvalidValue;
}

cudaError_t launch_merge(const AttnParams& p, int q_dtype, cudaStream_t stream) {
  if (q_dtype == PA_F32) return launch_merge_t<PA_F32>(p, stream);
  if (q_dtype == PA_F16) return launch_merge_t<PA_F16>(p, stream);
  if (q_dtype == PA_BF16) return launch_merge_t<PA_BF16>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_varlen_plan(const AttnParams& p, int32_t* part_off, int4* work,
                               int32_t* work_count, int max_work, cudaStream_t stream) {
  varlen_plan_kernel<<<1, 1024, 0, stream>>>(p, part_off, work, work_count,
                                             const_cast<int32_t*>(p.plan_ok), max_work,
                                             prefill_tile_tokens(p.group));
  return cudaGetLastError();
}

}  // namespace pa
