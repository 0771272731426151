// Portable kernels of the attention path:
//  * attn_generic_kernel -- one warp per (query row, query head, partition), plain
//    fp32 FMAs, 32 keys per step (a lane per key for the scores, a lane per head
//    dimension for the weighted sum); serves fp32 caches and every shape the
//    tensor-core kernels do not;
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

// A token row of a cache tile (= physical block x Hkv + KV head): the address of its
// first element (NVFP4: of its code row) and, for NVFP4, of its block-scale row.
struct KvRow {
  const uint8_t* row;
  const uint8_t* scales;
};

template <int KVDT>
__device__ __forceinline__ KvRow kv_row(const void* cache, long long tile, int bs, int d, int off) {
  const uint8_t* base = static_cast<const uint8_t*>(cache);
  if constexpr (is_nvfp4<KVDT>()) {
    const uint8_t* t = base + tile * nvfp4_tile_bytes(bs, d);
    return {t + off * (d / 2), t + bs * (d / 2) + off * (d / 16)};
  } else {
    return {base + ((tile * bs + off) * d) * Elem<KVDT>::bytes, nullptr};
  }
}

// Stored value (without the fp32 scale) of element dd of a token row.
template <int KVDT>
__device__ __forceinline__ float kv_elem(const KvRow& r, int dd) {
  if constexpr (is_nvfp4<KVDT>()) {
    const uint32_t byte = r.row[dd >> 1];
    const __half2_raw c = __nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>(byte), __NV_E2M1);
    __half_raw v;
    v.x = (dd & 1) ? c.y : c.x;
    const __half_raw b = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(r.scales[dd >> 4]), __NV_E4M3);
    return __half2float(__half(v)) * __half2float(__half(b));
  } else {
    using KE = Elem<KVDT>;
    return KE::load(reinterpret_cast<const typename KE::T*>(r.row) + dd);
  }
}

template <int QDT, int KVDT>
__global__ void __launch_bounds__(128, 1)
    attn_generic_kernel(const AttnParams p, int only_multi_token) {
  using QE = Elem<QDT>;
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
  const int t0 = ri.origin + z * ri.part;  // partition z of the row's keys
  const int t1 = min(t0 + ri.part, ri.kv_len);
  float kscale = 1.f, vscale = 1.f;
  if (is_scaled<KVDT>()) {
    kscale = p.k_scale[kvh * p.scale_stride];
    vscale = p.v_scale[kvh * p.scale_stride];
  }
  const float c = p.scale * kscale * kLog2e;

  // The warp's query row in shared memory (every lane reads all of it below).
  __shared__ float sq[4][kGenericMaxPerLane * 32];
  float* q_s = sq[threadIdx.x >> 5];
  const typename QE::T* qrow =
      reinterpret_cast<const typename QE::T*>(p.q) + ((long long)row * p.num_q_heads + head) * d;
  for (int dd = lane; dd < d; dd += 32) q_s[dd] = QE::load(qrow + dd);
  __syncwarp();
  float acc[kGenericMaxPerLane];
#pragma unroll
  for (int i = 0; i < kGenericMaxPerLane; ++i) acc[i] = 0.f;
  const int32_t* table = p.block_tables + (long long)ri.request * p.max_blocks_per_seq;
  float m = -INFINITY, l = 0.f;
  // 32 keys at a time (keys before the window are not read): lane j scores key tb + j
  // on its own, so the warp reduces once per 32 keys; then lane i accumulates
  // dimensions i, i + 32, ... of the 32 weighted V rows (coalesced row reads).
  for (int tb = max(t0, ri.lo); tb < t1; tb += 32) {
    const int tt = tb + lane;
    float sj = -INFINITY;
    long long tile = -1;
    if (tt < t1) {
      const int phys = table[tt / p.block_size];
      if (phys < 0 || phys >= p.num_blocks) {
        flag_error(p.err, PA_ERRFLAG_BLOCK_TABLE);
      } else {
        tile = (long long)phys * p.num_kv_heads + kvh;
        const KvRow kr = kv_row<KVDT>(p.k_cache, tile, p.block_size, d, tt % p.block_size);
        // 32 independent loads in flight per round, four accumulation chains
        float dot[4] = {0.f, 0.f, 0.f, 0.f};
        int dd = 0;
        for (; dd + 32 <= d; dd += 32) {
          float kv[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) kv[e] = kv_elem<KVDT>(kr, dd + e);
#pragma unroll
          for (int e = 0; e < 32; ++e) dot[e & 3] = fmaf(q_s[dd + e], kv[e], dot[e & 3]);
        }
        for (; dd + 8 <= d; dd += 8) {
          float kv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) kv[e] = kv_elem<KVDT>(kr, dd + e);
#pragma unroll
          for (int e = 0; e < 8; ++e) dot[e & 3] = fmaf(q_s[dd + e], kv[e], dot[e & 3]);
        }
        for (; dd < d; ++dd) dot[0] = fmaf(q_s[dd], kv_elem<KVDT>(kr, dd), dot[0]);
        sj = ((dot[0] + dot[1]) + (dot[2] + dot[3])) * c;
      }
    }
    const float m_new = fmaxf(m, warp_max_xor(sj, 1, 16));
    if (m_new == -INFINITY) continue;  // no attended key in this group of 32
    const float alpha = exp2f(m - m_new);  // m == -inf before the first key -> 0
    const float pj = exp2f(sj - m_new);
    l = l * alpha + warp_sum_xor(pj, 1, 16);
#pragma unroll
    for (int i = 0; i < kGenericMaxPerLane; ++i) acc[i] *= alpha;
    const int n = min(32, t1 - tb);
    // lane j's V row, handed to every lane; eight rows at a time, so that the loads
    // of eight keys are in flight together
    const KvRow my_v = tile >= 0 ? kv_row<KVDT>(p.v_cache, tile, p.block_size, d, tt % p.block_size)
                                 : KvRow{nullptr, nullptr};
    for (int j0 = 0; j0 < n; j0 += 8) {
      float pv[8];
      KvRow vr[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u;  // < 32
        pv[u] = __shfl_sync(0xffffffffu, pj, j);
        vr[u].row = reinterpret_cast<const uint8_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(my_v.row), j));
        vr[u].scales = nullptr;
        if constexpr (is_nvfp4<KVDT>())
          vr[u].scales = reinterpret_cast<const uint8_t*>(
              __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(my_v.scales), j));
        // keys past the group, or in an unreadable block (flagged above): not read
        if (j >= n) vr[u].row = nullptr;
      }
#pragma unroll
      for (int i = 0; i < kGenericMaxPerLane; ++i) {
        const int dd = lane + 32 * i;
        if (dd < d) {
          float v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) v[u] = vr[u].row != nullptr ? kv_elem<KVDT>(vr[u], dd) : 0.f;
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[i] = fmaf(pv[u], v[u], acc[i]);
        }
      }
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

// One warp per (row, head), four per CTA: out = sum_j acc_j * 2^(m_j - M) /
// sum_j l_j * 2^(m_j - M) with M = max_j m_j.  (M, L) come from one pass over the
// partial states with an online combine; then each lane owns four output
// dimensions and streams the partials with 16-byte loads, eight in flight.
constexpr int kMergeThreads = 128;

__device__ __forceinline__ void combine_ml(float& m, float& l, float m2, float l2) {
  if (l2 <= 0.f) return;
  if (l <= 0.f) {
    m = m2;
    l = l2;
    return;
  }
  const float nm = fmaxf(m, m2);
  l = l * exp2f(m - nm) + l2 * exp2f(m2 - nm);
  m = nm;
}

template <int QDT>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const AttnParams p) {
  using QE = Elem<QDT>;
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5);
  if (gw >= (long long)p.num_rows * p.num_q_heads || plan_rejected(p)) return;
  const int row = static_cast<int>(gw / p.num_q_heads);
  const int head = static_cast<int>(gw % p.num_q_heads);
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
  const float2* ml = p.ws_ml + base * hq + head;  // partial j at ml[j * hq]
  if (np <= 8 && (d & 3) == 0 && d <= 128) {
    // A few partials: every load (each lane's four dimensions of every partial, and
    // every partial's max and sum, the same for all lanes) issued at once, one trip
    // to memory; each lane combines the maxima itself.
    const int nv = d >> 2;
    const float4* acc4 = reinterpret_cast<const float4*>(p.ws_acc + (base * hq + head) * d);
    const long long stride4 = (long long)hq * nv;
    float2 v[8];
    float4 a[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      v[u] = make_float2(-INFINITY, 0.f);
      a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (u < np) {
        v[u] = ml[(long long)u * hq];
        if (lane < nv) a[u] = acc4[u * stride4 + lane];
      }
    }
    float M = -INFINITY, L = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) combine_ml(M, L, v[u].x, v[u].y);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float w = v[u].y > 0.f ? exp2f(v[u].x - M) : 0.f;
      o.x = fmaf(a[u].x, w, o.x);
      o.y = fmaf(a[u].y, w, o.y);
      o.z = fmaf(a[u].z, w, o.z);
      o.w = fmaf(a[u].w, w, o.w);
    }
    if (lane < nv) {
      typename QE::T* out = reinterpret_cast<typename QE::T*>(p.out) + ((long long)row * hq + head) * d;
      out[4 * lane + 0] = QE::from_float(o.x * inv);
      out[4 * lane + 1] = QE::from_float(o.y * inv);
      out[4 * lane + 2] = QE::from_float(o.z * inv);
      out[4 * lane + 3] = QE::from_float(o.w * inv);
    }
    return;
  }
  float M = -INFINITY, L = 0.f;
  for (int j = lane; j < np; j += 32) {
    const float2 v = ml[(long long)j * hq];
    combine_ml(M, L, v.x, v.y);
  }
  for (int o = 16; o >= 1; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, M, o), l2 = __shfl_xor_sync(0xffffffffu, L, o);
    combine_ml(M, L, m2, l2);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  typename QE::T* out = reinterpret_cast<typename QE::T*>(p.out) + ((long long)row * hq + head) * d;
  const long long stride = (long long)hq * d;  // floats between consecutive partials
  const float* acc = p.ws_acc + (base * hq + head) * d;
  if ((d & 3) == 0) {
    for (int c = lane; c < (d >> 2); c += 32) {
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      int j = 0;
      for (; j + 8 <= np; j += 8) {
        float4 a[8];
        float w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float2 v = ml[(long long)(j + u) * hq];
          w[u] = v.y > 0.f ? exp2f(v.x - M) : 0.f;
          a[u] = reinterpret_cast<const float4*>(acc + (j + u) * stride)[c];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          o.x = fmaf(a[u].x, w[u], o.x);
          o.y = fmaf(a[u].y, w[u], o.y);
          o.z = fmaf(a[u].z, w[u], o.z);
          o.w = fmaf(a[u].w, w[u], o.w);
        }
      }
      if (j < np) {  // the last np - j < 8 partials: every load issued before the first use
        float4 a[8];
        float w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          w[u] = 0.f;
          a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (j + u < np) {
            const float2 v = ml[(long long)(j + u) * hq];
            w[u] = v.y > 0.f ? exp2f(v.x - M) : 0.f;
            a[u] = reinterpret_cast<const float4*>(acc + (j + u) * stride)[c];
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          o.x = fmaf(a[u].x, w[u], o.x);
          o.y = fmaf(a[u].y, w[u], o.y);
          o.z = fmaf(a[u].z, w[u], o.z);
          o.w = fmaf(a[u].w, w[u], o.w);
        }
      }
      out[4 * c + 0] = QE::from_float(o.x * inv);
      out[4 * c + 1] = QE::from_float(o.y * inv);
      out[4 * c + 2] = QE::from_float(o.z * inv);
      out[4 * c + 3] = QE::from_float(o.w * inv);
    }
  } else {
    for (int dd = lane; dd < d; dd += 32) {
      float o = 0.f;
      for (int j = 0; j < np; ++j) {
        const float2 v = ml[(long long)j * hq];
        if (v.y > 0.f) o = fmaf(acc[j * stride + dd], exp2f(v.x - M), o);
      }
      out[dd] = QE::from_float(o * inv);
    }
  }
}

// Rows with many partials: one CTA of four warps per (row, head); the warps split
// the partitions (each lane owning four output dimensions, four loads in flight)
// and their sums meet in shared memory.
template <int QDT>
__global__ void __launch_bounds__(kMergeThreads) merge_wide_kernel(const AttnParams p) {
  using QE = Elem<QDT>;
  constexpr int kWarps = kMergeThreads / 32;
  __shared__ float red_m[kWarps], red_l[kWarps];
  __shared__ float4 red_o[kWarps][64];  // head_size <= 256
  const long long gid = blockIdx.x;
  const int row = static_cast<int>(gid / p.num_q_heads);
  const int head = static_cast<int>(gid % p.num_q_heads);
  if (row >= p.num_rows || plan_rejected(p)) return;
  const RowInfo ri = row_info(p, row);
  if (!ri.ok) return;
  int np = ri.parts_row;
  if (p.force_partials) {
    const int start = shared_prefix_tokens(p, row);
    np = (start > 0 ? (start + p.part_shared - 1) / p.part_shared : 0) +
         (ri.seq_len - start + ri.part - 1) / ri.part;
  } else if (np <= 1) {
    return;
  }
  const long long base = row_partial_base(p, ri, row);
  const int hq = p.num_q_heads, d = p.head_size, nv = d >> 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float2* ml = p.ws_ml + base * hq + head;
  float M = -INFINITY, L = 0.f;
  for (int j = threadIdx.x; j < np; j += kMergeThreads) {
    const float2 v = ml[(long long)j * hq];
    combine_ml(M, L, v.x, v.y);
  }
  for (int o = 16; o >= 1; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, M, o), l2 = __shfl_xor_sync(0xffffffffu, L, o);
    combine_ml(M, L, m2, l2);
  }
  if (lane == 0) {
    red_m[warp] = M;
    red_l[warp] = L;
  }
  __syncthreads();
  M = red_m[0];
  L = red_l[0];
  for (int w = 1; w < kWarps; ++w) combine_ml(M, L, red_m[w], red_l[w]);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const long long stride = (long long)hq * d;
  const float* acc = p.ws_acc + (base * hq + head) * d;
  for (int c = lane; c < nv; c += 32) {
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    int j = warp;
    for (; j + 3 * kWarps < np; j += 4 * kWarps) {
      float4 a[4];
      float w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int jj = j + u * kWarps;
        const float2 v = ml[(long long)jj * hq];
        w[u] = v.y > 0.f ? exp2f(v.x - M) : 0.f;
        a[u] = reinterpret_cast<const float4*>(acc + jj * stride)[c];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        o.x = fmaf(a[u].x, w[u], o.x);
        o.y = fmaf(a[u].y, w[u], o.y);
        o.z = fmaf(a[u].z, w[u], o.z);
        o.w = fmaf(a[u].w, w[u], o.w);
      }
    }
    for (; j < np; j += kWarps) {
      const float2 v = ml[(long long)j * hq];
      const float w = v.y > 0.f ? exp2f(v.x - M) : 0.f;
      const float4 a = reinterpret_cast<const float4*>(acc + j * stride)[c];
      o.x = fmaf(a.x, w, o.x);
      o.y = fmaf(a.y, w, o.y);
      o.z = fmaf(a.z, w, o.z);
      o.w = fmaf(a.w, w, o.w);
    }
    red_o[warp][c] = o;
  }
  __syncthreads();
  typename QE::T* out = reinterpret_cast<typename QE::T*>(p.out) + ((long long)row * hq + head) * d;
  for (int c = threadIdx.x; c < nv; c += kMergeThreads) {
    float4 o = red_o[0][c];
    for (int w = 1; w < kWarps; ++w) {
      o.x += red_o[w][c].x;
      o.y += red_o[w][c].y;
      o.z += red_o[w][c].z;
      o.w += red_o[w][c].w;
    }
    out[4 * c + 0] = QE::from_float(o.x * inv);
    out[4 * c + 1] = QE::from_float(o.y * inv);
    out[4 * c + 2] = QE::from_float(o.z * inv);
    out[4 * c + 3] = QE::from_float(o.w * inv);
  }
}

// One request's plan: where its partial rows go and which prefill tiles it needs.  A
// row tile of tile_tokens query tokens needs the partitions up to its last key; all
// but the last of them span a whole partition.
struct RequestPlan {
  int q_len, seq_len, part, origin, parts;
  int full_tiles;  // prefill tiles over a whole partition
  int last_tiles;  // prefill tiles over a row tile's last partition
  bool ok;
};

__device__ int tile_partitions(const AttnParams& p, const RequestPlan& rp, int t0, int tile_tokens) {
  const int last = min(t0 + tile_tokens, rp.q_len) - 1;
  const int kv = p.causal ? rp.seq_len - rp.q_len + last + 1 : rp.seq_len;
  return ceil_div_dev(kv - rp.origin, rp.part);
}

__device__ RequestPlan plan_request(const AttnParams& p, int r, int tile_tokens) {
  RequestPlan rp;
  rp.q_len = p.query_start_loc[r + 1] - p.query_start_loc[r];
  rp.seq_len = p.seq_lens[r];
  rp.part = p.part;
  rp.origin = 0;
  rp.parts = 0;
  rp.full_tiles = 0;
  rp.last_tiles = 0;
  rp.ok = rp.q_len >= 0 && rp.q_len <= p.max_query_len && rp.q_len <= rp.seq_len &&
          rp.seq_len <= p.max_seq_len && (long long)rp.seq_len <= (long long)p.max_blocks_per_seq * p.block_size;
  if (rp.ok && rp.q_len > 0 && rp.seq_len >= 1) {
    rp.part = rp.q_len == 1 ? p.part : p.part_pf;
    rp.origin = window_origin(p, rp.seq_len, rp.q_len);
    rp.parts = ceil_div_dev(rp.seq_len - rp.origin, rp.part);
    if (rp.q_len > 1) {
      for (int t0 = 0; t0 < rp.q_len; t0 += tile_tokens) {
        const int np = tile_partitions(p, rp, t0, tile_tokens);
        if (np > 0) {
          rp.full_tiles += np - 1;
          rp.last_tiles += 1;
        }
      }
    }
  }
  return rp;
}

// Single CTA.  For each request: validates its query range and computes
//   part_off[r] = sum over earlier requests of q_len * ceil(seq_len / part_r),
// the index of its first partial row, and lists its prefill tiles (requests with
// q_len > 1) as (request, first query row, partition, 0): first every tile over a
// whole partition (work_full of them), then each row tile's last, shorter one, so
// that the persistent tile grids claim the long tiles first and the short ones fill
// the tail.
__global__ void __launch_bounds__(1024)
    varlen_plan_kernel(const AttnParams p, int32_t* part_off, int4* work, int32_t* work_count,
                       int32_t* plan_ok, int max_work, int tile_tokens) {
  __shared__ int warp_tot[3][32];
  __shared__ int carry[3];
  __shared__ int bad, full_total;
  const int tid = threadIdx.x;
  const int lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  if (tid == 0) {
    carry[0] = carry[1] = carry[2] = 0;
    full_total = 0;
    const int q0 = p.query_start_loc[0], qn = p.query_start_loc[p.num_seqs];
    bad = (q0 != 0 || qn != p.num_rows) ? 1 : 0;
  }
  __syncthreads();
  // pass 1: the number of whole-partition tiles, after which the last tiles start
  for (int base = 0; base < p.num_seqs; base += blockDim.x) {
    const int r = base + tid;
    int nf = r < p.num_seqs ? plan_request(p, r, tile_tokens).full_tiles : 0;
    for (int o = 16; o > 0; o >>= 1) nf += __shfl_xor_sync(0xffffffffu, nf, o);
    if (lane == 0 && nf) atomicAdd(&full_total, nf);
  }
  __syncthreads();
  // pass 2: exclusive scans of (partial rows, whole-partition tiles, last tiles)
  for (int base = 0; base < p.num_seqs; base += blockDim.x) {
    const int r = base + tid;
    RequestPlan rp;
    rp.q_len = 0;
    rp.parts = 0;
    rp.full_tiles = 0;
    rp.last_tiles = 0;
    if (r < p.num_seqs) {
      rp = plan_request(p, r, tile_tokens);
      if (rp.q_len < 0) atomicOr(&bad, 1);
      if (!rp.ok && rp.q_len != 0)
        flag_error(p.err, rp.q_len < 0 || rp.q_len > p.max_query_len || rp.q_len > rp.seq_len
                              ? PA_ERRFLAG_QUERY : PA_ERRFLAG_SEQ_LEN);
    }
    const int v[3] = {rp.q_len > 0 ? rp.q_len * rp.parts : 0, rp.full_tiles, rp.last_tiles};
    int sc[3] = {v[0], v[1], v[2]};
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int a = __shfl_up_sync(0xffffffffu, sc[k], o);
        if (lane >= o) sc[k] += a;
      }
    }
    if (lane == 31)
      for (int k = 0; k < 3; ++k) warp_tot[k][wid] = sc[k];
    __syncthreads();
    if (wid == 0) {
      for (int k = 0; k < 3; ++k) {
        int a = lane < nw ? warp_tot[k][lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
          const int x = __shfl_up_sync(0xffffffffu, a, o);
          if (lane >= o) a += x;
        }
        warp_tot[k][lane] = a;
      }
    }
    __syncthreads();
    int ex[3];
    for (int k = 0; k < 3; ++k) ex[k] = carry[k] + (wid ? warp_tot[k][wid - 1] : 0) + sc[k] - v[k];
    if (r < p.num_seqs) {
      part_off[r] = ex[0];
      if (rp.full_tiles + rp.last_tiles) {
        int kf = ex[1], kl = full_total + ex[2];
        const int row0 = p.query_start_loc[r];
        // partition-major: the row tiles that read one partition are listed (and so
        // claimed) one after another, and read its K/V from L2 while it is there
        const int last_t0 = (rp.q_len - 1) / tile_tokens * tile_tokens;
        const int np_max = tile_partitions(p, rp, last_t0, tile_tokens);  // the most any row tile has
        for (int z = 0; z < np_max; ++z) {
          for (int t0 = 0; t0 < rp.q_len; t0 += tile_tokens) {
            const int np = tile_partitions(p, rp, t0, tile_tokens);
            if (z >= np) continue;
            const int k = z + 1 < np ? kf++ : kl++;
            if (k < max_work) work[k] = make_int4(r, row0 + t0, z, 0);
          }
        }
      }
    }
    __syncthreads();
    if (tid == 0)
      for (int k = 0; k < 3; ++k) carry[k] += warp_tot[k][nw - 1];
    __syncthreads();
  }
  if (tid == 0) {
    const int count = bad ? 0 : min(full_total + carry[2], max_work);
    *work_count = count;
    if (p.work_full) *p.work_full = min(full_total, count);
    *plan_ok = bad ? 0 : 1;
    if (p.work_claim) *p.work_claim = 0;
    if (bad) flag_error(p.err, PA_ERRFLAG_QUERY);
  }
}

template <int QDT, int KVDT>
cudaError_t launch_generic_t(const AttnParams& p, int grid_z, int only_multi, cudaStream_t s) {
  dim3 grid(p.num_rows, (p.num_q_heads + 3) / 4, grid_z);
  attn_generic_kernel<QDT, KVDT><<<grid, 128, 0, s>>>(p, only_multi);
  return cudaGetLastError();
}

// Rows may carry up to p.max_partitions partials: with many, four warps per row.
template <int QDT>
cudaError_t launch_merge_t(const AttnParams& p, cudaStream_t s) {
  const long long rows = (long long)p.num_rows * p.num_q_heads;
  if (p.max_partitions > 32 && (p.head_size & 3) == 0 && p.head_size <= 256) {
    merge_wide_kernel<QDT><<<(unsigned)rows, kMergeThreads, 0, s>>>(p);
  } else {
    const long long ctas = (rows + kMergeThreads / 32 - 1) / (kMergeThreads / 32);
    merge_kernel<QDT><<<(unsigned)ctas, kMergeThreads, 0, s>>>(p);
  }
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
  PA_GEN(PA_F16, PA_FP8_E5M2)
  PA_GEN(PA_BF16, PA_FP8_E5M2)
  PA_GEN(PA_F32, PA_FP8_E5M2)
  PA_GEN(PA_F16, PA_NVFP4)
  PA_GEN(PA_BF16, PA_NVFP4)
  PA_GEN(PA_F32, PA_NVFP4)
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
