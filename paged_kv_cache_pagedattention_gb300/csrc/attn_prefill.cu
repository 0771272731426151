// Tensor-core tiles for the multi-token (chunked-prefill) rows of a varlen batch.
//
// [LINEAGE] "Chunked prefill" / [ARCH] Part 2 (chunked prefill): a long prompt is
// processed in chunks; each chunk's query tokens attend the request's cached
// prefix and, causally, the chunk itself.  [NOTES] "Prefill 与 Decode" / [ARCH]
// Part 1: prefill work is dense and compute-bound, so these tiles run on the
// tensor cores.
//
// Work item (built by the varlen plan kernel): (request, first query row of the
// tile, partition of the keys).  The CTA's grid y picks the KV head and a group of
// <= 8 query heads.  A tile holds 128 query rows = (token, head) pairs, token-major
// (row = token * GP + head, GP = the head group padded to a power of two), so every
// K/V element loaded serves all heads of the group and all tokens of the tile.
//
// Warp roles: warps 0..7 each own 16 query rows (Q fragments and the O accumulator
// stay in registers, FlashAttention-2 style); warp 8 produces: its lane 0 walks the
// partition's blocks through the block table and issues TMA bulk-tensor copies of
// the K/V tiles into a ring of stages shared by the CTA (full / empty mbarriers).
// Per 16-token block and warp:
//   S = Q K^T   (m16n8k16, M = 16 rows, N = 8 tokens, K = head dim)
//   online softmax per row (running max / sum, exp2, fp32), causal mask by position
//   O += P V    (P straight from the S accumulators as the A operand)
// The output is written directly when the row needs one partition, else as a
// partial state (unnormalised O, max, sum) merged later.
#include "pa_common.cuh"

namespace pa {

int prefill_tile_tokens(int group) {
  int g8 = 1;
  while (g8 < group && g8 < 8) g8 <<= 1;
  return 128 / g8;
}

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int HEAD, int BS>
struct PrefillGeom {
  static constexpr int kRowBytes = HEAD * 2;
  static constexpr int kTileBytes = BS * kRowBytes;
  static constexpr int kSub = kRowBytes / 128;
  static constexpr int kStages = kTileBytes <= 4096 ? 8 : 5;
  static constexpr int kKSteps = HEAD / 16;  // QK k-steps over the head dim
  static constexpr int kNTok = BS / 8;       // QK n-tiles over tokens
  static constexpr int kNDim = HEAD / 8;     // PV n-tiles over the head dim
  static __device__ __forceinline__ uint32_t off(int tok, int chunk) {
    return static_cast<uint32_t>((chunk >> 3) * BS * 128) + swz128(tok, chunk & 7);
  }
};

template <int HEAD, int BS>
constexpr int prefill_smem_bytes() {
  using G = PrefillGeom<HEAD, BS>;
  return G::kStages * 2 * G::kTileBytes + 2 * G::kStages * 8 + 1024;
}

template <int QDT, int HEAD, int BS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_mma_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv) {
  using G = PrefillGeom<HEAD, BS>;
  using QE = Elem<QDT>;
  constexpr int ST = G::kStages;
  constexpr int TB = G::kTileBytes;

  if (plan_rejected(p) || (int)blockIdx.x >= *p.work_count) return;
  const int4 item = p.work[blockIdx.x];
  const int r = item.x, row0 = item.y, z = item.z;
  const int kvh = blockIdx.y / p.num_head_groups, hg = blockIdx.y % p.num_head_groups;
  const int h0 = kvh * p.group + hg * 8;
  const int nh = min(8, p.group - hg * 8);
  int gp = 1;
  while (gp < min(p.group, 8)) gp <<= 1;
  const int tile_tokens = 128 / gp;

  const int qs = p.query_start_loc[r];
  const int q_len = p.query_start_loc[r + 1] - qs;
  const int seq_len = p.seq_lens[r];
  const int t0 = row0 - qs;                            // first token of the tile in its request
  const int ntok = min(tile_tokens, q_len - t0);       // tokens in this tile
  const int pos0 = seq_len - q_len + t0;               // position of the tile's first token
  const int kv_end = p.causal ? pos0 + ntok : seq_len; // keys the tile's last row attends
  const int part = p.part_pf;
  const int parts_req = (seq_len + part - 1) / part;
  const int k0 = z * part, k1 = min(k0 + part, kv_end);
  const int kb0 = k0 / BS, kb1 = (k1 + BS - 1) / BS;
  const int nblocks = kb1 - kb0;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ST * 2 * TB);
  uint64_t* empty = full + ST;
  __shared__ int s_failed;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_failed = 0;
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    for (int i = 0; i < ST; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int32_t* table = p.block_tables + (long long)r * p.max_blocks_per_seq;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      auto phys_of = [&](int kb) {
        const int ph = table[kb];
        return (ph >= 0 && ph < p.num_blocks) ? ph : -1;
      };
      for (int i = 0; i < nblocks; ++i) {
        const int s = i % ST;
        if (i >= ST && !mbar_wait_bounded(empty + s, ((i / ST) - 1) & 1)) {
          flag_error(p.err, PA_ERRFLAG_TIMEOUT);
          s_failed = 1;
          break;
        }
        const int ph = phys_of(kb0 + i);
        if (ph < 0) {
          flag_error(p.err, PA_ERRFLAG_BLOCK_TABLE);
          mbar_arrive(full + s);
        } else {
          uint8_t* st = smem + s * 2 * TB;
          mbar_arrive_expect_tx(full + s, 2 * TB);
          tma_load_4d(st, &tmk, 0, kvh * BS, 0, ph, full + s);
          tma_load_4d(st + TB, &tmv, 0, kvh * BS, 0, ph, full + s);
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // this thread's two rows: warp-local rows lane/4 and lane/4 + 8
  int rt[2], rn[2], rpos[2];
  bool rvalid[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int rho = 16 * warp + (lane >> 2) + 8 * h;
    rt[h] = rho / gp;
    rn[h] = rho % gp;
    rvalid[h] = rt[h] < ntok && rn[h] < nh;
    rpos[h] = pos0 + rt[h];
  }
  // rows covered by this warp: tokens 16w/gp .. (16w+15)/gp
  const int warp_tok_lo = (16 * warp) / gp;
  const int warp_last_pos = pos0 + min((16 * warp + 15) / gp, ntok - 1);
  const bool warp_active = warp_tok_lo < ntok;

  // Q fragments (A operand, rows x head dim), zero for padding rows
  uint32_t qa[G::kKSteps][4];
  {
    const uint32_t* qw[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
      qw[h] = rvalid[h] ? reinterpret_cast<const uint32_t*>(
                              reinterpret_cast<const typename QE::T*>(p.q) +
                              ((long long)(row0 + rt[h]) * p.num_q_heads + h0 + rn[h]) * HEAD)
                        : nullptr;
    const int qq = lane & 3;
#pragma unroll
    for (int ks = 0; ks < G::kKSteps; ++ks) {
      qa[ks][0] = qw[0] ? qw[0][8 * ks + qq] : 0u;
      qa[ks][1] = qw[1] ? qw[1][8 * ks + qq] : 0u;
      qa[ks][2] = qw[0] ? qw[0][8 * ks + 4 + qq] : 0u;
      qa[ks][3] = qw[1] ? qw[1][8 * ks + 4 + qq] : 0u;
    }
  }
  const float c = p.scale * kLog2e;
  float acc[G::kNDim][4];
#pragma unroll
  for (int i = 0; i < G::kNDim; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

  for (int i = 0; i < nblocks; ++i) {
    const int s = i % ST;
    const bool got = mbar_wait_bounded(full + s, (i / ST) & 1);
    if (!__all_sync(0xffffffffu, got)) {
      if (lane == 0) {
        flag_error(p.err, PA_ERRFLAG_TIMEOUT);
        s_failed = 1;
      }
      break;
    }
    const int kb = kb0 + i;
    const int ph = table[kb];
    const int kbase_tok = kb * BS;
    // skip blocks that no row of this warp can see (all keys after its last position)
    const bool useful = warp_active && (ph >= 0 && ph < p.num_blocks) &&
                        (!p.causal || kbase_tok <= warp_last_pos);
    if (useful) {
      const uint32_t kbase = smem_u32(smem + s * 2 * TB);
      const uint32_t vbase = kbase + TB;
      // ---- S = Q K^T over this block's tokens
      float sc[G::kNTok][4];
#pragma unroll
      for (int nt = 0; nt < G::kNTok; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < G::kKSteps; ++ks) {
#pragma unroll
        for (int np2 = 0; np2 < G::kNTok / 2; ++np2) {
          const int mi = lane >> 3;
          const int tok = 16 * np2 + (lane & 7) + 8 * (mi >> 1);
          const int chunk = 2 * ks + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + G::off(tok, chunk), b0, b1, b2, b3);
          mma_16816<QDT>(sc[2 * np2], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_16816<QDT>(sc[2 * np2 + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
      }
      // ---- mask, scale, online softmax (rows h = 0: c0,c1; h = 1: c2,c3)
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < G::kNTok; ++nt) {
        const int key = kbase_tok + 8 * nt + 2 * (lane & 3);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const int k = key + (e & 1);
          const bool ok = rvalid[h] && k < seq_len && k >= k0 && k < k1 && (!p.causal || k <= rpos[h]);
          sc[nt][e] = ok ? sc[nt][e] * c : -INFINITY;
          mx[h] = fmaxf(mx[h], sc[nt][e]);
        }
      }
      float alpha[2], use[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = warp_max_xor(mx[h], 1, 2);
        const float nm = fmaxf(m[h], mx[h]);
        use[h] = nm == -INFINITY ? 0.f : nm;
        alpha[h] = exp2f(m[h] - use[h]);
        m[h] = nm;
      }
      uint32_t pa[G::kNTok][2];
      float add[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < G::kNTok; ++nt) {
        pa[nt][0] = pack2<QDT>(exp2f(sc[nt][0] - use[0]), exp2f(sc[nt][1] - use[0]));
        pa[nt][1] = pack2<QDT>(exp2f(sc[nt][2] - use[1]), exp2f(sc[nt][3] - use[1]));
        const float2 f0 = unpack2<QDT>(pa[nt][0]), f1 = unpack2<QDT>(pa[nt][1]);
        add[0] += f0.x + f0.y;
        add[1] += f1.x + f1.y;
      }
      l[0] = l[0] * alpha[0] + add[0];
      l[1] = l[1] * alpha[1] + add[1];
#pragma unroll
      for (int dn = 0; dn < G::kNDim; ++dn) {
        acc[dn][0] *= alpha[0];
        acc[dn][1] *= alpha[0];
        acc[dn][2] *= alpha[1];
        acc[dn][3] *= alpha[1];
      }
      // ---- O += P V; V tokens past seq_len are zeroed (their P is 0, their bits arbitrary)
      const int rem = seq_len - kbase_tok;
#pragma unroll
      for (int kt = 0; kt < BS / 16; ++kt) {
        const int tk = 16 * kt + 2 * (lane & 3);
        const uint32_t m01 = (tk < rem ? 0xffffu : 0u) | (tk + 1 < rem ? 0xffff0000u : 0u);
        const uint32_t m23 = (tk + 8 < rem ? 0xffffu : 0u) | (tk + 9 < rem ? 0xffff0000u : 0u);
        const bool tail = rem < 16 * kt + 16;
#pragma unroll
        for (int dp = 0; dp < G::kNDim / 2; ++dp) {
          const int mi = lane >> 3;
          const int tok = 16 * kt + (lane & 7) + 8 * (mi & 1);
          const int chunk = 2 * dp + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(vbase + G::off(tok, chunk), b0, b1, b2, b3);
          if (tail) {
            b0 &= m01;
            b1 &= m23;
            b2 &= m01;
            b3 &= m23;
          }
          mma_16816<QDT>(acc[2 * dp], pa[2 * kt][0], pa[2 * kt][1], pa[2 * kt + 1][0], pa[2 * kt + 1][1], b0, b1);
          mma_16816<QDT>(acc[2 * dp + 1], pa[2 * kt][0], pa[2 * kt][1], pa[2 * kt + 1][0], pa[2 * kt + 1][1], b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }
  if (s_failed) return;

  // ---- epilogue: each thread writes its two rows' columns
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l[h] = warp_sum_xor(l[h], 1, 2);
    if (!rvalid[h]) continue;
    const int kv_len = p.causal ? rpos[h] + 1 : seq_len;
    const int parts_row = (kv_len + part - 1) / part;
    if (z >= parts_row) continue;  // this row has no keys in this partition
    const int t = t0 + rt[h];
    const int head = h0 + rn[h];
    const int dcol = 2 * (lane & 3);
    if (parts_row == 1) {
      const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
      typename QE::T* o = reinterpret_cast<typename QE::T*>(p.out) + ((long long)(qs + t) * p.num_q_heads + head) * HEAD;
#pragma unroll
      for (int dn = 0; dn < G::kNDim; ++dn) {
        const uint32_t v = pack2<QDT>(acc[dn][2 * h] * inv, acc[dn][2 * h + 1] * inv);
        *reinterpret_cast<uint32_t*>(o + 8 * dn + dcol) = v;
      }
    } else {
      const long long pi = (long long)p.part_off[r] + (long long)t * parts_req + z;
      float* wa = p.ws_acc + (pi * p.num_q_heads + head) * HEAD;
#pragma unroll
      for (int dn = 0; dn < G::kNDim; ++dn)
        *reinterpret_cast<float2*>(wa + 8 * dn + dcol) = make_float2(acc[dn][2 * h], acc[dn][2 * h + 1]);
      if ((lane & 3) == 0) p.ws_ml[pi * p.num_q_heads + head] = make_float2(m[h], l[h]);
    }
  }
}

template <int QDT, int HEAD, int BS>
cudaError_t launch_t(const AttnParams& p, int num_items, const CUtensorMap* tk, const CUtensorMap* tv,
                     cudaStream_t stream) {
  constexpr int smem = prefill_smem_bytes<HEAD, BS>();
  auto kern = prefill_mma_kernel<QDT, HEAD, BS>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();  // consume it: the caller reports the failure
      return e;
    }
    configured_device = dev;
  }
  dim3 grid(num_items, p.num_kv_heads * p.num_head_groups);
  kern<<<grid, kThreads, smem, stream>>>(p, *tk, *tv);
  return cudaGetLastError();
}

template <int QDT>
cudaError_t launch_shape(const AttnParams& p, int num_items, const CUtensorMap* tk, const CUtensorMap* tv,
                         cudaStream_t s) {
  const int d = p.head_size, bs = p.block_size;
  if (d == 128 && bs == 16) return launch_t<QDT, 128, 16>(p, num_items, tk, tv, s);
  if (d == 128 && bs == 32) return launch_t<QDT, 128, 32>(p, num_items, tk, tv, s);
  if (d == 64 && bs == 16) return launch_t<QDT, 64, 16>(p, num_items, tk, tv, s);
  if (d == 64 && bs == 32) return launch_t<QDT, 64, 32>(p, num_items, tk, tv, s);
  return cudaErrorInvalidValue;
}

}  // namespace

bool prefill_mma_supported(int q_dtype, int kv_dtype, int head_size, int block_size, int group) {
  (void)group;
  if (!(q_dtype == PA_BF16 || q_dtype == PA_F16) || kv_dtype != q_dtype) return false;
  return (head_size == 64 || head_size == 128) && (block_size == 16 || block_size == 32);
}

cudaError_t launch_prefill_mma(const AttnParams& p, int q_dtype, int kv_dtype, int num_items,
                               const CUtensorMap* tmap_k, const CUtensorMap* tmap_v, cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  if (kv_dtype != q_dtype) return cudaErrorInvalidValue;
  if (q_dtype == PA_BF16) return launch_shape<PA_BF16>(p, num_items, tmap_k, tmap_v, stream);
  if (q_dtype == PA_F16) return launch_shape<PA_F16>(p, num_items, tmap_k, tmap_v, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
