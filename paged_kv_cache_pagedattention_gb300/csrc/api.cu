// The C ABI declared in include/pa.h: argument validation, workspace layout,
// tensor-map encoding, kernel selection and launch, the device error word and
// optional event-based kernel tracing.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "pa_internal.h"

namespace {

using pa::AttnParams;

__device__ unsigned g_pa_error_word;

constexpr int kMaxDevices = 64;
// Share of the SMs the prefill tiles' first grid (on the caller's stream) holds while
// the decode rows of a varlen step run beside it on the side stream.
constexpr int kPrefillShareNum = 2;
constexpr int kPrefillShareDen = 3;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

// Per-device lookups below are cached in atomics: host threads may call on the
// same or different devices at once, and a repeated lookup stores the same value.
unsigned* error_word() {
  static std::atomic<unsigned*> cache[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned* w = cache[dev].load(std::memory_order_acquire);
  if (!w) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_pa_error_word) != cudaSuccess) {
      (void)cudaGetLastError();  // consume it: a later launch check must not see it
      return nullptr;
    }
    w = static_cast<unsigned*>(ptr);
    cache[dev].store(w, std::memory_order_release);
  }
  return w;
}

int sm_count() {
  static std::atomic<int> cache[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int dtype_bytes(int dt) {
  switch (dt) {
    case PA_F32: return 4;
    case PA_F16: return 2;
    case PA_BF16: return 2;
    case PA_FP8_E4M3: return 1;
    case PA_FP8_E5M2: return 1;
    case PA_FP8_E4M3_PER_HEAD: return 1;
    case PA_FP8_E5M2_PER_HEAD: return 1;
    default: return 0;
  }
}

// Scaled formats with one scale per KV head are the base format with a scale
// stride of 1 (the kernels read the scale of KV head h at scale[h * stride]).
pa_dtype base_dtype(pa_dtype dt) {
  if (dt == PA_FP8_E4M3_PER_HEAD) return PA_FP8_E4M3;
  if (dt == PA_FP8_E5M2_PER_HEAD) return PA_FP8_E5M2;
  if (dt == PA_NVFP4_PER_HEAD) return PA_NVFP4;
  return dt;
}
int scale_stride_of(pa_dtype dt) {
  return dt == PA_FP8_E4M3_PER_HEAD || dt == PA_FP8_E5M2_PER_HEAD || dt == PA_NVFP4_PER_HEAD ? 1 : 0;
}

// Cache formats (after base_dtype) whose values carry fp32 scales.
bool scaled_dtype(pa_dtype dt) { return dt == PA_FP8_E4M3 || dt == PA_FP8_E5M2 || dt == PA_NVFP4; }

// NVFP4 tiles: whole 16-element groups per row and whole 16-byte pieces per tile.
bool nvfp4_shape_ok(int head_size, int block_size) {
  return head_size % 16 == 0 && ((long long)block_size * head_size) % 256 == 0;
}

// Bytes of one (block, KV head) tile of a cache.
long long tile_bytes(pa_dtype dt, int block_size, int head_size) {
  if (dt == PA_NVFP4) return pa::nvfp4_tile_bytes(block_size, head_size);
  return (long long)block_size * head_size * dtype_bytes(dt);
}

// ------------------------------------------------------------------ partitions

int round_up(int x, int m) { return static_cast<int>(ceil_div(x, m) * m); }

// Partition tokens: doubled from 64 (capped at 4096) until the units of work times
// the partitions fit `ctas_per_sm` CTAs per SM (16 by default: on the Llama-shaped decode,
// 64 x U[512, 4096] tokens x 8 KV heads, 1024-token partitions measured 94.6 us against
// 97.2 us for 512 and 103.9 us for 4096).  Each partition adds a partial state
// per row for the merge, so finer partitions balance the attention grid better but
// cost merge time.  The starting size matters only for small batches, which never
// fill the SMs: on 4 fp32 sequences of 17 to 200 tokens (8 / 2 heads, head 64) the
// attention kernel took 36.6 us with 128-token partitions and 22.0 us with 64.
int default_partition(int num_seqs, int num_kv_heads, int max_seq_len, int block_size, int ctas_per_sm = 16) {
  const long long units = (long long)(num_seqs > 0 ? num_seqs : 1) * (num_kv_heads > 0 ? num_kv_heads : 1);
  const long long target = (long long)ctas_per_sm * sm_count();
  int part = round_up(64, block_size);
  const int cap = round_up(4096, block_size);
  while (part < cap && units * ceil_div(max_seq_len, part) > target) part *= 2;
  while (ceil_div(max_seq_len, part) > 65535) part *= 2;
  return part;
}

int resolve_partition(int requested, int num_seqs, int num_kv_heads, int max_seq_len, int block_size) {
  int part = requested > 0 ? requested : default_partition(num_seqs, num_kv_heads, max_seq_len, block_size);
  while (ceil_div(max_seq_len, part) > 65535) part *= 2;
  return part;
}

// Partitions a row can use under a sliding window: its keys span at most
// window + q_len - 1 positions from a block-aligned origin.
int window_partitions(long long parts, int window, int max_query_len, int block_size, int part) {
  if (window <= 0) return static_cast<int>(parts);
  const long long span = (long long)window + max_query_len - 1 + block_size - 1;
  return static_cast<int>(std::min<long long>(parts, ceil_div(span, part)));
}

int prefill_partition(int part) { return part > 16384 ? part : 16384 / part * part; }

struct DecodeLayout {
  int part;
  long long parts;
  size_t ml_off, acc_off, total;
};

DecodeLayout decode_layout(int num_seqs, int hq, int d, int max_seq_len, int bs, int hkv, int requested) {
  DecodeLayout L;
  L.part = resolve_partition(requested, num_seqs, hkv, max_seq_len, bs);
  L.parts = ceil_div(max_seq_len, L.part);
  const size_t rows = (size_t)num_seqs * (size_t)L.parts;
  L.ml_off = 256;
  L.acc_off = L.ml_off + align256(rows * hq * sizeof(float2));
  L.total = L.acc_off + align256(rows * hq * (size_t)d * sizeof(float));
  return L;
}

struct VarlenLayout {
  int part, part_pf;
  long long parts, parts_pf, max_work;
  size_t off_off, work_off, ml_off, acc_off, total;
};

VarlenLayout varlen_layout(int num_seqs, int total_q, int hq, int hkv, int d, int max_seq_len, int bs,
                           int requested) {
  VarlenLayout L;
  L.part = resolve_partition(requested, num_seqs, hkv, max_seq_len, bs);
  L.part_pf = requested > 0 ? L.part : prefill_partition(L.part);
  L.parts = ceil_div(max_seq_len, L.part);
  L.parts_pf = ceil_div(max_seq_len, L.part_pf);
  const int group = hq / (hkv > 0 ? hkv : 1);
  L.max_work = (ceil_div(total_q, pa::prefill_tile_tokens(group)) + num_seqs) * L.parts_pf;
  const size_t rows = (size_t)num_seqs * (size_t)L.parts + (size_t)total_q * (size_t)L.parts_pf;
  L.off_off = 256;
  L.work_off = L.off_off + align256((size_t)num_seqs * sizeof(int32_t));
  L.ml_off = L.work_off + align256((size_t)L.max_work * sizeof(int4));
  L.acc_off = L.ml_off + align256(rows * hq * sizeof(float2));
  L.total = L.acc_off + align256(rows * hq * (size_t)d * sizeof(float));
  return L;
}

// Shared-prefix decode: partitions of the shared prefixes (part_shared, sized by
// the groups x KV heads units) followed by partitions of the private rests (part).
struct SharedLayout {
  int part, part_shared;
  long long parts_shared, parts_private, parts;
  size_t ml_off, acc_off, total;
};

SharedLayout shared_layout(int num_seqs, int num_groups, int hq, int hkv, int d, int max_seq_len, int bs,
                           int requested) {
  SharedLayout L;
  // The private remainders: in a batch of forks most are short, so the private grid's
  // real CTAs are far fewer than sequences x KV heads x partitions, and a sequence with
  // a long private range (one that shares nothing) is streamed by few long CTAs, each
  // bound by its own copies in flight.  Partitions of at most 2048 tokens give such a
  // sequence twice the CTAs of the plain decode's 4096-token cap (agentic forks + one
  // lone parent: span 0.3681 -> 0.3626 ms; with the earlier tile producer 1024 / 512
  // tokens measured 0.380 / 0.440 ms against 0.364 for 2048: the short remainders'
  // empty CTAs then dominate).
  L.part = requested > 0 ? requested
                         : resolve_partition(std::min(default_partition(num_seqs, hkv, max_seq_len, bs),
                                                      round_up(2048, bs)),
                                             num_seqs, hkv, max_seq_len, bs);
  // The shared-prefix tiles carry a whole group per CTA: ~8 partitions' worth of work
  // items per SM (the persistent tile kernel takes them in turn), and coarser
  // partitions halve the shared partials the merge reads (measured on the agentic
  // forks: 0.442 -> 0.413 ms per step against 32 per SM).  Fixed partitions that fit
  // the resident CTAs in exactly one wave were faster on that workload (8192 tokens:
  // span 0.355 against 0.364 ms) but fall off a cliff when the wave is missed by a few
  // items (6144: 0.452 ms), and the host cannot tell which groups share nothing.
  L.part_shared = requested > 0
                      ? L.part
                      : resolve_partition(default_partition(num_groups > 0 ? num_groups : 1, hkv, max_seq_len, bs, 8),
                                          num_groups > 0 ? num_groups : 1, hkv, max_seq_len, bs);
  L.parts_shared = ceil_div(max_seq_len, L.part_shared);
  L.parts_private = ceil_div(max_seq_len, L.part);
  L.parts = L.parts_shared + L.parts_private;
  const size_t rows = (size_t)num_seqs * (size_t)L.parts;
  L.ml_off = 256;
  L.acc_off = L.ml_off + align256(rows * hq * sizeof(float2));
  L.total = L.acc_off + align256(rows * hq * (size_t)d * sizeof(float));
  return L;
}

// ------------------------------------------------------------------ tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// The cache as a 4-D tensor: dim0 = 128 bytes of a token's row, dim1 = the tokens
// of all heads of one block (Hkv x block_size, stride one row), dim2 = which
// 128-byte piece of the row (stride 128 bytes), dim3 = physical block.  One box is
// a whole (block, head) tile, {128 bytes, block_size, pieces, 1}; in shared memory
// it lands piece-major ([piece][token][128 bytes]) with the 128-byte swizzle.
// With `one_piece` the box is a single piece, {128 bytes, block_size, 1, 1}, so
// the copies of consecutive blocks can be placed side by side per piece.
bool encode_cache_map(CUtensorMap* m, const void* base, int kv_dtype, int num_blocks, int hkv, int bs, int d,
                      bool one_piece = false) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int eb = dtype_bytes(kv_dtype);
  const int row_bytes = d * eb;
  if (row_bytes % 128) return false;
  const int pieces = row_bytes / 128;
  cuuint64_t dims[4] = {(cuuint64_t)(128 / eb), (cuuint64_t)hkv * bs, (cuuint64_t)pieces, (cuuint64_t)num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)row_bytes, 128, (cuuint64_t)hkv * bs * row_bytes};
  cuuint32_t box[4] = {(cuuint32_t)(128 / eb), (cuuint32_t)bs, one_piece ? 1u : (cuuint32_t)pieces, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType t = eb == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  return fn(m, t, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of the K and V caches for the tensor-core kernels.  NVFP4 tiles are
// moved with 1-D bulk copies; their maps are zeroed and never read.
bool cache_maps(CUtensorMap* tk, CUtensorMap* tv, const void* k_cache, const void* v_cache, int kv_dtype,
                int num_blocks, int hkv, int bs, int d) {
  if (kv_dtype == PA_NVFP4) {
    memset(tk, 0, sizeof(*tk));
    memset(tv, 0, sizeof(*tv));
    return true;
  }
  return encode_cache_map(tk, k_cache, kv_dtype, num_blocks, hkv, bs, d) &&
         encode_cache_map(tv, v_cache, kv_dtype, num_blocks, hkv, bs, d);
}

// ------------------------------------------------------------------ tracing

constexpr int kTraceKinds = 9;
bool g_trace_on = false;
struct TraceSlot {
  int kind;
  cudaEvent_t a, b;
};
std::vector<TraceSlot> g_pending;
std::vector<cudaEvent_t> g_event_pool;
int64_t g_launches[kTraceKinds];
double g_ms[kTraceKinds];

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

struct TraceScope {
  int kind;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  TraceScope(int k, cudaStream_t st) : kind(k), s(st) {
    if (g_trace_on) {
      a = take_event();
      if (a) cudaEventRecord(a, s);
    }
  }
  ~TraceScope() {
    if (a) {
      cudaEvent_t b = take_event();
      if (b) {
        cudaEventRecord(b, s);
        g_pending.push_back({kind, a, b});
      } else {
        g_event_pool.push_back(a);
      }
    }
  }
};

void collect_trace() {
  for (const TraceSlot& t : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(t.b) == cudaSuccess && cudaEventElapsedTime(&ms, t.a, t.b) == cudaSuccess) {
      g_launches[t.kind] += 1;
      g_ms[t.kind] += ms;
    }
    g_event_pool.push_back(t.a);
    g_event_pool.push_back(t.b);
  }
  g_pending.clear();
}

// A second stream per device, created on first use, onto which the shared-prefix
// decode forks its private-remainder kernel so both run at once; joined back with
// events before the merge.  Guarded by a mutex: the fork / join pair must not
// interleave between host threads.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool failed = false;
};
std::mutex g_side_mutex;
SideStream g_side[kMaxDevices];

SideStream* side_stream() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& sd = g_side[dev];
  if (sd.failed) return nullptr;
  if (!sd.stream) {
    if (cudaStreamCreateWithFlags(&sd.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess) {
      (void)cudaGetLastError();
      sd.failed = true;
      return nullptr;
    }
  }
  return &sd;
}

pa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks shared by pa_decode and pa_varlen_attn, but for the workspace.
pa_status check_attention_inputs(const void* out, const void* q, const void* k_cache, const void* v_cache,
                                 int32_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* seq_lens, int32_t max_seq_len, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                 pa_dtype q_dtype, pa_dtype kv_dtype, const float* k_scale,
                                 const float* v_scale, int32_t partition_size) {
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PA_ERR_INVALID_ARG;
  if (num_blocks < 1 || max_blocks_per_seq < 1 || max_seq_len < 1 || num_q_heads < 1 || num_kv_heads < 1 ||
      head_size < 1 || block_size < 1)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
  if (partition_size < 0 || (partition_size > 0 && partition_size % block_size)) return PA_ERR_INVALID_ARG;
  if (q_dtype != PA_F32 && q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  const bool kv_scaled = scaled_dtype(kv_dtype);
  if (kv_dtype != q_dtype && !kv_scaled) return PA_ERR_UNSUPPORTED;
  if (kv_scaled && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  if (kv_dtype == PA_NVFP4 && !nvfp4_shape_ok(head_size, block_size)) return PA_ERR_UNSUPPORTED;
  if (head_size > 256) return PA_ERR_UNSUPPORTED;
  if (num_kv_heads * ((num_q_heads / num_kv_heads + 7) / 8) > 65535) return PA_ERR_UNSUPPORTED;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

// Checks shared by pa_decode and pa_varlen_attn.
pa_status check_attention_args(const void* out, const void* q, const void* k_cache, const void* v_cache,
                               int32_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* seq_lens, int32_t max_seq_len, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                               pa_dtype q_dtype, pa_dtype kv_dtype, const float* k_scale,
                               const float* v_scale, int32_t partition_size, void* workspace) {
  const pa_status st = check_attention_inputs(out, q, k_cache, v_cache, num_blocks, block_tables,
                                              max_blocks_per_seq, seq_lens, max_seq_len, num_q_heads,
                                              num_kv_heads, head_size, block_size, q_dtype, kv_dtype, k_scale,
                                              v_scale, partition_size);
  if (st != PA_OK) return st;
  if (!workspace) return PA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return PA_ERR_WORKSPACE;
  return PA_OK;
}

AttnParams base_params(void* out, const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
                       const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                       int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_size, int32_t block_size, float scale, const float* k_scale,
                       const float* v_scale) {
  AttnParams p;
  memset(&p, 0, sizeof(p));
  p.out = out;
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.err = error_word();
  p.num_seqs = num_seqs;
  p.num_blocks = num_blocks;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.head_size = head_size;
  p.block_size = block_size;
  p.group = num_q_heads / num_kv_heads;
  p.num_head_groups = (p.group + 7) / 8;
  p.max_seq_len = max_seq_len;
  p.causal = 1;
  p.scale = scale;
  return p;  // part / part_pf / part_shared are set by the caller
}

}  // namespace

namespace pa {

// The checks pa_decode makes on everything but the workspace, for entry points that
// supply their own workspace (pa_decode_static_workspace), so that they report an
// invalid argument before a size problem, as pa_decode does.
pa_status check_decode_args(const void* out, const void* q, const void* k_cache, const void* v_cache,
                            int32_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, int32_t max_seq_len, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_size, int32_t block_size, float scale,
                            pa_dtype q_dtype, pa_dtype kv_dtype, const float* k_scale, const float* v_scale,
                            int32_t partition_size) {
  const pa_status st = check_attention_inputs(out, q, k_cache, v_cache, num_blocks, block_tables,
                                              max_blocks_per_seq, seq_lens, max_seq_len, num_q_heads,
                                              num_kv_heads, head_size, block_size, q_dtype, base_dtype(kv_dtype),
                                              k_scale, v_scale, partition_size);
  if (st != PA_OK) return st;
  if (!(scale > 0.f) || !(scale < INFINITY)) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

}  // namespace pa

extern "C" {

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG: invalid argument";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: unsupported dtype or shape";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case PA_ERR_BOUNDS: return "PA_ERR_BOUNDS: a device-side bounds check fired";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT: a bounded device wait gave up";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA call or kernel launch failed";
    default: return "unknown pa_status";
  }
}

int32_t pa_version(void) { return 100; }

pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                               int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                               pa_dtype src_dtype, pa_dtype cache_dtype, const float* k_scale,
                               const float* v_scale, pa_stream_t stream) {
  const int scale_stride = scale_stride_of(cache_dtype);
  cache_dtype = base_dtype(cache_dtype);
  if (num_tokens < 0 || num_blocks < 1 || num_kv_heads < 1 || head_size < 1 || block_size < 1)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (src_dtype != PA_F32 && src_dtype != PA_F16 && src_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  const bool cache_scaled = scaled_dtype(cache_dtype);
  if (cache_dtype != src_dtype && !cache_scaled) return PA_ERR_UNSUPPORTED;
  if (cache_scaled && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  if ((head_size * dtype_bytes(src_dtype)) % 16) return PA_ERR_UNSUPPORTED;
  if (cache_dtype == PA_NVFP4 ? !nvfp4_shape_ok(head_size, block_size) : (head_size * dtype_bytes(cache_dtype)) % 16)
    return PA_ERR_UNSUPPORTED;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return PA_ERR_INVALID_ARG;
  pa::ScatterParams p;
  p.scale_stride = scale_stride;
  p.key = key;
  p.value = value;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.slot_mapping = slot_mapping;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.err = error_word();
  p.num_tokens = num_tokens;
  p.num_blocks = num_blocks;
  p.num_kv_heads = num_kv_heads;
  p.head_size = head_size;
  p.block_size = block_size;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TraceScope t(0, s);
  return cuda_status(pa::launch_reshape_and_cache(p, src_dtype, cache_dtype, s));
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping, int32_t num_pairs,
                         int32_t num_blocks, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                         pa_dtype cache_dtype, pa_stream_t stream) {
  if (num_pairs < 0 || num_blocks < 1 || num_kv_heads < 1 || head_size < 1 || block_size < 1)
    return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_mapping) return PA_ERR_INVALID_ARG;
  cache_dtype = base_dtype(cache_dtype);
  if (cache_dtype == PA_NVFP4) {
    if (!nvfp4_shape_ok(head_size, block_size)) return PA_ERR_UNSUPPORTED;
  } else {
    const int eb = dtype_bytes(cache_dtype);
    if (eb == 0) return PA_ERR_UNSUPPORTED;
    if ((head_size * eb) % 16) return PA_ERR_UNSUPPORTED;
  }
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return PA_ERR_INVALID_ARG;
  pa::CopyParams p;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_mapping = block_mapping;
  p.err = error_word();
  p.num_pairs = num_pairs;
  p.num_blocks = num_blocks;
  p.block_bytes = (long long)num_kv_heads * tile_bytes(cache_dtype, block_size, head_size);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TraceScope t(7, s);
  return cuda_status(pa::launch_copy_blocks(p, s));
}

int32_t pa_default_partition_size(int32_t num_seqs, int32_t num_kv_heads, int32_t max_seq_len,
                                  int32_t block_size) {
  if (block_size < 1 || max_seq_len < 1) return 0;
  return default_partition(num_seqs, num_kv_heads, max_seq_len, block_size);
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_size, int32_t max_seq_len, int32_t block_size,
                                int32_t partition_size) {
  if (num_seqs < 1 || num_q_heads < 1 || head_size < 1 || max_seq_len < 1 || block_size < 1) return 256;
  return decode_layout(num_seqs, num_q_heads, head_size, max_seq_len, block_size, num_kv_heads,
                       partition_size)
      .total;
}

pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
                    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                    int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                    int32_t head_size, int32_t block_size, float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                    const float* k_scale, const float* v_scale, int32_t partition_size, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream) {
  return pa_decode_windowed(out, q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                            num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, scale, 0,
                            q_dtype, kv_dtype, k_scale, v_scale, partition_size, workspace, workspace_bytes, stream);
}

pa_status pa_decode_windowed(void* out, const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
                             const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                             int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_size, int32_t block_size, float scale, int32_t window,
                             pa_dtype q_dtype, pa_dtype kv_dtype, const float* k_scale, const float* v_scale,
                             int32_t partition_size, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  const int scale_stride = scale_stride_of(kv_dtype);
  kv_dtype = base_dtype(kv_dtype);
  if (num_seqs < 0 || window < 0) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  pa_status st = check_attention_args(out, q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq,
                                      seq_lens, max_seq_len, num_q_heads, num_kv_heads, head_size, block_size,
                                      q_dtype, kv_dtype, k_scale, v_scale, partition_size, workspace);
  if (st != PA_OK) return st;
  if (!(scale > 0.f) || !(scale < INFINITY)) return PA_ERR_INVALID_ARG;
  const DecodeLayout L =
      decode_layout(num_seqs, num_q_heads, head_size, max_seq_len, block_size, num_kv_heads, partition_size);
  if (workspace_bytes < L.total) return PA_ERR_WORKSPACE;
  AttnParams p = base_params(out, q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                             num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, scale,
                             k_scale, v_scale);
  p.scale_stride = scale_stride;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.num_rows = num_seqs;
  p.max_query_len = 1;
  p.part = p.part_pf = L.part;
  p.part_shared = L.part;
  p.max_partitions = static_cast<int>(L.parts);
  p.window = window;
  p.ws_ml = reinterpret_cast<float2*>(ws + L.ml_off);
  p.ws_acc = reinterpret_cast<float*>(ws + L.acc_off);
  const int grid_z = window_partitions(L.parts, window, 1, block_size, L.part);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (pa::decode_mma_supported(q_dtype, kv_dtype, head_size, block_size, p.group)) {
    CUtensorMap tk, tv;
    if (!cache_maps(&tk, &tv, k_cache, v_cache, kv_dtype, num_blocks, num_kv_heads, block_size, head_size))
      return PA_ERR_CUDA;
    TraceScope t(1, s);
    e = pa::launch_decode_mma(p, q_dtype, kv_dtype, grid_z, &tk, &tv, s);
  } else {
    TraceScope t(1, s);
    e = pa::launch_attn_generic(p, q_dtype, kv_dtype, grid_z, -1, s);
  }
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (L.parts > 1) {
    TraceScope t(2, s);
    e = pa::launch_merge(p, q_dtype, s);
  }
  return cuda_status(e);
}

size_t pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_groups, int32_t num_q_heads,
                                              int32_t num_kv_heads, int32_t head_size, int32_t max_seq_len,
                                              int32_t block_size, int32_t partition_size) {
  if (num_seqs < 1 || num_q_heads < 1 || head_size < 1 || max_seq_len < 1 || block_size < 1) return 256;
  return shared_layout(num_seqs, num_groups, num_q_heads, num_kv_heads, head_size, max_seq_len, block_size,
                       partition_size)
      .total;
}

pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  int32_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                  int32_t block_size, float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                                  const float* k_scale, const float* v_scale, const int32_t* group_start,
                                  const int32_t* group_shared_blocks, int32_t num_groups,
                                  int32_t max_group_size, int32_t partition_size, void* workspace,
                                  size_t workspace_bytes, pa_stream_t stream) {
  const int scale_stride = scale_stride_of(kv_dtype);
  kv_dtype = base_dtype(kv_dtype);
  if (num_seqs < 0 || num_groups < 0) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  pa_status st = check_attention_args(out, q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq,
                                      seq_lens, max_seq_len, num_q_heads, num_kv_heads, head_size, block_size,
                                      q_dtype, kv_dtype, k_scale, v_scale, partition_size, workspace);
  if (st != PA_OK) return st;
  if (!(scale > 0.f) || !(scale < INFINITY)) return PA_ERR_INVALID_ARG;
  if (num_groups > 0 && (!group_start || !group_shared_blocks)) return PA_ERR_INVALID_ARG;
  if (max_group_size < 1 || max_group_size > 8) return PA_ERR_UNSUPPORTED;
  const SharedLayout L = shared_layout(num_seqs, num_groups, num_q_heads, num_kv_heads, head_size, max_seq_len,
                                       block_size, partition_size);
  if (workspace_bytes < L.total) return PA_ERR_WORKSPACE;
  const bool fast = pa::decode_mma_supported(q_dtype, kv_dtype, head_size, block_size,
                                             num_q_heads / num_kv_heads);
  if (!fast || num_groups == 0 || max_group_size < 2)  // nothing to share, or no tensor-core path
    return pa_decode(out, q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                     num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, scale, q_dtype,
                     kv_dtype, k_scale, v_scale, partition_size, workspace, workspace_bytes, stream);
  AttnParams p = base_params(out, q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                             num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, scale,
                             k_scale, v_scale);
  p.scale_stride = scale_stride;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.num_rows = num_seqs;
  p.max_query_len = 1;
  p.part = p.part_pf = L.part;
  p.part_shared = L.part_shared;
  p.max_partitions = static_cast<int>(L.parts);
  p.ws_ml = reinterpret_cast<float2*>(ws + L.ml_off);
  p.ws_acc = reinterpret_cast<float*>(ws + L.acc_off);
  p.group_start = group_start;
  p.group_shared_blocks = group_shared_blocks;
  p.num_groups = num_groups;
  p.max_group_size = max_group_size;
  p.force_partials = 1;
  CUtensorMap tk, tv;
  if (!cache_maps(&tk, &tv, k_cache, v_cache, kv_dtype, num_blocks, num_kv_heads, block_size, head_size))
    return PA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  {
    std::lock_guard<std::mutex> lock(g_side_mutex);
    SideStream* side = side_stream();
    TraceScope span(6, s);  // shared prefixes and private rests together
    cudaStream_t s2 = s;
    if (side && cudaEventRecord(side->fork, s) == cudaSuccess &&
        cudaStreamWaitEvent(side->stream, side->fork, 0) == cudaSuccess)
      s2 = side->stream;
    {
      TraceScope t(5, s);
      e = scaled_dtype(kv_dtype)
              ? pa::launch_shared_prefix(p, q_dtype, kv_dtype, static_cast<int>(L.parts_shared), &tk, &tv, s)
              : pa::launch_shared_prefix_tiles(p, q_dtype, static_cast<int>(L.parts_shared), &tk, &tv, s);
    }
    if (e == cudaSuccess) {
      TraceScope t(1, s2);
      e = pa::launch_decode_mma(p, q_dtype, kv_dtype, static_cast<int>(L.parts_private), &tk, &tv, s2);
    }
    if (s2 != s) {  // join, even after a failed launch, so the caller's stream stays ordered
      if (cudaEventRecord(side->join, s2) != cudaSuccess || cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess)
        e = cudaErrorUnknown;
    }
  }
  if (e != cudaSuccess) return PA_ERR_CUDA;
  TraceScope t(2, s);
  return cuda_status(pa::launch_merge(p, q_dtype, s));
}

size_t pa_varlen_workspace_size(int32_t num_seqs, int32_t total_q_tokens, int32_t max_query_len,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                int32_t max_seq_len, int32_t block_size, int32_t partition_size) {
  (void)max_query_len;
  if (num_seqs < 1 || total_q_tokens < 1 || num_q_heads < 1 || num_kv_heads < 1 || head_size < 1 ||
      max_seq_len < 1 || block_size < 1)
    return 256;
  return varlen_layout(num_seqs, total_q_tokens, num_q_heads, num_kv_heads, head_size, max_seq_len, block_size,
                       partition_size)
      .total;
}

pa_status pa_varlen_attn(void* out, const void* q, const void* k_cache, const void* v_cache, int32_t num_blocks,
                         const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* query_start_loc,
                         const int32_t* seq_lens, int32_t num_seqs, int32_t total_q_tokens, int32_t max_query_len,
                         int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                         int32_t block_size, float scale, int32_t causal, pa_dtype q_dtype, pa_dtype kv_dtype,
                         const float* k_scale, const float* v_scale, int32_t partition_size, void* workspace,
                         size_t workspace_bytes, pa_stream_t stream) {
  return pa_varlen_attn_windowed(out, q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq,
                                 query_start_loc, seq_lens, num_seqs, total_q_tokens, max_query_len, max_seq_len,
                                 num_q_heads, num_kv_heads, head_size, block_size, scale, 0, causal, q_dtype,
                                 kv_dtype, k_scale, v_scale, partition_size, workspace, workspace_bytes, stream);
}

pa_status pa_varlen_attn_windowed(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  int32_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* query_start_loc, const int32_t* seq_lens, int32_t num_seqs,
                                  int32_t total_q_tokens, int32_t max_query_len, int32_t max_seq_len,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                  float scale, int32_t window, int32_t causal, pa_dtype q_dtype, pa_dtype kv_dtype,
                                  const float* k_scale, const float* v_scale, int32_t partition_size,
                                  void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  const int scale_stride = scale_stride_of(kv_dtype);
  kv_dtype = base_dtype(kv_dtype);
  if (num_seqs < 0 || total_q_tokens < 0 || window < 0) return PA_ERR_INVALID_ARG;
  if (window > 0 && !causal) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q_tokens == 0) return PA_OK;
  if (!query_start_loc || max_query_len < 1) return PA_ERR_INVALID_ARG;
  pa_status st = check_attention_args(out, q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq,
                                      seq_lens, max_seq_len, num_q_heads, num_kv_heads, head_size, block_size,
                                      q_dtype, kv_dtype, k_scale, v_scale, partition_size, workspace);
  if (st != PA_OK) return st;
  if (!(scale > 0.f) || !(scale < INFINITY)) return PA_ERR_INVALID_ARG;
  const VarlenLayout L = varlen_layout(num_seqs, total_q_tokens, num_q_heads, num_kv_heads, head_size,
                                       max_seq_len, block_size, partition_size);
  if (workspace_bytes < L.total) return PA_ERR_WORKSPACE;
  AttnParams p = base_params(out, q, k_cache, v_cache, num_blocks, block_tables, max_blocks_per_seq, seq_lens,
                             num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, scale,
                             k_scale, v_scale);
  p.scale_stride = scale_stride;
  // prefill tiles are claimed by index over (work item, KV head group)
  if (L.max_work * p.num_kv_heads * p.num_head_groups > (1LL << 30)) return PA_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.query_start_loc = query_start_loc;
  p.num_rows = total_q_tokens;
  p.max_query_len = max_query_len;
  p.part = L.part;
  p.part_pf = L.part_pf;
  p.part_shared = L.part;
  p.max_partitions = static_cast<int>(L.parts);
  p.causal = causal ? 1 : 0;
  p.window = window;
  const int grid_dec = window_partitions(L.parts, window, 1, block_size, L.part);
  const int grid_all = window_partitions(L.parts, window, max_query_len, block_size, L.part);
  const int grid_pf = window_partitions(L.parts_pf, window, max_query_len, block_size, L.part_pf);
  int32_t* work_count = reinterpret_cast<int32_t*>(ws);
  p.plan_ok = reinterpret_cast<int32_t*>(ws + 4);
  p.work_claim = reinterpret_cast<int32_t*>(ws + 8);
  p.work_full = reinterpret_cast<int32_t*>(ws + 12);
  int32_t* part_off = reinterpret_cast<int32_t*>(ws + L.off_off);
  int4* work = reinterpret_cast<int4*>(ws + L.work_off);
  p.part_off = part_off;
  p.work = work;
  p.work_count = work_count;
  p.ws_ml = reinterpret_cast<float2*>(ws + L.ml_off);
  p.ws_acc = reinterpret_cast<float*>(ws + L.acc_off);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  {
    TraceScope t(3, s);
    e = pa::launch_varlen_plan(p, part_off, work, work_count, static_cast<int>(L.max_work), s);
  }
  if (e != cudaSuccess) return PA_ERR_CUDA;
  const bool fast_decode = pa::decode_mma_supported(q_dtype, kv_dtype, head_size, block_size, p.group);
  const bool fast_prefill = pa::prefill_tc_supported(q_dtype, kv_dtype, head_size, block_size);
  // whole-tile boxes for K and V; the prefill tiles copy K one piece at a time
  CUtensorMap tk, tv, tk1;
  const bool prefill_tiles = fast_prefill && max_query_len > 1;
  if (fast_decode || prefill_tiles) {
    if (!cache_maps(&tk, &tv, k_cache, v_cache, kv_dtype, num_blocks, num_kv_heads, block_size, head_size))
      return PA_ERR_CUDA;
  }
  if (prefill_tiles && kv_dtype == PA_NVFP4) {
    memset(&tk1, 0, sizeof(tk1));  // NVFP4 tiles move with 1-D bulk copies
  } else if (prefill_tiles &&
             !encode_cache_map(&tk1, k_cache, kv_dtype, num_blocks, num_kv_heads, block_size, head_size, true)) {
    return PA_ERR_CUDA;
  }
  // Single-token rows: tensor-core decode kernel, else the generic kernel.
  // Multi-token rows: tensor-core prefill tiles, else the generic kernel.
  const bool multi = max_query_len > 1;
  if (!fast_decode && !(multi && fast_prefill)) {
    TraceScope t(1, s);  // generic kernel for every row
    e = pa::launch_attn_generic(p, q_dtype, kv_dtype, std::max(grid_all, grid_pf), -1, s);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  } else {
    // The decode rows (HBM-bound) and the prefill tiles (tensor-bound) touch disjoint
    // rows and partial slots, so they run concurrently: the tiles on the caller's
    // stream, right behind the plan, so that their CTAs are resident first; the decode
    // rows on the side stream, joined back before the merge.  The tiles' persistent
    // grid then holds about two thirds of the SMs (one CTA per SM) and the decode rows
    // keep the rest: HBM stays near its copy rate from ~80 free SMs on (an SM-holding
    // probe measured 6.9 of 7.1 TB/s).  A second grid over every SM follows the decode
    // rows and claims whatever tiles are left, so SMs the decode rows free up go to the
    // tiles; if the tiles finish first, the decode grid spreads over every SM.
    std::lock_guard<std::mutex> lock(g_side_mutex);
    SideStream* side = multi ? side_stream() : nullptr;
    TraceScope span(8, s);  // decode rows and prefill tiles together
    cudaStream_t s2 = s;
    if (side && cudaEventRecord(side->fork, s) == cudaSuccess &&
        cudaStreamWaitEvent(side->stream, side->fork, 0) == cudaSuccess)
      s2 = side->stream;
    const int sms = sm_count();
    const bool split = multi && fast_prefill && s2 != s;
    if (multi && fast_prefill) {
      TraceScope t(4, s);
      const int ctas = split ? std::max(1, (sms * kPrefillShareNum) / kPrefillShareDen) : sms;
      e = pa::launch_prefill_tc(p, q_dtype, kv_dtype, static_cast<int>(L.max_work), ctas, &tk1, &tv, s);
    } else if (multi) {
      TraceScope t(1, s);
      e = pa::launch_attn_generic(p, q_dtype, kv_dtype, grid_pf, 1, s);
    }
    if (e == cudaSuccess) {
      TraceScope t(1, s2);
      e = fast_decode ? pa::launch_decode_mma(p, q_dtype, kv_dtype, grid_dec, &tk, &tv, s2)
                      : pa::launch_attn_generic(p, q_dtype, kv_dtype, grid_dec, 0, s2);
    }
    if (e == cudaSuccess && split) {  // the tiles still unclaimed
      TraceScope t(4, s2);
      e = pa::launch_prefill_tc(p, q_dtype, kv_dtype, static_cast<int>(L.max_work), sms, &tk1, &tv, s2);
    }
    if (s2 != s) {  // join, even after a failed launch, so the caller's stream stays ordered
      if (cudaEventRecord(side->join, s2) != cudaSuccess || cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess)
        e = cudaErrorUnknown;
    }
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  if (L.parts > 1 || L.parts_pf > 1) {
    TraceScope t(2, s);
    e = pa::launch_merge(p, q_dtype, s);
  }
  return cuda_status(e);
}

pa_status pa_get_error_flags(uint32_t* flags, int32_t clear, pa_stream_t stream) {
  if (!flags) return PA_ERR_INVALID_ARG;
  unsigned* w = error_word();
  if (!w) return PA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned host = 0;
  if (cudaMemcpyAsync(&host, w, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  if (clear) {
    if (cudaMemsetAsync(w, 0, sizeof(unsigned), s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  }
  *flags = host;
  const unsigned errors = host & ~PA_ERRFLAG_SHARED_MISMATCH;  // the diagnostic bit is no error
  if (errors & ~PA_ERRFLAG_TIMEOUT) return PA_ERR_BOUNDS;
  if (errors & PA_ERRFLAG_TIMEOUT) return PA_ERR_TIMEOUT;
  return PA_OK;
}

pa_status pa_trace_enable(int32_t on) {
  g_trace_on = on != 0;
  return PA_OK;
}

pa_status pa_trace_read(int32_t kind, int64_t* launches, double* total_ms, int32_t reset) {
  if (kind < 0 || kind >= kTraceKinds) return PA_ERR_INVALID_ARG;
  collect_trace();
  if (launches) *launches = g_launches[kind];
  if (total_ms) *total_ms = g_ms[kind];
  if (reset) {
    for (int k = 0; k < kTraceKinds; ++k) {
      g_launches[k] = 0;
      g_ms[k] = 0.0;
    }
  }
  return PA_OK;
}

}  // extern "C"
