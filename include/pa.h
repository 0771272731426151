/*
 * pa.h -- C ABI of the paged KV cache attention library (libpa.so), GB300 / sm_103a.
 *
 * The library implements the data-parallel hot path of paged KV cache serving:
 *   1. pa_reshape_and_cache  writes the K/V of new tokens into fixed-size physical
 *                            blocks through a per-token slot mapping
 *                            (pa_copy_blocks duplicates blocks for copy-on-write);
 *   2. pa_decode             PagedAttention decode: one query token per sequence
 *                            attends the sequence's whole cached context, read
 *                            through its block table (split-K over the context
 *                            plus a merge of the partial softmax states);
 *   3. pa_varlen_attn        attention of a flattened variable-length batch that
 *                            mixes chunked-prefill requests (many query tokens on
 *                            a cached prefix, causal within the chunk) and decode
 *                            requests (one query token).
 *
 * Sources, cited by key:
 *   [AGENTIC] "宣稱省下 106 倍成本：vLLM 怎麼把 Serving 系統校準給 Agentic Workload"
 *             (datasciocean.com, ai-concept/vllm-agentic-serving)
 *   [NOTES]   "大模型推理优化学习笔记" (fishingrodd.cn, 2026/10/30)
 *   [LINEAGE] "从静态批处理到状态化推理集群" (wineandchord.com,
 *             llm/landscape/lineages/inference-serving)
 *   [ARCH]    summary of a vLLM V1 architecture deep-dive
 *             (ai.youdonthavefriends.com, llm/ai/deep-analysis/2026/08/08/vllm-architecture)
 *   [DSV41]   vLLM x DeepSeek-V4.1-Flash agentic throughput write-up (yaoyouai.cn)
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory.  Every array argument is a DEVICE pointer owned by the caller, unless
 *   the argument says otherwise.  The library allocates no device memory and keeps
 *   no per-call state; scratch memory is the caller's `workspace`, sized by the
 *   matching *_workspace_size() query.  This follows [LINEAGE]'s rule that
 *   running out of memory is handled at admission, never while writing KV.
 * Library state.  What the library does hold, once per device and for the life of
 *   the process: one CUDA stream and two events, created by the first
 *   pa_decode_shared_prefix call or pa_varlen_attn call with multi-token rows
 *   (those calls run two kernels at once: they fork the second stream from
 *   `stream` and join it back); two file-scope device symbols, the error word
 *   (pa_get_error_flags) and the pa_decode_static_workspace array; and, on the
 *   host, each kernel's shared-memory opt-in and occupancy figure, and the
 *   tracing counters.
 * Sizes and partitions.  The attention calls and their workspace queries take a
 *   partition_size (0 = the default): split-K splits each context into partitions
 *   of that many tokens, and the partition count sizes the workspace.  The default
 *   depends on the number of (sequence, KV head) units and the SM count, which is
 *   why the workspace queries also take num_kv_heads.
 * Streams.  All compute calls are asynchronous on `stream` (a cudaStream_t;
 *   NULL is the legacy default stream).  Calls on one stream run in issue order:
 *   write the new tokens with pa_reshape_and_cache, then attend.
 * Cache layout.  k_cache and v_cache are separate tensors of shape
 *   [num_blocks][num_kv_heads][block_size][head_size], row-major, element type
 *   kv_dtype.  One (block, kv head) tile of block_size x head_size elements is
 *   contiguous.  Bytes per block per layer (K and V together) are
 *   2 x block_size x num_kv_heads x head_size x dtype_bytes ([ARCH] Part 1,
 *   KV cache manager).  Both tensors must start on a 16-byte boundary.
 * NVFP4 caches.  [DSV41] "三、第二招：把能合的内核全合成一个" names an NVFP4 KV
 *   format 45% smaller than FP8; read as NVIDIA's NVFP4: 4-bit E2M1 elements (1 sign,
 *   2 exponent bits with bias 1, 1 mantissa bit: +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}), one
 *   E4M3 block scale per 16 consecutive elements of a token's head vector, and the
 *   fp32 scale k_scale / v_scale.  Shape [num_blocks][num_kv_heads][tile_bytes]
 *   bytes, tile_bytes = 9 x block_size x head_size / 16: a tile holds block_size
 *   code rows of head_size/2 bytes (element 2i in the low nibble of byte i,
 *   element 2i+1 in the high nibble), then block_size scale rows of head_size/16
 *   bytes.  head_size must be a multiple of 16 and block_size x head_size a
 *   multiple of 256 (whole 16-byte tiles).  Element value = E2M1(code) x
 *   E4M3(block scale) x scale.
 * Slots.  A token with flat slot s lives in physical block s / block_size at
 *   offset s % block_size ([ARCH] Part 1, forward pass: slot_mapping).  A
 *   negative slot marks a padding token and is skipped.
 * Block tables.  block_tables is int32 [num_seqs][max_blocks_per_seq]; entry
 *   [i][j] is the physical block that holds logical block j of sequence i
 *   ([LINEAGE] "PagedAttention": (sequence, logical block) -> physical block).
 *   Physical blocks may be in any order and may be shared by several sequences
 *   ([AGENTIC] "統一分頁 + 共用池").  Only the first ceil(seq_len/block_size)
 *   entries of a row are read.
 * Heads.  num_q_heads is a multiple of num_kv_heads; query head h reads KV head
 *   h / (num_q_heads / num_kv_heads) (grouped-query attention).
 * Positions.  seq_lens[i] counts all tokens of sequence i INCLUDING the new
 *   ones.  The q_len new query tokens of a request are its last q_len positions;
 *   query j (0-based) sits at position seq_len - q_len + j and, when causal,
 *   attends keys 0..position ([ARCH] Part 1: flattened batch, positions + mask).
 * Numerics.  Scores and the softmax run in fp32 with a running max and sum
 *   ([AGENTIC] "Online softmax"); the output is rounded once to q_dtype.
 *   FP8 caches carry fp32 scales (k_scale, v_scale: device pointers to one float
 *   each, or to num_kv_heads floats with the *_PER_HEAD formats, KV head h using
 *   [h]): stored code = fp8(x / scale), rounded to nearest even with saturation to
 *   +-448 (e4m3) or +-57344 (e5m2); value = fp8 decode x scale.  NVFP4 caches
 *   (PA_NVFP4, PA_NVFP4_PER_HEAD) carry the same fp32 scales; see pa_reshape_and_cache.
 * Errors.  Argument checks that need no device data return synchronously with
 *   a status and launch nothing.  Inputs that live on the device (block-table
 *   entries, slots, sequence lengths, query offsets) are checked by the kernels:
 *   an out-of-range value is never dereferenced -- the access is skipped and a
 *   bit is OR-ed into the device error word, which pa_get_error_flags() reads.
 *   Launch failures return PA_ERR_CUDA.  No C++ exception crosses this ABI.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pa_stream_t; /* same type as cudaStream_t */

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* a null pointer, a non-positive size, inconsistent shapes */
  PA_ERR_UNSUPPORTED = 2, /* a dtype combination or shape the library does not handle */
  PA_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or smaller than required */
  PA_ERR_BOUNDS = 4,      /* returned by pa_get_error_flags when a device check fired */
  PA_ERR_TIMEOUT = 5,     /* a bounded device wait gave up (see PA_ERRFLAG_TIMEOUT) */
  PA_ERR_CUDA = 6         /* a CUDA runtime call or kernel launch failed */
} pa_status;

/* Element formats.  The first four are the formats of the serving path (queries and
 * caches in fp32 / f16 / bf16, caches in FP8 e4m3); the rest are more KV formats:
 * FP8 e5m2, one FP8 scale per KV head, and NVFP4 ([DSV41] "三、第二招"). */
typedef enum pa_dtype {
  PA_F32 = 0,
  PA_F16 = 1,
  PA_BF16 = 2,
  PA_FP8_E4M3 = 3, /* cache only: stored as uint8 codes with a per-tensor fp32 scale */
  PA_FP8_E5M2 = 4, /* cache only: as PA_FP8_E4M3, 5 exponent and 2 mantissa bits */
  PA_FP8_E4M3_PER_HEAD = 5, /* as PA_FP8_E4M3 with one scale per KV head: k_scale and */
  PA_FP8_E5M2_PER_HEAD = 6, /* v_scale point to num_kv_heads floats (head h: [h]) */
  PA_NVFP4 = 7,             /* cache only: E2M1 codes + E4M3 block scales + fp32 scale */
  PA_NVFP4_PER_HEAD = 8     /* as PA_NVFP4 with one fp32 scale per KV head */
} pa_dtype;

/* Bits of the device error word (pa_get_error_flags). */
#define PA_ERRFLAG_BLOCK_TABLE 0x1u /* a block-table entry outside [0, num_blocks) */
#define PA_ERRFLAG_SLOT 0x2u        /* a slot >= num_blocks * block_size */
#define PA_ERRFLAG_SEQ_LEN 0x4u     /* seq_len <= 0, > max_seq_len or > max_blocks_per_seq*block_size */
#define PA_ERRFLAG_QUERY 0x8u       /* query_start_loc decreasing, q_len > seq_len or > max_query_len */
#define PA_ERRFLAG_TIMEOUT 0x10u    /* a bounded wait for an asynchronous copy gave up */
/* Diagnostic, not an error: pa_decode_shared_prefix met a member whose block-table
 * entry differs from the group's first member on a block declared shared.  The
 * output is unaffected: that member read its own block. */
#define PA_ERRFLAG_SHARED_MISMATCH 0x20u

/* Human-readable name of a status code.  Never NULL. */
const char* pa_status_string(pa_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t pa_version(void);

/*
 * pa_reshape_and_cache -- scatter new tokens' K and V into the paged cache.
 * [NOTES] "Prefill 与 Decode": prefill stores K/V for every prompt token and each
 * decode step appends the new token's K/V.  [ARCH] Part 1, forward pass: input
 * preparation builds slot_mapping, one flat slot per new token.
 *
 *   key, value     [num_tokens][num_kv_heads][head_size], src_dtype, rows contiguous
 *   k_cache, v_cache  cache tensors (layout above), cache_dtype
 *   slot_mapping   int64 [num_tokens]; slot < 0 skips the token; a slot >=
 *                  num_blocks*block_size is skipped and sets PA_ERRFLAG_SLOT.
 *                  Two tokens with the same slot in one call: which one lands is
 *                  unspecified.
 *   cache_dtype == src_dtype copies the bits exactly.  cache_dtype == PA_FP8_E4M3
 *   or PA_FP8_E5M2 (src f32/f16/bf16) stores fp8_rne_satfinite(float(x) / *k_scale)
 *   (resp. v; saturation at +-448 for e4m3, +-57344 for e5m2),
 *   the division being IEEE fp32 division.  k_scale / v_scale: device pointers to
 *   one float each, used only for FP8 and NVFP4 (may be NULL otherwise).
 *   cache_dtype == PA_NVFP4 (src f32/f16/bf16): for each group of 16 consecutive
 *   elements of a (token, head) row with largest magnitude a, with s = *k_scale
 *   (resp. v) and every product / quotient one IEEE fp32 operation: the block
 *   scale is e4m3_rne_satfinite(a / (6 s)), of value b; each element x is stored as
 *   e2m1_rne_satfinite(x / (s b)) (ties to the even code, saturating at +-6, the
 *   sign kept, so small negatives give code 0x8); a group with b == 0 stores zero
 *   codes.  Non-finite inputs give unspecified codes.
 *   head_size * dtype_bytes must be a multiple of 16 bytes for both dtypes (NVFP4:
 *   the tile rule of the cache layout above).
 */
pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int32_t num_tokens, int32_t num_blocks,
                               int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                               pa_dtype src_dtype, pa_dtype cache_dtype, const float* k_scale,
                               const float* v_scale, pa_stream_t stream);

/*
 * pa_copy_blocks -- copy whole physical blocks of the paged cache (copy-on-write).
 * [AGENTIC] "統一分頁 + 共用池": with reference counting and copy-on-write, forked
 * sequences' block tables point at the same physical blocks, and a block is
 * duplicated only when shared content has to change.  [LINEAGE] "Prefix reuse":
 * a shared block that is not yet full must be copied before either branch writes
 * its next token into it; otherwise one branch overwrites the other's history.
 * The caller (which owns the reference counts) picks the destination block, calls
 * this, points the writing branch's block table at the copy, then writes.
 *
 *   k_cache, v_cache  cache tensors (layout above), cache_dtype (any pa_dtype;
 *                  only its size matters: the bytes are copied exactly; an NVFP4
 *                  block is num_kv_heads tiles of codes and block scales)
 *   block_mapping  int64 [num_pairs][2], pairs (src, dst): block dst of both
 *                  tensors becomes a copy of block src (all KV heads, all
 *                  block_size slots).  A pair with src or dst outside
 *                  [0, num_blocks) is skipped and sets PA_ERRFLAG_BLOCK_TABLE;
 *                  src == dst is a no-op.  Destinations must be distinct and no
 *                  destination may also be a source in the same call (otherwise
 *                  the result is unspecified).
 *   head_size * dtype_bytes must be a multiple of 16; both tensors 16-byte aligned.
 * num_pairs == 0 returns PA_OK and launches nothing.
 */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping, int32_t num_pairs,
                         int32_t num_blocks, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                         pa_dtype cache_dtype, pa_stream_t stream);

/*
 * Context tokens per split-K partition that pa_decode / pa_varlen_attn use when
 * called with partition_size == 0.  A multiple of block_size.  Chosen from the
 * problem size and the device's SM count (current device).
 */
int32_t pa_default_partition_size(int32_t num_seqs, int32_t num_kv_heads, int32_t max_seq_len,
                                  int32_t block_size);

/*
 * Bytes of workspace pa_decode needs.  partition_size == 0 means the default
 * (pa_default_partition_size with the current device; pass num_kv_heads through
 * num_kv_heads).  Always >= 256: the first bytes hold internal bookkeeping.
 * num_kv_heads and partition_size are parameters because the partition count
 * sizes the workspace (one partial state per sequence, query head and partition)
 * and the default partition size depends on sequences x KV heads.
 */
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_size, int32_t max_seq_len, int32_t block_size,
                                int32_t partition_size);

/*
 * pa_decode -- PagedAttention decode, one query token per sequence.
 * [NOTES] "Prefill 与 Decode" / "Decode": the new token's Q attends the K/V of all
 * the sequence's cached tokens (including its own, written just before);
 * [LINEAGE] "PagedAttention": the kernel reads K/V through the block table.
 * Long contexts are split into partitions of partition_size tokens whose partial
 * softmax states (running max, weight sum, weighted sum) are merged afterwards
 * with the rescale-and-add rule of [AGENTIC] "Online softmax".
 *
 *   out            [num_seqs][num_q_heads][head_size], q_dtype (written)
 *   q              [num_seqs][num_q_heads][head_size], q_dtype (f32, f16 or bf16)
 *   k_cache, v_cache  cache tensors, kv_dtype; kv_dtype == q_dtype, or an FP8 / NVFP4
 *                  format with q_dtype f16/bf16 (k_scale / v_scale then required)
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]
 *   seq_lens       int32 [num_seqs], each in [1, max_seq_len]
 *   max_seq_len    host-side upper bound of seq_lens (sizes the launch)
 *   scale          softmax scale applied to q.k (e.g. 1/sqrt(head_size)); positive and
 *                  finite, else PA_ERR_INVALID_ARG (the same for every attention call).
 *                  FP8 scales (*k_scale, *v_scale) must be positive as well.
 *   partition_size 0 for the default, else a positive multiple of block_size
 *                  (lets a caller force or tune split-K; the tests force it)
 *   workspace      device scratch of >= pa_decode_workspace_size(...) bytes,
 *                  256-byte aligned; contents need no initialisation
 * A sequence whose seq_len is out of range gets an all-zero output row and sets
 * PA_ERRFLAG_SEQ_LEN.
 */
pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    int32_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                    int32_t block_size, float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                    const float* k_scale, const float* v_scale, int32_t partition_size,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_windowed -- pa_decode with sliding-window attention.
 * [AGENTIC] "為什麼需要「分頁」記憶體管理": sliding-window attention only looks at
 * the most recent fixed range, and blocks that leave it are reclaimed at once
 * into the shared pool.  The query of sequence i (at position seq_lens[i] - 1)
 * attends keys seq_lens[i] - window .. seq_lens[i] - 1 (all of them when the
 * sequence is shorter).  Entries of blocks that lie wholly before the window may
 * hold anything (released blocks): they are never read and never checked.
 * window == 0 is pa_decode; window < 0 is PA_ERR_INVALID_ARG.  The workspace size
 * is pa_decode_workspace_size(...) as for pa_decode; other arguments as pa_decode.
 */
pa_status pa_decode_windowed(void* out, const void* q, const void* k_cache, const void* v_cache,
                             int32_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                             int32_t block_size, float scale, int32_t window, pa_dtype q_dtype,
                             pa_dtype kv_dtype, const float* k_scale, const float* v_scale,
                             int32_t partition_size, void* workspace, size_t workspace_bytes,
                             pa_stream_t stream);

/*
 * Bytes of workspace pa_decode_shared_prefix needs (>= 256) for num_groups groups;
 * partition_size as for pa_decode_workspace_size (0: the shared prefixes get their
 * own default partition size, sized by groups x KV heads).
 */
size_t pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_groups, int32_t num_q_heads,
                                              int32_t num_kv_heads, int32_t head_size, int32_t max_seq_len,
                                              int32_t block_size, int32_t partition_size);

/*
 * pa_decode_shared_prefix -- pa_decode for batches whose sequences share prefix
 * blocks.  [AGENTIC] "統一分頁 + 共用池": sequences that share a prefix (forked
 * subagents, parallel samples) point at the same physical blocks through reference
 * counts.  Same result as pa_decode; each shared (block, KV head) tile is read once
 * per group and applied to every member's query heads, then each member's
 * remaining (private) tokens are attended as in pa_decode and the two partial
 * states are merged.
 *
 *   group_start        device int32 [num_groups + 1], non-decreasing, [0] = 0,
 *                      [num_groups] = num_seqs: group g is the run of consecutive
 *                      sequences group_start[g] .. group_start[g+1]-1
 *   group_shared_blocks device int32 [num_groups]: the first that-many block-table
 *                      entries are identical for every member of group g (clamped
 *                      to the full blocks of the group's shortest member)
 *   num_groups         number of groups (0: plain pa_decode)
 *   max_group_size     host bound on the members of any group, 1..8; groups larger
 *                      than the bound share nothing (still correct)
 *   the rest as pa_decode; workspace >= pa_decode_shared_prefix_workspace_size(...).
 * The declaration is a hint, checked block by block.  [AGENTIC] "統一分頁 + 共用池":
 * shared blocks are copied on write, so a hint can be stale (a member already
 * holds its own copy of a block) or wrong.  A member whose entry for a declared
 * block names another physical block than the group's first sequence reads its own
 * block (loaded separately, for that member alone), so the output is always that of
 * pa_decode; the call sets the diagnostic PA_ERRFLAG_SHARED_MISMATCH.  Entries
 * outside [0, num_blocks) are skipped and set PA_ERRFLAG_BLOCK_TABLE, as in
 * pa_decode.  Without a tensor-core path for the dtypes/shape (or with no groups)
 * this is exactly pa_decode (with a workspace of the size above).
 * The shared-prefix and private-remainder kernels run at once: the call forks a
 * second stream of its own (created on the device's first call, with two events;
 * make that first call before any CUDA stream capture) and joins it back into
 * `stream` before the merge.  Calls from several host threads are serialised
 * around that fork / join.
 */
pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  int32_t num_blocks, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                  int32_t block_size, float scale, pa_dtype q_dtype, pa_dtype kv_dtype,
                                  const float* k_scale, const float* v_scale, const int32_t* group_start,
                                  const int32_t* group_shared_blocks, int32_t num_groups,
                                  int32_t max_group_size, int32_t partition_size, void* workspace,
                                  size_t workspace_bytes, pa_stream_t stream);

/*
 * Size of the fixed device array pa_decode_static_workspace uses as scratch:
 * 32 MiB, held on every GPU that loads this library until the process exits.
 */
#define PA_STATIC_WORKSPACE_BYTES (32u << 20)

/*
 * pa_decode_static_workspace -- pa_decode without a caller-provided workspace.
 * The serving pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory where attention runs: runtimes whose memory
 * planner only provides the tensors it planned (inputs, outputs, KV cache) and no
 * operator scratch, and plug-ins that must not call cudaMalloc or a caching
 * allocator on the serving path (it can synchronise the device, or fail when the
 * pool is exhausted).  The caller passes inputs and outputs only; the split-K
 * partial states go to a file-scope device array of PA_STATIC_WORKSPACE_BYTES.
 *
 *   Arguments as pa_decode.  partition_size 0 picks the default partitioning,
 *   coarsened (doubled) until the partial states fit the array; an explicit
 *   partition_size is used as given.  If the partial states do not fit (many
 *   sequences x heads), returns PA_ERR_WORKSPACE and launches nothing.
 *   Allocates nothing: no cudaMalloc / cudaFree and no allocating library call.
 *   The first call on a device looks up the array's device address (with that
 *   device current); make that first call before any CUDA stream capture.
 *   Every call on a device shares the one array and leaves its contents behind.
 *   Nothing in it needs to start at zero (each call writes every partial it later
 *   reads), but calls that overlap on the GPU -- on different streams, or from
 *   different host threads -- race on it: serialise them.
 */
pa_status pa_decode_static_workspace(void* out, const void* q, const void* k_cache, const void* v_cache,
                                     int32_t num_blocks, const int32_t* block_tables,
                                     int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                                     int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_size, int32_t block_size, float scale, pa_dtype q_dtype,
                                     pa_dtype kv_dtype, const float* k_scale, const float* v_scale,
                                     int32_t partition_size, pa_stream_t stream);

/*
 * Bytes of workspace pa_varlen_attn needs (>= 256).  Same partition_size rule
 * as pa_decode_workspace_size.  The workspace holds the partial states of every
 * row (single-token rows by the decode partition size, multi-token rows by
 * partitions of >= 16384 tokens) and the plan of the prefill tiles, whose length
 * follows total_q_tokens and the query heads per KV head.
 */
size_t pa_varlen_workspace_size(int32_t num_seqs, int32_t total_q_tokens, int32_t max_query_len,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                int32_t max_seq_len, int32_t block_size, int32_t partition_size);

/*
 * pa_varlen_attn -- attention of a flattened variable-length batch.
 * [ARCH] Part 1: all sequences are concatenated into one long sequence with no
 * padding, and V1 mixes decode requests and chunked-prefill requests in one
 * step; [LINEAGE] "静态 batching" / "Chunked prefill": each step holds
 * sum_i q_i <= K tokens, q_i = 1 for a decode, a chunk's tokens for a prefill.
 *
 *   out            [total_q_tokens][num_q_heads][head_size], q_dtype (written)
 *   q              [total_q_tokens][num_q_heads][head_size], q_dtype
 *   query_start_loc int32 [num_seqs + 1], non-decreasing, [0] = 0,
 *                  [num_seqs] = total_q_tokens; request r owns query rows
 *                  query_start_loc[r] .. query_start_loc[r+1]-1
 *   seq_lens       int32 [num_seqs], context length including the new tokens;
 *                  q_len_r <= seq_lens[r] is required
 *   max_query_len, max_seq_len  host-side upper bounds (size the launch)
 *   causal         1: query at position p attends keys 0..p; 0: all seq_len keys
 *   partition_size 0: defaults (single-token rows as pa_decode, rows of
 *                  multi-token requests in partitions of >= 16384 tokens); > 0:
 *                  that many tokens for every row
 *   the rest as pa_decode.  A request with q_len == 0 is skipped.
 * pa_decode equals pa_varlen_attn with q_len = 1 for every request.
 * The single-token rows and the multi-token rows' tiles run concurrently: the
 * call forks a library-owned side stream from `stream` with events and joins it
 * back before its last kernel, so the call stays ordered on `stream` (and can be
 * captured into a CUDA graph).  The tiles are claimed through a counter in the
 * workspace, which the call's own plan kernel resets.
 */
pa_status pa_varlen_attn(void* out, const void* q, const void* k_cache, const void* v_cache,
                         int32_t num_blocks, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* query_start_loc,
                         const int32_t* seq_lens, int32_t num_seqs, int32_t total_q_tokens,
                         int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                         float scale, int32_t causal, pa_dtype q_dtype, pa_dtype kv_dtype,
                         const float* k_scale, const float* v_scale, int32_t partition_size,
                         void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_varlen_attn_windowed -- pa_varlen_attn with sliding-window attention
 * (causal only; window > 0 with causal == 0 is PA_ERR_UNSUPPORTED).  Query j of a
 * request (position p = seq_len - q_len + j) attends keys max(0, p - window + 1)
 * .. p.  Entries of blocks wholly before the window of the request's first query
 * may hold anything (released blocks): they are never read.  window == 0 is
 * pa_varlen_attn; the workspace is sized by pa_varlen_workspace_size as for it.
 */
pa_status pa_varlen_attn_windowed(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  int32_t num_blocks, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* query_start_loc,
                                  const int32_t* seq_lens, int32_t num_seqs, int32_t total_q_tokens,
                                  int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                  float scale, int32_t window, int32_t causal, pa_dtype q_dtype,
                                  pa_dtype kv_dtype, const float* k_scale, const float* v_scale,
                                  int32_t partition_size, void* workspace, size_t workspace_bytes,
                                  pa_stream_t stream);

/*
 * Read the device error word of the current device (host pointer `flags`),
 * after synchronising `stream`.  clear != 0 resets it to zero.  Returns
 * PA_ERR_BOUNDS if any error bit other than TIMEOUT is set, PA_ERR_TIMEOUT if
 * TIMEOUT is the only error bit set, PA_OK otherwise (no bit, or only the
 * diagnostic PA_ERRFLAG_SHARED_MISMATCH; `flags` still reports it).
 */
pa_status pa_get_error_flags(uint32_t* flags, int32_t clear, pa_stream_t stream);

/*
 * Kernel-level tracing.  While enabled, every kernel the library launches is
 * bracketed by CUDA events recorded on its launch stream.  pa_trace_read()
 * synchronises those events and, for kernel kind `kind` (0 = reshape_and_cache,
 * 1 = attention main kernel, 2 = partial merge, 3 = varlen plan,
 * 4 = prefill tiles (two launches per pa_varlen_attn call when single-token rows
 * run beside them), 5 = shared-prefix tiles, 6 = the span of the shared-prefix
 * and private-remainder kernels of pa_decode_shared_prefix, 7 = copy_blocks,
 * 8 = the span of the single-token-row and multi-token-row kernels of
 * pa_varlen_attn, which run concurrently on two streams),
 * returns the launch count and the summed device milliseconds since the last
 * reset (reset != 0 clears every kind).
 * Tracing is off by default and costs nothing when off.  Not thread-safe.
 */
pa_status pa_trace_enable(int32_t on);
pa_status pa_trace_read(int32_t kind, int64_t* launches, double* total_ms, int32_t reset);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
