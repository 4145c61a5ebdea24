/*
 * pkv.h -- C ABI of the paged-KV hot path for GB300 (sm_103a).
 *
 * Four device computations and their host-side checks:
 *   pkv_compute_slot_mapping   new-token positions -> flat cache slots
 *   pkv_store_kvcache          scatter fresh K/V rows into the paged cache
 *   pkv_paged_attention_decode one query per sequence, GQA, split-K + LSE combine
 *   pkv_unpack_block_paged     CSR block-paged snapshot -> contiguous [T, H, d]
 *
 * Sources (page title -- section):
 *   "Paged KV Cache - AI infra interview lesson": Walk the Shapes First;
 *     Step 1: slot_mapping and store_kvcache; Step 2: paged_attention_decode.
 *   "Block-Paged KV Cache" (Hurray format documentation): The three buffers;
 *     Element lookup through the block table; Validating the storage invariants.
 *
 * Conventions shared by every entry point
 *   - Plain pointers and sizes only.  "device" pointers must be CUDA device
 *     (or managed) memory of the current device; "host" pointers are CPU memory.
 *   - The caller owns every buffer.  The library never allocates, frees or
 *     synchronises; work is enqueued on `stream` (a cudaStream_t passed as
 *     void*, NULL = the legacy default stream) and the call returns at once.
 *   - Shapes and arguments are checked synchronously, before anything is
 *     enqueued; a failed check returns an error status and enqueues nothing.
 *     pkv_last_error_string() then describes the failure (thread-local).
 *   - Errors that depend on device data (a slot or block id out of range, a
 *     context longer than declared) cannot be seen on the host.  The kernels
 *     skip the offending element, apply the documented fallback and OR a bit
 *     (PKV_ERRBIT_*) into `err_flag`, an optional device int32 that the
 *     caller zeroes and reads back; pass NULL to ignore such errors.
 *   - Floating-point tensors are contiguous, row-major, in one storage type
 *     (pkv_dtype) shared by q / key / value / caches / out.  All offsets are
 *     computed in 64-bit.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* a size, pointer or shape is invalid */
    PKV_ERR_UNSUPPORTED = 2,   /* valid, but not a combination this build handles */
    PKV_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (launch, tensor map) */
    PKV_ERR_OUT_OF_RANGE = 4,  /* host-side index check failed (validators) */
    PKV_ERR_WORKSPACE = 5      /* workspace missing or smaller than the size query says */
} pkv_status;

typedef enum pkv_dtype { PKV_F32 = 0, PKV_F16 = 1, PKV_BF16 = 2 } pkv_dtype;

/* Width of the CSR index buffers ("BlockTableIndexType" U32 / U64). */
typedef enum pkv_index_type { PKV_U32 = 0, PKV_U64 = 1 } pkv_index_type;

/* Quantization scheme tags ("Block-Paged KV Cache", Quantization compatibility). */
enum { PKV_QUANT_NONE = 0x00, PKV_QUANT_PER_TENSOR = 0x01, PKV_QUANT_PER_CHANNEL = 0x02, PKV_QUANT_PER_BLOCK = 0x03 };

/* Bits OR-ed into *err_flag by the kernels. */
#define PKV_ERRBIT_SLOT_RANGE   0x01 /* store: slot not -1 and outside [0, num_slots) */
#define PKV_ERRBIT_BLOCK_RANGE  0x02 /* a used block-table entry outside [0, num_blocks) */
#define PKV_ERRBIT_CONTEXT      0x04 /* context length < 0, > max_context_len or > table */
#define PKV_ERRBIT_CSR_PAGE     0x08 /* unpack: a token's page lies outside its seq_ptr slice */
#define PKV_ERRBIT_CSR_PHYS     0x10 /* unpack: physical page id >= num_pages */
#define PKV_ERRBIT_SPAN         0x20 /* slot mapping: cu_new disagrees with [start, end) */
#define PKV_ERRBIT_TIMEOUT      0x40 /* an internal pipeline wait gave up (never expected) */

/* Text of the last error returned on this thread ("" after success). */
PKV_API const char *pkv_last_error_string(void);

/* Library version string. */
PKV_API const char *pkv_version(void);

/*
 * pkv_selftest_wait_timeout -- failure-detection self-test of the bounded
 * pipeline wait.  Launches one warp on `stream` that waits on an mbarrier
 * nothing completes, with the deadline mechanism every attention-kernel stage
 * uses (a wall-clock limit read from %globaltimer).  When the limit passes, the
 * kernel ORs PKV_ERRBIT_TIMEOUT into *err_flag and returns; nothing faults or
 * hangs, and the context stays usable.
 *   err_flag    device int32, 4-byte aligned (required)
 *   timeout_us  the wait's limit, in (0, 1000000] microseconds
 * Returns PKV_ERR_INVALID_ARG for a NULL or misaligned flag or a limit out of
 * range, PKV_ERR_CUDA if the launch fails.
 */
PKV_API pkv_status pkv_selftest_wait_timeout(int32_t *err_flag, uint32_t timeout_us, void *stream);

/*
 * pkv_compute_slot_mapping -- "Walk the Shapes First" and "Step 1": the slot
 * of position p of sequence b is block_tables[b][p / block_size] * block_size
 * + p % block_size; the mapping covers only the positions written this step.
 *
 *   block_tables    device int32 [num_seqs, max_blocks_per_seq], row-major;
 *                   entries past a sequence's last block may be -1.
 *   starts, ends    device int32 [num_seqs]: positions [starts[b], ends[b]).
 *   cu_new          device int32 [num_seqs + 1]: sequence b's slots go to
 *                   slot_mapping[cu_new[b] .. cu_new[b+1]); cu_new[0] == 0.
 *   num_blocks      pool size in blocks; block_size * num_blocks < 2^31.
 *   slot_mapping    device int32 [num_new_tokens] (output).
 * Device errors: a position whose block is missing (-1 / beyond the row) or
 * >= num_blocks gets slot -1 and PKV_ERRBIT_BLOCK_RANGE; a sequence whose
 * cu_new span differs from ends-starts, or exceeds num_new_tokens, writes
 * only what fits and sets PKV_ERRBIT_SPAN.
 */
PKV_API pkv_status pkv_compute_slot_mapping(const int32_t *block_tables, int32_t max_blocks_per_seq,
                                    const int32_t *starts, const int32_t *ends,
                                    const int32_t *cu_new, int32_t num_seqs,
                                    int32_t block_size, int32_t num_blocks,
                                    int32_t *slot_mapping, int64_t num_new_tokens,
                                    int32_t *err_flag, void *stream);

/*
 * pkv_store_kvcache -- "Step 1: slot_mapping and store_kvcache": with the caches
 * viewed as [num_slots, num_kv_heads * head_dim] rows, row slot_mapping[i]
 * receives key[i] (and value[i]); slot -1 is padding and is skipped.
 *
 *   key, value        device [num_tokens, num_kv_heads, head_dim]
 *   k_cache, v_cache  device [num_blocks, block_size, num_kv_heads, head_dim],
 *                     num_slots = num_blocks * block_size rows (modified in place)
 *   slot_mapping      device int32 [num_tokens]; non-(-1) slots must be
 *                     distinct (duplicates race: which row wins is undefined).
 * Device errors: a slot that is neither -1 nor in [0, num_slots) is skipped
 * and sets PKV_ERRBIT_SLOT_RANGE.
 */
PKV_API pkv_status pkv_store_kvcache(const void *key, const void *value, void *k_cache, void *v_cache,
                             const int32_t *slot_mapping, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim, int64_t num_slots,
                             pkv_dtype dtype, int32_t *err_flag, void *stream);

/*
 * pkv_paged_attention_decode -- "Step 2: paged_attention_decode": for every
 * sequence b (one query token) and query head h, with n = context_lens[b],
 *   out[b,h] = softmax_t( scale * q[b,h] . K_t ) . V_t,   t = 0 .. n-1,
 * where token t lives in cache row block_tables[b][t / block_size] *
 * block_size + t % block_size, KV head h / (num_q_heads / num_kv_heads).
 * Only the first ceil(n / block_size) table entries are read (later ones may
 * be -1); the unused tail of the last block is never read.  The context is
 * split into partitions that are reduced independently and merged with a
 * log-sum-exp combine (flash-decoding), so long contexts fill the GPU.
 *
 *   out              device [num_seqs, num_q_heads, head_dim] (output, dtype)
 *   q                device [num_seqs, num_q_heads, head_dim]
 *   k_cache, v_cache device [num_blocks, block_size, num_kv_heads, head_dim]
 *   block_tables     device int32 [num_seqs, max_blocks_per_seq]
 *   context_lens     device int32 [num_seqs], each in [0, max_context_len]
 *   max_context_len  host bound on context_lens; sizes the grid and workspace
 *   workspace        device scratch of at least
 *                    pkv_paged_attention_decode_workspace_size(...) bytes,
 *                    256-byte aligned; contents need not be initialised.
 * num_q_heads must be a multiple of num_kv_heads.  Accumulation is fp32; the
 * result is rounded once to dtype.  n == 0 gives a zero row.
 * Device errors: a context length < 0, > max_context_len or needing more than
 * max_blocks_per_seq blocks gives a zero row and PKV_ERRBIT_CONTEXT; a used
 * block id outside [0, num_blocks) drops that block's tokens from the softmax
 * and sets PKV_ERRBIT_BLOCK_RANGE.
 */
PKV_API pkv_status pkv_paged_attention_decode(void *out, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens,
                                      int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int32_t num_blocks,
                                      int32_t max_context_len, float scale, pkv_dtype dtype,
                                      void *workspace, size_t workspace_bytes,
                                      int32_t *err_flag, void *stream);

/*
 * pkv_paged_attention_decode_append -- one decode step of the pages'
 * "Walk the Shapes First" trace in one call: every sequence's new token sits
 * at position context_lens[b] - 1 (context_lens counts it), its K/V rows are
 * written to the paged caches at that position's slot
 * (block_tables[b][p / block_size] * block_size + p % block_size, as in
 * "Step 1: slot_mapping and store_kvcache"), and then the attention of
 * pkv_paged_attention_decode runs over the whole context, the new token
 * included ("Step 2: paged_attention_decode").  The result equals
 * pkv_compute_slot_mapping over [ctx - 1, ctx) + pkv_store_kvcache +
 * pkv_paged_attention_decode with the same arguments.
 *
 *   key, value       device [num_seqs, num_kv_heads, head_dim]: the new token's
 *                    K/V rows (dtype), read only
 *   k_cache, v_cache modified in place (one row per sequence)
 *   all other arguments, the workspace and the output as in
 *                    pkv_paged_attention_decode.
 * On the tensor-core path with the work-balanced schedule (at most 512
 * sequences) and 8-byte aligned key/value, the rows are written by the
 * attention kernel itself right before it reads that block; otherwise a
 * separate append kernel runs first on the same stream.
 * Device errors: a sequence whose context length is invalid (see
 * pkv_paged_attention_decode) is neither appended nor attended
 * (PKV_ERRBIT_CONTEXT, zero row); a block id outside [0, num_blocks) at
 * position ctx - 1 skips the append and sets PKV_ERRBIT_BLOCK_RANGE.
 */
PKV_API pkv_status pkv_paged_attention_decode_append(void *out, const void *q, const void *key,
                                             const void *value, void *k_cache, void *v_cache,
                                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                                             const int32_t *context_lens, int32_t num_seqs,
                                             int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                             int32_t max_context_len, float scale, pkv_dtype dtype,
                                             void *workspace, size_t workspace_bytes,
                                             int32_t *err_flag, void *stream);

/* Workspace bytes pkv_paged_attention_decode needs for these sizes (0 is a
 * valid answer).  Pure host arithmetic; never fails (returns 0 on bad sizes,
 * which the decode call then rejects). */
PKV_API size_t pkv_paged_attention_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                                 int32_t num_kv_heads, int32_t head_dim,
                                                 int32_t block_size, int32_t max_context_len,
                                                 pkv_dtype dtype);

/* How pkv_paged_attention_decode will split the context for these sizes:
 * tokens per partition, number of partitions covering max_context_len
 * (1 = no combine pass), and whether the TMA/tensor-core path is used
 * (fp16/bf16, head_dim 128, Hq/Hkv <= 8, block_size a multiple of 16 and
 * 16-byte aligned pools; 0 = the CUDA-core path).  Any output may be NULL. */
PKV_API pkv_status pkv_paged_attention_decode_plan(int32_t num_seqs, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_dim,
                                           int32_t block_size, int32_t max_context_len,
                                           pkv_dtype dtype, int32_t *partition_tokens,
                                           int32_t *num_partitions, int32_t *fast_path);

/*
 * pkv_paged_attention_decode_static_ws -- the same computation and arguments
 * as pkv_paged_attention_decode, minus the workspace: this variant allocates
 * nothing and needs nothing allocated for it.  (No counterpart on the pages;
 * it exists for callers, not for the method.)
 *
 * Who needs it: code that cannot allocate device memory where it runs
 * attention.  One example is a plugin inside an inference engine, whose enqueue
 * hook may only use memory the engine handed it.  Another is a service that
 * reserves a fixed memory budget at start-up and must not call cudaMalloc
 * afterwards.  Such callers still pass q, the caches, the tables and out; the
 * split-K scratch comes from a fixed region built into the library instead.
 *
 * The region is PKV_STATIC_WORKSPACE_BYTES (16 MiB) of device memory that
 * every GPU loading the library holds until the process exits.  Sizes whose
 * pkv_paged_attention_decode_workspace_size exceeds it are rejected with
 * PKV_ERR_WORKSPACE before anything is enqueued; use the workspace variant
 * for those.  Argument errors (bad sizes, NULL pointers) are reported as
 * PKV_ERR_INVALID_ARG first, exactly as by pkv_paged_attention_decode.  The
 * size bound assumes every sequence holds max_context_len tokens: 8 x 32768
 * tokens at Hq 32 / Hkv 8 needs about 15.9 MB and fits, as do 64 x 4096 at
 * Hq = Hkv = 32 (14.6 MB) and 8 x 8192 (7.4 MB); 128 sequences of up to 8192
 * tokens at Hq 16 / Hkv 8 need about 27 MB and do not.
 *
 * Every call looks up the region's device address (cudaGetSymbolAddress)
 * with the calling thread's current device; the lookup allocates nothing.
 * The first call on a device may load the library's device code, so make it
 * before any stream capture.
 *
 * All calls share the one region, and it keeps whatever the last call left
 * there.  Nothing in it has to start at zero: every call writes each scratch
 * value before reading it.  Calls whose GPU work overlaps (for example on two
 * streams at once) race on the region and give wrong results; serialise
 * them.  The function calls no cudaMalloc/cudaFree and no allocating library
 * routine.
 */
#define PKV_STATIC_WORKSPACE_BYTES (16u * 1024u * 1024u)
PKV_API pkv_status pkv_paged_attention_decode_static_ws(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int32_t num_blocks, int32_t max_context_len, float scale,
    pkv_dtype dtype, int32_t *err_flag, void *stream);

/*
 * pkv_unpack_block_paged -- "The three buffers" and "Element lookup through
 * the block table": resolve one {kv_role, layer} snapshot into its logical
 * tensor out[total_tokens, num_heads, head_dim], element by element
 *   flat = ((block_table[seq_ptr[s] + t / page_size] * page_size
 *            + t % page_size) * num_heads + h) * head_dim + dim,
 * for token t of sequence s written to row token_ptr[s] + t.  Pages that
 * several sequences name (prefix sharing) are read, never copied in the pool.
 * Call once per role (keys, values) over the same index buffers.
 *
 *   page_pool    device [num_pages, page_size, num_heads, head_dim] (paged axis 0)
 *   block_table  device u32/u64 [nnz]; seq_ptr device u32/u64 [num_seqs + 1]
 *   token_ptr    device int64 [num_seqs + 1]: sequence s owns output rows
 *                token_ptr[s] .. token_ptr[s+1]-1 (the CSR buffers do not carry
 *                per-sequence token counts); token_ptr[num_seqs] == total_tokens.
 *   out          device [total_tokens, num_heads, head_dim] (output)
 * Run pkv_validate_index_buffers / pkv_validate_token_ptr on the host copies
 * first.  Device errors: rows whose page lies outside the sequence's slice
 * are zero-filled (PKV_ERRBIT_CSR_PAGE); rows on a page id >= num_pages are
 * zero-filled (PKV_ERRBIT_CSR_PHYS).
 */
PKV_API pkv_status pkv_unpack_block_paged(void *out, const void *page_pool, const void *block_table,
                                  const void *seq_ptr, pkv_index_type index_type,
                                  const int64_t *token_ptr, int32_t num_seqs, int64_t nnz,
                                  int32_t page_size, int64_t num_pages, int32_t num_heads,
                                  int32_t head_dim, int64_t total_tokens, pkv_dtype dtype,
                                  int32_t *err_flag, void *stream);

/*
 * pkv_validate_index_buffers -- "Validating the storage invariants" (host
 * pointers): seq_ptr[0] == 0; seq_ptr non-decreasing; seq_ptr[num_seqs] ==
 * nnz; every block_table entry < num_pages.  The empty batch (num_seqs == 0,
 * seq_ptr == {0}) is valid.  Returns PKV_OK or PKV_ERR_OUT_OF_RANGE (with the
 * broken invariant in pkv_last_error_string()), PKV_ERR_INVALID_ARG for NULL
 * pointers or negative sizes.
 */
PKV_API pkv_status pkv_validate_index_buffers(const void *seq_ptr, const void *block_table,
                                      pkv_index_type index_type, int64_t num_seqs, int64_t nnz,
                                      int64_t num_pages);

/*
 * pkv_validate_quantization_compatibility -- "Block-Paged KV Cache",
 * Quantization compatibility: whether a quantization scheme's scales fit the
 * block-paged layout (host only, no pointers).
 *   scheme_tag  PKV_QUANT_NONE (0x00), PKV_QUANT_PER_TENSOR (0x01),
 *               PKV_QUANT_PER_CHANNEL (0x02), PKV_QUANT_PER_BLOCK (0x03,
 *               per-block-affine)
 *   axis        the axis the scales run along (0 is the paged axis)
 *   block_size  elements per scale block (per-block-affine only)
 *   page_size   tokens per page
 * Per-block-affine is valid only along axis 0 with block_size == page_size,
 * so a shared page carries its own scales; per-channel scales along the paged
 * axis are refused; no-scale and per-tensor schemes always fit (the page
 * states only the first two rules; the rest is this library's reading).
 * Returns PKV_OK, or PKV_ERR_INVALID_ARG naming the broken rule (also for an
 * unknown tag or page_size <= 0).  The library's fp8 and int8 caches keep one
 * scale per (block, KV head): per-block-affine with block_size == page_size.
 */
PKV_API pkv_status pkv_validate_quantization_compatibility(int32_t scheme_tag, int32_t axis, int32_t block_size,
                                                   int32_t page_size);

/*
 * pkv_validate_token_ptr -- host check that token_ptr (host int64 [num_seqs+1])
 * fits the snapshot: token_ptr[0] == 0, non-decreasing, token_ptr[num_seqs] ==
 * total_tokens, and every sequence's tokens fit its pages:
 * ceil(len_s / page_size) <= seq_ptr[s+1] - seq_ptr[s] (seq_ptr host).
 */
PKV_API pkv_status pkv_validate_token_ptr(const int64_t *token_ptr, const void *seq_ptr,
                                  pkv_index_type index_type, int64_t num_seqs,
                                  int32_t page_size, int64_t total_tokens);

/*
 * pkv_validate_block_paged_shape -- "Building a descriptor": a block-paged
 * snapshot is rank-3 only, [total_tokens, num_heads, head_dim] (host array
 * `shape` of `rank` entries).  PKV_OK when rank == 3, every extent is >= 0
 * and the last two equal num_heads and head_dim; PKV_ERR_INVALID_ARG otherwise.
 */
PKV_API pkv_status pkv_validate_block_paged_shape(const int64_t *shape, int32_t rank,
                                                  int32_t num_heads, int32_t head_dim);

/*
 * pkv_block_paged_element_offset -- "Element lookup through the block table"
 * on host pointers: writes the flat page_pool offset of (seq, token, head, dim)
 * to *flat_out.  PKV_ERR_OUT_OF_RANGE when seq, head or dim is out of range,
 * the token's page lies outside the sequence's slice, or the physical page is
 * >= num_pages.
 */
PKV_API pkv_status pkv_block_paged_element_offset(int64_t seq, int64_t token, int64_t head, int64_t dim,
                                          int32_t page_size, int64_t num_pages,
                                          int32_t num_heads, int32_t head_dim,
                                          const void *block_table, const void *seq_ptr,
                                          pkv_index_type index_type, int64_t num_seqs,
                                          int64_t *flat_out);

/*
 * pkv_paged_attention_prefill -- causal varlen / chunked prefill over the paged
 * cache ("Paged KV Cache - AI infra interview lesson": Step 3, varlen
 * attention and cu_seqlens, is named there without content; the reading here
 * is the plain one its Steps 1 and 2 support).  Sequence b's new tokens sit
 * at positions [starts[b], starts[b] + n_b), n_b = cu_q[b+1] - cu_q[b], and
 * their K/V are already stored in the caches (pkv_compute_slot_mapping over
 * that range + pkv_store_kvcache), as are those of positions [0, starts[b])
 * (a cached prefix or earlier chunks).  For query i of sequence b, at position
 * p = starts[b] + i, and query head h:
 *   out[cu_q[b] + i, h] = softmax_{t <= p}(scale * q[cu_q[b] + i, h] . K_t) . V_t
 * with K_t / V_t read through the block table and KV head h / (Hq / Hkv).
 *
 *   out, q         device [cu_q[num_seqs], num_q_heads, head_dim] (dtype)
 *   starts         device int32 [num_seqs], first new position per sequence
 *   cu_q           device int32 [num_seqs + 1], offsets of each sequence's queries
 *   max_q_len      host bound on n_b (sizes the grid)
 *   caches, block_tables, num_blocks as in pkv_paged_attention_decode.
 * fp32 accumulation (tcgen05 tensor cores, accumulators in tensor memory; P
 * enters the PV product rounded to dtype and the row sum adds the same rounded
 * values), one rounding of the output to dtype.  fp16 or bf16, head_dim 128,
 * num_q_heads / num_kv_heads in {1, 2, 4, 8}, block_size a multiple of 16,
 * 16-byte aligned pools, q and out; other shapes or alignments return
 * PKV_ERR_UNSUPPORTED.  No workspace.  One CTA per two tiles of 128 query
 * rows of a KV head, using all 512 tensor-memory columns of its SM.
 * Device errors: starts[b] < 0 or a span needing more than max_blocks_per_seq
 * blocks gives zero rows and PKV_ERRBIT_CONTEXT; n_b < 0 or n_b > max_q_len
 * sets PKV_ERRBIT_CONTEXT (rows past max_q_len are not written); a used block
 * id outside [0, num_blocks) drops that block's tokens and sets
 * PKV_ERRBIT_BLOCK_RANGE.
 */
PKV_API pkv_status pkv_paged_attention_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
                                               const int32_t *block_tables, int32_t max_blocks_per_seq,
                                               const int32_t *starts, const int32_t *cu_q, int32_t num_seqs,
                                               int32_t max_q_len, int32_t num_q_heads, int32_t num_kv_heads,
                                               int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                               float scale, pkv_dtype dtype, int32_t *err_flag, void *stream);

/*
 * fp8 (E4M3) paged caches -- "Block-Paged KV Cache", Quantization
 * compatibility: per-block-affine scales with block_size == page_size stay per
 * page slot, so a shared page carries its own scales.  The pages give that
 * placement rule only.  This library's reading: the caches hold OCP E4M3
 * codes (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, largest finite 448), [num_blocks, block_size, num_kv_heads,
 * head_dim] bytes, and every (physical block, KV head) has one float32 scale
 * for K and one for V, k_scale / v_scale [num_blocks, num_kv_heads].  A
 * stored value is scale * decode(code).  Encoding divides by the scale in
 * binary32 and rounds to the nearest even code, saturating at +-448; a zero
 * scale stores +0.
 *
 * pkv_quantize_kvcache_fp8: a 16-bit or fp32 cache `src` of `dtype` -> codes
 *   and scales, per (block, head) s = max|x| / 448 (NaN ignored).  Used to
 *   fill a cache (e.g. after a prefill); head_dim must be even.
 * pkv_store_kvcache_fp8: "Step 1" into an fp8 cache: row slot_mapping[i]
 *   receives encode(key[i] / s) with the scale of the row's block and head
 *   (a value beyond 448 * s saturates).  Slot -1 is skipped; other slots
 *   outside [0, num_slots) set PKV_ERRBIT_SLOT_RANGE and are skipped.
 * pkv_paged_attention_decode_fp8: "Step 2" over fp8 caches, q and out in
 *   fp16 or bf16, with the arguments, workspace
 *   (pkv_paged_attention_decode_workspace_size with the q dtype) and device
 *   errors of pkv_paged_attention_decode.  Codes are widened exactly to f16
 *   and the products run on f16 tensor cores (q is rounded to f16 once;
 *   values beyond 65504 overflow).  Only the tensor-core, work-balanced
 *   shapes run: head_dim 128, num_q_heads / num_kv_heads <= 8, block_size a
 *   multiple of 16, 16-byte aligned q and code pools; others return
 *   PKV_ERR_UNSUPPORTED.  Batches of more than 512 sequences run as
 *   consecutive launches over groups of at most 512 (one workspace, reused in
 *   stream order).
 * pkv_paged_attention_decode_append_fp8: the fused decode step over fp8
 *   caches ("Step 1" then "Step 2" for one new token per sequence): key[b]
 *   and value[b] ([num_seqs, num_kv_heads, head_dim], the q dtype, 8-byte
 *   aligned) are encoded as by pkv_store_kvcache_fp8, under the scales
 *   already in k_scale / v_scale, into the cache row of position
 *   context_lens[b] - 1, and the attention of pkv_paged_attention_decode_fp8
 *   runs over the whole context, the new token included.  The scales are not
 *   changed.  Arguments, workspace, limits and errors as
 *   pkv_paged_attention_decode_fp8; a block id out of range at position
 *   ctx - 1 skips the append and sets PKV_ERRBIT_BLOCK_RANGE.
 */
PKV_API pkv_status pkv_quantize_kvcache_fp8(const void *src, void *codes, float *scales, int32_t num_blocks,
                                            int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                            pkv_dtype dtype, void *stream);
PKV_API pkv_status pkv_store_kvcache_fp8(const void *key, const void *value, void *k_cache, void *v_cache,
                                         const float *k_scale, const float *v_scale, const int32_t *slot_mapping,
                                         int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                         int64_t num_slots, int32_t block_size, pkv_dtype dtype,
                                         int32_t *err_flag, void *stream);
PKV_API pkv_status pkv_paged_attention_decode_fp8(void *out, const void *q, const void *k_cache,
                                                  const void *v_cache, const float *k_scale, const float *v_scale,
                                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                  const int32_t *context_lens, int32_t num_seqs,
                                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                  int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                                                  float scale, pkv_dtype dtype, void *workspace,
                                                  size_t workspace_bytes, int32_t *err_flag, void *stream);
PKV_API pkv_status pkv_paged_attention_decode_append_fp8(void *out, const void *q, const void *key,
                                                         const void *value, void *k_cache, void *v_cache,
                                                         const float *k_scale, const float *v_scale,
                                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                         const int32_t *context_lens, int32_t num_seqs,
                                                         int32_t num_q_heads, int32_t num_kv_heads,
                                                         int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                                         int32_t max_context_len, float scale, pkv_dtype dtype,
                                                         void *workspace, size_t workspace_bytes,
                                                         int32_t *err_flag, void *stream);

/*
 * int8 paged caches -- "Block-Paged KV Cache", Quantization compatibility
 * names int8 caches beside fp8 ones under the same placement rule.  This
 * library's reading (symmetric): the caches hold signed bytes c in
 * [-127, 127], [num_blocks, block_size, num_kv_heads, head_dim], with the
 * k_scale / v_scale layout of the fp8 caches, a stored value being scale * c.
 * The scale of a (block, head) is max|x| / 127 (binary32, NaN ignored).
 * Encoding divides by the scale in binary32, rounds to the nearest integer
 * (ties to even), clamps to +-127 and stores NaN as 0; a zero scale stores 0.
 *
 * pkv_quantize_kvcache_int8, pkv_store_kvcache_int8,
 * pkv_paged_attention_decode_int8 and pkv_paged_attention_decode_append_int8
 * take the arguments, and have the ownership, shape limits, errors and
 * device error bits, of their fp8 counterparts above; only the code format
 * differs.  Codes are widened exactly to f16 for the products.
 */
PKV_API pkv_status pkv_quantize_kvcache_int8(const void *src, void *codes, float *scales, int32_t num_blocks,
                                             int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                             pkv_dtype dtype, void *stream);
PKV_API pkv_status pkv_store_kvcache_int8(const void *key, const void *value, void *k_cache, void *v_cache,
                                          const float *k_scale, const float *v_scale, const int32_t *slot_mapping,
                                          int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                          int64_t num_slots, int32_t block_size, pkv_dtype dtype,
                                          int32_t *err_flag, void *stream);
PKV_API pkv_status pkv_paged_attention_decode_int8(void *out, const void *q, const void *k_cache,
                                                   const void *v_cache, const float *k_scale, const float *v_scale,
                                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                   const int32_t *context_lens, int32_t num_seqs,
                                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                   int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                                                   float scale, pkv_dtype dtype, void *workspace,
                                                   size_t workspace_bytes, int32_t *err_flag, void *stream);
PKV_API pkv_status pkv_paged_attention_decode_append_int8(void *out, const void *q, const void *key,
                                                          const void *value, void *k_cache, void *v_cache,
                                                          const float *k_scale, const float *v_scale,
                                                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                          const int32_t *context_lens, int32_t num_seqs,
                                                          int32_t num_q_heads, int32_t num_kv_heads,
                                                          int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                                          int32_t max_context_len, float scale, pkv_dtype dtype,
                                                          void *workspace, size_t workspace_bytes,
                                                          int32_t *err_flag, void *stream);

/*
 * Host block allocator -- which physical block of the pool each sequence
 * owns ("Paged KV Cache - AI infra interview lesson": Walk the Shapes First;
 * Append slots during decode; Separate allocation, sharing and release).
 * Host memory only, no CUDA call; thread-safe per handle.  It hands out the
 * lowest-numbered free block first, so traces are deterministic, and keeps a
 * reference count per block: the number of block-table entries that point at
 * it.  A block returns to the free pool when its count reaches zero.
 *
 *   pkv_allocator_create       pool of num_blocks blocks of block_size tokens
 *                              (num_blocks * block_size < 2^31)
 *   pkv_allocator_add_sequence new sequence `seq` holding num_tokens tokens:
 *                              ceil(num_tokens / block_size) blocks, taken from
 *                              the pool, or the caller's `blocks` (host int32
 *                              list; each must be free) when not NULL
 *   pkv_allocator_fork         new sequence `child` sharing the first
 *                              num_tokens tokens (whole blocks) of `parent`;
 *                              the shared blocks' counts go up
 *   pkv_allocator_append       grows `seq` by num_tokens tokens, taking a new
 *                              block whenever a position p has p % block_size
 *                              == 0; writes their slots
 *                              (block_table[p / bs] * bs + p % bs) to the host
 *                              int32 `slots` [num_tokens] if not NULL
 *   pkv_allocator_release      drops `seq`; its blocks' counts go down
 *   pkv_allocator_block_table  host int32 row [max_blocks] of `seq` (padded
 *                              with -1), its length and block count
 *   pkv_allocator_stats        free, allocated (count > 0) and referenced
 *                              blocks, live sequences; any output may be NULL
 *   pkv_allocator_check        0 when every accounting invariant holds, else
 *                              the first broken one: 1 free + allocated !=
 *                              pool, 2 a count differs from the table entries
 *                              that point at the block, 3 a block is both free
 *                              and referenced (or neither), 4 a sequence's
 *                              partly filled last block is shared, 5 a table
 *                              does not cover its sequence's length
 *                              ("Chapter 2 -- KV cache, memory hierarchy,
 *                              continuous batching, and PagedAttention",
 *                              Deterministic evals for this layer)
 * Errors: PKV_ERR_INVALID_ARG (unknown or duplicate sequence id, a prefix that
 * is not whole blocks, a block that is not free); PKV_ERR_OUT_OF_RANGE (not
 * enough free blocks, or a row too short).  A failed call changes nothing.
 */
typedef struct pkv_block_allocator pkv_block_allocator;
PKV_API pkv_status pkv_allocator_create(int32_t num_blocks, int32_t block_size, pkv_block_allocator **out);
PKV_API void pkv_allocator_destroy(pkv_block_allocator *a);
PKV_API pkv_status pkv_allocator_add_sequence(pkv_block_allocator *a, int64_t seq, int64_t num_tokens,
                                              const int32_t *blocks);
PKV_API pkv_status pkv_allocator_fork(pkv_block_allocator *a, int64_t parent, int64_t child, int64_t num_tokens);
PKV_API pkv_status pkv_allocator_append(pkv_block_allocator *a, int64_t seq, int64_t num_tokens, int32_t *slots);
PKV_API pkv_status pkv_allocator_release(pkv_block_allocator *a, int64_t seq);
PKV_API pkv_status pkv_allocator_block_table(pkv_block_allocator *a, int64_t seq, int32_t *row,
                                             int32_t max_blocks, int64_t *num_tokens, int32_t *num_used);
PKV_API pkv_status pkv_allocator_stats(pkv_block_allocator *a, int64_t *free_blocks, int64_t *allocated_blocks,
                                       int64_t *referenced_blocks, int64_t *num_seqs);
PKV_API int32_t pkv_allocator_check(pkv_block_allocator *a);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
