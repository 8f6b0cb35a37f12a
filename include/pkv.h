/*
 * pkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache decode-attention library.
 *
 * The operations follow the problem statement of these web pages:
 *   [ENG26]  "The engineering truth of long-context inference 2026: PagedAttention,
 *            Ring Attention and KV-cache offload from 128K to 1M context"
 *            (blog.lonae.com), sections 1.1, 2.1-2.3, 3.1.
 *   [UNLOCK] "Unlocking long context: engineering practice for million-token LLM
 *            inference" (ybb.press), sections 3.1, 3.2, 4.1, 5.1.
 *   [MHPN]   long-context article at mhpn.cn (news 2466452), sections 1.1, 3.1, 3.2.
 *   [SEQPAR] "Sequence-parallel engineering for long-context LLM inference: Ring
 *            Attention and distributed KV cache" (ybb.press), section
 *            "numerically stable incremental softmax".
 *
 * Conventions shared by every call:
 *   - Every device buffer is owned by the caller (for example a torch tensor);
 *     the library never allocates device memory.  `d_` marks a device pointer,
 *     `h_` or no prefix a host pointer.  On a host whose pinned memory the GPU
 *     maps (a Grace host), the decode calls also take q, the new token's k and
 *     v, the lengths, the tables and out in pinned host memory (the kernels read
 *     and write them over the CPU-GPU link); the workspace is device memory,
 *     and every buffer must stay allocated until the launches that use it end.
 *   - Shapes are row-major: q and out [batch, num_q_heads, head_dim];
 *     k and v of new tokens [tokens, num_kv_heads, head_dim]; block tables
 *     int32 [batch, max_blocks_per_seq] (entries past ceil(seq_len/block_size)
 *     are never read).
 *   - The pool has the pages' layout [num_blocks, 2, num_layers, num_kv_heads,
 *     block_size, head_dim] ([ENG26] 2.2): the K (index 0) and V (index 1)
 *     tiles of one (block, layer, kv head) are block_size x head_dim contiguous
 *     elements.
 *   - GQA ([MHPN] 3.2): G = num_q_heads / num_kv_heads consecutive query heads
 *     share one KV head: query head h reads KV head h / G.
 *   - Calls that take a cudaStream_t are asynchronous on that stream; their
 *     return code reports host-side validation and launch errors only.  Errors
 *     found on the device (a block id outside the pool, a bounded wait that ran
 *     out) are recorded in the pool's status word and read by pkv_check_status.
 *   - No C++ exception crosses this boundary.  Functions returning int return a
 *     pkv_status (0 = success, negative = error).
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_API __attribute__((visibility("default")))

typedef enum {
  PKV_OK = 0,
  PKV_EINVAL = -1,       /* an argument is out of range or inconsistent */
  PKV_ENOMEM = -2,       /* the pool has too few free blocks, or the workspace is too small */
  PKV_ECUDA = -3,        /* a CUDA runtime call failed */
  PKV_EBOUNDS = -4,      /* (device) a block id or position outside the pool or table */
  PKV_ETIMEOUT = -5,     /* (device) a bounded wait inside a kernel ran out */
  PKV_EUNSUPPORTED = -6  /* a valid combination the library has no kernel for */
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_F16 = 1, PKV_BF16 = 2, PKV_FP8_E4M3 = 3 } pkv_dtype;

/* Geometry of one pool.  kv_dtype is fixed for the pool's lifetime. */
typedef struct {
  int32_t num_layers, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks;
  int32_t kv_dtype; /* a pkv_dtype */
} pkv_geometry;

/* Opaque, library-owned host state of a pool: geometry, the caller's device
 * buffer, the host block allocator (free list plus per-block reference counts)
 * and cached TMA descriptors. */
typedef struct pkv_pool pkv_pool;

/* Bytes of a device status word (int32 x 4) that kv_pool_create accepts. */
#define PKV_STATUS_BYTES 16

/* ---------------------------------------------------------------- pool sizing */

/* [MHPN] 3.1, [ENG26] 1.1: 2 x num_layers x num_kv_heads x head_dim x
 * (num_blocks x block_size) x bytes(kv_dtype).  Returns 0 for an invalid
 * geometry. */
PKV_API size_t kv_pool_bytes(const pkv_geometry* geom);

/* ---------------------------------------------------------------- pool lifetime */

/* Create the host state for a pool whose storage the caller owns.
 *   d_pool     device buffer of at least kv_pool_bytes(geom) bytes, 16-byte aligned
 *   pool_bytes its size
 *   d_status   device buffer of PKV_STATUS_BYTES bytes for the device error word
 *              (zeroed here), or NULL to not record device errors
 * Supported: head_dim in [8, 256] and a multiple of 8 (16 for E4M3);
 * block_size in [1, 256]; num_q_heads a multiple of num_kv_heads.
 * All blocks start free.  Returns PKV_OK and *out, or PKV_EINVAL. */
PKV_API int kv_pool_create(const pkv_geometry* geom, void* d_pool, size_t pool_bytes,
                           int32_t* d_status, pkv_pool** out);
PKV_API int kv_pool_destroy(pkv_pool* pool);
PKV_API int kv_pool_geometry(const pkv_pool* pool, pkv_geometry* out);

/* ---------------------------------------------------------------- host block allocator */
/* [ENG26] 2.2 allocate_block and [UNLOCK] 3.1 on-demand allocation: a
 * sequence's table grows by one block when its next token starts a new block.
 * The allocator is host-only and not thread-safe; ids are in [0, num_blocks). */

/* Take n free blocks (all or nothing: PKV_ENOMEM leaves the pool unchanged).
 * Each gets reference count 1.  out_block_ids: host int32[n]. */
PKV_API int kv_pool_alloc(pkv_pool* pool, int n, int32_t* out_block_ids);
/* Take these specific free blocks (all or nothing; PKV_EINVAL if one is taken
 * or repeated).  Lets a caller lay tables out over chosen ids. */
PKV_API int kv_pool_reserve(pkv_pool* pool, int n, const int32_t* block_ids);
/* Drop one reference from each block; a block whose count reaches 0 is free
 * again.  PKV_EINVAL (and no change) if any id is free or out of range. */
PKV_API int kv_pool_free(pkv_pool* pool, int n, const int32_t* block_ids);
/* Add one reference to each block (a shared prefix, [UNLOCK] 3.1 copy-on-write). */
PKV_API int kv_pool_share(pkv_pool* pool, int n, const int32_t* block_ids);
/* Reference count of a block (0 = free), or PKV_EINVAL. */
PKV_API int kv_pool_refcount(const pkv_pool* pool, int32_t block_id);
PKV_API int kv_pool_num_free(const pkv_pool* pool);
/* Copy-on-write before writing into block `id`: if its count is 1, *out_id = id;
 * otherwise take a free block, copy all of `id`'s bytes (every layer, K and V)
 * into it on `stream`, drop one reference from `id` and return the new id.
 * PKV_ENOMEM if no block is free. */
PKV_API int kv_pool_cow(pkv_pool* pool, int32_t id, int32_t* out_id, cudaStream_t stream);

/* Room for the next tokens of every sequence, before they are appended ([ENG26]
 * 2.2: append_token calls allocate_block when a token starts a new block;
 * [UNLOCK] 3.1: on-demand allocation, and copy-on-write of a block shared with
 * another sequence before it is written).  For s in [0, batch), sequence s holds
 * n = h_seq_lens[s] tokens and will append k = h_new_tokens[s] (NULL: 1 each):
 *   - table entries [ceil(n / bs), ceil((n + k) / bs)) get freshly taken blocks;
 *   - if k > 0 and n % bs != 0, the block at entry n / bs (the partly filled one
 *     the first new token lands in) is copied into a fresh block when its
 *     reference count is above 1, on `stream` (all layers, K and V), the entry
 *     is replaced and the shared block loses one reference.  Sequences sharing
 *     one tail are resolved in order: the last of them keeps the original.
 * h_block_tables: host int32 [batch, max_blocks_per_seq], updated in place (the
 * caller uploads the rows that changed before the append).  h_first_changed:
 * host int32 [batch] or NULL; receives the first changed entry of each row, or
 * -1.  All or nothing: PKV_ENOMEM if the free blocks do not cover every
 * sequence's need, PKV_EINVAL if a count is negative, a sequence would outgrow
 * max_blocks_per_seq or its tail entry is not a live block, PKV_ECUDA if a copy
 * cannot be issued; in each case pool and tables are unchanged.  Host-side and
 * not thread-safe with the other allocator calls. */
PKV_API int kv_pool_prepare_append(pkv_pool* pool, int batch, const int32_t* h_seq_lens,
                                   const int32_t* h_new_tokens, int32_t* h_block_tables,
                                   int max_blocks_per_seq, int32_t* h_first_changed,
                                   cudaStream_t stream);

/* ---------------------------------------------------------------- append (reshape_and_cache) */

/* [ENG26] 2.2 append_token, one token per sequence: for s in [0, batch),
 *   pos = d_positions[s], block = d_block_tables[s][pos / block_size],
 *   offset = pos % block_size,
 *   pool[block, 0, layer, :, offset, :] = d_k[s];  pool[block, 1, layer, :, offset, :] = d_v[s].
 * d_k, d_v: [batch, num_kv_heads, head_dim] in in_dtype.  For a pool of
 * kv_dtype f32/f16/bf16, in_dtype must equal kv_dtype and the bytes are copied.
 * For an E4M3 pool ([UNLOCK] 3.2, per-tensor FP8) in_dtype is f32, f16 or bf16
 * and each element is stored as e4m3(x / scale): IEEE fp32 division, round to
 * nearest even, finite overflow and +-Inf saturate to +-448, NaN -> 0x7F;
 * k_scale / v_scale (> 0) are used only for E4M3.  A negative position means
 * "no token for this sequence" and is skipped (padding).  A position past the
 * table, or a block id outside the pool, records PKV_EBOUNDS and skips that
 * token. */
PKV_API int kv_append(pkv_pool* pool, int layer, const void* d_k, const void* d_v,
                      pkv_dtype in_dtype, const int32_t* d_block_tables, int max_blocks_per_seq,
                      const int32_t* d_positions, int batch, float k_scale, float v_scale,
                      cudaStream_t stream);

/* The same store for num_tokens tokens: token i belongs to sequence
 * d_seq_ids[i] (< batch) at position d_positions[i] (a prefill or bulk fill).
 * Several tokens may target one sequence; two tokens must not target one slot
 * unless their values are equal. */
PKV_API int kv_append_tokens(pkv_pool* pool, int layer, const void* d_k, const void* d_v,
                             pkv_dtype in_dtype, const int32_t* d_block_tables,
                             int max_blocks_per_seq, int batch, const int32_t* d_seq_ids,
                             const int32_t* d_positions, int64_t num_tokens, float k_scale,
                             float v_scale, cudaStream_t stream);

/* Block-wise FP8 scaling ([UNLOCK] 3.2: one scale per 64-128 tokens).  Storage
 * is one fp32 scale per pool block, K or V, layer and KV head: d_scales is a
 * caller-owned device array [num_blocks, 2, num_layers, num_kv_heads] of fp32
 * (16-byte aligned); a scale group spanning several blocks stores its scale in
 * each of them (kv_block_scales).  While it is attached to an E4M3 pool,
 * kv_append, kv_append_tokens, paged_decode_step and every decode call encode and
 * dequantise each tile with its own slot's scale (x / scale stored, value x
 * scale read) and ignore their k_scale / v_scale arguments.  NULL detaches it.
 * PKV_EINVAL for a pool that is not E4M3. */
PKV_API int kv_pool_set_block_scales(pkv_pool* pool, float* d_scales);
/* Compute the attached block scales of every scale group the given tokens land
 * in (token i: sequence d_seq_ids[i], or i when d_seq_ids is NULL, at
 * d_positions[i]).  A scale group is group_tokens consecutive positions of a
 * sequence, [g x group_tokens, (g + 1) x group_tokens), a multiple of the block
 * size (0: one block; the pages' reading is 64 or 128); groups of sequences that
 * share their first block (a shared prefix) are one group.  Its scale is
 * amax / 448 over those tokens' finite elements (IEEE fp32 division; amax = 0
 * gives 1), written into the slot of every block of the group present in the
 * table; other slots keep their scales.  Run it on the tokens that fill a group
 * before storing them (a prefill): a group's scale must not change while it
 * holds encoded tokens, so later appends into its blocks reuse the scale and
 * values beyond 448 x scale saturate (a block taken later for a group's
 * remaining positions needs its slot set to the group's scale, for example by
 * this call over the group's tokens).  PKV_EINVAL for a group size that is not
 * a positive multiple of the block size. */
PKV_API int kv_block_scales(pkv_pool* pool, int layer, const void* d_k, const void* d_v,
                            pkv_dtype in_dtype, const int32_t* d_block_tables,
                            int max_blocks_per_seq, int batch, const int32_t* d_seq_ids,
                            const int32_t* d_positions, int64_t num_tokens, int group_tokens,
                            cudaStream_t stream);

/* Absolute maximum behind the per-tensor FP8 scale ([UNLOCK] 3.2): the largest
 * |x| over the finite elements of d_x (n elements of f32/f16/bf16; NaN and +-Inf
 * are left out, 0 if none is finite), written to *d_amax (device float) on
 * `stream`.  PKV_EINVAL for a NULL pointer, n < 0 or another dtype. */
PKV_API int kv_absmax(const void* d_x, pkv_dtype dtype, int64_t n, float* d_amax,
                      cudaStream_t stream);

/* Per-tensor FP8 E4M3 scale ([UNLOCK] 3.2, "per-tensor" FP8 with one fp32 scale
 * for K and one for V): *d_scale = amax / 448 in IEEE fp32 (round to nearest),
 * where amax is the largest of d_amax[0 .. n) -- the kv_absmax results of the
 * pieces a tensor is held in (for example the cached tokens and the new ones) --
 * and 448 is the largest finite E4M3 value, so the largest element is stored as
 * +-448.  amax = 0 gives 1.  Both pointers are device floats; asynchronous on
 * `stream`.  The result is what kv_append, kv_append_tokens and the decode calls
 * take as k_scale / v_scale.  PKV_EINVAL for a NULL pointer or n < 1. */
PKV_API int kv_fp8_scale(const float* d_amax, int n, float* d_scale, cudaStream_t stream);

/* ---------------------------------------------------------------- decode attention */

/* Workspace bytes paged_decode_attention needs on the current device for this
 * geometry, batch and num_splits (0 = automatic).  max_seq_len is the largest
 * seq_len the call will see. */
PKV_API size_t paged_decode_workspace_bytes(const pkv_geometry* geom, int batch, int max_seq_len,
                                            int num_splits);

/* Decode attention over the paged pool ([UNLOCK] 4.1 and 5.1, [MHPN] 1.1, 3.2):
 * for each sequence s < batch and query head h < num_q_heads, with
 * n = d_seq_lens[s] >= 0 tokens and kv head h / G,
 *   s_j = scale * <q[s,h,:], K_s[j,:]>,  w = softmax(s),  out[s,h,:] = sum_j w_j V_s[j,:]
 * where token j of sequence s is read from pool[table[s][j / bs], *, layer, kv, j % bs, :]
 * and E4M3 elements are dequantised as value x k_scale (K) or x v_scale (V).
 * A sequence with n = 0 gets out = 0.  On E4M3 pools bf16 / f16 q run on f16
 * tensor-core operands after an exact power-of-two prescale; f32 q runs on the
 * fp32 CUDA-core kernel.
 * The key range of each sequence is cut into partitions whose partial results
 * are merged by log-sum-exp ([SEQPAR] incremental softmax, [ENG26] 3.1):
 *   num_splits = 0: automatic.  The token stream of all sequences is cut into
 *     equal contiguous runs of blocks, one per resident CTA, so every SM reads
 *     the same number of bytes; sequences spanning several runs are merged.
 *   num_splits = S >= 1: every sequence is cut into S block-aligned partitions
 *     (partials in the workspace as [batch, num_q_heads, S, head_dim] fp32 plus
 *     [batch, num_q_heads, S] log-sum-exp, then merge_partials); S = 1 writes
 *     out directly.
 * d_q: [batch, num_q_heads, head_dim] in q_dtype; d_out same shape in out_dtype
 * (f32, f16 or bf16).  scale is the softmax scale (the pages use 1/sqrt(head_dim)).
 * d_workspace: at least paged_decode_workspace_bytes(...) bytes, 16-byte
 * aligned, device memory; it is scratch and needs no initialisation.
 * Errors: PKV_EINVAL (shapes, dtypes, batch < 0, max_seq_len < 0),
 * PKV_ENOMEM (workspace too small), PKV_EUNSUPPORTED, PKV_ECUDA. */
PKV_API int paged_decode_attention(void* d_out, pkv_dtype out_dtype, const void* d_q,
                                   pkv_dtype q_dtype, const pkv_pool* pool, int layer,
                                   const int32_t* d_block_tables, int max_blocks_per_seq,
                                   const int32_t* d_seq_lens, int batch, int max_seq_len,
                                   float scale, float k_scale, float v_scale, int num_splits,
                                   void* d_workspace, size_t ws_bytes, cudaStream_t stream);

/* Partial decode attention over the tokens this pool holds, for a key range of
 * each sequence split across GPUs ([SEQPAR] "numerically stable incremental
 * softmax": every device attends over its own range and the partial results are
 * combined by log-sum-exp; [ENG26] 3.1).  Same computation as
 * paged_decode_attention over the d_seq_lens[s] tokens of each sequence's table,
 * but it returns, per row (s, h) of batch x num_q_heads, the normalised fp32
 * output d_out [batch, num_q_heads, head_dim] and the natural log-sum-exp of the
 * row's scaled scores d_lse [batch, num_q_heads] (-inf and out = 0 for a
 * sequence with no tokens here).  Partials of the ranges of one sequence, stacked
 * as [batch, num_q_heads, ranges, head_dim] and [batch, num_q_heads, ranges],
 * give its whole attention through merge_partials.  Runs on the tensor-core
 * kernel (bf16 / f16 pools with q in the pool's dtype, E4M3 pools with bf16 / f16
 * q; head_dim 128), else PKV_EUNSUPPORTED.  The workspace is
 * paged_decode_workspace_bytes(geom, batch, max_seq_len, 0); other arguments and
 * errors as in paged_decode_attention. */
PKV_API int paged_decode_attention_partial(float* d_out, float* d_lse, const void* d_q,
                                           pkv_dtype q_dtype, const pkv_pool* pool, int layer,
                                           const int32_t* d_block_tables, int max_blocks_per_seq,
                                           const int32_t* d_seq_lens, int batch, int max_seq_len,
                                           float scale, float k_scale, float v_scale,
                                           void* d_workspace, size_t ws_bytes,
                                           cudaStream_t stream);

/* Launch choices a caller may force (tests, ablations, benchmarks).  Zero-filled
 * means "automatic" for every field. */
typedef struct {
  int32_t kernel;          /* 0 auto, 1 the SIMT kernel, 2 the mma.sync tensor-core kernel,
                              3 the tcgen05 chunked-prefill kernel (multi-token calls with
                              num_splits = 0; the shared-prefix entry reads 2 / 3 as its
                              plain / prefix-pass route) */
  int32_t ctas_per_sm;     /* 0 auto; the persistent grid is SMs x this */
  int32_t kv_heads_per_cta;/* 0 auto */
  int32_t stages;          /* 0 auto; shared-memory pipeline depth */
  int32_t phase;           /* 0 attention then merge, 1 attention only, 2 merge only */
  int32_t pdl;             /* 1: launch the attention kernel with programmatic dependent
                              launch, so that it starts while the launches before it in
                              the stream (for example the previous decode step's attention
                              and merge, chained the same way) finish.  Only valid when
                              those launches write none of q, the block tables, seq_lens or
                              k/v_new, and write the pool only within the last two blocks
                              of each sequence (a previous decode step's new token): the
                              kernel waits for them before it loads those two blocks and
                              before any write to out, the workspace and the pool. */
  int32_t reserved[2];
} pkv_launch_opts;

/* paged_decode_attention with forced launch choices.  phase 1 and 2 split the
 * call into its two kernels so a caller can time them apart; the workspace
 * carries the partial results from phase 1 to phase 2. */
PKV_API int paged_decode_attention_ex(void* d_out, pkv_dtype out_dtype, const void* d_q,
                                      pkv_dtype q_dtype, const pkv_pool* pool, int layer,
                                      const int32_t* d_block_tables, int max_blocks_per_seq,
                                      const int32_t* d_seq_lens, int batch, int max_seq_len,
                                      float scale, float k_scale, float v_scale, int num_splits,
                                      void* d_workspace, size_t ws_bytes,
                                      const pkv_launch_opts* opts, cudaStream_t stream);

/* One decode step for one layer: for every sequence s with n = d_seq_lens[s] >= 1
 * tokens (counting the new one), store the new token's d_k_new[s] / d_v_new[s]
 * ([batch, num_kv_heads, head_dim] in new_dtype) at position n - 1 exactly as
 * kv_append does ([ENG26] 2.2, [UNLOCK] 3.2), then compute
 * paged_decode_attention over the n tokens.  On the tensor-core kernel the store
 * is fused into the attention launch: the CTA that reads a sequence's last block
 * writes the token into it just before loading it, so the step is one attention
 * launch plus the merge.  The slot written must not be shared with another
 * sequence (copy it with kv_pool_cow first).  Other arguments and errors as in
 * paged_decode_attention_ex. */
PKV_API int paged_decode_step(void* d_out, pkv_dtype out_dtype, const void* d_q, pkv_dtype q_dtype,
                              const void* d_k_new, const void* d_v_new, pkv_dtype new_dtype,
                              const pkv_pool* pool, int layer, const int32_t* d_block_tables,
                              int max_blocks_per_seq, const int32_t* d_seq_lens, int batch,
                              int max_seq_len, float scale, float k_scale, float v_scale,
                              int num_splits, void* d_workspace, size_t ws_bytes,
                              const pkv_launch_opts* opts, cudaStream_t stream);

/* Multi-token decode: every sequence s has n = d_seq_lens[s] tokens in the pool,
 * the last q_len of which are new (already stored, e.g. by kv_append_tokens).
 * Query token i (0 <= i < q_len) of sequence s sits at position n - q_len + i and
 * attends causally over tokens 0 .. n - q_len + i -- the chunked-prefill /
 * speculative-verification reading of [UNLOCK] 5.2; q_len = 1 is
 * paged_decode_attention.  A query whose position is negative gets out = 0.
 * d_q and d_out: [batch, q_len, num_q_heads, head_dim].  The tensor-core kernel
 * (mma.sync) takes q_len * (num_q_heads / num_kv_heads) <= 16 rows per KV head
 * (<= 8 at block_size 64); larger chunks run on the tcgen05 kernel: UMMA tiles
 * of 128 query rows x 64 keys with S and O in tensor memory (num_splits must be
 * 0 there), head_dim 128, num_q_heads / num_kv_heads dividing 128.  bf16 / f16
 * pools take q in the pool's dtype; E4M3 pools take bf16 or f16 q (f32 q only
 * for q_len = 1, on the fp32 CUDA-core kernel).  E4M3 tiles become f16 operands
 * (exactly with per-tensor scales; with per-block ones each value times its
 * block's scale over the largest power of two among the blocks read, rounded to
 * f16), and q is multiplied by a power of two that puts its largest magnitude
 * just below f16's maximum before it is rounded to f16 (exact for bf16 and f16
 * values), so any finite q and any positive scales stay in range.  Other
 * combinations return PKV_EUNSUPPORTED.  Other arguments and errors as in
 * paged_decode_attention_ex; the workspace is paged_decode_workspace_bytes_mq. */
PKV_API int paged_decode_attention_mq(void* d_out, pkv_dtype out_dtype, const void* d_q,
                                      pkv_dtype q_dtype, int q_len, const pkv_pool* pool,
                                      int layer, const int32_t* d_block_tables,
                                      int max_blocks_per_seq, const int32_t* d_seq_lens,
                                      int batch, int max_seq_len, float scale, float k_scale,
                                      float v_scale, int num_splits, void* d_workspace,
                                      size_t ws_bytes, const pkv_launch_opts* opts,
                                      cudaStream_t stream);
/* Workspace bytes of paged_decode_attention_mq (an upper bound over launch plans). */
PKV_API size_t paged_decode_workspace_bytes_mq(const pkv_geometry* geom, int batch, int q_len,
                                               int max_seq_len, int num_splits);

/* Decode attention over sequences that share a prefix of blocks ([UNLOCK] 3.1:
 * a shared prompt prefix is one set of physical blocks referenced by many
 * tables, copy-on-write).  The result equals paged_decode_attention_ex over each
 * sequence's own table; the shared blocks are read once per KV head for all
 * sequences instead of once per sequence:
 *   1. sequence s's first d_prefix_lens[s] tokens (a multiple of block_size,
 *      0 .. prefix_len_max) must be blocks d_prefix_table[0 .. d_prefix_lens[s] /
 *      block_size) -- the same ids as its own table (checked on the device;
 *      a mismatch, a length that is not a multiple of block_size or exceeds the
 *      sequence or prefix_len_max is reported by pkv_check_status as PKV_EINVAL);
 *   2. the prefix keys are attended by all batch x num_q_heads query rows at
 *      once on the tcgen05 kernel (128-row query tiles, key range split across
 *      CTAs), each row limited to its own prefix length, giving fp32 partials;
 *   3. each sequence's remaining tokens go through the decode kernel, which
 *      reads its own table from entry d_prefix_lens[s] / block_size on (a
 *      sequence whose prefix fails the check of step 1 is read from its first
 *      token), and one merge combines all partials by log-sum-exp ([SEQPAR]
 *      incremental softmax).
 * d_prefix_table: int32 [prefix_blocks], prefix_len_max <= prefix_blocks *
 * block_size (0: plain decode through the same path).  bf16 / f16 pools with q
 * in the pool's dtype, or E4M3 pools with bf16 / f16 q (k_scale / v_scale as in
 * paged_decode_attention, > 0, ignored for other pools and when the pool has
 * per-block scales attached); head_dim 128, num_q_heads / num_kv_heads dividing
 * 128 and at most 8 (16 at block size <= 32); otherwise PKV_EUNSUPPORTED (bad
 * scales: PKV_EINVAL).  The workspace (caller-owned, 16-byte aligned) is
 * paged_decode_workspace_bytes_cascade; other arguments, ownership and errors as
 * in paged_decode_attention_ex.
 * When it pays: the prefix pass replaces one read of the shared blocks per
 * sequence.  A prefix whose K/V (prefix_len_max x 2 x num_kv_heads x head_dim
 * elements) fill at most a quarter of the device's L2 is read from HBM about
 * once by the plain decode too (the sequences reach their first blocks together
 * and the repeats hit in L2); the extra pass and merge would then cost more than
 * they save, so such a call runs steps 2-3 as paged_decode_attention over the
 * sequences' own tables, after the same check of step 1.  opts->kernel (opts
 * may be NULL): 0 that automatic choice, 2 always the plain decode, 3 always the
 * prefix pass; other values PKV_EINVAL.  opts->phase splits the call so that a
 * caller can time its parts: 0 everything, 1 steps 1-2 (the prefix check and
 * the prefix pass), 2 step 3 (the suffix decode and the merge; needs a phase-1
 * call with the same arguments and workspace before it on the stream); other
 * values PKV_EINVAL.  The other fields are ignored.
 * Measured on one GB300: 32 sequences sharing 64K tokens (268 MB of K/V), 7.6x
 * faster than paged_decode_attention; 64 sequences sharing 4K tokens (17 MB),
 * the prefix pass (the automatic choice there) 3% faster than the plain decode. */
PKV_API int paged_decode_attention_cascade(void* d_out, pkv_dtype out_dtype, const void* d_q,
                                           pkv_dtype q_dtype, const pkv_pool* pool, int layer,
                                           const int32_t* d_prefix_table, int prefix_blocks,
                                           int prefix_len_max, const int32_t* d_prefix_lens,
                                           const int32_t* d_block_tables, int max_blocks_per_seq,
                                           const int32_t* d_seq_lens, int batch, int max_seq_len,
                                           float scale, float k_scale, float v_scale,
                                           void* d_workspace, size_t ws_bytes,
                                           const pkv_launch_opts* opts, cudaStream_t stream);
/* Workspace bytes of paged_decode_attention_cascade (an upper bound over launch plans). */
PKV_API size_t paged_decode_workspace_bytes_cascade(const pkv_geometry* geom, int batch,
                                                    int max_blocks_per_seq, int max_seq_len,
                                                    int prefix_len_max);

/* Log-sum-exp merge of partial results ([SEQPAR] incremental softmax,
 * [ENG26] 3.1): for each row r = (s, h) of batch x num_q_heads,
 *   M = max_p lse[r,p],  w_p = exp(lse[r,p] - M),
 *   out[r,:] = sum_p w_p O[r,p,:] / sum_p w_p.
 * d_part_o: fp32 [batch, num_q_heads, num_splits, head_dim], each partial
 * already normalised; d_part_lse: fp32 [batch, num_q_heads, num_splits],
 * natural log-sum-exp of that partition's scores.  A partial with lse = -inf
 * has weight 0; a row whose partials are all -inf gets out = 0.
 * d_out: [batch, num_q_heads, head_dim] in out_dtype (f32, f16, bf16). */
PKV_API int merge_partials(void* d_out, pkv_dtype out_dtype, const float* d_part_o,
                           const float* d_part_lse, int batch, int num_q_heads, int head_dim,
                           int num_splits, cudaStream_t stream);

/* ---------------------------------------------------------------- decode without a workspace */

/* Size of the library's built-in scratch array used by
 * paged_decode_attention_static (16 MiB per GPU that loads the library). */
#define PKV_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/* paged_decode_attention for callers that cannot allocate device memory when
 * they run it (an allocator frozen during graph capture, a plugin that only
 * receives its input and output buffers, a loop that must not allocate after
 * start-up).  The source pages have no counterpart: this is an interface
 * convenience of this library.
 * Same arguments and result as paged_decode_attention, minus the workspace:
 * the partial results live in a fixed array inside the library
 * (PKV_STATIC_SCRATCH_BYTES), so the call allocates nothing.
 *   - Returns PKV_ENOMEM, launching nothing, if the workspace this call's
 *     launch plan needs is larger than the array (paged_decode_workspace_bytes
 *     is an upper bound of that need).
 *   - Every call on a device shares the array and the array keeps what the last
 *     call left; no part of it needs to start at zero.  Calls whose kernels may
 *     overlap on the GPU (unordered streams) race on it and must be serialised.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture. */
PKV_API int paged_decode_attention_static(void* d_out, pkv_dtype out_dtype, const void* d_q,
                                          pkv_dtype q_dtype, const pkv_pool* pool, int layer,
                                          const int32_t* d_block_tables, int max_blocks_per_seq,
                                          const int32_t* d_seq_lens, int batch, int max_seq_len,
                                          float scale, float k_scale, float v_scale,
                                          int num_splits, cudaStream_t stream);

/* ---------------------------------------------------------------- status */

/* Synchronise `stream`, read and clear the pool's device status word and
 * return the first error recorded since the last check (PKV_OK if none;
 * PKV_OK too if the pool has no status word). */
PKV_API int pkv_check_status(const pkv_pool* pool, cudaStream_t stream);
/* A static string naming a pkv_status. */
PKV_API const char* pkv_strerror(int status);
/* Failure-detection self-test.  One warp waits, through the bounded wait every
 * kernel of this library uses on its mbarriers, on a barrier that nothing
 * arrives on; when the bound runs out (1 s of the GPU's global timer) it
 * records PKV_ETIMEOUT in the pool's status word and the kernel exits, so the
 * next pkv_check_status returns PKV_ETIMEOUT and the context stays usable.
 * Asynchronous on `stream`; returns PKV_EINVAL for a NULL pool or one without a
 * status word, PKV_ECUDA if the launch fails. */
PKV_API int pkv_wait_selftest(const pkv_pool* pool, cudaStream_t stream);
/* Number of kernel launches this library has issued in this process (a
 * counter the benchmark reads to report its launches). */
PKV_API uint64_t pkv_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H_ */
