/*
 * tq.h - C ABI of libtq: TurboQuant KV-cache hot path on one GB300 (sm_103a).
 *
 * The method, as the sources state it. [Guide] = the TurboQuant-on-vLLM guide at
 * hotelren.com/news/5528865.
 *   - quantize-on-append ([Guide] §二, the five-step pipeline): rotate each key/value head vector
 *     with a seeded randomised Hadamard transform and store the key norm. Then code the key with a
 *     2-bit Lloyd-Max codebook for the rotated-coordinate (Beta) distribution, and add one QJL
 *     sign bit per dimension on the key residual (3-bit keys). Values are quantised symmetrically
 *     at 2 or 4 bits in groups of 32 with an fp16 scale per group. Everything is bit-packed.
 *   - hybrid decode attention ([Guide] §五.1 and §七): scores are estimated straight from the
 *     packed keys plus the QJL correction, against a rotated, projected query. Values are
 *     dequantised inside an online softmax. The result is merged exactly with a bf16 ring buffer
 *     of the most recent 128 tokens (buffer_size=128, [Guide] §五.1).
 *
 * Conventions (all calls):
 *   - Pointers prefixed d_ are DEVICE pointers; all others are host pointers.
 *   - The caller owns every device buffer (tables, cache, workspace). The library never allocates
 *     device memory; it allocates only its small host-side context.
 *   - Work is enqueued asynchronously on the caller's CUDA stream `stream`. Calls on one layer must
 *     be ordered by the caller (same stream, or events).
 *   - Kernels are launched with programmatic dependent launch: a kernel may start, and read its
 *     inputs (q, k, v, seq_ids, n_new, the tables, the packed pages), as soon as the previous kernel
 *     on the stream releases its dependents. Every kernel of this library does that only after it
 *     has itself waited for its own predecessor. A caller kernel that releases dependents early
 *     (griddepcontrol.launch_dependents) must have finished writing those inputs first; kernels that
 *     do not use that instruction, and copies, need no care.
 *   - Every argument is validated on the host before any launch. A bad argument returns
 *     TQ_ERR_INVALID_ARG and an unsupported shape returns TQ_ERR_UNSUPPORTED; nothing is launched
 *     in either case. A launch failure returns TQ_ERR_CUDA. tq_last_error() gives the reason
 *     (thread-local string).
 *   - Conditions that only the device can see (a sequence growing past max_ctx, a bad sequence id)
 *     set bits of a device status word instead of faulting. tq_check_status() reads that word.
 *     Kernels never trap and never wait without a bound.
 *   - No C++ exception crosses this ABI.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tq_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum tq_status {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,
  TQ_ERR_UNSUPPORTED = 2,
  TQ_ERR_CAPACITY = 3,
  TQ_ERR_CUDA = 4,
  TQ_ERR_DEVICE = 5 /* the device status word is non-zero (see tq_check_status) */
} tq_status;

typedef enum tq_dtype { TQ_BF16 = 0, TQ_F32 = 1 } tq_dtype;

/* Device status word bits. */
#define TQ_DEV_ERR_CAPACITY 0x1u /* an append would grow a sequence past max_ctx; the row was skipped */
#define TQ_DEV_ERR_SEQ_ID 0x2u   /* a sequence id outside [0, max_seqs); the row was skipped */
#define TQ_DEV_ERR_SPLITS 0x4u   /* decode saw more packed pages than its grid covers (max_ctx_hint too small) */
#define TQ_DEV_ERR_TIMEOUT 0x8u  /* a bounded wait on a bulk copy gave up; that split was dropped */
#define TQ_DEV_ERR_BLOCK 0x10u   /* paged cache: a page that an append or decode touched has no valid block in
                                  * the block table; the append skipped it, the decode result is undefined */

/* Configuration. The key has key_bits bits per coordinate: a (key_bits - 1)-bit Lloyd-Max code plus 1 QJL
 * sign bit ([Guide] §二 steps 2-3; §五.1 key_bits=3). key_bits 4 is the 4-bit TurboQuant row of the
 * overview's table (§性能表现与实测数据), read as a 3-bit code plus the sign; it is served with
 * value_bits 4. */
typedef struct tq_config {
  int32_t head_dim;    /* d: 64, 128 or 256 */
  int32_t key_bits;    /* 3, or 4 with value_bits 4 (TQ_ERR_UNSUPPORTED otherwise) */
  int32_t value_bits;  /* 2 or 4 ([Guide] §二 step 4) */
  int32_t value_group; /* 32 ([Guide] §二 step 4) */
  int32_t ring_size;   /* 128: hybrid mode, exact recent buffer ([Guide] §五.1 buffer_size=128);
                        * 0: full_tq mode ([Guide] §三): every token is quantised by its append and decode
                        * reads only packed tokens. The bf16 ring is still allocated, as a staging copy of
                        * the current block: each append codes the 32-token blocks that hold its new tokens
                        * (older tokens of such a block again, with identical codes) and publishes F = L - Np. */
  int32_t n_layers;
  int32_t n_kv_heads;
  int32_t n_q_heads;   /* multiple of n_kv_heads, with n_q_heads / n_kv_heads in {1, 2, 4} (GQA) */
  int32_t max_seqs;    /* number of sequence slots in the cache */
  int32_t max_ctx;     /* maximum tokens per sequence (packed + ring) */
  uint64_t seed;       /* seeds the rotation signs D and the QJL matrix S (SplitMix64) */
  int32_t n_blocks;    /* 0: every (layer, slot, KV head) owns max_pages = ceil(max_ctx / 128) contiguous
                        * pages. > 0: paged cache ([Guide] §七: the engine's KV cache lives in paged blocks). Each layer
                        * holds a pool of n_blocks blocks; a block is one 128-token page of every KV head. The
                        * int32 block table [max_seqs][max_pages] (in the cache buffer, see
                        * tq_block_table_offset) maps (slot, page) to a block; the caller fills it before an
                        * append or decode touches the page, with ids in [0, n_blocks) and no block shared by
                        * two live pages. It is the same table for every layer. */
} tq_config;

typedef struct tq_ctx tq_ctx; /* opaque host object owned by the library */

/* Bytes of the device tables buffer (rotation signs, S, S^T, codebook) for `cfg`; 0 if cfg is invalid. */
size_t tq_tables_bytes(const tq_config* cfg);

/* Bytes of the device cache buffer for `cfg`; 0 if invalid. Layout, in order:
 *   - packed pages [layer][slot][kv_head][page][page_bytes], or for a paged cache (n_blocks > 0)
 *     [layer][block][kv_head][page_bytes];
 *   - bf16 ring K and V [layer][slot][kv_head][ring][d];
 *   - int32 state [layer][slot][2]: total length L and flushed ring prefix F;
 *   - the int32 device status word. */
size_t tq_cache_bytes(const tq_config* cfg);

/* Bytes of one packed page of 128 tokens of one KV head (the fragment-major record layout). */
size_t tq_page_bytes(const tq_config* cfg);

/* tq_init_codebooks: creates a context for `cfg`.
 *   - Computes on the host, in fp64: the 2-bit Lloyd-Max codebook of the density
 *     f_d(x) ~ (1-x^2)^((d-3)/2) ([Guide] §二 step 2: "Beta-distribution-optimal codebook").
 *   - Computes the seeded rotation signs D and QJL matrix S (SplitMix64, Box-Muller, bf16).
 *   - Uploads both with cudaMemcpyAsync on `stream` into the caller's d_tables (at least
 *     tq_tables_bytes(cfg) bytes, 256-byte aligned).
 * The context is bound to the current CUDA device. *out is freed by tq_destroy. */
tq_status tq_init_codebooks(const tq_config* cfg, void* d_tables, size_t tables_bytes, tq_stream_t stream,
                            tq_ctx** out);

/* Binds the caller's cache buffer: d_cache (at least tq_cache_bytes, 256-byte aligned). The
 * sequence state and status word are zeroed on `stream`, so every slot starts empty. */
tq_status tq_cache_bind(tq_ctx* ctx, void* d_cache, size_t cache_bytes, tq_stream_t stream);

/* Empties the sequences d_seq_ids[0..batch) of `layer` (layer = -1: every layer). */
tq_status tq_reset_seqs(tq_ctx* ctx, int layer, const int32_t* d_seq_ids, int batch, tq_stream_t stream);

/* tq_quantize_append: appends new tokens to sequences of one layer ([Guide] §二 pipeline and §五.1:
 * prefill is captured in bulk, decode tokens go into the ring buffer).
 *   - k, v: device arrays [batch][max_new][n_kv_heads][d] of dtype `dt`. Row b uses its first
 *     d_n_new[b] tokens.
 *   - d_seq_ids[b]: the cache slot of row b. d_n_new[b] is in [0, max_new].
 *   - Ring semantics: the ring holds the last R = L - 128*floor((L-1)/128) tokens of a length-L
 *     sequence, so decode reads 128*floor((L-1)/128) packed tokens + R ring tokens. An append
 *     quantises every 128-token block it completes into its packed page at once, including the
 *     block that fills the ring to R = 128 (decode keeps reading those from the ring until the next
 *     token starts a new ring block); so the pages of all blocks below 128*floor(L/128) are written.
 *   - f32 inputs enter the ring rounded to bf16. Blocks that never pass through the ring are
 *     quantised from the f32 values.
 *   - A row that would exceed max_ctx is skipped and sets TQ_DEV_ERR_CAPACITY.
 *   - Launches: for max_new < 128, one kernel (the page of a block the append completes, the ring rows
 *     and the new length); otherwise one quantize kernel over the pages to write (for bf16 tokens a
 *     persistent tensor-core coder, one CTA per SM, at head_dim 64, 128 and 256; for f32 tokens four
 *     CTAs per page), then the ring rows and the new lengths (two kernels; in full_tq mode followed by
 *     the two launches of tq_ring_flush). */
tq_status tq_quantize_append(tq_ctx* ctx, int layer, const void* k, const void* v, tq_dtype dt,
                             const int32_t* d_seq_ids, const int32_t* d_n_new, int batch, int max_new,
                             tq_stream_t stream);

/* tq_ring_flush: quantises the ring of each row into the packed history now ("periodically flush
 * the residual cache into the main cache", [Overview] §核心技术解析, Bonsai residual cache).
 *   - Afterwards decode treats all L tokens as packed.
 *   - The bf16 copies stay in the ring until the block is complete, and that block is re-quantised
 *     with identical codes when it completes. Quantisation is per token, so the codes do not change.
 *   - Rows with an empty ring are unchanged. */
tq_status tq_ring_flush(tq_ctx* ctx, int layer, const int32_t* d_seq_ids, int batch, tq_stream_t stream);

/* tq_dequantize_tokens: reconstructs packed tokens [t0, t0 + count) of (layer, seq_slot, kv_head) in the
 * original basis, for fidelity reports and tests (the decode never dequantises keys; [Guide] §六 quotes the
 * cosine similarity of such reconstructions):
 *   k_hat = n Pi^T (c[idx] + sqrt(pi/2)/d gamma S^T sigma)   (with_qjl = 1; with_qjl = 0 drops the QJL term)
 *   v_hat = Pi^T ((code - 2^(value_bits-1) + 1/2) s_g)
 * with Pi = H diag(D) / sqrt(d), sigma_i = +1 where the stored sign bit is set and -1 elsewhere, and n,
 * gamma, s_g the stored fp16 values ([Guide] §二 steps 1-4).
 *   - d_k_out, d_v_out: device fp32 [count][head_dim], row i for token t0 + i. Caller-owned; not aliased.
 *   - Tokens are positions in the sequence; only positions below the row's packed count (its length less
 *     the ring) hold codes, and others give unspecified values. A paged cache's page without a block gives
 *     zeros and TQ_DEV_ERR_BLOCK on the status word.
 *   - Asynchronous on `stream`, ordered after earlier appends on it. Errors (on the host, before launch):
 *     TQ_ERR_INVALID_ARG for a bad layer, slot, head, negative t0 or count, with_qjl not 0 or 1, NULL
 *     outputs with count > 0, or no cache bound; TQ_ERR_CAPACITY for tokens past the sequence's pages. */
tq_status tq_dequantize_tokens(tq_ctx* ctx, int layer, int seq_slot, int kv_head, int t0, int count, int with_qjl,
                               float* d_k_out, float* d_v_out, tq_stream_t stream);

/* Bytes of the decode workspace for `batch` rows and a longest sequence of `max_ctx_hint` tokens
 * (0 = cfg.max_ctx). The same workspace serves tq_decode_attention, tq_decode_phase and
 * tq_decode_step. */
size_t tq_workspace_bytes(const tq_ctx* ctx, int batch, int max_ctx_hint);

/* tq_decode_attention: one decode step of hybrid attention for one layer ([Guide] §五.1 and §七).
 *   - q: device bf16 [batch][n_q_heads][d] (one query token per row).
 *   - out: device f32 [batch][n_q_heads][d].
 *   - Query head h attends KV head h / (n_q_heads / n_kv_heads).
 *   - softmax_scale <= 0 selects 1/sqrt(d).
 *   - Scores use the TurboQuant estimator n*(<Pi q, c[idx]> + sqrt(pi/2)/d * gamma * <S Pi q, sign>)
 *     over the packed history, and exact dot products over the ring.
 *   - One softmax runs over both.
 *   - d_workspace: at least tq_workspace_bytes(ctx, batch, max_ctx_hint) bytes, 256-byte aligned,
 *     scratch owned by the caller. It starts with per-(row, KV head) and per-row arrival counters
 *     that must be zero before the first call on a workspace (zero-fill it once); every call leaves
 *     them at zero again.
 *   - max_ctx_hint: an upper bound on every row's length (0 = cfg.max_ctx). It only sizes the grid;
 *     a row longer than the hint sets TQ_DEV_ERR_SPLITS.
 *   - Launches: one split-K decode kernel (+ the ring split). Every split CTA rotates and projects
 *     the query itself; the last CTA of each (row, KV head) runs the combine. */
tq_status tq_decode_attention(tq_ctx* ctx, int layer, const void* q, float* out, const int32_t* d_seq_ids,
                              int batch, float softmax_scale, void* d_workspace, size_t workspace_bytes,
                              int max_ctx_hint, tq_stream_t stream);

/* tq_decode_step: one decode step of one layer in one launch: appends one new token to every row
 * and attends q over the sequence that includes it. The results, the cache contents and the sequence
 * state are identical to tq_quantize_append with d_n_new[b] = 1 followed by tq_decode_attention, in
 * one kernel instead of two ([Guide] §五.1 ring buffer, §三 hybrid decode, §二 pipeline).
 *   - k_new, v_new: device [batch][n_kv_heads][d] of dtype dt (bf16 or f32), aligned to 4 elements.
 *   - q, out, d_seq_ids, softmax_scale, d_workspace, workspace_bytes: as tq_decode_attention.
 *     max_ctx_hint must cover every row's length after its new token.
 *   - The ring split of each (row, KV head) takes the new token from k_new / v_new, attends to it and
 *     writes it into the ring. When the token fills the ring to 128, that CTA also codes the 128
 *     ring tokens into their packed page (the next step then starts a new ring block over it). The
 *     last (row, KV head) of a row to finish publishes the row's new length.
 *   - A row already at max_ctx gets no token (TQ_DEV_ERR_CAPACITY) and is decoded as it stands; an
 *     invalid slot sets TQ_DEV_ERR_SEQ_ID.
 *   - A launch of this library that directly follows a decode step of the same layer on the same
 *     stream reads the sequence state only after its stream wait (the step publishes it at its end).
 *   - full_tq contexts (ring_size 0) run it as the append and decode launches. */
tq_status tq_decode_step(tq_ctx* ctx, int layer, const void* k_new, const void* v_new, tq_dtype dt, const void* q,
                         float* out, const int32_t* d_seq_ids, int batch, float softmax_scale, void* d_workspace,
                         size_t workspace_bytes, int max_ctx_hint, tq_stream_t stream);

/* tq_decode_phase: launches one phase of tq_decode_attention with the same arguments, for callers that
 * interleave the phases with other work or time them one by one. The two phases run in order on one
 * workspace:
 *   0 = zero the workspace's arrival counters (a memset; needed once before the first phase-1 call
 *       on a workspace that was not zero-filled);
 *   1 = split-K decode over packed pages (each split CTA prepares the query: rotation, projection,
 *       f16 operands of the key bit-plane MMAs) plus the exact ring split. The last CTA of every
 *       (row, KV head) also runs the combine: log-sum-exp merge, inverse rotation, ring merge -> out.
 * Any other phase returns TQ_ERR_INVALID_ARG. Phase 1 leaves the counters at zero, so calling 0 and
 * then 1, or just 1 on a zeroed workspace, is equivalent to one tq_decode_attention call. */
tq_status tq_decode_phase(tq_ctx* ctx, int phase, int layer, const void* q, float* out, const int32_t* d_seq_ids,
                          int batch, float softmax_scale, void* d_workspace, size_t workspace_bytes,
                          int max_ctx_hint, tq_stream_t stream);

/* tq_prefill_attention: attention of a prefill chunk over the cache of one layer. The chunk's tokens
 * must already be appended (tq_quantize_append); row b's queries are its sequence's last d_n_q[b]
 * tokens. Query i of the row (position L - n_q + i) attends causally to every position up to its own,
 * through the same estimator as tq_decode_attention: packed tokens through their codes, ring tokens
 * exactly ([Guide] §七: prefill attention; here over the packed history).
 *   - q: device bf16 [batch][q_per_row][n_q_heads][d]; out: device f32 of the same shape. Queries
 *     i >= d_n_q[b] of a row are padding: their outputs are zero.
 *   - d_n_q[b] in [0, q_per_row] and at most the row's length; d_seq_ids as for decode.
 *   - d_workspace: at least tq_prefill_workspace_bytes(ctx, batch, q_per_row, max_ctx_hint) bytes,
 *     256-byte aligned; its arrival counters are zeroed by every call (one memset).
 *   - batch * q_per_row <= 65535.
 *   - Launches, head_dim 128 with key_bits 3, 4 query heads per KV head and q_per_row >= 32:
 *       1. a kernel that expands every packed page of every (row, KV head) once, into f16 tensor-core
 *          tiles in the workspace (128.5 KB per page and KV head, for the pages of max_ctx_hint tokens);
 *       2. a tcgen05 kernel over tiles of 128 query rows (32 queries x the 4 query heads of one KV head)
 *          that copies those tiles in and computes scores and P.V on the tensor cores into TMEM, writing
 *          one partial per (query, KV head, history split);
 *       3. a kernel with one CTA per (query, KV head): the exact ring split of the ring tokens that the
 *          query sees, the log-sum-exp merge of the history partials, the inverse rotation, the merge.
 *     A row longer than max_ctx_hint sets TQ_DEV_ERR_SPLITS and leaves its pages past the hint out.
 *   - Other shapes: the memset and one split-K decode kernel over batch * q_per_row query rows (the
 *     rows of one sequence read the same pages, mostly from L2). With an even q_per_row and a
 *     contiguous cache, each CTA takes two adjacent query rows of a sequence in the MMAs' 8 query
 *     columns, so they share the expanded key bits.
 *   - The workspace size depends on these choices; tq_prefill_workspace_bytes makes the same ones. */
size_t tq_prefill_workspace_bytes(const tq_ctx* ctx, int batch, int q_per_row, int max_ctx_hint);
tq_status tq_prefill_attention(tq_ctx* ctx, int layer, const void* q, float* out, const int32_t* d_seq_ids,
                               const int32_t* d_n_q, int batch, int q_per_row, float softmax_scale,
                               void* d_workspace, size_t workspace_bytes, int max_ctx_hint, tq_stream_t stream);

/* tq_decode_attention_noalloc: the same decode step as tq_decode_attention, for callers that cannot
 * allocate device memory when they decode. Examples: code on a path where cudaMalloc's implicit
 * synchronisation is forbidden, or a host runtime that owns all device memory and only hands over the
 * operation's own tensors. The sources have no counterpart of this call; it is an ABI convenience.
 *   - The caller passes only inputs and outputs (q, out, d_seq_ids). The scratch lives in a 4 MiB
 *     device array inside libtq, which every GPU that loads the library holds until the process exits.
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 *   - Sizes whose scratch (tq_workspace_bytes(ctx, batch, max_ctx_hint)) exceeds 4 MiB are rejected
 *     with TQ_ERR_CAPACITY and a message; nothing is launched.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress) with
 *     that device current. Make that first call before any stream capture.
 *   - Every call shares the one array, whose contents persist between calls. The only entries that
 *     must start at zero are the arrival counters: 16384 of them, one per (row, KV head), in a fixed
 *     region at the start of the array for every context (so batch x n_kv_heads <= 16384, else
 *     TQ_ERR_CAPACITY); the split partials follow that region. The array is zero-filled when the library
 *     loads and every call leaves the counters at zero; everything else a call reads, it writes first, so
 *     calls on contexts of different shapes may alternate. Calls that overlap on the GPU (on different
 *     streams, or from different host threads) race on it and give wrong results; order them. */
tq_status tq_decode_attention_noalloc(tq_ctx* ctx, int layer, const void* q, float* out, const int32_t* d_seq_ids,
                                      int batch, float softmax_scale, int max_ctx_hint, tq_stream_t stream);

/* Test hook for the bounded waits of the decode kernels (not part of the decode itself). stage >= 0 makes
 * every following tq_decode_attention / tq_decode_phase / tq_decode_attention_noalloc launch at head_dim 128
 * leave one page stage without its copy: in the first split CTA of row 0, KV head 0, the first page stream issues neither
 * the copy nor the expected-byte count of page stage `stage` (0 .. stages - 1; a stage the kernel does not
 * have is ignored), and its wait on that stage gives up after `polls` polls (1 .. 2^22). The kernel then
 * sets TQ_DEV_ERR_TIMEOUT, waits (bounded) for every copy it did issue, and returns; that unit's output is
 * unspecified, every other unit's is exact, and the workspace stays usable. Nothing faults or hangs.
 * stage = -1 turns the hook off (the default). Returns TQ_ERR_INVALID_ARG for values out of range.
 * Process-wide; set it only while no other thread launches decodes. */
tq_status tq_debug_decode_wait_fault(int stage, int polls);

/* Test hook for the bounded waits of the tcgen05 bulk coders (bf16 appends of >= 128 tokens at head_dim 64,
 * 128 and 256; not part of the append itself). task >= 0 makes every following such tq_quantize_append skip the
 * TMA copy of page task `task`, numbered (row * n_kv_heads + head) * pages_per_row + j with
 * pages_per_row = ceil(max_new / 128) and j the j-th complete block the append codes for that row: the CTA
 * that owns the task issues neither the copy nor its expected-byte count, and its wait on it gives up after
 * `polls` polls (1 .. 2^22). That CTA then sets TQ_DEV_ERR_TIMEOUT, waits (bounded) for every copy and MMA
 * batch it did issue, frees its tensor memory and returns: the pages it had not finished are unspecified,
 * every other page is exact, and the cache stays usable. A task that is not a TMA copy (a page that starts
 * in the ring, or no such task) changes nothing. Nothing faults or hangs. task = -1 turns the hook off (the
 * default). Returns TQ_ERR_INVALID_ARG for values out of range. Process-wide; set it only while no other
 * thread appends. */
tq_status tq_debug_append_wait_fault(int task, int polls);

/* Test hook for the bounded waits of the tcgen05 prefill kernel (not part of the prefill itself). While
 * page >= 0, CTA (0, 0, 0) of every following tcgen05 prefill launch (query tile 0, KV head 0, batch row 0,
 * history split 0) issues neither the copy of the expanded h and l tiles of the page with index `page`
 * within its split nor that copy's expected-byte count, and its wait for them gives up after `polls` polls
 * (1 .. 2^22). That CTA then
 * sets TQ_DEV_ERR_TIMEOUT, waits (bounded) for every copy and MMA batch it did issue, frees its tensor
 * memory and writes an empty partial: the outputs of its 32 queries x 4 query heads are unspecified, every
 * other output is as without the hook, and the context stays usable. A page index the CTA does not reach
 * changes nothing. Nothing faults or hangs. page = -1 turns the hook off (the default). Returns
 * TQ_ERR_INVALID_ARG for values out of range. Process-wide; set it only while no other thread calls the
 * prefill. */
tq_status tq_debug_prefill_wait_fault(int page, int polls);

/* Test hook for the two prefill paths (not part of the prefill itself): mode 1 makes every following
 * tq_prefill_attention (and tq_prefill_workspace_bytes) take the CUDA-core decode-kernel path even where
 * the tcgen05 path applies; mode 0 (the default) chooses automatically. Returns TQ_ERR_INVALID_ARG for
 * other values. Process-wide; set it only while no other thread calls the prefill. */
tq_status tq_debug_prefill_path(int mode);

/* Synchronises `stream` and reads the device status word. It returns TQ_OK if the word is zero.
 * Otherwise it returns TQ_ERR_DEVICE and stores the word in *word (if non-NULL). `clear` != 0
 * zeroes the word afterwards. */
tq_status tq_check_status(tq_ctx* ctx, tq_stream_t stream, uint32_t* word, int clear);

/* Frees the host context (device buffers stay owned by the caller). */
void tq_destroy(tq_ctx* ctx);

/* Thread-local description of the last error (empty string if none). */
const char* tq_last_error(void);

/* ---- Comparison codecs (stateless; no context) ----
 * KIVI 2-bit and Bonsai 1-bit, the two other KV codecs of the TurboQuant-vLLM overview
 * (§核心技术解析, sizes in §性能表现与实测数据). The overview names the schemes but not their parameters.
 * These entry points take the plainest reading that gives its table's sizes (KIVI 2-bit 1,024 MB,
 * Bonsai 1-bit 288 MB for Llama-3.1-8B at 32K tokens).
 *
 * Inputs are bf16 K and V laid out [n_tokens][n_heads][head_dim] (row-major, device). Groups never
 * cross a head. Every pointer is a device pointer owned by the caller, and every call is asynchronous
 * on `stream`. Returns TQ_ERR_INVALID_ARG for bad sizes, NULL outputs or misaligned pointers; nothing
 * is launched then. Values at or beyond the fp16 range (|x| >= 65504) are outside the codecs' domain.
 * Codes are undefined there.
 *
 * KIVI 2-bit ([Overview] §KIVI非对称量化):
 *   - Keys are grouped per channel over 16 consecutive tokens; values per token over 16 consecutive
 *     channels.
 *   - Per group: zero z = fp16(min) and scale s = fp16((max - min) / 3), with the difference and
 *     quotient in fp32.
 *   - code = clamp(rint((x - z) * (1/s)), 0, 3), each step in fp32 round-to-nearest-even; code 0 if
 *     s = 0.
 *   - Reconstruction: x_hat = z + code * s.
 *   Layouts, with C = n_heads * head_dim:
 *   - k_codes  uint32 [n_tokens/16][C]: word (g, c) holds tokens 16g..16g+15 of channel c; token 16g+t
 *     is at bits 2t..2t+1.
 *   - k_scale, k_zero  fp16 bits [n_tokens/16][C].
 *   - v_codes  uint32 [n_tokens][C/16]: channel 16j+i is at bits 2i..2i+1 of word (t, j).
 *   - v_scale, v_zero  fp16 bits [n_tokens][C/16].
 *   Requirements:
 *   - head_dim is a multiple of 16. When keys are given, n_tokens is a multiple of 16.
 *   - k and v are 16-byte aligned; k_codes is 8-byte aligned; k_scale, k_zero and v_codes are 4-byte
 *     aligned.
 *   - k or v may be NULL to skip that tensor; its outputs are then unused.
 *   One launch codes both tensors. */
tq_status tq_kivi2_quantize(const void* k, const void* v, int n_tokens, int n_heads, int head_dim,
                            uint32_t* k_codes, uint16_t* k_scale, uint16_t* k_zero, uint32_t* v_codes,
                            uint16_t* v_scale, uint16_t* v_zero, tq_stream_t stream);
/* Inverse of tq_kivi2_quantize. It writes bf16 x_hat = z + code * s (computed in fp32, rounded to
 * nearest even) to k_out and v_out, in the input layout. Either output may be NULL. Alignment is the
 * same as for tq_kivi2_quantize, with k_out and v_out 16-byte aligned. */
tq_status tq_kivi2_dequantize(const uint32_t* k_codes, const uint16_t* k_scale, const uint16_t* k_zero,
                              const uint32_t* v_codes, const uint16_t* v_scale, const uint16_t* v_zero,
                              int n_tokens, int n_heads, int head_dim, void* k_out, void* v_out,
                              tq_stream_t stream);
/* Bonsai 1-bit Q1_0_g128 ([Overview] §Bonsai 1-bit). Each of the n_rows rows (a token's head vector)
 * splits into groups of 128 channels.
 *   - bit = 1 where x >= 0.
 *   - scale = fp16(mean |x|) of the group, the least-squares scale for fixed signs. The sum runs in
 *     fp32 in a fixed order, so it can sit one fp16 ulp from the exact mean.
 *   - Reconstruction: x_hat = +scale or -scale.
 *   Layouts:
 *   - bits  uint32 [n_rows][head_dim/32]: channel 32w+b is at bit b of word w.
 *   - scale  fp16 bits [n_rows][head_dim/128].
 *   Requirements:
 *   - head_dim is a multiple of 128.
 *   - k and v are 16-byte aligned; bits are 4-byte aligned.
 *   - Either input may be NULL.
 *   One launch codes both tensors. The fp16 residual cache of recent tokens that the overview pairs
 *   with this codec is the ring of the hybrid mode above; it is not part of these calls. */
tq_status tq_bonsai1_quantize(const void* k, const void* v, int64_t n_rows, int head_dim, uint32_t* k_bits,
                              uint16_t* k_scale, uint32_t* v_bits, uint16_t* v_scale, tq_stream_t stream);
/* Inverse of tq_bonsai1_quantize: bf16 +-scale per channel into k_out and v_out (16-byte aligned;
 * either may be NULL). */
tq_status tq_bonsai1_dequantize(const uint32_t* k_bits, const uint16_t* k_scale, const uint32_t* v_bits,
                                const uint16_t* v_scale, int64_t n_rows, int head_dim, void* k_out, void* v_out,
                                tq_stream_t stream);

/* Stored K + V bytes of a cache of n_tokens tokens in n_layers layers of n_kv_heads heads under each
 * codec. These are the codes and their parameters only, with no ring and no alignment padding. The
 * rows of the overview's table in §性能表现与实测数据 are:
 *   - FP16: 2 bytes per element.
 *   - KIVI 2-bit: 2 bits plus fp16 scale and zero per 16 elements.
 *   - Bonsai 1-bit: 1 bit plus an fp16 scale per 128 elements.
 * This library's own records are:
 *   - key: d/4 + d/8 + 4 bytes;
 *   - value: d/4 (2-bit) or d/2 (4-bit), plus d/16 bytes.
 * Returns 0 for an unknown codec, bad sizes, or a head_dim that the codec does not accept. */
typedef enum tq_codec {
  TQ_CODEC_FP16 = 0,
  TQ_CODEC_KIVI2 = 1,
  TQ_CODEC_BONSAI1 = 2,
  TQ_CODEC_TQ_K3V2 = 3,
  TQ_CODEC_TQ_K3V4 = 4
} tq_codec;
size_t tq_codec_kv_bytes(int codec, int n_layers, int n_kv_heads, int head_dim, int64_t n_tokens);

/* ---- Host-only inspection helpers (tests and tools; no device work) ---- */

/* Byte offset, inside the cache buffer, of one packed page of (layer, slot, kv_head, page); (size_t)-1
 * for a paged cache (the page's block comes from the device block table). */
size_t tq_page_offset(const tq_ctx* ctx, int layer, int slot, int kv_head, int page);
/* Paged cache: byte offset of the page of (layer, block, kv_head); (size_t)-1 when not paged. */
size_t tq_block_page_offset(const tq_ctx* ctx, int layer, int block, int kv_head);
/* Paged cache: byte offset of the int32 block table [max_seqs][max_pages] inside the cache buffer
 * (tq_cache_bind sets every entry to -1, "no block"); (size_t)-1 when not paged. */
size_t tq_block_table_offset(const tq_ctx* ctx);
/* Byte offsets of the ring K (which = 0) / V (which = 1) block of (layer, slot, kv_head). */
size_t tq_ring_offset(const tq_ctx* ctx, int layer, int slot, int kv_head, int which);
/* Byte offset of the int32 pair {L, F} of (layer, slot), and of the status word. */
size_t tq_state_offset(const tq_ctx* ctx, int layer, int slot);
size_t tq_status_offset(const tq_ctx* ctx);

/* Converts the first n_tokens of one packed page (a host copy of tq_page_bytes bytes) into canonical
 * records ([Guide] §二 step 5 bit packing, little-endian within bytes):
 *   - key record = idx (key_bits - 1 bits/coord, a little-endian bit stream: bit i of coordinate j is bit
 *     (key_bits - 1) j + i of the stream) | QJL sign (1 bit/coord, 1 = projection >= 0) | fp16 n | fp16 gamma;
 *   - value record = codes (value_bits/coord) | fp16 scale per 32 coords.
 * out_keys holds n_tokens * (d*(key_bits-1)/8 + d/8 + 4) bytes; out_values holds n_tokens * (d*vb/8 + d/16). */
tq_status tq_page_to_records(const tq_ctx* ctx, const void* h_page, int n_tokens, uint8_t* out_keys,
                             uint8_t* out_values);
/* Inverse of tq_page_to_records (host): builds a page from canonical records (unused tokens zero). */
tq_status tq_records_to_page(const tq_ctx* ctx, const uint8_t* keys, const uint8_t* values, int n_tokens,
                             void* h_page);

/* Host copies of the tables this context uploaded:
 *   - D: float[d] (+-1);
 *   - S_bf16: uint16[d*d], row-major bf16 bits;
 *   - centroids: double[2^(key_bits-1)] (4 or 8);
 *   - boundaries: double[2^(key_bits-1) - 1] (3 or 7).
 * Any pointer may be NULL. */
tq_status tq_get_tables(const tq_ctx* ctx, float* D, uint16_t* S_bf16, double* centroids, double* boundaries);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
