/*
 * pagedkv.h -- C ABI of the GB300 paged KV cache decode-step library
 * (libpagedkv.so).
 *
 * The library implements the data-parallel hot path of PagedAttention:
 * a host-side block manager (free-block queue, per-block reference counts,
 * per-sequence block tables with #filled, fork / append / free,
 * copy-on-write of shared last blocks) and three sm_103a CUDA kernels that
 * consume its output -- the fused slot write, the fused block copy and
 * single-query paged decode attention with an optional split-context merge.
 *
 * Sources for the operations (pages are cited by title and section):
 *   [review]   "Efficient Memory Management for Large Language Model Serving
 *              with PagedAttention" paper review, mz-moonzoo.tistory.com/116
 *   [tutorial] "KV 캐시 관리와 PagedAttention" (KV cache management and
 *              PagedAttention), llm-systems-engineering.pages.dev/posts/paged-kv-cache
 *   [teardown] vLLM PagedAttention teardown, arcyou.ai/ko/teardowns/vllm-paged-attention
 *   [notes]    PagedAttention notes, unpurerationalist.github.io/posts/2026/11/3919429635
 *
 * Conventions
 *   - Every function returns PA_OK (0) or a PA_ERR_* code; no exception or
 *     longjmp crosses the ABI.  pa_last_error_string() describes the last
 *     failure of the calling thread.
 *   - Host pointers are marked (host), device pointers (device).  The caller
 *     owns every buffer it passes, host or device, and the CUDA stream
 *     (passed as void*, a cudaStream_t; NULL = the legacy default stream).
 *     The library owns only the pa_pool object.
 *   - Device calls validate their scalar arguments and pointer alignment on
 *     the host, then enqueue work on the stream and return; they do not
 *     synchronise.  Problems found by a kernel (a block id or slot outside
 *     the pool, a wait that ran out) are reported through the optional
 *     device status word: the kernel skips the bad access and stores the
 *     error code there if it still holds 0.  The status word is never reset
 *     by the library.
 *   - Host block-manager calls are synchronous and not thread-safe for one
 *     pool; different pools are independent.
 *   - Cache layout, one K and one V array per layer, fp16:
 *       cache[num_blocks][num_heads][block_size][head_dim]
 *     so that one (block, head) pair is block_size*head_dim*2 contiguous
 *     bytes.  New keys / values, queries and outputs are [n][num_heads][head_dim].
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define PA_OK                0
#define PA_ERR_INVALID_ARG   1  /* bad scalar, shape, alignment or capacity    */
#define PA_ERR_OUT_OF_BLOCKS 2  /* free queue cannot cover the request          */
#define PA_ERR_NO_SEQ        3  /* unknown sequence id / id already in use      */
#define PA_ERR_CUDA          4  /* a CUDA runtime call or launch failed         */
#define PA_ERR_TIMEOUT       5  /* (device status) a bounded wait ran out       */
#define PA_ERR_BAD_BLOCK     6  /* (device status) block id / slot outside pool */

#define PA_DTYPE_F16 0

/* Default split-context partition: a context longer than this many tokens
 * is split into partitions of this size whose partial results are merged. */
#define PA_DEFAULT_PARTITION_TOKENS 512

/* Pool geometry, shared by the block manager and the device calls.
 *   num_blocks        physical blocks in the pool (>= 0)
 *   block_size        tokens per block B: 4, 8, 16 or 32 for the device calls
 *                     (any value >= 1 for the host block manager)
 *   num_layers        layers whose caches share the block ids (>= 1)
 *   num_heads         attention heads H (>= 1)
 *   head_dim          D: 8, 16, 32, 64, 128 or 256 for the device calls
 *   dtype             PA_DTYPE_F16 (the only one)
 *   partition_tokens  split-context partition size in tokens; 0 selects
 *                     PA_DEFAULT_PARTITION_TOKENS; otherwise a positive
 *                     multiple of block_size (a value at least as long as
 *                     every context turns the split off)
 *   flags             0 or PA_POOL_PREFIX_CACHING (host block manager only)
 *   free_order        (host, optional) initial order of the free-block queue,
 *                     a permutation of 0..num_blocks-1; NULL = 0,1,2,...
 *                     Read by pa_pool_create only.                          */
typedef struct pa_pool_desc {
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_layers;
    int32_t num_heads;
    int32_t head_dim;
    int32_t dtype;
    int32_t partition_tokens;
    int32_t flags;
    const int32_t *free_order;
} pa_pool_desc;

/* pa_pool_desc.flags */
#define PA_POOL_PREFIX_CACHING 1   /* keep full prompt blocks for reuse (pa_seq_add_tokens) */

typedef struct pa_pool pa_pool;

/* Text of the calling thread's last error ("" if none).  The pointer stays
 * valid until the thread's next failing call. */
const char *pa_last_error_string(void);

/* ---- host block manager ---------------------------------------------------
 * A fixed pool of equal-size physical blocks, sized once at creation; new
 * blocks are taken from the head of a FIFO free queue ([teardown]
 * "PagedAttention" section; [review] §4.2).  Each sequence has a block table
 * mapping its logical blocks to physical blocks; only its last block may be
 * partly filled ([review] §4.3; [notes] §3.3).  Token position p of a sequence
 * is stored in slot  table[p / B] * B + p % B  ([tutorial] Fig. 2). */

/* Create a pool from *desc.  *out receives the handle.
 * Errors: PA_ERR_INVALID_ARG (bad geometry, free_order not a permutation). */
int pa_pool_create(const pa_pool_desc *desc, pa_pool **out);

/* Destroy a pool (NULL is accepted). */
int pa_pool_destroy(pa_pool *pool);

/* Admit sequence seq_id with a prompt of n_tokens tokens: takes
 * ceil(n_tokens / B) blocks from the free queue, in queue order
 * ([review] §4.3, 7-token prompt example; [tutorial] Fig. 1).
 * slots_out (host, optional, n_tokens entries) receives the slot of each
 * prompt token.  All-or-nothing.
 * Errors: PA_ERR_NO_SEQ (id in use), PA_ERR_OUT_OF_BLOCKS, PA_ERR_INVALID_ARG. */
int pa_seq_add(pa_pool *pool, int32_t seq_id, int32_t n_tokens, int64_t *slots_out);

/* Admit a sequence from its prompt's token ids, reusing cached blocks
 * ([teardown] "PagedAttention" section, prefix sharing).  In a pool created
 * with PA_POOL_PREFIX_CACHING every full block of a prompt is keyed by a hash
 * chain over (its parent block's key, its B token ids, extra_key), so a key
 * names the whole prefix up to that block.  The leading full blocks whose
 * keys are cached (checked against the stored tokens, parent key and extra
 * key) are touched instead of allocated: their reference count goes up and a
 * cached block that was free leaves the free queue, no copy.  The scan stops
 * at the first block that is not cached, and never reuses the block holding
 * the last prompt token (a prompt that is all cached still gets that block
 * new, so at least its last token is computed and nothing writes into a
 * shared block).  The remaining blocks come from the
 * free queue, and the new full blocks are cached.  A cached block keeps its
 * key while its count is 0 -- freed blocks join the tail of the free queue,
 * so they are evicted (dropped from the cache) last, least recently freed
 * first -- and loses it when the free queue hands it out again.  Blocks
 * filled by later appends are not cached.
 *   token_ids   (host) n_tokens int32 token ids
 *   extra_key   mixed into every key (requests with different extra keys,
 *               e.g. adapters, never share)
 *   slots_out   (host, optional) slot of every prompt token
 *   n_cached_out (host, optional) leading tokens whose K/V are already in
 *               the cache (reused blocks x B): only the tokens after them need
 *               their K/V written.
 * Without PA_POOL_PREFIX_CACHING this is pa_seq_add (nothing is cached).
 * All-or-nothing.  Errors: PA_ERR_NO_SEQ, PA_ERR_OUT_OF_BLOCKS,
 * PA_ERR_INVALID_ARG.  pa_pool_cached_blocks: blocks currently cached. */
int pa_seq_add_tokens(pa_pool *pool, int32_t seq_id, int32_t n_tokens, const int32_t *token_ids,
                      int64_t extra_key, int64_t *slots_out, int32_t *n_cached_out);
int pa_pool_cached_blocks(const pa_pool *pool, int32_t *n_cached);

/* fork: the child gets a copy of the parent's block table and length, and
 * every block's reference count goes up by one ([notes] §4.2 fork;
 * [review] §5 "Fork").  Errors: PA_ERR_NO_SEQ (no parent / child exists). */
int pa_seq_fork(pa_pool *pool, int32_t parent, int32_t child);

/* free: every block of the sequence loses one reference; a block whose count
 * reaches 0 goes to the tail of the free queue.  Blocks are released from the
 * sequence's last block backwards ([tutorial] "returning blocks after a
 * request ends"; [notes] §3.4.2, §4.2; [teardown] tail blocks go first).
 * Errors: PA_ERR_NO_SEQ. */
int pa_seq_free(pa_pool *pool, int32_t seq_id);

/* Batched fork and free for beam search ([notes] §3.4.2: beams fork at
 * every step and pruned beams release their blocks): the same operations as
 * pa_seq_fork / pa_seq_free, applied in order; pa_seq_fork_batch's parents
 * may be children created earlier in the same call.  Every argument is
 * checked before anything changes.  Errors: PA_ERR_NO_SEQ,
 * PA_ERR_INVALID_ARG. */
int pa_seq_fork_batch(pa_pool *pool, int32_t n, const int32_t *parents, const int32_t *children);
int pa_seq_free_batch(pa_pool *pool, int32_t n, const int32_t *seq_ids);

/* One pruning step of beam search for n_groups groups of `width` beams
 * ([notes] §3.4.2: beams fork where a candidate is kept several times and
 * pruned beams drop their references; [review] §4.4 (2)).  beams (host,
 * n_groups x width int32, in/out) holds each group's beam sequence ids;
 * counts (host, n_groups x width int32) how many of the group's `width`
 * survivors each beam is (each row sums to width).  Per group, in order:
 * every surviving beam keeps its id and is forked count - 1 times into new
 * ids *next_id, *next_id + 1, ... (pa_seq_fork), placed right after it;
 * beams with count 0 are freed, in beam order (pa_seq_free).  The group's
 * new ids are written back into its row of beams and *next_id advances.
 * Everything is checked before anything changes.  Errors: PA_ERR_NO_SEQ (a
 * beam does not exist or a new id is in use), PA_ERR_INVALID_ARG (a row
 * that does not sum to width, a beam listed twice, a negative count). */
int pa_beam_prune(pa_pool *pool, int32_t n_groups, int32_t width, int32_t *beams,
                  const int32_t *counts, int32_t *next_id);

/* append, for a batch: one new token for each of seq_ids[0..n_seqs), handled
 * in the order given ([review] §4.3 steps 1-2; [tutorial] Fig. 3, Fig. 6):
 *   - no block yet, or the last block is full (shared or not): take a new
 *     block from the free queue and append it to the table (no copy);
 *   - last block partly filled and shared (count > 1): copy-on-write -- take
 *     a new block, emit the pair (old, new) to copies_out, decrement the old
 *     block's count and point the table's last entry at the new block;
 *   - otherwise write in place.
 * The token's slot goes to slot_mapping_out[i] (host, n_seqs entries).
 * copies_out (host, copies_cap x 2 int32: src, dst) receives the block copies
 * that must run (pa_copy_blocks) before the slot write (pa_write_kv);
 * *n_copies_out their number.  A sequence may appear once per call.
 * All-or-nothing: on PA_ERR_OUT_OF_BLOCKS (the queue cannot cover every new
 * block) or a too-small copies_cap (PA_ERR_INVALID_ARG) nothing changes
 * ([teardown]: allocate_slots reports failure, which the scheduler answers by
 * preempting).  Errors: PA_ERR_NO_SEQ, PA_ERR_INVALID_ARG, PA_ERR_OUT_OF_BLOCKS. */
int pa_alloc_slots(pa_pool *pool, int32_t n_seqs, const int32_t *seq_ids,
                   int64_t *slot_mapping_out, int32_t *copies_out, int32_t copies_cap,
                   int32_t *n_copies_out);

/* One decode step's host work for a batch, in one call: pa_alloc_slots
 * for seq_ids (one new token each, copy-on-write pairs to copies_out), then
 * the batch's block tables and context lengths as pa_get_block_tables
 * exports them, after the append ([review] §4.3 decoding: the block manager
 * maps each new token to a slot; §4.6: the scheduler hands the block tables
 * to the workers).  Written for a serving loop that stages these arrays in
 * page-locked host memory and uploads them with one copy:
 *   slot_mapping_out (host, n_seqs int64), ctx_lens_out (host, n_seqs int32),
 *   tables_out (host, n_seqs x max_blocks int32, padded with -1),
 *   copies_out (host, copies_cap x 2 int32), *n_copies_out.
 * All-or-nothing: also fails with no change when a table would grow beyond
 * max_blocks (PA_ERR_INVALID_ARG).  Errors: as pa_alloc_slots. */
int pa_decode_step_prepare(pa_pool *pool, int32_t n_seqs, const int32_t *seq_ids,
                           int32_t max_blocks, int64_t *slot_mapping_out, int32_t *ctx_lens_out,
                           int32_t *tables_out, int32_t *copies_out, int32_t copies_cap,
                           int32_t *n_copies_out);

/* pa_decode_step_prepare for a staging buffer that a serving loop reuses
 * step after step: the outputs and their meaning are the same, but row i of
 * tables_out is written only when sequence seq_ids[i]'s block table changed
 * since this call last wrote that row.  row_versions (host, n_seqs uint64,
 * owned by the caller) records what each row holds: zero it before the first
 * call, and keep one such array per tables_out buffer and max_blocks (reset
 * it to zero when either changes, or when anything else writes tables_out).
 * A table changes when its sequence is added, forked, moved between pools,
 * or takes a new or copied block; in a decode step that is about one
 * sequence in B, so most rows are left as they are.  Table versions are
 * unique in the process, so a row never matches another sequence or pool.
 * Errors: as pa_decode_step_prepare; PA_ERR_INVALID_ARG for a NULL
 * row_versions when rows are to be written. */
int pa_decode_step_prepare_rows(pa_pool *pool, int32_t n_seqs, const int32_t *seq_ids,
                                int32_t max_blocks, int64_t *slot_mapping_out,
                                int32_t *ctx_lens_out, int32_t *tables_out,
                                uint64_t *row_versions, int32_t *copies_out, int32_t copies_cap,
                                int32_t *n_copies_out);

/* Swapping ([review] §4.5 (1) swapping; [notes] §3.5 Swapping, CPU block
 * manager): a preempted group of sequences moves, all its blocks at once,
 * from the GPU pool to a second pool that manages swap space in host memory,
 * and later back (pa_swap_out from gpu to cpu, pa_swap_in from cpu to gpu;
 * the two pools must have the same block size).  The group must hold every
 * reference to its blocks ([review] §4.5 (2): sequences that share blocks
 * are evicted together); each distinct block gets one block of the target
 * pool (with the same reference count), the sequences' tables are rewritten
 * to the new ids, and the source blocks return to their free queue, the
 * last-used first.  pairs_out (host, pairs_cap x 2 int32) receives the
 * (source block, target block) pairs in first-use order -- the copies that
 * pa_swap_blocks must perform.  All-or-nothing.
 * Errors: PA_ERR_NO_SEQ, PA_ERR_OUT_OF_BLOCKS (target pool full),
 * PA_ERR_INVALID_ARG (a block shared outside the group, small pairs_cap,
 * different block sizes). */
int pa_swap_out(pa_pool *gpu, pa_pool *cpu, int32_t n_seqs, const int32_t *seq_ids,
                int32_t *pairs_out, int32_t pairs_cap, int32_t *n_pairs_out);
int pa_swap_in(pa_pool *cpu, pa_pool *gpu, int32_t n_seqs, const int32_t *seq_ids,
               int32_t *pairs_out, int32_t pairs_cap, int32_t *n_pairs_out);

/* append, several tokens per sequence (chunked prefill, [review] §4.3 "all
 * tokens of the step are concatenated"; [teardown] chunked prefill): like
 * pa_alloc_slots with counts[i] >= 0 new tokens for seq_ids[i] -- the first
 * may copy a shared, partly filled last block (copy-on-write), the tokens
 * fill the last block's free slots and then take new blocks in queue order.
 * slot_mapping_out (host, sum(counts) int64) gets the slots sequence by
 * sequence, in the order given.  All-or-nothing.  Errors: as pa_alloc_slots. */
int pa_alloc_slots_n(pa_pool *pool, int32_t n_seqs, const int32_t *seq_ids,
                     const int32_t *counts, int64_t *slot_mapping_out, int32_t *copies_out,
                     int32_t copies_cap, int32_t *n_copies_out);

/* Export block tables and context lengths for a batch, in the layout the
 * attention kernel reads: tables_out (host, n_seqs x max_blocks int32,
 * row-major) gets each sequence's physical block ids, padded with -1;
 * ctx_lens_out (host, n_seqs int32) gets each sequence's token count.
 * Errors: PA_ERR_NO_SEQ, PA_ERR_INVALID_ARG (a table longer than max_blocks;
 * the outputs are then unspecified). */
int pa_get_block_tables(const pa_pool *pool, int32_t n_seqs, const int32_t *seq_ids,
                        int32_t max_blocks, int32_t *tables_out, int32_t *ctx_lens_out);

/* Introspection.  pa_seq_info: token count and table length of a sequence.
 * pa_pool_num_free: blocks in the free queue.  pa_pool_free_queue: the
 * queue from head to tail into out (host, cap entries), *n_out = its length
 * (PA_ERR_INVALID_ARG if cap is too small).  pa_pool_refcounts: every
 * block's reference count into out (host, num_blocks entries). */
int pa_seq_info(const pa_pool *pool, int32_t seq_id, int32_t *num_tokens, int32_t *num_blocks);
int pa_pool_num_free(const pa_pool *pool, int32_t *n_free);
int pa_pool_free_queue(const pa_pool *pool, int32_t *out, int32_t cap, int32_t *n_out);
int pa_pool_refcounts(const pa_pool *pool, int32_t *out);

/* ---- device kernels -------------------------------------------------------
 * All pointers below are device pointers unless marked (host).  Tensors must
 * be contiguous and 16-byte aligned; desc supplies the geometry (its
 * free_order is ignored).  status (device, optional, one int32) receives the
 * first error a kernel detects; NULL disables reporting but not the checks. */

/* Fused reshape and block write ([review] §5.1 (1); [notes] §4.1): for every
 * token t < n_tokens and head h,
 *     k_cache[slot / B][h][slot % B][:] = k[t][h][:],  same for v,
 * with slot = slot_mapping[t] (int64).  A negative slot skips the token;
 * a slot >= num_blocks * B is skipped and reported as PA_ERR_BAD_BLOCK.
 * k, v: [n_tokens][num_heads][head_dim] fp16.  One layer per call.
 * Errors: PA_ERR_INVALID_ARG, PA_ERR_CUDA. */
int pa_write_kv(const void *k, const void *v, const int64_t *slot_mapping, int32_t n_tokens,
                void *k_cache, void *v_cache, const pa_pool_desc *desc,
                int32_t *status, void *stream);

/* Fused block copy for copy-on-write ([review] §5.1 (3); [notes] §4.1): for
 * every pair (src, dst) in pairs (device, n_pairs x 2 int32) and every layer
 * l < num_layers, block dst of k_caches[l] and v_caches[l] becomes a copy of
 * block src, in one launch.  k_caches / v_caches are (host) arrays of
 * num_layers device pointers (num_layers <= 128).  The destinations must be
 * distinct and no destination may be the source of another pair (true of the
 * pairs pa_alloc_slots emits: every destination is a newly taken block).
 * Pairs outside the pool are skipped and reported as PA_ERR_BAD_BLOCK.
 * Errors: PA_ERR_INVALID_ARG, PA_ERR_CUDA. */
int pa_copy_blocks(void *const *k_caches, void *const *v_caches, int32_t num_layers,
                   const int32_t *pairs, int32_t n_pairs, const pa_pool_desc *desc,
                   int32_t *status, void *stream);

/* Block copies between two cache sets (swap out / swap in, [review] §5.1 (3)
 * fused block copy): for every pair (a, b) in pairs (device-accessible,
 * n_pairs x 2 int32) and every layer, block b of dst_k[l] / dst_v[l] becomes
 * a copy of block a of src_k[l] / src_v[l], in one launch.  The caches are
 * device memory or page-locked host memory mapped into the device's address
 * space (e.g. swap space in Grace memory, reached over NVLink-C2C); src and
 * dst hold src_num_blocks / dst_num_blocks blocks of the layout above.
 * Pairs outside either pool are skipped and reported as PA_ERR_BAD_BLOCK.
 * num_layers <= 128.  Errors: PA_ERR_INVALID_ARG, PA_ERR_CUDA. */
int pa_swap_blocks(const void *const *src_k, const void *const *src_v, int32_t src_num_blocks,
                   void *const *dst_k, void *const *dst_v, int32_t dst_num_blocks,
                   int32_t num_layers, const int32_t *pairs, int32_t n_pairs,
                   const pa_pool_desc *desc, int32_t *status, void *stream);

/* Bytes of device workspace pa_decode_attention needs for a batch of n_seqs
 * sequences whose tables have max_blocks columns: 256 bytes of scheduling
 * state, plus room for the partial results of split contexts when a context
 * can be longer than one partition.  0 for an empty batch. */
size_t pa_decode_workspace_bytes(int32_t n_seqs, int32_t max_blocks, const pa_pool_desc *desc);

/* Single-query paged decode attention ([notes] §3.1 blockwise attention
 * equation; [review] §4.1 and §5.1 (2); [tutorial] Fig. 4): for every
 * sequence s < n_seqs and head h,
 *     o[s][h] = sum_{p < ctx} softmax_p(scale * q[s][h] . k_p) v_p,
 * where k_p, v_p are read from physical block block_tables[s][p / B] at
 * offset p % B and ctx = ctx_lens[s] counts every stored token of the
 * sequence, the one written in this step included.  Slots past ctx are never
 * used.  ctx <= 0 gives o = 0; a ctx above max_blocks * B is reported as
 * PA_ERR_BAD_BLOCK and its output left unwritten.  Contexts longer than
 * partition_tokens are
 * split into partitions whose partial (max, sum, unnormalised output) go to
 * the workspace and are merged by a second kernel; results agree with the
 * unsplit sum to rounding.
 *   out, q        [n_seqs][num_heads][head_dim] fp16
 *   k_cache, v_cache  one layer, layout above
 *   block_tables  [n_seqs][max_blocks] int32 (entries past ceil(ctx/B) unread)
 *   ctx_lens      [n_seqs] int32, each <= max_blocks * B
 *   workspace     >= pa_decode_workspace_bytes(n_seqs, max_blocks, desc)
 *                 bytes, 256-byte aligned (may be NULL when that is 0); its
 *                 contents need no initialisation and are not preserved (the
 *                 call clears its scheduling word on the stream first).  Two
 *                 calls must not use one workspace concurrently.
 * Errors: PA_ERR_INVALID_ARG, PA_ERR_CUDA. */
int pa_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, const int32_t *ctx_lens, int32_t n_seqs,
                        int32_t max_blocks, float scale, void *workspace, size_t workspace_bytes,
                        int32_t *status, const pa_pool_desc *desc, void *stream);

/* One decode step's slot write and attention in one call ([review] §5.1 (1)
 * fused reshape and block write; §4.3 decoding): for every sequence s <
 * n_seqs, the step's new key and value rows k_new[s], v_new[s] (device,
 * [n_seqs][num_heads][head_dim] fp16, 16-byte aligned) are stored at
 * slot_mapping[s] (device, n_seqs int64, the slot pa_alloc_slots /
 * pa_decode_step_prepare returned for the token), exactly as pa_write_kv
 * with one token per sequence, and then attention runs as
 * pa_decode_attention (same arguments and workspace), the new token
 * included.  Where the persistent decode kernel runs (batches whose
 * per-sequence plan fits its shared memory) the write happens inside it: the
 * unit that reads a sequence's last context block first stores the new rows
 * into it, so the step takes one launch fewer; otherwise the slot write runs
 * as its own launch first, on the same stream.
 * slot_mapping[s] must be the slot of position ctx_lens[s] - 1 (the token
 * just appended); the in-kernel write checks it against the block table and
 * reports PA_ERR_INVALID_ARG in *status (writing nothing) when it is not.  A
 * negative slot skips the sequence's write, as in pa_write_kv.
 * Errors: as pa_decode_attention; PA_ERR_INVALID_ARG also for NULL or
 * misaligned k_new, v_new or slot_mapping. */
int pa_decode_step_attention(void *out, const void *q, const void *k_new, const void *v_new,
                             const int64_t *slot_mapping, void *k_cache, void *v_cache,
                             const int32_t *block_tables, const int32_t *ctx_lens, int32_t n_seqs,
                             int32_t max_blocks, float scale, void *workspace,
                             size_t workspace_bytes, int32_t *status, const pa_pool_desc *desc,
                             void *stream);

/* Causal paged prefill attention ([review] §4.3, the prompt phase: the
 * prompt's tokens are processed together, each attending to the tokens
 * before it and itself; [notes] §3.1 blockwise attention equation, applied
 * to each of those queries).  Sequence s < n_seqs has
 * q_len = q_starts[s+1] - q_starts[s] queries, rows q_starts[s] .. of q, and
 * a context of ctx = ctx_lens[s] stored tokens that includes the queries' own
 * tokens (written beforehand with pa_write_kv).  Row q_starts[s] + i is the
 * query at position p = ctx - q_len + i and, for every head h,
 *     out[row][h] = sum_{j <= p} softmax_j(scale * q[row][h] . k_j) v_j,
 * with k_j, v_j read through block_tables[s] as in pa_decode_attention.
 * q_len == ctx is a whole prompt; q_len < ctx continues a sequence whose
 * first ctx - q_len tokens are already cached (a later chunk of a long
 * prompt, or a prompt whose leading blocks came from the prefix cache).
 * q_len == 1 is a decode query.
 *   out, q        [q_rows][num_heads][head_dim] fp16, 16-byte aligned like
 *                 the caches; every sequence's rows lie in [0, q_rows)
 *   block_tables  [n_seqs][max_blocks] int32 (entries past ceil(ctx/B) unread)
 *   ctx_lens      [n_seqs] int32
 *   q_starts      [n_seqs + 1] int32, non-decreasing
 *   max_q_len     host bound on every q_len (sizes the launch)
 *   q_rows        rows of q and out (0: nothing to do)
 *   scale         finite and > 0 (1/sqrt(head_dim) in the pages)
 * head_dim 64 or 128, block_size 4..32.  Tensor cores: fp16 products, fp32
 * accumulation; the probabilities (at most 2^8 after a lazy rescale of the
 * running maximum) enter the second product as fp16, whose rounding stays
 * below the fp16 rounding of the output.
 * Device-side problems go to *status and leave that sequence's rows
 * unwritten: PA_ERR_INVALID_ARG for q_len < 0, q_len > ctx,
 * q_len > max_q_len or rows outside [0, q_rows); PA_ERR_BAD_BLOCK for
 * ctx > max_blocks * B or a table entry outside the pool (that entry is not
 * read and the sequence's output is unspecified).
 * Work is balanced across the GPU through a unit counter in the library's
 * device memory that each launch sets back to zero when it ends; calls take
 * the library's 64 counters in turn, so up to 64 calls may be in flight at
 * once on different streams (a captured call replayed from a CUDA graph
 * reuses its counter, which its previous replay left at zero).
 * Errors: PA_ERR_INVALID_ARG (geometry, sizes, NULL or misaligned
 * pointers), PA_ERR_CUDA. */
int pa_prefill_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *ctx_lens,
                         const int32_t *q_starts, int32_t n_seqs, int32_t max_blocks,
                         int32_t max_q_len, int32_t q_rows, float scale, int32_t *status,
                         const pa_pool_desc *desc, void *stream);

/* The prompt phase's slot write and causal prefill attention in one call,
 * for whole prompts ([review] §4.3 prompt phase; §5.1 (1) fused reshape and
 * block write): every sequence s must have q_len == ctx_lens[s] (its
 * prompt, with blocks already allocated through pa_seq_add /
 * pa_alloc_slots_n), and k_new, v_new (device, [q_rows][num_heads][head_dim]
 * fp16, 16-byte aligned, finite) hold its keys and values on the same rows as
 * q.  The result is that of pa_write_kv of those rows into the prompts'
 * slots (positions 0 .. q_len - 1 through block_tables) followed by
 * pa_prefill_attention; the kernel reads the keys and values from k_new and
 * v_new (once per query-tile pair, no read back from the cache) and the unit
 * that reaches a prompt's last key stores every key tile's blocks into the
 * cache as it goes.  block_size 8, 16 or 32; other arguments and errors as
 * pa_prefill_attention; a sequence with q_len != ctx is reported as
 * PA_ERR_INVALID_ARG in *status (that sequence is neither written nor
 * attended). */
int pa_prefill_step_attention(void *out, const void *q, const void *k_new, const void *v_new,
                              void *k_cache, void *v_cache, const int32_t *block_tables,
                              const int32_t *ctx_lens, const int32_t *q_starts, int32_t n_seqs,
                              int32_t max_blocks, int32_t max_q_len, int32_t q_rows, float scale,
                              int32_t *status, const pa_pool_desc *desc, void *stream);

/* ---- decode attention without a caller-provided workspace ------------------
 * No counterpart on the pages: this entry point exists for callers that
 * cannot allocate device memory when they run attention -- for instance a
 * runtime that reserves all device memory up front and gives its kernels no
 * allocator, or a plugin host that forbids cudaMalloc (an allocation can
 * fail or synchronise the device) once serving has started.
 *
 * Same arguments and result as pa_decode_attention, minus the workspace: the
 * library uses a fixed scratch area of PA_NOALLOC_SCRATCH_BYTES compiled into
 * it as a static device array.  Every GPU on which the library is loaded
 * holds that array until the process exits.  The call allocates nothing
 * (no cudaMalloc / cudaFree or allocating library routine); it clears the
 * scratch's scheduling word on the stream itself.
 *
 *   - Every argument is checked before any CUDA call; a batch whose
 *     pa_decode_workspace_bytes(n_seqs, max_blocks, desc) exceeds
 *     PA_NOALLOC_SCRATCH_BYTES is rejected with PA_ERR_INVALID_ARG.
 *   - The first call on a device looks up the scratch's device address
 *     (cudaGetSymbolAddress, with that device current, which may load the
 *     library's device code); make that first call before any stream
 *     capture on the device.  A first call whose stream is being captured
 *     is refused with PA_ERR_INVALID_ARG before the lookup; a lookup that
 *     fails (PA_ERR_CUDA) is tried again by the next call.
 *   - All calls share the one scratch area, which keeps the last call's
 *     contents: calls whose work overlaps on the GPU (different streams,
 *     threads or processes sharing the context, without ordering between
 *     them) race and give wrong results.  Order them, e.g. on one stream.
 * Errors: as pa_decode_attention, plus PA_ERR_INVALID_ARG for a batch too
 * large for the scratch and PA_ERR_CUDA if the scratch address lookup fails. */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)

int pa_decode_attention_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *block_tables, const int32_t *ctx_lens,
                                int32_t n_seqs, int32_t max_blocks, float scale,
                                int32_t *status, const pa_pool_desc *desc, void *stream);

/* Diagnostic for the bounded waits that every kernel of this library uses
 * (no counterpart on the pages).  Launches one thread on `stream` that
 * waits, through the library's bounded wait, for an mbarrier phase that
 * nothing completes; the wait gives up after its limit (200 ms) and the
 * thread writes PA_ERR_TIMEOUT into *status, as a kernel whose producer
 * never arrives would.  Nothing faults and the context stays usable.
 *   status  device int32, caller-owned; reads PA_ERR_TIMEOUT once the
 *           stream has completed the call.
 * Errors: PA_ERR_INVALID_ARG for a NULL status (nothing launched);
 * PA_ERR_CUDA if the launch fails. */
int pa_selftest_bounded_wait(int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
