/*
 * pagedkv.h — C ABI of the GB300 (sm_103a) paged KV-cache decode library.
 *
 * What the library computes comes from four web pages on vLLM's PagedAttention:
 *   [HowVLLM]   "How vLLM gets real throughput on H100s: PagedAttention and
 *               continuous batching explained"
 *   [DeepDive]  "High-Throughput LLM Inference & Training: A Deep Dive into vLLM"
 *               (single paragraph; Figures 1 and 2; the KV-footprint equation)
 *   [ArchBench] "vLLM architecture, memory and benchmarks deep dive"
 *   [Dissect]   "Dissecting vLLM: How PagedAttention and Continuous Batching
 *               Maximize Throughput"
 *
 * The KV cache of every layer is a pool of fixed-size physical blocks of
 * B = 16 or 32 tokens ([HowVLLM] "PagedAttention borrows from operating
 * systems"; [ArchBench] "PagedAttention: a 1960s idea for modern GPUs"). Each
 * sequence owns a block table: logical block i of the sequence lives in
 * physical block block_tables[s][i]. The decode kernel walks that table and
 * gathers K/V from the scattered blocks ([Dissect] "PagedAttention: Virtual
 * Memory for KV Cache", last paragraph).
 *
 * Cache layout (the pages only say that the kernel assumes one fixed layout,
 * [Dissect] "A Balanced Take: The Sharp Edges"; this is the one used here):
 *   k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim],
 *                      row-major; element type bf16 (2 bytes) or OCP FP8 E4M3
 *                      (1 byte). One (block, head) page is one contiguous run
 *                      of block_size*head_dim elements.
 *   q, out           : [num_seqs][num_heads][head_dim] bf16.
 *                      Query head j reads KV head j / (num_heads/num_kv_heads).
 *   block_tables     : int32 [num_seqs][max_blocks_per_seq]; entries past
 *                      ceil(context_len/block_size) are never read.
 *   context_lens     : int32 [num_seqs], number of cached tokens to attend to
 *                      (the token written this step included).
 *   slot_mapping     : int64 [num_tokens], slot = block*block_size + offset;
 *                      -1 means "skip this token".
 *
 * Conventions shared by every entry point:
 *   - Pointers named as "device" must point to device memory (any allocator);
 *     the library never allocates or frees device memory and never keeps a
 *     pointer after the call returns.
 *   - Device buffers must be 16-byte aligned (q, out, k, v, caches, workspace);
 *     a misaligned pointer returns PKV_ERR_INVALID_ARG.
 *   - Every launch is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). PKV_OK means "validated and enqueued". A launch failure
 *     returns PKV_ERR_CUDA. Faults inside a kernel surface at the caller's
 *     next synchronisation. The decode and merge kernels are launched as
 *     programmatic dependents of the work before them on the stream: their
 *     CTAs may be scheduled early, but they wait for that work to complete
 *     before reading global memory, so stream order holds as usual.
 *   - Kernels check every block id and slot they dereference. An out-of-range
 *     id is skipped (the affected output is unspecified) and, if a device
 *     error word was registered with pkv_set_device_check, an error code is
 *     written there. Every wait inside a kernel is bounded; a wait that runs
 *     out also sets the error word and the kernel returns normally.
 *   - No function throws, prints or aborts. Functions are re-entrant except the
 *     allocator, whose handle must have one owner at a time.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, bad size or shape   */
  PKV_ERR_UNSUPPORTED = -2,   /* shape outside the supported set (see below)  */
  PKV_ERR_CUDA = -3,          /* a CUDA runtime call failed                   */
  PKV_ERR_OUT_OF_BLOCKS = -4, /* allocator: free pool exhausted (state kept)  */
  PKV_ERR_NOT_FOUND = -5,     /* allocator: unknown sequence id               */
  PKV_ERR_DEVICE_CHECK = -6   /* a kernel reported a bad id or a timed-out wait */
} pkv_status;

typedef enum { PKV_DTYPE_BF16 = 0, PKV_DTYPE_FP8_E4M3 = 1 } pkv_dtype;

/* Device error codes written into the registered error word (first error wins). */
#define PKV_DEVERR_NONE 0
#define PKV_DEVERR_BLOCK_ID 1    /* block table entry outside [0, num_blocks) */
#define PKV_DEVERR_SLOT 2        /* slot_mapping entry outside the pool       */
#define PKV_DEVERR_WAIT_TIMEOUT 3 /* a bounded barrier wait gave up           */
#define PKV_DEVERR_CONTEXT 4     /* context_len outside [0, max_blocks_per_seq*block_size],
                                    or longer than the call's context bound */
#define PKV_DEVERR_ORDER 5       /* seq_order entry outside [0, num_seqs)      */

/* Geometry of one layer's K and V pools (both share it). */
typedef struct {
  int num_blocks;   /* physical blocks in the pool                     */
  int block_size;   /* tokens per block: 16 or 32                      */
  int num_kv_heads; /* KV heads                                        */
  int head_dim;     /* 128 or 256                                      */
  int dtype;        /* pkv_dtype                                       */
} pkv_cache_desc;

/* Supported shapes: head_dim in {128, 256}; block_size in {16, 32};
 * num_heads / num_kv_heads (the GQA group) in [1, 8]; Q and out bf16. */

/* ------------------------------------------------------------------------ *
 * kv_cache_write: store this step's new K/V into their slots.
 *
 * Blocks are filled only as tokens are produced ([HowVLLM] "PagedAttention
 * borrows from operating systems"; [ArchBench] "PagedAttention: a 1960s
 * idea for modern GPUs"), so every decode step scatters one K and one V row
 * per sequence into the slot the allocator handed out.
 *
 *   k, v         : device bf16 [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping : device int64 [num_tokens]; -1 skips the token
 *   k_cache, v_cache : device pools described by `cache`
 *   k_scale, v_scale : device fp32 [num_kv_heads], FP8 pools only (else NULL).
 *     FP8 code = round-to-nearest-even, saturating to +-448, of the fp32
 *     quotient x / scale[h] (IEEE division), OCP E4M3.
 * For bf16 pools the copy is bit-exact.
 * Errors: PKV_ERR_INVALID_ARG (null pointers, num_tokens < 0, misaligned),
 * PKV_ERR_UNSUPPORTED (shape), PKV_ERR_CUDA. num_tokens == 0 is a no-op.
 * ------------------------------------------------------------------------ */
int pkv_kv_cache_write(const void* k, const void* v, const int64_t* slot_mapping,
                       int num_tokens, void* k_cache, void* v_cache,
                       pkv_cache_desc cache, const float* k_scale,
                       const float* v_scale, void* stream);

/* ------------------------------------------------------------------------ *
 * paged_attention_decode: one query token per sequence, grouped-query
 * attention over the paged cache ([Dissect] "PagedAttention: Virtual Memory
 * for KV Cache"; decode as the bandwidth-bound phase: [HowVLLM] "Decode is a
 * memory problem, not a math problem").
 *
 * For sequence s and query head j (KV head h = j / g, g = num_heads /
 * num_kv_heads), with K_s, V_s the sequence's logical rows 0..ctx-1:
 *     z_t = scale * <q[s,j,:], K_s[t,:]>,  out[s,j,:] = sum_t softmax(z)_t V_s[t,:]
 * FP8 pools dequantise as code * k_scale[h] (resp. v_scale[h]).
 * The softmax is the max-subtracted one, accumulated online in fp32.
 *
 *   out       : device bf16 [num_seqs][num_heads][head_dim] (written when
 *               partition_size == 0; untouched otherwise)
 *   q         : device bf16 [num_seqs][num_heads][head_dim]
 *   block_tables : device int32 [num_seqs][max_blocks_per_seq]
 *   context_lens : device int32 [num_seqs]; a context of 0 yields zeros
 *   max_context  : host upper bound of context_lens (sizes the grid)
 *   scale        : logit scale, normally 1/sqrt(head_dim)
 *   partition_size : 0 = one pass: the result goes to `out` directly (the
 *               library spreads each sequence over a thread-block cluster of up
 *               to 8 CTAs and merges their softmax states on chip; no
 *               workspace). Otherwise a multiple of block_size: the context is cut
 *               into partitions [p*P, (p+1)*P) starting at token 0, and each
 *               partition's (max, sum, normalised output) is written to
 *               `workspace`; pkv_paged_attention_reduce then merges them.
 *   workspace, workspace_bytes : device scratch for the split form, at least
 *               pkv_decode_workspace_bytes(...) bytes (ignored when
 *               partition_size == 0; may be NULL then).
 *   seq_order : NULL, or device int32 [num_seqs], a permutation of
 *               0..num_seqs-1: the order in which the kernel's CTAs take the
 *               sequences (the grid's first CTAs work on seq_order[0]). Every
 *               order gives the same bits; only the schedule changes. With
 *               contexts of very different lengths, longest first
 *               (pkv_longest_first_order) starts the long sequences while
 *               the short ones fill in behind them, instead of leaving a long
 *               one to run alone at the end of the grid. An entry outside
 *               [0, num_seqs) is reported as PKV_DEVERR_ORDER and its CTAs
 *               do nothing; a sequence that no entry names (because of such
 *               an entry or a repeated one) is not decoded, and its result
 *               is undefined (the split form's merge still combines that
 *               row's workspace slots).
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 * ------------------------------------------------------------------------ */
size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                  int max_context, int partition_size);

/* Host helper: a split size near partition_size without a nearly empty last
 * partition. With n = max(1, round(max_context / partition_size)) (halves
 * round up), the result is the smallest multiple of block_size that covers
 * max_context in n partitions, so the longest context takes n partitions of
 * about equal length instead of, e.g., two full ones and a few-token third
 * (1033 tokens at P = 512, B = 16: 528, two partitions). It equals
 * partition_size whenever partition_size divides max_context. Any result is
 * a valid partition_size for the calls above (size the workspace with it).
 * Returns partition_size if max_context <= 0, PKV_ERR_INVALID_ARG if
 * block_size <= 0 or partition_size is not a positive multiple of it. (The
 * pages leave the split size open; this is a load-balancing choice.) */
int pkv_split_partition_size(int max_context, int block_size, int partition_size);

/* Host helper: order[0..n) = the indices 0..n-1 sorted by lengths[i], longest
 * first, equal lengths in index order (a stable sort), for the seq_order
 * arguments below. lengths and order are host arrays of n int32.
 * Returns PKV_OK; PKV_ERR_INVALID_ARG if n < 0 or (n > 0 and a pointer is
 * NULL). */
int pkv_longest_first_order(const int32_t* lengths, int n, int32_t* order);

int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                               const void* v_cache, pkv_cache_desc cache,
                               const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs,
                               int num_heads, int max_context, float scale,
                               int partition_size, void* workspace,
                               size_t workspace_bytes, const int32_t* seq_order,
                               void* stream);

/* ------------------------------------------------------------------------ *
 * paged_attention_reduce: merge the per-partition partials of a split decode.
 * With m_p, l_p the partition's running max and exp-sum and o_p its
 * normalised output, M = max_p m_p, w_p = l_p * exp(m_p - M):
 *     out = sum_p (w_p / sum_q w_q) * o_p          over p < ceil(ctx / P).
 * One partition reproduces o_0 exactly. The split form is not described on
 * the pages; it is the log-sum-exp merge that makes the split result equal
 * to the one-pass softmax.
 *
 *   out       : device bf16 [num_seqs][num_heads][head_dim]
 *   workspace : the same buffer the split decode wrote
 *   other args: as passed to the split decode
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 * ------------------------------------------------------------------------ */
int pkv_paged_attention_reduce(void* out, const void* workspace,
                               size_t workspace_bytes,
                               const int32_t* context_lens, int num_seqs,
                               int num_heads, int head_dim, int max_context,
                               int partition_size, void* stream);

/* ------------------------------------------------------------------------ *
 * paged_attention: the decode attention of one step in one call, the result
 * in `out`: pkv_paged_attention_decode, then (partition_size > 0)
 * pkv_paged_attention_reduce on the same workspace, both on `stream`.
 * Arguments as for pkv_paged_attention_decode; `out` is always written.
 * Errors: those of the two calls (the merge is not launched after a failed
 * decode).
 * ------------------------------------------------------------------------ */
int pkv_paged_attention(void* out, const void* q, const void* k_cache,
                        const void* v_cache, pkv_cache_desc cache,
                        const float* k_scale, const float* v_scale,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* context_lens, int num_seqs, int num_heads,
                        int max_context, float scale, int partition_size,
                        void* workspace, size_t workspace_bytes, const int32_t* seq_order,
                        void* stream);

/* ------------------------------------------------------------------------ *
 * paged_attention_decode_shared_prefix: decode for groups of sequences that
 * share a prompt's physical blocks (rollouts forked from one prompt,
 * [HowVLLM] "PagedAttention borrows from operating systems"; [Dissect]
 * "PagedAttention: Virtual Memory for KV Cache"). The result is the same
 * attention as pkv_paged_attention_decode; the shared pages are read once per
 * group (per row tile of a large group, below) instead of once per member.
 *
 *   group_start   : device int32 [num_groups + 1]; group i is the sequences
 *                   [group_start[i], group_start[i+1]) of the batch;
 *                   sequences outside every group are fine
 *   max_group_members : host bound on the members of any group (>= 1 when
 *                   num_groups > 0, <= num_seqs). A group's query rows
 *                   (members x g) are covered by tiles of floor(128/g)
 *                   members; every tile reads the shared pages (adjacent
 *                   tiles of a partition run together, so the second read
 *                   of a page is served by L2). A group larger than the
 *                   bound is reported as PKV_DEVERR_CONTEXT and its uncovered
 *                   members get their result without the shared part.
 *   prefix_blocks : device int32 [num_seqs]; the number of leading blocks of
 *                   each sequence that are its group's shared prefix: the same
 *                   value and the same physical ids for every member, full
 *                   blocks only, prefix_blocks[s]*block_size <= context_lens[s];
 *                   0 for a sequence outside every group
 *   max_prefix_blocks : host upper bound of prefix_blocks
 *   max_own_context : host upper bound of each sequence's own part,
 *                   context_lens[s] - prefix_blocks[s]*block_size (the whole
 *                   context for a sequence outside every group); it sizes the
 *                   own-part grid and slots, so a tight bound saves launching
 *                   CTAs with no page (a longer own part is reported as
 *                   PKV_DEVERR_CONTEXT and cut); the other arguments as for
 *                   pkv_paged_attention_decode
 *   partition_size: split size P of each member's own part (multiple of
 *                   block_size, at most 2048 blocks); the shared part uses
 *                   partitions of Pp tokens, a power-of-two multiple of P
 *                   chosen for the current device (the smallest for which the
 *                   prefix grid fits the SM count, at most 2048 blocks):
 *                   pkv_shared_prefix_partition_size returns it
 *   workspace     : at least pkv_shared_prefix_workspace_bytes(...) bytes.
 *                   Layout (fp32), with NPP = ceil(max_prefix_blocks *
 *                   block_size / Pp), NPS = ceil(max_own_context / P),
 *                   NPT = NPP + NPS and R = num_seqs * num_heads rows:
 *                   tmp_out [R][NPT][head_dim] | max_logits [R][NPT] |
 *                   exp_sums [R][NPT]. Slot p < NPP of a row holds the shared
 *                   partition p (tokens [p*Pp, min((p+1)*Pp, prefix tokens))),
 *                   slot NPP + p the own partition p (tokens from
 *                   prefix_blocks[s]*block_size + p*P on), in the form of
 *                   pkv_paged_attention_decode's partials.
 *   k_scale, v_scale : device fp32 [num_kv_heads] dequantisation scales of
 *                   an E4M3 pool (required then, else ignored), as for
 *                   pkv_paged_attention_decode
 *   seq_order     : NULL or a permutation of the sequences, the order in
 *                   which the own-block decode takes them, as for
 *                   pkv_paged_attention_decode (there, longest own part
 *                   first: pkv_longest_first_order of context_lens[s] -
 *                   prefix_blocks[s]*block_size)
 * Per group, KV head and row tile, a kernel computes partials of the members'
 * query heads over the shared pages (the members' queries form the rows of
 * one tensor-core product; for E4M3 pools the codes are turned into exact f16
 * operands in shared memory and P is one f16 part); each member's own blocks
 * go through the split decode; the merge combines both.
 * ------------------------------------------------------------------------ */
size_t pkv_shared_prefix_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                         int max_own_context, int max_prefix_tokens,
                                         int partition_size);
/* Pp, the shared part's partition size that
 * pkv_paged_attention_decode_shared_prefix uses on the current device for
 * these arguments (> 0), or a negative pkv_status. */
int pkv_shared_prefix_partition_size(int num_groups, int max_group_members, int num_kv_heads,
                                     int num_heads, int block_size, int max_prefix_blocks,
                                     int partition_size);
int pkv_paged_attention_decode_shared_prefix(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    pkv_cache_desc cache, const float* k_scale, const float* v_scale,
    const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int num_seqs, int num_heads, int max_own_context,
    float scale, const int32_t* group_start, int num_groups, int max_group_members,
    const int32_t* prefix_blocks, int max_prefix_blocks, int partition_size,
    void* workspace, size_t workspace_bytes, const int32_t* seq_order, void* stream);

/* ------------------------------------------------------------------------ *
 * copy_blocks: copy-on-write duplication. Sequences forked from one prompt
 * share its physical blocks; a block is cloned only when a sibling is about
 * to write into it ([HowVLLM] "PagedAttention borrows from operating
 * systems"; [ArchBench] "PagedAttention: a 1960s idea for modern GPUs";
 * [Dissect] "PagedAttention: Virtual Memory for KV Cache").
 * For every pair (src, dst): k_cache[dst] = k_cache[src] and
 * v_cache[dst] = v_cache[src], all heads, byte for byte.
 *
 *   block_pairs : device int32 [num_pairs][2] = {src, dst}
 * Destinations must be distinct and must not appear as a source of another
 * pair in the same call (the allocator guarantees this).
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA.
 * num_pairs == 0 is a no-op.
 * ------------------------------------------------------------------------ */
int pkv_copy_blocks(void* k_cache, void* v_cache, pkv_cache_desc cache,
                    const int32_t* block_pairs, int num_pairs, void* stream);

/* ------------------------------------------------------------------------ *
 * paged_attention_decode_noalloc: split decode + merge that allocates
 * nothing. (The pages have no counterpart; this is a service for callers.)
 *
 * For callers that cannot call cudaMalloc or provide a workspace: code
 * running inside a framework that owns the whole device-memory budget and
 * forbids allocations outside its arena, C callers without a device
 * allocator, and latency-critical paths where an allocation (which can
 * synchronise the device) is not acceptable. The per-partition partials go
 * to a fixed array of PKV_NOALLOC_SCRATCH_BYTES bytes of device memory that
 * belongs to the library; every GPU that loads this part of the library
 * holds that array until the process exits.
 *
 * Arguments and result are those of pkv_paged_attention_decode with
 * partition_size > 0 (and seq_order NULL) followed by
 * pkv_paged_attention_reduce: `out` receives the merged bf16 output. The
 * caller still passes every input and output.
 *   - Returns PKV_ERR_UNSUPPORTED when the partials,
 *     pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context,
 *     partition_size), exceed PKV_NOALLOC_SCRATCH_BYTES (use a larger
 *     partition_size or the workspace form), PKV_ERR_INVALID_ARG for
 *     partition_size <= 0, and every error of the two calls it makes.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it per device and context (a new
 *     context on the device, e.g. after cudaDeviceReset, looks it up again);
 *     make that first call before any stream capture.
 *   - All calls in the process share the one array and it keeps the last
 *     call's contents; nothing in it needs to start at zero. Calls whose
 *     kernels may overlap on the GPU (other streams, other host threads)
 *     race on it: serialise them.
 * ------------------------------------------------------------------------ */
#define PKV_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

int pkv_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, pkv_cache_desc cache,
                                       const float* k_scale, const float* v_scale,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, int num_seqs,
                                       int num_heads, int max_context, float scale,
                                       int partition_size, void* stream);

/* ------------------------------------------------------------------------ *
 * swap_out / swap_in: move whole blocks (K and V, all heads) between a pool
 * and a packed buffer, for preemption by swapping ([Dissect] "Continuous
 * Batching: Breaking the Sequence Barrier" and "FAQ": a running sequence's
 * blocks go to CPU RAM, the device blocks are freed, and they come back
 * later).
 *
 *   blocks  : int32 [n] block ids, readable by the device (device memory or
 *             pinned host memory)
 *   k_buf, v_buf : [n][num_kv_heads*block_size*head_dim*esz] bytes, block i of
 *             the list at row i; device memory or pinned host memory the device
 *             can address (the kernel reads/writes it directly)
 * swap_out: buf[i] = pool[blocks[i]]; swap_in: pool[blocks[i]] = buf[i]
 * (byte for byte). The allocator side (freeing a sequence, re-creating it
 * with fresh blocks on the way back) is the caller's.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA; n == 0 is a
 * no-op. Out-of-range ids are skipped and reported.
 * ------------------------------------------------------------------------ */
int pkv_swap_out(const void* k_cache, const void* v_cache, pkv_cache_desc cache,
                 const int32_t* blocks, int num_blocks_to_move, void* k_buf, void* v_buf,
                 void* stream);
int pkv_swap_in(void* k_cache, void* v_cache, pkv_cache_desc cache, const int32_t* blocks,
                int num_blocks_to_move, const void* k_buf, const void* v_buf, void* stream);

/* Register a device int32 that kernels write a PKV_DEVERR_* code into (first
 * error wins; the caller clears it). NULL switches reporting off; the kernels
 * still skip out-of-range ids. Process-wide; returns PKV_OK. */
int pkv_set_device_check(int* dev_error_flag);

/* Failure-detection self-test: launches one kernel whose barrier wait can never
 * complete; the bounded wait gives up after limit_us microseconds (1..2e6),
 * writes PKV_DEVERR_WAIT_TIMEOUT into *dev_error_flag (device int32, first
 * error wins) and the kernel returns, leaving the context usable. Every wait
 * in the library's kernels is bounded the same way (2 s). */
int pkv_selftest_wait_timeout(int* dev_error_flag, int limit_us, void* stream);

/* Static description of a status code. Never NULL. */
const char* pkv_status_string(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int pkv_version(void);

/* ------------------------------------------------------------------------ *
 * Host block allocator ([HowVLLM] "PagedAttention borrows from operating
 * systems" and "Continuous batching removes straggler bubbles"; [ArchBench]
 * "PagedAttention: a 1960s idea for modern GPUs"; [Dissect] "PagedAttention:
 * Virtual Memory for KV Cache"; [DeepDive] Figures 1 and 2).
 *
 * - Free list: at creation the pool's block ids are shuffled with a seeded
 *   Fisher-Yates (std::mt19937_64); blocks are popped from and pushed back to
 *   the same end (last freed, first reused).
 * - A sequence holds exactly ceil(len / block_size) blocks: a block is taken
 *   only when the previous one is full.
 * - fork gives the child the parent's table and adds one reference to each
 *   block; no device work happens.
 * - append of a token into a block whose reference count is > 1 takes a fresh
 *   block, emits the pair (old, new) for pkv_copy_blocks and drops one
 *   reference from the old block (copy-on-write). A holder that finds the
 *   count at 1 writes in place.
 * - free drops one reference from each block; blocks that reach 0 go back to
 *   the free list.
 * All calls are O(blocks touched). A failing call leaves the state unchanged.
 * The handle is not thread-safe.
 * ------------------------------------------------------------------------ */
typedef struct pkv_allocator pkv_allocator;

int pkv_alloc_create(int num_blocks, int block_size, uint64_t seed,
                     pkv_allocator** out);
void pkv_alloc_destroy(pkv_allocator* a);
/* New empty sequence; its id is written to *seq_id. */
int pkv_seq_new(pkv_allocator* a, int* seq_id);
/* New sequence sharing every block of `parent`. */
int pkv_seq_fork(pkv_allocator* a, int parent, int* child);
/* Reserve n_tokens new slots at the end of `seq`.
 *   slots_out     : host int64 [n_tokens], the slot of each new token
 *   cow_pairs_out : host int32 [n_tokens][2] (may be NULL if the caller knows
 *                   no block is shared); receives the (src, dst) pairs
 *   n_cow         : number of pairs written (NULL allowed when cow_pairs_out
 *                   is NULL)
 * PKV_ERR_OUT_OF_BLOCKS if the pool cannot hold the new tokens (nothing is
 * changed); PKV_ERR_INVALID_ARG if a shared block must be cloned but
 * cow_pairs_out is NULL. */
int pkv_seq_append(pkv_allocator* a, int seq, int n_tokens, int64_t* slots_out,
                   int32_t* cow_pairs_out, int* n_cow);
/* Release the sequence and its references. */
int pkv_seq_free(pkv_allocator* a, int seq);
/* Copy the sequence's block table into out[0..cap); *n_blocks = its length.
 * Returns PKV_ERR_INVALID_ARG if cap is too small (nothing written). */
int pkv_seq_block_table(const pkv_allocator* a, int seq, int32_t* out, int cap,
                        int* n_blocks);
int pkv_seq_len(const pkv_allocator* a, int seq, int* len);
/* Reference count of one physical block (0 = free). */
int pkv_block_refcount(const pkv_allocator* a, int block, int* refcount);
/* free_blocks + used_blocks == num_blocks; used_slots = sum of live lengths
 * counted once per physical slot (shared slots count once). */
int pkv_alloc_stats(const pkv_allocator* a, int* free_blocks, int* used_blocks,
                    long long* used_slots);
/* Checkpoint / resume of the allocator (the pages have no counterpart; with
 * pkv_swap_out of the used blocks it saves a whole cache state, e.g. before
 * moving a batch off the GPU). pkv_alloc_save writes the complete state (free
 * list order, refcounts, fill, every sequence's table and length, next id)
 * as a flat record of *n bytes into buf (host memory, cap bytes); with buf
 * NULL it only reports *n. pkv_alloc_load creates an allocator from such a
 * record; it checks the record against itself (sizes, ranges, each block
 * free exactly once or held by exactly refcount tables) and returns
 * PKV_ERR_INVALID_ARG, creating nothing, on any mismatch. */
int pkv_alloc_save(const pkv_allocator* a, void* buf, size_t cap, size_t* n);
int pkv_alloc_load(const void* buf, size_t n, pkv_allocator** out);

/* ------------------------------------------------------------------------ *
 * Iteration-level (continuous) batching scheduler over an allocator
 * ([HowVLLM] "Continuous batching removes straggler bubbles"; [Dissect]
 * "Continuous Batching: Breaking the Sequence Barrier"; [ArchBench]
 * "Continuous batching and the straggler problem").
 *
 * A request is (id, prompt length, token budget); it ends (EOS) when it has
 * produced max_new_tokens tokens. pkv_sched_step runs one iteration:
 *   1. eject the requests that produced their last token in the previous
 *      iteration; their blocks return to the free list at once;
 *   2. admit waiting requests in arrival order while the batch has fewer than
 *      max_num_seqs requests and the free blocks cover the prompt and its first
 *      new token on top of what the running requests need this iteration
 *      (the prompt slots are reported: the caller stores the prompt's K/V);
 *   3. give every running request one slot for this iteration's token; if the
 *      pool runs dry, the most recently admitted request is preempted (freed
 *      and put back at the head of the queue, to be recomputed).
 * Swap mode (pkv_sched_set_preemption(s, PKV_PREEMPT_SWAP); [Dissect]
 * "Continuous Batching: Breaking the Sequence Barrier" and "FAQ": preempted
 * sequences' blocks go to CPU RAM): a preempted request keeps its progress;
 * its block list is reported (event 3, pkv_sched_swap_blocks) and the caller
 * copies those blocks out (pkv_swap_out) before anything is written in this
 * iteration, since the blocks are already free. Swapped requests are resumed
 * first, before step 2, when the free blocks cover their length plus one
 * token: fresh blocks for the whole length are reported (event 4,
 * pkv_sched_swap_blocks) and the caller copies the saved blocks back
 * (pkv_swap_in) before this iteration's writes. Nothing is recomputed.
 * After a step, the running batch (admission order) is read with
 * pkv_sched_running / pkv_sched_block_tables; context_len counts the token of
 * this iteration. The scheduler uses the allocator through its public calls;
 * neither is thread-safe.
 * ------------------------------------------------------------------------ */
typedef struct pkv_scheduler pkv_scheduler;

int pkv_sched_create(pkv_allocator* alloc, int block_size, int max_num_seqs,
                     pkv_scheduler** out);
void pkv_sched_destroy(pkv_scheduler* s);
int pkv_sched_add_request(pkv_scheduler* s, int64_t request_id, int prompt_len,
                          int max_new_tokens);
/* A request for n sampled continuations of one prompt (n = 1: the call
 * above). It is admitted as a unit once the batch has room for n rows and
 * the free blocks cover the prompt plus one block per sample: the prompt is
 * stored once (its slots reported under request_id) and n - 1 forks share
 * its blocks ([HowVLLM] "PagedAttention borrows from operating systems";
 * [Dissect] "PagedAttention: Virtual Memory for KV Cache": copy-on-write
 * among sequences of one prompt). The samples run as requests request_id,
 * request_id + 1, ..., request_id + n - 1;
 * each has the token budget max_new_tokens. A sample that writes into a block
 * still shared gets a copy (pkv_sched_cow_pairs). A preempted sample comes
 * back as a request of its own (recompute: from the prompt; swap: its blocks,
 * shared ones included, are copied out and back into private blocks).
 * PKV_ERR_INVALID_ARG if n < 1 or n > max_num_seqs, if request_id < 0, or if
 * any id in [request_id, request_id + n) belongs to a request that is
 * waiting (with its samples' ids), running or swapped out (ids of finished
 * requests may be reused); the same check applies to
 * pkv_sched_add_request. */
int pkv_sched_add_request_n(pkv_scheduler* s, int64_t request_id, int prompt_len,
                            int max_new_tokens, int n);
/* One iteration; reports the batch size, the requests admitted in it and
 * those ejected at its start. */
int pkv_sched_step(pkv_scheduler* s, int* num_running, int* num_admitted,
                   int* num_finished);
/* Running batch: request ids, context lengths and the slot of this
 * iteration's token, each [cap >= num_running] (any may be NULL). */
int pkv_sched_running(const pkv_scheduler* s, int64_t* request_ids,
                      int32_t* context_lens, int64_t* new_slots, int cap);
/* Block tables of the running batch, [rows >= num_running][max_blocks],
 * padded with -1. PKV_ERR_INVALID_ARG if a table is longer than max_blocks. */
int pkv_sched_block_tables(const pkv_scheduler* s, int32_t* tables, int max_blocks,
                           int rows);
/* Prompt slots of a request admitted in the last step (n = prompt length). */
int pkv_sched_prompt_slots(const pkv_scheduler* s, int64_t request_id,
                           int64_t* slots, int cap, int* n);
/* Ids of the last step's events: kind 0 admitted, 1 finished, 2 preempted,
 * 3 swapped out, 4 swapped in (resumed). A request resumed and preempted
 * again in the same step appears in neither 3 nor 4 (its saved copy stays
 * valid). */
int pkv_sched_events(const pkv_scheduler* s, int kind, int64_t* ids, int cap, int* n);
/* Copy-on-write pairs (src, dst) of the last step, host int32 [n][2]: blocks
 * still shared with other samples that a sample cloned to write this
 * iteration's token. Within an iteration the caller applies, in this order:
 * swap-outs (events 3), swap-ins (events 4), the admitted prompts' K/V,
 * pkv_copy_blocks of these pairs, this iteration's K/V (pkv_kv_cache_write),
 * then the decode. n = 0 when no block was shared. PKV_ERR_INVALID_ARG if cap
 * is below n (n is still reported). */
int pkv_sched_cow_pairs(const pkv_scheduler* s, int32_t* pairs, int cap, int* n);
/* waiting counts queued and swapped-out requests. */
int pkv_sched_counts(const pkv_scheduler* s, int* waiting, int* running,
                     long long* steps);

#define PKV_PREEMPT_RECOMPUTE 0
#define PKV_PREEMPT_SWAP 1
/* Preemption policy (default PKV_PREEMPT_RECOMPUTE). */
int pkv_sched_set_preemption(pkv_scheduler* s, int mode);
#define PKV_BATCH_ADMISSION 0
#define PKV_BATCH_LONGEST_FIRST 1
/* Row order of the batch reported by pkv_sched_running and
 * pkv_sched_block_tables (the same order in both): PKV_BATCH_ADMISSION
 * (default) or PKV_BATCH_LONGEST_FIRST, by decreasing context length, ties in
 * admission order. (The pages have no counterpart; a split decode launches a
 * batch's rows in order, and longest first its tail is shortest: a batch of
 * 256 lengths log-uniform in [16, 16384] took 0.3416 ms in arrival order and
 * 0.3355 ms longest first on GB300.) Preemption still takes the most recently
 * admitted request. PKV_ERR_INVALID_ARG for another value. */
int pkv_sched_set_batch_order(pkv_scheduler* s, int order);
/* Block list (logical order) of a request swapped out or in during the last
 * step: the blocks to copy to host memory, or the fresh blocks to copy back
 * into. n = number of blocks; PKV_ERR_NOT_FOUND for any other request. */
int pkv_sched_swap_blocks(const pkv_scheduler* s, int64_t request_id, int32_t* blocks,
                          int cap, int* n);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
