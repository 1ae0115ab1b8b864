/*
 * kshipra.h -- C ABI of the GB300 (sm_103a) paged GQA attention library.
 *
 * The operations follow the pages "Building Kshipra" part 3 (kshipra-3):
 *  - section 1 "Block-Arena KV Cache": keys and values live in one arena of
 *    fixed-size blocks reserved once; nothing is allocated per token.  KV
 *    bytes per token = 2 x layers x KV heads x head dim x bytes per element.
 *  - section 4 "Chunked Prefill": attention runs an online softmax (running
 *    max, running sum, rescaled accumulator) across KV blocks read in place
 *    from the arena, with no gather copy; RoPE uses absolute positions (a
 *    chunk after P cached tokens starts at position P); the causal mask lets
 *    each query see the cached prefix and the earlier tokens of its chunk.
 *  - section 3 "Radix-Tree Prefix Cache": several block tables may name the
 *    same physical blocks (shared prefixes); the kernels only read them.
 *  - section 5 "Continuous Batching": one call may mix prefill chunks and
 *    single-token decodes.
 *
 * Conventions for every entry point
 *  - Pointers documented as "device" are CUDA device pointers owned by the
 *    caller; the library never frees or keeps them past the call.  Pointers
 *    documented as "host" are ordinary host memory.
 *  - Calls that take a `stream` (a cudaStream_t passed as void*; NULL is the
 *    legacy default stream) only enqueue work on it and return without
 *    waiting, except kshipra_device_status, which waits for that stream.
 *  - The library allocates no memory per call.  Scratch space is the
 *    caller's `workspace`.
 *  - The return value is a status code: KSHIPRA_OK or one of the errors
 *    below.  Host-side checks run before anything is enqueued, so a call that
 *    returns an argument error has touched no device memory.
 *    kshipra_last_error() gives a one-line description of the last error
 *    raised on the calling thread.
 *  - Facts held only in device arrays (block ids inside [0, num_blocks),
 *    positions consistent with context lengths, num_tokens ==
 *    query_start_loc[num_seqs]) cannot be checked on the host.  They are
 *    preconditions; kernels that meet a violation skip the offending access,
 *    never trap, and set a bit in the device status word read by
 *    kshipra_device_status.
 *
 * Layouts (element type `dtype`: 0 = IEEE binary16, 1 = bfloat16)
 *  - token rows q, k, v, q_rot, out: [num_tokens][heads][head_dim], tokens of
 *    sequence s contiguous in query_start_loc order.
 *  - arena: k_arena and v_arena are each [num_blocks][num_kv_heads]
 *    [block_size][head_dim]; slot p % block_size of logical block
 *    p / block_size holds position p.
 *  - block_tables: int32 [num_seqs][max_blocks_per_seq]; entry j of row s is
 *    the physical block holding logical block j of sequence s.  Entries past
 *    ceil(context_len / block_size) are never read.
 *  - query q head h uses kv head h / (num_q_heads / num_kv_heads).
 *
 * Supported shapes: head_dim 64 or 128; block_size 16 or 32; num_q_heads /
 * num_kv_heads in {1, 2, 4, 8, 16}; dtype 0 or 1.
 */
#ifndef KSHIPRA_H
#define KSHIPRA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define KSHIPRA_OK 0
#define KSHIPRA_ERR_INVALID_ARG 1        /* null pointer, negative size, heads not divisible */
#define KSHIPRA_ERR_UNSUPPORTED 2        /* head_dim, block_size, group size or dtype not built */
#define KSHIPRA_ERR_WORKSPACE_TOO_SMALL 3
#define KSHIPRA_ERR_CUDA 4               /* a CUDA call failed; see kshipra_last_error() */
#define KSHIPRA_ERR_OUT_OF_BLOCKS 5      /* the block pool has fewer free blocks than requested */

/* ---- device status word bits (kshipra_device_status) ----------------- */
#define KSHIPRA_DEV_BAD_BLOCK_ID 0x1     /* a block-table entry outside [0, num_blocks) */
#define KSHIPRA_DEV_BAD_POSITION 0x2     /* a position outside [0, rope_max_pos) or past the table */
#define KSHIPRA_DEV_BAD_LENGTHS 0x4      /* context/query lengths inconsistent with the arguments */
#define KSHIPRA_DEV_TIMEOUT 0x8          /* a bounded wait inside a kernel gave up */

#define KSHIPRA_DTYPE_F16 0
#define KSHIPRA_DTYPE_BF16 1

/* ---- options (kshipra_set_option) ------------------------------------ */
/* Options belong to the calling host thread (each thread starts with the
 * defaults): a call uses the settings of the thread that makes it, so a
 * workspace size queried on a thread fits that thread's later calls, and
 * threads that set different values never affect each other. */
/* Keys per decode split (0 = automatic).  Nonzero values must be multiples
 * of 64.  Affects the workspace size. */
#define KSHIPRA_OPT_SPLIT_TOKENS 0
/* A sequence whose query_len x group size is at most this many rows runs on
 * the split-KV decode kernel, all others on the tensor-core prefill kernel.
 * 0..16, default 16; 0 sends every sequence to the prefill kernel. */
#define KSHIPRA_OPT_DECODE_MAX_ROWS 1

/*
 * KV bytes one token occupies across all layers:
 *   2 (K and V) x num_layers x num_kv_heads x head_dim x element size.
 * (kshipra-3, section 1: 128 KiB per token for 32 layers, 8 KV heads, head
 * dim 128, FP16.)  Host only.  Returns 0 for a non-positive argument or an
 * unknown dtype.
 */
size_t kshipra_kv_bytes_per_token(int num_layers, int num_kv_heads, int head_dim, int dtype);

/*
 * RoPE table on the host: host_out[p][i][0] = cos(p * theta^(-2i/d)),
 * host_out[p][i][1] = sin(...), for p < max_pos, i < head_dim / 2
 * (rotate-half convention: element i pairs with i + d/2).  The angle, cos and
 * sin are evaluated in float64 and each entry is rounded once to float32.
 * (kshipra-3, section 4: RoPE uses absolute positions.)  The caller copies it
 * to the device once and passes that copy to kshipra_kv_append_rope.
 * host_out must hold max_pos * head_dim floats.  Host only, no CUDA calls.
 * Errors: INVALID_ARG (null, max_pos < 0, head_dim odd or < 2, theta <= 0).
 */
int kshipra_rope_table_build(float* host_out, int max_pos, int head_dim, double theta);

/*
 * RoPE and append (kshipra-3, sections 1 and 4).  For every token t of
 * sequence s (query_start_loc[s] <= t < query_start_loc[s+1]) at position
 * p = positions[t]:
 *   - q_rot[t][h] = RoPE(q[t][h], p) for every q head (skipped when q and
 *     q_rot are both NULL, e.g. when filling a cached prefix);
 *   - k_arena[b][h][p % block_size] = RoPE(k[t][h], p) and
 *     v_arena[b][h][p % block_size] = v[t][h] for every kv head, where
 *     b = block_tables[s][p / block_size].
 * The rotation is computed in float32 from rope_table (two separately
 * rounded products, then one rounded add or subtract; no fused multiply-add)
 * and rounded once to dtype (nearest, ties to even), so the arena contents
 * are reproducible bit for bit.  V rows are copied bit for
 * bit.  q_rot may alias q.  Other arena slots are not touched.
 *
 * q, q_rot [num_tokens][num_q_heads][head_dim]; k, v [num_tokens]
 * [num_kv_heads][head_dim]; k_arena, v_arena, block_tables, query_start_loc
 * [num_seqs + 1], positions [num_tokens], rope_table [rope_max_pos]
 * [head_dim/2][2] float32: all device pointers.
 * Device-side violations: a block id outside [0, num_blocks), a logical block
 * index >= max_blocks_per_seq or a position outside [0, rope_max_pos) skip
 * that token's writes and set KSHIPRA_DEV_BAD_BLOCK_ID / _BAD_POSITION.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA.  num_tokens == 0 is a no-op.
 */
int kshipra_kv_append_rope(const void* q, const void* k, const void* v, void* q_rot, void* k_arena,
                           void* v_arena, const int32_t* block_tables, const int32_t* query_start_loc,
                           const int32_t* positions, const float* rope_table, int rope_max_pos, int num_seqs,
                           int num_tokens, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int max_blocks_per_seq, int num_blocks, int dtype, void* stream);

/* ---------------------------------------------------------------------------
 * Block management (kshipra-3, section 1: the arena is reserved once and a
 * LIFO free list hands blocks out and takes them back; section 3: reference
 * counts keep shared prefix blocks alive and a block is copied before a
 * request that diverges inside it writes it; section 5: a preempted
 * sequence's blocks are swapped out of the arena and restored later).
 *
 * The pool is host state (thread-safe); it decides block ids and never
 * touches device memory.  The move calls below do the device side.
 */
typedef struct kshipra_block_pool kshipra_block_pool;

/* A pool over blocks 0 .. num_blocks-1, all free.  The free list starts as
 * 0, 1, ..., num_blocks-1 and allocation takes from its end, so the first
 * allocation returns num_blocks-1.  Errors: INVALID_ARG. */
int kshipra_block_pool_create(int num_blocks, kshipra_block_pool** pool_out);
void kshipra_block_pool_destroy(kshipra_block_pool* pool);
/* Free blocks, or -1 for a NULL pool. */
int kshipra_block_pool_num_free(kshipra_block_pool* pool);
/* n blocks into ids_out (host array), each with reference count 1, taken
 * from the end of the free list (the most recently released first).  All or
 * nothing.  Errors: INVALID_ARG, OUT_OF_BLOCKS. */
int kshipra_block_alloc(kshipra_block_pool* pool, int n, int32_t* ids_out);
/* One more reference to each listed (allocated) block: another sequence maps
 * it, e.g. a shared prefix.  Errors: INVALID_ARG (a block not allocated). */
int kshipra_block_share(kshipra_block_pool* pool, const int32_t* ids, int n);
/* Drops one reference per listed block, in order; a block whose count
 * reaches 0 goes to the end of the free list (the next allocation reuses it).
 * Nothing changes if any entry would drop below 0.  Errors: INVALID_ARG. */
int kshipra_block_release(kshipra_block_pool* pool, const int32_t* ids, int n);
/* Reference count of one block (0 = free), or -1 for a bad id / NULL pool. */
int kshipra_block_refcount(kshipra_block_pool* pool, int id);
/* Before writing into block *id_inout: if it is shared (count > 1), takes a
 * fresh block for the writer, drops the writer's reference to the shared
 * one, stores the fresh id in *id_inout and the shared id in *copy_from_out
 * (the caller then copies the block with kshipra_blocks_copy); if it is
 * private, *copy_from_out = -1 and nothing changes.
 * Errors: INVALID_ARG, OUT_OF_BLOCKS. */
int kshipra_block_make_private(kshipra_block_pool* pool, int32_t* id_inout, int32_t* copy_from_out);

/* Device side, asynchronous on `stream`; arenas as for the attention calls
 * ([num_blocks][num_kv_heads][block_size][head_dim], K and V), ids are device
 * int32 arrays of n entries.  Ids outside the arena are reported through the
 * device status word (KSHIPRA_DEV_BAD_BLOCK_ID) and skipped.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
/* Copies block src_ids[i] to block dst_ids[i] (all kv heads, K and V) within
 * the arena.  The copies run in no fixed order, so the destination ids must
 * be distinct and no destination may also be a source (a block copied while
 * it is overwritten gives either content); the lists are device memory and
 * are not checked. */
int kshipra_blocks_copy(void* k_arena, void* v_arena, const int32_t* src_ids, const int32_t* dst_ids, int n,
                        int num_kv_heads, int block_size, int head_dim, int num_blocks, int dtype, void* stream);
/* Gathers blocks ids[0..n) into k_out, v_out [n][num_kv_heads][block_size]
 * [head_dim]: device memory or pinned host memory (written over the CPU-GPU
 * link, no staging copy). */
int kshipra_blocks_swap_out(void* k_out, void* v_out, const void* k_arena, const void* v_arena, const int32_t* ids,
                            int n, int num_kv_heads, int block_size, int head_dim, int num_blocks, int dtype,
                            void* stream);
/* Scatters k_in, v_in [n][num_kv_heads][block_size][head_dim] (device or
 * pinned host memory) into blocks ids[0..n) of the arena. */
int kshipra_blocks_swap_in(void* k_arena, void* v_arena, const void* k_in, const void* v_in, const int32_t* ids,
                           int n, int num_kv_heads, int block_size, int head_dim, int num_blocks, int dtype,
                           void* stream);

/* ---------------------------------------------------------------------------
 * Radix-tree prefix cache (kshipra-3, section 3): cached KV blocks form a tree
 * whose edges are blocks of block_size tokens; a request walks it from the
 * root and reuses every matching block; under memory pressure the least
 * recently used leaf is evicted, looked up again after each eviction so that
 * a parent left without children is considered too.
 *
 * Host state (thread-safe) over a block pool, which must outlive the cache.
 * The tree holds one pool reference to each block it caches.  Recency is a
 * logical clock that advances once per match or insert and stamps every node
 * the call walks; ties in recency (and in the partial match below) go to the
 * smaller block id.
 */
typedef struct kshipra_prefix_cache kshipra_prefix_cache;

/* An empty cache over `pool` for blocks of block_size tokens.
 * Errors: INVALID_ARG. */
int kshipra_prefix_cache_create(kshipra_block_pool* pool, int block_size, kshipra_prefix_cache** cache_out);
/* Drops the tree's references (blocks nobody else holds return to the pool's
 * free list) and frees the cache. */
void kshipra_prefix_cache_destroy(kshipra_prefix_cache* cache);
/* The longest cached prefix of tokens[0..num_tokens): full blocks while one
 * matches, then, if tokens remain and no full block matches them, the child
 * sharing the longest run of leading tokens with the rest.  Writes the
 * matched blocks to blocks_out (host array of max_blocks >=
 * ceil(num_tokens / block_size) entries), their number to *num_blocks_out and
 * the matched token count to *num_matched_out; the caller gets one reference
 * to each returned block.  When *num_matched_out is not a multiple of
 * block_size, the last block is shared and only partly the caller's: it must
 * go through kshipra_block_make_private (and kshipra_blocks_copy) before the
 * caller writes slot *num_matched_out % block_size.  Errors: INVALID_ARG. */
int kshipra_prefix_cache_match(kshipra_prefix_cache* cache, const int32_t* tokens, int num_tokens,
                               int32_t* blocks_out, int max_blocks, int* num_blocks_out, int* num_matched_out);
/* Caches the full blocks of a computed sequence: block j of tokens (tokens
 * [j * block_size, (j + 1) * block_size)) lives in blocks[j], for j <
 * num_tokens / block_size (num_blocks may be larger; the partial tail is not
 * cached).  Where the same tokens are cached already under the same parent,
 * the cached block stays and blocks[j] is not added.  Each added block gets
 * the tree's reference; *num_added_out (may be NULL) is their number.  All or
 * nothing.  Errors: INVALID_ARG (too few ids, an added block not allocated,
 * cached elsewhere already, or listed twice). */
int kshipra_prefix_cache_insert(kshipra_prefix_cache* cache, const int32_t* tokens, int num_tokens,
                                const int32_t* blocks, int num_blocks, int* num_added_out);
/* Frees up to num_blocks blocks: repeatedly removes the least recently used
 * leaf whose block only the tree holds and drops that reference.  Stops early
 * when nothing is evictable; *num_freed_out (may be NULL) is the count.
 * Errors: INVALID_ARG. */
int kshipra_prefix_cache_evict(kshipra_prefix_cache* cache, int num_blocks, int* num_freed_out);
/* Blocks evict() could free now, cascades included: nodes whose whole
 * subtree only the tree holds (the "evictable" term of section 5's admission
 * test, free + evictable >= reserved + needed).  -1 for a NULL cache. */
int kshipra_prefix_cache_evictable(kshipra_prefix_cache* cache);
/* Cached blocks (tree nodes), or -1 for a NULL cache. */
int kshipra_prefix_cache_num_nodes(kshipra_prefix_cache* cache);

/*
 * Bytes of device workspace kshipra_paged_attention needs for these sizes,
 * written to *bytes_out (host pointer).  sm_count is the number of SMs of the
 * device the call will run on (0 = ask the current device, which needs a
 * CUDA device).  The result depends on KSHIPRA_OPT_SPLIT_TOKENS.
 * Errors: INVALID_ARG, CUDA (sm_count == 0 and no device).
 */
int kshipra_paged_attention_workspace_size(int num_seqs, int num_tokens, int max_context_len, int num_q_heads,
                                           int num_kv_heads, int head_dim, int sm_count, size_t* bytes_out);

/*
 * Paged GQA attention over the arena (kshipra-3, section 4; mixed batches,
 * section 5).  For every query token t of sequence s at position
 * p = positions[t] and every q head h:
 *   out[t][h] = sum_j softmax_j(scale * q_rot[t][h] . K_s[j]) V_s[j]
 * over keys j = 0..p of sequence s, where K_s[j] / V_s[j] are read in place
 * from the arena through block_tables (no gather copy).  Requires
 * positions[t] < context_lens[s] and context_lens[s] <= max_context_len.
 * Accumulation is float32; out is rounded once to dtype.
 *
 * Sequences with query_len x group <= KSHIPRA_OPT_DECODE_MAX_ROWS run on a
 * split-KV decode kernel (partial results of sequences cut into several
 * splits in `workspace`, merged inside the same kernel by the split that
 * finishes last); the others on a tcgen05 tensor-core chunked-prefill kernel with
 * fully masked key tiles skipped.  The split is decided on the device, so
 * one call may mix both kinds.  When both kinds may be present, the prefill
 * kernel runs beside the decode kernel: on a side stream of the
 * calling thread (created on first use, highest priority, released when the
 * thread ends), forked from and joined back into `stream` with events, so the
 * call stays ordered on `stream` as a whole and can be captured in a CUDA
 * graph; the prefill kernel keeps the SMs the decode kernel does not need to
 * reach full HBM bandwidth.  kshipra_paged_attention_noalloc runs the two
 * kernels one after the other on `stream` instead.
 *
 * out, q_rot [num_tokens][num_q_heads][head_dim]; k_arena, v_arena,
 * block_tables, context_lens [num_seqs], query_start_loc [num_seqs + 1],
 * positions [num_tokens], workspace: device pointers.  workspace must be
 * 256-byte aligned and at least kshipra_paged_attention_workspace_size()
 * bytes (it may be NULL when that size is 0).  out must not alias q_rot.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA.
 */
int kshipra_paged_attention(void* out, const void* q_rot, const void* k_arena, const void* v_arena,
                            const int32_t* block_tables, const int32_t* context_lens,
                            const int32_t* query_start_loc, const int32_t* positions, int num_seqs,
                            int num_tokens, int max_query_len, int max_context_len, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                            int num_blocks, float scale, int dtype, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * One step: kshipra_kv_append_rope followed by kshipra_paged_attention
 * (kshipra-3, sections 1 and 4), with the same arguments and results -- the
 * arena gets the new tokens' rotated K and raw V bit for bit as the append
 * writes them, out is the attention of the rotated q, bit for bit as the two
 * calls give it -- with fewer launches and no q_rot round trip:
 *  - every sequence of the decode class (max_query_len x group <=
 *    KSHIPRA_OPT_DECODE_MAX_ROWS): ONE launch; each decode CTA rotates its
 *    query rows from q in registers, and in the CTA whose key split holds a
 *    new token's position the warp that reads that position writes the
 *    token's K and V first;
 *  - otherwise: the append writes K and V only, then the attention kernels
 *    rotate q themselves (the prefill kernels in shared memory, the decode
 *    kernel in registers); with head_dim 128 they start while the append
 *    finishes.  This relies on no sequence's new tokens landing in a block
 *    that another sequence of the call reads as its cached prefix (a shared
 *    block is copied before it is written: kshipra_block_make_private).
 *
 * q [num_tokens][num_q_heads][head_dim], k, v [num_tokens][num_kv_heads]
 * [head_dim], rope_table as for kshipra_kv_append_rope; the other arguments
 * as for kshipra_paged_attention, with the same workspace size.  q_rot
 * (device, [num_tokens][num_q_heads][head_dim]) receives the rotated q; it
 * may be NULL.  q_rot must not alias out or q.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA.
 */
int kshipra_decode_step(void* out, const void* q, const void* k, const void* v, void* q_rot, void* k_arena,
                       void* v_arena, const int32_t* block_tables, const int32_t* context_lens,
                       const int32_t* query_start_loc, const int32_t* positions, const float* rope_table,
                       int rope_max_pos, int num_seqs, int num_tokens, int max_query_len, int max_context_len,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                       int num_blocks, float scale, int dtype, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * Paged attention without any allocation and without a caller workspace.
 * The paper has no counterpart; this is a convenience of this library.
 *
 * For callers that can't allocate device memory: a server that reserved all
 * free device memory for its KV arena up front (a later cudaMalloc would
 * fail), a host framework whose allocator owns every device byte, or a
 * latency-critical loop that must not pay cudaMalloc's implicit
 * synchronisation.  Same arguments, computation and errors as
 * kshipra_paged_attention minus the workspace: the split-KV partials live in
 * a fixed scratch array of KSHIPRA_NOALLOC_SCRATCH_BYTES bytes inside the
 * library, which every GPU that loads the library holds until the process
 * exits.  Sizes whose partials need more than that are rejected with
 * KSHIPRA_ERR_WORKSPACE_TOO_SMALL before anything is launched.  The need
 * depends on the calling thread's KSHIPRA_OPT_SPLIT_TOKENS (shorter splits,
 * more partials) and on the device's SM count (the automatic split size
 * follows it), so a size that fits under one setting or device may not fit
 * under another: query it with kshipra_paged_attention_workspace_size on the
 * same thread, with the same option and the device's SM count.  The first call on a device
 * looks up the scratch address on that device (make it before any stream
 * capture).  All calls share the one array: calls that overlap on the GPU
 * (different streams, or several host threads) race and corrupt each
 * other's results; serialise them.  Nothing in the scratch has to start at
 * zero: each call writes every partial it reads.
 * Errors: as kshipra_paged_attention; KSHIPRA_ERR_CUDA also when the scratch
 * address cannot be looked up.
 */
#define KSHIPRA_NOALLOC_SCRATCH_BYTES (16u << 20)
int kshipra_paged_attention_noalloc(void* out, const void* q_rot, const void* k_arena, const void* v_arena,
                                    const int32_t* block_tables, const int32_t* context_lens,
                                    const int32_t* query_start_loc, const int32_t* positions, int num_seqs,
                                    int num_tokens, int max_query_len, int max_context_len, int num_q_heads,
                                    int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                                    int num_blocks, float scale, int dtype, void* stream);

/*
 * Reads the current device's status word into *code_out (host pointer) and
 * clears it, after waiting for `stream`.  0 means no kernel reported a
 * violation since the last read.  Errors: INVALID_ARG, CUDA.
 */
int kshipra_device_status(int32_t* code_out, void* stream);

/* Sets a tuning option (KSHIPRA_OPT_*) for the calling host thread only;
 * it applies to that thread's later calls.  Errors: INVALID_ARG. */
int kshipra_set_option(int option, int value);

/* Static description of a status code. */
const char* kshipra_status_string(int code);

/* One-line description of the last error on the calling thread ("" if none). */
const char* kshipra_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KSHIPRA_H */
