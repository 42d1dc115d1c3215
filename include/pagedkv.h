/*
 * pagedkv.h -- C ABI of libpagedkv.so: the decode hot path of a paged KV
 * cache on one GPU (sm_103a).
 *
 * What the operations are (web pages on paged KV caches; page title, then
 * section):
 *   - tonho.wtf "vllm", "como funciona": the KV cache of a sequence is cut
 *     into fixed-size blocks (16 tokens by default) that are slices of one
 *     GPU pool; a per-sequence block table maps logical blocks to physical
 *     ones; a new physical block is taken only when the last one is full;
 *     decode attention takes the current token's query against the keys of
 *     one block at a time and accumulates the output against that block's
 *     values, so blocks need not be adjacent; sequences share blocks through
 *     reference counts, and a write into the last shared block copies that
 *     block and only it.
 *   - tonho.wtf "vllm", "o que isso custou": the three kernels the method
 *     needs -- block write, paged read fused with attention, batched block
 *     copy.  They are paged_kv_append, paged_attention_decode and
 *     copy_blocks below.
 *   - techtrendfeed "KV Cache Administration: PagedAttention &
 *     RadixAttention", "How PagedAttention Works", steps 1-4 (blocks of 16
 *     or 32 tokens; block table used by the kernel to gather K and V; growth
 *     one block at a time; copy-on-write), and "Why this modified LLM
 *     serving" (paging changes neither the attention result nor the model's
 *     outputs).
 *
 * Conventions shared by every call:
 *   - Cache layout: k_cache and v_cache are each
 *       [num_blocks][num_kv_heads][block_size][head_dim]
 *     row-major, elements of pkv_cache_desc.dtype.  Token position t of a
 *     sequence sits in logical block t / block_size at offset
 *     t % block_size; the (block, KV head) tile is contiguous.
 *   - A slot is physical_block * block_size + offset.
 *   - GQA: query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   - Ownership: every data pointer is a caller-owned DEVICE pointer unless
 *     stated otherwise; the library keeps no pointer after a call returns,
 *     allocates no memory, and never synchronises except in
 *     pkv_check_device_error.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *     default stream).  Every call is asynchronous on it.
 *   - Errors found on the host (null or misaligned pointers, unsupported
 *     shapes, too small a workspace) return a status and launch nothing.
 *     Bad metadata that lives on the device (a slot, block id or context
 *     length outside the pool) never faults: the kernel skips the access,
 *     zero-fills the affected output, and records the first such error in a
 *     per-device error word that pkv_check_device_error reads and clears.
 *   - Kernels never wait on another kernel or CTA.  Waits inside one CTA
 *     (its copy pipeline) are bounded; a wait that runs out records
 *     PKV_DEVERR_TIMEOUT and the CTA returns.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,     /* null/misaligned pointer or bad size */
    PKV_ERR_UNSUPPORTED = 2,     /* valid but not implemented shape or dtype */
    PKV_ERR_WORKSPACE = 3,       /* workspace missing or too small */
    PKV_ERR_CUDA = 4,            /* a CUDA runtime or driver call failed */
    PKV_ERR_DEVICE_METADATA = 5  /* reported by pkv_check_device_error */
} pkv_status;

typedef enum { PKV_BF16 = 0, PKV_FP16 = 1, PKV_FP32 = 2 } pkv_dtype;

/* Codes stored in the device error word (first error wins). */
enum {
    PKV_DEVERR_NONE = 0,
    PKV_DEVERR_SLOT = 1,        /* append / compact_tokens: slot >= num_blocks * block_size */
    PKV_DEVERR_COPY_ID = 2,     /* copy_blocks / swap_blocks: src or dst outside its pool */
    PKV_DEVERR_CONTEXT_LEN = 3, /* decode: context_lens[s] < 0, above the table's capacity, or above max_context_len */
    PKV_DEVERR_BLOCK_ID = 4,    /* decode: block_tables entry outside the pool */
    PKV_DEVERR_TIMEOUT = 5,     /* a bounded in-CTA wait ran out */
    PKV_DEVERR_PREFIX_LEN = 6,  /* grouped decode: prefix_lens[s] < 0, above context_lens[s] or
                                   max_prefix_len, or not a multiple of block_size */
    PKV_DEVERR_GROUP = 7        /* grouped decode: group_starts out of order or range, or a sequence
                                   with a shared prefix in no group or beyond max_group_size members */
};

/* Shape of one layer's paged cache (host struct, read during the call). */
typedef struct {
    int64_t num_blocks;  /* physical blocks in the pool, >= 1 */
    int32_t num_kv_heads;
    int32_t block_size;  /* tokens per block: 16 or 32 */
    int32_t head_dim;    /* 128 */
    int32_t dtype;       /* pkv_dtype: PKV_BF16 or PKV_FP16 */
} pkv_cache_desc;

/* Human-readable name of a status. Never NULL. */
const char* pkv_status_string(pkv_status status);

/* Library version as 10000*major + 100*minor + patch. */
int pkv_version(void);

/*
 * Block write ("vllm", "como funciona" and "o que isso custou").
 * For every token t with slot_mapping[t] >= 0 and every KV head h:
 *     k_cache[slot / bs][h][slot % bs][:] = k[t][h][:]   (same for v)
 * k, v:          [num_tokens][num_kv_heads][head_dim], cache dtype, 16-byte
 *                aligned device memory.
 * slot_mapping:  [num_tokens] int64 device memory; a negative slot marks a
 *                padding token, which is skipped.
 * k_cache, v_cache: the pool (layout above), 16-byte aligned.
 * num_tokens == 0 is a no-op.  Two tokens with the same slot race (last
 * writer undefined).  A slot >= num_blocks * block_size is skipped and
 * recorded as PKV_DEVERR_SLOT.  The copy is bit-exact.
 */
pkv_status paged_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                           void* k_cache, void* v_cache, const pkv_cache_desc* cache, void* stream);

/*
 * Bytes of workspace paged_attention_decode needs for these sizes (0 when
 * the call runs in a single pass).  partition_size as for
 * paged_attention_decode; with 0 (automatic) the size covers the smallest
 * automatic partition, so it is enough whatever the call picks.  Returns 0
 * for invalid sizes.
 */
size_t paged_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                       int32_t max_context_len, int32_t partition_size);

/* How paged_attention_decode divides the work (see paged_attention_plan). */
enum {
    PKV_PLAN_SINGLE = 0,       /* one CTA per (sequence, head group): no partials */
    PKV_PLAN_SPLIT = 1,        /* split-K, merged by the last partition of each row */
    PKV_PLAN_SPLIT_REDUCE = 2  /* split-K with more than 16 partitions, merged by a second kernel */
};

/*
 * The decomposition paged_attention_decode uses for these sizes on the
 * current device; -1 for invalid sizes.  block_size is the cache's.
 */
int32_t paged_attention_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t block_size,
                             int32_t max_context_len, int32_t partition_size);

/*
 * The split-K partition size (tokens) paged_attention_decode uses for these
 * sizes on the current device: partition_size itself when it is non-zero,
 * else the automatic choice.  Returns 0 for invalid sizes.
 */
int32_t paged_attention_partition_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t max_context_len, int32_t partition_size);

/*
 * Paged decode attention ("vllm", "como funciona": the query of the current
 * token against the keys of one block at a time, output accumulated against
 * the same block's values; blocks need not be adjacent).
 * For every sequence s and query head h, with L = context_lens[s] and
 * kvh = h / (num_q_heads / num_kv_heads):
 *     out[s][h][:] = sum_{t<L} softmax_t(scale * q[s][h] . K[t]) V[t]
 * where K[t], V[t] are row t % bs of tile (block_tables[s][t / bs], kvh).
 * L counts every attended token, including the one appended this step;
 * L == 0 gives zeros.
 *
 * q:               [num_seqs][num_q_heads][head_dim], cache dtype, 16-byte aligned.
 * k_cache, v_cache: the pool, 16-byte aligned.
 * block_tables:    [num_seqs][max_blocks_per_seq] int32; entries past
 *                  ceil(L / bs) are never read.
 * context_lens:    [num_seqs] int32, each in [0, min(max_context_len,
 *                  max_blocks_per_seq * bs)].
 * max_context_len: host-side upper bound of context_lens; it sizes the
 *                  split-K partitions and the workspace.
 * out:             [num_seqs][num_q_heads][head_dim] of out_dtype (PKV_FP32,
 *                  PKV_BF16 or PKV_FP16), 16-byte aligned.
 * partition_size:  tokens per split-K partition, a multiple of block_size;
 *                  0 picks 512, 1024, 2048 or 4096 from the amount of work
 *                  and the device's SM count (the largest that still gives
 *                  every resident decode CTA two work units).  When max_context_len > partition_size
 *                  each partition writes (o_p, lse_p) to the workspace and
 *                  they are merged through their log-sum-exp: by the last
 *                  partition of each (sequence, head group) to finish when a
 *                  sequence has at most 16 partitions, else by a second
 *                  kernel.  Otherwise one kernel writes out directly.
 * workspace:       device memory of at least
 *                  paged_attention_workspace_bytes(...) bytes, 256-byte
 *                  aligned (may be NULL when that is 0).  Contents on entry
 *                  are ignored: the merge's arrival counters carry the
 *                  epoch of the call that wrote them, and a counter of any
 *                  other epoch counts as zero.  Two calls whose kernels may
 *                  overlap on the GPU must not share a workspace.
 * Supported: head_dim 128; block_size 16 or 32; bf16 or fp16 caches;
 * num_q_heads a multiple of num_kv_heads; num_seqs <= 65535.
 * Results depend only on logical token order: permuting physical block ids
 * leaves the output bit-for-bit unchanged.
 */
pkv_status paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_context_len, float scale, void* out, int32_t out_dtype,
                                  const pkv_cache_desc* cache, int32_t partition_size, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * A decode step in one launch: the block write of one new token per
 * sequence ("vllm", "o que isso custou": block write) fused into
 * paged_attention_decode.  The result, and the cache afterwards, are those
 * of paged_kv_append(k_new, v_new, slot_mapping, num_seqs, ...) followed by
 * paged_attention_decode(...), provided that each sequence's new token is its
 * last context position: slot_mapping[s] must be the slot of position
 * context_lens[s] - 1 of sequence s (block_tables[s][(L-1)/bs] * bs +
 * (L-1) % bs), or negative when sequence s has no new token, and no other
 * sequence may read that slot in this call.  A slot that is not that position
 * is not written and is recorded as PKV_DEVERR_SLOT.
 * k_new, v_new:  [num_seqs][num_kv_heads][head_dim], cache dtype, 16-byte
 *                aligned device memory.
 * slot_mapping:  [num_seqs] int64 device memory.
 * Other arguments as for paged_attention_decode; k_cache and v_cache are
 * written.
 */
pkv_status paged_attention_append_decode(const void* q, const void* k_new, const void* v_new,
                                         const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_context_len, float scale, void* out, int32_t out_dtype,
                                         const pkv_cache_desc* cache, int32_t partition_size, void* workspace,
                                         size_t workspace_bytes, void* stream);

/*
 * paged_attention_decode for batches whose sequences share prompt blocks
 * (samples forked from one prompt, a common system prompt).  Forked
 * sequences map the prompt's logical blocks to the same physical blocks,
 * counted by reference ("vllm", "como funciona"; techtrendfeed "KV Cache
 * Administration", "How PagedAttention Works", step 4), and a shared prefix
 * is read once and reused (aitalk.it "PagedAttention e RadixAttention").
 * Here each shared block is read from HBM once per (group, KV head) and
 * attended by every member's query heads together; each member's own
 * blocks are attended as in paged_attention_decode, and the two parts are
 * merged through their log-sum-exp.
 *
 * The result is paged_attention_decode's on the same q, cache, tables and
 * lengths, provided that for every member s of group g, positions
 * 0 .. prefix_lens[s]-1 of s sit in the same physical blocks as the same
 * positions of the group's first member (block_tables rows agree there).
 *
 * group_starts:   [num_groups + 1] int32 device memory: the members of group
 *                 g are sequences group_starts[g] .. group_starts[g+1]-1, in
 *                 order; groups must not overlap.
 * max_group_size: host-side upper bound of group_starts[g+1] - group_starts[g].
 * prefix_lens:    [num_seqs] int32 device memory: tokens of s attended through
 *                 its group's first member's block table, a multiple of
 *                 block_size in [0, min(context_lens[s], max_prefix_len)].
 *                 Members of one group may differ.  A sequence with
 *                 prefix_lens[s] == 0 need not be in any group.
 * max_prefix_len: host-side upper bound of prefix_lens, <= max_context_len.
 * workspace:      at least paged_attention_grouped_workspace_bytes(...)
 *                 bytes, 256-byte aligned; always needed.  Contents on entry
 *                 are ignored.
 * Other arguments as for paged_attention_decode.  Supported: as for
 * paged_attention_decode, with num_q_heads / num_kv_heads <= 64 and
 * num_groups <= 65535.  Bad metadata never faults: a prefix length out of
 * range (PKV_DEVERR_PREFIX_LEN), or a sequence with a nonzero prefix length
 * that lies in no group or in a group beyond max_group_size members
 * (PKV_DEVERR_GROUP), zeroes that sequence's output.  A group whose range
 * is out of order or out of bounds is skipped (PKV_DEVERR_GROUP); the
 * groups on either side of it may then overlap, and a sequence in two of
 * them gets a finite but unspecified output.  The pages describe the
 * sharing, not this kernel: the grouped read is an addition of this
 * library.
 */
pkv_status paged_attention_decode_grouped(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                          int32_t max_context_len, const int32_t* group_starts,
                                          int32_t num_groups, int32_t max_group_size, const int32_t* prefix_lens,
                                          int32_t max_prefix_len, float scale, void* out, int32_t out_dtype,
                                          const pkv_cache_desc* cache, int32_t partition_size, void* workspace,
                                          size_t workspace_bytes, void* stream);

/*
 * A grouped decode step in one call: the block write of one new token per
 * sequence (as paged_attention_append_decode) fused into
 * paged_attention_decode_grouped.  The result, and the cache afterwards, are
 * those of paged_kv_append(k_new, v_new, slot_mapping, num_seqs, ...)
 * followed by paged_attention_decode_grouped(...), provided that each
 * sequence's new token is its last context position and lies past its
 * shared prefix (prefix_lens[s] < context_lens[s]; a write into a shared
 * block is preceded by its copy, "vllm", "como funciona"): slot_mapping[s]
 * must be the slot of position context_lens[s] - 1, or negative when
 * sequence s has no new token.  A slot that is not that position is not
 * written and is recorded as PKV_DEVERR_SLOT.  Arguments as for
 * paged_attention_append_decode and paged_attention_decode_grouped.
 */
pkv_status paged_attention_append_decode_grouped(const void* q, const void* k_new, const void* v_new,
                                                 const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                 const int32_t* context_lens, int32_t num_seqs,
                                                 int32_t num_q_heads, int32_t max_context_len,
                                                 const int32_t* group_starts, int32_t num_groups,
                                                 int32_t max_group_size, const int32_t* prefix_lens,
                                                 int32_t max_prefix_len, float scale, void* out, int32_t out_dtype,
                                                 const pkv_cache_desc* cache, int32_t partition_size,
                                                 void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes paged_attention_decode_grouped needs (0 for invalid sizes). */
size_t paged_attention_grouped_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                               int32_t max_context_len, int32_t max_prefix_len,
                                               int32_t partition_size);

/*
 * paged_attention_decode without a workspace argument, for callers that
 * cannot allocate device memory: a process whose device memory is all owned
 * by another allocator (such as a serving engine that reserved nearly all of
 * HBM for its KV pool at start-up), or a latency-critical loop that must not
 * call cudaMalloc because it can implicitly synchronise the device.  The
 * pages have no counterpart to this call; it is an addition of this library.
 *
 * Arguments and results are those of paged_attention_decode.  The split-K
 * partials live in a file-scope device array of 16 MiB that every GPU which
 * loads the library holds until the process exits; a call whose
 * paged_attention_workspace_bytes(...) exceeds 16 MiB is rejected with
 * PKV_ERR_WORKSPACE before anything is launched.  The call allocates nothing.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  The array is shared by every call on the
 * device and keeps the last call's contents; nothing in it needs to start at
 * zero.  Calls whose kernels overlap on the GPU race on the array: the caller
 * must serialise them.
 */
pkv_status paged_attention_decode_static(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_context_len, float scale, void* out, int32_t out_dtype,
                                         const pkv_cache_desc* cache, int32_t partition_size, void* stream);

/*
 * Batched copy-on-write block copy ("vllm", "como funciona": a write into
 * the last shared block copies that block and only it; "o que isso
 * custou": batched block copy).
 * For each pair i and each layer l:
 *     k_caches[l][dst] = k_caches[l][src], v_caches[l][dst] = v_caches[l][src]
 * (whole blocks: every KV head and slot), with (src, dst) =
 * (src_dst_pairs[2i], src_dst_pairs[2i+1]).
 * k_caches, v_caches: HOST arrays of num_layers device pointers (each
 *                  16-byte aligned), all layers of the shape in `cache`.
 * src_dst_pairs:   [num_pairs][2] int64 DEVICE memory.
 * Destinations must be distinct and no destination may also be a source
 * (otherwise the result depends on block scheduling); an id outside the
 * pool skips that pair and records PKV_DEVERR_COPY_ID.  Bit-exact.
 */
pkv_status copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                       const int64_t* src_dst_pairs, int32_t num_pairs, const pkv_cache_desc* cache,
                       void* stream);

/*
 * Swap-out / swap-in of whole blocks between two pools ("vllm", "como
 * funciona": a preempted sequence's blocks go to CPU RAM and come back).
 * For each pair i and each layer l:
 *     dst_k_caches[l][dst] = src_k_caches[l][src]   (and the V caches)
 * with (src, dst) = (src_dst_pairs[2i], src_dst_pairs[2i+1]), src a block of
 * the source pool (src_num_blocks blocks) and dst one of the destination
 * pool (dst_num_blocks blocks).  Either pool may be GPU memory or page-locked
 * host memory that the GPU addresses directly (cudaHostAlloc, or
 * cudaHostRegister'ed memory, on a unified-addressing system; on GB300 the
 * copy runs over NVLink-C2C).  Both pools have the per-block shape of
 * `cache` (its num_blocks is not used).
 * src_k_caches, ...: HOST arrays of num_layers pointers, 16-byte aligned.
 * src_dst_pairs:    [num_pairs][2] int64, GPU-addressable memory.
 * An id outside its pool skips that pair and records PKV_DEVERR_COPY_ID.
 * Destinations must be distinct.  Bit-exact.
 */
pkv_status swap_blocks(void* const* src_k_caches, void* const* src_v_caches, int64_t src_num_blocks,
                       void* const* dst_k_caches, void* const* dst_v_caches, int64_t dst_num_blocks,
                       int32_t num_layers, const int64_t* src_dst_pairs, int32_t num_pairs,
                       const pkv_cache_desc* cache, void* stream);

/*
 * Token-level compaction into fresh target blocks (gist.science "Zipage",
 * Compressed PagedAttention: once a request holds N_max blocks and the last
 * one is full, the tokens it keeps are rewritten into new target blocks --
 * the first N_max - 1 of its new table -- so that prefix blocks shared with
 * other requests stay intact).  For each i with both slots >= 0:
 *     k_cache[dst slot row of head h] = k_cache[src slot row of head h]
 * for every KV head h, and the same for v_cache.  The caller chooses the
 * kept tokens (their scoring is not part of this library) and the target
 * blocks.  No destination slot may also be a source slot, and destinations
 * must be distinct.  A slot >= num_blocks * block_size skips the token and
 * records PKV_DEVERR_SLOT.  src_slots, dst_slots: [num_tokens] int64 device
 * memory.  Bit-exact.
 */
pkv_status compact_tokens(const int64_t* src_slots, const int64_t* dst_slots, int64_t num_tokens, void* k_cache,
                          void* v_cache, const pkv_cache_desc* cache, void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns PKV_OK (and *first_error_code = 0) when no kernel recorded
 * an error since the last check, PKV_ERR_DEVICE_METADATA with the first
 * PKV_DEVERR_* code otherwise, or PKV_ERR_CUDA.  first_error_code may be
 * NULL.
 * The word is one per device, shared by the library's calls on every stream,
 * and only `stream` is synchronised: an error recorded by a kernel still
 * running on another stream is not seen by this check, and is reported by a
 * later one (or, if it lands between the read and the clear, lost).  To check
 * the calls of several streams, synchronise all of them (or the device)
 * before calling this.
 */
pkv_status pkv_check_device_error(void* stream, int32_t* first_error_code);

/*
 * Self-test of the bounded-wait error path, with no fault and no hang.
 * Launches one CTA that waits, through the same bounded mbarrier wait the
 * copy pipelines use but with a limit of limit_us microseconds, on a phase
 * that nothing completes.  The wait runs out, the CTA records
 * PKV_DEVERR_TIMEOUT in the device error word (as a stalled pipeline would)
 * and returns; the context stays usable.  limit_us: 1 .. 2,000,000, else
 * PKV_ERR_INVALID_ARG with nothing launched.  Asynchronous on `stream`.
 */
pkv_status pkv_wait_selftest(int32_t limit_us, void* stream);

/* Number of kernels this library has launched in this process. */
uint64_t pkv_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
