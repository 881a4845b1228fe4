/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) PagedAttention library: decode
 * and prefill attention over a paged KV cache and the block moves around it.
 *
 * The operations follow the pages on PagedAttention and continuous batching:
 *
 *  - paged_decode_attention: "PagedAttention: gestionar la KV cache como
 *    memoria de un sistema operativo" (josueisai.com), section "Cómo funciona
 *    por dentro" -- the attention kernel reads non-contiguous KV memory by
 *    looking up each stretch of the sequence in its block table, scores the
 *    query against every block's keys and takes the softmax-weighted sum of
 *    the values.  One call performs this decode step for every sequence of a
 *    continuously batched set ("Batching Continuo y PagedAttention",
 *    cruxr.ai, section "Batching continuo (In-Flight Batching)").
 *  - kv_append: same page and section -- a new token's key and value go into
 *    the last block of the table (a new block is taken only when the last is
 *    full; the host block manager decides, this call writes the slot).
 *  - copy_blocks: iplexlaw.co.kr "pagedattention-vllm-kv-cache", section
 *    "Dos respuestas a una entrada: ejemplo hipotético" -- a shared block that
 *    still has room is copied when written while other references to it
 *    exist (copy-on-write, "Batching Continuo y PagedAttention", section
 *    "PagedAttention: Memoria virtual para la KV cache").
 *  - paged_decode_step: the three calls above as one decode step (copies,
 *    append, attention), every argument checked before anything launches.
 *  - Beyond the decode step: paged_prefill_attention (causal attention of a
 *    prompt or chunk over the cache), paged_decode_attention_shared_prefix
 *    (decode reading blocks shared by a group of sequences once), swap_blocks
 *    (blocks between a device pool and a pinned host pool, for preemption),
 *    copy_blocks_layers / kv_append_layers (every layer in one launch), and
 *    paged_decode_attention_static_workspace (decode with library scratch).
 *    Each cites its passage below.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Block size P = 16 tokens ("típicamente P = 16").
 *  - Cache layout, for one layer: k_cache and v_cache are two arrays
 *      [num_blocks][num_kv_heads][16][head_dim]
 *    so each (physical block, kv head) tile is one contiguous 16*head_dim run
 *    (a block for one layer and one head stores 2*P*d_h elements, K and V).
 *    Slot s of the pool is block s / 16, offset s % 16.
 *  - q and out: [num_seqs][num_q_heads][head_dim]; k, v of kv_append:
 *    [num_tokens][num_kv_heads][head_dim]. All row-major, contiguous.
 *  - dtype: PKV_BF16 (bf16 storage, fp32 accumulation, bf16 output rounded to
 *    nearest even) or PKV_F32 (fp32 throughout). q, caches and out share it.
 *    The decode calls (paged_decode_attention, paged_decode_step,
 *    paged_decode_attention_static_workspace and the planning queries) also
 *    take PKV_BF16_OUT_F32: bf16 q and caches, the bf16 arithmetic unchanged,
 *    and out fp32 -- the accumulated O / L before it would be rounded to bf16,
 *    so the kernel's own error can be measured apart from the output rounding
 *    (append and copy inside paged_decode_step move bf16).
 *  - head_dim is 64 or 128; num_q_heads is a multiple of num_kv_heads and the
 *    group size g = num_q_heads / num_kv_heads is at most 16. Query head hq
 *    reads kv head hq / g (consecutive grouping).
 *  - Every pointer is a DEVICE pointer unless stated otherwise (the per-step
 *    arguments of decode, append and copy may be page-locked host memory),
 *    16-byte aligned. The caller owns all memory (including the workspace) and the
 *    stream; the library never allocates, frees or synchronises. `stream` is a
 *    cudaStream_t (NULL = the legacy default stream); calls are asynchronous.
 *  - Return value: PKV_OK, or a negative status (pkv_status_string). Only
 *    scalar arguments and pointer alignment can be checked without a
 *    synchronisation; checks of device contents go through pkv_validate /
 *    pkv_validate_slots, and the kernels themselves never fault on bad
 *    contents: they skip the offending element (or read zeros) and raise a bit
 *    in the device error word (pkv_device_error).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_BF16_OUT_F32 = 2 } pkv_dtype;

#define PKV_OK 0
#define PKV_ERR_ARG -1          /* bad scalar argument, null pointer, shape mismatch */
#define PKV_ERR_UNSUPPORTED -2  /* head_dim, dtype or group size not supported */
#define PKV_ERR_INDEX -3        /* index out of range (copy pairs checked on the host) */
#define PKV_ERR_OVERLAP -4      /* copy pairs overlap: repeated destination, or a destination that is also a source */
#define PKV_ERR_CUDA -5         /* a CUDA runtime/driver call or launch failed */
#define PKV_ERR_WORKSPACE -6    /* workspace missing or smaller than pkv_decode_workspace_bytes */
#define PKV_ERR_ALIGN -7        /* a pointer is not 16-byte aligned */

/* partition_tokens value that asks for the persistent balanced split (bf16). */
#define PKV_PARTITION_BALANCED -1

/* Bits of the device error word. */
#define PKV_DEVERR_BLOCK_ID 0x1u    /* a block-table entry outside [0, num_blocks): its K/V read as zeros */
#define PKV_DEVERR_SLOT 0x2u        /* a slot >= num_blocks*16 in kv_append: that token was skipped */
#define PKV_DEVERR_PAIR 0x4u        /* a copy pair outside [0, num_blocks): that pair was skipped */
#define PKV_DEVERR_TIMEOUT 0x8u     /* a bounded wait inside a kernel ran out: output unspecified */
#define PKV_DEVERR_LENGTH 0x10u     /* context_len < 0, > max_blocks_per_seq*16 or > max_context_len: clamped */
#define PKV_DEVERR_POINTER 0x20u    /* a pointer in a per-layer pointer array is null or not 16-byte aligned: skipped */

/* Human-readable name of a status code (static storage). */
const char *pkv_status_string(int status);

/* Library version: major*10000 + minor*100 + patch. */
int pkv_version(void);

/*
 * Tokens per split-context partition for a decode call (a multiple of 16):
 * partition_tokens > 0 is returned as is (it must be a multiple of 16); 0
 * (automatic) and PKV_PARTITION_BALANCED give 512. A sequence of L tokens is
 * processed as ceil(L / partition) partitions whose partial softmax
 * statistics are merged by a log-sum-exp reduce; the result does not depend
 * on the choice.
 *
 * bf16 has a second decomposition, chosen with PKV_PARTITION_BALANCED, or
 * automatically (partition_tokens == 0) when the batch has at least a quarter
 * as many (sequence, kv head) pairs as the GPU runs persistent warps (12 per
 * SM): the blocks of all pairs are cut into equal shares, one per warp of a
 * persistent kernel (one CTA per SM), and the pieces of a cut sequence are
 * merged with the same log-sum-exp rule inside that kernel. Batches of a few
 * long sequences keep fixed partitions, which merge faster.
 */
int pkv_decode_partition_tokens(int num_seqs, int num_kv_heads, int max_context_len, int partition_tokens);

/*
 * Kernel launches one paged_decode_attention call makes with these arguments:
 * 1 (persistent balanced kernel, or no sequence longer than one partition),
 * 2 (partition kernel + log-sum-exp reduce kernel), 0 for an empty batch or
 * bad arguments. Queries the current device's SM count.
 */
int pkv_decode_launches(int num_seqs, int num_kv_heads, int max_context_len, int partition_tokens, pkv_dtype dtype);

/*
 * 1 if paged_decode_attention with these arguments runs the persistent
 * balanced kernel (bf16 only: PKV_PARTITION_BALANCED, or automatic
 * partitioning on a batch with at least a quarter as many (sequence, kv head)
 * units as the GPU has persistent warps), else 0. Queries the current
 * device's SM count.
 */
int pkv_decode_persistent(int num_seqs, int num_kv_heads, int partition_tokens, pkv_dtype dtype);

/*
 * Layout of every decode workspace (paged_decode_attention, paged_decode_step,
 * paged_decode_attention_shared_prefix, and the library's own array behind
 * paged_decode_attention_static_workspace): the first PKV_DECODE_COUNTER_BYTES
 * bytes hold the persistent kernel's arrival counters, then come partial
 * softmax states (max in the log2 domain, sum, partial output, fp32).
 *  - The counters must be zero before the first call that uses the buffer
 *    (zero-fill it once after allocating it, e.g. cudaMemsetAsync). Every
 *    call that completes without a device error leaves them zero, and no
 *    decode path writes anything else into them.
 *  - The partial states need no initial value: a call writes every state it
 *    reads earlier in the same call.
 * So one buffer, sized for the largest call, serves calls of any shape on any
 * decode path in turn (split grid, persistent, shared prefix), with no
 * clearing between them. After a call that raised PKV_DEVERR_TIMEOUT, zero
 * the counters again.
 */
#define PKV_DECODE_COUNTER_BYTES 10240u

/*
 * Bytes of device workspace paged_decode_attention needs with these
 * arguments (0 when it needs none): the counter header and the partial
 * states, laid out as above.
 */
size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int max_context_len, int partition_tokens);

/*
 * One decode step of attention for every sequence:
 *   out[s][hq][:] = sum_t softmax_t(scale * <q[s][hq], K_t>) V_t
 * over the context_lens[s] tokens of sequence s, token t read from physical
 * block block_tables[s][t / 16] at offset t % 16, kv head hq / g.
 *
 * block_tables: int32 [num_seqs][max_blocks_per_seq] (entries past
 *   ceil(len/16) are never read); context_lens: int32 [num_seqs].
 * max_context_len: host-side upper bound on every context_lens[s] (sizes the
 *   launch); longer lengths are clamped and flagged (PKV_DEVERR_LENGTH).
 * A context length of 0 yields a zero output row.
 * workspace / workspace_bytes: device scratch of at least
 *   pkv_decode_workspace_bytes(...) bytes, laid out and initialised as
 *   described above PKV_DECODE_COUNTER_BYTES (may be NULL when that size is
 *   0). Concurrent calls must not share a workspace.
 * q, out, block_tables and context_lens may point to page-locked host memory
 *   (mapped into the device's address space, as cudaHostAlloc gives): the
 *   kernels read and write them in place over the host link. The caches and
 *   the workspace must be device memory.
 */
int paged_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens, float scale,
                           int num_kv_heads, int num_seqs, int num_q_heads, int head_dim,
                           int max_blocks_per_seq, int num_blocks, int max_context_len, pkv_dtype dtype,
                           int partition_tokens, void *workspace, size_t workspace_bytes, void *stream);

/*
 * One whole decode step in one call ("Batching Continuo y PagedAttention",
 * cruxr.ai, section "Juntándolo todo: Arquitectura de vLLM": each iteration
 * copies shared blocks that are about to be written, appends every running
 * sequence's new token, then runs attention): copy_blocks(src_dst_pairs),
 * then kv_append(k_new, v_new, slot_mapping), then paged_decode_attention,
 * with the arguments and semantics of those three calls (num_pairs = 0 or
 * num_tokens = 0 skips a stage). Every argument is checked before anything
 * is launched; a failing check launches nothing.
 * Because the library launches the append itself, the attention kernels are
 * launched programmatically after it: they read block_tables, context_lens
 * and q (which the append does not write) while the append still runs, and
 * wait for it only before reading the caches. Nothing changes for the
 * caller: work enqueued on the stream before the call finishes before the
 * step's first launch, as usual.
 */
int paged_decode_step(void *out, const void *q, void *k_cache, void *v_cache, const int32_t *block_tables,
                      const int32_t *context_lens, float scale, int num_kv_heads, int num_seqs, int num_q_heads,
                      int head_dim, int max_blocks_per_seq, int num_blocks, int max_context_len, pkv_dtype dtype,
                      int partition_tokens, void *workspace, size_t workspace_bytes, const void *k_new,
                      const void *v_new, const int64_t *slot_mapping, int num_tokens, const int64_t *src_dst_pairs,
                      int num_pairs, void *stream);

/*
 * paged_decode_attention for a batch whose sequences share leading blocks --
 * parallel samples of one prompt, a common system prompt ("Batching Continuo
 * y PagedAttention", cruxr.ai, copy-on-write paragraph: the tables of requests
 * with a common prefix point at the same physical blocks; "PagedAttention:
 * gestionar la KV cache como memoria de un sistema operativo", section "El
 * regalo extra: compartir memoria"). Results are those of
 * paged_decode_attention on the same tables; the shared blocks are read from
 * HBM once per group instead of once per sequence: a group's unit attends the
 * union of its members' blocks -- the shared ones once for every member's
 * query heads, each member's own blocks for that member's heads only.
 *
 * group_members: int32 [num_groups][group_size], sequence ids (-1 = empty
 *   slot). The groups partition the batch: every sequence is listed exactly
 *   once, a sequence that shares nothing as a group of one (a sequence not
 *   listed gets no output); so num_groups <= num_seqs (else PKV_ERR_ARG).
 * shared_blocks: int32 [num_groups]: leading blocks all members' tables hold
 *   in common (same physical ids). The kernel uses at most the full blocks of
 *   the group's shortest member and reads them through the first member's
 *   table; the caller guarantees the members agree on them.
 * group_size x (num_q_heads / num_kv_heads) must be at most 16. bf16 only.
 * Partitions of partition_tokens split each group's union of blocks.
 * workspace: at least pkv_shared_prefix_workspace_bytes(...) bytes; it
 *   needs no zero-fill of its own and may be the buffer other decode calls
 *   use (it never writes the counter header). partition_tokens as for paged_decode_attention (> 0 or
 *   0 for 512). Two launches: the prefix/suffix kernel and a merge kernel.
 */
int paged_decode_attention_shared_prefix(void *out, const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, const int32_t *context_lens, float scale,
                                         int num_kv_heads, int num_seqs, int num_q_heads, int head_dim,
                                         int max_blocks_per_seq, int num_blocks, int max_context_len,
                                         const int32_t *group_members, const int32_t *shared_blocks, int num_groups,
                                         int group_size, pkv_dtype dtype, int partition_tokens, void *workspace,
                                         size_t workspace_bytes, void *stream);

/* Workspace bytes paged_decode_attention_shared_prefix needs (the decode
 * workspace layout above: its counter header is left untouched). */
size_t pkv_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_context_len,
                                         int group_size, int partition_tokens);

/*
 * Causal prefill attention over the paged cache: several new tokens per
 * sequence -- a prompt, or a chunk of one that follows earlier context
 * ("Batching Continuo y PagedAttention", cruxr.ai, section "Juntándolo todo:
 * Arquitectura de vLLM": the prefill pass over the whole prompt fills the KV
 * cache; "Continuous Batching", ultralytics.com glossary, chunked prefill).
 * The new tokens' K and V must already be in the cache (kv_append).
 *
 * Sequence s owns query rows query_start[s] .. query_start[s+1]-1, n_s rows:
 * its last n_s context positions, context_lens[s] - n_s .. context_lens[s]-1.
 * Query i of s (position pos = context_lens[s] - n_s + i) attends to the
 * sequence's tokens at positions 0 .. pos:
 *   out[r][hq][:] = sum_{t<=pos} softmax_t(scale * q[r][hq] . K_t[hkv]) V_t[hkv],
 *   hkv = hq / (num_q_heads / num_kv_heads).
 * q, out: bf16 [num_queries][num_q_heads][head_dim]; caches, block_tables,
 *   context_lens as for paged_decode_attention. query_start: int32
 *   [num_seqs + 1], device, non-decreasing from 0, query_start[num_seqs] <=
 *   num_queries.
 * max_query_len: host-side upper bound on every n_s (sizes the launch);
 *   max_context_len as for paged_decode_attention.
 * n_s < 0, n_s > context_lens[s], n_s > max_query_len or rows past
 *   num_queries: the sequence's rows are left unwritten and PKV_DEVERR_LENGTH
 *   is raised.
 * bf16 only; head_dim 64 or 128; num_q_heads / num_kv_heads at most 64.
 * No workspace; one launch.
 */
int paged_prefill_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *context_lens, const int32_t *query_start,
                            float scale, int num_kv_heads, int num_seqs, int num_q_heads, int head_dim,
                            int max_blocks_per_seq, int num_blocks, int num_queries, int max_query_len,
                            int max_context_len, pkv_dtype dtype, void *stream);

/*
 * KV append: for each token t with slot = slot_mapping[t] >= 0,
 *   k_cache[slot / 16][h][slot % 16][:] = k[t][h][:]   (and v) for every kv head h.
 * Negative slots are skipped (padding). Slots >= num_blocks*16 are skipped
 * and flagged (PKV_DEVERR_SLOT). Two tokens with the same slot race.
 * slot_mapping: int64 [num_tokens]. Bit-exact copy.
 * k, v and slot_mapping may point to page-locked host memory (read in place).
 */
int kv_append(const void *k, const void *v, const int64_t *slot_mapping, void *k_cache, void *v_cache,
              int num_tokens, int num_kv_heads, int head_dim, int num_blocks, pkv_dtype dtype, void *stream);

/*
 * Block copy (copy-on-write): for each pair i, copy physical block
 * src_dst_pairs[i][0] onto src_dst_pairs[i][1] -- all kv heads, all 16
 * slots -- in both k_cache and v_cache. src_dst_pairs: int64 [num_pairs][2],
 * device or page-locked host memory. Pairs must not overlap (all destinations distinct, no destination
 * also a source): check them on the host with pkv_check_copy_pairs. Pairs out
 * of range are skipped and flagged (PKV_DEVERR_PAIR). Bit-exact copy.
 */
int copy_blocks(void *k_cache, void *v_cache, const int64_t *src_dst_pairs, int num_pairs, int num_kv_heads,
                int head_dim, int num_blocks, pkv_dtype dtype, void *stream);

/*
 * Block swap between two pools ("Batching Continuo y PagedAttention",
 * cruxr.ai, section "Juntándolo todo: Arquitectura de vLLM": under memory
 * pressure the scheduler copies a low-priority request's KV blocks to CPU
 * memory, frees the GPU blocks, and copies them back to resume). For each pair
 * i, block src_dst_pairs[i][0] of the source pool is copied onto block
 * src_dst_pairs[i][1] of the destination pool, all kv heads and 16 slots, in
 * both caches. Each pool is [num_blocks][num_kv_heads][16][head_dim] in device
 * memory or in pinned host memory the GPU can address (cudaHostAlloc or
 * cudaHostRegister with unified addressing: the host pointer is used as is).
 * src_dst_pairs: int64 [num_pairs][2] in device-accessible memory. Swap-out
 * is device -> host pool, swap-in host -> device pool; device -> device moves
 * between pools too. Destinations must be distinct (pkv_check_swap_pairs);
 * pairs out of range are skipped and flagged (PKV_DEVERR_PAIR). Bit-exact.
 */
int swap_blocks(void *dst_k_cache, void *dst_v_cache, int dst_num_blocks, const void *src_k_cache,
                const void *src_v_cache, int src_num_blocks, const int64_t *src_dst_pairs, int num_pairs,
                int num_kv_heads, int head_dim, pkv_dtype dtype, void *stream);

/*
 * Host-side check of swap pairs (HOST pointer): PKV_ERR_INDEX if an id is
 * outside its pool, PKV_ERR_OVERLAP if a destination repeats. No CUDA call.
 */
int pkv_check_swap_pairs(const int64_t *host_pairs, int num_pairs, int src_num_blocks, int dst_num_blocks);

/*
 * copy_blocks for num_layers layers in one launch: a logical block spans all
 * layers ("Batching Continuo y PagedAttention", section "PagedAttention:
 * Memoria virtual para la KV cache"), so one copy-on-write copies it in every
 * layer's cache. k_caches, v_caches: arrays of num_layers cache pointers, the
 * arrays themselves in device-accessible memory; every layer's pool has
 * num_blocks blocks of the same shape. A null or misaligned pointer skips
 * that layer (PKV_DEVERR_POINTER). Same pair rules as copy_blocks.
 */
int copy_blocks_layers(void *const *k_caches, void *const *v_caches, int num_layers, const int64_t *src_dst_pairs,
                       int num_pairs, int num_kv_heads, int head_dim, int num_blocks, pkv_dtype dtype, void *stream);

/*
 * kv_append for num_layers layers in one launch: layer l writes k[l][t], v[l][t]
 * ([num_tokens][num_kv_heads][head_dim]) into k_caches[l], v_caches[l] at
 * slot_mapping[t] (one slot mapping for all layers). Pointer arrays in
 * device-accessible memory; same slot rules as kv_append.
 */
int kv_append_layers(const void *const *k, const void *const *v, const int64_t *slot_mapping, void *const *k_caches,
                     void *const *v_caches, int num_layers, int num_tokens, int num_kv_heads, int head_dim,
                     int num_blocks, pkv_dtype dtype, void *stream);

/*
 * Host-side check of copy pairs (HOST pointer, int64 [num_pairs][2]):
 * PKV_ERR_INDEX if an id is outside [0, num_blocks), PKV_ERR_OVERLAP if a
 * destination repeats or is also a source, else PKV_OK. No CUDA call.
 */
int pkv_check_copy_pairs(const int64_t *host_pairs, int num_pairs, int num_blocks);

/*
 * Device-side check of decode metadata. Clears *dev_err_word (device int32)
 * on `stream`, then ORs into it PKV_DEVERR_BLOCK_ID for any entry
 * block_tables[s][j], j < ceil(context_lens[s] / 16), outside [0, num_blocks),
 * and PKV_DEVERR_LENGTH for any length < 0, > max_blocks_per_seq*16 or
 * > max_context_len. Never traps.
 */
int pkv_validate(const int32_t *block_tables, const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                 int num_blocks, int max_context_len, int32_t *dev_err_word, void *stream);

/* Same for a slot mapping: PKV_DEVERR_SLOT for any slot >= num_blocks*16. */
int pkv_validate_slots(const int64_t *slot_mapping, int num_tokens, int num_blocks, int32_t *dev_err_word,
                       void *stream);

/*
 * Reads (synchronously, on the current device) the library's device error
 * word -- the OR of PKV_DEVERR_* bits raised by kernels since it was last
 * cleared -- into *value, and clears it when `clear` is nonzero.
 */
int pkv_device_error(uint32_t *value, int clear);

/*
 * Bytes of the library's built-in decode scratch (32 MiB), used by
 * paged_decode_attention_static_workspace.
 */
#define PKV_STATIC_WORKSPACE_BYTES (32u << 20)

/*
 * paged_decode_attention without a caller-provided workspace. No part of the
 * pages corresponds to this call: it exists for callers that cannot allocate
 * device memory where they call the library -- e.g. a plugin or extension hook
 * that is handed raw device pointers and has no allocator of its own, or a
 * serving loop that owns every byte of device memory from start-up and forbids
 * later cudaMalloc (which can synchronise the device, fail under a fixed
 * budget, or fragment a carefully sized pool).
 *
 * Arguments, layout, results and errors are those of paged_decode_attention;
 * the split-context scratch lives instead in a file-scope device array of
 * PKV_STATIC_WORKSPACE_BYTES that every GPU which loads the library holds
 * until the process exits. A call whose split needs more than that returns
 * PKV_ERR_WORKSPACE and launches nothing (a larger partition_tokens needs
 * less scratch). The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *
 * The first call on a device looks up the array's device address with that
 * device current and caches it; make that first call before any stream
 * capture. All calls share the one array, laid out like any decode
 * workspace (see PKV_DECODE_COUNTER_BYTES), and it keeps the last call's
 * contents: its counter header starts at zero when the library loads and
 * every call that completes without a device error leaves it zero, whatever
 * path (persistent or split grid) and shape the calls before it took; the
 * partial states after it need no clearing, because a call writes every state
 * it reads. After a call that raised PKV_DEVERR_TIMEOUT the header may hold
 * stale counts: no entry point clears it, so such a process should stop
 * using this call. Calls that
 * overlap on the GPU (different streams, or different host threads, without
 * ordering between them) race on the array: order them, or use
 * paged_decode_attention with separate workspaces.
 */
int paged_decode_attention_static_workspace(void *out, const void *q, const void *k_cache, const void *v_cache,
                                            const int32_t *block_tables, const int32_t *context_lens, float scale,
                                            int num_kv_heads, int num_seqs, int num_q_heads, int head_dim,
                                            int max_blocks_per_seq, int num_blocks, int max_context_len,
                                            pkv_dtype dtype, int partition_tokens, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
