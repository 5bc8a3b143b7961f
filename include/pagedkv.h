/*
 * pagedkv.h -- C ABI of the GB300 paged KV cache library (libpagedkv.so).
 *
 * The library implements the data-parallel hot path of PagedAttention
 * decoding, as described by the web pages on vLLM's PagedAttention:
 *
 *  [P1] "vLLM 高性能大语言模型推理引擎深度技术评估与分布式架构展望", sections
 *       "PagedAttention 内存管理与核心数据结构" (KV split into fixed-size
 *       physical blocks), "逻辑块到物理块的映射转换" (block tables; the kernel
 *       walks the physical-block mapping and gathers K/V in place), and
 *       "束搜索与并行采样的三大调度原语" (fork / append with copy-on-write / free).
 *  [P2] openEuler essay on vLLM, section "PagedAttention：把操作系统的分页搬上
 *       GPU" (block table indirection; split of long contexts into
 *       partitions, grid (heads, seqs, partitions)).
 *  [P3] "vLLM：大语言模型推理与服务库", section 4.2 (physical block, block table,
 *       block pool with an O(1) free list), 4.3 (allocate on demand when the
 *       last block is full, then update the table and write the KV) and 4.4
 *       (PagedAttention kernel: inputs q, k_cache, v_cache, block_tables,
 *       context lengths; q.K -> softmax -> weighted sum of V; 16-byte
 *       vectorised coalesced loads, shared-memory staging).
 *  [P4] "vLLM 深度解析：从 PagedAttention 到生产部署", sections "PagedAttention
 *       的解法" (block table example) and "Prefix Caching 与 Copy-on-Write".
 *
 * Conventions for every call below.
 *  - Device pointers are CUDA global-memory addresses owned by the caller
 *    (typically torch tensors).  The library never allocates or frees device
 *    memory and keeps no pointer after a call returns.
 *  - Every device pointer must be 16-byte aligned.
 *  - GPU calls are asynchronous on the given stream (0 = legacy default
 *    stream) and return after enqueueing; ordering between calls is the
 *    stream order the caller chooses.
 *  - Arguments are validated on the host before any launch: a bad shape,
 *    size, null pointer or misalignment returns PKV_ERR_INVALID and launches
 *    nothing; a valid but unimplemented combination returns
 *    PKV_ERR_UNSUPPORTED.  A failed launch returns PKV_ERR_CUDA.
 *  - Data-dependent errors found on the device (a block id outside the
 *    pool, a slot outside the pool, a seq_len beyond the block table) never
 *    trap: the kernel skips the offending access and ORs a bit into a device
 *    error word that pkv_get_device_error() reads and clears.
 *  - No C++ exception crosses this interface.
 *
 * KV pool layout (part of the ABI).  K and V are two separate pools, each
 *     [num_blocks][num_kv_heads][block_size][head_size]
 * row-major in the cache element type, so the (block, kv head) tile is one
 * contiguous run of block_size*head_size elements (4 KiB for bf16 at
 * head_size 128) and one token of one head is a contiguous head_size row.
 * Token position t of a sequence lives in physical block
 * block_tables[seq][t / block_size] at offset t % block_size.
 * A slot is physical_block * block_size + offset.
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
    PKV_ERR_INVALID = 1,      /* bad argument; nothing launched / state unchanged */
    PKV_ERR_UNSUPPORTED = 2,  /* valid but not implemented (dtype, head_size, group) */
    PKV_ERR_OOM = 3,          /* host allocator has no free block; state unchanged */
    PKV_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    PKV_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required */
    PKV_ERR_NOT_FOUND = 6     /* unknown sequence id (host allocator) */
} pkv_status;

typedef enum {
    PKV_F16 = 0,       /* IEEE binary16 */
    PKV_BF16 = 1,      /* bfloat16 */
    PKV_FP8_E4M3 = 2   /* OCP E4M3FN, per-tensor scale: value = code * scale */
} pkv_dtype;

/* Bits of the device error word (pkv_get_device_error). */
#define PKV_DEVERR_BLOCK_ID   0x1u  /* block table entry outside [0, num_blocks) */
#define PKV_DEVERR_SEQ_LEN    0x2u  /* seq_len < 0 or > max_blocks_per_seq * block_size */
#define PKV_DEVERR_SLOT       0x4u  /* slot >= num_blocks * block_size */
#define PKV_DEVERR_COPY_PAIR  0x8u  /* copy pair id outside [0, num_blocks) */
#define PKV_DEVERR_TIMEOUT    0x10u /* an internal pipeline wait gave up */

/* Description of one KV pool pair (K pool and V pool share it). */
typedef struct {
    int32_t num_blocks;    /* NB >= 1 */
    int32_t block_size;    /* b; only 16 is implemented */
    int32_t num_kv_heads;  /* Hkv >= 1 */
    int32_t head_size;     /* D; 64 or 128 */
    int32_t kv_dtype;      /* pkv_dtype of the pool elements */
    float k_scale;         /* fp8 only: stored key = code * k_scale (> 0); ignored otherwise */
    float v_scale;         /* fp8 only: stored value = code * v_scale (> 0) */
} pkv_cache_desc;

/* ------------------------------------------------------------------ GPU */

/*
 * Slot-mapped append of this step's new keys and values into the paged pool
 * ([P3] 4.3 step 2: allocate a block when the last is full -> update the
 * block table -> write the KV; [P1] prefill/decode paragraph: each decode
 * step appends the new token's KV vector).
 *
 * k, v: device [num_tokens][num_kv_heads][head_size] in in_dtype.  in_dtype
 *   equals the cache dtype, or for an fp8 cache is PKV_BF16 or PKV_F16.
 * slot_mapping: device int64 [num_tokens]; slot < 0 skips the token (padding).
 *   Token t is written to block slot / b at offset slot % b of every KV
 *   head.  For an fp8 cache each element is stored as the E4M3 code nearest
 *   (ties to even, saturating at +-448) to binary32(x) / k_scale (v_scale).
 *   Two tokens with the same slot race (which one lands is unspecified).
 * k_cache, v_cache: device pools in the layout above, written in place.
 * A slot >= num_blocks * b sets PKV_DEVERR_SLOT and that token is skipped.
 * num_tokens == 0 is a no-op.
 */
pkv_status pkv_paged_kv_append(const void* k, const void* v, int32_t in_dtype, int32_t num_tokens,
                               const int64_t* slot_mapping, void* k_cache, void* v_cache,
                               const pkv_cache_desc* desc, void* stream);

/*
 * Block copy behind copy-on-write ([P4] "Prefix Caching 与 Copy-on-Write":
 * a block shared by several sequences is copied only when one of them is
 * about to modify it; [P1] append primitive).
 *
 * pairs: device int32 [num_pairs][2] = (src, dst).  Every byte of K[src]
 *   and V[src] (all KV heads, all b slots) is copied to K[dst] and V[dst].
 *   The dst ids must be distinct and no dst may be a src of another pair
 *   (the host allocator only produces such sets); otherwise the result is
 *   unspecified.  An id outside [0, num_blocks) sets PKV_DEVERR_COPY_PAIR
 *   and skips the pair.  Enqueue before pkv_paged_kv_append of the same
 *   step so the appended token lands in the private copy.
 * num_pairs == 0 is a no-op.
 */
pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                           const int32_t* pairs, int32_t num_pairs, void* stream);

/*
 * Block swap between the device pool and a host pool, for preemption by
 * swapping ([P1] scheduling section: under memory pressure a sequence's KV
 * blocks are moved to CPU memory and brought back later instead of being
 * recomputed).
 *
 * k_host, v_host: host pools in the pool layout ([num_host_blocks][Hkv][16]
 *   [D] each), pinned and mapped into the device address space (e.g.
 *   cudaHostAlloc with cudaHostAllocMapped, or registered with
 *   cudaHostRegisterMapped); otherwise PKV_ERR_INVALID.  The copy runs as
 *   one kernel that reads or writes host memory directly.
 * pairs: device int32 [num_pairs][2] = (device block, host block).
 * direction 0 copies device -> host (swap out), 1 host -> device (swap in).
 *   Every byte of both pools' blocks is copied.  Destination blocks must be
 *   distinct.  An id out of range sets PKV_DEVERR_COPY_PAIR and skips the
 *   pair.  The host data is complete once the stream reaches this point.
 */
pkv_status pkv_swap_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* desc, void* k_host, void* v_host,
                           int32_t num_host_blocks, const int32_t* pairs, int32_t num_pairs, int32_t direction,
                           void* stream);

/*
 * Bytes of device workspace pkv_paged_attention_decode needs for these sizes
 * (split-K partials: per (seq, query head, partition) a running max, a sum
 * and a normalised head_size-vector, all fp32).  partition_tokens = 0 asks
 * for the size the automatic choice can need (its largest case).
 * Returns 0 on invalid sizes.
 */
size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                                  int32_t max_seq_len, int32_t partition_tokens);

/*
 * Decode (single-query) attention over the paged pool ([P3] 4.4: inputs q,
 * k_cache, v_cache, block_tables, context lengths; per query walk the block
 * table, q.K -> softmax -> weighted sum of V; [P1] "逻辑块到物理块的映射转换"
 * step 4; [P2] partitions of long contexts).
 *
 * For every sequence s and query head i (KV head h = i / (num_q_heads /
 * num_kv_heads)):
 *     out[s][i] = sum_{t < seq_lens[s]} softmax_t(scale * q[s][i] . K_t) V_t
 * with K_t, V_t read from block block_tables[s][t / b], offset t % b, head h
 * (for fp8 pools multiplied by k_scale / v_scale).  Accumulation is fp32;
 * out is rounded once to q_dtype.  seq_lens[s] == 0 gives a zero row.
 *
 * q: device [num_seqs][num_q_heads][head_size] in q_dtype (PKV_F16 or
 *   PKV_BF16; for f16/bf16 pools it must equal the pool dtype).
 * block_tables: device int32 [num_seqs][max_blocks_per_seq]; entries past a
 *   sequence's last block are never read.
 * seq_lens: device int32 [num_seqs]; max_seq_len (host) must be >= every
 *   entry (it sizes the launch).  An entry that is negative or beyond
 *   min(max_blocks_per_seq * b, max_seq_len rounded up to whole partitions)
 *   sets PKV_DEVERR_SEQ_LEN and is clamped into that range.
 * out: device [num_seqs][num_q_heads][head_size] in q_dtype.
 * partition_tokens: tokens per split-K partition (a positive multiple of
 *   the block size), or 0 to let the library choose from the sizes and the
 *   SM count.  When a sequence spans more than one partition its partials go
 *   to the workspace and a log-sum-exp merge kernel finishes the row.
 * workspace: device buffer of at least
 *   pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_size,
 *   max_seq_len, partition_tokens) bytes (may be NULL when that is 0);
 *   otherwise PKV_ERR_WORKSPACE.
 * Implemented: block_size 16; head_size 64 or 128; num_q_heads / num_kv_heads
 *   in {1, 2, 4, 8}; pools f16, bf16 or fp8 E4M3.
 */
pkv_status pkv_paged_attention_decode(const void* q, int32_t q_dtype, int32_t num_seqs,
                                      int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                      const pkv_cache_desc* desc, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                      int32_t max_seq_len, float scale, void* out, void* workspace,
                                      size_t workspace_bytes, int32_t partition_tokens, void* stream);

/*
 * Decode attention that allocates nothing and needs no workspace argument.
 * The pages have no counterpart to this call: it exists for callers that
 * cannot hand the library a device buffer -- a plug-in inside a framework
 * that owns all device memory and exposes no allocator, or a latency-
 * critical loop that must not call cudaMalloc (which can synchronise the
 * device).  Arguments and results are those of pkv_paged_attention_decode
 * without workspace / workspace_bytes.
 *
 * The split-K scratch is a 32 MiB array inside the library (held on every
 * GPU that loads it until the process exits).  A call whose scratch need,
 * pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_size, max_seq_len,
 * P) for the partition size P actually used, exceeds 32 MiB returns
 * PKV_ERR_WORKSPACE and launches nothing.  Every call looks up the array's
 * device address in the current context (cudaGetSymbolAddress, which
 * allocates nothing); the first lookup on a device may load the library's
 * device code, so make the first call on a device before any stream
 * capture.  No cudaMalloc, cudaFree or allocating
 * routine is called.  All calls share the one array and it keeps whatever
 * the last call left there; nothing in it needs to start at zero (every
 * partial the merge reads is written first in the same call).  Calls whose
 * kernels may overlap on the GPU (different streams without ordering) race
 * on the array and give undefined results.
 */
pkv_status pkv_paged_attention_decode_noalloc(const void* q, int32_t q_dtype, int32_t num_seqs,
                                              int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                              const pkv_cache_desc* desc, const int32_t* block_tables,
                                              int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                              int32_t max_seq_len, float scale, void* out,
                                              int32_t partition_tokens, void* stream);

/*
 * One decode step's copy-on-write copies, append and attention in one
 * launch: the same result as
 *   pkv_copy_blocks(pairs (cow_src[s], the block of slot_mapping[s]) ...),
 *   pkv_paged_kv_append(k_new, v_new, in_dtype, num_seqs, slot_mapping, ...),
 *   pkv_paged_attention_decode(q, ...),
 * with one new token per batch row (row s of k_new / v_new, [num_seqs]
 * [Hkv][head_size]; slot_mapping[s] < 0: row s appends nothing).  Each
 * decode CTA that covers a row's last position (seq_lens[s] - 1) writes its
 * KV head's part of that token before reading the pool, which saves the
 * append kernel's launch and its pass over the slot rows.  slot_mapping[s]
 * must be the slot of position seq_lens[s] - 1 in row s's block table (what
 * the allocator's append returned); otherwise PKV_DEVERR_SLOT is set and
 * nothing is written for that row.  in_dtype: the cache's 16-bit type, or
 * f16 / bf16 for an fp8 cache (encoded as pkv_paged_kv_append does); an fp8
 * input returns PKV_ERR_UNSUPPORTED.
 * cow_src (device int32 [num_seqs], may be NULL): for a row whose append
 *   took a fresh copy of a shared partial block (the allocator's copy-on-
 *   write pair (src, dst) with dst the block of slot_mapping[s]), src; else
 *   -1.  The CTA copies its head's tile of src into dst, except the appended
 *   row, before writing the row (other sharers write only that row of src,
 *   in place).  An src outside the pool, or equal to dst, sets
 *   PKV_DEVERR_COPY_PAIR and nothing is written for the row.  Other
 *   copy-on-write pairs (not into an appending row's last block) must be
 *   copied with pkv_copy_blocks first.  Other arguments, errors and
 *   workspace as for pkv_paged_attention_decode.
 * work_units, num_work_units (device int32, may be NULL / 0): the order in
 *   which the CTAs start.  A CTA covers unit u = s * NP + partition (NP =
 *   ceil(max_seq_len / P), P the partition size this call uses) for one KV
 *   head; the list's units run in order, each for every KV head.  NULL: the
 *   grid order (partition, KV head, sequence).  pkv_decode_plan writes every
 *   unit of a batch longest first.  A list must hold every unit of the batch
 *   (a row whose units are missing is left undefined, and so is its append);
 *   a unit outside [0, num_seqs * NP) sets PKV_DEVERR_SEQ_LEN and is skipped.
 *   With a list and partition_tokens 0 the automatic partition size has no
 *   2048-token cap (long CTAs start first, so it only adds merge work);
 *   pkv_decode_plan with partition_tokens 0 uses that same size.
 */
pkv_status pkv_paged_attention_decode_append(const void* k_new, const void* v_new, int32_t in_dtype,
                                             const int64_t* slot_mapping, const int32_t* cow_src,
                                             const void* q, int32_t q_dtype,
                                             int32_t num_seqs, int32_t num_q_heads, void* k_cache, void* v_cache,
                                             const pkv_cache_desc* desc, const int32_t* block_tables,
                                             int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                             int32_t max_seq_len, float scale, void* out, void* workspace,
                                             size_t workspace_bytes, int32_t partition_tokens,
                                             const int32_t* work_units, int32_t num_work_units, void* stream);

/*
 * Host work plan for pkv_paged_attention_decode_append (plain C++, no GPU
 * work; with partition_tokens 0 it asks the device for its SM count, as the
 * decode's automatic choice does).  Writes to units[0 .. *num_units) every
 * unit s * NP + partition of the batch (every partition of every row, one
 * for a zero-length row), sorted by its tokens, longest first (ties: unit
 * order), so that the last CTAs to start are the shortest
 * (longest-processing-time-first list scheduling).  seq_lens: HOST copy of
 * the decode call's array; num_kv_heads, max_seq_len, partition_tokens: as
 * passed to it.  *num_units always receives the count; PKV_ERR_WORKSPACE if
 * it exceeds units_cap (nothing written).  A length outside [0,
 * max_seq_len] returns PKV_ERR_INVALID.
 */
pkv_status pkv_decode_plan(const int32_t* seq_lens, int32_t num_seqs, int32_t num_kv_heads, int32_t max_seq_len,
                           int32_t partition_tokens, int32_t* units, int32_t units_cap, int32_t* num_units);

/*
 * Shared-prefix ("cascade") decode attention: the same function as
 * pkv_paged_attention_decode, computed so that blocks shared by a group of
 * sequences are read once per group rather than once per sequence.  Shared
 * blocks arise from fork, prefix sharing and parallel sampling ([P4]
 * "Prefix Caching 与 Copy-on-Write"; [P1] "束搜索与并行采样的三大调度原语").
 * Each member's attention is split into the group's shared leading blocks
 * (all member query heads attend to them together, on the tensor cores) and
 * the member's own remaining tokens; the two are combined exactly by the
 * log-sum-exp merge.
 *
 * Arguments as for pkv_paged_attention_decode, plus the groups (device
 * int32 arrays, as produced by pkv_alloc_prefix_groups):
 *   seq_group[num_seqs]: group of each batch row, or -1;
 *   group_blocks[num_groups]: leading blocks shared by every member -- the
 *     first group_blocks[g] entries of every member's block table must be
 *     identical and each of those blocks full (16 valid tokens);
 *   group_offsets[num_groups + 1], group_members[]: CSR list of the batch
 *     rows of each group;
 *   max_group_members, max_group_blocks: host bounds of the two (size the
 *     launch).
 * workspace must hold pkv_decode_cascade_workspace_bytes(...) bytes, plus,
 * for an fp8 pool, pkv_decode_cascade_staging_bytes(...) more: there the
 * prefix pass first copies every group's shared blocks once into q's 16-bit
 * type (exact: every E4M3 value is an f16 and a bf16 value) in the
 * workspace, after the partials at the next 256-byte boundary, and reads
 * that copy, with k_scale in the score scale and v_scale on the output.
 * scale must be finite and > 0 (else PKV_ERR_INVALID).
 * Implemented for f16 / bf16 pools (q of the same type) and fp8 E4M3 pools
 * (q f16 or bf16; k_scale, v_scale > 0), head_size 64 or 128, num_q_heads /
 * num_kv_heads in {1, 2, 4, 8}.  The own tokens use the kernels plain decode
 * uses.  A member index or block count out of range sets
 * PKV_DEVERR_SEQ_LEN and the offending rows are skipped.
 * Streams: every launch goes to `stream`.  The own-token decode is a
 * programmatic dependent of the prefix pass and runs beside it; one extra
 * CTA of its grid waits for the prefix pass, and the merge waits for that
 * grid.  The call is ordered on `stream` like any other and can be captured
 * into a CUDA graph.  num_seqs above 65534 returns PKV_ERR_UNSUPPORTED.
 */
pkv_status pkv_paged_attention_decode_cascade(const void* q, int32_t q_dtype, int32_t num_seqs,
                                              int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                              const pkv_cache_desc* desc, const int32_t* block_tables,
                                              int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                              int32_t max_seq_len, const int32_t* seq_group,
                                              const int32_t* group_blocks, const int32_t* group_offsets,
                                              const int32_t* group_members, int32_t num_groups,
                                              int32_t max_group_members, int32_t max_group_blocks, float scale,
                                              void* out, void* workspace, size_t workspace_bytes,
                                              int32_t partition_tokens, void* stream);

/* Workspace bytes of pkv_paged_attention_decode_cascade (0 on invalid sizes;
 * partition_tokens = 0 sizes for the automatic choice's largest case). */
size_t pkv_decode_cascade_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                                          int32_t max_seq_len, int32_t partition_tokens,
                                          int32_t max_group_blocks);

/* Extra workspace bytes of pkv_paged_attention_decode_cascade over an fp8
 * pool (the groups' 16-bit prefix copy and its block table): 0 for f16 / bf16
 * pools, for no groups, or on invalid sizes.  The whole workspace is then
 * round_up(pkv_decode_cascade_workspace_bytes(...), 256) + this. */
size_t pkv_decode_cascade_staging_bytes(int32_t kv_dtype, int32_t num_seqs, int32_t max_blocks_per_seq,
                                        int32_t num_groups, int32_t max_group_blocks, int32_t num_kv_heads,
                                        int32_t head_size);

/*
 * Paged (chunked) prefill attention, causal, on the tensor cores.  Prefill
 * processes a prompt's tokens together; chunked prefill cuts a long prompt
 * into chunks that run in successive iterations, each attending to the KV
 * of the earlier chunks already in the pool ([P1] "PagedAttention 内存管理与
 * 核心数据结构" and the scheduling section on chunked prefill).
 *
 * q, out: [num_tokens][num_q_heads][head_size] (q_dtype); the new tokens of
 *   all sequences packed back to back.
 * query_start: device int32 [num_seqs + 1]: sequence s owns rows
 *   [query_start[s], query_start[s+1]) of q and out, n_s rows in all.
 * seq_lens: device int32 [num_seqs]: tokens of sequence s in the pool,
 *   counting its n_s new ones, whose K/V must already be appended (the last
 *   n_s positions).  Row j of sequence s sits at position seq_lens[s] - n_s + j
 *   and attends to positions 0..that position:
 *     out[query_start[s] + j][i] = sum_{t <= pos} softmax_t(scale * q.k_t) v_t
 *   with query head i reading KV head i / (num_q_heads / num_kv_heads).
 * max_query_len: host bound on every n_s (sizes the grid); a larger n_s sets
 *   PKV_DEVERR_SEQ_LEN and its rows past the bound may be left unwritten.
 * Rows of out outside every sequence's range are not written.
 * scale must be finite and > 0 (else PKV_ERR_INVALID).
 * Implemented for f16 / bf16 pools with q of the same type, fp8 E4M3 pools
 * with f16 or bf16 q, head_size 64 or 128, num_q_heads / num_kv_heads in
 * {1, 2, 4, 8}, and at most 2^31 - 1 CTAs (ceil(max_query_len * G / 256) *
 * num_kv_heads * num_seqs, G = num_q_heads / num_kv_heads); others return
 * PKV_ERR_UNSUPPORTED.  out has q's type.
 * fp8 pools: the keys and values are desc->k_scale * code and
 * desc->v_scale * code (both finite and > 0, else PKV_ERR_INVALID).  A first
 * kernel, on the same stream, copies the blocks the batch reaches (the first
 * ceil(seq_lens[s] / 16) entries of each block-table row) into 16-bit
 * blocks of q's type in the workspace -- exact, since every E4M3 value is an
 * f16 and a bf16 value -- and the attention pass reads that copy.
 * workspace, workspace_bytes: device memory of at least
 * pkv_prefill_workspace_bytes(desc->kv_dtype, num_seqs, num_kv_heads,
 * head_size, max_blocks_per_seq) bytes, 16-byte aligned, owned by the
 * caller and not read or written by any other work until this call's
 * kernels finish in stream order (else PKV_ERR_WORKSPACE).  16-bit pools
 * need none (NULL, 0).  num_seqs * max_blocks_per_seq * num_kv_heads * 16
 * must stay below 2^31 for an fp8 pool (else PKV_ERR_UNSUPPORTED).
 * work_units, num_work_units: the order in which units are taken.  A unit
 * u = s * nq + qt (sequence s, its query rows [qt * r, (qt + 1) * r) with
 * r = 256 / G tokens, nq = ceil(max_query_len / r)) runs for one KV head.
 * Null (num_work_units 0): every unit, each (sequence, KV head) from its last
 * rows down.  Otherwise a device int32 array of num_work_units units, each
 * run for every KV head in that order, and only those; pkv_prefill_plan
 * writes the batch's units longest causal key range first.  A unit outside
 * [0, num_seqs * nq) sets PKV_DEVERR_SEQ_LEN and is skipped.
 * The attention kernel is persistent: one CTA per SM takes (unit, KV head)
 * pairs in list order from a device counter as it finishes the one before.
 * The library owns 1024 such counters and hands one to each call in turn;
 * the kernel returns its counter to zero when it ends.  Calls that run at
 * the same time (other streams, or two different captured graphs) must
 * not hold the same counter, i.e. must be fewer than 1024 calls apart.
 * Inconsistent query_start / seq_lens (n_s < 0,
 * n_s > seq_lens[s], past num_tokens or the block table) set
 * PKV_DEVERR_SEQ_LEN and the sequence is skipped; a block id outside the pool
 * sets PKV_DEVERR_BLOCK_ID (for an fp8 pool the block reads as zeros).
 */
pkv_status pkv_paged_attention_prefill(const void* q, int32_t q_dtype, int32_t num_tokens, int32_t num_q_heads,
                                       int32_t num_seqs, const int32_t* query_start, int32_t max_query_len,
                                       const void* k_cache, const void* v_cache, const pkv_cache_desc* desc,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, const int32_t* work_units,
                                       int32_t num_work_units, float scale, void* out, void* workspace,
                                       size_t workspace_bytes, void* stream);

/*
 * Workspace bytes pkv_paged_attention_prefill needs: 0 for an f16 / bf16
 * pool; for an fp8 E4M3 pool 2 * 2 * num_seqs * max_blocks_per_seq *
 * num_kv_heads * 16 * head_size bytes of 16-bit block copies plus a 4-byte
 * block-table entry per (sequence, block), each part rounded up to 256 bytes.
 * Returns 0 for a negative count or a non-positive num_kv_heads / head_size.
 */
size_t pkv_prefill_workspace_bytes(int32_t kv_dtype, int32_t num_seqs, int32_t num_kv_heads, int32_t head_size,
                                   int32_t max_blocks_per_seq);

/*
 * Host work plan for pkv_paged_attention_prefill (plain C++, no GPU):
 * writes to units[0 .. *num_units) every non-empty unit s * nq + qt of the
 * batch (see work_units above), sorted by the causal key range of the
 * unit's last query row, longest first (ties: sequence, then query tile,
 * ascending), so that the last units to start are the shortest.  The batch
 * may mix chunks over contexts of any length; scheduling long units first
 * keeps the tail short.
 * query_start [num_seqs + 1], seq_lens [num_seqs]: HOST copies of the
 *   prefill call's arrays.  max_query_len, num_q_heads, num_kv_heads: as
 *   passed to the prefill call.
 * *num_units always receives the count; PKV_ERR_WORKSPACE if it exceeds
 * units_cap (nothing written).  Inconsistent sequences (n_s < 0, n_s >
 * max_query_len, n_s > seq_lens[s], query_start[s] < 0) return
 * PKV_ERR_INVALID; a head ratio outside {1, 2, 4, 8} PKV_ERR_UNSUPPORTED.
 */
pkv_status pkv_prefill_plan(const int32_t* query_start, const int32_t* seq_lens, int32_t num_seqs,
                            int32_t num_q_heads, int32_t num_kv_heads, int32_t max_query_len, int32_t* units,
                            int32_t units_cap, int32_t* num_units);

/*
 * Partition size the automatic choice (partition_tokens = 0) would use for
 * these sizes on the current device, or a negative pkv_status on error.
 * planned != 0: the size for a launch with a work list (no 2048-token cap,
 * see pkv_paged_attention_decode_append); 0: grid order (every other decode
 * entry point).
 */
int32_t pkv_decode_auto_partition(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_size, int32_t max_seq_len, int32_t planned);

/*
 * Decode kernel selection for subsequent pkv_paged_attention_decode calls
 * (process-wide): 0 = automatic (tensor-core kernel when num_q_heads /
 * num_kv_heads >= 2 and head_size == 128, CUDA-core kernel otherwise),
 * 1 = always the CUDA-core kernel, 2 = always the tensor-core kernel (a call
 * it cannot serve then returns PKV_ERR_UNSUPPORTED).  Both compute the same
 * function; the switch exists so each can be tested and timed.
 * PKV_ERR_INVALID for another value.
 */
pkv_status pkv_set_decode_path(int32_t path);
int32_t pkv_get_decode_path(void);

/*
 * Reads and clears the device error word of the current device (the OR of
 * PKV_DEVERR_* bits set by every kernel since the last call).  Synchronises
 * the given stream first.  *flags receives the bits.
 */
pkv_status pkv_get_device_error(uint32_t* flags, void* stream);

/*
 * Check of the failure path of the kernels' bounded waits (no counterpart on
 * the pages, which describe no device-side failure handling).  Enqueues one
 * 32-thread CTA on `stream` that waits on a shared-memory mbarrier nothing
 * ever arrives at and no copy feeds, with the wait routine of the decode
 * kernels' copy pipelines (which = 0: at most 2^14 polls of up to 100 us
 * each) or of the prefill's tensor-core pipeline (which = 1: 2 s of the
 * global timer).  The wait gives up, PKV_DEVERR_TIMEOUT is set in the device
 * error word and the kernel returns, leaving the context usable.  Expect the
 * launch to take up to about 2 s.  PKV_ERR_INVALID for another `which`.
 */
pkv_status pkv_check_wait_timeout(int32_t which, void* stream);

/* Static description of a status code (never NULL). */
const char* pkv_status_string(int32_t status);

/* Library version, "major.minor.patch". */
const char* pkv_version(void);

/* -------------------------------------------------------- host allocator */

/*
 * Host-side block allocator: plain C++, host memory only (it hands out block
 * ids; the caller owns the device pool they index).
 *
 * [P3] 4.2 "Block Pool": a pool split into fixed-size blocks, a free list,
 *   O(1) allocate (take the last free id; fail when empty) and O(1) free.
 * [P3] 4.3: a sequence gets a new block only when its last block is full.
 * [P1] "束搜索与并行采样的三大调度原语": fork copies the parent's block table
 *   (same physical ids, reference count +1); append on a shared block uses
 *   copy-on-write; free decrements reference counts and returns blocks
 *   whose count reaches zero to the free list at once.
 * [P4] "Prefix Caching 与 Copy-on-Write": shared blocks carry a reference
 *   count > 1 and are copied only when modified.
 *
 * Readings: the free list is a stack; copy-on-write happens when the block
 * the next token goes to is partial AND shared; a sequence's blocks are
 * released last block first.  Every call either succeeds completely or
 * returns an error with the allocator unchanged.  The handle is not
 * thread-safe: one thread at a time per handle.
 */
typedef struct pkv_alloc pkv_alloc;

/* free_order: NULL (ids 0..num_blocks-1, so block num_blocks-1 is taken
 * first) or a permutation of 0..num_blocks-1 whose LAST entry is taken
 * first.  Returns NULL on invalid arguments. */
pkv_alloc* pkv_alloc_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order);
void pkv_alloc_destroy(pkv_alloc* a);

/* New sequence holding num_tokens >= 0 tokens (ceil(num_tokens / b) blocks). */
pkv_status pkv_alloc_seq_new(pkv_alloc* a, int64_t seq_id, int32_t num_tokens);
/* child gets parent's table and length; every block's count +1. */
pkv_status pkv_alloc_fork(pkv_alloc* a, int64_t parent_id, int64_t child_id);
/* Reserve the slot for one more token of seq_id.  *slot receives it.  When
 * the token would go into a partial block shared with another sequence, a
 * private block is allocated, the table is repointed, and (*cow_src,
 * *cow_dst) receive the pair to pass to pkv_copy_blocks; otherwise both are
 * -1.  cow_src / cow_dst may be NULL only if the caller does not care. */
pkv_status pkv_alloc_append_slot(pkv_alloc* a, int64_t seq_id, int64_t* slot, int32_t* cow_src,
                                 int32_t* cow_dst);
/* Grow seq_id by num_tokens tokens without returning slots (prefill of new
 * tokens).  PKV_ERR_INVALID if that would write into a shared partial block. */
pkv_status pkv_alloc_seq_extend(pkv_alloc* a, int64_t seq_id, int32_t num_tokens);
/* Release every block of seq_id and forget it. */
pkv_status pkv_alloc_free(pkv_alloc* a, int64_t seq_id);

/* One decode step for a batch: append_slot for seq_ids[0..n) in order.
 * slots[i] receives row i's slot (or -1 where seq_ids[i] < 0: padding row);
 * pairs receives the copy-on-write pairs ([*num_pairs][2], capacity
 * pairs_cap >= n).  All or nothing: on any error the allocator is restored
 * to its state before the call. */
pkv_status pkv_alloc_append_batch(pkv_alloc* a, const int64_t* seq_ids, int32_t n, int64_t* slots,
                                  int32_t* pairs, int32_t pairs_cap, int32_t* num_pairs);
/* Chunked prefill: reserve counts[i] new token slots for sequence seq_ids[i]
 * (each sequence at most once; counts[i] >= 0), in order, as append_slot
 * would one token at a time.  slots (capacity slots_cap >= sum counts)
 * receives the slots sequence after sequence; pairs receives the
 * copy-on-write pairs ([*num_pairs][2], capacity pairs_cap >= n: only a
 * sequence's first new token can land in a shared partial block).  All or
 * nothing, like append_batch. */
pkv_status pkv_alloc_append_tokens(pkv_alloc* a, const int64_t* seq_ids, const int32_t* counts, int32_t n,
                                   int64_t* slots, int64_t slots_cap, int32_t* pairs, int32_t pairs_cap,
                                   int32_t* num_pairs);
/* Export padded block tables and lengths for a batch: tables is
 * [n][max_blocks] (unused entries -1), seq_lens [n]; a row whose seq_id is
 * negative gets length 0.  PKV_ERR_INVALID if a table does not fit. */
pkv_status pkv_alloc_export(const pkv_alloc* a, const int64_t* seq_ids, int32_t n, int32_t* tables,
                            int32_t max_blocks, int32_t* seq_lens);

pkv_status pkv_alloc_block_table(const pkv_alloc* a, int64_t seq_id, int32_t* out, int32_t cap,
                                 int32_t* n);
pkv_status pkv_alloc_seq_len(const pkv_alloc* a, int64_t seq_id, int64_t* n);
/* Reference count of a block (0 = free), or -1 for an id outside the pool. */
int32_t pkv_alloc_refcount(const pkv_alloc* a, int32_t block);
int32_t pkv_alloc_num_free(const pkv_alloc* a);
int32_t pkv_alloc_num_seqs(const pkv_alloc* a);
/* Groups of batch rows that share leading blocks, for cascade decode.  Rows
 * (seq_ids[i] >= 0) with at least min_blocks full blocks are bucketed by their
 * first block id; a bucket of two or more rows becomes a group whose shared
 * prefix is the longest run of identical leading block ids, counting only
 * blocks full in every member, if that run is >= min_blocks.  Outputs:
 * seq_group[n] (-1 when ungrouped), group_blocks[*num_groups],
 * group_offsets[*num_groups + 1], group_members (batch rows; capacity n),
 * the largest group and the largest prefix.  Capacities of group_blocks and
 * group_offsets: n and n + 1. */
pkv_status pkv_alloc_prefix_groups(const pkv_alloc* a, const int64_t* seq_ids, int32_t n, int32_t min_blocks,
                                   int32_t* seq_group, int32_t* group_blocks, int32_t* group_offsets,
                                   int32_t* group_members, int32_t* num_groups, int32_t* max_members,
                                   int32_t* max_blocks);
/* Swap a sequence between a device allocator and a host-block allocator
 * (a second pkv_alloc over the host pool's block ids, same block size).
 * swap_out moves seq_id from `dev` to `host`; swap_in moves it back.  One new
 * block is taken per block of the sequence, the old ones are released, and
 * pairs ([*n][2], capacity cap) receive (device block, host block) for
 * pkv_swap_blocks in either direction.  Every block of the sequence must
 * be held by it alone (refcount 1), else PKV_ERR_INVALID; PKV_ERR_OOM if
 * the target has too few free blocks.  All or nothing. */
pkv_status pkv_alloc_swap_out(pkv_alloc* dev, pkv_alloc* host, int64_t seq_id, int32_t* pairs, int32_t cap,
                              int32_t* n);
pkv_status pkv_alloc_swap_in(pkv_alloc* dev, pkv_alloc* host, int64_t seq_id, int32_t* pairs, int32_t cap,
                             int32_t* n);
/*
 * Automatic prefix caching ([P1] "基于级联哈希的缓存结构设计" and "缓存分配、
 * 触碰与驱逐闭环").  A full block is identified by its cascaded hash
 *   hash(parent hash, the block's token ids, extra hashes)
 * (the parent of the first block is 0; extra hashes carry whatever else fixes
 * the block's KV, e.g. a LoRA adapter id; a per-request cache salt joins the
 * first block's extra hashes only, so different salts never share blocks).
 * The hash is 64-bit FNV-1a over the little-endian bytes of: parent (8),
 * token count (4), each token id (4), extra count (4), each extra (8).
 *
 * Allocator side: commit registers a sequence's full blocks under their
 * hashes; lookup counts the leading hashes of a prompt found in the table
 * (get_computed_blocks); seq_new_prefix touches those blocks (a reference
 * each; a block no sequence held becomes live again) and allocates the rest.
 * A committed block whose count drops to zero stays cached and evictable.
 * Allocation uses never-cached free blocks first, then evicts the cached
 * block released longest ago; a sequence's blocks are released last to
 * first, so the leaf end of a chain is evicted before its root.
 * num_free counts never-cached and evictable blocks.
 */
uint64_t pkv_block_hash(uint64_t parent_hash, const int32_t* tokens, int32_t num_tokens, const uint64_t* extras,
                        int32_t num_extras);
/* Hashes of the num_tokens / block_size full blocks of a token sequence
 * (capacity cap), the same extras for every block and *salt (if salt is not
 * NULL) added to the first block's. */
pkv_status pkv_prefix_block_hashes(const int32_t* tokens, int64_t num_tokens, int32_t block_size,
                                   const uint64_t* extras, int32_t num_extras, const uint64_t* salt,
                                   uint64_t* hashes, int64_t cap, int64_t* num_hashes);
/* Leading hashes[0..n) present in the table (no state change); -1 on a bad
 * argument. */
int32_t pkv_alloc_lookup(const pkv_alloc* a, const uint64_t* hashes, int32_t n);
/* New sequence of num_tokens tokens whose first full blocks have the given
 * hashes (num_hashes * block_size <= num_tokens): the leading hits
 * (*hit_blocks) are shared, the other blocks allocated.  All or nothing;
 * PKV_ERR_OOM if the pool cannot hold the rest. */
pkv_status pkv_alloc_seq_new_prefix(pkv_alloc* a, int64_t seq_id, const uint64_t* hashes, int32_t num_hashes,
                                    int32_t num_tokens, int32_t* hit_blocks);
/* Registers the sequence's first num_hashes blocks (all full) under the
 * given hashes once their KV is written; a block already committed keeps its
 * hash (a different one is PKV_ERR_INVALID), a hash already held by another
 * block is skipped.  *committed (may be NULL) = blocks newly registered. */
pkv_status pkv_alloc_commit(pkv_alloc* a, int64_t seq_id, const uint64_t* hashes, int32_t num_hashes,
                            int32_t* committed);
/* Cached blocks that no sequence holds (evictable). */
int32_t pkv_alloc_num_cached(const pkv_alloc* a);
/* 1 and *hash if the block is committed, 0 if not, -1 on a bad argument. */
int64_t pkv_alloc_block_hash_of(const pkv_alloc* a, int32_t block, uint64_t* hash);
/* Forgets every hash; evictable blocks become plain free blocks. */
void pkv_alloc_reset_prefix_cache(pkv_alloc* a);

/* Fault injection for tests: the k-th block allocation from now (k >= 1)
 * fails as if the pool were empty; k <= 0 disables. */
void pkv_alloc_fail_after(pkv_alloc* a, int64_t k);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
