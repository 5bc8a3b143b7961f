// pkv_cascade.cu -- shared-prefix (cascade) decode attention.
//
// When several sequences share their leading physical blocks (prefix
// sharing and parallel sampling: "vLLM 深度解析：从 PagedAttention 到生产部署",
// "Prefix Caching 与 Copy-on-Write"; "vLLM 高性能大语言模型推理引擎深度技术评估
// 与分布式架构展望", "束搜索与并行采样的三大调度原语": fork shares the parent's
// physical blocks), plain decode reads the shared blocks once per sequence.
// Cascade decode splits every member's attention into the shared part and
// its own part, which are combined exactly by the log-sum-exp merge:
//
//   1. the prefix pass (the tcgen05 attention tile of pkv_prefill.cu): for
//      each group, KV head and 1024-token prefix partition, the query heads of
//      the group's members (128 / G members x G heads per CTA, on the MMA's
//      M dimension) attend to the shared blocks, read once per CTA; partials
//      go to partition indices [0, NPP);
//   2. the regular decode kernel attends each sequence's own tokens (from
//      the end of its group's prefix), partials at indices NPP + p;
//   3. the merge kernel combines prefix and own partials of every row.
//
// The three run in this order on the caller's stream, each later one a
// programmatic dependent of the one before.  The prefix pass lets the
// own-token decode start at once (it reads the pool and writes other
// partials), so the two run side by side; one extra CTA of the decode grid
// waits for the prefix pass to complete, so the merge, which waits for the
// decode grid, sees both.  No second stream or event is involved, and the
// call can be captured into a CUDA graph.
//
// The result is the same function as pkv_paged_attention_decode.
#include <cstdint>

#include "pkv_internal.h"

namespace pkv {

namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
}  // namespace

}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_decode_cascade_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                                                     int32_t max_seq_len, int32_t partition_tokens,
                                                     int32_t max_group_blocks) {
    if (num_seqs < 0 || num_q_heads <= 0 || head_size <= 0 || max_seq_len < 0 || partition_tokens < 0 ||
        max_group_blocks < 0 || partition_tokens % kBlockSize)
        return 0;
    const int64_t P = partition_tokens > 0 ? partition_tokens : kAutoMinPartition;
    const int64_t NP = prefix_partitions(max_group_blocks) + (max_seq_len > 0 ? cdiv(max_seq_len, P) : 1);
    return partials_bytes(num_seqs, num_q_heads, head_size, NP);
}

extern "C" size_t pkv_decode_cascade_staging_bytes(int32_t kv_dtype, int32_t num_seqs, int32_t max_blocks_per_seq,
                                                   int32_t num_groups, int32_t max_group_blocks, int32_t num_kv_heads,
                                                   int32_t head_size) {
    if (kv_dtype != PKV_FP8_E4M3 || num_seqs <= 0 || max_blocks_per_seq <= 0 || num_groups <= 0 ||
        max_group_blocks <= 0 || num_kv_heads <= 0 || head_size <= 0)
        return 0;
    return static_cast<size_t>(
        cascade_stage_layout(num_seqs, max_blocks_per_seq, num_groups, max_group_blocks, num_kv_heads, head_size)
            .bytes);
}

extern "C" pkv_status pkv_paged_attention_decode_cascade(
    const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads, const void* k_cache, const void* v_cache,
    const pkv_cache_desc* d, const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
    int32_t max_seq_len, const int32_t* seq_group, const int32_t* group_blocks, const int32_t* group_offsets,
    const int32_t* group_members, int32_t num_groups, int32_t max_group_members, int32_t max_group_blocks, float scale,
    void* out, void* workspace, size_t ws_bytes, int32_t partition_tokens, void* stream) {
    // ---- validation (host, before any launch)
    if (!d || num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0 ||
        partition_tokens < 0 || num_groups < 0 || max_group_members < 0 || max_group_blocks < 0)
        return PKV_ERR_INVALID;
    if (d->num_blocks <= 0 || d->num_kv_heads <= 0 || d->head_size <= 0 || d->block_size <= 0)
        return PKV_ERR_INVALID;
    if (d->kv_dtype < PKV_F16 || d->kv_dtype > PKV_FP8_E4M3) return PKV_ERR_INVALID;
    if (q_dtype != PKV_F16 && q_dtype != PKV_BF16) return PKV_ERR_INVALID;
    if (num_q_heads % d->num_kv_heads || !(scale > 0.f) || scale > 3.0e38f) return PKV_ERR_INVALID;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * d->block_size)
        return PKV_ERR_INVALID;
    if (max_group_blocks > max_blocks_per_seq || partition_tokens % kBlockSize) return PKV_ERR_INVALID;
    const bool fp8 = d->kv_dtype == PKV_FP8_E4M3;
    if (!fp8 && q_dtype != d->kv_dtype) return PKV_ERR_UNSUPPORTED;
    if (d->block_size != kBlockSize || (d->head_size != 64 && d->head_size != 128)) return PKV_ERR_UNSUPPORTED;
    if (fp8 && !(d->k_scale > 0.f && d->v_scale > 0.f)) return PKV_ERR_INVALID;
    const int G = num_q_heads / d->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65534 || d->num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;  // + the decode's join layer
    if (num_seqs == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out || !seq_group) return PKV_ERR_INVALID;
    if (num_groups > 0 && (!group_blocks || !group_offsets || !group_members)) return PKV_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PKV_ERR_INVALID;
    const int64_t pool_rows = static_cast<int64_t>(d->num_blocks) * d->num_kv_heads * kBlockSize;
    if (pool_rows > 0x7fffffff) return PKV_ERR_UNSUPPORTED;

    const int P = partition_tokens > 0 ? partition_tokens : auto_partition(num_seqs, d->num_kv_heads, max_seq_len, false);
    const int npp = num_groups > 0 ? prefix_partitions(max_group_blocks) : 0;
    const int64_t nps = max_seq_len > 0 ? cdiv(max_seq_len, P) : 1;
    const int64_t NP = npp + nps;
    const int64_t row_chunks = cdiv(static_cast<int64_t>(max_group_members) * G, 128);  // one 128-row Q tile per CTA
    if (NP > 0x7fffffff || static_cast<int64_t>(num_groups) * row_chunks > 65535) return PKV_ERR_UNSUPPORTED;
    const size_t part_bytes = partials_bytes(num_seqs, num_q_heads, d->head_size, NP);
    // an fp8 pool's staged 16-bit prefix copy follows the partials
    const size_t stage_off = (part_bytes + 255) / 256 * 256;
    const int64_t stage_rows = static_cast<int64_t>(num_groups) * max_group_blocks * d->num_kv_heads * kBlockSize;
    const bool staged = fp8 && num_groups > 0 && max_group_blocks > 0 && row_chunks > 0;
    if (staged && stage_rows > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
    const size_t need =
        staged ? stage_off + static_cast<size_t>(cascade_stage_layout(num_seqs, max_blocks_per_seq, num_groups,
                                                                      max_group_blocks, d->num_kv_heads, d->head_size)
                                                     .bytes)
               : part_bytes;
    if (!workspace || ws_bytes < need || !aligned16(workspace)) return PKV_ERR_WORKSPACE;
    unsigned int* err = error_word();
    if (!err) return PKV_ERR_CUDA;

    DecodeParams p{};
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.out = out;
    p.S = num_seqs;
    p.Hq = num_q_heads;
    p.Hkv = d->num_kv_heads;
    p.D = d->head_size;
    p.NB = d->num_blocks;
    p.MB = max_blocks_per_seq;
    p.P = P;
    p.NP = static_cast<int32_t>(NP);
    const float log2e = 1.4426950408889634f;
    p.qk_scale = scale * log2e * (fp8 ? d->k_scale : 1.f);
    p.v_scale = fp8 ? d->v_scale : 1.f;
    p.err = err;
    p.seq_group = seq_group;
    p.group_blocks = group_blocks;
    p.part_base = npp;
    p.cascade = 1;
    partials_layout(p, workspace);

    // The own-token decode: the kernels plain decode would use (tensor cores
    // for grouped heads at head_size 128, CUDA cores otherwise), on the pool
    // itself.
    const bool use_mma = d->head_size == 128 && G >= 2;
    const int eb = fp8 ? 1 : 2;
    CUtensorMap tk, tv, tq, tpk, tpv;
    if ((use_mma && (!encode_pool_map(&tk, k_cache, eb, pool_rows, d->head_size) ||
                     !encode_pool_map(&tv, v_cache, eb, pool_rows, d->head_size))) ||
        !encode_token_head_map(&tq, q, d->head_size, num_q_heads, num_seqs, G, 1))
        return PKV_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    const bool prefix = npp > 0 && row_chunks > 0;
    // 1. shared prefixes, after everything before this call
    if (prefix) {
        CascadeParams cp{p, group_offsets, group_members, G, static_cast<int32_t>(row_chunks), npp,
                         block_tables, d->num_blocks, p.qk_scale, 1.f};
        void* staging = static_cast<unsigned char*>(workspace) + stage_off;
        if (staged) {
            // the prefix pass reads a 16-bit copy (q's type) of the groups' blocks
            const CascadeStage lay = cascade_stage_layout(num_seqs, max_blocks_per_seq, num_groups, max_group_blocks,
                                                          d->num_kv_heads, d->head_size);
            unsigned char* sw = static_cast<unsigned char*>(staging);
            cp.prefix_tables = reinterpret_cast<const int32_t*>(sw + lay.table_off);
            cp.prefix_nb = num_groups * max_group_blocks;
            cp.prefix_o_scale = d->v_scale;
            if (!encode_pool_map(&tpk, sw + lay.k_off, 2, stage_rows, d->head_size) ||
                !encode_pool_map(&tpv, sw + lay.v_off, 2, stage_rows, d->head_size))
                return PKV_ERR_CUDA;
        } else if (!use_mma) {
            if (!encode_pool_map(&tpk, k_cache, 2, pool_rows, d->head_size) ||
                !encode_pool_map(&tpv, v_cache, 2, pool_rows, d->head_size))
                return PKV_ERR_CUDA;
        }
        const CUtensorMap& pk = (staged || !use_mma) ? tpk : tk;
        const CUtensorMap& pv = (staged || !use_mma) ? tpv : tv;
        if (staged) e = launch_cascade_stage_fp8(cp, num_groups, max_group_blocks, q_dtype, k_cache, v_cache, staging, st);
        if (e == cudaSuccess) e = launch_cascade_prefix_tc(cp, num_groups, q_dtype, d->head_size, tq, pk, pv, st);
        if (e != cudaSuccess) return PKV_ERR_CUDA;
        p.join_primary = 1;
    }
    // 2. each sequence's own tokens, beside the prefix pass
    if (use_mma) {
        e = launch_decode_gqa(p, G, d->kv_dtype, q_dtype, tk, tv, st);
    } else if (d->kv_dtype == PKV_BF16) {
        e = launch_decode_bf16(p, G, st);
    } else if (d->kv_dtype == PKV_F16) {
        e = launch_decode_f16(p, G, st);
    } else if (q_dtype == PKV_BF16) {
        e = launch_decode_fp8_bf16q(p, G, st);
    } else {
        e = launch_decode_fp8_f16q(p, G, st);
    }
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    // 3. merge every row, once the decode grid (and with it the prefix pass) is complete
    e = launch_merge(p, q_dtype, st);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
