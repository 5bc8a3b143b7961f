// pkv_noalloc.cu -- decode attention for callers that cannot allocate device
// memory.
//
// pkv_paged_attention_decode needs a caller-provided workspace whenever a
// sequence is split into several partitions (the per-partition max, sum and
// partial output that the merge kernel combines).  Some callers have no way
// to provide one: a plug-in running inside a host framework that owns all
// device memory and offers no allocator, or a latency-critical loop that
// must not call cudaMalloc (which can synchronise the whole device).  This
// entry point serves them with a fixed scratch buffer that lives in the
// library itself, as a static device array of kNoAllocScratchBytes bytes.
// Every GPU that loads the library holds that buffer until the process
// exits.
//
// Nothing here calls cudaMalloc, cudaFree or any routine that allocates.
#include <cstdint>

#include "pkv_internal.h"

namespace pkv {
namespace {

// Maximum scratch this entry point can use: 32 MiB, enough for e.g. 8
// sequences x 64 query heads x 64 partitions of head_size 128 (17 MiB).
constexpr size_t kNoAllocScratchBytes = 32u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch in the current context.  In host code
// the array's name is only a host-side handle, so the address is looked up
// with cudaGetSymbolAddress -- on every call, not cached: a cached address
// would outlive a cudaDeviceReset or belong to another context of the same
// device.  The lookup allocates nothing; the first one on a device may load
// the library's device code, which is why the first call should come before
// any stream capture.
void* scratch_address(pkv_status* st) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        *st = PKV_ERR_CUDA;
        return nullptr;
    }
    *st = PKV_OK;
    return ptr;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_paged_attention_decode_noalloc(const void* q, int32_t q_dtype, int32_t num_seqs,
                                                         int32_t num_q_heads, const void* k_cache,
                                                         const void* v_cache, const pkv_cache_desc* desc,
                                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                         const int32_t* seq_lens, int32_t max_seq_len, float scale,
                                                         void* out, int32_t partition_tokens, void* stream) {
    if (!desc || partition_tokens < 0) return PKV_ERR_INVALID;
    // Resolve the partition size first so the scratch need is exact.
    int32_t P = partition_tokens;
    if (P == 0) {
        P = pkv_decode_auto_partition(num_seqs, num_q_heads, desc->num_kv_heads, desc->head_size, max_seq_len, 0);
        if (P < 0) return static_cast<pkv_status>(-P);
    }
    const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, desc->head_size, max_seq_len, P);
    if (need > kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;  // beyond the built-in maximum
    pkv_status st = PKV_OK;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = scratch_address(&st);
        if (st != PKV_OK) return st;
    }
    return pkv_paged_attention_decode(q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, desc, block_tables,
                                      max_blocks_per_seq, seq_lens, max_seq_len, scale, out, scratch,
                                      need > 0 ? kNoAllocScratchBytes : 0, P, stream);
}
