// pkv_api.cu -- C ABI entry points for decode attention, the device error
// word, status strings.  Argument meaning, layout, ownership and error
// behaviour are specified in include/pagedkv.h.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "pkv_decode_impl.cuh"
#include "pkv_merge.cuh"

namespace pkv {

// Device error word: the OR of PKV_DEVERR_* bits reported by the kernels.
__device__ unsigned int g_device_error = 0;

namespace {
using CtxGetCurrent = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (no libcuda link).
CtxGetCurrent ctx_get_current() {
    static CtxGetCurrent fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrent>(f);
    });
    return fn;
}
}  // namespace

// The error word's device address is cached per device together with the
// context it was looked up in, and looked up again whenever the current
// context differs (after a cudaDeviceReset, or under another context of the
// same device), so a stale address is never handed to a kernel.
unsigned int* error_word() {
    static CUcontext ctxs[kMaxDevices] = {};
    static unsigned int* ptrs[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    const CtxGetCurrent get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev] || !ctx || ctx != ctxs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<unsigned int*>(p);
        CUcontext now = nullptr;  // the lookup may have made the primary context current
        if (get && get(&now) != CUDA_SUCCESS) now = nullptr;
        ctxs[dev] = now;
    }
    return ptrs[dev];
}

namespace {
// Launches the merge as a programmatic dependent of the kernel before it on
// the stream (the decode that wrote the partials): its CTAs may start while
// that kernel's last CTAs run and wait in griddepcontrol.wait for its
// completion, which hides the launch gap.  A driver that refuses the
// attribute gets a plain launch.
template <int D, typename QT, int WPR>
cudaError_t launch_merge_t(const DecodeParams& p, int64_t rows, cudaStream_t st) {
    constexpr int RPC = 8 / WPR;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + RPC - 1) / RPC));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, merge_kernel<D, QT, WPR>, p);
    if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) {
        (void)cudaGetLastError();
        merge_kernel<D, QT, WPR><<<cfg.gridDim, 256, 0, st>>>(p);
        e = cudaGetLastError();
    }
    return e;
}

template <int D, typename QT>
cudaError_t launch_merge_d(const DecodeParams& p, int64_t rows, cudaStream_t st) {
    switch (merge_warps_per_row(p.NP)) {
    case 1: return launch_merge_t<D, QT, 1>(p, rows, st);
    case 2: return launch_merge_t<D, QT, 2>(p, rows, st);
    case 4: return launch_merge_t<D, QT, 4>(p, rows, st);
    default: return launch_merge_t<D, QT, 8>(p, rows, st);
    }
}
}  // namespace

cudaError_t launch_merge(const DecodeParams& p, int q_dtype, cudaStream_t st) {
    const int64_t rows = static_cast<int64_t>(p.S) * p.Hq;
    if (rows <= 0) return cudaSuccess;
    if (q_dtype == PKV_BF16)
        return p.D == 128 ? launch_merge_d<128, BF16>(p, rows, st) : launch_merge_d<64, BF16>(p, rows, st);
    return p.D == 128 ? launch_merge_d<128, F16>(p, rows, st) : launch_merge_d<64, F16>(p, rows, st);
}

int num_sms() {
    static int cached[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

namespace {
std::atomic<int> g_decode_path{0};  // 0 auto, 1 CUDA cores, 2 tensor cores
}  // namespace

cudaError_t launch_decode_gqa(const DecodeParams& p, int G, int kv_dtype, int q_dtype, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t st) {
    if (kv_dtype == PKV_F16) return launch_decode_mma_f16(p, G, tk, tv, st);
    if (kv_dtype == PKV_BF16) return launch_decode_mma_bf16(p, G, tk, tv, st);
    return q_dtype == PKV_BF16 ? launch_decode_mma_fp8_bf16q(p, G, tk, tv, st)
                               : launch_decode_mma_fp8_f16q(p, G, tk, tv, st);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 2-D view of a pool as [NB*Hkv*16 rows][D] elements, 128-byte inner box of
// 16 rows, 128-byte swizzle (matches swz128() in the kernel).
bool encode_pool_map(CUtensorMap* map, const void* base, int elem_bytes, int64_t rows, int D) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * elem_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem_bytes), static_cast<cuuint32_t>(kBlockSize)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_token_head_map(CUtensorMap* map, const void* base, int D, int H, int64_t T, int box_h, int box_t) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_h), static_cast<cuuint32_t>(box_t)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

// Tokens per split-K partition when the caller passes 0.  Enough CTAs for a
// few waves of resident CTAs keep the SMs evenly loaded when sequence
// lengths differ; beyond that, splitting only adds partial-result traffic.
// In grid order a CTA never takes more than kAutoMaxPartition tokens, so a
// few long sequences cannot leave the last wave running alone (measured on
// GB300: 64 x U[512, 4096] MHA decodes 2.4 % faster with 2048-token
// partitions; sequences of <= 2048 tokens are not split by this cap).  A
// launch in a host plan's longest-first order (planned) starts the long
// CTAs first, so there the cap only adds merge work and is dropped (the same
// batch: 341.4 against 346.2 us).
constexpr int kAutoMaxPartition = 2048;

int auto_partition(int S, int Hkv, int max_seq_len, bool planned) {
    const int64_t units = static_cast<int64_t>(S) * Hkv;
    const int64_t want = static_cast<int64_t>(num_sms()) * 2 * 4;
    int64_t parts = ceil_div(want, units > 0 ? units : 1);
    if (parts < 1) parts = 1;
    int64_t P = ceil_div(ceil_div(max_seq_len > 0 ? max_seq_len : 1, parts), kBlockSize) * kBlockSize;
    if (!planned && P > kAutoMaxPartition) P = kAutoMaxPartition;
    if (P < kAutoMinPartition) P = kAutoMinPartition;
    return static_cast<int>(P);
}

size_t partials_bytes(int64_t S, int64_t Hq, int64_t D, int64_t NP) {
    // m, l and o rows, each region 256-byte aligned
    const int64_t rows = S * Hq * NP;
    const int64_t ml = ceil_div(rows * 4, 256) * 256;
    return static_cast<size_t>(2 * ml + rows * D * 4);
}

void partials_layout(DecodeParams& p, void* workspace) {
    const int64_t rows = static_cast<int64_t>(p.S) * p.Hq * p.NP;
    const int64_t ml = ceil_div(rows * 4, 256) * 256;
    unsigned char* w = static_cast<unsigned char*>(workspace);
    p.part_m = reinterpret_cast<float*>(w);
    p.part_l = reinterpret_cast<float*>(w + ml);
    p.part_o = reinterpret_cast<float*>(w + 2 * ml);
}

namespace {
size_t workspace_bytes(int64_t S, int64_t Hq, int64_t D, int64_t max_seq_len, int64_t P) {
    const int64_t NP = max_seq_len > 0 ? ceil_div(max_seq_len, P) : 1;
    if (NP <= 1) return 0;
    return partials_bytes(S, Hq, D, NP);
}
}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_set_decode_path(int32_t path) {
    if (path < 0 || path > 2) return PKV_ERR_INVALID;
    g_decode_path.store(path);
    return PKV_OK;
}

extern "C" int32_t pkv_get_decode_path(void) { return g_decode_path.load(); }

extern "C" size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                                             int32_t max_seq_len, int32_t partition_tokens) {
    if (num_seqs < 0 || num_q_heads <= 0 || head_size <= 0 || max_seq_len < 0 || partition_tokens < 0)
        return 0;
    if (partition_tokens % kBlockSize) return 0;
    const int64_t P = partition_tokens > 0 ? partition_tokens : kAutoMinPartition;
    return workspace_bytes(num_seqs, num_q_heads, head_size, max_seq_len, P);
}

extern "C" int32_t pkv_decode_auto_partition(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_size, int32_t max_seq_len, int32_t planned) {
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_size <= 0 || max_seq_len < 0)
        return -static_cast<int32_t>(PKV_ERR_INVALID);
    return auto_partition(num_seqs, num_kv_heads, max_seq_len, planned != 0);
}

namespace {
// The step's new tokens for the decode with a fused append (null: plain decode).
struct FusedAppend {
    const void* k;
    const void* v;
    int32_t in_dtype;
    const int64_t* slots;    // [num_seqs]
    const int32_t* cow_src;  // [num_seqs] or null
};

pkv_status decode_common(const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads,
                         const void* k_cache, const void* v_cache, const pkv_cache_desc* d,
                         const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                         int32_t max_seq_len, float scale, void* out, void* workspace, size_t ws_bytes,
                         int32_t partition_tokens, void* stream, const FusedAppend* app,
                         const int32_t* work = nullptr, int32_t num_work = 0) {
    // ---- validation (host, before any launch)
    if (num_work < 0 || (!work && num_work > 0)) return PKV_ERR_INVALID;
    if (!d || num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0 ||
        partition_tokens < 0)
        return PKV_ERR_INVALID;
    if (d->num_blocks <= 0 || d->num_kv_heads <= 0 || d->head_size <= 0 || d->block_size <= 0)
        return PKV_ERR_INVALID;
    if (d->kv_dtype < PKV_F16 || d->kv_dtype > PKV_FP8_E4M3) return PKV_ERR_INVALID;
    if (q_dtype != PKV_F16 && q_dtype != PKV_BF16) return PKV_ERR_INVALID;
    if (num_q_heads % d->num_kv_heads) return PKV_ERR_INVALID;
    if (!(scale == scale)) return PKV_ERR_INVALID;
    if (d->kv_dtype == PKV_FP8_E4M3 && !(d->k_scale > 0.f && d->v_scale > 0.f)) return PKV_ERR_INVALID;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * d->block_size)
        return PKV_ERR_INVALID;
    if (partition_tokens % kBlockSize) return PKV_ERR_INVALID;
    if (d->kv_dtype != PKV_FP8_E4M3 && q_dtype != d->kv_dtype) return PKV_ERR_UNSUPPORTED;
    if (d->block_size != kBlockSize || (d->head_size != 64 && d->head_size != 128)) return PKV_ERR_UNSUPPORTED;
    const int G = num_q_heads / d->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || d->num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || (work && num_work == 0)) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out) return PKV_ERR_INVALID;
    if (static_cast<int64_t>(num_work) * d->num_kv_heads > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return PKV_ERR_INVALID;
    if (app) {
        if (!app->k || !app->v || !app->slots || !aligned16(app->k) || !aligned16(app->v) ||
            (reinterpret_cast<uintptr_t>(app->slots) & 7u) || (reinterpret_cast<uintptr_t>(app->cow_src) & 3u))
            return PKV_ERR_INVALID;
        if (app->in_dtype < PKV_F16 || app->in_dtype > PKV_FP8_E4M3) return PKV_ERR_INVALID;
        const bool same16 = d->kv_dtype != PKV_FP8_E4M3 && app->in_dtype == d->kv_dtype;
        const bool to_fp8 = d->kv_dtype == PKV_FP8_E4M3 && (app->in_dtype == PKV_BF16 || app->in_dtype == PKV_F16);
        if (!same16 && !to_fp8) return PKV_ERR_UNSUPPORTED;
    }

    const int P =
        partition_tokens > 0 ? partition_tokens : auto_partition(num_seqs, d->num_kv_heads, max_seq_len, work != nullptr);
    const int64_t NP = max_seq_len > 0 ? ceil_div(max_seq_len, P) : 1;
    if (NP > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
    const size_t need = workspace_bytes(num_seqs, num_q_heads, d->head_size, max_seq_len, P);
    if (need > 0 && (!workspace || ws_bytes < need || !aligned16(workspace))) return PKV_ERR_WORKSPACE;

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
    p.qk_scale = scale * log2e * (d->kv_dtype == PKV_FP8_E4M3 ? d->k_scale : 1.f);
    p.v_scale = d->kv_dtype == PKV_FP8_E4M3 ? d->v_scale : 1.f;
    p.err = err;
    p.work = work;
    p.num_work = num_work;
    if (need > 0) partials_layout(p, workspace);
    if (app) {
        p.k_new = app->k;
        p.v_new = app->v;
        p.slots = app->slots;
        p.cow_src = app->cow_src;
        p.in_dtype = app->in_dtype;
        p.k_enc_scale = d->k_scale;
        p.v_enc_scale = d->v_scale;
    }

    // Tensor-core kernel for grouped-query heads at head_size 128; CUDA
    // cores otherwise (one query row per KV head is not a dense tile).
    const int64_t pool_rows = static_cast<int64_t>(d->num_blocks) * d->num_kv_heads * kBlockSize;
    const bool mma_ok = d->head_size == 128 && G >= 2 && pool_rows <= 0x7fffffff;
    const int path = g_decode_path.load();
    if (path == 2 && !mma_ok) return PKV_ERR_UNSUPPORTED;
    const bool use_mma = mma_ok && path != 1;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (use_mma) {
        CUtensorMap tk, tv;
        const int eb = d->kv_dtype == PKV_FP8_E4M3 ? 1 : 2;
        if (!encode_pool_map(&tk, k_cache, eb, pool_rows, d->head_size) ||
            !encode_pool_map(&tv, v_cache, eb, pool_rows, d->head_size))
            return PKV_ERR_CUDA;
        e = launch_decode_gqa(p, G, d->kv_dtype, q_dtype, tk, tv, st);
    } else if (d->kv_dtype == PKV_F16) {
        e = launch_decode_f16(p, G, st);
    } else if (d->kv_dtype == PKV_BF16) {
        e = launch_decode_bf16(p, G, st);
    } else if (q_dtype == PKV_BF16) {
        e = launch_decode_fp8_bf16q(p, G, st);
    } else {
        e = launch_decode_fp8_f16q(p, G, st);
    }
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    if (NP > 1) {
        e = launch_merge(p, q_dtype, st);
        if (e != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}
}  // namespace

extern "C" pkv_status pkv_paged_attention_decode(const void* q, int32_t q_dtype, int32_t num_seqs,
                                                 int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                                 const pkv_cache_desc* d, const int32_t* block_tables,
                                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                                 int32_t max_seq_len, float scale, void* out, void* workspace,
                                                 size_t ws_bytes, int32_t partition_tokens, void* stream) {
    return decode_common(q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, d, block_tables, max_blocks_per_seq,
                         seq_lens, max_seq_len, scale, out, workspace, ws_bytes, partition_tokens, stream, nullptr);
}

extern "C" pkv_status pkv_paged_attention_decode_append(const void* k_new, const void* v_new, int32_t in_dtype,
                                                        const int64_t* slot_mapping, const int32_t* cow_src,
                                                        const void* q, int32_t q_dtype,
                                                        int32_t num_seqs, int32_t num_q_heads, void* k_cache,
                                                        void* v_cache, const pkv_cache_desc* d,
                                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                        const int32_t* seq_lens, int32_t max_seq_len, float scale,
                                                        void* out, void* workspace, size_t ws_bytes,
                                                        int32_t partition_tokens, const int32_t* work_units,
                                                        int32_t num_work_units, void* stream) {
    const FusedAppend app{k_new, v_new, in_dtype, slot_mapping, cow_src};
    return decode_common(q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, d, block_tables, max_blocks_per_seq,
                         seq_lens, max_seq_len, scale, out, workspace, ws_bytes, partition_tokens, stream,
                         num_seqs > 0 ? &app : nullptr, work_units, num_work_units);
}

// Host work plan for the decode: the batch's (sequence, partition) units,
// longest first.  See pagedkv.h.
extern "C" pkv_status pkv_decode_plan(const int32_t* seq_lens, int32_t num_seqs, int32_t num_kv_heads,
                                      int32_t max_seq_len, int32_t partition_tokens, int32_t* units,
                                      int32_t units_cap, int32_t* num_units) {
    if (!num_units) return PKV_ERR_INVALID;
    *num_units = 0;
    if (num_seqs < 0 || num_kv_heads <= 0 || max_seq_len < 0 || partition_tokens < 0 || units_cap < 0 ||
        partition_tokens % kBlockSize)
        return PKV_ERR_INVALID;
    if (num_seqs == 0) return PKV_OK;
    if (!seq_lens) return PKV_ERR_INVALID;
    const int P = partition_tokens > 0 ? partition_tokens : auto_partition(num_seqs, num_kv_heads, max_seq_len, true);
    const int64_t NP = max_seq_len > 0 ? ceil_div(max_seq_len, P) : 1;
    if (NP * num_seqs > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
    std::vector<std::pair<int64_t, int32_t>> list;  // (tokens, unit)
    for (int32_t s = 0; s < num_seqs; ++s) {
        int64_t L = seq_lens[s];
        if (L < 0 || L > max_seq_len) return PKV_ERR_INVALID;
        const int64_t n = L > 0 ? ceil_div(L, P) : 1;  // a zero-length row still has a unit (it writes zeros)
        for (int64_t part = 0; part < n; ++part)
            list.emplace_back(std::min<int64_t>(P, L - part * P), static_cast<int32_t>(s * NP + part));
    }
    std::stable_sort(list.begin(), list.end(),
                     [](const std::pair<int64_t, int32_t>& a, const std::pair<int64_t, int32_t>& b) {
                         return a.first > b.first;
                     });
    *num_units = static_cast<int32_t>(list.size());
    if (static_cast<int64_t>(list.size()) > units_cap) return PKV_ERR_WORKSPACE;
    if (!units) return PKV_ERR_INVALID;
    for (size_t i = 0; i < list.size(); ++i) units[i] = list[i].second;
    return PKV_OK;
}

extern "C" pkv_status pkv_get_device_error(uint32_t* flags, void* stream) {
    if (!flags) return PKV_ERR_INVALID;
    unsigned int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int v = 0;
    if (cudaMemcpyAsync(&v, err, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaMemsetAsync(err, 0, sizeof(unsigned int), st) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PKV_ERR_CUDA;
    *flags = v;
    return PKV_OK;
}

extern "C" const char* pkv_status_string(int32_t status) {
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported combination";
    case PKV_ERR_OOM: return "out of blocks";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_NOT_FOUND: return "unknown sequence";
    default: return "unknown status";
    }
}

extern "C" const char* pkv_version(void) { return "0.1.0"; }
