// pkv_cache_ops.cu -- slot-mapped KV append and copy-on-write block copy.
//
// Append: "vLLM：大语言模型推理与服务库" section 4.3 (a new token is written into
// the block the table maps its position to, after a block is allocated when
// the last one is full) and "vLLM 高性能大语言模型推理引擎深度技术评估与分布式
// 架构展望" (each decode step appends the new token's KV vector to GPU memory).
// Copy: "vLLM 深度解析：从 PagedAttention 到生产部署", "Prefix Caching 与
// Copy-on-Write" (a shared block is copied when it is about to be modified).
//
// Both are pure data movement in the [NB][Hkv][16][D] pool layout: one token
// of one head is a contiguous D-element row, one block of one pool is a
// contiguous Hkv*16*D-element run.  Threads move 16-byte vectors.
#include <cstdint>

#include "pkv_append.cuh"

namespace pkv {
namespace {

// One thread per 16-byte chunk of input row (t, h), for K (blockIdx.y = 0)
// and V (blockIdx.y = 1).  Same element type in and out: a plain copy.
__global__ void __launch_bounds__(256) append_copy_kernel(const unsigned char* __restrict__ k,
                                                          const unsigned char* __restrict__ v,
                                                          const int64_t* __restrict__ slots,
                                                          unsigned char* kc, unsigned char* vc, int T,
                                                          int Hkv, int row_bytes, int64_t num_slots,
                                                          unsigned int* err) {
    const int chunks = row_bytes / 16;
    const int64_t total = static_cast<int64_t>(T) * Hkv * chunks;
    const unsigned char* src = blockIdx.y == 0 ? k : v;
    unsigned char* dst = blockIdx.y == 0 ? kc : vc;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i % chunks);
        const int64_t row = i / chunks;  // t * Hkv + h
        const int t = static_cast<int>(row / Hkv), h = static_cast<int>(row % Hkv);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (h == 0 && c == 0 && blockIdx.y == 0) report(err, PKV_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
        const int64_t drow = (blk * Hkv + h) * kBlockSize + off;
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(src + row * row_bytes) + c);
        reinterpret_cast<uint4*>(dst + drow * row_bytes)[c] = x;
    }
}

// fp8 E4M3 cache, 16-bit input: each thread encodes 8 input elements (16
// bytes in, 8 bytes out).  code = e4m3_rn_satfinite(x / scale) with an IEEE
// binary32 division.
template <typename IT>
__global__ void __launch_bounds__(256) append_fp8_kernel(const unsigned char* __restrict__ k,
                                                         const unsigned char* __restrict__ v,
                                                         const int64_t* __restrict__ slots,
                                                         unsigned char* kc, unsigned char* vc, int T,
                                                         int Hkv, int D, int64_t num_slots, float k_scale,
                                                         float v_scale, unsigned int* err) {
    const int chunks = D / 8;
    const int64_t total = static_cast<int64_t>(T) * Hkv * chunks;
    const unsigned char* src = blockIdx.y == 0 ? k : v;
    unsigned char* dst = blockIdx.y == 0 ? kc : vc;
    const float sc = blockIdx.y == 0 ? k_scale : v_scale;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i % chunks);
        const int64_t row = i / chunks;
        const int t = static_cast<int>(row / Hkv), h = static_cast<int>(row % Hkv);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (h == 0 && c == 0 && blockIdx.y == 0) report(err, PKV_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
        const int64_t drow = (blk * Hkv + h) * kBlockSize + off;
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(src + row * D * 2) + c);
        const uint2 out2 = encode_e4m3x8<IT>(x, sc);
        const uint32_t out[2] = {out2.x, out2.y};
        *reinterpret_cast<uint2*>(dst + drow * D + c * 8) = make_uint2(out[0], out[1]);
    }
}

// Block copy: grid (num_pairs, kCopySplit, 2 pools); each CTA moves 1/kCopySplit
// of one block of one pool with 16-byte vectors.
constexpr int kCopySplit = 8;

__global__ void __launch_bounds__(256) copy_blocks_kernel(unsigned char* kc, unsigned char* vc,
                                                          const int32_t* __restrict__ pairs, int NB,
                                                          int64_t block_bytes, unsigned int* err) {
    const int pr = blockIdx.x;
    const int32_t src = __ldg(pairs + 2 * pr), dst = __ldg(pairs + 2 * pr + 1);
    if (src < 0 || src >= NB || dst < 0 || dst >= NB) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) report(err, PKV_DEVERR_COPY_PAIR);
        return;
    }
    if (src == dst) return;
    unsigned char* pool = blockIdx.z == 0 ? kc : vc;
    const int64_t vecs = block_bytes / 16;
    const int64_t per = (vecs + kCopySplit - 1) / kCopySplit;
    const int64_t lo = blockIdx.y * per, hi = min(vecs, lo + per);
    const uint4* s4 = reinterpret_cast<const uint4*>(pool + src * block_bytes);
    uint4* d4 = reinterpret_cast<uint4*>(pool + dst * block_bytes);
    for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) d4[i] = s4[i];
}

// Swap: grid (num_pairs, kCopySplit, 2 pools); moves 1/kCopySplit of one
// block of one pool between the device pool and the host pool (pinned,
// device-mapped memory, same [blocks][Hkv][16][D] layout) with 16-byte
// vectors.  direction 0: device -> host, 1: host -> device.
__global__ void __launch_bounds__(256) swap_blocks_kernel(unsigned char* kc, unsigned char* vc, unsigned char* kh,
                                                          unsigned char* vh, const int32_t* __restrict__ pairs,
                                                          int NB, int NH, int64_t block_bytes, int direction,
                                                          unsigned int* err) {
    const int pr = blockIdx.x;
    const int32_t dblk = __ldg(pairs + 2 * pr), hblk = __ldg(pairs + 2 * pr + 1);
    if (dblk < 0 || dblk >= NB || hblk < 0 || hblk >= NH) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) report(err, PKV_DEVERR_COPY_PAIR);
        return;
    }
    unsigned char* dev = (blockIdx.z == 0 ? kc : vc) + dblk * block_bytes;
    unsigned char* host = (blockIdx.z == 0 ? kh : vh) + hblk * block_bytes;
    const uint4* src = reinterpret_cast<const uint4*>(direction == 0 ? dev : host);
    uint4* dst = reinterpret_cast<uint4*>(direction == 0 ? host : dev);
    const int64_t vecs = block_bytes / 16;
    const int64_t per = (vecs + kCopySplit - 1) / kCopySplit;
    const int64_t lo = blockIdx.y * per, hi = min(vecs, lo + per);
    for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) dst[i] = src[i];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool desc_ok(const pkv_cache_desc* d) {
    if (!d) return false;
    if (d->num_blocks <= 0 || d->num_kv_heads <= 0 || d->head_size <= 0 || d->block_size <= 0) return false;
    if (d->kv_dtype < PKV_F16 || d->kv_dtype > PKV_FP8_E4M3) return false;
    if (d->kv_dtype == PKV_FP8_E4M3 && !(d->k_scale > 0.f && d->v_scale > 0.f)) return false;
    return true;
}

bool desc_supported(const pkv_cache_desc* d) {
    return d->block_size == kBlockSize && (d->head_size == 64 || d->head_size == 128);
}

int grid_for(int64_t work) {
    const int64_t per = 256;
    int64_t g = (work + per - 1) / per;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
    if (g > cap) g = cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_paged_kv_append(const void* k, const void* v, int32_t in_dtype, int32_t num_tokens,
                                          const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                          const pkv_cache_desc* desc, void* stream) {
    if (!desc_ok(desc) || num_tokens < 0) return PKV_ERR_INVALID;
    if (!desc_supported(desc)) return PKV_ERR_UNSUPPORTED;
    if (in_dtype < PKV_F16 || in_dtype > PKV_FP8_E4M3) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PKV_ERR_INVALID;
    const bool same = in_dtype == desc->kv_dtype;
    const bool to_fp8 = desc->kv_dtype == PKV_FP8_E4M3 && (in_dtype == PKV_BF16 || in_dtype == PKV_F16);
    if (!same && !to_fp8) return PKV_ERR_UNSUPPORTED;
    unsigned int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int Hkv = desc->num_kv_heads, D = desc->head_size;
    const int64_t num_slots = static_cast<int64_t>(desc->num_blocks) * kBlockSize;
    if (same) {
        const int row_bytes = D * (desc->kv_dtype == PKV_FP8_E4M3 ? 1 : 2);
        const int64_t work = static_cast<int64_t>(num_tokens) * Hkv * (row_bytes / 16);
        dim3 grid(grid_for(work), 2);
        append_copy_kernel<<<grid, 256, 0, st>>>(static_cast<const unsigned char*>(k),
                                                 static_cast<const unsigned char*>(v), slot_mapping,
                                                 static_cast<unsigned char*>(k_cache),
                                                 static_cast<unsigned char*>(v_cache), num_tokens, Hkv,
                                                 row_bytes, num_slots, err);
    } else {
        const int64_t work = static_cast<int64_t>(num_tokens) * Hkv * (D / 8);
        dim3 grid(grid_for(work), 2);
        auto kern = in_dtype == PKV_BF16 ? append_fp8_kernel<BF16> : append_fp8_kernel<F16>;
        kern<<<grid, 256, 0, st>>>(static_cast<const unsigned char*>(k), static_cast<const unsigned char*>(v),
                                   slot_mapping, static_cast<unsigned char*>(k_cache),
                                   static_cast<unsigned char*>(v_cache), num_tokens, Hkv, D, num_slots,
                                   desc->k_scale, desc->v_scale, err);
    }
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                                      const int32_t* pairs, int32_t num_pairs, void* stream) {
    if (!desc_ok(desc) || num_pairs < 0) return PKV_ERR_INVALID;
    if (!desc_supported(desc)) return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !pairs || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(pairs) & 3u))
        return PKV_ERR_INVALID;
    if (num_pairs > 65535 * 1024) return PKV_ERR_UNSUPPORTED;
    unsigned int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    const int64_t block_bytes = static_cast<int64_t>(desc->num_kv_heads) * kBlockSize * desc->head_size *
                                (desc->kv_dtype == PKV_FP8_E4M3 ? 1 : 2);
    dim3 grid(num_pairs, kCopySplit, 2);
    copy_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<unsigned char*>(k_cache), static_cast<unsigned char*>(v_cache), pairs, desc->num_blocks,
        block_bytes, err);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" pkv_status pkv_swap_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* desc, void* k_host,
                                      void* v_host, int32_t num_host_blocks, const int32_t* pairs,
                                      int32_t num_pairs, int32_t direction, void* stream) {
    if (!desc_ok(desc) || num_pairs < 0 || num_host_blocks < 0 || (direction != 0 && direction != 1))
        return PKV_ERR_INVALID;
    if (!desc_supported(desc)) return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !k_host || !v_host || !pairs || num_host_blocks == 0) return PKV_ERR_INVALID;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_host) || !aligned16(v_host) ||
        (reinterpret_cast<uintptr_t>(pairs) & 3u))
        return PKV_ERR_INVALID;
    // The host pools must be pinned and mapped into the device address space.
    void* kd = nullptr;
    void* vd = nullptr;
    if (cudaHostGetDevicePointer(&kd, k_host, 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&vd, v_host, 0) != cudaSuccess || !kd || !vd) {
        cudaGetLastError();  // clear the sticky-free error of the failed query
        return PKV_ERR_INVALID;
    }
    if (!aligned16(kd) || !aligned16(vd)) return PKV_ERR_INVALID;
    unsigned int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    const int64_t block_bytes = static_cast<int64_t>(desc->num_kv_heads) * kBlockSize * desc->head_size *
                                (desc->kv_dtype == PKV_FP8_E4M3 ? 1 : 2);
    dim3 grid(num_pairs, kCopySplit, 2);
    swap_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<unsigned char*>(k_cache), static_cast<unsigned char*>(v_cache),
        static_cast<unsigned char*>(kd), static_cast<unsigned char*>(vd), pairs, desc->num_blocks, num_host_blocks,
        block_bytes, direction, err);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
