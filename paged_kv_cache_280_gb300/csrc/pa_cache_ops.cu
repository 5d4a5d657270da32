// Slot-mapped append (reshape_and_cache) and copy-on-write block copy.
//
// Both are HBM copies of 16-byte vectors; a thread moves one 16-byte chunk of
// K and the matching chunk of V per iteration of a grid-stride loop, so
// consecutive threads touch consecutive bytes of one row (coalesced on both
// sides).  Indices are checked against the pool before any access.
#include <cuda_fp8.h>

#include <cmath>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// "破局思路/按需分配" (ohmygp.com) and "非连续存储" ("Q32" §2): token i goes to
// slot s = slot_mapping[i]: block s / BS, offset s % BS, every KV head.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const uint4* __restrict__ k_new,
                                                                const uint4* __restrict__ v_new, uint4* k_pool,
                                                                uint4* v_pool, const int64_t* __restrict__ slots,
                                                                int32_t num_tokens, int32_t num_kv_heads,
                                                                int32_t row_chunks, int32_t block_size,
                                                                int64_t pool_slots, int32_t* status) {
    pdl_launch_dependents();  // the decode that follows may start its prologue now
    const int64_t per_token = (int64_t)num_kv_heads * row_chunks;
    const int64_t total = (int64_t)num_tokens * per_token;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / per_token;
        const int64_t within = idx - i * per_token;  // h * row_chunks + chunk
        const int64_t s = __ldg(slots + i);
        if (s < 0) continue;
        if (s >= pool_slots) {
            flag_status(status, PA_DEV_BAD_SLOT);
            continue;
        }
        const int64_t blk = s / block_size, off = s - blk * block_size;
        const int64_t h = within / row_chunks, chunk = within - h * row_chunks;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * row_chunks + chunk;
        k_pool[dst] = __ldg(k_new + idx);
        v_pool[dst] = __ldg(v_new + idx);
    }
}

// Slot-mapped append into FP8 (E4M3) pools: each element is quantised as
// code = E4M3(fp32(x / scale)) with round-to-nearest-even and saturation to
// +-448 (the hardware conversion with satfinite).  One thread converts 8
// elements: 16 bytes of bf16 in, 8 bytes of codes out.
template <typename TIn>
__global__ void __launch_bounds__(256) reshape_and_cache_fp8_kernel(
    const TIn* __restrict__ k_new, const TIn* __restrict__ v_new, uint2* k_pool, uint2* v_pool,
    const int64_t* __restrict__ slot_mapping, int32_t num_tokens, int32_t num_kv_heads, int32_t row_groups,
    int32_t block_size, int64_t num_slots, float k_scale, float v_scale, int32_t* status) {
    pdl_launch_dependents();
    const int64_t total = (int64_t)num_tokens * num_kv_heads * row_groups;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tok = idx / ((int64_t)num_kv_heads * row_groups);
        const int64_t rem = idx - tok * num_kv_heads * row_groups;
        const int64_t slot = __ldg(slot_mapping + tok);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            flag_status(status, PA_DEV_BAD_SLOT);
            continue;
        }
        const int64_t blk = slot / block_size, off = slot % block_size;
        const int64_t h = rem / row_groups, grp = rem - h * row_groups;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * row_groups + grp;
        uint32_t kc[2], vc[2];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t kw = 0, vw = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t src = idx * 8 + half * 4 + e;
                const float kx = static_cast<float>(k_new[src]) / k_scale;
                const float vx = static_cast<float>(v_new[src]) / v_scale;
                kw |= (uint32_t)__nv_cvt_float_to_fp8(kx, __NV_SATFINITE, __NV_E4M3) << (8 * e);
                vw |= (uint32_t)__nv_cvt_float_to_fp8(vx, __NV_SATFINITE, __NV_E4M3) << (8 * e);
            }
            kc[half] = kw;
            vc[half] = vw;
        }
        k_pool[dst] = make_uint2(kc[0], kc[1]);
        v_pool[dst] = make_uint2(vc[0], vc[1]);
    }
}

// "Copy-on-Write" ("Q32" §3): pool[dst] <- pool[src] for a whole block, K and V.
// blockIdx.y selects the pair, blockIdx.x a slice of the block.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* k_pool, uint4* v_pool, const int32_t* __restrict__ pairs,
                                                          int32_t num_pairs, int64_t block_chunks, int32_t num_blocks,
                                                          int32_t* status) {
    const int32_t pair = blockIdx.y;
    const int32_t src = __ldg(pairs + 2 * pair), dst = __ldg(pairs + 2 * pair + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, PA_DEV_BAD_BLOCK_ID);
        return;
    }
    const uint4* ks = k_pool + (int64_t)src * block_chunks;
    const uint4* vs = v_pool + (int64_t)src * block_chunks;
    uint4* kd = k_pool + (int64_t)dst * block_chunks;
    uint4* vd = v_pool + (int64_t)dst * block_chunks;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < block_chunks;
         c += (int64_t)gridDim.x * blockDim.x) {
        const uint4 a = ks[c];
        const uint4 b = vs[c];
        kd[c] = a;
        vd[c] = b;
    }
}

// Swap-out / swap-in of whole blocks between the pools and a block store
// [n][Hkv][block_size][head_dim] that may live in pinned host memory (written
// and read over NVLink-C2C by these kernels, no staging copy).  blockIdx.y
// selects the block, blockIdx.x a slice of it.
template <bool kOut>
__global__ void __launch_bounds__(256) swap_blocks_kernel(uint4* k_pool, uint4* v_pool, const int32_t* __restrict__ blocks,
                                                          uint4* k_store, uint4* v_store, int64_t block_chunks,
                                                          int32_t num_blocks, int32_t* status) {
    const int32_t i = blockIdx.y;
    const int32_t b = blocks[i];
    if (b < 0 || b >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, PA_DEV_BAD_BLOCK_ID);
        return;
    }
    uint4* kp = k_pool + (int64_t)b * block_chunks;
    uint4* vp = v_pool + (int64_t)b * block_chunks;
    uint4* ks = k_store + (int64_t)i * block_chunks;
    uint4* vs = v_store + (int64_t)i * block_chunks;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < block_chunks;
         c += (int64_t)gridDim.x * blockDim.x) {
        if (kOut) {
            const uint4 a = kp[c], v = vp[c];
            ks[c] = a;
            vs[c] = v;
        } else {
            const uint4 a = ks[c], v = vs[c];
            kp[c] = a;
            vp[c] = v;
        }
    }
}

static int sm_count_of_current_device() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool shape_ok(int32_t head_dim, int32_t block_size) {
    return (head_dim == 64 || head_dim == 128) && (block_size == 16 || block_size == 32);
}

}  // namespace pa

extern "C" pa_status pa_reshape_and_cache(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                                          const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size, int32_t num_blocks, pa_dtype dtype,
                                          int32_t* dev_status, void* stream) {
    using namespace pa;
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (!shape_ok(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !k_pool || !v_pool || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) || (reinterpret_cast<uintptr_t>(dev_status) & 3u))
        return PA_ERR_INVALID_ARG;
    const int elem = dtype == PA_F32 ? 4 : 2;
    const int32_t row_chunks = head_dim * elem / 16;
    const int64_t total = (int64_t)num_tokens * num_kv_heads * row_chunks;
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return PA_ERR_CUDA;
    const int64_t want = (total + 255) / 256;
    const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    reshape_and_cache_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), static_cast<uint4*>(k_pool),
        static_cast<uint4*>(v_pool), slot_mapping, num_tokens, num_kv_heads, row_chunks, block_size,
        (int64_t)num_blocks * block_size, dev_status);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* src_dst_pairs, int32_t num_pairs,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                    pa_dtype dtype, int32_t* dev_status, void* stream) {
    using namespace pa;
    if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
    if (!shape_ok(head_dim, block_size) || (dtype == PA_FP8_E4M3 && head_dim != 128)) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (num_pairs > 65535) return PA_ERR_UNSUPPORTED;  // one grid row per pair
    if (!k_pool || !v_pool || !src_dst_pairs) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || (reinterpret_cast<uintptr_t>(src_dst_pairs) & 3u) ||
        (reinterpret_cast<uintptr_t>(dev_status) & 3u))
        return PA_ERR_INVALID_ARG;
    const int elem = dtype == PA_F32 ? 4 : (dtype == PA_BF16 ? 2 : 1);
    const int64_t block_chunks = (int64_t)num_kv_heads * block_size * head_dim * elem / 16;
    int64_t slices = (block_chunks + 256 * 4 - 1) / (256 * 4);  // ~4 chunks per thread
    if (slices < 1) slices = 1;
    if (slices > 1024) slices = 1024;
    dim3 grid((unsigned)slices, (unsigned)num_pairs);
    copy_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), src_dst_pairs, num_pairs, block_chunks, num_blocks,
        dev_status);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

namespace pa {

static pa_status swap_blocks(bool out, void* k_pool, void* v_pool, const int32_t* blocks, int32_t n, void* k_store,
                             void* v_store, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int32_t num_blocks, pa_dtype dtype, int32_t* dev_status, void* stream) {
    if (n < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
    if (!shape_ok(head_dim, block_size) || (dtype == PA_FP8_E4M3 && head_dim != 128)) return PA_ERR_UNSUPPORTED;
    if (n == 0) return PA_OK;
    if (n > 65535) return PA_ERR_UNSUPPORTED;  // one grid row per block
    if (!k_pool || !v_pool || !blocks || !k_store || !v_store) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_store) || !aligned16(v_store) ||
        (reinterpret_cast<uintptr_t>(blocks) & 3u) || (reinterpret_cast<uintptr_t>(dev_status) & 3u))
        return PA_ERR_INVALID_ARG;
    const int elem = dtype == PA_F32 ? 4 : (dtype == PA_BF16 ? 2 : 1);
    const int64_t block_chunks = (int64_t)num_kv_heads * block_size * head_dim * elem / 16;
    int64_t slices = (block_chunks + 256 * 4 - 1) / (256 * 4);  // ~4 chunks per thread
    if (slices < 1) slices = 1;
    if (slices > 1024) slices = 1024;
    dim3 grid((unsigned)slices, (unsigned)n);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (out)
        swap_blocks_kernel<true><<<grid, 256, 0, st>>>(static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), blocks,
                                                       static_cast<uint4*>(k_store), static_cast<uint4*>(v_store),
                                                       block_chunks, num_blocks, dev_status);
    else
        swap_blocks_kernel<false><<<grid, 256, 0, st>>>(static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
                                                        blocks, static_cast<uint4*>(k_store),
                                                        static_cast<uint4*>(v_store), block_chunks, num_blocks,
                                                        dev_status);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa

extern "C" pa_status pa_swap_out(const void* k_pool, const void* v_pool, const int32_t* blocks, int32_t num,
                                 void* k_store, void* v_store, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int32_t num_blocks, pa_dtype dtype, int32_t* dev_status,
                                 void* stream) {
    return pa::swap_blocks(true, const_cast<void*>(k_pool), const_cast<void*>(v_pool), blocks, num, k_store, v_store,
                           num_kv_heads, head_dim, block_size, num_blocks, dtype, dev_status, stream);
}

extern "C" pa_status pa_swap_in(const void* k_store, const void* v_store, const int32_t* blocks, int32_t num,
                                void* k_pool, void* v_pool, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                int32_t num_blocks, pa_dtype dtype, int32_t* dev_status, void* stream) {
    return pa::swap_blocks(false, k_pool, v_pool, blocks, num, const_cast<void*>(k_store), const_cast<void*>(v_store),
                           num_kv_heads, head_dim, block_size, num_blocks, dtype, dev_status, stream);
}

extern "C" pa_status pa_reshape_and_cache_fp8(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                                              const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                                              int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                              pa_dtype in_dtype, float k_scale, float v_scale, int32_t* dev_status,
                                              void* stream) {
    using namespace pa;
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (in_dtype != PA_F32 && in_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (head_dim != 128 || (block_size != 16 && block_size != 32)) return PA_ERR_UNSUPPORTED;
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !k_pool || !v_pool || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) || (reinterpret_cast<uintptr_t>(dev_status) & 3u))
        return PA_ERR_INVALID_ARG;
    const int32_t row_groups = head_dim / 8;
    const int64_t total = (int64_t)num_tokens * num_kv_heads * row_groups;
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return PA_ERR_CUDA;
    const int64_t want = (total + 255) / 256;
    const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (in_dtype == PA_BF16)
        reshape_and_cache_fp8_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
            static_cast<uint2*>(k_pool), static_cast<uint2*>(v_pool), slot_mapping, num_tokens, num_kv_heads,
            row_groups, block_size, (int64_t)num_blocks * block_size, k_scale, v_scale, dev_status);
    else
        reshape_and_cache_fp8_kernel<float><<<grid, 256, 0, st>>>(
            static_cast<const float*>(k_new), static_cast<const float*>(v_new), static_cast<uint2*>(k_pool),
            static_cast<uint2*>(v_pool), slot_mapping, num_tokens, num_kv_heads, row_groups, block_size,
            (int64_t)num_blocks * block_size, k_scale, v_scale, dev_status);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
