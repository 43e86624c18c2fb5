// Fused block copy (vLLM paper review, mz-moonzoo.tistory.com/116, §5.1 (3);
// PagedAttention notes, unpurerationalist.github.io, §4.1): the copies that
// copy-on-write asks for -- whole physical blocks, every layer, keys and
// values -- in one launch instead of one cudaMemcpyAsync per block.
//
// grid = (vector chunk, pair, layer * 2 + {K, V}); each thread moves 16-byte
// vectors of one block of one layer's K or V cache.  A block of one layer is
// H * B * D * 2 contiguous bytes in the cache layout [num_blocks][H][B][D].
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pagedkv {

namespace {

constexpr int kMaxLayers = 128;

struct LayerPtrs {
    uint4 *k[kMaxLayers];
    uint4 *v[kMaxLayers];
};

constexpr int kVecPerThread = 4;

__global__ void __launch_bounds__(256)
copy_blocks_kernel(const __grid_constant__ LayerPtrs ptrs, const int32_t *__restrict__ pairs,
                   int32_t n_pairs, int64_t vec_per_block, int32_t num_blocks, int32_t *status) {
    const int layer = blockIdx.z >> 1;
    uint4 *cache = (blockIdx.z & 1) ? ptrs.v[layer] : ptrs.k[layer];
    for (int32_t pi = blockIdx.y; pi < n_pairs; pi += gridDim.y) {
        const int32_t src = pairs[2 * pi];
        const int32_t dst = pairs[2 * pi + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (blockIdx.x == 0 && threadIdx.x == 0) report(status, PA_ERR_BAD_BLOCK);
            continue;
        }
        const uint4 *s = cache + (int64_t)src * vec_per_block;
        uint4 *d = cache + (int64_t)dst * vec_per_block;
        const int64_t base = (int64_t)blockIdx.x * blockDim.x * kVecPerThread + threadIdx.x;
        uint4 tmp[kVecPerThread];
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int64_t e = base + (int64_t)u * blockDim.x;
            if (e < vec_per_block) tmp[u] = s[e];
        }
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int64_t e = base + (int64_t)u * blockDim.x;
            if (e < vec_per_block) d[e] = tmp[u];
        }
    }
}

struct SwapPtrs {
    const uint4 *sk[kMaxLayers];
    const uint4 *sv[kMaxLayers];
    uint4 *dk[kMaxLayers];
    uint4 *dv[kMaxLayers];
};

// Block pairs (src in one cache set, dst in another), every layer, K and V.
__global__ void __launch_bounds__(256)
swap_blocks_kernel(const __grid_constant__ SwapPtrs ptrs, const int32_t *__restrict__ pairs,
                   int32_t n_pairs, int64_t vec_per_block, int32_t src_blocks, int32_t dst_blocks,
                   int32_t *status) {
    const int layer = blockIdx.z >> 1;
    const bool is_v = blockIdx.z & 1;
    const uint4 *src = is_v ? ptrs.sv[layer] : ptrs.sk[layer];
    uint4 *dst = is_v ? ptrs.dv[layer] : ptrs.dk[layer];
    for (int32_t pi = blockIdx.y; pi < n_pairs; pi += gridDim.y) {
        const int32_t a = pairs[2 * pi];
        const int32_t b = pairs[2 * pi + 1];
        if (a < 0 || a >= src_blocks || b < 0 || b >= dst_blocks) {
            if (blockIdx.x == 0 && threadIdx.x == 0) report(status, PA_ERR_BAD_BLOCK);
            continue;
        }
        const uint4 *s = src + (int64_t)a * vec_per_block;
        uint4 *d = dst + (int64_t)b * vec_per_block;
        const int64_t base = (int64_t)blockIdx.x * blockDim.x * kVecPerThread + threadIdx.x;
        uint4 tmp[kVecPerThread];
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int64_t e = base + (int64_t)u * blockDim.x;
            if (e < vec_per_block) tmp[u] = s[e];
        }
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int64_t e = base + (int64_t)u * blockDim.x;
            if (e < vec_per_block) d[e] = tmp[u];
        }
    }
}

}  // namespace

int launch_swap_blocks(const void *const *src_k, const void *const *src_v, int32_t src_blocks,
                       void *const *dst_k, void *const *dst_v, int32_t dst_blocks,
                       int32_t num_layers, const int32_t *pairs, int32_t n_pairs,
                       const pa_pool_desc *d, int32_t *status, void *stream) {
    std::string why;
    if (!d) return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: NULL desc");
    if (!device_geometry_ok(d, &why))
        return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: %s", why.c_str());
    if (n_pairs < 0 || num_layers < 1 || num_layers > kMaxLayers || src_blocks < 0 ||
        dst_blocks < 0)
        return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: n_pairs=%d, num_layers=%d (1..%d)",
                    n_pairs, num_layers, kMaxLayers);
    if (n_pairs == 0) return PA_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !pairs)
        return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: NULL pointer");
    SwapPtrs sp{};
    auto bad = [](const void *p) { return !p || (reinterpret_cast<uintptr_t>(p) & 15); };
    for (int l = 0; l < num_layers; ++l) {
        if (bad(src_k[l]) || bad(src_v[l]) || bad(dst_k[l]) || bad(dst_v[l]))
            return fail(PA_ERR_INVALID_ARG, "pa_swap_blocks: layer %d cache NULL or misaligned", l);
        sp.sk[l] = static_cast<const uint4 *>(src_k[l]);
        sp.sv[l] = static_cast<const uint4 *>(src_v[l]);
        sp.dk[l] = static_cast<uint4 *>(dst_k[l]);
        sp.dv[l] = static_cast<uint4 *>(dst_v[l]);
    }
    const int64_t vec_per_block = (int64_t)d->num_heads * d->block_size * d->head_dim / 8;
    const int64_t per_cta = 256 * kVecPerThread;
    dim3 grid((unsigned)((vec_per_block + per_cta - 1) / per_cta),
              (unsigned)(n_pairs < 65535 ? n_pairs : 65535), (unsigned)(2 * num_layers));
    swap_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        sp, pairs, n_pairs, vec_per_block, src_blocks, dst_blocks, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "pa_swap_blocks: launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

int launch_copy_blocks(void *const *k_caches, void *const *v_caches, int32_t num_layers,
                       const int32_t *pairs, int32_t n_pairs, const pa_pool_desc *d,
                       int32_t *status, void *stream) {
    std::string why;
    if (!d) return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: NULL desc");
    if (!device_geometry_ok(d, &why))
        return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: %s", why.c_str());
    if (n_pairs < 0 || num_layers < 1 || num_layers > kMaxLayers)
        return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: n_pairs=%d, num_layers=%d (1..%d)",
                    n_pairs, num_layers, kMaxLayers);
    if (n_pairs == 0) return PA_OK;
    if (!k_caches || !v_caches || !pairs) return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: NULL pointer");
    LayerPtrs lp{};
    for (int l = 0; l < num_layers; ++l) {
        if (!k_caches[l] || !v_caches[l] || (reinterpret_cast<uintptr_t>(k_caches[l]) & 15) ||
            (reinterpret_cast<uintptr_t>(v_caches[l]) & 15))
            return fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: layer %d cache NULL or misaligned", l);
        lp.k[l] = static_cast<uint4 *>(k_caches[l]);
        lp.v[l] = static_cast<uint4 *>(v_caches[l]);
    }
    const int64_t vec_per_block = (int64_t)d->num_heads * d->block_size * d->head_dim / 8;
    const int64_t per_cta = 256 * kVecPerThread;
    dim3 grid((unsigned)((vec_per_block + per_cta - 1) / per_cta),
              (unsigned)(n_pairs < 65535 ? n_pairs : 65535), (unsigned)(2 * num_layers));
    copy_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        lp, pairs, n_pairs, vec_per_block, d->num_blocks, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "pa_copy_blocks: launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

}  // namespace pagedkv
