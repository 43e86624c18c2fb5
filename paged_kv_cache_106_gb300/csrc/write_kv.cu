// Fused reshape and block write (vLLM paper review, mz-moonzoo.tistory.com/116,
// §5.1 (1); PagedAttention notes, unpurerationalist.github.io, §4.1): the
// new key and value of every token go straight from the projection layout
// [n_tokens][H][D] to their slot in the block-structured cache
// [num_blocks][H][B][D], one launch for the whole batch.
//
// Two launch shapes, both moving 16-byte vectors with shift-only index
// arithmetic (D / 8 and B are powers of two); reads are fully coalesced and
// writes are contiguous runs of D*2 bytes per (token, head).  The call moves
// 2 * n_tokens * H * D * 2 bytes each way (5.2 MB for 256 OPT-13B tokens).
//  * few tokens (a decode step): one thread per key vector and the matching
//    value vector, CTAs of 128 consecutive vectors of one token, so every
//    load of the call is in flight at once (with a CTA per token only a
//    fifth of them were, and the write was latency-bound);
//  * many tokens (a prompt batch): token-major, a CTA takes a token
//    (grid-stride), reads its slot once and its threads loop over the
//    token's vectors (measured faster there than a thread per vector).
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pagedkv {

namespace {

constexpr int kWriteThreads = 128;

__global__ void __launch_bounds__(kWriteThreads)
write_kv_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                const int64_t *__restrict__ slot_mapping, int32_t n_tokens, int vec_per_tok,
                int row_shift, int bshift, int H, int64_t num_slots, uint4 *__restrict__ k_cache,
                uint4 *__restrict__ v_cache, int32_t *status) {
    const int row_mask = (1 << row_shift) - 1;   // vectors per (token, head) row - 1
    for (int32_t t = blockIdx.x; t < n_tokens; t += gridDim.x) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;                 // token not stored
        if (slot >= num_slots) {
            if (threadIdx.x == 0) report(status, PA_ERR_BAD_BLOCK);
            continue;
        }
        const int64_t blk = slot >> bshift;
        const int off = (int)(slot & ((1 << bshift) - 1));
        const uint4 *ks = k + (int64_t)t * vec_per_tok, *vs = v + (int64_t)t * vec_per_tok;
        // run of head h in the cache: ((blk * H + h) * B + off) rows of D / 8 vectors
        const int64_t base = ((blk * H) << bshift) + off;
#pragma unroll 4
        for (int j = threadIdx.x; j < vec_per_tok; j += kWriteThreads) {
            const int h = j >> row_shift, c = j & row_mask;
            const int64_t dst = ((base + ((int64_t)h << bshift)) << row_shift) + c;
            k_cache[dst] = ks[j];
            v_cache[dst] = vs[j];
        }
    }
}

// One thread per 16-byte vector: CTA b covers vectors [c * 128, c * 128 +
// 128) of token t, with b = t * chunks + c.
__global__ void __launch_bounds__(kWriteThreads)
write_kv_vec_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                    const int64_t *__restrict__ slot_mapping, int vec_per_tok, int chunks,
                    int row_shift, int bshift, int H, int64_t num_slots,
                    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, int32_t *status) {
    const int t = blockIdx.x / chunks;
    const int j = (blockIdx.x - t * chunks) * kWriteThreads + threadIdx.x;
    const int64_t slot = slot_mapping[t];
    if (slot < 0 || j >= vec_per_tok) return;
    if (slot >= num_slots) {
        if (j == 0) report(status, PA_ERR_BAD_BLOCK);
        return;
    }
    const uint4 kv = k[(int64_t)t * vec_per_tok + j];
    const uint4 vv = v[(int64_t)t * vec_per_tok + j];
    const int64_t blk = slot >> bshift;
    const int off = (int)(slot & ((1 << bshift) - 1));
    const int h = j >> row_shift, c = j & ((1 << row_shift) - 1);
    const int64_t dst = (((((blk * H) + h) << bshift) + off) << row_shift) + c;
    k_cache[dst] = kv;
    v_cache[dst] = vv;
}

}  // namespace

int launch_write_kv(const void *k, const void *v, const int64_t *slot_mapping, int32_t n_tokens,
                    void *k_cache, void *v_cache, const pa_pool_desc *d, int32_t *status,
                    void *stream) {
    std::string why;
    if (!d) return fail(PA_ERR_INVALID_ARG, "pa_write_kv: NULL desc");
    if (!device_geometry_ok(d, &why)) return fail(PA_ERR_INVALID_ARG, "pa_write_kv: %s", why.c_str());
    if (n_tokens < 0) return fail(PA_ERR_INVALID_ARG, "pa_write_kv: n_tokens < 0");
    if (n_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache)
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv: NULL pointer");
    auto mis16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
    if (mis16(k) || mis16(v) || mis16(k_cache) || mis16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7))
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv: misaligned pointer");
    const int vec_per_row = d->head_dim / 8;
    int row_shift = 0, bshift = 0;
    while ((1 << row_shift) < vec_per_row) ++row_shift;
    while ((1 << bshift) < d->block_size) ++bshift;
    if ((1 << row_shift) != vec_per_row || (1 << bshift) != d->block_size)
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv: head_dim / 8 and block_size must be powers of two");
    if ((int64_t)d->num_heads * vec_per_row > (1 << 30))
        return fail(PA_ERR_INVALID_ARG, "pa_write_kv: num_heads * head_dim too large");
    const int vec_per_tok = d->num_heads * vec_per_row;
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t num_slots = (int64_t)d->num_blocks * d->block_size;
    const int chunks = (vec_per_tok + kWriteThreads - 1) / kWriteThreads;
    if (n_tokens < sms * 16 && (int64_t)n_tokens * chunks < (1ll << 31)) {
        write_kv_vec_kernel<<<(unsigned)(n_tokens * chunks), kWriteThreads, 0, st>>>(
            static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping,
            vec_per_tok, chunks, row_shift, bshift, d->num_heads, num_slots,
            static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), status);
    } else {
        // resident CTAs: 16 per SM of 128 threads, grid-stride over the tokens
        write_kv_kernel<<<sms * 16, kWriteThreads, 0, st>>>(
            static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, n_tokens,
            vec_per_tok, row_shift, bshift, d->num_heads, num_slots,
            static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), status);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_write_kv: launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

}  // namespace pagedkv
