// Fused reshape and block write (vLLM paper review, mz-moonzoo.tistory.com/116,
// §5.1 (1); PagedAttention notes, unpurerationalist.github.io, §4.1): the
// new key and value of every token go straight from the projection layout
// [n_tokens][H][D] to their slot in the block-structured cache
// [num_blocks][H][B][D], one launch for the whole batch.
//
// One thread moves one 16-byte vector (8 halves) of a key row and the same
// vector of the value row: reads are fully coalesced, writes are contiguous
// runs of D*2 bytes per (token, head).  This kernel moves
// 2 * n_tokens * H * D * 2 bytes each way (~2.6 MB for 256 OPT-13B tokens),
// microseconds next to the attention it feeds.
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pagedkv {

namespace {

__global__ void __launch_bounds__(256)
write_kv_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                const int64_t *__restrict__ slot_mapping, int64_t n_vec, int vec_per_tok,
                int vec_per_row, int H, int B, int64_t num_slots, uint4 *__restrict__ k_cache,
                uint4 *__restrict__ v_cache, int32_t *status) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_vec;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / vec_per_tok;
        const int rem = (int)(i - t * vec_per_tok);
        const int h = rem / vec_per_row;
        const int c = rem - h * vec_per_row;
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;                 // token not stored
        if (slot >= num_slots) {
            report(status, PA_ERR_BAD_BLOCK);
            continue;
        }
        const int64_t blk = slot / B;
        const int off = (int)(slot - blk * B);
        const int64_t dst = ((blk * H + h) * B + off) * vec_per_row + c;
        k_cache[dst] = k[i];
        v_cache[dst] = v[i];
    }
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
    const int vec_per_tok = d->num_heads * vec_per_row;
    const int64_t n_vec = (int64_t)n_tokens * vec_per_tok;
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (n_vec + 255) / 256;
    const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    write_kv_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, n_vec,
        vec_per_tok, vec_per_row, d->num_heads, d->block_size,
        (int64_t)d->num_blocks * d->block_size, static_cast<uint4 *>(k_cache),
        static_cast<uint4 *>(v_cache), status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_write_kv: launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

}  // namespace pagedkv
