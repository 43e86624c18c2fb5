// C ABI entry points of the device calls, the thread-local error text and the
// geometry checks they share.  The block-manager entry points are in pool.cpp.
#include <cstring>
#include <string>

#include "pa_internal.h"

namespace pagedkv {

namespace {
thread_local std::string g_last_error;
}

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

const char *last_error() { return g_last_error.c_str(); }

int partition_tokens_of(const pa_pool_desc *d) {
    return d->partition_tokens > 0 ? d->partition_tokens : PA_DEFAULT_PARTITION_TOKENS;
}

bool device_geometry_ok(const pa_pool_desc *d, std::string *why) {
    char buf[256];
    const int B = d->block_size, D = d->head_dim;
    if (d->dtype != PA_DTYPE_F16) {
        *why = "dtype must be PA_DTYPE_F16";
        return false;
    }
    if (!(B == 4 || B == 8 || B == 16 || B == 32)) {
        std::snprintf(buf, sizeof buf, "block_size %d not in {4, 8, 16, 32}", B);
        *why = buf;
        return false;
    }
    if (!(D == 8 || D == 16 || D == 32 || D == 64 || D == 128 || D == 256)) {
        std::snprintf(buf, sizeof buf, "head_dim %d not in {8, 16, 32, 64, 128, 256}", D);
        *why = buf;
        return false;
    }
    if (d->num_heads < 1 || d->num_blocks < 0) {
        *why = "num_heads must be >= 1 and num_blocks >= 0";
        return false;
    }
    const int pt = partition_tokens_of(d);
    if (d->partition_tokens < 0 || pt % B != 0) {
        std::snprintf(buf, sizeof buf, "partition_tokens %d is not a positive multiple of %d",
                      d->partition_tokens, B);
        *why = buf;
        return false;
    }
    return true;
}

}  // namespace pagedkv

using namespace pagedkv;

extern "C" {

const char *pa_last_error_string(void) { return last_error(); }

int pa_selftest_bounded_wait(int32_t *status, void *stream) {
    return launch_selftest_bounded_wait(status, stream);
}

int pa_write_kv(const void *k, const void *v, const int64_t *slot_mapping, int32_t n_tokens,
                void *k_cache, void *v_cache, const pa_pool_desc *desc, int32_t *status,
                void *stream) {
    return launch_write_kv(k, v, slot_mapping, n_tokens, k_cache, v_cache, desc, status, stream);
}

int pa_copy_blocks(void *const *k_caches, void *const *v_caches, int32_t num_layers,
                   const int32_t *pairs, int32_t n_pairs, const pa_pool_desc *desc,
                   int32_t *status, void *stream) {
    return launch_copy_blocks(k_caches, v_caches, num_layers, pairs, n_pairs, desc, status,
                              stream);
}

int pa_swap_blocks(const void *const *src_k, const void *const *src_v, int32_t src_num_blocks,
                   void *const *dst_k, void *const *dst_v, int32_t dst_num_blocks,
                   int32_t num_layers, const int32_t *pairs, int32_t n_pairs,
                   const pa_pool_desc *desc, int32_t *status, void *stream) {
    return launch_swap_blocks(src_k, src_v, src_num_blocks, dst_k, dst_v, dst_num_blocks,
                              num_layers, pairs, n_pairs, desc, status, stream);
}

size_t pa_decode_workspace_bytes(int32_t n_seqs, int32_t max_blocks, const pa_pool_desc *desc) {
    return decode_workspace_bytes(n_seqs, max_blocks, desc);
}

int pa_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, const int32_t *ctx_lens, int32_t n_seqs,
                        int32_t max_blocks, float scale, void *workspace, size_t workspace_bytes,
                        int32_t *status, const pa_pool_desc *desc, void *stream) {
    return launch_decode_attention(out, q, k_cache, v_cache, block_tables, ctx_lens, n_seqs,
                                   max_blocks, scale, workspace, workspace_bytes, status, desc,
                                   stream);
}

int pa_decode_step_attention(void *out, const void *q, const void *k_new, const void *v_new,
                             const int64_t *slot_mapping, void *k_cache, void *v_cache,
                             const int32_t *block_tables, const int32_t *ctx_lens, int32_t n_seqs,
                             int32_t max_blocks, float scale, void *workspace,
                             size_t workspace_bytes, int32_t *status, const pa_pool_desc *desc,
                             void *stream) {
    return launch_decode_step_attention(out, q, k_new, v_new, slot_mapping, k_cache, v_cache,
                                        block_tables, ctx_lens, n_seqs, max_blocks, scale,
                                        workspace, workspace_bytes, status, desc, stream);
}

int pa_prefill_step_attention(void *out, const void *q, const void *k_new, const void *v_new,
                              void *k_cache, void *v_cache, const int32_t *block_tables,
                              const int32_t *ctx_lens, const int32_t *q_starts, int32_t n_seqs,
                              int32_t max_blocks, int32_t max_q_len, int32_t q_rows, float scale,
                              int32_t *status, const pa_pool_desc *desc, void *stream) {
    return launch_prefill_step_attention(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                                         ctx_lens, q_starts, n_seqs, max_blocks, max_q_len, q_rows,
                                         scale, status, desc, stream);
}

int pa_prefill_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *ctx_lens,
                         const int32_t *q_starts, int32_t n_seqs, int32_t max_blocks,
                         int32_t max_q_len, int32_t q_rows, float scale, int32_t *status,
                         const pa_pool_desc *desc, void *stream) {
    return launch_prefill_attention(out, q, k_cache, v_cache, block_tables, ctx_lens, q_starts,
                                    n_seqs, max_blocks, max_q_len, q_rows, scale, status, desc,
                                    stream);
}

}  // extern "C"
