// Internal declarations shared by the library's translation units.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "../../include/pagedkv.h"

namespace pagedkv {

// Records a formatted message as the calling thread's last error and
// returns `code`, so call sites can write `return fail(PA_ERR_..., "...")`.
int fail(int code, const char *fmt, ...);

// Clears nothing: successful calls leave the last error untouched.
const char *last_error();

// Geometry checks shared by the device entry points.
bool device_geometry_ok(const pa_pool_desc *d, std::string *why);
int partition_tokens_of(const pa_pool_desc *d);

// Kernel launchers (device code lives in the .cu files).
int launch_selftest_bounded_wait(int32_t *status, void *stream);
int launch_write_kv(const void *k, const void *v, const int64_t *slot_mapping, int32_t n_tokens,
                    void *k_cache, void *v_cache, const pa_pool_desc *d, int32_t *status,
                    void *stream);
int launch_copy_blocks(void *const *k_caches, void *const *v_caches, int32_t num_layers,
                       const int32_t *pairs, int32_t n_pairs, const pa_pool_desc *d,
                       int32_t *status, void *stream);
int launch_swap_blocks(const void *const *src_k, const void *const *src_v, int32_t src_blocks,
                       void *const *dst_k, void *const *dst_v, int32_t dst_blocks,
                       int32_t num_layers, const int32_t *pairs, int32_t n_pairs,
                       const pa_pool_desc *d, int32_t *status, void *stream);
size_t decode_workspace_bytes(int32_t n_seqs, int32_t max_blocks, const pa_pool_desc *d);
int launch_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *ctx_lens, int32_t n_seqs,
                            int32_t max_blocks, float scale, void *workspace,
                            size_t workspace_bytes, int32_t *status, const pa_pool_desc *d,
                            void *stream);
int launch_decode_step_attention(void *out, const void *q, const void *k_new, const void *v_new,
                                 const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                 const int32_t *block_tables, const int32_t *ctx_lens,
                                 int32_t n_seqs, int32_t max_blocks, float scale, void *workspace,
                                 size_t workspace_bytes, int32_t *status, const pa_pool_desc *d,
                                 void *stream);
int launch_prefill_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, const int32_t *ctx_lens,
                             const int32_t *q_starts, int32_t n_seqs, int32_t max_blocks,
                             int32_t max_q_len, int32_t q_rows, float scale, int32_t *status,
                             const pa_pool_desc *d, void *stream);

int launch_prefill_step_attention(void *out, const void *q, const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache, const int32_t *block_tables,
                                  const int32_t *ctx_lens, const int32_t *q_starts, int32_t n_seqs,
                                  int32_t max_blocks, int32_t max_q_len, int32_t q_rows,
                                  float scale, int32_t *status, const pa_pool_desc *d, void *stream);

}  // namespace pagedkv
