// Single-query paged decode attention for sm_103a, with split-context
// partitions and a log-sum-exp merge.
//
// What is computed (PagedAttention notes, unpurerationalist.github.io, §3.1,
// blockwise attention equation; vLLM paper review, mz-moonzoo.tistory.com/116,
// §4.1): for each sequence s and head h,
//     o = sum_p softmax_p(scale * q . k_p) v_p   over the ctx stored positions,
// with position p read from physical block table[p / B] at offset p % B
// (KV cache management and PagedAttention tutorial,
// llm-systems-engineering.pages.dev/posts/paged-kv-cache, Fig. 2, Fig. 4).
// The review's §5.1 (2) describes the kernel the pages had: a fused block
// read + attention adapted from FasterTransformer, one warp per block for
// coalesced reads.  This design keeps "one warp owns whole blocks" but moves
// the bytes with the Blackwell bulk-copy engine:
//
//  * grid = (partition, head, sequence); a partition is partition_tokens
//    tokens of one sequence's context (contexts up to one partition need no
//    merge);
//  * each warp owns every WARPS-th block of its partition and runs its own
//    ring of STAGES shared-memory stages; lane 0 issues two 1-D bulk copies
//    per block (the (block, head) key rows and value rows are each one
//    contiguous B*D*2-byte run in the cache layout) completing on that
//    stage's mbarrier, so each warp keeps STAGES-1 blocks in flight with no
//    CTA-wide synchronisation in the main loop;
//  * q.k: lane (g, r) holds dims [8r, 8r+8) of token g of each pass (16-byte
//    shared loads, conflict free); the NP partial dot products per lane are
//    reduced across the row's lanes with a reduce-scatter butterfly, so one
//    block costs NP-1+log2(TPR/NP) shuffles instead of NP*log2(TPR);
//  * online softmax in base 2 (q is pre-scaled by scale*log2 e) with fp32
//    running max / sum per warp; p.v accumulates in fp32 registers;
//  * warps are combined through shared memory; a partition of a split
//    context writes (max, sum, unnormalised output) to the workspace and the
//    merge kernel combines partitions: m = max m_p, l = sum 2^(m_p-m) l_p,
//    o = sum 2^(m_p-m) acc_p / l.  (The pages do not cover the split or the
//    merge; this is the standard log-sum-exp combination of the same sum.)
//
// Slots of the last block past ctx are neither copied (the bulk copy of a
// partial block moves only its valid rows) nor used.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pagedkv {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, int B>
struct Geo {
    static_assert(D % 8 == 0 && D >= 8 && D <= 256, "head_dim");
    static constexpr int TPR = D / 8;                     // lanes per token row
    static constexpr int TPP = 32 / TPR;                  // tokens per pass
    static constexpr int NP = (B + TPP - 1) / TPP;        // passes per block
    static_assert(NP <= TPR, "reduce-scatter layout");
    static constexpr int DUP = TPR / NP;                  // lanes sharing one score
    static constexpr int CHUNK = B * D * 2;               // K (or V) bytes of one (block, head)
    static constexpr int STAGE = 2 * CHUNK;
};

#ifndef PA_ATTN_TARGET_STAGE_BYTES
#define PA_ATTN_TARGET_STAGE_BYTES (96 * 1024)
#endif

template <int D, int B>
struct DefaultCfg {
    static constexpr int STAGE = Geo<D, B>::STAGE;
    static constexpr int WARPS = (8 * STAGE > 200 * 1024) ? 2 : 4;
    static constexpr int S0 = PA_ATTN_TARGET_STAGE_BYTES / (WARPS * STAGE);
    static constexpr int STAGES = S0 < 2 ? 2 : (S0 > 8 ? 8 : S0);
};

template <int D, int B, int WARPS, int STAGES>
struct Smem {
    static constexpr int STAGE_BYTES = WARPS * STAGES * Geo<D, B>::STAGE;
    static constexpr int BAR_OFF = STAGE_BYTES;
    static constexpr int COMB_OFF = BAR_OFF + WARPS * STAGES * 8;
    static constexpr int TOTAL = COMB_OFF + WARPS * (D + 2) * 4 + 128;   // +128: base alignment
};

struct DecodeParams {
    __half *out;
    const __half *q;
    const __half *k_cache;
    const __half *v_cache;
    const int32_t *block_tables;
    const int32_t *ctx_lens;
    float *ws_ml;      // [S][H][max_parts][2]  (max, sum)
    float *ws_acc;     // [S][H][max_parts][D]  unnormalised output
    int32_t *status;
    int32_t n_seqs;
    int32_t num_heads;
    int32_t num_blocks;
    int32_t max_blocks;
    int32_t part_blocks;
    int32_t max_parts;
    float qscale;      // scale * log2(e)
};

// Sum NP partial values over the TPR lanes of a row group.  On return the
// lane holds the full sum of value index idx(r) (see token_index_of).
template <int NP, int TPR>
__device__ __forceinline__ float row_reduce_scatter(float (&v)[NP], int r) {
#pragma unroll
    for (int k = 0; (NP >> k) > 1; ++k) {
        const int half = NP >> (k + 1);
        const int off = TPR >> (k + 1);
        const bool upper = (r & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(kFull, send, off);
        }
    }
    float x = v[0];
#pragma unroll
    for (int off = TPR / NP / 2; off >= 1; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
    return x;
}

template <int NP, int TPR>
__device__ __forceinline__ int token_index_of(int r) {
    int idx = 0;
#pragma unroll
    for (int k = 0; (NP >> k) > 1; ++k)
        if (r & (TPR >> (k + 1))) idx += NP >> (k + 1);
    return idx;
}

template <int D, int B, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32)
paged_decode_kernel(const DecodeParams p) {
    using G = Geo<D, B>;
    using L = Smem<D, B, WARPS, STAGES>;
    constexpr int TPR = G::TPR, TPP = G::TPP, NP = G::NP, DUP = G::DUP;
    constexpr int CHUNK = G::CHUNK, STAGE = G::STAGE;

    const int part = blockIdx.x;
    const int h = blockIdx.y;
    const int s = blockIdx.z;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int H = p.num_heads;

    const int ctx = p.ctx_lens[s];
    __half *out_row = p.out + ((size_t)s * H + h) * D;
    if (ctx <= 0) {
        if (part == 0)
            for (int i = tid; i < D; i += WARPS * 32) out_row[i] = __float2half(0.f);
        return;
    }
    if (ctx > p.max_blocks * B) {   // the table row cannot hold this context
        if (part == 0 && tid == 0) report(p.status, PA_ERR_BAD_BLOCK);
        return;
    }
    const int nblk = (ctx + B - 1) / B;
    const int n_parts = (nblk + p.part_blocks - 1) / p.part_blocks;
    if (part >= n_parts) return;
    const int j0 = part * p.part_blocks;
    const int nb_part = min(p.part_blocks, nblk - j0);
    const int n_w = nb_part > warp ? (nb_part - warp + WARPS - 1) / WARPS : 0;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint8_t *stages = smem + warp * STAGES * STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF) + warp * STAGES;
    float *comb = reinterpret_cast<float *>(smem + L::COMB_OFF);

    const int r = lane % TPR;
    const int g = lane / TPR;

    // q, dims [8r, 8r+8), pre-scaled into log2 units.
    float qf[8];
    {
        const uint4 u =
            *reinterpret_cast<const uint4 *>(p.q + ((size_t)s * H + h) * D + r * 8);
        half8_to_float8(u, qf);
#pragma unroll
        for (int i = 0; i < 8; ++i) qf[i] *= p.qscale;
    }

    const size_t blk_stride = (size_t)H * B * D;
    const __half *kbase = p.k_cache + (size_t)h * B * D;
    const __half *vbase = p.v_cache + (size_t)h * B * D;
    const int32_t *trow = p.block_tables + (size_t)s * p.max_blocks + j0 + warp;

    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < STAGES; ++st) mbar_init(smem_addr(&bars[st]), 1);
        fence_barrier_init();
    }
    __syncwarp();

    const uint64_t policy = l2_evict_first_policy();
    int tbl = -1;   // lane i: physical block of this warp's block (32*chunk + i)

    // Issue the copies of this warp's i-th block into stage i % STAGES.
    // Called by the whole warp with increasing i.
    auto issue = [&](int i) {
        if ((i & 31) == 0) {
            const int e = i + lane;
            tbl = e < n_w ? trow[(size_t)e * WARPS] : -1;
        }
        const int phys = __shfl_sync(kFull, tbl, i & 31);
        if (lane == 0) {
            const int j = j0 + warp + WARPS * i;
            const int nv = min(B, ctx - j * B);
            const uint32_t bytes = (uint32_t)nv * D * 2;
            const int st = i % STAGES;
            const uint32_t bar = smem_addr(&bars[st]);
            const uint32_t dst = smem_addr(stages + st * STAGE);
            if (phys >= 0 && phys < p.num_blocks) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, 2 * bytes);
                bulk_g2s(dst, kbase + (size_t)phys * blk_stride, bytes, bar, policy);
                bulk_g2s(dst + CHUNK, vbase + (size_t)phys * blk_stride, bytes, bar, policy);
            } else {
                report(p.status, PA_ERR_BAD_BLOCK);
                mbar_arrive(bar);
            }
        }
    };

    const int pro = min(STAGES, n_w);
    for (int i = 0; i < pro; ++i) issue(i);

    const int my_idx = token_index_of<NP, TPR>(r);
    const int my_tok = my_idx * TPP + g;

    float m = -INFINITY;
    float lsum = 0.f;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;

    for (int i = 0; i < n_w; ++i) {
        const int st = i % STAGES;
        const uint32_t parity = (uint32_t)(i / STAGES) & 1u;
        if (!mbar_wait_bounded(smem_addr(&bars[st]), parity, p.status, true)) {
            report(p.status, PA_ERR_TIMEOUT);
            // Let copies already in flight land before the CTA can exit.
            const int last = min(n_w, i + STAGES);
            for (int k = i; k < last; ++k)
                mbar_wait_bounded(smem_addr(&bars[k % STAGES]), (uint32_t)(k / STAGES) & 1u,
                                  p.status, false);
            break;
        }
        const int j = j0 + warp + WARPS * i;
        const int nv = min(B, ctx - j * B);
        const uint8_t *kst = stages + st * STAGE;
        const uint8_t *vst = kst + CHUNK;

        // scores: partial q.k over this lane's 8 dims, one per pass
        float part_dot[NP];
#pragma unroll
        for (int ps = 0; ps < NP; ++ps) {
            const int t = ps * TPP + g;
            float d = 0.f;
            if (TPP * NP == B || t < B) {
                const uint4 u = *reinterpret_cast<const uint4 *>(kst + t * (D * 2) + r * 16);
                float kf[8];
                half8_to_float8(u, kf);
#pragma unroll
                for (int c = 0; c < 8; ++c) d = fmaf(qf[c], kf[c], d);
            }
            part_dot[ps] = d;
        }
        float sc = row_reduce_scatter<NP, TPR>(part_dot, r);
        if (my_tok >= nv) sc = -INFINITY;

        float bm = sc;
#pragma unroll
        for (int off = DUP; off < 32; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, off));
        if (bm > m) {   // warp-uniform
            const float a = exp2f(m - bm);
            lsum *= a;
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] *= a;
            m = bm;
        }
        const float pr = exp2f(sc - m);
        lsum += pr;

#pragma unroll
        for (int ps = 0; ps < NP; ++ps) {
            const int t = ps * TPP + g;
            const float pt = __shfl_sync(kFull, pr, g * TPR + ps * DUP);
            if (t < nv) {
                const uint4 u = *reinterpret_cast<const uint4 *>(vst + t * (D * 2) + r * 16);
                float vf[8];
                half8_to_float8(u, vf);
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[c] = fmaf(pt, vf[c], acc[c]);
            }
        }
        __syncwarp();
        if (i + STAGES < n_w) issue(i + STAGES);
    }

    // warp totals: output over token groups, sum over all lanes
#pragma unroll
    for (int off = TPR; off < 32; off <<= 1)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += __shfl_xor_sync(kFull, acc[c], off);
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) lsum += __shfl_xor_sync(kFull, lsum, off);
    lsum *= 1.0f / DUP;

    float *cw = comb + warp * (D + 2);
    if (g == 0) {
#pragma unroll
        for (int c = 0; c < 8; ++c) cw[r * 8 + c] = acc[c];
    }
    if (lane == 0) {
        cw[D] = m;
        cw[D + 1] = lsum;
    }
    __syncthreads();

    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, comb[w * (D + 2) + D]);
    float wgt[WARPS];
    float Lt = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        wgt[w] = exp2f(comb[w * (D + 2) + D] - M);
        Lt = fmaf(wgt[w], comb[w * (D + 2) + D + 1], Lt);
    }
    if (n_parts == 1) {
        const float inv = 1.0f / Lt;
        for (int i = tid; i < D; i += WARPS * 32) {
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < WARPS; ++w) o = fmaf(wgt[w], comb[w * (D + 2) + i], o);
            out_row[i] = __float2half(o * inv);
        }
    } else {
        const size_t idx = ((size_t)s * H + h) * p.max_parts + part;
        if (tid == 0) {
            p.ws_ml[2 * idx] = M;
            p.ws_ml[2 * idx + 1] = Lt;
        }
        float *wacc = p.ws_acc + idx * D;
        for (int i = tid; i < D; i += WARPS * 32) {
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < WARPS; ++w) o = fmaf(wgt[w], comb[w * (D + 2) + i], o);
            wacc[i] = o;
        }
    }
}

// One warp per (sequence, head) whose context spans more than one partition.
template <int D>
__global__ void __launch_bounds__(128) paged_merge_kernel(const DecodeParams p, int part_tokens) {
    const int gw = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    const int H = p.num_heads;
    if (gw >= p.n_seqs * H) return;
    const int s = gw / H;
    const int h = gw % H;
    const int ctx = p.ctx_lens[s];
    const int n_parts = ctx > 0 ? (ctx + part_tokens - 1) / part_tokens : 0;
    if (n_parts <= 1 || n_parts > p.max_parts) return;
    const size_t base = ((size_t)s * H + h) * p.max_parts;
    float M = -INFINITY;
    for (int q = lane; q < n_parts; q += 32) M = fmaxf(M, p.ws_ml[2 * (base + q)]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    float Lt = 0.f;
    for (int q = lane; q < n_parts; q += 32)
        Lt += exp2f(p.ws_ml[2 * (base + q)] - M) * p.ws_ml[2 * (base + q) + 1];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) Lt += __shfl_xor_sync(kFull, Lt, off);
    const float inv = 1.0f / Lt;
    __half *out_row = p.out + ((size_t)s * H + h) * D;
    for (int d = lane; d < D; d += 32) {
        float o = 0.f;
        for (int q = 0; q < n_parts; ++q)
            o = fmaf(exp2f(p.ws_ml[2 * (base + q)] - M), p.ws_acc[(base + q) * D + d], o);
        out_row[d] = __float2half(o * inv);
    }
}

template <int D, int B, int WARPS, int STAGES>
int launch_cfg(const DecodeParams &prm, int part_tokens, cudaStream_t stream) {
    using L = Smem<D, B, WARPS, STAGES>;
    auto kern = paged_decode_kernel<D, B, WARPS, STAGES>;
    // Raising the dynamic shared-memory limit is per device; do it once each.
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return fail(PA_ERR_CUDA, "pa_decode_attention: cudaGetDevice failed");
    std::call_once(once[dev], [&] {
        attr_err[dev] =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    });
    if (attr_err[dev] != cudaSuccess)
        return fail(PA_ERR_CUDA, "pa_decode_attention: cudaFuncSetAttribute: %s",
                    cudaGetErrorString(attr_err[dev]));
    dim3 grid(prm.max_parts, prm.num_heads, prm.n_seqs);
    kern<<<grid, WARPS * 32, L::TOTAL, stream>>>(prm);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "pa_decode_attention: launch: %s", cudaGetErrorString(e));
    if (prm.max_parts > 1) {
        const int64_t warps = (int64_t)prm.n_seqs * prm.num_heads;
        const unsigned blocks = (unsigned)((warps + 3) / 4);
        paged_merge_kernel<D><<<blocks, 128, 0, stream>>>(prm, part_tokens);
        e = cudaGetLastError();
        if (e != cudaSuccess)
            return fail(PA_ERR_CUDA, "pa_decode_attention: merge launch: %s",
                        cudaGetErrorString(e));
    }
    return PA_OK;
}

template <int D, int B>
int launch_db(const DecodeParams &prm, int part_tokens, cudaStream_t stream) {
#if defined(PA_TUNE_WARPS) && defined(PA_TUNE_STAGES)
    if (D == 128 && B == 16)
        return launch_cfg<D, B, PA_TUNE_WARPS, PA_TUNE_STAGES>(prm, part_tokens, stream);
#endif
    return launch_cfg<D, B, DefaultCfg<D, B>::WARPS, DefaultCfg<D, B>::STAGES>(prm, part_tokens,
                                                                             stream);
}

template <int D>
int launch_d(int B, const DecodeParams &prm, int part_tokens, cudaStream_t stream) {
    switch (B) {
        case 4: return launch_db<D, 4>(prm, part_tokens, stream);
        case 8: return launch_db<D, 8>(prm, part_tokens, stream);
        case 16: return launch_db<D, 16>(prm, part_tokens, stream);
        case 32: return launch_db<D, 32>(prm, part_tokens, stream);
    }
    return fail(PA_ERR_INVALID_ARG, "pa_decode_attention: unsupported block_size %d", B);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int max_parts_of(int32_t max_blocks, int part_blocks) {
    return max_blocks > 0 ? (max_blocks + part_blocks - 1) / part_blocks : 1;
}

}  // namespace

size_t decode_workspace_bytes(int32_t n_seqs, int32_t max_blocks, const pa_pool_desc *d) {
    std::string why;
    if (!d || n_seqs < 0 || max_blocks < 0 || !device_geometry_ok(d, &why)) return 0;
    const int part_blocks = partition_tokens_of(d) / d->block_size;
    const int mp = max_parts_of(max_blocks, part_blocks);
    if (mp <= 1) return 0;
    const size_t rows = (size_t)n_seqs * d->num_heads * mp;
    return align256(rows * 2 * sizeof(float)) + align256(rows * d->head_dim * sizeof(float));
}

int launch_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *ctx_lens, int32_t n_seqs,
                            int32_t max_blocks, float scale, void *workspace,
                            size_t workspace_bytes, int32_t *status, const pa_pool_desc *d,
                            void *stream) {
    std::string why;
    if (!d) return fail(PA_ERR_INVALID_ARG, "pa_decode_attention: NULL desc");
    if (!device_geometry_ok(d, &why))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_attention: %s", why.c_str());
    if (n_seqs < 0 || n_seqs > 65535 || max_blocks < 0 || d->num_heads > 65535)
        return fail(PA_ERR_INVALID_ARG,
                    "pa_decode_attention: n_seqs=%d (<= 65535), max_blocks=%d, num_heads=%d",
                    n_seqs, max_blocks, d->num_heads);
    if (n_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !ctx_lens || (max_blocks > 0 && !block_tables))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_attention: NULL pointer");
    auto mis16 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) != 0; };
    if (mis16(out) || mis16(q) || mis16(k_cache) || mis16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_attention: out/q/caches must be 16-byte aligned");
    if (!std::isfinite(scale))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_attention: scale is not finite");
    const int part_tokens = partition_tokens_of(d);
    const int part_blocks = part_tokens / d->block_size;
    const int mp = max_parts_of(max_blocks, part_blocks);
    const size_t need = decode_workspace_bytes(n_seqs, max_blocks, d);
    if (need > 0) {
        if (!workspace || workspace_bytes < need)
            return fail(PA_ERR_INVALID_ARG,
                        "pa_decode_attention: workspace of %zu bytes needed, %zu given", need,
                        workspace ? workspace_bytes : (size_t)0);
        if (reinterpret_cast<uintptr_t>(workspace) & 255)
            return fail(PA_ERR_INVALID_ARG, "pa_decode_attention: workspace must be 256-byte aligned");
    }
    DecodeParams prm{};
    prm.out = static_cast<__half *>(out);
    prm.q = static_cast<const __half *>(q);
    prm.k_cache = static_cast<const __half *>(k_cache);
    prm.v_cache = static_cast<const __half *>(v_cache);
    prm.block_tables = block_tables;
    prm.ctx_lens = ctx_lens;
    const size_t rows = (size_t)n_seqs * d->num_heads * mp;
    prm.ws_ml = need ? static_cast<float *>(workspace) : nullptr;
    prm.ws_acc = need ? reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                  align256(rows * 2 * sizeof(float)))
                      : nullptr;
    prm.status = status;
    prm.n_seqs = n_seqs;
    prm.num_heads = d->num_heads;
    prm.num_blocks = d->num_blocks;
    prm.max_blocks = max_blocks;
    prm.part_blocks = part_blocks;
    prm.max_parts = mp;
    prm.qscale = scale * kLog2e;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (d->head_dim) {
        case 8: return launch_d<8>(d->block_size, prm, part_tokens, st);
        case 16: return launch_d<16>(d->block_size, prm, part_tokens, st);
        case 32: return launch_d<32>(d->block_size, prm, part_tokens, st);
        case 64: return launch_d<64>(d->block_size, prm, part_tokens, st);
        case 128: return launch_d<128>(d->block_size, prm, part_tokens, st);
        case 256: return launch_d<256>(d->block_size, prm, part_tokens, st);
    }
    return fail(PA_ERR_INVALID_ARG, "pa_decode_attention: unsupported head_dim %d", d->head_dim);
}

}  // namespace pagedkv
