// Causal paged prefill attention: every query of a prompt (or of a chunk
// appended to a cached prefix) attends to the positions up to its own,
// reading keys and values through the block table.
//
// What it computes: the prompt phase of the vLLM paper review (§4.3), where
// the prompt's tokens are processed together and each one attends to the
// tokens before it and itself, with the blockwise attention equation of the
// PagedAttention notes (§3.1) evaluated for each of those queries.
//
// Kernel design (sm_103a, tensor cores through mma.sync m16n8k16):
//   - one CTA = (sequence, head, tile of 64 consecutive queries); 4 warps,
//     16 query rows each.  Later query tiles (more keys) are launched first.
//   - keys and values stream through shared memory in tiles of 64 positions,
//     double-buffered with 16-byte cp.async copies.  A row's physical address
//     comes from the block table (block j / B, offset j % B); in the cache
//     layout [block][head][B][D] each (block, head) run is B*D*2 contiguous
//     bytes, so a tile is a handful of contiguous runs.  Rows are stored
//     with the 16-byte chunks XOR-swizzled by (row % 8), so ldmatrix reads
//     hit eight different bank groups.
//   - S = Q K^T accumulates in fp32; the online softmax runs in base 2 on the
//     accumulator fragments; P V uses P as the sum of two fp16 terms
//     (hi = fp16(p), lo = fp16(p - hi)), which keeps the probabilities to
//     about 22 bits so the fp16 output is limited by its own rounding.
//   - positions past the causal end of the tile are zero-filled, and scores
//     of keys after a row's own position are masked to -inf.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pagedkv {
namespace {

constexpr int kBM = 64;        // queries per CTA
constexpr int kBN = 64;        // key positions per tile
constexpr int kThreads = 128;  // 4 warps x 16 query rows

struct PrefillParams {
    __half *out;
    const __half *q;
    const __half *k_cache;
    const __half *v_cache;
    const int32_t *tables;
    const int32_t *ctx_lens;
    const int32_t *q_starts;
    int32_t num_heads, num_blocks, max_blocks, max_q_len, q_tiles, bshift;
    float qscale;  // scale * log2(e): softmax evaluated with exp2
    int32_t *status;
};

// Byte offset of 16-byte chunk c of row r in a swizzled [rows][D] fp16 tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// c += a (16x16, row) * b (16x8, col); fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two probabilities as fp16 pairs hi + lo (lower column in the low half).
__device__ __forceinline__ void split_pair(float p0, float p1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(p0, p1);
    const __half2 l = __floats2half2_rn(p0 - __low2float(h), p1 - __high2float(h));
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

template <int D>
constexpr int prefill_smem_bytes() {
    return kBM * D * 2 + 4 * kBN * D * 2;  // Q tile + two K and two V tiles
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2) paged_prefill_mma(const PrefillParams p) {
    constexpr int CPR = D / 8;                 // 16-byte chunks per row
    constexpr int RPP = kThreads / CPR;        // rows covered by one pass of the CTA
    constexpr int NLD = kBN * CPR / kThreads;  // chunks per thread per tile
    constexpr int TILE = kBN * D * 2;
    static_assert(kBM == kBN && CPR >= 8 && kThreads % CPR == 0, "tile geometry");
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sQ = smem_addr(smem);
    const uint32_t sK = sQ + kBM * D * 2;
    const uint32_t sV = sK + 2 * TILE;

    const int s = blockIdx.z, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q_beg = p.q_starts[s];
    const int ql = p.q_starts[s + 1] - q_beg;
    const int ctx = p.ctx_lens[s];
    const bool bad_len = ql < 0 || ql > ctx || ql > p.max_q_len;
    const bool bad_ctx = (int64_t)ctx > ((int64_t)p.max_blocks << p.bshift);
    if (bad_len || bad_ctx) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0)
            report(p.status, bad_len ? PA_ERR_INVALID_ARG : PA_ERR_BAD_BLOCK);
        return;
    }
    const int q0 = (p.q_tiles - 1 - (int)blockIdx.x) * kBM;  // later tiles first
    if (q0 >= ql) return;

    const int pos0 = ctx - ql;                   // position of query 0 of the sequence
    const int rows = min(kBM, ql - q0);
    const int n_end = pos0 + q0 + rows;          // this tile needs keys [0, n_end)
    const int n_tiles = (n_end + kBN - 1) / kBN;
    const int B = 1 << p.bshift;
    const int c = tid % CPR, r0 = tid / CPR;
    const int32_t *table = p.tables + (size_t)s * p.max_blocks;

    // Q tile: rows past the sequence's last query are zero-filled.
    for (int i = 0; i < NLD; ++i) {
        const int r = r0 + i * RPP;
        const bool v = r < rows;
        const __half *src = p.q + ((size_t)(q_beg + q0 + (v ? r : 0)) * p.num_heads + h) * D + c * 8;
        cp_async16(sQ + swz<D>(r, c), src, v);
    }
    auto load_kv = [&](int t, int buf) {
        const int n0 = t * kBN;
        for (int i = 0; i < NLD; ++i) {
            const int r = r0 + i * RPP;
            const int j = n0 + r;
            bool v = j < n_end;
            size_t off = 0;
            if (v) {
                const int phys = __ldg(table + (j >> p.bshift));
                if (phys < 0 || phys >= p.num_blocks) {
                    report(p.status, PA_ERR_BAD_BLOCK);
                    v = false;
                } else {
                    off = (((size_t)phys * p.num_heads + h) * B + (j & (B - 1))) * D + c * 8;
                }
            }
            cp_async16(sK + buf * TILE + swz<D>(r, c), p.k_cache + off, v);
            cp_async16(sV + buf * TILE + swz<D>(r, c), p.v_cache + off, v);
        }
        cp_async_commit();
    };
    load_kv(0, 0);  // one group: Q and the first key/value tile
    cp_async_wait<0>();
    __syncthreads();

    const int mi = lane >> 3;                   // ldmatrix: which 8x8 matrix this lane addresses
    uint32_t qf[D / 16][4];
    {
        const int r = warp * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            ldsm_x4(sQ + swz<D>(r, 2 * kk + (mi >> 1)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
    }

    const int g = lane >> 2, tq = lane & 3;
    const int wq = q0 + warp * 16;               // first query of this warp
    const bool active = wq < ql;
    const int pos_r[2] = {pos0 + min(wq + g, ql - 1), pos0 + min(wq + g + 8, ql - 1)};
    const int wpos_min = pos0 + min(wq, ql - 1);
    const int wpos_max = pos0 + min(wq + 15, ql - 1);

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    for (int t = 0; t < n_tiles; ++t) {
        const int buf = t & 1;
        if (t + 1 < n_tiles) {
            load_kv(t + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int n0 = t * kBN;
        if (active && n0 <= wpos_max) {
            // S = Q K^T for this warp's 16 rows and the tile's 64 keys
            float sc[kBN / 8][4];
#pragma unroll
            for (int j = 0; j < kBN / 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
            const uint32_t kb = sK + buf * TILE;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
                for (int jp = 0; jp < kBN / 16; ++jp) {
                    const int r = jp * 16 + (mi >> 1) * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + swz<D>(r, 2 * kk + (mi & 1)), b0, b1, b2, b3);
                    mma16816(sc[2 * jp], qf[kk], b0, b1);
                    mma16816(sc[2 * jp + 1], qf[kk], b2, b3);
                }
            }
            // online softmax, base 2
            const bool mask = n0 + kBN - 1 > wpos_min;
            float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < kBN / 8; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float x = sc[j][e] * p.qscale;
                    if (mask && n0 + 8 * j + 2 * tq + (e & 1) > pos_r[e >> 1]) x = -INFINITY;
                    sc[j][e] = x;
                    mt[e >> 1] = fmaxf(mt[e >> 1], x);
                }
            }
            float corr[2], ls[2] = {0.f, 0.f};
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                mt[rr] = fmaxf(mt[rr], __shfl_xor_sync(0xffffffffu, mt[rr], 1));
                mt[rr] = fmaxf(mt[rr], __shfl_xor_sync(0xffffffffu, mt[rr], 2));
                const float mn = fmaxf(m_run[rr], mt[rr]);  // finite: key 0 is in tile 0
                corr[rr] = exp2f(m_run[rr] - mn);
                m_run[rr] = mn;
            }
#pragma unroll
            for (int j = 0; j < kBN / 8; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float pe = exp2f(sc[j][e] - m_run[e >> 1]);
                    sc[j][e] = pe;
                    ls[e >> 1] += pe;
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) l_run[rr] = l_run[rr] * corr[rr] + ls[rr];
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                o[i][0] *= corr[0];
                o[i][1] *= corr[0];
                o[i][2] *= corr[1];
                o[i][3] *= corr[1];
            }
            // O += P V, P as hi + lo fp16 operands
            const uint32_t vb = sV + buf * TILE;
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk) {
                uint32_t ah[4], al[4];
                split_pair(sc[2 * kk][0], sc[2 * kk][1], ah[0], al[0]);
                split_pair(sc[2 * kk][2], sc[2 * kk][3], ah[1], al[1]);
                split_pair(sc[2 * kk + 1][0], sc[2 * kk + 1][1], ah[2], al[2]);
                split_pair(sc[2 * kk + 1][2], sc[2 * kk + 1][3], ah[3], al[3]);
                const int r = kk * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vb + swz<D>(r, 2 * dp + (mi >> 1)), b0, b1, b2, b3);
                    mma16816(o[2 * dp], ah, b0, b1);
                    mma16816(o[2 * dp], al, b0, b1);
                    mma16816(o[2 * dp + 1], ah, b2, b3);
                    mma16816(o[2 * dp + 1], al, b2, b3);
                }
            }
        }
        __syncthreads();  // every warp is done with buffer `buf` before it is refilled
    }

    // Normalise, stage the warp's rows in its own part of the Q tile, then
    // store them as 16-byte vectors.
    if (!active) return;
    float inv[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        float l = l_run[rr];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        inv[rr] = 1.f / l;
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        const __half2 a = __floats2half2_rn(o[i][0] * inv[0], o[i][1] * inv[0]);
        const __half2 b = __floats2half2_rn(o[i][2] * inv[1], o[i][3] * inv[1]);
        const int ra = warp * 16 + g, rb = ra + 8;
        asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sQ + swz<D>(ra, i) + 4 * tq),
                     "r"(*reinterpret_cast<const uint32_t *>(&a))
                     : "memory");
        asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sQ + swz<D>(rb, i) + 4 * tq),
                     "r"(*reinterpret_cast<const uint32_t *>(&b))
                     : "memory");
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 16 * CPR / 32; ++i) {
        const int idx = lane + 32 * i;
        const int r = idx / CPR, cc = idx % CPR;
        if (wq + r < ql) {
            uint4 val;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                         : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                         : "r"(sQ + swz<D>(warp * 16 + r, cc)));
            *reinterpret_cast<uint4 *>(p.out + ((size_t)(q_beg + wq + r) * p.num_heads + h) * D +
                                       cc * 8) = val;
        }
    }
}

template <int D>
cudaError_t set_prefill_smem_once() {
    static std::once_flag once[64];
    static cudaError_t err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        err[dev] = cudaFuncSetAttribute(paged_prefill_mma<D>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        prefill_smem_bytes<D>());
    });
    return err[dev];
}

template <int D>
int launch_d(const PrefillParams &p, int n_seqs, cudaStream_t st) {
    cudaError_t e = set_prefill_smem_once<D>();
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "prefill smem attribute: %s", cudaGetErrorString(e));
    const dim3 grid((unsigned)p.q_tiles, (unsigned)p.num_heads, (unsigned)n_seqs);
    paged_prefill_mma<D><<<grid, kThreads, prefill_smem_bytes<D>(), st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

}  // namespace

int launch_prefill_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, const int32_t *ctx_lens,
                             const int32_t *q_starts, int32_t n_seqs, int32_t max_blocks,
                             int32_t max_q_len, float scale, int32_t *status,
                             const pa_pool_desc *d, void *stream) {
    if (!d) return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: desc is NULL");
    std::string why;
    if (!device_geometry_ok(d, &why)) return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: %s", why.c_str());
    if (d->head_dim != 64 && d->head_dim != 128)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: head_dim %d not in {64, 128}",
                    d->head_dim);
    if (n_seqs < 0 || max_blocks < 0 || max_q_len < 0)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: negative size");
    if (n_seqs > 65535 || d->num_heads > 65535)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: more than 65535 sequences or heads");
    if (n_seqs == 0 || max_q_len == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !ctx_lens || !q_starts)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: NULL pointer");
    if (((uintptr_t)out | (uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache) & 15)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: out, q and caches must be 16-byte aligned");
    if (max_blocks < 1) return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: max_blocks < 1");
    int bshift = 0;
    while ((1 << bshift) < d->block_size) ++bshift;
    PrefillParams p;
    p.out = static_cast<__half *>(out);
    p.q = static_cast<const __half *>(q);
    p.k_cache = static_cast<const __half *>(k_cache);
    p.v_cache = static_cast<const __half *>(v_cache);
    p.tables = block_tables;
    p.ctx_lens = ctx_lens;
    p.q_starts = q_starts;
    p.num_heads = d->num_heads;
    p.num_blocks = d->num_blocks;
    p.max_blocks = max_blocks;
    p.max_q_len = max_q_len;
    p.q_tiles = (max_q_len + kBM - 1) / kBM;
    p.bshift = bshift;
    p.qscale = scale * 1.4426950408889634f;
    p.status = status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return d->head_dim == 64 ? launch_d<64>(p, n_seqs, st) : launch_d<128>(p, n_seqs, st);
}

}  // namespace pagedkv
