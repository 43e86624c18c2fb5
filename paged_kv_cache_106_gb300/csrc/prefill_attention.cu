// Causal paged prefill attention: every query of a prompt (or of a chunk
// appended to a cached prefix) attends to the positions up to its own,
// reading keys and values through the block table.
//
// What it computes: the prompt phase of the vLLM paper review (§4.3), where
// the prompt's tokens are processed together and each one attends to the
// tokens before it and itself, with the blockwise attention equation of the
// PagedAttention notes (§3.1) evaluated for each of those queries.
//
// Kernel design (sm_103a, 5th-generation tensor cores through tcgen05):
//   - one CTA = (sequence, head, tile of 128 consecutive queries); later
//     query tiles (more keys) are launched first.  Warp roles:
//       warps 0-7  softmax: query row i is tensor-memory lane i; warps w and
//                  w + 4 share the 32 rows of lane quarter w % 4, each taking
//                  half of a tile's key columns, and meet once per tile to
//                  combine their row maxima;
//       warp 8     one thread issues every tcgen05.mma and commit;
//       warps 9-10 gather K tiles, warps 11-12 the Q tile and V tiles.
//   - keys and values stream through shared-memory rings (3 K stages, 2 V) in
//     tiles of 128 positions.  Position j lives in block table[j / B] at
//     offset j % B; in the cache layout [block][head][B][D] each (block,
//     head) run is B*D*2 contiguous bytes.  For B >= 8 a lane per block
//     issues one 2-D TMA copy per 64-column panel of the run (a tensor map
//     over the cache's rows), which lands already in the 128-byte-swizzled
//     layout the tensor cores read; for B = 4 the loader threads gather the
//     same layout with 16-byte cp.async.  The same bytes are the K-major B
//     operand of S = Q K^T and the MN-major B operand of O = P V.  Rows past
//     the context in the last V tile are zeroed before the product.
//   - tensor memory (512 columns): three 128-column S buffers, so Q K^T for
//     tile t+2 runs while tile t is in softmax, and the fp32 output
//     accumulator O (D columns).  Softmax overwrites its S buffer with P as
//     fp16 pairs, which the P V product reads as its A operand straight from
//     tensor memory.
//   - the softmax is online, in base 2 (ex2.approx), with a lazy rescale: a row's
//     reference maximum moves only when a tile raises it by more than 2^8,
//     so O is rescaled in tensor memory rarely; P <= 2^8 stays exact enough
//     in fp16.  P enters P V as hi + lo fp16 terms (hi = fp16(p),
//     lo = fp16(p - hi)), keeping about 22 bits of each probability, so the
//     fp16 rounding of the output dominates the error.
//   - positions past the causal end of the tile are zero-filled, and scores
//     of keys after a row's own position are masked to -inf.
//   - the epilogue stages each row half as fp16 in shared memory and writes
//     it with one bulk copy (rows of a head are H*D*2 bytes apart in out).
//   - every mbarrier wait is bounded; a wait that runs out reports
//     PA_ERR_TIMEOUT, and the CTA drains its MMAs (bounded) and frees its
//     tensor memory before it returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "tc_device.cuh"

namespace pagedkv {
namespace {

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

// 2^x by the PTX approximation instruction (relative error about 2^-22;
// -inf gives +0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Barrier among `count` threads of the CTA (ids 1.. are free; 0 is
// __syncthreads) that also returns whether `v` held for all of them.
__device__ __forceinline__ bool group_all(int id, int count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// 2-D tensor copy global -> shared (box of the tensor map at element
// coordinates x, y); completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Two probabilities as fp16 pairs hi + lo (lower column in the low half).
// hi is p rounded to fp16's 11 significant bits by integer arithmetic (exact
// in fp16 for p >= 2^-14), so only the two packing conversions use the
// conversion pipe; lo = p - hi is exact in fp32.  hi + lo carries p to about
// 2^-22 relative, or to fp16's subnormal spacing (2^-24) for tiny p.
__device__ __forceinline__ void split_pair(float p0, float p1, uint32_t &hi, uint32_t &lo) {
    const float h0 = __uint_as_float((__float_as_uint(p0) + 0x1000u) & 0xFFFFE000u);
    const float h1 = __uint_as_float((__float_as_uint(p1) + 0x1000u) & 0xFFFFE000u);
    const __half2 h = __floats2half2_rn(h0, h1);
    const __half2 l = __floats2half2_rn(p0 - h0, p1 - h1);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

constexpr int TBM = 128;          // queries per CTA (= tensor-memory lanes)
constexpr int TBN = 128;          // key positions per tile
constexpr int NST = 3;            // K ring stages and S buffers
constexpr int NSV = 2;            // V ring stages
constexpr int kMmaWarp = 8, kKWarp0 = 9, kVWarp0 = 11;
constexpr int kTcThreads = 416;   // 13 warps
constexpr uint32_t kPanel = TBM * 128;   // bytes of one 64-column panel of a 128-row tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = NST * 128;    // output accumulator after the S buffers
constexpr float kRescaleLog2 = 8.f;      // lazy-rescale threshold (log2 units)

template <int D>
struct TcLayout {
    static constexpr uint32_t TILE = (D / 64) * kPanel;
    static constexpr uint32_t Q = 0, K = TILE, V = K + NST * TILE, END = V + NSV * TILE;
    static constexpr uint32_t OUT_STRIDE = D * 2 + 16;   // output staging rows (in the K ring)
    // at least 116 KB so that one CTA holds an SM (its 512 tensor-memory
    // columns are the whole SM's), plus 1 KB to align the tiles to 1024 bytes
    static constexpr uint32_t BYTES = (END > 116u * 1024u ? END : 116u * 1024u) + 1024u;
};

struct TcBars {
    uint64_t q_full;
    uint64_t k_full[NST], k_empty[NST], v_full[NSV], v_empty[NSV];
    uint64_t s_full[NST], p_full[NST], pv_done[NST];
    uint64_t done, v_raw;
    uint32_t tmem;
    int32_t tab[2][2][TBN / 4];   // per loader group, double-buffered block ids of a tile
    float red[2][2][TBM];         // per tile parity and column half: row maxima, then sums
};

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// TMA: K / V tiles arrive by 2-D tensor copies of whole (block, head) runs
// (block sizes 8..32, whose runs start on 1024-byte boundaries of the
// swizzle pattern); otherwise (block size 4) by 16-byte cp.async.
template <int D, bool TMA>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_tc(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
    using L = TcLayout<D>;
    constexpr int CPR = D / 8;        // 16-byte chunks per row
    constexpr int RPP = 64 / CPR;     // rows one pass of a 64-thread loader group covers
    extern __shared__ uint8_t smem_raw[];
    __shared__ TcBars bars;
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = base + L::Q, sK = base + L::K, sV = base + L::V;

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
    const int q0 = (p.q_tiles - 1 - (int)blockIdx.x) * TBM;  // later tiles first
    if (q0 >= ql) return;
    const int pos0 = ctx - ql;                 // position of query 0 of the sequence
    const int rows = min(TBM, ql - q0);
    const int n_end = pos0 + q0 + rows;        // this tile needs keys [0, n_end)
    const int n_tiles = (n_end + TBN - 1) / TBN;

    const uint32_t b_q = smem_addr(&bars.q_full), b_done = smem_addr(&bars.done);
    auto bar = [](uint64_t *arr, int i) { return smem_addr(arr + i); };
    if (tid == 0) {
        mbar_init(b_q, 64);
        for (int i = 0; i < NST; ++i) {
            mbar_init(bar(bars.k_full, i), TMA ? 1 : 64);
            mbar_init(bar(bars.k_empty, i), 1);
            mbar_init(bar(bars.s_full, i), 1);
            mbar_init(bar(bars.p_full, i), 256);
            mbar_init(bar(bars.pv_done, i), 1);
        }
        for (int i = 0; i < NSV; ++i) {
            mbar_init(bar(bars.v_full, i), TMA ? 1 : 64);
            mbar_init(bar(bars.v_empty, i), 1);
        }
        mbar_init(b_done, 1);
        mbar_init(smem_addr(&bars.v_raw), 1);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) tc::alloc(smem_addr(&bars.tmem), kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = bars.tmem;

    if (warp >= kKWarp0) {
        // ---- loaders: 64 threads gather K tiles, 64 gather the Q tile and V tiles
        const bool is_k = warp < kVWarp0;
        const int g = is_k ? 0 : 1;
        const int lt = tid - (is_k ? kKWarp0 : kVWarp0) * 32;
        const int c = lt % CPR, r0 = lt / CPR;
        const int B = 1 << p.bshift;
        const int32_t *table = p.tables + (size_t)s * p.max_blocks;
        if (!is_k) {
#pragma unroll 4
            for (int r = r0; r < TBM; r += RPP) {
                const bool v = r < rows;
                const __half *src =
                    p.q + ((size_t)(q_beg + q0 + (v ? r : 0)) * p.num_heads + h) * D + c * 8;
                cp_async16(sQ + tc::sw128(TBM, r, c), src, v);
            }
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(b_q);
        }
        const uint32_t ring = is_k ? sK : sV;
        uint64_t *full = is_k ? bars.k_full : bars.v_full;
        uint64_t *empty = is_k ? bars.k_empty : bars.v_empty;
        const int nb = TBN >> p.bshift;   // blocks per tile (tiles start on a block)
        const int NS = is_k ? NST : NSV;   // ring stages of this group
        if constexpr (TMA) {
            // One warp per group issues the tensor copies, lane i for block i
            // of the tile; the V group's second warp helps zero the rows past
            // the context in the last V tile.
            const CUtensorMap *map = is_k ? &tmk : &tmv;
            const uint32_t run_bytes = (uint32_t)B * 128u * (D / 64);
            const uint32_t b_raw = smem_addr(&bars.v_raw);
            bool dead = false;   // a wait ran out: issue nothing more, but still meet the group
            for (int t = 0; t < n_tiles; ++t) {
                const int st = t % NS;
                const int n0 = t * TBN;
                // rows past the context must read as zeros in V (0 * garbage
                // could be NaN); only the last tile has such rows
                const bool fix = !is_k && t == n_tiles - 1 && n_end - n0 < TBN;
                if (lt < 32 && !dead) {
                    const bool ok = warp_all(t < NS || mbar_wait_bounded(bar(empty, st),
                                                                         ((t / NS) - 1) & 1,
                                                                         p.status, true));
                    if (!ok) report(p.status, PA_ERR_TIMEOUT);
                    dead = !ok;
                }
                if (lt < 32 && !dead) {
                    const int j = n0 + (lt << p.bshift);
                    const bool valid = lt < nb && j < n_end;
                    const int phys = valid ? __ldg(table + (j >> p.bshift)) : -1;
                    const bool in_pool = valid && phys >= 0 && phys < p.num_blocks;
                    if (valid && !in_pool) report(p.status, PA_ERR_BAD_BLOCK);
                    const uint32_t n_runs = __popc(__ballot_sync(0xffffffffu, in_pool));
                    const uint32_t tgt = fix ? b_raw : bar(full, st);
                    if (lt == 0) mbar_arrive_expect_tx(tgt, n_runs * run_bytes);
                    __syncwarp();
                    if (in_pool) {
                        const uint32_t dst = ring + st * L::TILE + (uint32_t)(lt << p.bshift) * 128u;
                        const int y = (phys * p.num_heads + h) << p.bshift;
#pragma unroll
                        for (int pn = 0; pn < D / 64; ++pn)
                            tma_load_2d(dst + pn * kPanel, map, pn * 64, y, tgt);
                    }
                }
                if (fix) {
                    // both V warps: wait for the copies, zero rows [n_end - n0, TBN)
                    const bool ok = mbar_wait_bounded(b_raw, 0, p.status, true);
                    if (ok) {
                        const int first = n_end - n0;
                        const uint32_t span = (uint32_t)(TBN - first) * 128u;
                        for (int pn = 0; pn < D / 64; ++pn) {
                            const uint32_t z = ring + st * L::TILE + pn * kPanel + first * 128u;
                            for (uint32_t o = (uint32_t)lt * 16u; o < span; o += 64u * 16u)
                                asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(z + o),
                                             "r"(0)
                                             : "memory");
                        }
                        fence_proxy_async_smem();
                    }
                    if (group_all(2, 64, ok)) {
                        if (lt == 0) mbar_arrive(bar(full, st));
                    } else {
                        report(p.status, PA_ERR_TIMEOUT);
                    }
                }
            }
        } else {
            const __half *cache = is_k ? p.k_cache : p.v_cache;
            // Tile t is issued before tile t-1 is waited for, so two tiles of
            // copies are in flight per thread.
            int t = 0;
            for (; t < n_tiles; ++t) {
                const int st = t % NS;
                const int n0 = t * TBN;
                int32_t *tab = bars.tab[g][t & 1];
                if (lt < nb) {   // the tile's physical block ids, read once by the group
                    const int j = n0 + (lt << p.bshift);
                    tab[lt] = j < n_end ? __ldg(table + (j >> p.bshift)) : -1;
                }
                const bool free_ok =
                    t < NS || mbar_wait_bounded(bar(empty, st), ((t / NS) - 1) & 1, p.status, true);
                // one decision for the whole group, and the block ids visible to it
                if (!group_all(1 + g, 64, free_ok)) {
                    report(p.status, PA_ERR_TIMEOUT);
                    break;
                }
                const uint32_t dst = ring + st * L::TILE;
#pragma unroll 4
                for (int r = r0; r < TBN; r += RPP) {
                    const int j = n0 + r;
                    const int phys = tab[r >> p.bshift];
                    bool v = j < n_end;
                    size_t off = 0;
                    if (v) {
                        if (phys < 0 || phys >= p.num_blocks) {
                            report(p.status, PA_ERR_BAD_BLOCK);
                            v = false;
                        } else {
                            off = (((size_t)phys * p.num_heads + h) * B + (j & (B - 1))) * D + c * 8;
                        }
                    }
                    cp_async16(dst + tc::sw128(TBN, r, c), cache + off, v);
                }
                cp_async_commit();
                if (t > 0) {
                    cp_async_wait<1>();
                    fence_proxy_async_smem();
                    mbar_arrive(bar(full, (t - 1) % NS));
                }
            }
            cp_async_wait<0>();
            if (t == n_tiles && n_tiles > 0) {
                fence_proxy_async_smem();
                mbar_arrive(bar(full, (n_tiles - 1) % NS));
            }
        }
    } else if (warp == kMmaWarp) {
        // ---- one thread issues the MMAs
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_f16(TBM, TBN, false);
            constexpr uint32_t idO = tc::idesc_f16(TBM, D, true);
            auto issue_s = [&](int t) -> bool {
                const int st = t % NST;
                if (!mbar_wait_bounded(bar(bars.k_full, st), (t / NST) & 1, p.status, true))
                    return false;
                tc::fence_after();
                const uint32_t kb = sK + st * L::TILE;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
                    tc::mma_ss(tmem + st * 128, tc::smem_desc(sQ + off, 16, 1024),
                               tc::smem_desc(kb + off, 16, 1024), idS, kk > 0 ? 1u : 0u);
                }
                tc::commit(bar(bars.s_full, st));
                tc::commit(bar(bars.k_empty, st));
                return true;
            };
            bool ok = mbar_wait_bounded(b_q, 0, p.status, true);
            if (ok) ok = issue_s(0);
            if (ok && n_tiles > 1) ok = issue_s(1);
            for (int t = 0; ok && t < n_tiles; ++t) {
                const int b = t % NST, bv = t % NSV;
                ok = mbar_wait_bounded(bar(bars.p_full, b), (t / NST) & 1, p.status, true) &&
                     mbar_wait_bounded(bar(bars.v_full, bv), (t / NSV) & 1, p.status, true);
                if (!ok) break;
                tc::fence_after();
                const uint32_t vb = sV + bv * L::TILE;
#pragma unroll
                for (int kk = 0; kk < TBN / 16; ++kk) {
                    const uint64_t dv = tc::smem_desc(vb + kk * 2048, kPanel, 1024);
                    const uint32_t pa = tmem + b * 128 + (kk >> 1) * 32 + (kk & 1) * 8;
                    tc::mma_ts(tmem + kOCol, pa, dv, idO, (t > 0 || kk > 0) ? 1u : 0u);
                    tc::mma_ts(tmem + kOCol, pa + 16, dv, idO, 1u);
                }
                tc::commit(bar(bars.v_empty, bv));
                tc::commit(bar(bars.pv_done, b));
                if (t + 2 < n_tiles) {
                    // S(t+2) goes to the buffer whose P the product of tile t-1 read
                    if (t >= 1)
                        ok = mbar_wait_bounded(bar(bars.pv_done, (t - 1) % NST),
                                               ((t - 1) / NST) & 1, p.status, true);
                    if (ok) ok = issue_s(t + 2);
                }
            }
            if (!ok) report(p.status, PA_ERR_TIMEOUT);
            tc::commit(b_done);   // lets the teardown wait for every MMA issued
        }
        __syncwarp();
    } else {
        // ---- softmax warps: warps w and w + 4 share the query rows of tensor-memory
        // lane quarter w % 4 (row = lane of that quarter); warp w < 4 takes key
        // columns 0-63 of each tile, warp w + 4 columns 64-127
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const int qi = q0 + row;
        const bool valid = qi < ql;
        const int pos = pos0 + min(qi, ql - 1);
        const float qs = p.qscale;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int t = 0; t < n_tiles; ++t) {
            const int b = t % NST;
            ok = ok && warp_all(mbar_wait_bounded(bar(bars.s_full, b), (t / NST) & 1, p.status, true));
            const uint32_t sb = lane_base + b * 128 + half * 64;
            const int n0 = t * TBN + half * 64;   // first key of this warp's columns
            // keys past this row's position are masked: key n0 + 32 cc + i with i > lim
            const bool need_mask = n0 + 63 > pos0 + q0;
            float mt = -INFINITY;
            if (ok) {
                tc::fence_after();
#pragma unroll 1
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t r[32];
                    tc::ld32(sb + cc * 32, r);
                    tc::wait_ld();
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                    if (need_mask) {
                        const int lim = pos - (n0 + cc * 32);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            m4[i & 3] = fmaxf(m4[i & 3], i > lim ? -INFINITY : __uint_as_float(r[i]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) m4[i & 3] = fmaxf(m4[i & 3], __uint_as_float(r[i]));
                    }
                    mt = fmaxf(mt, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
                }
                mt *= qs;   // scale > 0: the maximum of the scaled scores
            }
            bars.red[t & 1][half][row] = mt;
            // the two halves of each row meet here once per tile: one exit
            // decision for all softmax warps, and the partner's maximum
            if (!group_all(3, 256, ok)) {
                ok = false;
                break;
            }
            mt = fmaxf(mt, bars.red[t & 1][half ^ 1][row]);
            float corr = 1.f;
            const bool resc = mt > m_run + kRescaleLog2;
            if (resc) {
                corr = ex2(m_run - mt);
                m_run = mt;
                l_run *= corr;
            }
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t r[32], w[32];
                tc::ld32(sb + cc * 32, r);
                tc::wait_ld();
                if (need_mask) {
                    const int lim = pos - (n0 + cc * 32);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float p0 = 2 * i > lim ? 0.f : ex2(fmaf(__uint_as_float(r[2 * i]), qs, -m_run));
                        const float p1 =
                            2 * i + 1 > lim ? 0.f : ex2(fmaf(__uint_as_float(r[2 * i + 1]), qs, -m_run));
                        ls[i & 3] += p0 + p1;
                        split_pair(p0, p1, w[i], w[16 + i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float p0 = ex2(fmaf(__uint_as_float(r[2 * i]), qs, -m_run));
                        const float p1 = ex2(fmaf(__uint_as_float(r[2 * i + 1]), qs, -m_run));
                        ls[i & 3] += p0 + p1;
                        split_pair(p0, p1, w[i], w[16 + i]);
                    }
                }
                tc::st32(sb + cc * 32, w);
            }
            l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            tc::wait_st();
            if (__any_sync(0xffffffffu, resc && t > 0)) {
                // O holds tiles < t: wait until their product is complete, then
                // scale this warp's half of the output columns
                if (warp_all(mbar_wait_bounded(bar(bars.pv_done, (t - 1) % NST),
                                               ((t - 1) / NST) & 1, p.status, true))) {
                    tc::fence_after();
#pragma unroll 1
                    for (int cc = 0; cc < D / 64; ++cc) {
                        const uint32_t oc = lane_base + kOCol + half * (D / 2) + cc * 32;
                        uint32_t r[32];
                        tc::ld32(oc, r);
                        tc::wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
                        tc::st32(oc, r);
                    }
                    tc::wait_st();
                } else {
                    ok = false;   // every softmax warp leaves at the next meeting
                }
            }
            tc::fence_before();
            mbar_arrive(bar(bars.p_full, b));
        }
        if (ok)
            ok = warp_all(mbar_wait_bounded(bar(bars.pv_done, (n_tiles - 1) % NST),
                                            ((n_tiles - 1) / NST) & 1, p.status, true));
        bars.red[n_tiles & 1][half][row] = l_run;
        if (group_all(3, 256, ok)) {
            // this warp's half of the row: normalise, stage as fp16 in the
            // (now idle) K ring, store with one bulk copy per row half
            tc::fence_after();
            const float inv = 1.f / (l_run + bars.red[n_tiles & 1][half ^ 1][row]);
            const uint32_t stage = sK + (uint32_t)row * L::OUT_STRIDE + half * D;
#pragma unroll 1
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t r[32];
                tc::ld32(lane_base + kOCol + half * (D / 2) + cc * 32, r);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t hv[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const __half2 v2 = __floats2half2_rn(__uint_as_float(r[8 * i + 2 * k]) * inv,
                                                             __uint_as_float(r[8 * i + 2 * k + 1]) * inv);
                        hv[k] = *reinterpret_cast<const uint32_t *>(&v2);
                    }
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                     stage + cc * 64 + i * 16),
                                 "r"(hv[0]), "r"(hv[1]), "r"(hv[2]), "r"(hv[3])
                                 : "memory");
                }
            }
            fence_proxy_async_smem();
            if (valid) {
                __half *dst = p.out + ((size_t)(q_beg + qi) * p.num_heads + h) * D + half * (D / 2);
                asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                             "r"(stage), "r"(D)
                             : "memory");
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            }
        } else {
            report(p.status, PA_ERR_TIMEOUT);
        }
    }

    // ---- teardown: every MMA drained (bounded), then tensor memory freed
    tc::fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        if (lane == 0 && !mbar_wait_bounded(b_done, 0, p.status, false))
            report(p.status, PA_ERR_TIMEOUT);
        __syncwarp();
        tc::fence_after();
        tc::dealloc(tmem, kTmemCols);
    }
}

template <int D, bool TMA>
cudaError_t set_prefill_smem_once() {
    static std::once_flag once[64];
    static cudaError_t err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        err[dev] = cudaFuncSetAttribute(paged_prefill_tc<D, TMA>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)TcLayout<D>::BYTES);
    });
    return err[dev];
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (the library does not link the driver library itself).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// One layer's cache seen as a 2-D fp16 tensor of num_blocks*H*B rows of D
// values; a box is 64 values (one 128-byte swizzle row) by B rows, i.e. one
// (block, head) run of one 64-column panel.
int encode_cache_map(CUtensorMap *m, const void *cache, const pa_pool_desc *d) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail(PA_ERR_CUDA, "pa_prefill_attention: cuTensorMapEncodeTiled unavailable");
    const uint64_t rows = (uint64_t)d->num_blocks * d->num_heads * d->block_size;
    cuuint64_t dims[2] = {(cuuint64_t)d->head_dim, (cuuint64_t)(rows ? rows : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)d->head_dim * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)d->block_size};
    cuuint32_t elem[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(cache), dims,
                           strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PA_ERR_CUDA, "pa_prefill_attention: cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PA_OK;
}

template <int D, bool TMA>
int launch_d(PrefillParams p, int n_seqs, const pa_pool_desc *d, cudaStream_t st) {
    cudaError_t e = set_prefill_smem_once<D, TMA>();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "prefill smem attribute: %s", cudaGetErrorString(e));
    CUtensorMap tmk, tmv;
    std::memset(&tmk, 0, sizeof tmk);
    std::memset(&tmv, 0, sizeof tmv);
    if (TMA) {
        int rc = encode_cache_map(&tmk, p.k_cache, d);
        if (rc == PA_OK) rc = encode_cache_map(&tmv, p.v_cache, d);
        if (rc != PA_OK) return rc;
    }
    p.q_tiles = (p.max_q_len + TBM - 1) / TBM;
    const dim3 grid((unsigned)p.q_tiles, (unsigned)p.num_heads, (unsigned)n_seqs);
    paged_prefill_tc<D, TMA><<<grid, kTcThreads, TcLayout<D>::BYTES, st>>>(p, tmk, tmv);
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
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: scale must be finite and > 0");
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
    p.q_tiles = 0;   // set by the launcher from its tile height
    p.bshift = bshift;
    p.qscale = scale * 1.4426950408889634f;
    p.status = status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool tma = d->block_size >= 8;
    if (d->head_dim == 64)
        return tma ? launch_d<64, true>(p, n_seqs, d, st) : launch_d<64, false>(p, n_seqs, d, st);
    return tma ? launch_d<128, true>(p, n_seqs, d, st) : launch_d<128, false>(p, n_seqs, d, st);
}

}  // namespace pagedkv
