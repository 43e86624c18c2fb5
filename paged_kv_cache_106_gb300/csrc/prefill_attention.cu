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
//   - persistent: one CTA per SM walks units of work, a unit being 128
//     consecutive queries of one (sequence, head); units are taken in the
//     order (sequence, query tile from the last, head), strided by CTA: all
//     heads of a query tile run side by side (different keys and values, no
//     hot spots), and the next tile of the same (sequence, head), which
//     re-reads a prefix of those keys and values, follows while they are
//     still in L2 (measured: 5 % faster than interleaving 8 sequences).  Tensor memory,
//     barriers and the pipeline carry over from unit to unit.  Warp roles:
//       warps 0-7  softmax and epilogue: query row i is tensor-memory lane i;
//                  warps w and w + 4 share the 32 rows of lane quarter w % 4,
//                  each taking half of a tile's key columns, and meet once per
//                  tile to combine their row maxima;
//       warp 8     one thread issues every tcgen05.mma and commit, polling its
//                  dependencies so Q K^T and P V of different tiles interleave;
//       warp 9     Q rows and K tiles by TMA, warp 10 V tiles by TMA;
//       warp 11    scheduler: finds this CTA's non-empty units and publishes
//                  them through a 4-slot descriptor ring;
//       warps 12-15 epilogue: warp 12 + q normalises and writes the rows of
//                  lane quarter q once a unit's last P V is done.
//   - Q (two buffers), K and V (two-stage rings, with the runs of the tile
//     two steps further prefetched into L2) move in tiles of 128
//     positions.  Position j lives in block table[j / B] at offset j % B; in
//     the cache layout [block][head][B][D] each (block, head) run is B*D*2
//     contiguous bytes.  K and V tiles sit in shared memory as 8-row groups,
//     [j / 8][64-column panel][j % 8][128 bytes], 128-byte swizzled, so that
//     a run of B >= 8 rows is whole groups: a loader lane per block moves it
//     with one 4-D TMA copy (at D = 128, 4 KB at B = 16; per-SM copy
//     throughput is higher for bigger boxes, and the copies bound the loop)
//     and it lands already in the layout the tensor cores read (the swizzle
//     follows the shared-memory address).  At B = 4, or D = 64, one 2-D copy
//     per panel (box 64 x B).  The same bytes are the K-major B operand of
//     S = Q K^T (8-row groups D/64 KB apart) and the MN-major B operand of
//     O = P V (panels 1 KB apart).  The V block holding the context's last
//     position is copied up to it in boxes of 8, 4, 2 and 1 rows, and the V
//     ring starts zeroed, so slots past the context are never read.  Q
//     arrives as one 128-row box per panel of a [rows][H][D] tensor map, in
//     [panel][128 rows] layout (rows past q_rows read as zeros).
//   - tensor memory (512 columns): three 128-column S buffers, so Q K^T for
//     tile t+2 runs while tile t is in softmax, and the fp32 output
//     accumulator O (D columns).  Softmax overwrites its S buffer with P as
//     fp16 pairs, which the P V product reads as its A operand straight from
//     tensor memory.
//   - the softmax is online, in base 2 (ex2.approx), with a lazy rescale: a row's
//     reference maximum moves only when a tile raises it by more than 2^8,
//     so O is rescaled in tensor memory rarely.  P (<= 2^8) enters P V as
//     fp16, 11 significant bits like the output: rounding p perturbs each
//     weight by at most 2^-12 relative, and the fp16 rounding of the output
//     stays the larger error (simulated: max |error| 1.03e-3 against 0.98e-3
//     with exact p, for prompts up to 1536 and peaked scores).
//   - blocks past the causal end of a tile are not copied; scores of keys
//     after a row's own position are masked to -inf (a select, so stale
//     shared memory there cannot leak in).
//   - the epilogue warps wait for a unit's last P V, read O from tensor
//     memory into registers (normalised, as fp16) and release it to the next
//     unit's first P V, which overwrites O; so the tensor pipe idles at a
//     unit boundary only for that read, and the softmax warps never stop
//     for an epilogue.  They write the rows with 16-byte streaming stores,
//     exchanged within groups of 8 lanes so that each store instruction
//     covers 4 whole 128-byte row segments (only the unit's rows).  A Q
//     buffer is free as soon as its unit's last Q K^T is done.
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
    int32_t num_heads, num_blocks, max_blocks, max_q_len, q_rows, q_tiles, bshift;
    float qscale;  // scale * log2(e): softmax evaluated with exp2
    int32_t *status;
};

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
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// L2 policies: keys and values are re-read by later query tiles (keep them),
// queries are read and outputs written once (let them go first).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Two probabilities as one fp16 pair (lower column in the low half).
__device__ __forceinline__ uint32_t pack_pair(float p0, float p1) {
    const __half2 h = __floats2half2_rn(p0, p1);
    return *reinterpret_cast<const uint32_t *>(&h);
}

constexpr int TBM = 128;          // queries per unit (= tensor-memory lanes)
constexpr int TBN = 128;          // key positions per tile
constexpr int NSB = 3;            // S buffers in tensor memory
constexpr int NSK = 2;            // K ring stages
constexpr int NSV = 2;            // V ring stages
constexpr int NU = 4;             // unit descriptors in flight
constexpr int kMmaWarp = 8, kKWarp = 9, kVWarp = 10, kSchedWarp = 11;   // 12-15: epilogue
constexpr int kTcThreads = 512;   // 16 warps
constexpr uint32_t kPanel = TBM * 128;   // bytes of one 64-column panel of a 128-row tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = NSB * 128;    // output accumulator after the S buffers
constexpr float kRescaleLog2 = 8.f;      // lazy-rescale threshold (log2 units)
// readers of a unit descriptor: K loader, V loader, MMA thread, 8 softmax warps, 4 epilogue warps
constexpr uint32_t kUnitReaders = 3 + 8 + 4;
constexpr int kPrefetchTiles = 2;  // K/V tiles prefetched into L2 ahead of their copies
constexpr int kSeqGroup = 1;     // sequences whose query tiles are interleaved (L2 reuse)
constexpr int kVPartMaps = 4;     // boxes of 8, 4, 2, 1 cache rows for a partial V block

template <int D>
struct TcLayout {
    static constexpr uint32_t TILE = (D / 64) * kPanel;
    static constexpr uint32_t Q = 0, K = 2 * TILE, V = K + NSK * TILE, END = V + NSV * TILE;
    // at least 116 KB so that one CTA holds an SM (its 512 tensor-memory
    // columns are the whole SM's), plus 1 KB to align the tiles to 1024 bytes
    static constexpr uint32_t BYTES = (END > 116u * 1024u ? END : 116u * 1024u) + 1024u;
};

// Byte offset of row r (panel 0) in a K or V tile.  Those tiles are laid out
// [r / 8][panel][r % 8][128 bytes]: 8-row groups of (D / 64) KB, each holding
// its rows' 64-column panels one after the other, so that a (block, head)
// run of B >= 8 rows is B / 8 whole groups, contiguous in shared memory, and
// one TMA box moves it.  Panel pn of a row is 1024 * pn bytes further.
template <int D>
__device__ __forceinline__ uint32_t kv_row_off(uint32_t r) {
    return (r >> 3) * (uint32_t)(D / 64) * 1024u + (r & 7u) * 128u;
}

// One unit of work: 128 queries of one (sequence, head).
struct Unit {
    int32_t s, h, q0, q_beg, ql, pos0, n_end, n_tiles;   // n_tiles == 0: no more units
};

// Tensor maps: K and V cache runs (D = 128 with B >= 8: a 4-D view
// [row / 8][panel][row % 8][64] with one box per (block, head) run; otherwise
// rows of D values, box 64 x B, one copy per panel), cache rows for the
// partial V block (boxes 64 x 8 .. 64 x 1), query rows and output rows as 3-D
// [rows][H][D] tensors (q: one box of 128 rows; out: boxes of 128 .. 1 rows).
struct TcMaps {
    CUtensorMap k, v, v_part[kVPartMaps], q;
};

struct TcBars {
    uint64_t unit_full[NU], unit_empty[NU];
    uint64_t q_full[2], q_empty[2];
    uint64_t k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV];
    uint64_t s_full[NSB], p_full[NSB], pv_done[NSB];
    uint64_t o_free;               // the epilogue has read a unit's O (one phase per unit)
    uint64_t l_full[2], l_empty[2]; // a unit's row sums (slot k & 1) written / read
    uint64_t done;
    uint32_t tmem;
    Unit unit[NU];
    float red[2][2][TBM];   // per tile parity and column half: row maxima
    float red_l[2][2][TBM]; // per unit parity and column half: a finished unit's row sums
};

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void zero_smem(uint32_t addr, uint32_t bytes, int lane) {
    for (uint32_t o = (uint32_t)lane * 16u; o < bytes; o += 32u * 16u)
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr + o), "r"(0) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
        : "memory");
}

// Persistent: one CTA per SM walks the units v = blockIdx.x + i * gridDim.x
// of the list ordered by group of kSeqGroup sequences, then query tile (the
// last, with the most keys, first), then sequence, then head; a scheduler
// warp skips the empty ones.  The query tiles of one (sequence, head) come
// about H units apart, while the keys and values they share are still in L2,
// and concurrent CTAs work on different (sequence, head).
template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_tc(const PrefillParams p, const __grid_constant__ TcMaps maps, int32_t n_seqs) {
    using L = TcLayout<D>;
    constexpr int NP = D / 64;   // 64-column panels
    extern __shared__ uint8_t smem_raw[];
    __shared__ TcBars bars;
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = base + L::Q, sK = base + L::K, sV = base + L::V;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.num_heads, B = 1 << p.bshift;
    auto bar = [](uint64_t *arr, int i) { return smem_addr(arr + i); };

    if (tid == 0) {
        for (int i = 0; i < NU; ++i) {
            mbar_init(bar(bars.unit_full, i), 1);
            mbar_init(bar(bars.unit_empty, i), kUnitReaders);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(bars.q_full, i), 1);
            mbar_init(bar(bars.q_empty, i), 1);   // the unit's last Q K^T is done
        }
        for (int i = 0; i < NSK; ++i) {
            mbar_init(bar(bars.k_full, i), 1);
            mbar_init(bar(bars.k_empty, i), 1);
        }
        for (int i = 0; i < NSV; ++i) {
            mbar_init(bar(bars.v_full, i), 1);
            mbar_init(bar(bars.v_empty, i), 1);
        }
        for (int i = 0; i < NSB; ++i) {
            mbar_init(bar(bars.s_full, i), 1);
            mbar_init(bar(bars.p_full, i), 256);
            mbar_init(bar(bars.pv_done, i), 1);
        }
        mbar_init(smem_addr(&bars.o_free), 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(bars.l_full, i), 256);
            mbar_init(bar(bars.l_empty, i), 128);
        }
        mbar_init(smem_addr(&bars.done), 1);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) tc::alloc(smem_addr(&bars.tmem), kTmemCols);
    // the V ring starts as zeros: rows no copy ever writes (values past a
    // context) must hold finite numbers, since they meet P = 0
    if (warp == kVWarp) zero_smem(sV, NSV * L::TILE, lane);
    fence_proxy_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = bars.tmem;
    const int q_tiles = p.q_tiles;

    // Reads unit k of this CTA from the ring (bounded wait); n_tiles < 0 on timeout.
    auto get_unit = [&](int k, Unit &u) {
        const bool ok =
            warp_all(mbar_wait_bounded(bar(bars.unit_full, k % NU), (k / NU) & 1, p.status, true));
        if (!ok) {
            u.n_tiles = -1;
            return;
        }
        u = bars.unit[k % NU];
    };

    if (warp == kSchedWarp) {
        // ---- scheduler: lanes test 32 candidate units at a time, the valid ones
        // are published in order
        const long long V = (long long)n_seqs * H * q_tiles;
        const long long group_units = (long long)kSeqGroup * H * q_tiles;
        int k = 0;
        bool ok = true;
        for (long long base_v = blockIdx.x; ok && base_v < V; base_v += 32ll * gridDim.x) {
            const long long v = base_v + (long long)lane * gridDim.x;
            Unit u{};
            bool valid = false;
            if (v < V) {
                // v -> (group of kSeqGroup sequences, query tile from the last,
                // sequence in the group, head)
                const int grp = (int)(v / group_units);
                const int gsz = min(kSeqGroup, n_seqs - grp * kSeqGroup);
                const long long r = v - (long long)grp * group_units;
                const int x = (int)(r / ((long long)gsz * H));
                const int r2 = (int)(r - (long long)x * gsz * H);
                u.s = grp * kSeqGroup + r2 / H;
                u.h = r2 - (r2 / H) * H;
                const int qt = q_tiles - 1 - x;
                u.q_beg = p.q_starts[u.s];
                u.ql = p.q_starts[u.s + 1] - u.q_beg;
                const int ctx = p.ctx_lens[u.s];
                const bool bad_len = u.ql < 0 || u.ql > ctx || u.ql > p.max_q_len ||
                                     u.q_beg < 0 || (int64_t)u.q_beg + u.ql > p.q_rows;
                const bool bad_ctx = (int64_t)ctx > ((int64_t)p.max_blocks << p.bshift);
                if ((bad_len || bad_ctx) && x == 0 && u.h == 0)
                    report(p.status, bad_len ? PA_ERR_INVALID_ARG : PA_ERR_BAD_BLOCK);
                u.q0 = qt * TBM;
                valid = !bad_len && !bad_ctx && u.q0 < u.ql;
                if (valid) {
                    u.pos0 = ctx - u.ql;
                    u.n_end = u.pos0 + u.q0 + min(TBM, u.ql - u.q0);
                    u.n_tiles = (u.n_end + TBN - 1) / TBN;
                }
            }
            uint32_t mask = __ballot_sync(0xffffffffu, valid);
            while (mask) {
                const int src = __ffs(mask) - 1;
                mask &= mask - 1;
                if (k >= NU)
                    ok = warp_all(mbar_wait_bounded(bar(bars.unit_empty, k % NU),
                                                    ((k / NU) - 1) & 1, p.status, true));
                if (!ok) break;
                if (lane == src) {
                    bars.unit[k % NU] = u;
                    mbar_arrive(bar(bars.unit_full, k % NU));
                }
                __syncwarp();
                ++k;
            }
        }
        // end marker
        if (ok && k >= NU)
            ok = warp_all(mbar_wait_bounded(bar(bars.unit_empty, k % NU), ((k / NU) - 1) & 1,
                                            p.status, true));
        if (lane == 0) {
            if (ok) {
                bars.unit[k % NU].n_tiles = 0;
                mbar_arrive(bar(bars.unit_full, k % NU));
            } else {
                report(p.status, PA_ERR_TIMEOUT);
            }
        }
    } else if (warp == kKWarp || warp == kVWarp) {
        // ---- loaders: lane i issues the TMA copies of block i of a tile
        const bool is_k = warp == kKWarp;
        const uint32_t run_bytes = (uint32_t)B * 128u * NP;
        const CUtensorMap *map = is_k ? &maps.k : &maps.v;
        uint64_t *full = is_k ? bars.k_full : bars.v_full;
        uint64_t *empty = is_k ? bars.k_empty : bars.v_empty;
        const uint32_t ring = is_k ? sK : sV;
        const int NS = is_k ? NSK : NSV;
        const int nb = TBN >> p.bshift;   // blocks per tile (tiles start on a block)
        const uint64_t keep = l2_policy_evict_last();
        int g = 0;                        // tiles issued so far (all units)
        bool ok = true;
        for (int k = 0; ok; ++k) {
            Unit u;
            get_unit(k, u);
            if (lane == 0 && u.n_tiles >= 0) mbar_arrive(bar(bars.unit_empty, k % NU));
            if (u.n_tiles <= 0) {
                ok = u.n_tiles == 0;
                break;
            }
            const int32_t *table = p.tables + (size_t)u.s * p.max_blocks;
            if (is_k) {
                // the unit's 128 query rows of head h (rows past the end of q read
                // as zeros; rows of the next sequence are harmless: never stored)
                const int qb = k & 1;
                if (k >= 2)
                    ok = warp_all(mbar_wait_bounded(bar(bars.q_empty, qb), ((k >> 1) - 1) & 1,
                                                    p.status, true));
                if (!ok) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(bars.q_full, qb), L::TILE);
#pragma unroll
                    for (int pn = 0; pn < NP; ++pn)
                        tma_load_3d(sQ + qb * L::TILE + pn * kPanel, &maps.q, pn * 64, u.h,
                                    u.q_beg + u.q0, bar(bars.q_full, qb), l2_evict_first_policy());
                }
                __syncwarp();
            }
            // block ids are read one tile ahead (and the runs of the tile
            // kPrefetchTiles ahead prefetched into L2), so that neither the table
            // read nor the copy waits on the other
            auto entry = [&](int t) {
                const int jt = t * TBN + (lane << p.bshift);
                return (t < u.n_tiles && lane < nb && jt < u.n_end) ? __ldg(table + (jt >> p.bshift)) : -1;
            };
            int phys_next = entry(0);
            for (int t = 0; t < u.n_tiles; ++t, ++g) {
                const int st = g % NS;
                const int phys = phys_next;
                phys_next = entry(t + 1);
                if (g >= NS)
                    ok = warp_all(mbar_wait_bounded(bar(empty, st), ((g / NS) - 1) & 1, p.status, true));
                if (!ok) break;
                const int n0 = t * TBN;
                const int j = n0 + (lane << p.bshift);   // first position of block `lane`
                const bool present = lane < nb && j < u.n_end;
                const bool in_pool = present && phys >= 0 && phys < p.num_blocks;
                if (present && !in_pool) report(p.status, PA_ERR_BAD_BLOCK);
                // V: the block holding the context's last position is copied up to
                // it, in boxes of 16, 8, 4, 2 and 1 rows (slots past it are never read)
                const int nv = min(B, u.n_end - j);
                const bool partial = !is_k && in_pool && nv < B;
                const uint32_t whole = __popc(__ballot_sync(0xffffffffu, in_pool && !partial));
                const uint32_t part_rows = __reduce_add_sync(0xffffffffu, partial ? (uint32_t)nv : 0u);
                if (lane == 0)
                    mbar_arrive_expect_tx(bar(full, st), whole * run_bytes + part_rows * 128u * NP);
                __syncwarp();
                const uint32_t jrow = (uint32_t)(lane << p.bshift);   // block's first tile row
                const uint32_t tile = ring + st * L::TILE;
                const int y = (phys * H + u.h) << p.bshift;
                if (in_pool && !partial) {
                    if (NP == 2 && B >= 8) {
                        tma_load_4d(tile + kv_row_off<D>(jrow), map, 0, 0, 0, y >> 3, bar(full, st), keep);
                    } else {
#pragma unroll
                        for (int pn = 0; pn < NP; ++pn)
                            tma_load_2d(tile + kv_row_off<D>(jrow) + pn * 1024u, map, pn * 64, y,
                                        bar(full, st), keep);
                    }
                } else if (partial) {
                    // pieces of 8 rows (each one whole group), then 4, 2 and 1
                    // (never crossing a group: the block starts on a group or, at
                    // B = 4, half-way into one)
                    int r = 0;
                    auto piece = [&](int m) {
#pragma unroll
                        for (int pn = 0; pn < NP; ++pn)
                            tma_load_2d(tile + kv_row_off<D>(jrow + (uint32_t)r) + pn * 1024u,
                                        &maps.v_part[m], pn * 64, y + r, bar(full, st), keep);
                        r += 8 >> m;
                    };
                    while (r + 8 <= nv) piece(0);
#pragma unroll
                    for (int m = 1; m < kVPartMaps; ++m)
                        if (nv & (8 >> m)) piece(m);
                }
                if (t + kPrefetchTiles < u.n_tiles) {
                    const int pp = entry(t + kPrefetchTiles);
                    if (pp >= 0 && pp < p.num_blocks)
                        prefetch_l2((is_k ? p.k_cache : p.v_cache) + ((size_t)pp * H + u.h) * ((size_t)B * D),
                                    (uint32_t)B * D * 2);
                }
            }
        }
        if (!ok) report(p.status, PA_ERR_TIMEOUT);
    } else if (warp == kMmaWarp) {
        // ---- one thread issues the MMAs; it polls its dependencies so that a
        // P V product never waits behind the next unit's Q K^T
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_f16(TBM, TBN, false);
            constexpr uint32_t idO = tc::idesc_f16(TBM, D, true);
            int ks = 0, ts = 0, gs = 0;   // S cursor: unit, tile in unit, global tile
            int kp = 0, tp = 0, gp = 0;   // P V cursor
            int s_tiles = -1;             // tiles of the S cursor's unit; -1: not read yet
            bool s_end = false, ok = true;
            uint64_t last = globaltimer_ns();
            uint32_t idle = 0;   // passes without progress
            while (ok) {
                bool progress = false;
                // read the S cursor's unit once it is published
                if (!s_end && s_tiles < 0 &&
                    mbar_test(bar(bars.unit_full, ks % NU), (ks / NU) & 1)) {
                    s_tiles = bars.unit[ks % NU].n_tiles;
                    if (s_tiles <= 0) s_end = true;
                    progress = true;
                }
                // P V of tile gp (its S was issued); a unit's first one overwrites O,
                // so it also waits for the epilogue to have read the previous unit's
                if (gp < gs && mbar_test(bar(bars.p_full, gp % NSB), (gp / NSB) & 1) &&
                    mbar_test(bar(bars.v_full, gp % NSV), (gp / NSV) & 1) &&
                    (tp > 0 || kp == 0 || mbar_test(smem_addr(&bars.o_free), (kp - 1) & 1))) {
                    tc::fence_after();
                    const uint32_t vb = sV + (gp % NSV) * L::TILE;
#pragma unroll
                    for (int kk = 0; kk < TBN / 16; ++kk) {
                        // 16 rows = 2 groups; panels 1 KB apart, groups NP KB apart
                        const uint64_t dv = tc::smem_desc(vb + kk * 2048u * NP, 1024, 1024u * NP);
                        // P of keys 16 kk .. 16 kk + 15: column half (kk / 4) * 64, then
                        // 16 columns per 32 keys, 8 columns (16 fp16) per slice
                        const uint32_t pa = tmem + (gp % NSB) * 128 + (kk >> 2) * 64 +
                                            ((kk >> 1) & 1) * 16 + (kk & 1) * 8;
                        tc::mma_ts(tmem + kOCol, pa, dv, idO, (tp > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::commit(bar(bars.v_empty, gp % NSV));
                    tc::commit(bar(bars.pv_done, gp % NSB));
                    ++gp;
                    if (++tp == bars.unit[kp % NU].n_tiles) {   // unit kp done for this thread
                        mbar_arrive(bar(bars.unit_empty, kp % NU));
                        ++kp;
                        tp = 0;
                    }
                    progress = true;
                }
                // Q K^T of tile gs: buffer gs % NSB is free once P V of gs - NSB is done
                if (!s_end && s_tiles > 0 && gs < gp + NSB &&
                    (ts > 0 || mbar_test(bar(bars.q_full, ks & 1), (ks >> 1) & 1)) &&
                    mbar_test(bar(bars.k_full, gs % NSK), (gs / NSK) & 1) &&
                    (gs < NSB || mbar_test(bar(bars.pv_done, gs % NSB), ((gs - NSB) / NSB) & 1))) {
                    tc::fence_after();
                    const uint32_t qb = sQ + (ks & 1) * L::TILE, kb = sK + (gs % NSK) * L::TILE;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        // Q: [panel][128 rows]; K: 8-row groups of NP panels
                        const uint32_t col = (kk & 3) * 32;
                        tc::mma_ss(tmem + (gs % NSB) * 128,
                                   tc::smem_desc(qb + (kk >> 2) * kPanel + col, 16, 1024),
                                   tc::smem_desc(kb + (kk >> 2) * 1024u + col, 16, 1024u * NP), idS,
                                   kk > 0 ? 1u : 0u);
                    }
                    tc::commit(bar(bars.s_full, gs % NSB));
                    tc::commit(bar(bars.k_empty, gs % NSK));
                    ++gs;
                    if (++ts == s_tiles) {   // last Q K^T of the unit: its Q buffer may go
                        tc::commit(bar(bars.q_empty, ks & 1));
                        ++ks;
                        ts = 0;
                        s_tiles = -1;
                    }
                    progress = true;
                }
                if (s_end && gp == gs) break;   // every issued tile has its product
                // timeout check every 256 idle passes (reading the timer is not free)
                if (progress) {
                    idle = 0;
                } else if ((++idle & 255) == 0) {
                    const uint64_t now = globaltimer_ns();
                    if (idle == 256) last = now;
                    if (now - last > kWaitLimitNs ||
                        *(volatile const int32_t *)p.status == PA_ERR_TIMEOUT)
                        ok = false;
                }
            }
            if (!ok) report(p.status, PA_ERR_TIMEOUT);
            if (s_end) mbar_arrive(bar(bars.unit_empty, ks % NU));   // the end marker's slot
            tc::commit(smem_addr(&bars.done));   // lets the teardown wait for every MMA issued
        }
        __syncwarp();
    } else if (warp < kMmaWarp) {
        // ---- softmax warps: warps w and w + 4 share the query rows of tensor-memory
        // lane quarter w % 4 (row = lane of that quarter); warp w < 4 takes key
        // columns 0-63 of each tile, warp w + 4 columns 64-127.  They leave the
        // loops only together, at a meeting (a unit's start or a tile's maxima
        // exchange), so that no meeting ever waits for a warp that has gone.
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const float qs = p.qscale;
        bool ok = true, stop = false;
        int g = 0;   // tiles processed so far (all units)
        for (int k = 0; !stop; ++k) {
            Unit u;
            get_unit(k, u);
            if (lane == 0 && u.n_tiles >= 0) mbar_arrive(bar(bars.unit_empty, k % NU));
            ok = ok && u.n_tiles >= 0;
            if (!group_all(3, 256, ok && u.n_tiles > 0)) break;   // end marker or a failure
            const int qi = u.q0 + row;
            const int pos = u.pos0 + min(qi, u.ql - 1);
            float m_run = -INFINITY, l_run = 0.f;
            for (int t = 0; t < u.n_tiles; ++t, ++g) {
                const int b = g % NSB;
                ok = ok && warp_all(mbar_wait_bounded(bar(bars.s_full, b), (g / NSB) & 1, p.status, true));
                const uint32_t sb = lane_base + b * 128 + half * 64;
                const int n0 = t * TBN + half * 64;   // first key of this warp's columns
                // keys past this row's position are masked: key n0 + 32 cc + i with i > lim
                const bool need_mask = n0 + 63 > u.pos0 + u.q0;
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
                bars.red[g & 1][half][row] = mt;
                // the two halves of each row meet here once per tile: one exit
                // decision for all softmax warps, and the partner's maximum
                if (!group_all(3, 256, ok)) {
                    stop = true;
                    break;
                }
                mt = fmaxf(mt, bars.red[g & 1][half ^ 1][row]);
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
                    uint32_t r[32], w[16];
                    tc::ld32(sb + cc * 32, r);
                    tc::wait_ld();
                    if (need_mask) {
                        const int lim = pos - (n0 + cc * 32);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float p0 =
                                2 * i > lim ? 0.f : ex2(fmaf(__uint_as_float(r[2 * i]), qs, -m_run));
                            const float p1 = 2 * i + 1 > lim
                                                 ? 0.f
                                                 : ex2(fmaf(__uint_as_float(r[2 * i + 1]), qs, -m_run));
                            ls[i & 3] += p0 + p1;
                            w[i] = pack_pair(p0, p1);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float p0 = ex2(fmaf(__uint_as_float(r[2 * i]), qs, -m_run));
                            const float p1 = ex2(fmaf(__uint_as_float(r[2 * i + 1]), qs, -m_run));
                            ls[i & 3] += p0 + p1;
                            w[i] = pack_pair(p0, p1);
                        }
                    }
                    // P of these 32 keys as 16 fp16 pairs over S columns already read
                    tc::st16(sb + cc * 16, w);
                }
                l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                tc::wait_st();
                if (__any_sync(0xffffffffu, resc && t > 0)) {
                    // O holds tiles < t of this unit: wait until their product is
                    // complete, then scale this warp's half of the output columns
                    if (warp_all(mbar_wait_bounded(bar(bars.pv_done, (g - 1) % NSB),
                                                   ((g - 1) / NSB) & 1, p.status, true))) {
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
            if (stop) break;
            // the unit's row sums for the epilogue warps (slot k & 1 is free once
            // the epilogue of unit k - 2 has read it)
            if (k >= 2)
                ok = ok && warp_all(mbar_wait_bounded(bar(bars.l_empty, k & 1), ((k >> 1) - 1) & 1,
                                                      p.status, true));
            if (ok) bars.red_l[k & 1][half][row] = l_run;
            mbar_arrive(bar(bars.l_full, k & 1));
        }
        if (!ok) report(p.status, PA_ERR_TIMEOUT);
    } else {
        // ---- epilogue warps 12-15: warp 12 + q takes the rows of tensor-memory
        // lane quarter q.  After a unit's last P V: read O, normalised and as
        // fp16, into registers, release O to the next unit's first product, then
        // write the rows.  Rows past the unit's queries are not written.
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        bool ok = true;
        int g = 0;   // tiles of this CTA's units so far
        for (int k = 0; ok; ++k) {
            Unit u;
            get_unit(k, u);
            if (lane == 0 && u.n_tiles >= 0) mbar_arrive(bar(bars.unit_empty, k % NU));
            if (u.n_tiles <= 0) {
                ok = u.n_tiles == 0;
                break;
            }
            g += u.n_tiles;
            const int last = g - 1;
            ok = warp_all(mbar_wait_bounded(bar(bars.l_full, k & 1), (k >> 1) & 1, p.status, true));
            const float inv = ok ? 1.f / (bars.red_l[k & 1][0][row] + bars.red_l[k & 1][1][row]) : 0.f;
            mbar_arrive(bar(bars.l_empty, k & 1));
            ok = ok && warp_all(mbar_wait_bounded(bar(bars.pv_done, last % NSB), (last / NSB) & 1,
                                                  p.status, true));
            uint32_t hv[D / 2];   // the row as fp16 pairs
            if (ok) {
                tc::fence_after();
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t r[32];
                    tc::ld32(lane_base + kOCol + cc * 32, r);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        hv[cc * 16 + i] = pack_pair(__uint_as_float(r[2 * i]) * inv,
                                                    __uint_as_float(r[2 * i + 1]) * inv);
                }
            }
            tc::fence_before();
            mbar_arrive(smem_addr(&bars.o_free));
            if (!ok) break;
            // 16-byte chunks transposed within groups of 8 lanes (an 8 x 8
            // exchange per 64 columns), so that each store instruction writes 4
            // whole 128-byte row segments
            const int qi = u.q0 + row;
            const unsigned long long mine =
                qi < u.ql ? reinterpret_cast<unsigned long long>(p.out + ((size_t)(u.q_beg + qi) * H + u.h) * D)
                          : 0ull;
            const int c = lane & 7;
#pragma unroll
            for (int pass = 0; pass < D / 64; ++pass) {
                uint32_t *x = hv + pass * 32;   // chunk e = x[4e .. 4e + 3]
#pragma unroll
                for (int m = 1; m < 8; m <<= 1) {
                    const bool up = (c & m) != 0;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (e & m) continue;
#pragma unroll
                        for (int wd = 0; wd < 4; ++wd) {
                            uint32_t &a = x[4 * e + wd], &b2 = x[4 * (e | m) + wd];
                            const uint32_t r = __shfl_xor_sync(0xffffffffu, up ? a : b2, m);
                            if (up) a = r; else b2 = r;
                        }
                    }
                }
                // lane c now holds chunk c of rows (lane - c) + e in x[4e ..]
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const unsigned long long ptr = __shfl_sync(0xffffffffu, mine, (lane & ~7) + e);
                    if (ptr)
                        __stcs(reinterpret_cast<uint4 *>(ptr) + pass * 8 + c,
                               make_uint4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]));
                }
            }
        }
        if (!ok) report(p.status, PA_ERR_TIMEOUT);
    }

    // ---- teardown: every MMA drained (bounded), then tensor memory freed
    tc::fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        if (lane == 0 && !mbar_wait_bounded(smem_addr(&bars.done), 0, p.status, false))
            report(p.status, PA_ERR_TIMEOUT);
        __syncwarp();
        tc::fence_after();
        tc::dealloc(tmem, kTmemCols);
    }
}

template <int D>
cudaError_t set_prefill_smem_once() {
    static std::once_flag once[64];
    static cudaError_t err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        err[dev] = cudaFuncSetAttribute(paged_prefill_tc<D>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)TcLayout<D>::BYTES);
    });
    return err[dev];
}

int sm_count_of_current_device() {
    static std::once_flag once[64];
    static int n[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::call_once(once[dev], [&] {
        if (cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            n[dev] = 0;
    });
    return n[dev];
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

// fp16 tensor of rank 2 ([rows][D]) or 3 ([rows][H][D]) with a box of 64
// values (one 128-byte swizzle row) by `box_rows` rows (and one head).
int encode_map(CUtensorMap *m, const void *base, int rank, uint64_t rows, int H, int D, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail(PA_ERR_CUDA, "pa_prefill_attention: cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3], elem[3] = {1, 1, 1};
    dims[0] = (cuuint64_t)D;
    strides[0] = (cuuint64_t)D * 2;
    box[0] = 64;
    if (rank == 2) {
        dims[1] = rows ? rows : 1;
        box[1] = (cuuint32_t)box_rows;
    } else {
        dims[1] = (cuuint64_t)H;
        dims[2] = rows ? rows : 1;
        strides[1] = (cuuint64_t)H * D * 2;
        box[1] = 1;
        box[2] = (cuuint32_t)box_rows;
    }
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)rank, const_cast<void *>(base),
                           dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PA_ERR_CUDA, "pa_prefill_attention: cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PA_OK;
}

// The cache as [row / 8][panel][row % 8][64] fp16 (D = 128, rows a multiple
// of 8), with a box of B / 8 such groups: one copy per (block, head) run that
// lands in the grouped shared-memory layout of the K and V tiles.
int encode_run_map(CUtensorMap *m, const void *base, uint64_t rows, int B) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail(PA_ERR_CUDA, "pa_prefill_attention: cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[4] = {64, 8, 2, rows / 8};
    const cuuint64_t strides[3] = {256, 128, 2048};   // bytes: next row, panel, 8-row group
    const cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)(B / 8)}, elem[4] = {1, 1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void *>(base), dims, strides,
                           box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PA_ERR_CUDA, "pa_prefill_attention: cuTensorMapEncodeTiled (run map) failed (%d)", (int)r);
    return PA_OK;
}

template <int D>
int launch_d(PrefillParams p, int n_seqs, const pa_pool_desc *d, cudaStream_t st) {
    cudaError_t e = set_prefill_smem_once<D>();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "prefill smem attribute: %s", cudaGetErrorString(e));
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return fail(PA_ERR_CUDA, "prefill: cannot read the SM count");
    const uint64_t cache_rows = (uint64_t)d->num_blocks * d->num_heads * d->block_size;
    const int H = d->num_heads;
    TcMaps maps;
    int rc;
    if (D == 128 && d->block_size >= 8) {   // the kernel's one-box-per-run path
        rc = encode_run_map(&maps.k, p.k_cache, cache_rows, d->block_size);
        if (rc == PA_OK) rc = encode_run_map(&maps.v, p.v_cache, cache_rows, d->block_size);
    } else {
        rc = encode_map(&maps.k, p.k_cache, 2, cache_rows, H, D, d->block_size);
        if (rc == PA_OK) rc = encode_map(&maps.v, p.v_cache, 2, cache_rows, H, D, d->block_size);
    }
    for (int m = 0; rc == PA_OK && m < kVPartMaps; ++m)
        rc = encode_map(&maps.v_part[m], p.v_cache, 2, cache_rows, H, D, 8 >> m);
    if (rc == PA_OK) rc = encode_map(&maps.q, p.q, 3, (uint64_t)p.q_rows, H, D, TBM);
    if (rc != PA_OK) return rc;
    p.q_tiles = (p.max_q_len + TBM - 1) / TBM;
    paged_prefill_tc<D><<<sms, kTcThreads, TcLayout<D>::BYTES, st>>>(p, maps, n_seqs);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

}  // namespace

int launch_prefill_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, const int32_t *ctx_lens,
                             const int32_t *q_starts, int32_t n_seqs, int32_t max_blocks,
                             int32_t max_q_len, int32_t q_rows, float scale, int32_t *status,
                             const pa_pool_desc *d, void *stream) {
    if (!d) return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: desc is NULL");
    std::string why;
    if (!device_geometry_ok(d, &why)) return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: %s", why.c_str());
    if (d->head_dim != 64 && d->head_dim != 128)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: head_dim %d not in {64, 128}",
                    d->head_dim);
    if (n_seqs < 0 || max_blocks < 0 || max_q_len < 0 || q_rows < 0)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: negative size");
    if (n_seqs > 65535 || d->num_heads > 65535)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_attention: more than 65535 sequences or heads");
    if (n_seqs == 0 || max_q_len == 0 || q_rows == 0) return PA_OK;
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
    p.q_rows = q_rows;
    p.q_tiles = 0;   // set by the launcher from its tile height
    p.bshift = bshift;
    p.qscale = scale * 1.4426950408889634f;
    p.status = status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return d->head_dim == 64 ? launch_d<64>(p, n_seqs, d, st) : launch_d<128>(p, n_seqs, d, st);
}

}  // namespace pagedkv
