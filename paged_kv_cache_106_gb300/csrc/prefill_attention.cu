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
//   - persistent: one CTA per SM walks units of work; a unit is one or two
//     query tiles (128 queries each) of one (sequence, head): tiles x and
//     x - 1 of a prompt share their keys and values, so each K/V tile is
//     copied once for both.  Each query tile has a slot: a Q buffer, S and O
//     in tensor memory (S0, S1, O0, O1: 128 columns each) and a softmax
//     warpgroup; a unit with one query tile takes the slots in turn.
//       warps 0-7 / 8-15  softmax and epilogue of slot 0 / 1: warps w and
//                  w + 4 share the query rows of tensor-memory lane quarter
//                  w % 4, each half of a tile's key columns, and meet once per
//                  tile (a named barrier of the two warps) to combine row
//                  maxima;
//       warp 16    one thread issues every tcgen05.mma and commit, in the
//                  order P V (slot 0), Q K^T of the next key tile (slot 0),
//                  then the same for slot 1, so one slot's products run on
//                  the tensor pipe while the other slot's softmax works;
//       warp 17    Q tiles and K tiles by TMA, warp 18 V tiles by TMA;
//       warp 19    scheduler: takes units one at a time from the launch's
//                  counter (CTAs that finish early take more) and publishes
//                  them through a 4-slot descriptor ring.
//     A job's output is written by its softmax warps at the slot's next job:
//     after writing that job's first P they read the old O (complete: the
//     new S was committed after its last P V), release it to the first P V,
//     and normalise and store while the tensor pipe works (16-byte streaming
//     stores, chunks exchanged between lanes so that each store instruction
//     writes whole row segments; only the unit's rows).
//   - K/V tiles are copied with an evict-last L2 policy (later query tiles
//     re-read them), query tiles with evict-first; the runs of the key tile
//     two steps ahead are prefetched into L2.
//   - K and V tiles sit in shared memory as 8-row groups, [j / 8][64-column
//     panel][j % 8][128 bytes], 128-byte swizzled; a (block, head) run of
//     B >= 8 rows is whole groups and one 4-D TMA copy moves it (at D = 128;
//     at B = 4 or D = 64, one 2-D copy per panel).  The same bytes are the
//     K-major B operand of S = Q K^T and the MN-major B operand of O = P V.
//     The V block holding the context's last position is copied up to it in
//     boxes of 8, 4, 2 and 1 rows, and the V ring starts zeroed, so slots
//     past the context are never read.
//   - the softmax is online, in base 2 (ex2.approx), with a lazy rescale: a
//     row's reference maximum moves only when a tile raises it by more than
//     2^8.  P (<= 2^8) is written over S as fp16 and read by P V straight
//     from tensor memory; fp16, like the output, keeps the output rounding
//     the larger error.
//   - keys after a row's own position are masked to -inf (a select, so
//     stale shared memory cannot leak in); blocks past the causal end of a
//     tile are not copied.
//   - every mbarrier wait is bounded; a wait that runs out reports
//     PA_ERR_TIMEOUT, and the CTA drains its MMAs (bounded) and frees its
//     tensor memory before it returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "tc_device.cuh"

namespace pagedkv {
namespace {

// Work counters of the prefill launches.  A launch takes its units one at a
// time from `next`; each block adds one to `done` when it takes no more, and
// the last one sets both back to zero, so that the next launch (on the same
// stream, or a replay of the same graph) finds zeros.  Launches pick counter
// (call number % kUnitCounters): calls on different streams stay apart while
// fewer than kUnitCounters of them are in flight at once.
struct UnitCounter {
    unsigned long long next;
    unsigned int done;
    unsigned int pad;
};
constexpr int kUnitCounters = 64;
__device__ UnitCounter g_unit_ctr[kUnitCounters];

struct PrefillParams {
    __half *out;
    const __half *q;
    const __half *k_cache;
    const __half *v_cache;
    const int32_t *tables;
    const int32_t *ctx_lens;
    const int32_t *q_starts;
    int32_t num_heads, num_blocks, max_blocks, max_q_len, q_rows, bshift;
    float qscale;  // scale * log2(e): softmax evaluated with exp2
    int32_t *status;
    UnitCounter *units;             // this launch's unit counter
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

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two fp32 values as one packed pair, and back.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// Packed fp32 pairs: a * b + c and a + b, element by element, one instruction
// each (round to nearest, as fmaf and + on each element).
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Two probabilities as one fp16 pair (lower column in the low half).
__device__ __forceinline__ uint32_t pack_pair(float p0, float p1) {
    const __half2 h = __floats2half2_rn(p0, p1);
    return *reinterpret_cast<const uint32_t *>(&h);
}

constexpr int TBM = 128;          // queries per query tile (= tensor-memory lanes)
constexpr int TBN = 128;          // key positions per key tile
constexpr int NSK = 2;            // K ring stages
constexpr int NSV = 2;            // V ring stages
static_assert(NSK == NSV, "the K and V rings advance together");
constexpr int NU = 4;             // unit descriptors in flight
constexpr int kLookahead = 2;     // units a block takes before its readers have fetched them all
// warps 0-7: softmax and epilogue of slot 0, 8-15: of slot 1
constexpr int kMmaWarp = 16, kKWarp = 17, kVWarp = 18, kSchedWarp = 19;
constexpr int kTcThreads = 640;   // 20 warps
constexpr uint32_t kPanel = TBM * 128;   // bytes of one 64-column panel of a 128-row tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;          // S of slot x at columns 128 x, its O at kOCol + 128 x
constexpr float kRescaleLog2 = 8.f;      // lazy-rescale threshold (log2 units)
// readers of a unit descriptor: K loader, V loader, MMA thread, 16 softmax warps
constexpr uint32_t kUnitReaders = 3 + 16;
constexpr int kPrefetchTiles = 2;  // K/V tiles prefetched into L2 ahead of their copies
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

// One unit of work: one or two query tiles of one (sequence, head) that share
// their keys and values, each on a slot (tensor-memory S and O, a Q buffer
// and a softmax warpgroup of its own).  A pair is query tiles x and x - 1;
// slot 0 takes x (the one with the most keys).
struct Unit {
    int32_t s, h, q_beg, ql, pos0;
    int32_t n_end, n_tiles;   // keys of the unit (its slots' union) and their key tiles; 0: no more units
    int32_t q0[2], nt[2];     // per slot: first query (within the prompt) and key tiles; nt 0: no job
};

// Tensor maps: K and V cache runs (D = 128 with B >= 8: a 4-D view
// [row / 8][panel][row % 8][64] with one box per (block, head) run; otherwise
// rows of D values, box 64 x B, one copy per panel), cache rows for the
// partial V block (boxes 64 x 8 .. 64 x 1), and query rows as a 3-D
// [rows][H][D] tensor with one box of 128 rows.
struct TcMaps {
    CUtensorMap k, v, v_part[kVPartMaps], q;
    // whole prompts written and attended in one call: the new keys and values
    // as 3-D [rows][H][D] tensors (boxes of 128 rows, like q), and the cache as
    // rows of D values with a box of 64 x B (one store per block and panel);
    // a prompt's last, partial block is stored in boxes of 8, 4, 2 and 1 rows
    // (v_part for values, k_part for keys)
    CUtensorMap kn, vn, ks, vs, k_part[kVPartMaps];
};

struct TcBars {
    uint64_t unit_full[NU], unit_empty[NU];
    uint64_t q_full[2], q_empty[2];           // per slot
    uint64_t k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV];
    uint64_t s_full[2], p_full[2];            // per slot: S written, P written
    uint64_t o_full[2];                       // per slot: a job's O complete
    uint64_t o_free[2];                       // per slot: a job's O read (the next job may overwrite it)
    uint64_t done;
    uint32_t tmem;
    Unit unit[NU];
    float red[2][2][2][TBM];                  // per slot, tile parity and column half: row maxima
    float red_l[2][2][TBM];                   // per slot and column half: a finished job's row sums
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

// 2-D tensor copy shared -> global (box of the tensor map at element
// coordinates x, y), in this thread's bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until every bulk group of this thread is complete (its writes done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Persistent: one CTA per SM takes units one at a time from the launch's
// counter, in the order sequence, then query-tile pair (the last, with the
// most keys, first), then head.  All heads of a pair run side by side on
// different SMs (different keys and values), and the next pair of the same
// (sequence, head), which re-reads a prefix of its keys and values, follows
// while they are still in L2.
// KN: every sequence is a whole prompt whose keys and values are read from
// the new rows (k_new, v_new) instead of the cache, and the unit that reaches
// a prompt's last key also stores every key tile's blocks into the cache
// (the prompt's slot write, done in the same pass).
template <int D, bool KN>
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
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(bars.q_full, x), 1);
            mbar_init(bar(bars.q_empty, x), 1);   // the job's last Q K^T is done
            mbar_init(bar(bars.s_full, x), 1);
            mbar_init(bar(bars.p_full, x), 8);    // the slot's softmax warps
            mbar_init(bar(bars.o_full, x), 1);
            mbar_init(bar(bars.o_free, x), 8);    // the slot's softmax warps
        }
        for (int i = 0; i < NSK; ++i) {
            mbar_init(bar(bars.k_full, i), 1);
            mbar_init(bar(bars.k_empty, i), 1);
        }
        for (int i = 0; i < NSV; ++i) {
            mbar_init(bar(bars.v_full, i), 1);
            mbar_init(bar(bars.v_empty, i), 1);
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
        // ---- scheduler: the launch's units in the order (sequence, pair of
        // query tiles from the last, head) are taken one at a time from the
        // launch's counter, so that blocks that finish early take more (with a
        // fixed share per block, the 256-prompt batch gave the heaviest block
        // about 5 % more work than the mean).  A unit
        // index is mapped to its sequence by a cursor that walks the sequences
        // 32 at a time, summing their units; the indices a block takes only
        // grow, so its cursor only moves forward.  A unit is taken only once
        // every reader has fetched the unit two before it: a block holds few
        // units it has not started.  A unit with one query tile takes the slots
        // in turn, so that consecutive such units overlap.
        int k = 0, singles = 0;
        bool ok = true;
        int w0 = -32;                      // first sequence of the cursor's window
        unsigned long long before = 0;     // units of the sequences before the window
        unsigned long long incl = 0;       // units of the window's sequences up to this lane's
        unsigned long long win = 0;        // units of the window
        unsigned long long own = 0;        // units of this lane's sequence
        for (;;) {
            if (k >= kLookahead)
                ok = warp_all(mbar_wait_bounded(bar(bars.unit_empty, (k - kLookahead) % NU),
                                                ((k - kLookahead) / NU) & 1, p.status, true));
            if (!ok) break;
            unsigned long long d = 0;
            if (lane == 0) d = atomicAdd(&p.units->next, 1ull);
            d = __shfl_sync(0xffffffffu, d, 0);
            while (d >= before + win && w0 + 32 < n_seqs) {
                before += win;
                w0 += 32;
                const int s = w0 + lane;
                unsigned long long n = 0;
                if (s < n_seqs) {
                    const int q_beg = p.q_starts[s], ql = p.q_starts[s + 1] - q_beg, ctx = p.ctx_lens[s];
                    // KN: whole prompts only (their keys and values are the new rows)
                    const bool bad_len = ql < 0 || ql > ctx || (KN && ql != ctx) || ql > p.max_q_len || q_beg < 0 ||
                                         (int64_t)q_beg + ql > p.q_rows;
                    const bool bad_ctx = (int64_t)ctx > ((int64_t)p.max_blocks << p.bshift);
                    // every block's cursor passes every sequence; one reports
                    if ((bad_len || bad_ctx) && blockIdx.x == 0)
                        report(p.status, bad_len ? PA_ERR_INVALID_ARG : PA_ERR_BAD_BLOCK);
                    if (!bad_len && !bad_ctx)
                        n = (unsigned long long)H * (unsigned long long)(((ql + TBM - 1) / TBM + 1) / 2);
                }
                own = n;
                incl = n;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                win = __shfl_sync(0xffffffffu, incl, 31);
            }
            if (d >= before + win) break;   // past the last unit
            const int src = __ffs(__ballot_sync(0xffffffffu, incl > d - before)) - 1;
            const unsigned long long excl = __shfl_sync(0xffffffffu, incl - own, src);
            Unit u{};
            u.s = w0 + src;
            const unsigned long long r = d - before - excl;   // unit within the sequence
            const int pr = (int)(r / (unsigned)H);
            u.h = (int)(r - (unsigned long long)pr * H);
            u.q_beg = p.q_starts[u.s];
            u.ql = p.q_starts[u.s + 1] - u.q_beg;
            const int ctx = p.ctx_lens[u.s];
            const int xa = (u.ql + TBM - 1) / TBM - 1 - 2 * pr;   // the pair's later query tile
            u.pos0 = ctx - u.ql;
            for (int x = 0; x < 2; ++x) {
                const int qt = xa - x;
                u.q0[x] = qt * TBM;
                const int end = u.pos0 + u.q0[x] + min(TBM, u.ql - u.q0[x]);
                u.nt[x] = qt >= 0 ? (end + TBN - 1) / TBN : 0;
            }
            u.n_end = u.pos0 + u.q0[0] + min(TBM, u.ql - u.q0[0]);
            u.n_tiles = u.nt[0];
            const bool single = u.nt[1] == 0;
            if (lane == 0) {
                if (single && (singles & 1)) {   // the lone tile goes to slot 1
                    u.q0[1] = u.q0[0];
                    u.nt[1] = u.nt[0];
                    u.nt[0] = 0;
                }
                bars.unit[k % NU] = u;
                mbar_arrive(bar(bars.unit_full, k % NU));
            }
            singles += single ? 1 : 0;
            __syncwarp();
            ++k;
        }
        // this block takes no more units; the last block resets the counter
        if (lane == 0 && atomicAdd(&p.units->done, 1u) == gridDim.x - 1) {
            p.units->next = 0;
            p.units->done = 0;
        }
        // end marker, once its ring slot is free
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
        // ---- loaders: lane i issues the TMA copies of block i of a key tile
        const bool is_k = warp == kKWarp;
        const uint32_t run_bytes = (uint32_t)B * 128u * NP;
        const CUtensorMap *map = is_k ? &maps.k : &maps.v;
        uint64_t *full = is_k ? bars.k_full : bars.v_full;
        uint64_t *empty = is_k ? bars.k_empty : bars.v_empty;
        const uint32_t ring = is_k ? sK : sV;
        const int NS = is_k ? NSK : NSV;
        const int nb = TBN >> p.bshift;   // blocks per key tile (tiles start on a block)
        const uint64_t keep = l2_policy_evict_last();
        int g = 0;                        // key tiles issued so far (all units)
        int job[2] = {0, 0};              // Q tiles loaded per slot (K loader)
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
                // each slot's 128 query rows of head h, into the slot's Q buffer once
                // its previous job's last Q K^T is done (rows past the end of q read
                // as zeros; rows of the next sequence are harmless: never stored)
                for (int x = 0; x < 2 && ok; ++x) {
                    if (u.nt[x] == 0) continue;
                    if (job[x] >= 1)
                        ok = warp_all(mbar_wait_bounded(bar(bars.q_empty, x), (job[x] - 1) & 1,
                                                        p.status, true));
                    if (!ok) break;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar(bars.q_full, x), L::TILE);
#pragma unroll
                        for (int pn = 0; pn < NP; ++pn)
                            tma_load_3d(sQ + x * L::TILE + pn * kPanel, &maps.q, pn * 64, u.h,
                                        u.q_beg + u.q0[x], bar(bars.q_full, x), l2_evict_first_policy());
                    }
                    __syncwarp();
                    ++job[x];
                }
                if (!ok) break;
            }
            // block ids are read one tile ahead (and the runs of the tile
            // kPrefetchTiles ahead prefetched into L2), so that neither the table
            // read nor the copy waits on the other
            auto entry = [&](int t) {
                const int jt = t * TBN + (lane << p.bshift);
                return (t < u.n_tiles && lane < nb && jt < u.n_end) ? __ldg(table + (jt >> p.bshift)) : -1;
            };
            int phys_next = entry(0);
            // KN: the unit whose key range ends at the prompt's end writes it
            const bool writer = KN && u.n_end == u.pos0 + u.ql;
            int phys_prev = -1;   // block of this lane in the tile before (KN stores)
            // KN: stores key tile tt (ring position gg; this lane's block phys_t)
            // into the cache once it has landed; one bulk group per call
            auto store_tile = [&](int tt, int gg, int phys_t) {
                const int sg = gg % NS;
                if (!warp_all(mbar_wait_bounded(bar(full, sg), (gg / NS) & 1, p.status, true))) {
                    ok = false;
                    return false;
                }
                const int jt = tt * TBN + (lane << p.bshift);   // first position of block `lane`
                if (lane < nb && jt < u.n_end && phys_t >= 0 && phys_t < p.num_blocks) {
                    const int y = (phys_t * H + u.h) << p.bshift;
                    const uint32_t src = ring + sg * L::TILE + ((uint32_t)lane << p.bshift) * 128u;
                    const int nrow = min(B, u.n_end - jt);   // the block's rows in the prompt
                    if (nrow == B) {
#pragma unroll
                        for (int pn = 0; pn < NP; ++pn)
                            tma_store_2d(is_k ? &maps.ks : &maps.vs, pn * 64, y, src + pn * kPanel);
                    } else {
                        // the last block up to the prompt's end only (the slots past
                        // it keep what they held, as with the slot write)
                        int r = 0;
                        auto piece = [&](int m) {
#pragma unroll
                            for (int pn = 0; pn < NP; ++pn)
                                tma_store_2d(is_k ? &maps.k_part[m] : &maps.v_part[m], pn * 64, y + r,
                                             src + (uint32_t)r * 128u + pn * kPanel);
                            r += 8 >> m;
                        };
                        while (r + 8 <= nrow) piece(0);
#pragma unroll
                        for (int m = 1; m < kVPartMaps; ++m)
                            if (nrow & (8 >> m)) piece(m);
                    }
                }
                bulk_commit();
                return true;
            };
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
                if constexpr (KN) {
                    // the tile's rows of the new keys (values), one box per panel
                    // into the Q-like layout [panel][row][128 bytes]; rows past the
                    // prompt belong to the next prompt (or read as zeros past the
                    // last row) and meet masked scores or P = 0.  First, this
                    // lane's stores from the stage (tile g - 2, stored while tile
                    // g - 1 loaded) have read it.
                    bulk_wait_read<0>();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar(full, st), L::TILE);
#pragma unroll
                        for (int pn = 0; pn < NP; ++pn)
                            tma_load_3d(ring + st * L::TILE + pn * kPanel, is_k ? &maps.kn : &maps.vn,
                                        pn * 64, u.h, u.q_beg + n0, bar(full, st), keep);
                    }
                    __syncwarp();
                    // the unit that reaches the prompt's last key stores each tile's
                    // blocks into the cache, one tile behind its loads
                    if (writer && t > 0 && !store_tile(t - 1, g - 1, phys_prev)) break;
                    phys_prev = phys;
                    continue;
                }
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
            if (KN && writer && ok) store_tile(u.n_tiles - 1, g - 1, phys_prev);   // the last tile
        }
        if (KN) bulk_wait_all();   // this lane's cache stores done before the CTA exits
        if (!ok) report(p.status, PA_ERR_TIMEOUT);
    } else if (warp == kMmaWarp) {
        // ---- one thread issues the MMAs in a fixed order, per key tile j of a
        // unit: P V of slot 0, then its Q K^T of key tile j + 1, then the same
        // for slot 1.  A Q K^T that overwrites a slot's S (where its P lies) is
        // issued right after the P V that reads that P: tcgen05.mma operations
        // of one thread execute in issue order.  While slot 0's softmax works,
        // the tensor pipe runs slot 1's products, and the other way round.
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_f16(TBM, TBN, false);
            constexpr uint32_t idO = tc::idesc_f16(TBM, D, true);
            int g = 0;                    // key tiles of the units so far (K/V ring position)
            int job[2] = {0, 0};          // jobs started per slot
            int pc[2] = {0, 0};           // P tiles consumed per slot
            bool ok = true;
            auto wait = [&](uint32_t b, uint32_t par) {
                if (ok) ok = mbar_wait_bounded(b, par, p.status, true);
                return ok;
            };
            // the same, polling: for what the next product waits on (a slot's P,
            // K, V, Q, O released), a polled wait sees the arrival sooner than a
            // suspended one (measured: 0.940 -> 0.918 ms on the 256-prompt batch)
            auto spin = [&](uint32_t b, uint32_t par) {
                if (!ok || mbar_test(b, par)) return ok;
                const uint64_t t0 = globaltimer_ns();
                for (uint32_t n = 1; !mbar_test(b, par); ++n)
                    if ((n & 1023) == 0 && (globaltimer_ns() - t0 > kWaitLimitNs ||
                                            *(volatile const int32_t *)p.status == PA_ERR_TIMEOUT))
                        return ok = false;
                return true;
            };
            // S_x = Q_x K^T for the key tile in K ring stage st.  A descriptor's
            // start address is its low field (address / 16; shared memory is far
            // below the field's range), so the descriptors of successive slices
            // are one base plus a constant.
            auto issue_s = [&](int x, int st) {
                const uint64_t dq = tc::smem_desc(sQ + x * L::TILE, 16, 1024);
                // K: 8-row groups of NP panels, or (KN) laid out like Q
                const uint64_t dk = tc::smem_desc(sK + st * L::TILE, 16, KN ? 1024u : 1024u * NP);
                constexpr uint32_t kPanelStep = KN ? kPanel : 1024u;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // Q: [panel][128 rows]
                    const uint32_t col = (kk & 3) * 32;
                    tc::mma_ss(tmem + x * 128, dq + (((kk >> 2) * kPanel + col) >> 4),
                               dk + (((kk >> 2) * kPanelStep + col) >> 4), idS, kk > 0 ? 1u : 0u);
                }
                tc::commit(bar(bars.s_full, x));
            };
            for (int k = 0; ok; ++k) {
                if (!wait(bar(bars.unit_full, k % NU), (k / NU) & 1)) break;
                const Unit u = bars.unit[k % NU];
                mbar_arrive(bar(bars.unit_empty, k % NU));
                if (u.n_tiles <= 0) break;
                // first key tile: S of each slot with a job
                if (!spin(bar(bars.k_full, g % NSK), (g / NSK) & 1)) break;
                for (int x = 0; x < 2; ++x) {
                    if (u.nt[x] == 0) continue;
                    if (!spin(bar(bars.q_full, x), job[x] & 1)) break;
                    tc::fence_after();
                    issue_s(x, g % NSK);
                    if (u.nt[x] == 1) tc::commit(bar(bars.q_empty, x));
                }
                tc::commit(bar(bars.k_empty, g % NSK));
                for (int j = 0; ok && j < u.n_tiles; ++j) {
                    const int gj = g + j;
                    if (!spin(bar(bars.v_full, gj % NSV), (gj / NSV) & 1)) break;
                    bool k_next = false;   // key tile j + 1 waited for
                    for (int x = 0; x < 2; ++x) {
                        if (j >= u.nt[x]) continue;
                        if (!spin(bar(bars.p_full, x), pc[x] & 1)) break;
                        ++pc[x];
                        // a job's first P V overwrites O: the epilogue must have read
                        // the slot's previous job
                        if (j == 0 && job[x] > 0 && !spin(bar(bars.o_free, x), (job[x] - 1) & 1)) break;
                        tc::fence_after();
                        // V: 16 rows = 2 groups; panels 1 KB apart, groups NP KB apart
                        // (KN: panels kPanel apart, groups 1 KB apart)
                        const uint64_t dv0 = KN ? tc::smem_desc(sV + (gj % NSV) * L::TILE, kPanel, 1024)
                                                : tc::smem_desc(sV + (gj % NSV) * L::TILE, 1024, 1024u * NP);
#pragma unroll
                        for (int kk = 0; kk < TBN / 16; ++kk) {
                            // P of keys 16 kk .. 16 kk + 15: column half (kk / 4) * 64, then
                            // 16 columns per 32 keys, 8 columns (16 fp16) per slice
                            const uint64_t dv = dv0 + ((kk * (KN ? 2048u : 2048u * NP)) >> 4);
                            const uint32_t pa =
                                tmem + x * 128 + (kk >> 2) * 64 + ((kk >> 1) & 1) * 16 + (kk & 1) * 8;
                            tc::mma_ts(tmem + kOCol + x * 128, pa, dv, idO, (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        if (j + 1 < u.nt[x]) {
                            if (!k_next && !spin(bar(bars.k_full, (gj + 1) % NSK), ((gj + 1) / NSK) & 1)) break;
                            k_next = true;
                            tc::fence_after();
                            issue_s(x, (gj + 1) % NSK);
                            if (j + 2 == u.nt[x]) tc::commit(bar(bars.q_empty, x));   // its last Q K^T
                        } else {
                            tc::commit(bar(bars.o_full, x));   // the job's O is complete
                            ++job[x];
                        }
                    }
                    if (!ok) break;
                    tc::commit(bar(bars.v_empty, gj % NSV));
                    if (k_next) tc::commit(bar(bars.k_empty, (gj + 1) % NSK));
                }
                g += u.n_tiles;
            }
            if (!ok) report(p.status, PA_ERR_TIMEOUT);
            tc::commit(smem_addr(&bars.done));   // lets the teardown wait for every MMA issued
        }
        __syncwarp();
    } else if (warp < kMmaWarp) {
        // ---- softmax and epilogue: warps 8x .. 8x + 7 serve slot x.  Warps w and
        // w + 4 of the slot share the query rows of tensor-memory lane quarter
        // w % 4; the first takes key columns 0-63 of each tile, the second
        // 64-127, and they meet once per tile (a named barrier of the two) to
        // combine their row maxima.  The slot's warps leave their loops only
        // together, at the vote that starts each unit.  A job's output is written at the start of
        // the slot's next job, when its O is complete (that job's first S was
        // committed after the last P V of the previous one), or after the last.
        const int x = warp >> 3, quarter = warp & 3, half = (warp >> 2) & 1;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t sb = lane_base + x * 128 + half * 64;
        const uint32_t ob = lane_base + kOCol + x * 128 + half * (D / 2);
        const int meet = 1 + x;   // named barrier of the slot (0 is __syncthreads)
        const int pair = 3 + 4 * x + quarter;   // named barrier of warps w and w + 4
        const float qs = p.qscale;
        bool ok = true;
        int sc = 0, job = 0;     // S tiles and jobs of this slot so far
        bool pend = false;       // the previous job's output is still in O
        float pend_l = 0.f;
        unsigned long long pend_out = 0;   // its row's half (none: a padded row)
        constexpr int NCH = D / 16;   // 16-byte chunks of a half row
        // this thread's half of the pending row, normalised, as fp16 pairs; after
        // a meeting, so that the partner's sum is in red_l
        auto epi_read = [&](uint32_t (&hv)[4 * NCH]) {
            const float inv = 1.f / (pend_l + bars.red_l[x][half ^ 1][row]);
            const uint64_t inv2 = pack_f32x2(inv, inv), zero2 = 0ull;
            tc::fence_after();
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t r[32];
                tc::ld32(ob + cc * 32, r);
                tc::wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float o0, o1;
                    unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(r[2 * i]),
                                                      __uint_as_float(r[2 * i + 1])),
                                           inv2, zero2),
                                 o0, o1);
                    hv[cc * 16 + i] = pack_pair(o0, o1);
                }
            }
        };
        // write it: chunks exchanged within groups of NCH lanes (an NCH x NCH
        // transpose), so that each store instruction writes whole row segments
        auto epi_store = [&](uint32_t (&hv)[4 * NCH]) {
            const int c = lane % NCH;
#pragma unroll
            for (int m = 1; m < NCH; m <<= 1) {
                const bool up = (c & m) != 0;
#pragma unroll
                for (int e = 0; e < NCH; ++e) {
                    if (e & m) continue;
#pragma unroll
                    for (int wd = 0; wd < 4; ++wd) {
                        uint32_t &a = hv[4 * e + wd], &b2 = hv[4 * (e | m) + wd];
                        const uint32_t r = __shfl_xor_sync(0xffffffffu, up ? a : b2, m);
                        if (up) a = r; else b2 = r;
                    }
                }
            }
            // lane c now holds chunk c of row (lane - c) + e in hv[4e ..]
#pragma unroll
            for (int e = 0; e < NCH; ++e) {
                const unsigned long long ptr = __shfl_sync(0xffffffffu, pend_out, lane - c + e);
                if (ptr)
                    __stcs(reinterpret_cast<uint4 *>(ptr) + c,
                           make_uint4(hv[4 * e], hv[4 * e + 1], hv[4 * e + 2], hv[4 * e + 3]));
            }
            pend = false;
        };
        for (int k = 0;; ++k) {
            Unit u;
            get_unit(k, u);
            if (lane == 0 && u.n_tiles >= 0) mbar_arrive(bar(bars.unit_empty, k % NU));
            ok = ok && u.n_tiles >= 0;
            if (!group_all(meet, 256, ok && u.n_tiles > 0)) break;   // end marker or a failure
            if (u.nt[x] == 0) continue;
            const int q0 = u.q0[x], qi = q0 + row;
            const int pos = u.pos0 + min(qi, u.ql - 1);   // this row's position
            // the last position among this warp's rows: key chunks after it are
            // masked for every row of the warp
            const int pos_w = u.pos0 + min(q0 + quarter * 32 + 31, u.ql - 1);
            // the position of this warp's first row: a chunk whose last key is at
            // or before it needs no mask for any real row of the warp (padded
            // rows past the queries are never stored)
            const int pos_f = u.pos0 + q0 + quarter * 32;
            float m_run = -INFINITY, l_run = 0.f;
            for (int t = 0; t < u.nt[x]; ++t, ++sc) {
                ok = ok && warp_all(mbar_wait_bounded(bar(bars.s_full, x), sc & 1, p.status, true));
                const int n0 = t * TBN + half * 64;   // first key of this warp's columns
                // keys past a row's position are masked: key n0 + 32 cc + i with i > lim
                float mt = -INFINITY;
                if (ok) {
                    tc::fence_after();
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
                    for (int cc = 0; cc < 2; ++cc) {
                        if (n0 + cc * 32 > pos_w) break;   // this chunk and the next: all masked
                        uint32_t r[32];
                        tc::ld32(sb + cc * 32, r);
                        tc::wait_ld();
                        if (n0 + cc * 32 + 31 > pos_f) {
                            const int lim = pos - (n0 + cc * 32);
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                m4[i & 3] = max3f(m4[i & 3], 2 * i > lim ? -INFINITY : __uint_as_float(r[2 * i]),
                                                  2 * i + 1 > lim ? -INFINITY : __uint_as_float(r[2 * i + 1]));
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                m4[i & 3] = max3f(m4[i & 3], __uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                        }
                    }
                    mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * qs;   // scale > 0
                }
                bars.red[x][sc & 1][half][row] = mt;
                if (t == 0 && pend) bars.red_l[x][half][row] = pend_l;
                // the two halves of each row meet (a barrier of the two warps): the
                // partner's maximum (and, on a job's first tile, the partner's sum
                // for the pending output).  A failed wait in either makes both
                // skip the rest of the unit's work, meeting at each tile still;
                // the slot's warps leave together at the next unit
                ok = group_all(pair, 64, ok);
                if (!ok) continue;
                mt = fmaxf(mt, bars.red[x][sc & 1][half ^ 1][row]);
                float corr = 1.f;
                const bool resc = mt > m_run + kRescaleLog2;
                if (resc) {
                    corr = ex2(m_run - mt);
                    m_run = mt;
                    l_run *= corr;
                }
                // x = s * qs - m_run and the running sum, two columns per instruction
                const uint64_t qs2 = pack_f32x2(qs, qs), negm2 = pack_f32x2(-m_run, -m_run);
                uint64_t ls2[2] = {0ull, 0ull};
#pragma unroll 1
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t r[32], w[16];
                    if (n0 + cc * 32 > pos_w) {   // all masked: P = 0, nothing to read
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = 0u;
                        tc::st16(sb + cc * 16, w);
                        continue;
                    }
                    tc::ld32(sb + cc * 32, r);
                    tc::wait_ld();
                    if (n0 + cc * 32 + 31 > pos_f) {
                        const int lim = pos - (n0 + cc * 32);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float x0, x1;
                            unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(r[2 * i]),
                                                              __uint_as_float(r[2 * i + 1])),
                                                   qs2, negm2),
                                         x0, x1);
                            const float p0 = 2 * i > lim ? 0.f : ex2(x0);
                            const float p1 = 2 * i + 1 > lim ? 0.f : ex2(x1);
                            ls2[i & 1] = add_f32x2(ls2[i & 1], pack_f32x2(p0, p1));
                            w[i] = pack_pair(p0, p1);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float x0, x1;
                            unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(r[2 * i]),
                                                              __uint_as_float(r[2 * i + 1])),
                                                   qs2, negm2),
                                         x0, x1);
                            const float p0 = ex2(x0), p1 = ex2(x1);
                            ls2[i & 1] = add_f32x2(ls2[i & 1], pack_f32x2(p0, p1));
                            w[i] = pack_pair(p0, p1);
                        }
                    }
                    // P of these 32 keys as 16 fp16 pairs, over S columns already read
                    tc::st16(sb + cc * 16, w);
                }
                {
                    float a0, a1, b0, b1;
                    unpack_f32x2(ls2[0], a0, a1);
                    unpack_f32x2(ls2[1], b0, b1);
                    l_run += (a0 + b0) + (a1 + b1);
                }
                tc::wait_st();
                if (__any_sync(0xffffffffu, resc && t > 0)) {
                    // O holds the job's tiles < t, complete (S of tile t was committed
                    // after their products): scale this warp's half of the columns
#pragma unroll 1
                    for (int cc = 0; cc < D / 64; ++cc) {
                        uint32_t r[32];
                        tc::ld32(ob + cc * 32, r);
                        tc::wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
                        tc::st32(ob + cc * 32, r);
                    }
                    tc::wait_st();
                }
                // one arrival per warp, once every lane's stores are done
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(bars.p_full, x));
                if (t == 0 && pend) {
                    // the previous job's O (complete: this tile's S was committed after
                    // its last P V) is read, then released to this job's first P V;
                    // its rows are written while the tensor pipe works
                    uint32_t hv[4 * NCH];
                    epi_read(hv);
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(bars.o_free, x));
                    epi_store(hv);
                }
            }
            pend = true;
            pend_l = l_run;
            pend_out = qi < u.ql ? reinterpret_cast<unsigned long long>(
                                       p.out + ((size_t)(u.q_beg + qi) * H + u.h) * D + half * (D / 2))
                                 : 0ull;
            ++job;
        }
        // the last job's output, once its last P V is done
        if (pend) {
            ok = ok && warp_all(mbar_wait_bounded(bar(bars.o_full, x), (job - 1) & 1, p.status, true));
            bars.red_l[x][half][row] = pend_l;
            if (group_all(meet, 256, ok)) {
                uint32_t hv[4 * NCH];
                epi_read(hv);
                epi_store(hv);
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

template <int D, bool KN>
cudaError_t set_prefill_smem_once() {
    static std::once_flag once[64];
    static cudaError_t err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        err[dev] = cudaFuncSetAttribute(paged_prefill_tc<D, KN>,
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

// The device address of the unit counters, per device, looked up once.
UnitCounter *unit_counters_of_current_device() {
    static std::once_flag once[64];
    static UnitCounter *ptr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::call_once(once[dev], [&] {
        void *a = nullptr;
        ptr[dev] = cudaGetSymbolAddress(&a, g_unit_ctr) == cudaSuccess
                       ? static_cast<UnitCounter *>(a) : nullptr;
    });
    return ptr[dev];
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

template <int D, bool KN>
int launch_d(PrefillParams p, int n_seqs, const pa_pool_desc *d, const void *k_new,
             const void *v_new, cudaStream_t st) {
    cudaError_t e = set_prefill_smem_once<D, KN>();
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
    if (KN) {   // the new rows, read like q; the cache, stored one block run and panel at a time
        if (rc == PA_OK) rc = encode_map(&maps.kn, k_new, 3, (uint64_t)p.q_rows, H, D, TBM);
        if (rc == PA_OK) rc = encode_map(&maps.vn, v_new, 3, (uint64_t)p.q_rows, H, D, TBM);
        if (rc == PA_OK) rc = encode_map(&maps.ks, p.k_cache, 2, cache_rows, H, D, d->block_size);
        if (rc == PA_OK) rc = encode_map(&maps.vs, p.v_cache, 2, cache_rows, H, D, d->block_size);
        for (int m = 0; rc == PA_OK && m < kVPartMaps; ++m)
            rc = encode_map(&maps.k_part[m], p.k_cache, 2, cache_rows, H, D, 8 >> m);
    } else {
        maps.kn = maps.vn = maps.ks = maps.vs = maps.q;   // unused
        for (int m = 0; m < kVPartMaps; ++m) maps.k_part[m] = maps.q;
    }
    if (rc != PA_OK) return rc;
    static std::atomic<uint32_t> calls{0};
    UnitCounter *ctrs = unit_counters_of_current_device();
    if (!ctrs) return fail(PA_ERR_CUDA, "prefill: cannot find the unit counters");
    p.units = ctrs + calls.fetch_add(1) % kUnitCounters;
    paged_prefill_tc<D, KN><<<sms, kTcThreads, TcLayout<D>::BYTES, st>>>(p, maps, n_seqs);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

}  // namespace

namespace {

int launch_prefill(void *out, const void *q, const void *k_new, const void *v_new,
                   const void *k_cache, const void *v_cache, const int32_t *block_tables,
                   const int32_t *ctx_lens, const int32_t *q_starts, int32_t n_seqs,
                   int32_t max_blocks, int32_t max_q_len, int32_t q_rows, float scale,
                   int32_t *status, const pa_pool_desc *d, void *stream) {
    const bool kn = k_new != nullptr;
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
    if (kn && (!v_new || (((uintptr_t)k_new | (uintptr_t)v_new) & 15)))
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_step_attention: k_new / v_new NULL or not 16-byte aligned");
    if (kn && d->block_size < 8)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_step_attention: block_size %d < 8", d->block_size);
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
    p.units = nullptr;   // set by the launcher
    p.bshift = bshift;
    p.qscale = scale * 1.4426950408889634f;
    p.status = status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (kn)
        return d->head_dim == 64 ? launch_d<64, true>(p, n_seqs, d, k_new, v_new, st)
                                 : launch_d<128, true>(p, n_seqs, d, k_new, v_new, st);
    return d->head_dim == 64 ? launch_d<64, false>(p, n_seqs, d, nullptr, nullptr, st)
                             : launch_d<128, false>(p, n_seqs, d, nullptr, nullptr, st);
}

}  // namespace

int launch_prefill_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, const int32_t *ctx_lens,
                             const int32_t *q_starts, int32_t n_seqs, int32_t max_blocks,
                             int32_t max_q_len, int32_t q_rows, float scale, int32_t *status,
                             const pa_pool_desc *d, void *stream) {
    return launch_prefill(out, q, nullptr, nullptr, k_cache, v_cache, block_tables, ctx_lens,
                          q_starts, n_seqs, max_blocks, max_q_len, q_rows, scale, status, d, stream);
}

int launch_prefill_step_attention(void *out, const void *q, const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache, const int32_t *block_tables,
                                  const int32_t *ctx_lens, const int32_t *q_starts, int32_t n_seqs,
                                  int32_t max_blocks, int32_t max_q_len, int32_t q_rows,
                                  float scale, int32_t *status, const pa_pool_desc *d, void *stream) {
    if (n_seqs > 0 && q_rows > 0 && !k_new)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_step_attention: NULL k_new");
    return launch_prefill(out, q, k_new, v_new, k_cache, v_cache, block_tables, ctx_lens, q_starts,
                          n_seqs, max_blocks, max_q_len, q_rows, scale, status, d, stream);
}

}  // namespace pagedkv
