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
// coalesced reads.  This design keeps "one warp owns whole blocks" and moves
// the bytes with the Blackwell bulk-copy engine.
//
// Work unit = (sequence, head, partition); a partition is partition_tokens
// tokens of one context (a context of at most one partition is one unit and
// needs no merge).  Two kernels compute units:
//
//  * paged_decode_persistent (the main path): one CTA per SM slot, each a
//    producer warp and C consumer warps.  CTAs take units from a global
//    ticket counter.  The producer decodes the ticket (per-CTA prefix sums
//    of partitions per sequence in shared memory), stages q, loads the
//    unit's block-table entries (coalesced) and streams every block of the
//    unit as two 1-D bulk copies (the (block, head) key rows and value rows
//    are each one contiguous B*D*2-byte run in the cache layout) into a
//    CTA-wide ring of STAGES shared-memory stages, across unit boundaries
//    without draining.  Stage i goes to consumer i % C; full / empty
//    mbarriers hand stages back and forth.  Each consumer keeps a running
//    softmax state per unit; at its last block of a unit it leaves a partial
//    (max, sum, output) in shared memory, and the last consumer to finish
//    the unit combines them and writes the output (one partition) or the
//    partition's partial to the workspace (split context).  CTA start-up
//    cost is paid once per CTA instead of once per unit.
//  * paged_decode_grid (fallback for batches too large for the per-CTA
//    prefix sums): grid = (partition, head, sequence), every warp owns every
//    WARPS-th block of its partition and runs its own bulk-copy ring.
//
// Per block (both kernels): lane (g, r) holds dims [8r, 8r+8) of token g of
// each pass (16-byte shared loads, conflict free); q.k uses the f16 x f16 ->
// f32 fused multiply-add (products exact, fp32 accumulation); the NP partial
// dot products per lane are reduced across the row's lanes with a
// reduce-scatter butterfly (NP-1+log2(TPR/NP) shuffles instead of
// NP*log2(TPR)); online softmax in base 2 (scale * log2 e applied to the
// reduced score) with fp32 running max / sum; p.v accumulates in fp32.
// Partials of a split context are merged by paged_merge_kernel:
// m = max m_p, l = sum 2^(m_p-m) l_p, o = sum 2^(m_p-m) acc_p / l.  (The
// pages do not cover the split or the merge; this is the standard
// log-sum-exp combination of the same sum.)
//
// Slots of the last block past ctx are neither copied (the bulk copy of a
// partial block moves only its valid rows) nor used.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pagedkv {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxPersistentSeqs = 2048;   // the per-CTA work plan lives in shared memory
constexpr size_t kCounterBytes = 256;      // workspace head: the unit ticket counter

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

struct DecodeParams {
    __half *out;
    const __half *q;
    const __half *k_cache;
    const __half *v_cache;
    const int32_t *block_tables;
    const int32_t *ctx_lens;
    float *ws_ml;      // [S][H][max_parts][2]  (max, sum)
    float *ws_acc;     // [S][H][max_parts][D]  unnormalised output
    int32_t *counter;  // unit tickets (persistent kernel), zeroed before each launch
    int32_t *status;
    int32_t n_seqs;
    int32_t num_heads;
    int32_t num_blocks;
    int32_t max_blocks;
    int32_t part_blocks;
    int32_t max_parts;
    float qscale;      // scale * log2(e)
    // optional slot write of the step's new token (persistent kernel): k_new /
    // v_new rows [n_seqs][H][D], slots[s] the slot of position ctx_lens[s] - 1
    // (NULL: no write)
    const __half *k_new;
    const __half *v_new;
    const int64_t *slots;
};

// ---------------------------------------------------------------- block math

// d += q . k over 8 halves (two 32-bit words hold four halves each), with
// f16 x f16 -> f32 fused multiply-adds: every product is exact in fp32.
__device__ __forceinline__ float dot8_f16(const uint4 &q, const uint4 &k, float d) {
    const uint32_t qa[4] = {q.x, q.y, q.z, q.w};
    const uint32_t ka[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
            "mov.b32 {a0, a1}, %1;\n\t"
            "mov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
            "fma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
            : "+f"(d)
            : "r"(qa[i]), "r"(ka[i]));
    return d;
}

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

// Running softmax state of one warp over the blocks it has seen of a unit.
template <int D, int B>
struct WarpAttn {
    using G = Geo<D, B>;
    int r, g, my_tok;
    uint4 qh;          // q halves, dims [8r, 8r+8)
    float m, lsum, acc[8];

    __device__ __forceinline__ void init_lane(int lane) {
        r = lane % G::TPR;
        g = lane / G::TPR;
        my_tok = token_index_of<G::NP, G::TPR>(r) * G::TPP + g;
    }
    __device__ __forceinline__ void reset() {
        m = -INFINITY;
        lsum = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = 0.f;
    }
    // One block: keys at kst, values at vst (row t at t * D * 2 bytes), nv valid rows.
    __device__ __forceinline__ void block(const uint8_t *kst, const uint8_t *vst, int nv,
                                          float qscale) {
        constexpr int TPR = G::TPR, TPP = G::TPP, NP = G::NP, DUP = G::DUP;
        float part_dot[NP];
#pragma unroll
        for (int ps = 0; ps < NP; ++ps) {
            const int t = ps * TPP + g;
            float d = 0.f;
            if (TPP * NP == B || t < B) {
                const uint4 u = *reinterpret_cast<const uint4 *>(kst + t * (D * 2) + r * 16);
                d = dot8_f16(qh, u, 0.f);
            }
            part_dot[ps] = d;
        }
        float sc = row_reduce_scatter<NP, TPR>(part_dot, r) * qscale;
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
    }
    // Totals over the warp: acc summed over token groups (lanes with g == 0
    // hold dims [8r, 8r+8)), lsum over all lanes.
    __device__ __forceinline__ void finalize() {
#pragma unroll
        for (int off = G::TPR; off < 32; off <<= 1)
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] += __shfl_xor_sync(kFull, acc[c], off);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) lsum += __shfl_xor_sync(kFull, lsum, off);
        lsum *= 1.0f / G::DUP;
    }
};

// Write one unit's combined result: the fp16 output when the context is one
// partition, else the partition's partial to the workspace.
template <int D>
__device__ __forceinline__ void store_unit(const DecodeParams &p, int s, int h, int part,
                                           int n_parts, int d, float M, float L, float o) {
    if (n_parts == 1) {
        p.out[((size_t)s * p.num_heads + h) * D + d] = __float2half(o / L);
    } else {
        const size_t idx = ((size_t)s * p.num_heads + h) * p.max_parts + part;
        if (d == 0) {
            p.ws_ml[2 * idx] = M;
            p.ws_ml[2 * idx + 1] = L;
        }
        p.ws_acc[idx * D + d] = o;
    }
}

// ------------------------------------------------------- persistent kernel

// A unit covers GH consecutive heads of one (sequence, partition): in the
// cache layout the key rows of those heads in one physical block are one
// contiguous GH * B * D * 2-byte run (same for values), so each block moves
// as two long bulk copies -- scattered short runs cost the memory system far
// more than their size.
constexpr int align16(int x) { return (x + 15) & ~15; }

template <int D, int B, int C, int SPC, int R, int GH>
struct PLayout {
    static constexpr int STAGES = C * SPC;
    static constexpr int CHUNK = Geo<D, B>::CHUNK;
    static constexpr int STAGE = 2 * GH * CHUNK;                     // K of GH heads, then V
    static_assert(STAGE % 128 == 0 || STAGE % 16 == 0, "bulk-copy destinations need 16 B");
    // every section starts on a 16-byte boundary (q rows are moved as uint4)
    static constexpr int FULL_OFF = align16(STAGES * STAGE);
    static constexpr int EMPTY_OFF = align16(FULL_OFF + STAGES * 8);
    static constexpr int DESC_OFF = align16(EMPTY_OFF + STAGES * 8);    // int2 per stage
    static constexpr int UNIT_OFF = align16(DESC_OFF + STAGES * 8);     // 16 int per unit slot
    static constexpr int Q_OFF = align16(UNIT_OFF + R * 64);            // GH * D halves per slot
    static constexpr int COMB_OFF = align16(Q_OFF + R * GH * D * 2);
    static constexpr int SEQ_OFF = align16(COMB_OFF + R * C * GH * (D + 2) * 4);  // plan, 2S+2 ints
    static_assert(Q_OFF % 16 == 0 && FULL_OFF % 8 == 0 && DESC_OFF % 8 == 0, "alignment");
    static constexpr int fixed_bytes() { return SEQ_OFF + 128; }     // +128: base alignment
    static size_t bytes(int n_seqs) { return fixed_bytes() + (size_t)(2 * n_seqs + 2) * 4; }
};

// unit slot fields (int32)
// U_DONE + g counts the groups that left their partial of head g; U_HDONE
// counts the heads combined.
enum { U_S = 0, U_H0, U_NH, U_PART, U_NPARTS, U_FIRSTC, U_NPARTIC, U_STATE, U_HDONE, U_DONE };
// stage descriptor flags
enum { F_FIRST = 1, F_LAST = 2, F_END = 4 };

template <int D, int B, int C, int SPC, int R, int GH, int PF>
__global__ void __launch_bounds__((C * GH + 1) * 32)
paged_decode_persistent(const DecodeParams p) {
    using G = Geo<D, B>;
    using L = PLayout<D, B, C, SPC, R, GH>;
    constexpr int STAGES = L::STAGES, STAGE = L::STAGE, CHUNK = G::CHUNK;
    constexpr int QVEC = GH * D / 8;                  // 16-byte pieces of a unit's q rows
    constexpr int QPL = (QVEC + 31) / 32;             // ... per producer lane
    // the step's new token is written here when its rows take one vector per
    // lane (else the launcher runs the slot write first)
    constexpr bool kWrite = QPL == 1;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::FULL_OFF);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L::EMPTY_OFF);
    int2 *sdesc = reinterpret_cast<int2 *>(smem + L::DESC_OFF);
    int32_t *units = reinterpret_cast<int32_t *>(smem + L::UNIT_OFF);
    __half *qs = reinterpret_cast<__half *>(smem + L::Q_OFF);
    float *comb = reinterpret_cast<float *>(smem + L::COMB_OFF);
    // Work plan (same in every CTA, so a ticket names the same unit everywhere):
    //  fullpre[s]  full partitions (every partition but a context's last one)
    //              of the sequences before s; fullpre[S] = F;
    //  order[r]    the r-th last partition, (s | partition << 16), grouped by
    //              size class, largest first, sequence order within a class.
    // Tickets F*HG.. run through order[]: big units go first and the stream
    // ends with the smallest ones, which keeps the CTAs' finishing times close.
    int32_t *fullpre = reinterpret_cast<int32_t *>(smem + L::SEQ_OFF);
    int32_t *order = fullpre + p.n_seqs + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int S = p.n_seqs;
    const int H = p.num_heads;
    const int HG = (H + GH - 1) / GH;             // head groups

    // ---- set-up: partitions per sequence (prefix sums), barriers
    if (tid == 0) {
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(smem_addr(&full[st]), 1);
            mbar_init(smem_addr(&empty[st]), GH);   // every warp of the stage's group
        }
        fence_barrier_init();
    }
    for (int i = tid; i < R * 16; i += blockDim.x) units[i] = 0;
    __syncthreads();
    // A context of 0 is one unit (its output is zero); a context the table
    // row cannot hold is reported and gets no unit.
    const int PB = p.part_blocks;
    auto plan_of = [&](int c, int &n_parts, int &cls) {
        if (c > p.max_blocks * B) {
            n_parts = 0;
            cls = 0;
            return;
        }
        const int nblk = c <= 0 ? 0 : (c + B - 1) / B;
        n_parts = c <= 0 ? 1 : (nblk + PB - 1) / PB;
        const int last = nblk - (n_parts - 1) * PB;     // blocks of the last partition
        cls = 4 * last >= 3 * PB ? 0 : (2 * last >= PB ? 1 : (4 * last >= PB ? 2 :
              (8 * last >= PB ? 3 : 4)));
    };
    constexpr int NCLS = 5;
    if (warp == 0) {
        const int per = (S + 31) / 32;
        const int lo = min(S, lane * per), hi = min(S, lo + per);
        int nfull = 0, ncls[NCLS] = {0, 0, 0, 0, 0};
        for (int s = lo; s < hi; ++s) {
            const int c = p.ctx_lens[s];
            if (c > p.max_blocks * B && blockIdx.x == 0) report(p.status, PA_ERR_BAD_BLOCK);
            int np, cls;
            plan_of(c, np, cls);
            if (np > 0) {
                nfull += np - 1;
#pragma unroll
                for (int k = 0; k < NCLS; ++k) ncls[k] += cls == k;
            }
        }
        // exclusive scans over lanes: full partitions, and each class
        auto scan = [&](int v, int &total) {
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(kFull, incl, off);
                if (lane >= off) incl += y;
            }
            total = __shfl_sync(kFull, incl, 31);
            return incl - v;
        };
        int F;
        int frun = scan(nfull, F);
        int cbase[NCLS], start = 0;
#pragma unroll
        for (int k = 0; k < NCLS; ++k) {
            int tot;
            cbase[k] = start + scan(ncls[k], tot);
            start += tot;
        }
        for (int s = lo; s < hi; ++s) {
            int np, cls;
            plan_of(p.ctx_lens[s], np, cls);
            fullpre[s] = frun;
            if (np > 0) {
                frun += np - 1;
                int r = 0;
#pragma unroll
                for (int k = 0; k < NCLS; ++k)
                    if (cls == k) r = cbase[k]++;
                order[r] = s | ((np - 1) << 16);
            }
        }
        if (lane == 0) {
            fullpre[S] = F;
            order[S] = start;          // number of last partitions (scratch slot)
        }
    }
    __syncthreads();
    const int n_full = fullpre[S];
    const int n_units = (n_full + order[S]) * HG;

    if (warp == C * GH) {
        // ================================================ producer warp
        // Software-pipelined: while unit k's blocks are issued, the ticket of
        // unit k+2 and the q rows and first table entries of unit k+1 are in
        // flight, so no global-memory latency sits between two units.
        const uint64_t policy = l2_evict_first_policy();
        const size_t blk_stride = (size_t)H * B * D;
        int i_stage = 0;
        int k_unit = 0;
        bool ok = true;

        struct Pending {
            int ticket, s, h0, nh, part, ctx, n_parts, j0, nb, tbl;
            uint4 q[QPL];
            int64_t wslot;          // the new token's slot (-1: nothing to write)
            uint4 kw, vw;           // this lane's piece of its key and value rows
        };
        // Decode a ticket (shared memory only) and start the loads of its
        // context length, q rows and first 32 table entries (lane t: entry
        // j0 + t, padding included).  None of these loads is waited on until
        // the unit becomes current, one unit later.
        auto prepare = [&](int ticket) {
            Pending u;
            u.ticket = ticket;
            u.s = u.h0 = u.nh = u.part = u.ctx = u.n_parts = u.j0 = u.nb = 0;
            u.tbl = -1;
            u.wslot = -1;
#pragma unroll
            for (int k = 0; k < QPL; ++k) u.q[k] = make_uint4(0, 0, 0, 0);
            u.kw = u.vw = make_uint4(0, 0, 0, 0);
            if (ticket >= n_units) return u;
            const int gp = ticket / HG;
            const int hg = ticket - gp * HG;
            u.h0 = hg * GH;
            u.nh = min(GH, H - u.h0);
            int lo;
            if (gp < n_full) {   // a full partition: last sequence s with fullpre[s] <= gp
                lo = 0;
                int hi = S - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (fullpre[mid] <= gp) lo = mid; else hi = mid - 1;
                }
                u.part = gp - fullpre[lo];
                u.n_parts = 2;       // more than one partition: the unit leaves a partial
            } else {             // a context's last partition
                const int e = order[gp - n_full];
                lo = e & 0xffff;
                u.part = e >> 16;
                u.n_parts = u.part + 1;
            }
            u.s = lo;
            u.j0 = u.part * p.part_blocks;
            u.ctx = p.ctx_lens[lo];
            if (u.j0 + lane < p.max_blocks)
                u.tbl = p.block_tables[(size_t)lo * p.max_blocks + u.j0 + lane];
            const uint4 *qsrc = reinterpret_cast<const uint4 *>(p.q + ((size_t)lo * H + u.h0) * D);
#pragma unroll
            for (int k = 0; k < QPL; ++k)
                if (lane + 32 * k < u.nh * (D / 8)) u.q[k] = qsrc[lane + 32 * k];
            if (kWrite && p.slots && gp >= n_full) {
                // a context's last partition holds the step's new token: this
                // unit writes its heads' key and value rows (loaded now, stored
                // before the copy of the block that holds them)
                u.wslot = p.slots[lo];
                const size_t row = ((size_t)lo * H + u.h0) * (D / 8) + lane;
                if (lane < u.nh * (D / 8)) {
                    u.kw = reinterpret_cast<const uint4 *>(p.k_new)[row];
                    u.vw = reinterpret_cast<const uint4 *>(p.v_new)[row];
                }
            }
            return u;
        };
        // blocks of the unit in its partition (needs the context length)
        auto blocks_of = [&](const Pending &u) {
            if (u.ticket >= n_units || u.ctx <= 0) return 0;
            return min(p.part_blocks, (u.ctx + B - 1) / B - u.j0);
        };

        // L2 prefetch runs PF blocks ahead of the shared-memory copies along
        // the stream of blocks (into the next unit when the current one ends),
        // so the number of bytes DRAM is working on is not bounded by the
        // stages that fit in shared memory.  pf_cur / pf_nxt: blocks of the
        // current / next unit already prefetched.
        auto prefetch = [&](const Pending &u, int b, int phys) {
            if (phys >= 0 && phys < p.num_blocks) {
                const size_t off = (size_t)phys * blk_stride + (size_t)u.h0 * B * D;
                prefetch_l2(p.k_cache + off, (uint32_t)u.nh * CHUNK);
                prefetch_l2(p.v_cache + off, (uint32_t)u.nh * CHUNK);
            }
        };
        int pf_cur = 0, pf_nxt = 0;

        int t_next = 0;
        if (lane == 0) t_next = atomicAdd(p.counter, 1);
        Pending cur = prepare(__shfl_sync(kFull, t_next, 0));
        if (lane == 0) t_next = atomicAdd(p.counter, 1);
        while (ok && cur.ticket < n_units) {
            cur.nb = blocks_of(cur);
            const int tn = __shfl_sync(kFull, t_next, 0);
            if (lane == 0) t_next = atomicAdd(p.counter, 1);
            Pending nxt = prepare(tn);
            if (PF > 0 && cur.ctx > 0) {
                // the first PF blocks of this unit, one lane per block
                const int upto = min(min(PF, cur.nb), 32);
                if (lane >= pf_cur && lane < upto) prefetch(cur, lane, cur.tbl);
                pf_cur = max(pf_cur, upto);
            }
            if (cur.ctx <= 0) {   // empty context (a negative length counts as 0): o = 0
                __half *o = p.out + ((size_t)cur.s * H + cur.h0) * D;
                for (int d = lane; d < cur.nh * D; d += 32) o[d] = __float2half(0.f);
            } else {
                const int slot = k_unit % R;
                int32_t *u = units + slot * 16;
                // wait until the slot's previous unit has been combined
                if (lane == 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (*(volatile int32_t *)&u[U_STATE] != 0) {
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            report(p.status, PA_ERR_TIMEOUT);
                            ok = false;
                            break;
                        }
                    }
                }
                ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                __threadfence_block();
                // stage q and the unit's description
#pragma unroll
                for (int k = 0; k < QPL; ++k)
                    if (lane + 32 * k < QVEC)
                        reinterpret_cast<uint4 *>(qs + slot * GH * D)[lane + 32 * k] = cur.q[k];
                if (lane == 0) {
                    u[U_S] = cur.s;
                    u[U_H0] = cur.h0;
                    u[U_NH] = cur.nh;
                    u[U_PART] = cur.part;
                    u[U_NPARTS] = cur.n_parts;
                    u[U_FIRSTC] = i_stage % C;
                    u[U_NPARTIC] = min(C, cur.nb);
                    u[U_HDONE] = 0;
#pragma unroll
                    for (int g = 0; g < GH; ++g) u[U_DONE + g] = 0;
                    u[U_STATE] = 1;
                }
                __syncwarp();
                __threadfence_block();
                const int32_t *trow = p.block_tables + (size_t)cur.s * p.max_blocks + cur.j0;
                const __half *kbase = p.k_cache + (size_t)cur.h0 * B * D;
                const __half *vbase = p.v_cache + (size_t)cur.h0 * B * D;
                int tbl = cur.tbl;
                for (int b = 0; b < cur.nb; ++b) {
                    if (b > 0 && (b & 31) == 0) tbl = b + lane < cur.nb ? trow[b + lane] : -1;
                    const int phys = __shfl_sync(kFull, tbl, b & 31);
                    if (PF > 0) {
                        const int tgt = b + PF;
                        const int pc = __shfl_sync(kFull, cur.tbl, tgt & 31);
                        const int tn2 = tgt - cur.nb;
                        const int pn = __shfl_sync(kFull, nxt.tbl, (tn2 < 0 ? 0 : tn2) & 31);
                        const int nxt_nb = tn2 >= 0 ? blocks_of(nxt) : 0;
                        if (lane == 0) {
                            if (tgt < cur.nb) {
                                if (tgt >= pf_cur && tgt < 32) prefetch(cur, tgt, pc);
                            } else if (tn2 < nxt_nb && tn2 >= pf_nxt && tn2 < 32) {
                                prefetch(nxt, tn2, pn);
                            }
                        }
                        if (tgt < cur.nb) pf_cur = max(pf_cur, tgt + 1);
                        else if (tn2 < nxt_nb) pf_nxt = max(pf_nxt, tn2 + 1);
                    }
                    if (kWrite && b == cur.nb - 1 && cur.wslot >= 0) {
                        // the new token: its slot must be position ctx - 1, in this
                        // block; its rows are stored, then fenced against the bulk
                        // copy below that reads them
                        const int64_t blk = cur.wslot / B;
                        const int off = (int)(cur.wslot % B);
                        if (blk == phys && off == (cur.ctx - 1) % B && phys >= 0 && phys < p.num_blocks) {
                            __half *kd = const_cast<__half *>(p.k_cache) + ((size_t)phys * H + cur.h0) * B * D + (size_t)off * D;
                            __half *vd = const_cast<__half *>(p.v_cache) + ((size_t)phys * H + cur.h0) * B * D + (size_t)off * D;
                            if (lane < cur.nh * (D / 8)) {
                                const int g = lane / (D / 8), c8 = lane % (D / 8);
                                reinterpret_cast<uint4 *>(kd + (size_t)g * B * D)[c8] = cur.kw;
                                reinterpret_cast<uint4 *>(vd + (size_t)g * B * D)[c8] = cur.vw;
                            }
                            fence_proxy_async_global();
                        } else if (lane == 0) {
                            report(p.status, PA_ERR_INVALID_ARG);
                        }
                        __syncwarp();
                    }
                    const int st = i_stage % STAGES;
                    const int use = i_stage / STAGES;
                    if (lane == 0) {
                        if (use > 0 && !mbar_wait_bounded(smem_addr(&empty[st]),
                                                          (uint32_t)(use - 1) & 1u, p.status, true)) {
                            report(p.status, PA_ERR_TIMEOUT);
                            ok = false;
                        } else {
                            const int nv = min(B, cur.ctx - (cur.j0 + b) * B);
                            const int flags =
                                (b < C ? F_FIRST : 0) | (b >= cur.nb - C ? F_LAST : 0);
                            sdesc[st] = make_int2(slot | (flags << 16), nv);
                            const uint32_t fb = smem_addr(&full[st]);
                            const uint32_t dk = smem_addr(smem + st * STAGE);
                            const uint32_t dv = dk + GH * CHUNK;
                            if (phys >= 0 && phys < p.num_blocks) {
                                const __half *sk = kbase + (size_t)phys * blk_stride;
                                const __half *sv = vbase + (size_t)phys * blk_stride;
                                if (nv == B) {   // the heads' full rows: one run each
                                    const uint32_t bytes = (uint32_t)cur.nh * CHUNK;
                                    mbar_arrive_expect_tx(fb, 2 * bytes);
                                    bulk_g2s(dk, sk, bytes, fb, policy);
                                    bulk_g2s(dv, sv, bytes, fb, policy);
                                } else {         // partial last block: valid rows per head
                                    const uint32_t bytes = (uint32_t)nv * D * 2;
                                    mbar_arrive_expect_tx(fb, 2 * bytes * cur.nh);
                                    for (int g = 0; g < cur.nh; ++g) {
                                        bulk_g2s(dk + g * CHUNK, sk + (size_t)g * B * D, bytes, fb,
                                                 policy);
                                        bulk_g2s(dv + g * CHUNK, sv + (size_t)g * B * D, bytes, fb,
                                                 policy);
                                    }
                                }
                            } else {
                                report(p.status, PA_ERR_BAD_BLOCK);
                                mbar_arrive(fb);
                            }
                        }
                    }
                    ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    ++i_stage;
                }
                ++k_unit;
            }
            cur = nxt;
            pf_cur = pf_nxt;
            pf_nxt = 0;
        }
        // end of stream: one END stage per consumer
        for (int c = 0; ok && c < C; ++c) {
            const int st = i_stage % STAGES;
            const int use = i_stage / STAGES;
            if (lane == 0) {
                if (use > 0 && !mbar_wait_bounded(smem_addr(&empty[st]), (uint32_t)(use - 1) & 1u,
                                                  p.status, true)) {
                    report(p.status, PA_ERR_TIMEOUT);
                    ok = false;
                } else {
                    sdesc[st] = make_int2(F_END << 16, 0);
                    mbar_arrive(smem_addr(&full[st]));
                }
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            ++i_stage;
        }
        if (!ok && lane == 0) {
            // let every issued copy land before the CTA can exit
            for (int k = max(0, i_stage - STAGES); k < i_stage; ++k)
                mbar_wait_bounded(smem_addr(&full[k % STAGES]), (uint32_t)(k / STAGES) & 1u,
                                  p.status, false);
        }
        return;
    }

    // ==================================================== consumer warps
    // Warp (c, g): group c takes every C-th stage, member g its head g.
    const int c = warp / GH;
    const int g = warp - c * GH;
    WarpAttn<D, B> wa;
    wa.init_lane(lane);
    wa.reset();
    int nh = 0;
    for (int i = c;; i += C) {
        const int st = i % STAGES;
        if (!mbar_wait_bounded(smem_addr(&full[st]), (uint32_t)(i / STAGES) & 1u, p.status, true)) {
            report(p.status, PA_ERR_TIMEOUT);
            return;
        }
        const int2 dsc = sdesc[st];
        const int flags = dsc.x >> 16;
        if (flags & F_END) return;
        const int slot = dsc.x & 0xffff;
        int32_t *u = units + slot * 16;
        if (flags & F_FIRST) {
            nh = u[U_NH];
            wa.reset();
            if (g < nh) wa.qh = reinterpret_cast<const uint4 *>(qs + (slot * GH + g) * D)[wa.r];
        }
        const uint8_t *kst = smem + st * STAGE;
        if (g < nh) wa.block(kst + g * CHUNK, kst + (GH + g) * CHUNK, dsc.y, p.qscale);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
        if ((flags & F_LAST) && g < nh) {
            wa.finalize();
            float *cw = comb + ((slot * C + c) * GH + g) * (D + 2);
            if (wa.g == 0) {
#pragma unroll
                for (int k = 0; k < 8; ++k) cw[wa.r * 8 + k] = wa.acc[k];
            }
            if (lane == 0) {
                cw[D] = wa.m;
                cw[D + 1] = wa.lsum;
            }
            __threadfence_block();
            __syncwarp();
            int last = 0;
            if (lane == 0) last = atomicAdd(&u[U_DONE + g], 1) == u[U_NPARTIC] - 1;
            last = __shfl_sync(kFull, last, 0);
            if (last) {   // every group has left its partial of head g: combine
                __threadfence_block();
                const int first_c = u[U_FIRSTC], np = u[U_NPARTIC];
                float M = -INFINITY;
                for (int t = 0; t < np; ++t)
                    M = fmaxf(M, comb[(((slot * C + (first_c + t) % C) * GH) + g) * (D + 2) + D]);
                float Lt = 0.f;
                for (int t = 0; t < np; ++t) {
                    const float *pw = comb + (((slot * C + (first_c + t) % C) * GH) + g) * (D + 2);
                    Lt = fmaf(exp2f(pw[D] - M), pw[D + 1], Lt);
                }
                const int s = u[U_S], h = u[U_H0] + g, part = u[U_PART], n_parts = u[U_NPARTS];
                for (int d = lane; d < D; d += 32) {
                    float o = 0.f;
                    for (int t = 0; t < np; ++t) {
                        const float *pw =
                            comb + (((slot * C + (first_c + t) % C) * GH) + g) * (D + 2);
                        o = fmaf(exp2f(pw[D] - M), pw[d], o);
                    }
                    store_unit<D>(p, s, h, part, n_parts, d, M, Lt, o);
                }
                __syncwarp();
                __threadfence_block();
                int free_it = 0;
                if (lane == 0) free_it = atomicAdd(&u[U_HDONE], 1) == nh - 1;
                free_it = __shfl_sync(kFull, free_it, 0);
                if (free_it && lane == 0) atomicExch(&u[U_STATE], 0);
            }
        }
    }
}

// -------------------------------------------------------- grid kernel

template <int D, int B>
struct GridCfg {
    static constexpr int STAGE = Geo<D, B>::STAGE;
    static constexpr int WARPS = (8 * STAGE > 200 * 1024) ? 2 : 4;
    static constexpr int S0 = (96 * 1024) / (WARPS * STAGE);
    static constexpr int STAGES = S0 < 2 ? 2 : (S0 > 8 ? 8 : S0);
    static constexpr int STAGE_BYTES = WARPS * STAGES * STAGE;
    static constexpr int BAR_OFF = STAGE_BYTES;
    static constexpr int COMB_OFF = BAR_OFF + WARPS * STAGES * 8;
    static constexpr int TOTAL = COMB_OFF + WARPS * (D + 2) * 4 + 128;
};

template <int D, int B>
__global__ void __launch_bounds__(GridCfg<D, B>::WARPS * 32)
paged_decode_grid(const DecodeParams p) {
    using G = Geo<D, B>;
    using L = GridCfg<D, B>;
    constexpr int WARPS = L::WARPS, STAGES = L::STAGES;
    constexpr int CHUNK = G::CHUNK, STAGE = G::STAGE;

    const int part = blockIdx.x;
    const int h = blockIdx.y;
    const int s = blockIdx.z;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int H = p.num_heads;

    const int ctx = p.ctx_lens[s];
    if (ctx <= 0) {   // empty context (a negative length counts as 0): o = 0
        if (part == 0)
            for (int i = tid; i < D; i += WARPS * 32)
                p.out[((size_t)s * H + h) * D + i] = __float2half(0.f);
        return;
    }
    if (ctx > p.max_blocks * B) {
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

    WarpAttn<D, B> wa;
    wa.init_lane(lane);
    wa.reset();
    wa.qh = *reinterpret_cast<const uint4 *>(p.q + ((size_t)s * H + h) * D + wa.r * 8);

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
        const uint8_t *kst = stages + st * STAGE;
        wa.block(kst, kst + CHUNK, min(B, ctx - j * B), p.qscale);
        __syncwarp();
        if (i + STAGES < n_w) issue(i + STAGES);
    }
    wa.finalize();

    float *cw = comb + warp * (D + 2);
    if (wa.g == 0) {
#pragma unroll
        for (int c = 0; c < 8; ++c) cw[wa.r * 8 + c] = wa.acc[c];
    }
    if (lane == 0) {
        cw[D] = wa.m;
        cw[D + 1] = wa.lsum;
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
    for (int i = tid; i < D; i += WARPS * 32) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) o = fmaf(wgt[w], comb[w * (D + 2) + i], o);
        store_unit<D>(p, s, h, part, n_parts, i, M, Lt, o);
    }
}

// One warp per (sequence, head) whose context spans more than one partition.
// All loads of a pass are issued before any is used: lane q holds partition
// q's (max, sum), every lane its D/32 output dims of up to 8 partitions.
template <int D>
__global__ void __launch_bounds__(128) paged_merge_kernel(const DecodeParams p, int part_tokens) {
    constexpr int DL = D >= 32 ? D / 32 : 1;   // dims per lane
    constexpr int QB = 8;                      // partitions per pass
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
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml) + base;
    float M = -INFINITY;
    for (int q = lane; q < n_parts; q += 32) M = fmaxf(M, ml[q].x);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    float o[DL];
#pragma unroll
    for (int k = 0; k < DL; ++k) o[k] = 0.f;
    float Lt = 0.f;
    for (int q0 = 0; q0 < n_parts; q0 += QB) {
        float a[QB][DL];
#pragma unroll
        for (int q = 0; q < QB; ++q)
#pragma unroll
            for (int k = 0; k < DL; ++k) {
                const int d = lane + 32 * k;
                a[q][k] = (q0 + q < n_parts && d < D) ? p.ws_acc[(base + q0 + q) * D + d] : 0.f;
            }
        const float2 mine = q0 + lane < n_parts && lane < QB ? ml[q0 + lane] : make_float2(-INFINITY, 0.f);
        const float w = exp2f(mine.x - M);
        float lw = w * mine.y;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) lw += __shfl_xor_sync(kFull, lw, off);
        Lt += lw;
#pragma unroll
        for (int q = 0; q < QB; ++q) {
            const float wq = __shfl_sync(kFull, w, q);
#pragma unroll
            for (int k = 0; k < DL; ++k) o[k] = fmaf(wq, a[q][k], o[k]);
        }
    }
    const float inv = 1.0f / Lt;
    __half *out_row = p.out + ((size_t)s * H + h) * D;
#pragma unroll
    for (int k = 0; k < DL; ++k) {
        const int d = lane + 32 * k;
        if (d < D) out_row[d] = __float2half(o[k] * inv);
    }
}

// ------------------------------------------------------------- launching

// Raise a kernel's dynamic shared-memory limit once per device.  Tag makes
// the once-flags distinct per kernel instantiation (they share one type).
template <typename Tag, typename K>
cudaError_t set_smem_once(K kern, int bytes) {
    static std::once_flag once[64];
    static cudaError_t err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    });
    return err[dev];
}

int sm_count() {
    static std::once_flag once[64];
    static int n[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::call_once(once[dev], [&] {
        n[dev] = 148;
        cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
    });
    return n[dev];
}

template <int D, int B>
struct PersistCfg {
    static constexpr int CHUNK = Geo<D, B>::CHUNK;
    // heads per unit: at least 8 KB of contiguous key (and value) rows per copy
    static constexpr int GH0 = 8192 / CHUNK;
    static constexpr int GH = GH0 < 1 ? 1 : (GH0 > 4 ? 4 : GH0);
    static constexpr int STAGE = 2 * GH * CHUNK;
    static constexpr int C = STAGE <= 8192 ? 4 : (STAGE <= 16384 ? 3 : 2);   // consumer warps
    static constexpr int SPC0 = (96 * 1024) / (C * STAGE);
    static constexpr int SPC = SPC0 < 2 ? 2 : (SPC0 > 8 ? 8 : SPC0);         // stages per consumer
    static constexpr int R = 3;       // unit slots (open units per CTA)
    static constexpr int PF = 0;      // L2 prefetch distance, blocks (0: none)
};

template <int D, int B, bool Persistent>
struct KernelTag {};

template <int D, int B>
int launch_db(const DecodeParams &prm_in, int part_tokens, const pa_pool_desc *d,
              cudaStream_t stream) {
    DecodeParams prm = prm_in;
    cudaError_t e;
    using PC = PersistCfg<D, B>;
    using L = PLayout<D, B, PC::C, PC::SPC, PC::R, PC::GH>;
    auto pkern = paged_decode_persistent<D, B, PC::C, PC::SPC, PC::R, PC::GH, PC::PF>;
    constexpr int threads = (PC::C * PC::GH + 1) * 32;
    // The persistent kernel's shared memory grows with the batch (its prefix
    // sums); it is used while that keeps the occupancy of a one-sequence
    // batch, else the grid kernel runs.  Found once per device.
    static std::once_flag once[64];
    static int max_seqs[64], per_sm_full[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return fail(PA_ERR_CUDA, "pa_decode_attention: cudaGetDevice failed");
    std::call_once(once[dev], [&] {
        max_seqs[dev] = 0;
        per_sm_full[dev] = 0;
        if (set_smem_once<KernelTag<D, B, true>>(pkern, (int)L::bytes(kMaxPersistentSeqs)) !=
            cudaSuccess)
            return;
        int base = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&base, pkern, threads,
                                                          (int)L::bytes(1)) != cudaSuccess ||
            base < 1)
            return;
        int lo = 1, hi = kMaxPersistentSeqs;   // largest batch with the same occupancy
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            int n = 0;
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pkern, threads, (int)L::bytes(mid));
            if (n >= base) lo = mid; else hi = mid - 1;
        }
        max_seqs[dev] = lo;
        per_sm_full[dev] = base;
    });
    // the persistent kernel writes the step's new token when a unit's rows
    // take one vector per producer lane; otherwise the slot write runs first
    constexpr bool kernel_writes = (PC::GH * D / 8 + 31) / 32 == 1;
    if (prm.slots && !(kernel_writes && prm.n_seqs <= max_seqs[dev])) {
        const int rc = launch_write_kv(prm.k_new, prm.v_new, prm.slots, prm.n_seqs,
                                       const_cast<__half *>(prm.k_cache),
                                       const_cast<__half *>(prm.v_cache), d, prm.status, stream);
        if (rc != PA_OK) return rc;
        prm.slots = nullptr;
    }
    if (prm.n_seqs <= max_seqs[dev]) {
        auto kern = pkern;
        const int use_smem = (int)L::bytes(prm.n_seqs);
        const int per_sm = per_sm_full[dev];
        const int64_t max_units =
            (int64_t)prm.n_seqs * ((prm.num_heads + PC::GH - 1) / PC::GH) * prm.max_parts;
        const int grid = (int)std::min<int64_t>((int64_t)sm_count() * per_sm, max_units);
        e = cudaMemsetAsync(prm.counter, 0, sizeof(int32_t), stream);
        if (e != cudaSuccess)
            return fail(PA_ERR_CUDA, "pa_decode_attention: memset: %s", cudaGetErrorString(e));
        kern<<<grid, threads, use_smem, stream>>>(prm);
    } else {
        using L = GridCfg<D, B>;
        auto kern = paged_decode_grid<D, B>;
        e = set_smem_once<KernelTag<D, B, false>>(kern, L::TOTAL);
        if (e != cudaSuccess)
            return fail(PA_ERR_CUDA, "pa_decode_attention: cudaFuncSetAttribute: %s",
                        cudaGetErrorString(e));
        dim3 grid(prm.max_parts, prm.num_heads, prm.n_seqs);
        kern<<<grid, L::WARPS * 32, L::TOTAL, stream>>>(prm);
    }
    e = cudaGetLastError();
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

template <int D>
int launch_d(int B, const DecodeParams &prm, int part_tokens, const pa_pool_desc *d,
             cudaStream_t stream) {
    switch (B) {
        case 4: return launch_db<D, 4>(prm, part_tokens, d, stream);
        case 8: return launch_db<D, 8>(prm, part_tokens, d, stream);
        case 16: return launch_db<D, 16>(prm, part_tokens, d, stream);
        case 32: return launch_db<D, 32>(prm, part_tokens, d, stream);
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
    if (n_seqs == 0) return 0;
    const int part_blocks = partition_tokens_of(d) / d->block_size;
    const int mp = max_parts_of(max_blocks, part_blocks);
    if (mp <= 1) return kCounterBytes;
    const size_t rows = (size_t)n_seqs * d->num_heads * mp;
    return kCounterBytes + align256(rows * 2 * sizeof(float)) +
           align256(rows * d->head_dim * sizeof(float));
}

namespace {

int launch_decode(void *out, const void *q, const void *k_new, const void *v_new,
                  const int64_t *slots, const void *k_cache, const void *v_cache,
                  const int32_t *block_tables, const int32_t *ctx_lens, int32_t n_seqs,
                  int32_t max_blocks, float scale, void *workspace, size_t workspace_bytes,
                  int32_t *status, const pa_pool_desc *d, void *stream) {
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
    if (slots && (!k_new || !v_new || mis16(k_new) || mis16(v_new) ||
                  (reinterpret_cast<uintptr_t>(slots) & 7)))
        return fail(PA_ERR_INVALID_ARG,
                    "pa_decode_step_attention: k_new / v_new NULL or not 16-byte aligned, or "
                    "slot_mapping not 8-byte aligned");
    const int part_tokens = partition_tokens_of(d);
    const int part_blocks = part_tokens / d->block_size;
    const int mp = max_parts_of(max_blocks, part_blocks);
    const size_t need = decode_workspace_bytes(n_seqs, max_blocks, d);
    if (!workspace || workspace_bytes < need)
        return fail(PA_ERR_INVALID_ARG,
                    "pa_decode_attention: workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (reinterpret_cast<uintptr_t>(workspace) & 255)
        return fail(PA_ERR_INVALID_ARG, "pa_decode_attention: workspace must be 256-byte aligned");
    DecodeParams prm{};
    prm.out = static_cast<__half *>(out);
    prm.q = static_cast<const __half *>(q);
    prm.k_cache = static_cast<const __half *>(k_cache);
    prm.v_cache = static_cast<const __half *>(v_cache);
    prm.block_tables = block_tables;
    prm.ctx_lens = ctx_lens;
    char *ws = static_cast<char *>(workspace);
    prm.counter = reinterpret_cast<int32_t *>(ws);
    const size_t rows = (size_t)n_seqs * d->num_heads * mp;
    prm.ws_ml = mp > 1 ? reinterpret_cast<float *>(ws + kCounterBytes) : nullptr;
    prm.ws_acc = mp > 1 ? reinterpret_cast<float *>(ws + kCounterBytes +
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
    prm.k_new = static_cast<const __half *>(k_new);
    prm.v_new = static_cast<const __half *>(v_new);
    prm.slots = slots;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (d->head_dim) {
        case 8: return launch_d<8>(d->block_size, prm, part_tokens, d, st);
        case 16: return launch_d<16>(d->block_size, prm, part_tokens, d, st);
        case 32: return launch_d<32>(d->block_size, prm, part_tokens, d, st);
        case 64: return launch_d<64>(d->block_size, prm, part_tokens, d, st);
        case 128: return launch_d<128>(d->block_size, prm, part_tokens, d, st);
        case 256: return launch_d<256>(d->block_size, prm, part_tokens, d, st);
    }
    return fail(PA_ERR_INVALID_ARG, "pa_decode_attention: unsupported head_dim %d", d->head_dim);
}

}  // namespace

int launch_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *ctx_lens, int32_t n_seqs,
                            int32_t max_blocks, float scale, void *workspace,
                            size_t workspace_bytes, int32_t *status, const pa_pool_desc *d,
                            void *stream) {
    return launch_decode(out, q, nullptr, nullptr, nullptr, k_cache, v_cache, block_tables,
                         ctx_lens, n_seqs, max_blocks, scale, workspace, workspace_bytes, status,
                         d, stream);
}

int launch_decode_step_attention(void *out, const void *q, const void *k_new, const void *v_new,
                                 const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                 const int32_t *block_tables, const int32_t *ctx_lens,
                                 int32_t n_seqs, int32_t max_blocks, float scale, void *workspace,
                                 size_t workspace_bytes, int32_t *status, const pa_pool_desc *d,
                                 void *stream) {
    if (n_seqs > 0 && !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "pa_decode_step_attention: NULL slot_mapping");
    return launch_decode(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                         ctx_lens, n_seqs, max_blocks, scale, workspace, workspace_bytes, status,
                         d, stream);
}

}  // namespace pagedkv

// ------------------------------------------------ workspace-free entry point
//
// For callers that cannot allocate device memory at call time (a runtime that
// owns all device memory, a plugin host that forbids cudaMalloc once serving
// has started): the workspace of pa_decode_attention comes from this fixed
// array instead.  Every device that loads the library holds it until exit.
// Host code cannot use the array's name as an address (on the host it is only
// a stand-in for the symbol): the device address is looked up with
// cudaGetSymbolAddress, with that device current, on the first call there
// that gets past the argument checks.  A failed lookup is not remembered (the
// next call tries again), and a first call made while its stream is being
// captured is refused before the lookup.  All calls share the array;
// concurrent calls race.
namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];   // guarded by g_noalloc_mu; null until a lookup succeeds

// The scratch's device address on the current device (looked up once).
int noalloc_scratch(cudaStream_t stream, void **out) {
    using namespace pagedkv;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "pa_decode_attention_noalloc: cudaGetDevice: %s",
                    cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(PA_ERR_CUDA, "pa_decode_attention_noalloc: device %d is beyond the %d "
                    "devices this library tracks", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev]) {
        *out = g_noalloc_ptr[dev];
        return PA_OK;
    }
    // The lookup may load the module; it must not run inside a stream capture.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) {
        cudaGetLastError();   // not sticky: keep it out of later launch checks
        return fail(PA_ERR_CUDA, "pa_decode_attention_noalloc: cudaStreamIsCapturing: %s",
                    cudaGetErrorString(e));
    }
    if (cap != cudaStreamCaptureStatusNone)
        return fail(PA_ERR_INVALID_ARG, "pa_decode_attention_noalloc: the first call on device "
                    "%d was made while its stream is being captured; make one call before any "
                    "capture (it looks up the scratch address)", dev);
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
        cudaGetLastError();
        return fail(PA_ERR_CUDA, "pa_decode_attention_noalloc: cudaGetSymbolAddress: %s",
                    cudaGetErrorString(e));
    }
    g_noalloc_ptr[dev] = ptr;
    *out = ptr;
    return PA_OK;
}
}  // namespace

extern "C" int pa_decode_attention_noalloc(void *out, const void *q, const void *k_cache,
                                           const void *v_cache, const int32_t *block_tables,
                                           const int32_t *ctx_lens, int32_t n_seqs,
                                           int32_t max_blocks, float scale, int32_t *status,
                                           const pa_pool_desc *desc, void *stream) {
    using namespace pagedkv;
    // every argument error is reported before any CUDA call
    std::string why;
    if (!desc) return fail(PA_ERR_INVALID_ARG, "pa_decode_attention_noalloc: NULL desc");
    if (!device_geometry_ok(desc, &why))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_attention_noalloc: %s", why.c_str());
    if (n_seqs < 0 || n_seqs > 65535 || max_blocks < 0 || desc->num_heads > 65535)
        return fail(PA_ERR_INVALID_ARG,
                    "pa_decode_attention_noalloc: n_seqs=%d (<= 65535), max_blocks=%d, "
                    "num_heads=%d", n_seqs, max_blocks, desc->num_heads);
    if (n_seqs == 0) return PA_OK;
    const size_t need = decode_workspace_bytes(n_seqs, max_blocks, desc);
    if (need > PA_NOALLOC_SCRATCH_BYTES)
        return fail(PA_ERR_INVALID_ARG,
                    "pa_decode_attention_noalloc: the batch needs %zu bytes of scratch, the "
                    "fixed scratch holds %zu (use pa_decode_attention with a workspace)",
                    need, (size_t)PA_NOALLOC_SCRATCH_BYTES);
    if (!out || !q || !k_cache || !v_cache || !ctx_lens || (max_blocks > 0 && !block_tables))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_attention_noalloc: NULL pointer");
    if (((uintptr_t)out | (uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache) & 15)
        return fail(PA_ERR_INVALID_ARG,
                    "pa_decode_attention_noalloc: out/q/caches must be 16-byte aligned");
    if (!std::isfinite(scale))
        return fail(PA_ERR_INVALID_ARG, "pa_decode_attention_noalloc: scale is not finite");
    void *scratch = nullptr;
    const int rc = noalloc_scratch(static_cast<cudaStream_t>(stream), &scratch);
    if (rc != PA_OK) return rc;
    return launch_decode_attention(out, q, k_cache, v_cache, block_tables, ctx_lens, n_seqs,
                                   max_blocks, scale, scratch, (size_t)PA_NOALLOC_SCRATCH_BYTES,
                                   status, desc, stream);
}
