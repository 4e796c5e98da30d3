// Paged decode attention for sm_103a.
//
// Problem ("Basics of LLM Inference and vLLM Internals", s.2 and s.4; "The
// Memory Trick Behind Fast LLM Serving", "PagedAttention changes the shape of
// the problem"): one query token per sequence attends to every cached token of
// that sequence; token t lives in physical block block_tables[s][t / 16] at
// offset t % 16; the query heads of a GQA group share one KV head.
//
// Design (one GB300, HBM-bound):
//  * Work unit = (sequence, KV head, group of <= 8 query heads).  The cached
//    blocks of all units are laid end to end and cut into equal contiguous
//    ranges, one per warp, so every warp streams the same number of 4 KiB tiles
//    whatever the length mix.  A unit a single warp covers is written directly;
//    a unit cut by range boundaries leaves one partial (unnormalised output,
//    running max and sum) per warp, merged by a log-sum-exp combine kernel
//    chained behind by programmatic dependent launch, so no streaming warp ever
//    waits on another.
//  * Each warp owns a ring of stages in shared memory.  One lane issues bulk
//    tensor copies (TMA, 128-byte swizzle) of the K and V tiles of a physical
//    block straight from the block table; the ring keeps several tiles per warp
//    in flight.  Block-table entries are fetched 32 at a time by the warp.
//  * Per 16-key block the warp computes S^T = K . Q^T with keys as the MMA M
//    dimension (16 keys = one block) and the <= 8 query heads of the group as N,
//    so no MMA row is padding when G = 8.  After an online softmax, the
//    probabilities are transposed in registers (movmatrix) into the B operand of
//    O^T = V^T . P^T, whose accumulator columns are again the heads.
//  * FP8-E4M3 tiles are widened to fp16 exactly on the fly (cvt e4m3x2) and the
//    per-tensor scales are folded into the softmax scale and the final divide.
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

template <int Kind, int Stages = 3>
struct DecodeCfg {
    static constexpr bool kFp8 = Kind == kKindFp8;
    static constexpr int kTileBytes = kFp8 ? 2048 : 4096;   // one (block, head) tile
    static constexpr int kStageBytes = 2 * kTileBytes;      // K then V
    static constexpr int kStages = Stages;                   // per warp
    static constexpr int kTileArea = kDecodeWarps * kStages * kStageBytes;
    static constexpr int kBarBytes = kDecodeWarps * kStages * 8;
};

// Flattened-order cursor over (sequence, unit-in-sequence, block).
struct Cursor {
    int s;    // sequence
    int uh;   // KV head * head_groups + head group
    int j;    // logical block
    int nb;   // blocks of sequence s
};

__device__ __forceinline__ void cursor_advance(Cursor& c, const int* cum, int B, int UH) {
    if (++c.j == c.nb) {
        c.j = 0;
        if (++c.uh == UH) {
            c.uh = 0;
            do {
                ++c.s;
            } while (c.s < B && cum[c.s + 1] == cum[c.s]);
            if (c.s < B) c.nb = (cum[c.s + 1] - cum[c.s]) / UH;
        }
    }
}

// Worker (warp) whose range holds flattened index f, for T indices over W workers
// with range w = [floor(w T / W), floor((w + 1) T / W)).
__device__ __forceinline__ int worker_of(long long f, long long T, int W) {
    return static_cast<int>(((f + 1) * W - 1) / T);
}

// How the flattened order [0, T) is cut.  Ranges 0 .. W-1 are static, one per
// worker, over [0, Ts); ranges W .. W+P-1 are pieces of S blocks over [Ts, T) that
// workers claim from a counter once their own range is done (SMs do not all stream
// at one rate, and the slow ones would otherwise set the end of the launch).  Range
// indices grow along the flattened order, so the ranges covering a unit are
// consecutive and a partial's slot is range + unit.
struct Split {
    int T, Ts, W, P, S;        // flattened indices fit in 32 bits (checked on the host)
    __device__ int range_of(int f) const { return f < Ts ? worker_of(f, Ts, W) : W + (f - Ts) / S; }
};

// dyn256 / 256 of the blocks go to pieces of an eighth of a static range (at least
// kMinPiece blocks), at most one piece per worker, when ranges are long enough to
// cut (kMinPieceRange blocks: a piece of a short range takes a warp as long as a
// range); every worker gets a non-empty static range or none.
__device__ __forceinline__ Split make_split(int T, int workers, int dyn256) {
    Split sp;
    sp.T = T;
    const int per = T / max(workers, 1);
    const int dyn = per < kMinPieceRange ? 0 : static_cast<int>(static_cast<long long>(T) * dyn256 / 256);
    const int P = min(workers, dyn / max(kMinPiece, per / 8));
    if (P <= 0) {
        sp.Ts = T;
        sp.P = 0;
        sp.S = 1;
    } else {
        sp.S = (dyn + P - 1) / P;
        sp.P = (dyn + sp.S - 1) / sp.S;
        sp.Ts = T - dyn;
    }
    sp.W = min(workers, sp.Ts);
    return sp;
}

// Cursor at flattened index f: the sequence s with cum[s] <= f < cum[s + 1].
__device__ __forceinline__ Cursor locate(int f, const int* cum, int B, int UH) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid] <= f) lo = mid; else hi = mid;
    }
    Cursor c;
    c.s = lo;
    c.nb = (cum[lo + 1] - cum[lo]) / UH;
    const int rem = f - cum[lo];
    c.uh = rem / c.nb;
    c.j = rem % c.nb;
    return c;
}

// Decode rows of a mixed batch are the sequences with q_len == 1 (whose row lies
// inside q: a malformed query_start_loc is recorded by the prologue and its rows skipped).
__device__ __forceinline__ bool decode_row(const DecodeParams& p, int s) {
    if (p.query_start_loc == nullptr) return true;
    const int a = p.query_start_loc[s];
    return p.query_start_loc[s + 1] - a == 1 && a >= 0 && a < p.total_rows;
}

// Blocks sequence s contributes to the flattened order (its blocks x units); a
// cascade decode covers only the blocks after the shared prefix.
// The flattened order counts 16-key units (one MMA tile each) whatever the
// physical block size: a 32-token block holds two units, an 8-token block half of one.
__device__ __forceinline__ int unit_blocks_of(const DecodeParams& p, int s, int UH) {
    if (!decode_row(p, s)) return 0;
    const int nb = (max(p.seq_lens[s], 0) + kBlockSize - 1) / kBlockSize;
    const int cap = (p.max_blocks * p.block_size + kBlockSize - 1) / kBlockSize;
    return max(min(nb, cap) - p.first_block, 0) * UH;
}

template <typename T>
__device__ __forceinline__ T shfl(T v, int src) {
    return __shfl_sync(0xffffffffu, v, src);
}

}  // namespace

template <int Kind, bool QBf16, bool Append, bool Dyn, int Stages = 3>
__device__ __forceinline__ void decode_body(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p) {
    using Cfg = DecodeCfg<Kind, Stages>;
    constexpr bool kFp8 = Cfg::kFp8;
    constexpr bool kMmaBf16 = Kind == kKindBf16;   // fp16 and FP8 (widened) use f16 MMA
    constexpr int NS = Cfg::kStages;
    constexpr int TILE = Cfg::kTileBytes;
    constexpr int STAGE = Cfg::kStageBytes;

    extern __shared__ uint8_t smem_raw[];
    __shared__ int warp_tot[kDecodeWarps];
    __shared__ int staged_unit[kDecodeWarps];   // static ranges: unit whose partial a warp left here
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t tiles = (raw_base + 1023u) & ~1023u;     // 128-byte swizzle needs 1 KiB alignment
    uint8_t* aligned = smem_raw + (tiles - raw_base);
    const uint32_t bars = tiles + Cfg::kTileArea;
    int* cum = reinterpret_cast<int*>(aligned + Cfg::kTileArea + Cfg::kBarBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t my_tiles = tiles + warp * NS * STAGE;
    const uint32_t my_bars = bars + warp * NS * 8;

    if (lane == 0) {
        for (int st = 0; st < NS; ++st) mbar_init(my_bars + 8 * st, 1);
        fence_barrier_init();
    }
    if (threadIdx.x == 0) {
        tmap_prefetch(&kmap);
        tmap_prefetch(&vmap);
    }

    if (!p.overlap_prior) grid_dependency_wait();

    const int B = p.num_seqs;
    const int UH = p.num_kv_heads * p.head_groups;
    const bool mixed = p.query_start_loc != nullptr;

    // ---- prologue: blocks per unit of every sequence, exclusive scan -> cum ----
    auto eligible = [&](int s) -> bool { return decode_row(p, s); };
    auto unit_blocks = [&](int s) -> int { return unit_blocks_of(p, s, UH); };
    {
        const int per = (B + blockDim.x - 1) / blockDim.x;
        const int beg = min(B, static_cast<int>(threadIdx.x) * per);
        const int end = min(B, beg + per);
        int local = 0;
        for (int s = beg; s < end; ++s) local += unit_blocks(s);
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int run = incl - local;
        for (int w = 0; w < warp; ++w) run += warp_tot[w];
        for (int s = beg; s < end; ++s) {
            cum[s] = run;
            run += unit_blocks(s);
        }
        if (threadIdx.x == blockDim.x - 1) cum[B] = run;
    }
    if (p.cascade) {
        // every table must start with sequence 0's first_block entries and every
        // sequence must hold the whole prefix
        const int shared = (p.first_block * kBlockSize) >> p.block_shift;   // shared table entries
        const long long checks = static_cast<long long>(B) * shared;
        for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < checks;
             i += static_cast<long long>(gridDim.x) * blockDim.x) {
            const int s = static_cast<int>(i / shared), j = static_cast<int>(i % shared);
            if (__ldg(p.block_tables + static_cast<size_t>(s) * p.max_blocks + j) != __ldg(p.block_tables + j) ||
                (j == 0 && p.seq_lens[s] < p.first_block * kBlockSize))   // first_block: 16-key units
                atomicOr(p.status, kDevErrRange);
        }
    }
    // empty decode rows produce zeros; over-long sequences are an input error
    for (int s = blockIdx.x; s < B; s += gridDim.x) {
        if (mixed && threadIdx.x == 0) {
            const int a = p.query_start_loc[s], b = p.query_start_loc[s + 1];
            if (a < 0 || b < a || b > p.total_rows) atomicOr(p.status, kDevErrRange);
        }
        if (!eligible(s)) continue;
        const int n = p.seq_lens[s];
        if (threadIdx.x == 0 && n > p.max_blocks * p.block_size) atomicOr(p.status, kDevErrRange);
        // a fused slot write needs a token to write: an empty sequence takes padding
        if (threadIdx.x == 0 && p.append && n <= 0 && p.slots[s] >= 0) atomicOr(p.status, kDevErrRange);
        if (n > 0) continue;
        const int row = mixed ? p.query_start_loc[s] : s;
        uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                            static_cast<size_t>(row) * p.num_q_heads * kHeadDim);
        for (int i = threadIdx.x; i < p.num_q_heads * kHeadDim / 8; i += blockDim.x)
            o[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    grid_launch_dependents();
    if (B > kCombineScanSeqs && blockIdx.x == 0) {
        // the block prefix, for the combine kernel of a large batch
        for (int i = threadIdx.x; i <= B; i += blockDim.x) p.plan[i] = cum[i];
    }

    const int T = cum[B];
    if (T == 0) return;
    const Split sp = make_split(T, p.num_workers, p.dyn256);
    const int wid = blockIdx.x * kDecodeWarps + warp;
    // With static ranges the warps of a CTA, whose ranges follow one another, merge
    // the partials of the unit their ranges end in before one of them writes it: a
    // unit then leaves one partial per CTA it spans, not one per warp.  Every warp
    // reaches that merge, with or without work.
    int my_staged = -1;
    if (wid < p.num_workers) do {
    // pieces are numbered from the counter's value when this call began (the
    // previous call's combine set claim[1] to the counter's final value)
    const unsigned claim_base = __ldcg(p.claim + 1);
    // a claim is sent kClaimAhead blocks before the producer needs it, so that the
    // atomic (all warps reach the end of their static ranges at about the same time)
    // returns while the ring still streams
    unsigned claim_got = 0;
    bool claim_sent = false;
    auto send_claim = [&]() {
        if (lane == 0) claim_got = atomicAdd(p.claim, 1u);
        claim_sent = true;
    };
    auto claim = [&](int& lo, int& hi, int& ri) -> bool {
        if (!claim_sent) send_claim();
        claim_sent = false;
        const unsigned k = shfl(claim_got, 0) - claim_base;     // modulo 2^32
        if (k >= static_cast<unsigned>(sp.P)) return false;
        lo = sp.Ts + static_cast<int>(k) * sp.S;
        hi = min(sp.T, lo + sp.S);
        ri = sp.W + static_cast<int>(k);
        return true;
    };
    // the consumer's range [c_lo, c_hi), index c_ri: first the worker's static range
    int c_lo = 0, c_hi = 0, c_ri = 0;
    if (wid < sp.W) {
        c_ri = wid;
        c_lo = static_cast<int>(static_cast<long long>(sp.Ts) * wid / sp.W);
        c_hi = static_cast<int>(static_cast<long long>(sp.Ts) * (wid + 1) / sp.W);
    } else if (!Dyn || !claim(c_lo, c_hi, c_ri)) {
        break;
    }
    const Cursor start = locate(c_lo, cum, B, UH);

    // per-lane fragment geometry
    const int g = lane >> 2;           // MMA group row
    const int t = lane & 3;            // MMA thread in group
    const int mi = lane >> 3;          // ldmatrix sub-matrix this lane addresses
    const int r8 = lane & 7;           // row within it
    const uint32_t k_row = static_cast<uint32_t>(r8 + ((mi & 1) << 3));
    const uint32_t v_row = kFp8 ? k_row : static_cast<uint32_t>(r8 + ((mi >> 1) << 3));

    // ---- producer: block-table window + TMA issue ----
    int tbl_s = -1, tbl_j0 = -1, tbl = 0;
    int pn_s = -1, pn_ent = 0, pn_n = 0;        // producer: sequence whose table entries are counted
    // fused slot write: the lane's 16 bytes of the next new-token row (k_new / v_new
    // row s H_kv + h), fetched when the unit holding it is issued and stored when it
    // is consumed, so that neither waits for the load
    const int part = lane & 15;
    const bool part_v = lane >= 16;
    const uint16_t* new_rows = part_v ? p.v_new : p.k_new;
    auto load_new = [&](int row) -> uint4 {
        return __ldg(reinterpret_cast<const uint4*>(new_rows + static_cast<size_t>(row) * kHeadDim) + part);
    };
    int pf_row = -1, pf_want = 0, pf_dst = 0;       // row fetched ahead (-1: none pending)
    long long pf_slot = -1;
    uint4 pf_x = make_uint4(0, 0, 0, 0);
    // A cascade's private blocks are read once, beside partials (the prefix grid's and
    // this grid's) that the combine reads back: the stream leaves L2 first, the
    // partials stay in it
    const bool stream_first = p.cascade != 0;
    const uint64_t pol = stream_first ? l2_policy_evict_first() : 0ull;
    auto load = [&](uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
        if (stream_first) tma_load_2d_hint(dst, map, x, y, bar, pol);
        else tma_load_2d(dst, map, x, y, bar);
    };
    auto issue = [&](const Cursor& c, int k) {
        // unit ja (16 keys) of the sequence: with blocks of 16 or 32 tokens it lies in
        // table entry 16 ja / bs at row offset 16 ja mod bs; with 8-token blocks it
        // spans entries 2 ja and 2 ja + 1 (the second only if the sequence reaches it)
        const int ja = c.j + p.first_block;
        const int bs = p.block_size, bsh = p.block_shift;
        if (c.s != pn_s) {
            pn_s = c.s;
            pn_n = max(p.seq_lens[c.s], 0);
            pn_ent = (pn_n + bs - 1) >> bsh;
        }
        const int ti = (ja * kBlockSize) >> bsh;
        if (c.s != tbl_s || (ti & ~31) != tbl_j0) {
            tbl_s = c.s;
            tbl_j0 = ti & ~31;
            const int jj = tbl_j0 + lane;
            tbl = jj < pn_ent && jj < p.max_blocks ? __ldg(p.block_tables + static_cast<size_t>(c.s) * p.max_blocks + jj) : 0;
        }
        const bool two = bs < kBlockSize && ti + 1 < pn_ent;
        int phys0 = shfl(tbl, ti & 31), phys1 = shfl(tbl, (ti + 1) & 31);
        if (static_cast<unsigned>(phys0) >= static_cast<unsigned>(p.num_blocks) ||
            (two && static_cast<unsigned>(phys1) >= static_cast<unsigned>(p.num_blocks))) {
            if (lane == 0) atomicOr(p.status, kDevErrRange);
            phys0 = static_cast<unsigned>(phys0) >= static_cast<unsigned>(p.num_blocks) ? 0 : phys0;
            phys1 = static_cast<unsigned>(phys1) >= static_cast<unsigned>(p.num_blocks) ? 0 : phys1;
        }
        const int h = c.uh / p.head_groups;
        const int y0 = ((phys0 * p.num_kv_heads + h) << bsh) + ((ja * kBlockSize) & (bs - 1));
        const int y1 = (phys1 * p.num_kv_heads + h) << bsh;
        if (Append && ja == ((pn_n - 1) >> 4) && pf_row < 0) {
            // the sequence's last 16 keys hold its new token (position n - 1): fetch the
            // lane's part of its row, its slot and where it belongs now, for the
            // consumer to store when this unit is consumed
            const int e = (pn_n - 1) >> bsh;                          // its table entry
            const int ph = e == ti ? phys0 : phys1;
            pf_row = c.s * p.num_kv_heads + h;
            pf_x = load_new(pf_row);
            pf_slot = __ldg(p.slots + c.s);
            pf_want = ph * bs + ((pn_n - 1) & (bs - 1));
            pf_dst = ((ph * p.num_kv_heads + h) << bsh) + ((pn_n - 1) & (bs - 1));
        }
        if (lane == 0) {
            const int st = k % NS;
            const uint32_t bar = my_bars + 8 * st;
            const uint32_t dst = my_tiles + st * STAGE;
            fence_proxy_async_smem();
            if (bs >= kBlockSize) {
                mbar_arrive_expect_tx(bar, STAGE);
                if constexpr (kFp8) {
                    load(dst, &kmap, 0, y0, bar);
                    load(dst + TILE, &vmap, 0, y0, bar);
                } else {
                    load(dst, &kmap, 0, y0, bar);
                    load(dst + 2048, &kmap, 64, y0, bar);
                    load(dst + TILE, &vmap, 0, y0, bar);
                    load(dst + TILE + 2048, &vmap, 64, y0, bar);
                }
            } else {
                // 8-row boxes: rows 0-7 of the tile from the first block, 8-15 from the second
                mbar_arrive_expect_tx(bar, two ? STAGE : STAGE / 2);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    if (e == 1 && !two) break;
                    const int y = e ? y1 : y0;
                    const uint32_t o = 1024u * e;
                    if constexpr (kFp8) {
                        load(dst + o, &kmap, 0, y, bar);
                        load(dst + TILE + o, &vmap, 0, y, bar);
                    } else {
                        load(dst + o, &kmap, 0, y, bar);
                        load(dst + 2048 + o, &kmap, 64, y, bar);
                        load(dst + TILE + o, &vmap, 0, y, bar);
                        load(dst + TILE + 2048 + o, &vmap, 64, y, bar);
                    }
                }
            }
        }
    };

    // producer: next flattened index p_f of its range [.., p_hi); a range it claims is
    // handed to the consumer (at most one waits: a piece is longer than the ring)
    Cursor P = start;
    int kp = 0;
    int p_f = c_lo, p_hi = c_hi;
    bool p_done = sp.P == 0, nx_valid = false;      // nothing to claim: no atomics at all
    int nx_lo = 0, nx_hi = 0, nx_ri = 0;
    auto produce = [&]() {
        if constexpr (!Dyn) {
            if (p_f == p_hi) return;
        } else if (!p_done && !claim_sent && p_hi - p_f <= kClaimAhead) {
            send_claim();
        }
        if (p_f == p_hi) {
            if (p_done || nx_valid) return;
            int lo, hi, ri;
            if (!claim(lo, hi, ri)) {
                p_done = true;
                return;
            }
            nx_lo = lo;
            nx_hi = hi;
            nx_ri = ri;
            nx_valid = true;
            p_f = lo;
            p_hi = hi;
            P = locate(lo, cum, B, UH);
        }
        issue(P, kp);
        cursor_advance(P, cum, B, UH);
        ++kp;
        ++p_f;
    };
    for (int i = 0; i < NS; ++i) produce();

    // FP8 scales of the current unit's KV head (set at each segment start)
    float s_log2 = p.scale_log2, vscale = 1.0f;

    Cursor C = start;
    float o[8][4];
    uint32_t qf[8][2];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int n_cur = 0, row_cur = 0;
    bool open = false;

    int c_f = c_lo;
    for (int kc = 0; kc < kp; ++kc) {
        if (!open) {
            // ---- segment start: query fragments of this unit ----
            open = true;
            n_cur = p.seq_lens[C.s];
            row_cur = mixed ? p.query_start_loc[C.s] : C.s;
            const int h = C.uh / p.head_groups;
            const int hg = C.uh % p.head_groups;
            const int gh = hg * kHeadsPerGroup + g;        // head within the GQA group
            if constexpr (kFp8) {
                s_log2 = p.scale_log2 * __ldg(p.k_scale + h * p.scale_stride);
                vscale = __ldg(p.v_scale + h * p.scale_stride);
            }
            const bool live = gh < p.group;
            const uint16_t* qrow = static_cast<const uint16_t*>(p.q) +
                                   (static_cast<size_t>(row_cur) * p.num_q_heads + h * p.group + (live ? gh : 0)) * kHeadDim;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                if constexpr (!kFp8) {
                    qf[kk][0] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * t) : 0u;
                    qf[kk][1] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * t + 8) : 0u;
                } else {
                    // k-slots (2t, 2t+1) <-> d (16kk+4t, +1); (2t+8, 2t+9) <-> d (16kk+4t+2, +3)
                    uint2 raw = live ? *reinterpret_cast<const uint2*>(qrow + 16 * kk + 4 * t) : make_uint2(0, 0);
                    qf[kk][0] = pack2<false>(to_float<QBf16>(raw.x & 0xffff), to_float<QBf16>(raw.x >> 16));
                    qf[kk][1] = pack2<false>(to_float<QBf16>(raw.y & 0xffff), to_float<QBf16>(raw.y >> 16));
                }
            }
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }

        // ---- wait for this block's tiles ----
        const int st = kc % NS;
        const uint32_t bar = my_bars + 8 * st;
        const uint32_t parity = (kc / NS) & 1;
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded(bar, parity, p.timeout_ns);
        ok = shfl(static_cast<int>(ok), 0) != 0;
        if (!ok) {
            if (lane == 0) {
                atomicOr(p.status, kDevErrTimeout);
                // let copies still in flight land before the warp leaves
                for (int k = kc; k < kp; ++k)
                    mbar_wait_bounded(my_bars + 8 * (k % NS), (k / NS) & 1, p.timeout_ns);
            }
            __syncwarp();
            break;
        }
        mbar_try_wait(bar, parity);   // phase is complete: acquire for every lane

        const uint32_t kt = my_tiles + st * STAGE;
        const uint32_t vt = kt + TILE;
        const int valid = min(kBlockSize, n_cur - (C.j + p.first_block) * kBlockSize);
        if constexpr (Append) {
            if (C.j + p.first_block == ((n_cur - 1) >> 4)) {
                // this unit holds the sequence's new token: store it into its slot and
                // over its row of the tile just copied (the copy may predate the store)
                const int h = C.uh / p.head_groups;
                const int nrow = C.s * p.num_kv_heads + h;
                uint4 x;
                long long slot;
                int want, dst;
                bool ok_row = true;
                if (nrow == pf_row) {
                    x = pf_x;
                    slot = pf_slot;
                    want = pf_want;
                    dst = pf_dst;
                    pf_row = -1;
                } else {   // a second new token inside the ring: fetched now
                    const int e = (n_cur - 1) >> p.block_shift;
                    const int ph = __ldg(p.block_tables + static_cast<size_t>(C.s) * p.max_blocks + e);
                    ok_row = static_cast<unsigned>(ph) < static_cast<unsigned>(p.num_blocks);
                    x = load_new(nrow);
                    slot = __ldg(p.slots + C.s);
                    want = ph * p.block_size + ((n_cur - 1) & (p.block_size - 1));
                    dst = ((ph * p.num_kv_heads + h) << p.block_shift) + ((n_cur - 1) & (p.block_size - 1));
                }
                if (slot >= 0) {
                    if (!ok_row || slot != want) {
                        if (lane == 0) atomicOr(p.status, kDevErrRange);
                    } else {
                        const uint32_t r = static_cast<uint32_t>((n_cur - 1) & 15);    // row in the tile
                        const uint32_t tile = part_v ? vt : kt;
                        if constexpr (!kFp8) {
                            uint16_t* gdst = static_cast<uint16_t*>(part_v ? p.v_cache_w : p.k_cache_w) +
                                             static_cast<size_t>(dst) * kHeadDim;
                            reinterpret_cast<uint4*>(gdst)[part] = x;
                            const uint32_t a = tile + ((part >> 3) << 11) + (r << 7) + (((part & 7) ^ (r & 7)) << 4);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x.x), "r"(x.y),
                                         "r"(x.z), "r"(x.w) : "memory");
                        } else {
                            const float sc = __ldg((part_v ? p.v_scale : p.k_scale) + h * p.scale_stride);
                            const uint32_t lo = e4m3_pair<QBf16>(x.x, sc) | (e4m3_pair<QBf16>(x.y, sc) << 16);
                            const uint32_t hi = e4m3_pair<QBf16>(x.z, sc) | (e4m3_pair<QBf16>(x.w, sc) << 16);
                            uint8_t* gdst = static_cast<uint8_t*>(part_v ? p.v_cache_w : p.k_cache_w) +
                                            static_cast<size_t>(dst) * kHeadDim;
                            reinterpret_cast<uint2*>(gdst)[part] = make_uint2(lo, hi);
                            const uint32_t a = tile + (r << 7) + ((((part >> 1) ^ (r & 7))) << 4) + ((part & 1) << 3);
                            asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(a), "r"(lo), "r"(hi) : "memory");
                        }
                        fence_proxy_async_smem();     // before a later copy into this stage
                    }
                }
                __syncwarp();
            }
        }

        // ---- S^T = K . Q^T : rows = 16 keys, cols = 8 heads ----
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (!kFp8) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t c = 2 * kk + (mi >> 1);
                const uint32_t addr = kt + ((c >> 3) << 11) + (k_row << 7) + (((c & 7) ^ r8) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(addr, a0, a1, a2, a3);
                if (kk & 1) mma16816<kMmaBf16>(sb, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
                else        mma16816<kMmaBf16>(sa, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
            }
        } else {
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
                const uint32_t c = 2 * kq + (mi >> 1);
                const uint32_t addr = kt + (k_row << 7) + ((c ^ r8) << 4);
                uint32_t x0, x1, x2, x3;
                ldsm_x4(addr, x0, x1, x2, x3);
                mma16816<false>(sa, e4m3x2_to_f16x2(x0 & 0xffff), e4m3x2_to_f16x2(x1 & 0xffff),
                                e4m3x2_to_f16x2(x0 >> 16), e4m3x2_to_f16x2(x1 >> 16), qf[2 * kq][0],
                                qf[2 * kq][1]);
                mma16816<false>(sb, e4m3x2_to_f16x2(x2 & 0xffff), e4m3x2_to_f16x2(x3 & 0xffff),
                                e4m3x2_to_f16x2(x2 >> 16), e4m3x2_to_f16x2(x3 >> 16), qf[2 * kq + 1][0],
                                qf[2 * kq + 1][1]);
            }
        }
        // element (key g | g+8, head 2t | 2t+1), in log2 units
        float s0 = (sa[0] + sb[0]) * s_log2;
        float s1 = (sa[1] + sb[1]) * s_log2;
        float s2 = (sa[2] + sb[2]) * s_log2;
        float s3 = (sa[3] + sb[3]) * s_log2;
        if (valid < kBlockSize) {
            if (g >= valid) s0 = s1 = -INFINITY;
            if (g + 8 >= valid) s2 = s3 = -INFINITY;
        }

        // ---- online softmax over keys (lanes with equal t share heads) ----
        float x0 = fmaxf(s0, s2), x1 = fmaxf(s1, s3);
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o2));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o2));
        }
        const float mn0 = fmaxf(m0, x0), mn1 = fmaxf(m1, x1);
        const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        const float p0 = exp2f(s0 - mn0), p1 = exp2f(s1 - mn1);
        const float p2 = exp2f(s2 - mn0), p3 = exp2f(s3 - mn1);
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
            o[dt][0] *= al0;
            o[dt][1] *= al1;
            o[dt][2] *= al0;
            o[dt][3] *= al1;
        }
        // P^T as the B operand: keys 2t,2t+1 (and +8) of head g
        const uint32_t pb0 = movmatrix_t(pack2<kMmaBf16>(p0, p1));
        const uint32_t pb1 = movmatrix_t(pack2<kMmaBf16>(p2, p3));

        // keys beyond the sequence end: zero V so stale or NaN slots cannot leak
        uint32_t vm01 = 0xffffffffu, vm23 = 0xffffffffu;
        if (valid < kBlockSize) {
            vm01 = (2 * t < valid ? 0x0000ffffu : 0u) | (2 * t + 1 < valid ? 0xffff0000u : 0u);
            vm23 = (2 * t + 8 < valid ? 0x0000ffffu : 0u) | (2 * t + 9 < valid ? 0xffff0000u : 0u);
        }

        // ---- O^T += V^T . P^T : rows = d, cols = heads ----
        if constexpr (!kFp8) {
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) {
                const uint32_t c = 2 * dt + (mi & 1);
                const uint32_t addr = vt + ((c >> 3) << 11) + (v_row << 7) + (((c & 7) ^ r8) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(addr, a0, a1, a2, a3);
                mma16816<kMmaBf16>(o[dt], a0 & vm01, a1 & vm01, a2 & vm23, a3 & vm23, pb0, pb1);
            }
        } else {
#pragma unroll
            for (int dq = 0; dq < 4; ++dq) {
                const uint32_t c = 2 * dq + (mi >> 1);
                const uint32_t addr = vt + (v_row << 7) + ((c ^ r8) << 4);
                uint32_t x0v, x1v, x2v, x3v;
                ldsm_x4_t(addr, x0v, x1v, x2v, x3v);
                // bytes [V(2t,d), V(2t,d+1), V(2t+1,d), V(2t+1,d+1)], d = 16c + 2g
                const uint32_t e0 = prmt(x0v, 0, 0x3120), e1 = prmt(x1v, 0, 0x3120);
                const uint32_t e2 = prmt(x2v, 0, 0x3120), e3 = prmt(x3v, 0, 0x3120);
                mma16816<false>(o[2 * dq], e4m3x2_to_f16x2(e0 & 0xffff) & vm01,
                                e4m3x2_to_f16x2(e0 >> 16) & vm01, e4m3x2_to_f16x2(e1 & 0xffff) & vm23,
                                e4m3x2_to_f16x2(e1 >> 16) & vm23, pb0, pb1);
                mma16816<false>(o[2 * dq + 1], e4m3x2_to_f16x2(e2 & 0xffff) & vm01,
                                e4m3x2_to_f16x2(e2 >> 16) & vm01, e4m3x2_to_f16x2(e3 & 0xffff) & vm23,
                                e4m3x2_to_f16x2(e3 >> 16) & vm23, pb0, pb1);
            }
        }
        __syncwarp();

        // refill the stage just consumed
        produce();

        // ---- segment end: unit finished or range finished ----
        if (C.j == C.nb - 1 || c_f == c_hi - 1) {
            open = false;
#pragma unroll
            for (int o2 = 4; o2 < 32; o2 <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
                l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
            }
            const int u = C.s * UH + C.uh;
            const int fu = cum[C.s] + C.uh * C.nb;
            // a unit one range covers is written directly, unless a prefix partial waits for it
            const bool write = !p.cascade && sp.range_of(fu) == sp.range_of(fu + C.nb - 1);
            // static ranges: a unit that goes on past this range's end (the range's last
            // segment; the ring is idle) is staged in the warp's ring for the CTA merge
            const bool stage = !Dyn && !write && C.j != C.nb - 1;
            if (!write) {
                // unit shared with other ranges: plain partial store, merged by combine_kernel
                const int slot = c_ri + u;
                float4* part = stage ? reinterpret_cast<float4*>(aligned + warp * NS * STAGE)
                                     : p.partial + static_cast<size_t>(slot) * 8 * 32;
#pragma unroll
                for (int dt = 0; dt < 8; ++dt) part[dt * 32 + lane] = make_float4(o[dt][0], o[dt][1], o[dt][2], o[dt][3]);
                if (lane < 4) {
                    float* ml = stage ? reinterpret_cast<float*>(part + 8 * 32) : p.ml + static_cast<size_t>(slot) * 16;
                    ml[2 * t] = m0;
                    ml[2 * t + 1] = m1;
                    ml[8 + 2 * t] = l0;
                    ml[8 + 2 * t + 1] = l1;
                }
                if (stage) my_staged = u;
            }
            if (write) {
                const int h = C.uh / p.head_groups;
                const int hg = C.uh % p.head_groups;
                const float inv0 = vscale / l0, inv1 = vscale / l1;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int gh = hg * kHeadsPerGroup + 2 * t + e;
                    if (gh >= p.group) continue;
                    const float inv = e ? inv1 : inv0;
                    uint16_t* orow = static_cast<uint16_t*>(p.out) +
                                     (static_cast<size_t>(row_cur) * p.num_q_heads + h * p.group + gh) * kHeadDim;
#pragma unroll
                    for (int dt = 0; dt < 8; ++dt) {
                        const uint16_t lo = from_float<QBf16>(o[dt][e] * inv);
                        const uint16_t hi = from_float<QBf16>(o[dt][2 + e] * inv);
                        if constexpr (kFp8) {
                            // rows g, g+8 of the tile are d = 16dt + 2g, 16dt + 2g + 1
                            *reinterpret_cast<uint32_t*>(orow + 16 * dt + 2 * g) =
                                static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
                        } else {
                            orow[16 * dt + g] = lo;
                            orow[16 * dt + g + 8] = hi;
                        }
                    }
                }
            }
        }
        if (++c_f == c_hi && Dyn) {
            if (!nx_valid) continue;          // the loop ends once every issued block is consumed
            c_lo = nx_lo;
            c_hi = nx_hi;
            c_ri = nx_ri;
            nx_valid = false;
            c_f = c_lo;
            C = locate(c_lo, cum, B, UH);
            open = false;
        } else {
            cursor_advance(C, cum, B, UH);
        }
    }
    } while (false);

    if constexpr (!Dyn) {
        // ---- CTA merge of staged partials: the first warp of each run of warps that
        // staged the same unit folds the run and writes one partial (slot wid + unit) ----
        if (lane == 0) staged_unit[warp] = my_staged;
        __syncthreads();
        if (my_staged >= 0 && (warp == 0 || staged_unit[warp - 1] != my_staged)) {
            const int t = lane & 3;
            float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
            float4 acc[8];
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) acc[dt] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int w2 = warp; w2 < kDecodeWarps && staged_unit[w2] == my_staged; ++w2) {
                const float4* part = reinterpret_cast<const float4*>(aligned + w2 * NS * STAGE);
                const float* ml = reinterpret_cast<const float*>(part + 8 * 32);
                const float m0w = ml[2 * t], m1w = ml[2 * t + 1], l0w = ml[8 + 2 * t], l1w = ml[8 + 2 * t + 1];
                const float n0 = fmaxf(M0, m0w), n1 = fmaxf(M1, m1w);
                const float r0 = exp2f(M0 - n0), r1 = exp2f(M1 - n1);      // 0 while nothing is summed
                const float w0 = exp2f(m0w - n0), w1 = exp2f(m1w - n1);
#pragma unroll
                for (int dt = 0; dt < 8; ++dt) {
                    const float4 x = part[dt * 32 + lane];
                    acc[dt] = make_float4(acc[dt].x * r0 + x.x * w0, acc[dt].y * r1 + x.y * w1,
                                          acc[dt].z * r0 + x.z * w0, acc[dt].w * r1 + x.w * w1);
                }
                L0 = L0 * r0 + l0w * w0;
                L1 = L1 * r1 + l1w * w1;
                M0 = n0;
                M1 = n1;
            }
            const int slot = wid + my_staged;
            float4* gpart = p.partial + static_cast<size_t>(slot) * 8 * 32;
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) gpart[dt * 32 + lane] = acc[dt];
            if (lane < 4) {
                float* gml = p.ml + static_cast<size_t>(slot) * 16;
                gml[2 * t] = M0;
                gml[2 * t + 1] = M1;
                gml[8 + 2 * t] = L0;
                gml[8 + 2 * t + 1] = L1;
            }
        }
    }
}

// 16-bit caches: at most 136 registers per thread, so that two CTAs (128 threads
// each) and a combine CTA (256 threads, at most 112) share an SM and the combine is
// resident, past its prologue, while the decode grid drains (with the two-stage
// ring, three CTAs per SM and the combine starts as they drain).  FP8 caches: 128,
// so that four CTAs fill the register file.
template <int Kind>
constexpr int decode_max_regs() { return Kind == kKindFp8 ? 128 : 136; }

template <int Kind, bool QBf16, bool Dyn, int Stages>
__global__ void __maxnreg__(decode_max_regs<Kind>())
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p) {
    decode_body<Kind, QBf16, false, Dyn, Stages>(kmap, vmap, p);
    // Overlapping a chunk launch of the same call (which neither reads what this grid
    // writes nor writes what it reads): the last CTA alone waits for it before exiting,
    // so that this grid, and the combine chained behind it, completes after it while
    // every other CTA frees its SM as soon as its range is done.
    if (p.overlap_prior && blockIdx.x == gridDim.x - 1) grid_dependency_wait();
}

// The same with the new tokens' slot write fused in (pa_decode_append).
template <int Kind, bool QBf16, bool Dyn>
__global__ void __maxnreg__(decode_max_regs<Kind>())
    decode_append_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                         const DecodeParams p) {
    decode_body<Kind, QBf16, true, Dyn>(kmap, vmap, p);
}


// Log-sum-exp combine of the units split across workers:
//   out = sum_i e^{m_i - M} o_i / sum_i e^{m_i - M} l_i,   M = max_i m_i,
// where worker i left its unnormalised output o_i, running max m_i (log2 units)
// and running sum l_i.  One CTA per unit at a time, one warp per 16-wide slice of
// d; a lane owns heads 2t, 2t+1 of the fragment layout.  The unit's place in the
// flattened order comes from `pre` (the block prefix per sequence, which the CTA
// computed from the lengths before waiting for the decode grid), or for large
// batches from the plan the decode grid published; after the wait one round trip
// brings up to kBatch slots' fragments together with their (m, l) for the lane's
// two heads, reduced in registers (online across batches): no shuffles.
template <bool OutBf16, bool Fp8Layout, bool Cascade, int kBatch>
__device__ __forceinline__ void combine_unit(const DecodeParams& p, int u, const int* pre_sum) {
    const int UH = p.num_kv_heads * p.head_groups;
    const int s = u / UH, uh = u % UH;
    const int B = p.num_seqs;
    const int dt = threadIdx.x >> 5, lane = threadIdx.x & 31, t = lane & 3, g = lane >> 2;
    long long lo = 0, T = 0;
    if (B <= kCombineScanSeqs) {
        lo = pre_sum[s];
        T = pre_sum[B];
    } else {
        grid_dependency_wait();
        lo = p.plan[s];
        T = p.plan[B];
    }
    const int nb = unit_blocks_of(p, s, UH) / UH;
    const bool pre = Cascade && p.first_block > 0;     // every row has a shared-prefix partial
    // the unit's partials: one per range it spans (ranges wa .. wb), or with static
    // ranges, where each CTA merged the partials of the unit its warps' ranges end in,
    // one for wa, one for the first warp of every later CTA before wb, and one for wb
    int wa = 0, wb = 0, nseg = 0, m0 = 0;
    const bool cta_merged = p.dyn256 == 0;
    if (nb > 0 && T > 0) {
        const Split sp = make_split(static_cast<int>(T), p.num_workers, p.dyn256);
        const int fu = static_cast<int>(lo) + uh * nb;
        wa = sp.range_of(fu);
        wb = sp.range_of(fu + nb - 1);
        if (wa == wb && !Cascade) return;     // its only range wrote the output
        if (!cta_merged || wa == wb) {
            nseg = wb - wa + 1;
        } else {
            m0 = (wa / kDecodeWarps + 1) * kDecodeWarps;
            nseg = 2 + (m0 <= wb - 1 ? (wb - 1 - m0) / kDecodeWarps + 1 : 0);
        }
    } else if (!pre) {
        return;   // an empty row: the decode grid wrote its zeros
    }
    const int h = uh / p.head_groups;
    const int hg = uh % p.head_groups;
    const int row = p.query_start_loc ? p.query_start_loc[s] : s;

    if (B <= kCombineScanSeqs) grid_dependency_wait();
    float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    // fold a batch of n pieces, each (fragment, max, sum) of the lane's two heads,
    // into the running (M, L, acc) (padding heads may turn to NaN: never written)
    auto fold = [&](const float4 (&v)[kBatch], const float2 (&mv)[kBatch], const float2 (&lv)[kBatch], int n) {
        float b0 = M0, b1 = M1;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            if (k < n) {
                b0 = fmaxf(b0, mv[k].x);
                b1 = fmaxf(b1, mv[k].y);
            }
        }
        // rescale what is summed so far (zero while nothing is: M = -inf)
        const float r0 = exp2f(M0 - b0), r1 = exp2f(M1 - b1);
        acc[0] *= r0;
        acc[2] *= r0;
        acc[1] *= r1;
        acc[3] *= r1;
        L0 *= r0;
        L1 *= r1;
        M0 = b0;
        M1 = b1;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            if (k < n) {
                const float w0 = exp2f(mv[k].x - M0), w1 = exp2f(mv[k].y - M1);
                acc[0] += v[k].x * w0;
                acc[1] += v[k].y * w1;
                acc[2] += v[k].z * w0;
                acc[3] += v[k].w * w1;
                L0 += lv[k].x * w0;
                L1 += lv[k].y * w1;
            }
        }
    };
    // the shared-prefix partials of the unit's rows, one per key segment of the
    // prefix, stored row-wise; fragment element (d, head 2t + e) of the lane is
    // d = dA (components 0, 1) and dB (2, 3)
    const int npre = pre ? p.prefix_splits : 0;
    if (Cascade && npre > 0) {
        const int dA = Fp8Layout ? 16 * dt + 2 * g : 16 * dt + g;
        const int dB = Fp8Layout ? dA + 1 : dA + 8;
        const size_t rows = static_cast<size_t>(B) * p.num_q_heads;
        for (int base = 0; base < npre; base += kBatch) {
            float4 v[kBatch];
            float2 mv[kBatch], lv[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int idx = min(base + k, npre - 1);
                const float* so = idx == 0 ? p.prefix_o : p.prefix_o_extra + (idx - 1) * rows * kHeadDim;
                const float* sm = idx == 0 ? p.prefix_ml : p.prefix_ml_extra + (idx - 1) * rows * 2;
                float o4[4] = {0.f, 0.f, 0.f, 0.f}, m2[2] = {-INFINITY, -INFINITY}, l2[2] = {0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int gh = hg * kHeadsPerGroup + 2 * t + e;
                    if (gh >= p.group) continue;
                    const size_t ri = static_cast<size_t>(row) * p.num_q_heads + h * p.group + gh;
                    const float2 ml2 = __ldcg(reinterpret_cast<const float2*>(sm + 2 * ri));
                    m2[e] = ml2.x;
                    l2[e] = ml2.y;
                    o4[e] = __ldcg(so + ri * kHeadDim + dA);
                    o4[2 + e] = __ldcg(so + ri * kHeadDim + dB);
                }
                v[k] = make_float4(o4[0], o4[1], o4[2], o4[3]);
                mv[k] = make_float2(m2[0], m2[1]);
                lv[k] = make_float2(l2[0], l2[1]);
            }
            fold(v, mv, lv, min(kBatch, npre - base));
        }
    }
    // range of the unit's k-th partial
    auto range_k = [&](int k) -> int {
        if (!cta_merged || wa == wb) return wa + k;
        return k == 0 ? wa : (k == nseg - 1 ? wb : m0 + kDecodeWarps * (k - 1));
    };
    // the decode slots of the unit's segments
    for (int base = 0; base < nseg; base += kBatch) {
        float4 v[kBatch];
        float2 mv[kBatch], lv[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int sl = range_k(min(base + k, nseg - 1)) + u;
            v[k] = __ldcg(p.partial + (static_cast<size_t>(sl) * 8 + dt) * 32 + lane);
            mv[k] = __ldcg(reinterpret_cast<const float2*>(p.ml + static_cast<size_t>(sl) * 16 + 2 * t));
            lv[k] = __ldcg(reinterpret_cast<const float2*>(p.ml + static_cast<size_t>(sl) * 16 + 8 + 2 * t));
        }
        fold(v, mv, lv, min(kBatch, nseg - base));
    }
    const float vscale = Fp8Layout ? __ldg(p.v_scale + h * p.scale_stride) : 1.0f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int gh = hg * kHeadsPerGroup + 2 * t + e;
        if (gh >= p.group) continue;
        const float inv = vscale / (e ? L1 : L0);
        uint16_t* orow = static_cast<uint16_t*>(p.out) +
                         (static_cast<size_t>(row) * p.num_q_heads + h * p.group + gh) * kHeadDim;
        const uint16_t lo16 = from_float<OutBf16>(acc[e] * inv);
        const uint16_t hi16 = from_float<OutBf16>(acc[2 + e] * inv);
        if constexpr (Fp8Layout) {
            *reinterpret_cast<uint32_t*>(orow + 16 * dt + 2 * g) =
                static_cast<uint32_t>(lo16) | (static_cast<uint32_t>(hi16) << 16);
        } else {
            orow[16 * dt + g] = lo16;
            orow[16 * dt + g + 8] = hi16;
        }
    }
}

// Grid-stride over the units: a few CTAs per SM cover any number of units without
// waves of one-CTA SMs.  At most 112 registers per thread, so that a combine CTA
// fits beside two decode CTAs (136 registers x 128 threads each) and is resident,
// past its prologue, while the decode grid drains.  For batches of up to kCombineScanSeqs sequences every CTA first builds the
// exclusive block prefix over the sequences in shared memory, overlapping the
// decode grid's tail; the units it then visits only look it up.
// The exclusive block prefix over the sequences (batches of up to kCombineScanSeqs),
// by a 256-thread CTA into shared memory.
__device__ __forceinline__ void combine_block_prefix(const DecodeParams& p, int* pre_sum, int* warp_sum) {
    const int B = p.num_seqs;
    const int UH = p.num_kv_heads * p.head_groups;
    {
        // thread i sums sequences [per i, per (i + 1)), then a scan over threads
        const int per = (B + 255) / 256;
        const int beg = min(B, static_cast<int>(threadIdx.x) * per), end = min(B, beg + per);
        int own = 0;
        for (int i = beg; i < end; ++i) own += unit_blocks_of(p, i, UH);
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        int inc = own;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o2);
            if (lane >= o2) inc += y;
        }
        if (lane == 31) warp_sum[warp] = inc;
        __syncthreads();
        int before = 0;
        for (int k = 0; k < warp; ++k) before += warp_sum[k];
        int run = before + inc - own;              // exclusive prefix of this thread's first sequence
        for (int i = beg; i < end; ++i) {
            pre_sum[i] = run;
            run += unit_blocks_of(p, i, UH);
        }
        if (threadIdx.x == 255) pre_sum[B] = before + inc;
        __syncthreads();
    }
}

template <bool OutBf16, bool Fp8Layout, bool Cascade, int kBatch>
__global__ void __maxnreg__(112) combine_kernel(const DecodeParams p) {
    __shared__ int pre_sum[kCombineScanSeqs + 1];
    __shared__ int warp_sum[8];
    // a launch chained behind (the next layer's decode) may become resident now and
    // wait for this grid's completion with its prologue done
    grid_launch_dependents();
    const int B = p.num_seqs;
    const int UH = p.num_kv_heads * p.head_groups;
    if (B <= kCombineScanSeqs) combine_block_prefix(p, pre_sum, warp_sum);
    const long long units = static_cast<long long>(B) * UH;
    for (long long u = blockIdx.x; u < units; u += gridDim.x)
        combine_unit<OutBf16, Fp8Layout, Cascade, kBatch>(p, static_cast<int>(u), pre_sum);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        // every claim of this call is made: the next call numbers its pieces from here
        grid_dependency_wait();
        p.claim[1] = __ldcg(p.claim);
    }
}

// Cascade combine, one warp per unit: every row of a cascade has a shared-prefix
// partial, so every unit is merged, and with many units a CTA per unit would run
// them in rounds.  A lane holds the fragments of heads 2t, 2t+1 in all eight
// 16-wide slices of d; partials are folded one per round trip.
template <bool OutBf16, bool Fp8Layout>
__device__ __forceinline__ void combine_unit_warp(const DecodeParams& p, int u, const int* pre_sum) {
    const int UH = p.num_kv_heads * p.head_groups;
    const int s = u / UH, uh = u % UH;
    const int B = p.num_seqs;
    const int lane = threadIdx.x & 31, t = lane & 3, g = lane >> 2;
    long long lo = 0, T = 0;
    if (B <= kCombineScanSeqs) {
        lo = pre_sum[s];
        T = pre_sum[B];
    } else {
        grid_dependency_wait();
        lo = p.plan[s];
        T = p.plan[B];
    }
    const int nb = unit_blocks_of(p, s, UH) / UH;
    // the unit's decode partials, as in combine_unit: one per range, or with static
    // ranges one per CTA run of the ranges it spans
    int wa = 0, wb = 0, nseg = 0, m0 = 0;
    const bool cta_merged = p.dyn256 == 0;
    if (nb > 0 && T > 0) {
        const Split sp = make_split(static_cast<int>(T), p.num_workers, p.dyn256);
        const int fu = static_cast<int>(lo) + uh * nb;
        wa = sp.range_of(fu);
        wb = sp.range_of(fu + nb - 1);
        if (!cta_merged || wa == wb) {
            nseg = wb - wa + 1;
        } else {
            m0 = (wa / kDecodeWarps + 1) * kDecodeWarps;
            nseg = 2 + (m0 <= wb - 1 ? (wb - 1 - m0) / kDecodeWarps + 1 : 0);
        }
    }
    const int npre = p.first_block > 0 ? p.prefix_splits : 0;
    if (nseg + npre == 0) return;     // an empty row: the decode grid wrote its zeros
    const int h = uh / p.head_groups, hg = uh % p.head_groups;
    const int row = p.query_start_loc ? p.query_start_loc[s] : s;
    const size_t rows = static_cast<size_t>(B) * p.num_q_heads;
    auto range_k = [&](int k) -> int {
        if (!cta_merged || wa == wb) return wa + k;
        return k == 0 ? wa : (k == nseg - 1 ? wb : m0 + kDecodeWarps * (k - 1));
    };
    // partial k: the prefix segments first, then the decode slots
    auto load = [&](int k, float (&v)[8][4], float& ma, float& mb, float& la, float& lb) {
        if (k < npre) {
            const float* so = k == 0 ? p.prefix_o : p.prefix_o_extra + (k - 1) * rows * kHeadDim;
            const float* sm = k == 0 ? p.prefix_ml : p.prefix_ml_extra + (k - 1) * rows * 2;
            float mm[2] = {-INFINITY, -INFINITY}, ll[2] = {0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int gh = hg * kHeadsPerGroup + 2 * t + e;
                const bool live = gh < p.group;
                const size_t ri = static_cast<size_t>(row) * p.num_q_heads + h * p.group + (live ? gh : 0);
                if (live) {
                    const float2 ml2 = __ldcg(reinterpret_cast<const float2*>(sm + 2 * ri));
                    mm[e] = ml2.x;
                    ll[e] = ml2.y;
                }
#pragma unroll
                for (int dt = 0; dt < 8; ++dt) {
                    const int dA = Fp8Layout ? 16 * dt + 2 * g : 16 * dt + g;
                    const int dB = Fp8Layout ? dA + 1 : dA + 8;
                    v[dt][e] = live ? __ldcg(so + ri * kHeadDim + dA) : 0.f;
                    v[dt][2 + e] = live ? __ldcg(so + ri * kHeadDim + dB) : 0.f;
                }
            }
            ma = mm[0];
            mb = mm[1];
            la = ll[0];
            lb = ll[1];
        } else {
            const size_t sl = static_cast<size_t>(range_k(k - npre)) + u;
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) {
                const float4 x = __ldcg(p.partial + (sl * 8 + dt) * 32 + lane);
                v[dt][0] = x.x;
                v[dt][1] = x.y;
                v[dt][2] = x.z;
                v[dt][3] = x.w;
            }
            const float2 mv = __ldcg(reinterpret_cast<const float2*>(p.ml + sl * 16 + 2 * t));
            const float2 lv = __ldcg(reinterpret_cast<const float2*>(p.ml + sl * 16 + 8 + 2 * t));
            ma = mv.x;
            mb = mv.y;
            la = lv.x;
            lb = lv.y;
        }
    };
    if (B <= kCombineScanSeqs) grid_dependency_wait();
    float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
    float acc[8][4];
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) acc[dt][0] = acc[dt][1] = acc[dt][2] = acc[dt][3] = 0.f;
    // fold one partial into the running (M, L, acc) (padding heads may turn to NaN: never written)
    auto fold = [&](const float (&v)[8][4], float ma, float mb, float la, float lb) {
        const float n0 = fmaxf(M0, ma), n1 = fmaxf(M1, mb);
        const float r0 = exp2f(M0 - n0), r1 = exp2f(M1 - n1);      // 0 while nothing is summed
        const float w0 = exp2f(ma - n0), w1 = exp2f(mb - n1);
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
            acc[dt][0] = acc[dt][0] * r0 + v[dt][0] * w0;
            acc[dt][1] = acc[dt][1] * r1 + v[dt][1] * w1;
            acc[dt][2] = acc[dt][2] * r0 + v[dt][2] * w0;
            acc[dt][3] = acc[dt][3] * r1 + v[dt][3] * w1;
        }
        L0 = L0 * r0 + la * w0;
        L1 = L1 * r1 + lb * w1;
        M0 = n0;
        M1 = n1;
    };
    const int nall = npre + nseg;
    for (int k = 0; k < nall; ++k) {
        float v[8][4];
        float ma, mb, la, lb;
        load(k, v, ma, mb, la, lb);
        fold(v, ma, mb, la, lb);
    }
    const float vscale = Fp8Layout ? __ldg(p.v_scale + h * p.scale_stride) : 1.0f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int gh = hg * kHeadsPerGroup + 2 * t + e;
        if (gh >= p.group) continue;
        const float inv = vscale / (e ? L1 : L0);
        uint16_t* orow = static_cast<uint16_t*>(p.out) +
                         (static_cast<size_t>(row) * p.num_q_heads + h * p.group + gh) * kHeadDim;
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
            const uint16_t lo16 = from_float<OutBf16>(acc[dt][e] * inv);
            const uint16_t hi16 = from_float<OutBf16>(acc[dt][2 + e] * inv);
            if constexpr (Fp8Layout) {
                *reinterpret_cast<uint32_t*>(orow + 16 * dt + 2 * g) =
                    static_cast<uint32_t>(lo16) | (static_cast<uint32_t>(hi16) << 16);
            } else {
                orow[16 * dt + g] = lo16;
                orow[16 * dt + g + 8] = hi16;
            }
        }
    }
}

// 8 units per 256-thread CTA, one per warp.  At most 112 registers, as combine_kernel.
template <bool OutBf16, bool Fp8Layout>
__global__ void __maxnreg__(112) combine_cascade_kernel(const DecodeParams p) {
    __shared__ int pre_sum[kCombineScanSeqs + 1];
    __shared__ int warp_sum[8];
    grid_launch_dependents();
    const int B = p.num_seqs;
    const int UH = p.num_kv_heads * p.head_groups;
    if (B <= kCombineScanSeqs) combine_block_prefix(p, pre_sum, warp_sum);
    const long long units = static_cast<long long>(B) * UH;
    const long long u = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (u < units) combine_unit_warp<OutBf16, Fp8Layout>(p, static_cast<int>(u), pre_sum);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        // every claim of this call is made: the next call numbers its pieces from here
        grid_dependency_wait();
        p.claim[1] = __ldcg(p.claim);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {
// narrow: the two-stage ring of the 16-bit decode kernel (no fused slot write)
template <int Kind, bool QBf16>
void* kernel_ptr(bool append, bool dyn, bool narrow) {
    if constexpr (Kind != kKindFp8) {
        if (narrow && !append)
            return dyn ? reinterpret_cast<void*>(&decode_kernel<Kind, QBf16, true, 2>)
                       : reinterpret_cast<void*>(&decode_kernel<Kind, QBf16, false, 2>);
    }
    if (dyn)
        return append ? reinterpret_cast<void*>(&decode_append_kernel<Kind, QBf16, true>)
                      : reinterpret_cast<void*>(&decode_kernel<Kind, QBf16, true, 3>);
    return append ? reinterpret_cast<void*>(&decode_append_kernel<Kind, QBf16, false>)
                  : reinterpret_cast<void*>(&decode_kernel<Kind, QBf16, false, 3>);
}

void* decode_fn(CacheKind kind, bool q_bf16, bool append, bool dyn, bool narrow) {
    switch (kind) {
        case kKindBf16: return kernel_ptr<kKindBf16, true>(append, dyn, narrow);
        case kKindFp16: return kernel_ptr<kKindFp16, false>(append, dyn, narrow);
        case kKindFp8:
            return q_bf16 ? kernel_ptr<kKindFp8, true>(append, dyn, false)
                          : kernel_ptr<kKindFp8, false>(append, dyn, false);
    }
    return nullptr;
}

int tile_area_bytes(CacheKind kind, bool narrow) {
    switch (kind) {
        case kKindBf16:
            return narrow ? DecodeCfg<kKindBf16, 2>::kTileArea + DecodeCfg<kKindBf16, 2>::kBarBytes
                          : DecodeCfg<kKindBf16>::kTileArea + DecodeCfg<kKindBf16>::kBarBytes;
        case kKindFp16:
            return narrow ? DecodeCfg<kKindFp16, 2>::kTileArea + DecodeCfg<kKindFp16, 2>::kBarBytes
                          : DecodeCfg<kKindFp16>::kTileArea + DecodeCfg<kKindFp16>::kBarBytes;
        case kKindFp8: return DecodeCfg<kKindFp8>::kTileArea + DecodeCfg<kKindFp8>::kBarBytes;
    }
    return 0;
}
}  // namespace

size_t decode_smem_bytes(CacheKind kind, int num_seqs, bool narrow) {
    // 1 KiB alignment slack + tiles + barriers + scan array
    return 1024 + static_cast<size_t>(tile_area_bytes(kind, narrow)) + static_cast<size_t>(num_seqs + 1) * 4;
}

cudaError_t decode_prepare(CacheKind kind, bool q_bf16, bool append, bool dyn, bool narrow, size_t max_smem) {
    // the largest request a call can make (kMaxSeqs sequences), within what the
    // device allows next to the kernel's static shared memory
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, decode_fn(kind, q_bf16, append, dyn, narrow));
    if (e != cudaSuccess) return e;
    size_t want = decode_smem_bytes(kind, kMaxSeqs, narrow);
    const size_t cap = max_smem > fa.sharedSizeBytes ? max_smem - fa.sharedSizeBytes : 0;
    if (want > cap) want = cap;
    return cudaFuncSetAttribute(decode_fn(kind, q_bf16, append, dyn, narrow),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(want));
}

cudaError_t decode_occupancy(CacheKind kind, bool q_bf16, bool append, bool dyn, bool narrow, size_t smem,
                             int* ctas_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, decode_fn(kind, q_bf16, append, dyn, narrow),
                                                         kDecodeWarps * 32, smem);
}

cudaError_t launch_decode(CacheKind kind, bool q_bf16, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const DecodeParams& p, int grid, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecodeWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<CUtensorMap*>(&kmap), const_cast<CUtensorMap*>(&vmap), const_cast<DecodeParams*>(&p)};
    const void* fn = decode_fn(kind, q_bf16, p.append != 0, p.dyn256 > 0, p.narrow != 0);
    if (!fn) return cudaErrorInvalidValue;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_combine(bool out_bf16, bool fp8_cache, const DecodeParams& p, int max_ctas,
                           cudaStream_t stream) {
    const long long units = static_cast<long long>(p.num_seqs) * p.num_kv_heads * p.head_groups;
    cudaLaunchConfig_t cfg = {};
    // a cascade with more units than resident combine CTAs: one warp per unit, 8 units
    // per CTA (a CTA per unit would take them in rounds); with fewer units a CTA per unit
    // batches a unit's partials (the prefix segments of a long prompt) in one round trip
    const bool warp_units = p.cascade && units > max_ctas;
    cfg.gridDim = dim3(static_cast<unsigned>(warp_units ? (units + 7) / 8 : (units < max_ctas ? units : max_ctas)));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // slots per round trip: 8 in the cascade variant (which also folds prefix
    // partials) and where units average under 8 partials, else 10 (at most 112
    // registers either way)
    // (with static ranges a unit leaves about one partial per CTA it spans, otherwise
    // one per range)
    const long long per_slot = p.dyn256 == 0 ? 4LL * kDecodeWarps : 8LL;
    const bool wide = !p.cascade && static_cast<long long>(p.num_workers) > per_slot * units;
    auto kernel = [&](auto ob, auto f8) -> const void* {
        constexpr bool O = decltype(ob)::value, F = decltype(f8)::value;
        if (warp_units) return reinterpret_cast<const void*>(&combine_cascade_kernel<O, F>);
        if (p.cascade) return reinterpret_cast<const void*>(&combine_kernel<O, F, true, 8>);
        return wide ? reinterpret_cast<const void*>(&combine_kernel<O, F, false, 10>)
                    : reinterpret_cast<const void*>(&combine_kernel<O, F, false, 8>);
    };
    using T = std::true_type;
    using Fa = std::false_type;
    const void* fn = out_bf16 ? (fp8_cache ? kernel(T{}, T{}) : kernel(T{}, Fa{}))
                              : (fp8_cache ? kernel(Fa{}, T{}) : kernel(Fa{}, Fa{}));
    void* args[] = {const_cast<DecodeParams*>(&p)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace pa
