// Prefill chunks of a mixed batch on the 5th-generation tensor cores (sm_103a).
//
// Problem ("Basics of LLM Inference and vLLM Internals", s.6 chunked prefill;
// "The Memory Trick Behind Fast LLM Serving", "Batching does not merge the
// conversations"): row j of a chunk of q_len new tokens sits at position
// seq_len - q_len + j and attends causally to tokens 0..pos of its own sequence,
// reached through the block table.  For a prompt chunk this is a dense
// contraction of the query rows against every cached key.
//
// One CTA = two consecutive tiles A and B of 128 MMA rows each (queries x all
// heads of one KV head, so every K/V tile in shared memory serves the whole
// GQA group twice) of one chunk; keys advance 64 at a time (4 blocks) through a
// 3-stage ring.  While one softmax warpgroup works on its tile, the tensor core
// runs the other tile's products (ping-pong).
//   warp 0       producer: bulk tensor copies (TMA, 128-byte swizzle) of each
//                step's K and V blocks (16-bit caches), one lane per block
//   warp 1       one lane issues tcgen05.mma: S_X(i) = Q_X K_i^T into a double
//                buffer in tensor memory, then O_X += P_X(i-1) V_(i-1)
//   warps 2-5    softmax of tile A, warps 6-9 softmax of tile B: one thread
//                per row, S from tensor memory, causal mask, online max/sum,
//                P to shared memory; O rescaled in tensor memory only when a
//                row maximum grows by more than 2^8
//   warps 10-13  FP8 caches only: gather e4m3 rows through the block table, widen
//                them exactly to f16 and store them in the MMA layout
// Every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kTcRows = 128;                 // MMA M of one tile
constexpr int kTcKeys = 64;                  // keys per step (MMA N of S, K of PV)
constexpr int kTcBlocksPerStep = kTcKeys / kBlockSize;
constexpr int kTcStages = 3;
constexpr uint32_t kQHalf = 16384;           // Q tile: [128 rows][64 elements] per d-half
constexpr uint32_t kKvHalf = 8192;           // K or V of a step: [64 rows][64 elements] per d-half
constexpr uint32_t kOffQ = 0;                // Q_A, Q_B: 32 KiB each
constexpr uint32_t kOffStage = 65536;        // stage s: K at +32768 s, V 16 KiB after it
constexpr uint32_t kStageBytes = 32768;
constexpr uint32_t kOffP = kOffStage + kTcStages * kStageBytes;   // P_A, P_B: [128 rows][64 keys]
constexpr uint32_t kPBytes = 16384;
constexpr uint32_t kOffBars = kOffP + 2 * kPBytes;
constexpr uint32_t kBarBytes = 256;          // barriers + tensor-memory address
constexpr uint32_t kOffCum = kOffBars + kBarBytes;
constexpr uint32_t kTmemCols = 512;          // S_A 0,64  S_B 128,192  O_A 256  O_B 384
constexpr float kRescaleLog2 = 8.0f;         // lazy rescale threshold (factor 256)

// barrier indices (8 bytes each from kOffBars)
enum {
    kBarKvFull = 0,     // [3]
    kBarKvEmpty = 3,    // [3]
    kBarSFull = 6,      // [tile][2]
    kBarSFree = 10,     // [tile][2]
    kBarPFull = 14,     // [tile]
    kBarPvDone = 16,    // [tile]
    kBarQFull = 18,
    kNumBars = 19
};

template <int Kind>
struct TcCfg {
    static constexpr bool kFp8 = Kind == kKindFp8;
    static constexpr bool kMmaBf16 = Kind == kKindBf16;
    static constexpr int kWarps = kFp8 ? 14 : 10;
};

// Bounded wait by lane 0 of the warp, then an acquire by every lane.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, limit);
    ok = __shfl_sync(0xffffffffu, static_cast<int>(ok), 0) != 0;
    if (ok) mbar_try_wait(bar, parity);
    return ok;
}

}  // namespace


template <int Kind, bool QBf16>
__global__ void __launch_bounds__(TcCfg<Kind>::kWarps * 32, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const ChunkParams p) {
    using Cfg = TcCfg<Kind>;
    constexpr bool kFp8 = Cfg::kFp8;
    constexpr bool kMmaBf16 = Cfg::kMmaBf16;
    constexpr int kThreads = Cfg::kWarps * 32;

    extern __shared__ uint8_t smem_raw[];
    __shared__ int warp_tot[Cfg::kWarps];
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw_base);
    int* cum = reinterpret_cast<int*>(sm + kOffCum);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffBars + kNumBars * 8);
    auto bar = [&](int i) -> uint32_t { return sbase + kOffBars + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(bar(kBarKvFull + s), kFp8 ? 4 : 1);
            mbar_init(bar(kBarKvEmpty + s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(bar(kBarSFull + 2 * x + b), 1);
                mbar_init(bar(kBarSFree + 2 * x + b), 4);
            }
            mbar_init(bar(kBarPFull + x), 4);
            mbar_init(bar(kBarPvDone + x), 1);
        }
        mbar_init(bar(kBarQFull), 8);
        fence_barrier_init();
        if constexpr (!kFp8) {
            tmap_prefetch(&kmap);
            tmap_prefetch(&vmap);
        }
    }

    grid_dependency_wait();

    // ---- tile pairs per chunk sequence, exclusive scan -> cum ----
    const int B = p.num_seqs;
    const int QT = p.queries_per_tile;
    auto pairs_of = [&](int s) -> int {
        const int ql = p.query_start_loc[s + 1] - p.query_start_loc[s];
        return ql >= 2 ? (ql + 2 * QT - 1) / (2 * QT) : 0;
    };
    {
        const int per = (B + kThreads - 1) / kThreads;
        const int beg = min(B, static_cast<int>(threadIdx.x) * per);
        const int end = min(B, beg + per);
        int local = 0;
        for (int s = beg; s < end; ++s) local += pairs_of(s);
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
            run += pairs_of(s);
        }
        if (threadIdx.x == kThreads - 1) cum[B] = run;
    }
    __syncthreads();
    grid_launch_dependents();

    const int R = cum[B];
    if (static_cast<int>(blockIdx.x) >= R) return;
    const int tau = R - 1 - static_cast<int>(blockIdx.x);   // heaviest pairs first
    int s = 0;
    {
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cum[mid] <= tau) lo = mid; else hi = mid;
        }
        s = lo;
    }
    const int pair = tau - cum[s];
    const int h = blockIdx.y;
    const int G = p.group;
    const int q0 = p.query_start_loc[s];
    const int q_len = p.query_start_loc[s + 1] - q0;
    const int n = p.seq_lens[s];
    if (n - q_len < 0 || n > p.max_blocks * kBlockSize) {   // inconsistent lengths
        if (threadIdx.x == 0) atomicOr(p.status, kDevErrRange);
        return;
    }
    // tile X (0 = A, 1 = B): queries j_first[X] .. j_last[X]; B may be absent
    const int jf0 = 2 * pair * QT;
    const int jf1 = jf0 + QT;
    const bool has_b = jf1 < q_len;
    const int jl0 = min(q_len, jf0 + QT) - 1;
    const int jl1 = has_b ? min(q_len, jf1 + QT) - 1 : jl0;
    const int pos_last_cta = n - q_len + jl1;
    const int nsteps = pos_last_cta / kTcKeys + 1;
    const int nsteps_a = (n - q_len + jl0) / kTcKeys + 1;
    const int nblocks = pos_last_cta / kBlockSize + 1;
    const int32_t* bt = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
    auto tile_steps = [&](int x) -> int { return x == 0 ? nsteps_a : (has_b ? nsteps : 0); };

    // ---- tensor memory ----
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto tS = [&](int x, int b) -> uint32_t { return tmem + 128u * x + 64u * b; };
    auto tO = [&](int x) -> uint32_t { return tmem + 256u + 128u * x; };
    bool ok = true;

    if (warp == 0) {
        // ================= producer (16-bit caches): lane b < 4 copies block b of a step =================
        if constexpr (!kFp8) {
            auto entry = [&](int i) -> int {
                const int j = i * kTcBlocksPerStep + lane;
                int phys = 0;
                if (lane < kTcBlocksPerStep && j < nblocks) {
                    phys = __ldg(bt + j);
                    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
                        atomicOr(p.status, kDevErrRange);
                        phys = 0;
                    }
                }
                return phys;
            };
            int phys = entry(0);
            for (int i = 0; i < nsteps && ok; ++i) {
                const int st = i % kTcStages;
                const int phys_next = i + 1 < nsteps ? entry(i + 1) : 0;
                if (i >= kTcStages &&
                    !warp_wait(bar(kBarKvEmpty + st), ((i / kTcStages) - 1) & 1, p.timeout_ns)) {
                    if (lane == 0) atomicOr(p.status, kDevErrTimeout);
                    ok = false;
                    break;
                }
                const int nb = min(kTcBlocksPerStep, nblocks - i * kTcBlocksPerStep);
                const uint32_t kdst = sbase + kOffStage + st * kStageBytes;
                const uint32_t vdst = kdst + 2 * kKvHalf;
                if (lane == 0) mbar_arrive_expect_tx(bar(kBarKvFull + st), static_cast<uint32_t>(nb) * 2 * 4096);
                __syncwarp();
                if (lane < nb) {
                    const int y = (phys * p.num_kv_heads + h) * kBlockSize;
                    // block b -> rows 16b..16b+15 of each d-half
                    tma_load_2d(kdst + lane * 2048, &kmap, 0, y, bar(kBarKvFull + st));
                    tma_load_2d(kdst + kKvHalf + lane * 2048, &kmap, 64, y, bar(kBarKvFull + st));
                    tma_load_2d(vdst + lane * 2048, &vmap, 0, y, bar(kBarKvFull + st));
                    tma_load_2d(vdst + kKvHalf + lane * 2048, &vmap, 64, y, bar(kBarKvFull + st));
                }
                phys = phys_next;
            }
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t idS = umma_idesc_f16<kMmaBf16>(kTcRows, kTcKeys, false);
            constexpr uint32_t idPV = umma_idesc_f16<kMmaBf16>(kTcRows, kHeadDim, true);
            auto issue_s = [&](int x, int i) -> bool {
                const int sb = i & 1;
                if (i >= 2 && !mbar_wait_bounded(bar(kBarSFree + 2 * x + sb), ((i >> 1) - 1) & 1, p.timeout_ns))
                    return false;
                tc_fence_after();
                const uint32_t qbase = sbase + kOffQ + x * 2 * kQHalf;
                const uint32_t kbase = sbase + kOffStage + (i % kTcStages) * kStageBytes;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint64_t a = umma_desc_sw128(qbase + (kk >> 2) * kQHalf + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = umma_desc_sw128(kbase + (kk >> 2) * kKvHalf + (kk & 3) * 32, 16, 1024);
                    umma_f16(tS(x, sb), a, b, idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(bar(kBarSFull + 2 * x + sb));
                return true;
            };
            auto issue_pv = [&](int x, int j) {
                const uint32_t vbase = sbase + kOffStage + (j % kTcStages) * kStageBytes + 2 * kKvHalf;
                const uint32_t pbase = sbase + kOffP + x * kPBytes;
#pragma unroll
                for (int kk = 0; kk < kTcKeys / 16; ++kk) {
                    const uint64_t a = umma_desc_sw128(pbase + kk * 32, 16, 1024);
                    const uint64_t b = umma_desc_sw128(vbase + kk * 2048, kKvHalf, 1024);
                    umma_f16(tO(x), a, b, idPV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(bar(kBarPvDone + x));
            };
            // Event loop: poll the barriers and issue whatever is ready, P.V first (it
            // unblocks that tile's softmax), then the next S into a free buffer, so that
            // one tile never waits behind the other.  No barrier can move past the
            // phase tested here: each one's next phase needs an MMA not yet issued.
            const int zt = has_b ? 1 : 0;             // tile that zeroes V rows in the last step
            int next_s[2] = {0, 0}, next_pv[2] = {0, 0};
            ok = mbar_wait_bounded(bar(kBarQFull), 0, p.timeout_ns);
            uint64_t t_last = global_timer_ns();
            while (ok && (next_pv[0] < tile_steps(0) || next_pv[1] < tile_steps(1))) {
                bool progress = false;
                for (int x = 0; x < 2; ++x) {
                    const int j = next_pv[x];
                    if (j < tile_steps(x) && j < next_s[x] && mbar_test(bar(kBarPFull + x), j & 1)) {
                        // a 16-bit cache's last step also waits for the zeroing tile
                        const bool blocked = !kFp8 && j == nsteps - 1 && x != zt && j < tile_steps(zt) &&
                                             !(next_pv[zt] > j || mbar_test(bar(kBarPFull + zt), j & 1));
                        if (!blocked) {
                            tc_fence_after();
                            issue_pv(x, j);
                            next_pv[x] = j + 1;
                            progress = true;
                            const int other = 1 - x;
                            if (j >= tile_steps(other) || next_pv[other] > j)
                                umma_commit(bar(kBarKvEmpty + (j % kTcStages)));   // both tiles done with stage
                        }
                    }
                }
                for (int x = 0; x < 2; ++x) {
                    const int i = next_s[x];
                    if (i < tile_steps(x) &&
                        mbar_test(bar(kBarKvFull + i % kTcStages), (i / kTcStages) & 1) &&
                        (i < 2 || mbar_test(bar(kBarSFree + 2 * x + (i & 1)), ((i >> 1) - 1) & 1))) {
                        ok = issue_s(x, i);
                        next_s[x] = i + 1;
                        progress = true;
                    }
                }
                if (progress) {
                    t_last = global_timer_ns();
                } else {
                    __nanosleep(32);          // leave issue slots to the softmax warps of this sub-partition
                    if (global_timer_ns() - t_last > p.timeout_ns) ok = false;
                }
            }
            if (!ok) atomicOr(p.status, kDevErrTimeout);
        }
        __syncwarp();
    } else if (warp < 10) {
        // ================= softmax: warps 2-5 tile A, 6-9 tile B; thread = one MMA row =================
        const int x = warp < 6 ? 0 : 1;
        const int quarter = warp & 3;                  // tensor-memory lanes 32 quarter .. + 31
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int steps = tile_steps(x);
        const int jf = x == 0 ? jf0 : jf1;
        const int jl = x == 0 ? jl0 : jl1;
        const int jq = r / G;
        const bool live = steps > 0 && r < QT * G && jf + jq <= jl;
        const int pos_first = n - q_len + jf;
        const int pos = live ? n - q_len + jf + jq : n - q_len + jl;
        const size_t qrow = (static_cast<size_t>(q0 + (live ? jf + jq : jf0)) * p.num_q_heads + h * G +
                             (live ? r % G : 0)) * kHeadDim;
        // Q row -> shared memory (MMA input type), 128-byte swizzle, two d-halves
        {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + qrow);
            uint8_t* qdst = sm + kOffQ + x * 2 * kQHalf;
#pragma unroll 4
            for (int c = 0; c < 16; ++c) {
                uint4 v = live ? src[c] : make_uint4(0, 0, 0, 0);
                if constexpr (kFp8 && QBf16) {
                    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack2<false>(to_float<true>(w[e] & 0xffffu), to_float<true>(w[e] >> 16));
                    v = make_uint4(w[0], w[1], w[2], w[3]);
                }
                *reinterpret_cast<uint4*>(qdst + (c >> 3) * kQHalf + sw128_offset(r, (c & 7) * 8)) = v;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarQFull));
        }
        const float kscale = kFp8 ? __ldg(p.k_scale) : 1.0f;
        const float vscale = kFp8 ? __ldg(p.v_scale) : 1.0f;
        const float s_log2 = p.scale_log2 * kscale;
        const bool pos_scale = s_log2 >= 0.f;
        float m_used = -INFINITY, l = 0.f;
        for (int i = 0; i < steps && ok; ++i) {
            const int sb = i & 1;
            if (!warp_wait(bar(kBarSFull + 2 * x + sb), (i >> 1) & 1, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int key0 = i * kTcKeys;
            const bool need_mask = key0 + kTcKeys - 1 > pos_first;
            const int lim = pos - key0;                 // columns > lim are masked
            const uint32_t s_addr = tS(x, sb) + lane_off;
            // pass 1: row maximum of the raw scores (scale > 0 keeps the order, < 0 reverses it)
            float hi = -INFINITY, lo = INFINITY;
#pragma unroll
            for (int c = 0; c < kTcKeys / 32; ++c) {
                uint32_t sv[32];
                tmem_ld32(s_addr + 32 * c, sv);
                tmem_wait_ld();
                if (!need_mask) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        hi = fmaxf(hi, __uint_as_float(sv[e]));
                        lo = fminf(lo, __uint_as_float(sv[e]));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const bool keep = 32 * c + e <= lim;
                        hi = fmaxf(hi, keep ? __uint_as_float(sv[e]) : -INFINITY);
                        lo = fminf(lo, keep ? __uint_as_float(sv[e]) : INFINITY);
                    }
                }
            }
            const float mx = (pos_scale ? hi : lo) * s_log2;   // -inf when every column is masked
            const bool need = mx > m_used + kRescaleLog2;
            const bool resc = __any_sync(0xffffffffu, need);
            const float m_new = need ? fmaxf(m_used, mx) : m_used;
            const float alpha = ex2_approx(m_used - m_new);    // 0 on the first step, 1 when kept
            m_used = m_new;
            // P buffer and O are busy until this tile's previous P.V is done
            if (i >= 1) {
                if (!warp_wait(bar(kBarPvDone + x), (i - 1) & 1, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (resc) {
#pragma unroll 1
                    for (int c = 0; c < kHeadDim / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(tO(x) + lane_off + 32 * c, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st32(tO(x) + lane_off + 32 * c, ov);
                    }
                    tmem_wait_st();
                }
            }
            // pass 2: p = 2^(s * scale - m), stored as the A operand of P.V
            float sum = 0.f;
            const float neg_m = -m_new;
            uint8_t* prow = sm + kOffP + x * kPBytes;
#pragma unroll
            for (int c = 0; c < kTcKeys / 32; ++c) {
                uint32_t sv[32];
                tmem_ld32(s_addr + 32 * c, sv);
                tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int e = 8 * q4 + 2 * k;
                        float p0 = ex2_approx(fmaf(__uint_as_float(sv[e]), s_log2, neg_m));
                        float p1 = ex2_approx(fmaf(__uint_as_float(sv[e + 1]), s_log2, neg_m));
                        if (need_mask) {
                            p0 = 32 * c + e <= lim ? p0 : 0.f;
                            p1 = 32 * c + e + 1 <= lim ? p1 : 0.f;
                        }
                        sum += p0 + p1;
                        w[k] = pack2<kMmaBf16>(p0, p1);
                    }
                    *reinterpret_cast<uint4*>(prow + sw128_offset(r, (4 * c + q4) * 8)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarSFree + 2 * x + sb));
            l = l * alpha + sum;
            if constexpr (!kFp8) {
                // keys past the CTA's last position get P = 0, but their V rows hold unloaded
                // (stale) or poisoned bytes and 0 x NaN is NaN: the last tile zeroes them
                if (i == nsteps - 1 && x == (has_b ? 1 : 0)) {
                    const int st = i % kTcStages;
                    if (!warp_wait(bar(kBarKvFull + st), (i / kTcStages) & 1, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    if (r < kTcKeys && key0 + r > pos_last_cta) {
                        uint8_t* vrow = sm + kOffStage + st * kStageBytes + 2 * kKvHalf + r * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            *reinterpret_cast<uint4*>(vrow + 16 * c) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4*>(vrow + kKvHalf + 16 * c) = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarPFull + x));
        }
        // ---- epilogue: O / l ----
        if (steps > 0) {
            if (ok && warp_wait(bar(kBarPvDone + x), (steps - 1) & 1, p.timeout_ns)) {
                tc_fence_after();
                const float inv = vscale / l;
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + qrow);
#pragma unroll 1
                for (int c = 0; c < kHeadDim / 32; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(tO(x) + lane_off + 32 * c, ov);
                    tmem_wait_ld();
                    if (live) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint32_t w[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                w[k] = static_cast<uint32_t>(from_float<QBf16>(__uint_as_float(ov[8 * e + 2 * k]) * inv)) |
                                       (static_cast<uint32_t>(from_float<QBf16>(__uint_as_float(ov[8 * e + 2 * k + 1]) * inv)) << 16);
                            dst[4 * c + e] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            } else if (lane == 0) {
                atomicOr(p.status, kDevErrTimeout);
            }
        }
    } else if constexpr (kFp8) {
        // ================= FP8 converters: thread = half a key row (64 d) of the step =================
        const int c = threadIdx.x - 10 * 32;           // 0..127
        const int krow = c >> 1;                       // key within the step
        const int half = c & 1;                        // d-half
        const uint8_t* kc = static_cast<const uint8_t*>(p.k_cache);
        const uint8_t* vc = static_cast<const uint8_t*>(p.v_cache);
        auto load_row = [&](int i, uint4 (&kx)[4], uint4 (&vx)[4]) {
            const int key = i * kTcKeys + krow;
            if (key <= pos_last_cta) {      // later keys get P = 0: store zeros
                int phys = __ldg(bt + (key >> 4));
                if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
                    atomicOr(p.status, kDevErrRange);
                    phys = 0;
                }
                const size_t off =
                    ((static_cast<size_t>(phys) * p.num_kv_heads + h) * kBlockSize + (key & 15)) * kHeadDim + 64 * half;
                const uint4* ks = reinterpret_cast<const uint4*>(kc + off);
                const uint4* vs = reinterpret_cast<const uint4*>(vc + off);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    kx[e] = __ldg(ks + e);
                    vx[e] = __ldg(vs + e);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) kx[e] = vx[e] = make_uint4(0, 0, 0, 0);
            }
        };
        auto widen_store = [&](uint8_t* dst, const uint4 (&x4)[4]) {
            // 64 e4m3 codes (d = 64 half + 16e ..) -> exact f16, 128-byte swizzle
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t w[4] = {x4[e].x, x4[e].y, x4[e].z, x4[e].w};
                uint32_t f[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    f[2 * k] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xffffu));
                    f[2 * k + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16));
                }
                *reinterpret_cast<uint4*>(dst + half * kKvHalf + sw128_offset(krow, 16 * e)) =
                    make_uint4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<uint4*>(dst + half * kKvHalf + sw128_offset(krow, 16 * e + 8)) =
                    make_uint4(f[4], f[5], f[6], f[7]);
            }
        };
        uint4 kx[4], vx[4], kn[4], vn[4];
        load_row(0, kx, vx);
        for (int i = 0; i < nsteps && ok; ++i) {
            const int st = i % kTcStages;
            if (i + 1 < nsteps) load_row(i + 1, kn, vn);          // in flight while this step converts
            if (i >= kTcStages &&
                !warp_wait(bar(kBarKvEmpty + st), ((i / kTcStages) - 1) & 1, p.timeout_ns)) {
                ok = false;
                break;
            }
            uint8_t* kdst = sm + kOffStage + st * kStageBytes;
            widen_store(kdst, kx);
            widen_store(kdst + 2 * kKvHalf, vx);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarKvFull + st));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kx[e] = kn[e];
                vx[e] = vn[e];
            }
        }
        if (!ok && lane == 0) atomicOr(p.status, kDevErrTimeout);
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {
void* chunk_tc_fn(CacheKind kind, bool q_bf16) {
    switch (kind) {
        case kKindBf16: return reinterpret_cast<void*>(&chunk_tc_kernel<kKindBf16, true>);
        case kKindFp16: return reinterpret_cast<void*>(&chunk_tc_kernel<kKindFp16, false>);
        case kKindFp8:
            return q_bf16 ? reinterpret_cast<void*>(&chunk_tc_kernel<kKindFp8, true>)
                          : reinterpret_cast<void*>(&chunk_tc_kernel<kKindFp8, false>);
    }
    return nullptr;
}
}  // namespace

size_t chunk_smem_bytes(CacheKind, int num_seqs) {
    return 1024 + kOffCum + static_cast<size_t>(num_seqs + 1) * 4;
}

int chunk_rows() { return kTcRows; }

int chunk_tiles_per_cta() { return 2; }

cudaError_t chunk_prepare(CacheKind kind, bool q_bf16, size_t max_smem) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, chunk_tc_fn(kind, q_bf16));
    if (e != cudaSuccess) return e;
    size_t want = chunk_smem_bytes(kind, kMaxSeqs);
    const size_t cap = max_smem > fa.sharedSizeBytes ? max_smem - fa.sharedSizeBytes : 0;
    if (want > cap) want = cap;
    return cudaFuncSetAttribute(chunk_tc_fn(kind, q_bf16), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(want));
}

cudaError_t launch_chunk(CacheKind kind, bool q_bf16, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         const ChunkParams& p, int grid_x, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, p.num_kv_heads);
    cfg.blockDim = dim3(kind == kKindFp8 ? TcCfg<kKindFp8>::kWarps * 32 : TcCfg<kKindBf16>::kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (kind) {
        case kKindBf16: return cudaLaunchKernelEx(&cfg, chunk_tc_kernel<kKindBf16, true>, kmap, vmap, p);
        case kKindFp16: return cudaLaunchKernelEx(&cfg, chunk_tc_kernel<kKindFp16, false>, kmap, vmap, p);
        case kKindFp8:
            return q_bf16 ? cudaLaunchKernelEx(&cfg, chunk_tc_kernel<kKindFp8, true>, kmap, vmap, p)
                          : cudaLaunchKernelEx(&cfg, chunk_tc_kernel<kKindFp8, false>, kmap, vmap, p);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pa
