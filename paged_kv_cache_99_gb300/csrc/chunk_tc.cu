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
// GQA group twice) of one chunk; keys advance 128 at a time (8 blocks).  Both
// products run at N = 128 (a kind::f16 MMA with M = 128, N = 128, K = 16 takes
// the tensor core 64 cycles): S = Q K^T over 128 keys and O += P V over
// d = 128.  While one softmax warpgroup works on its tile, the tensor core runs
// the other tile's products (ping-pong).  Twelve warps, three warpgroups:
//   warp 0       producer: bulk tensor copies (TMA, 128-byte swizzle) of each
//                step's K blocks and V blocks (16-bit caches) into separate
//                2-stage rings, one lane per block, K of step i+1 before V of i;
//                it zeroes the V rows past the CTA's last key in the last step
//   warp 1       one lane issues tcgen05.mma in a fixed order: per step
//                O_A += P_A(i) V_i, S_A(i+1) = Q_A K_{i+1}^T, then the same for
//                tile B (P read from tensor memory).  With 16-bit caches it takes
//                V_i and K_{i+1} before it waits for P, polls for P, and issues
//                the P.V of a step's first 64 keys while the softmax still works
//                on the other 64
//   warps 2, 3   FP8 caches only: gather e4m3 rows through the block table,
//                widen them exactly to f16 and store them in the MMA layout
//   warps 4-7    softmax of tile A, warps 8-11 softmax of tile B: one thread
//                per row holds its 128 scores in registers (one tensor-memory
//                read per step), causal mask, online max/sum, P (16-bit)
//                written back over the columns of S, with 16-bit caches released
//                in two halves of 64 keys; O rescaled in tensor memory (before
//                any of the step's P is released) only when a row maximum grows
//                by more than 2^8
// Warps 0-3 give registers to the softmax warpgroups (setmaxnreg).
// Per tile the chain is S(i) -> softmax(i) -> P.V(i) -> S(i+1): S(i+1) reuses
// the columns P(i) sits in, and the tensor core runs one thread's MMAs in
// order, so the completion of S(i+1) also means P.V(i) is done.
// Every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kTcRows = 128;                 // MMA M of one tile
constexpr int kTcKeys = 128;                 // keys per step (MMA N of S, K of P.V)
constexpr int kKStages = 2;                  // K ring (its copies run a step ahead of V's)
constexpr int kVStages = 2;                  // V ring
constexpr uint32_t kQHalf = 16384;           // Q tile: [128 rows][64 elements] per d-half
constexpr uint32_t kKvHalf = 16384;          // K or V of a step: [128 keys][64 elements] per d-half
constexpr uint32_t kKvBytes = 2 * kKvHalf;
constexpr uint32_t kOffQ = 0;                // Q_A, Q_B: 32 KiB each
constexpr uint32_t kOffK = 65536;            // K stages, 32 KiB each
constexpr uint32_t kOffV = kOffK + kKStages * kKvBytes;       // V stages, 32 KiB each
constexpr uint32_t kOffBars = kOffV + kVStages * kKvBytes;
constexpr uint32_t kBarBytes = 256;          // barriers + tensor-memory address
constexpr uint32_t kTmemCols = 512;          // S_A/P_A 0  S_B/P_B 128  O_A 256  O_B 384
constexpr float kRescaleLog2 = 8.0f;         // lazy rescale threshold (factor 256)
constexpr int kRegsFront = 104;              // registers per thread of warps 0-3 after the split
constexpr int kRegsSoftmax = 200;            // ... and of the softmax warps 4-11
static_assert(128 * kRegsFront + 256 * kRegsSoftmax <= 384 * 168, "register split above the launch total");

template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// barrier indices (8 bytes each from kOffBars)
enum {
    kBarKFull = 0,                          // [K stage]
    kBarKEmpty = kBarKFull + kKStages,      // [K stage]
    kBarVFull = kBarKEmpty + kKStages,      // [V stage]
    kBarVEmpty = kBarVFull + kVStages,      // [V stage]
    kBarSFull = kBarVEmpty + kVStages,      // [tile]
    kBarPFull = kBarSFull + 2,              // [tile]
    kBarPHalf = kBarPFull + 2,              // [tile] 16-bit caches: P of the step's first 64 keys stored
    kBarPvDone = kBarPHalf + 2,             // [tile]
    kBarQFull = kBarPvDone + 2,
    kBarVZero = kBarQFull + 1,              // 16-bit caches: V rows past the CTA's last key zeroed
    kNumBars = kBarVZero + 1
};
static_assert(kNumBars * 8 + 4 <= kBarBytes, "barriers");

template <int Kind>
struct TcCfg {
    static constexpr bool kFp8 = Kind == kKindFp8;
    static constexpr bool kMmaBf16 = Kind == kKindBf16;
    // warp 0: TMA producer (16-bit caches); 1: MMA issuer; 2-3: FP8 converters;
    // 4-7: softmax of tile A; 8-11: softmax of tile B.  Three warps share each
    // sub-partition's registers, which caps a thread at 168 at launch; the first
    // warpgroup then hands registers to the two softmax warpgroups.
    static constexpr int kWarps = 12;
};

// Bounded wait by lane 0 of the warp, then an acquire by every lane.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, limit);
    ok = __shfl_sync(0xffffffffu, static_cast<int>(ok), 0) != 0;
    if (ok) mbar_try_wait(bar, parity);
    return ok;
}

// Bounded wait that polls with the non-suspending test: for the MMA issuer, which
// must start the products the moment a softmax releases P.
__device__ __forceinline__ bool mbar_poll_bounded(uint32_t bar, uint32_t parity, uint64_t limit) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int k = 0; k < 64; ++k)
            if (mbar_test(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit) return false;
    }
}

// Three-input maximum / minimum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// 16 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
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
    __shared__ int pick[2];                  // this CTA's chunk sequence and tile pair
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (sbase - raw_base);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffBars + kNumBars * 8);
    auto bar = [&](int i) -> uint32_t { return sbase + kOffBars + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(bar(kBarKFull + s), kFp8 ? 2 : 1);
            mbar_init(bar(kBarKEmpty + s), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(bar(kBarVFull + s), kFp8 ? 2 : 1);
            mbar_init(bar(kBarVEmpty + s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(kBarSFull + x), 1);
            mbar_init(bar(kBarPFull + x), 4);
            mbar_init(bar(kBarPHalf + x), 4);
            mbar_init(bar(kBarPvDone + x), 1);
        }
        mbar_init(bar(kBarQFull), 8);
        mbar_init(bar(kBarVZero), 1);
        fence_barrier_init();
        if constexpr (!kFp8) {
            tmap_prefetch(&kmap);
            tmap_prefetch(&vmap);
        }
    }

    grid_dependency_wait();

    const int B = p.num_seqs;
    const int QT = p.queries_per_tile;
    // grid x = tile-pair slot x KV head, slot-major: every head's heaviest pair is
    // dispatched first, and the slots past the batch's pairs (the host bounds the
    // pair count without reading the query lengths) come last
    const int h = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.num_kv_heads));
    const int slot = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.num_kv_heads));
    const bool prefix = p.prefix_keys > 0;
    int s = 0, pair = 0, q0 = 0, q_len = 0, n = 0;
    if (!prefix) {
        // ---- tile pairs per chunk sequence: exclusive scan over contiguous runs of
        // sequences per thread; the thread whose run holds this CTA's pair names it ----
        auto pairs_of = [&](int sq) -> int {
            const int ql = p.query_start_loc[sq + 1] - p.query_start_loc[sq];
            return ql >= 2 ? (ql + 2 * QT - 1) / (2 * QT) : 0;
        };
        {
            const int per = (B + kThreads - 1) / kThreads;
            const int beg = min(B, static_cast<int>(threadIdx.x) * per);
            const int end = min(B, beg + per);
            int local = 0;
            for (int sq = beg; sq < end; ++sq) local += pairs_of(sq);
            int incl = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) warp_tot[warp] = incl;
            __syncthreads();
            int run = incl - local, total = 0;
            for (int w = 0; w < Cfg::kWarps; ++w) {
                run += w < warp ? warp_tot[w] : 0;
                total += warp_tot[w];
            }
            const int tau = total - 1 - slot;   // heaviest pairs first
            if (tau >= run && tau < run + local) {
                for (int sq = beg; sq < end; ++sq) {
                    const int np = pairs_of(sq);
                    if (tau < run + np) {
                        pick[0] = sq;
                        pick[1] = tau - run;
                        break;
                    }
                    run += np;
                }
            }
            if (tau < 0) pick[0] = -1;          // every thread agrees: no pair for this CTA
        }
        __syncthreads();
        grid_launch_dependents();

        s = pick[0];
        if (s < 0) return;
        pair = pick[1];
        q0 = p.query_start_loc[s];
        q_len = p.query_start_loc[s + 1] - q0;
        n = p.seq_lens[s];
        if (q0 < 0 || q_len < 0 || q0 + q_len > p.total_rows ||    // rows outside q
            n - q_len < 0 || n > p.max_blocks * p.block_size) {    // inconsistent lengths
            if (threadIdx.x == 0) atomicOr(p.status, kDevErrRange);
            return;
        }
    } else {
        // ---- prefix mode: query j is the decode row of sequence j; keys are the
        // shared prefix, read through sequence 0's table ----
        grid_launch_dependents();
        pair = slot;
        q_len = B;
        n = p.prefix_keys;
        if (2 * pair * QT >= B) return;
        if (n > p.max_blocks * p.block_size) {
            if (threadIdx.x == 0) atomicOr(p.status, kDevErrRange);
            return;
        }
    }
    const int G = p.group;
    // position of query j: causal chunk rows follow the cached tokens; in prefix mode
    // every row sits after the whole prefix
    auto qpos = [&](int j) -> int { return prefix ? n - 1 : n - q_len + j; };
    // tile X (0 = A, 1 = B): queries j_first[X] .. j_last[X]; B may be absent
    const int jf0 = 2 * pair * QT;
    const int jf1 = jf0 + QT;
    const bool has_b = jf1 < q_len;
    const int jl0 = min(q_len, jf0 + QT) - 1;
    const int jl1 = has_b ? min(q_len, jf1 + QT) - 1 : jl0;
    const int pos_last_cta = qpos(jl1);
    // steps of 128 keys this CTA covers: all up to its last position, or in prefix
    // mode the key segment blockIdx.z of prefix_steps steps (its own partial)
    int step0 = 0;
    int nsteps = pos_last_cta / kTcKeys + 1;
    int nsteps_a = qpos(jl0) / kTcKeys + 1;
    if (prefix && p.prefix_steps > 0) {
        step0 = static_cast<int>(blockIdx.z) * p.prefix_steps;
        nsteps = nsteps_a = max(min(nsteps - step0, p.prefix_steps), 0);
    }
    const int32_t* bt = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
    auto tile_steps = [&](int x) -> int { return x == 0 ? nsteps_a : (has_b ? nsteps : 0); };

    // ---- tensor memory ----
    if (warp == 1) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto tS = [&](int x) -> uint32_t { return tmem + 128u * x; };          // S, then P over its first 64 columns
    auto tO = [&](int x) -> uint32_t { return tmem + 256u + 128u * x; };
    bool ok = true;

    // 384 threads x 168 registers at launch = 128 x kRegsFront + 256 x kRegsSoftmax:
    // each warpgroup changes its share before it branches into its roles
    if (warp < 4) {
        setmaxnreg_dec<kRegsFront>();
        if (!kFp8 && warp == 0) {
            // ================= producer (16-bit caches) =================
            // A step's keys arrive as pieces of R = min(block size, 16) rows, one per lane:
            // piece c of the step holds keys c R .. c R + R - 1, read from table entry
            // key / bs at row key mod bs, and lands in rows c R.. of each d-half.
            {
                const int bsh = p.block_shift;
                const int rsh = min(bsh, 4);                          // log2(R)
                const int per_step = kTcKeys >> rsh;                  // pieces per step: 8 or 16
                const int npieces = (pos_last_cta >> rsh) + 1;        // pieces up to the CTA's last key
                auto entry = [&](int i) -> int {
                    const int c = (step0 + i) * per_step + lane;
                    int y = 0;
                    if (lane < per_step && c < npieces) {
                        const int key = c << rsh;
                        int phys = __ldg(bt + (key >> bsh));
                        if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
                            atomicOr(p.status, kDevErrRange);
                            phys = 0;
                        }
                        y = ((phys * p.num_kv_heads + h) << bsh) + (key & (p.block_size - 1));
                    }
                    return y;
                };
                auto copy = [&](const CUtensorMap* map, uint32_t dst, uint32_t full, int np, int y) {
                    if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(np) * 2 * (128u << rsh));
                    __syncwarp();
                    if (lane < np) {
                        tma_load_2d(dst + (lane << rsh) * 128, map, 0, y, full);
                        tma_load_2d(dst + kKvHalf + (lane << rsh) * 128, map, 64, y, full);
                    }
                };
                // order K(0), K(1), V(0), K(2), V(1), ...: each K a step ahead of its V
                auto pieces = [&](int i) { return min(per_step, npieces - (step0 + i) * per_step); };
                int y_v = entry(0);
                if (nsteps > 0) copy(&kmap, sbase + kOffK, bar(kBarKFull), pieces(0), y_v);
                int y_k = nsteps > 1 ? entry(1) : 0;
                for (int i = 0; i < nsteps && ok; ++i) {
                    const int y_after = i + 2 < nsteps ? entry(i + 2) : 0;
                    const int ik = i + 1;
                    if (ik < nsteps) {
                        const int st = ik % kKStages;
                        if (ik >= kKStages && !warp_wait(bar(kBarKEmpty + st), ((ik / kKStages) - 1) & 1, p.timeout_ns)) {
                            ok = false;
                            break;
                        }
                        copy(&kmap, sbase + kOffK + st * kKvBytes, bar(kBarKFull + st), pieces(ik), y_k);
                    }
                    const int st = i % kVStages;
                    if (i >= kVStages && !warp_wait(bar(kBarVEmpty + st), ((i / kVStages) - 1) & 1, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    copy(&vmap, sbase + kOffV + st * kKvBytes, bar(kBarVFull + st), pieces(i), y_v);
                    y_v = y_k;
                    y_k = y_after;
                }
                // keys past the CTA's last position get P = 0, but their V rows hold unloaded
                // (stale) or poisoned bytes and 0 x NaN is NaN: once the last step's V has
                // landed, its rows past that position are zeroed before any P.V reads them
                const int last = nsteps - 1;
                if (ok && last >= 0) {
                    const int st = last % kVStages;
                    if (!warp_wait(bar(kBarVFull + st), (last / kVStages) & 1, p.timeout_ns)) {
                        ok = false;
                    } else {
                        const int first = pos_last_cta - (step0 + last) * kTcKeys + 1;   // first row to zero
                        uint8_t* vst = sm + kOffV + st * kKvBytes;
                        for (int r = max(first, 0) + lane; r < kTcKeys; r += 32) {
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                *reinterpret_cast<uint4*>(vst + r * 128 + 16 * c) = make_uint4(0, 0, 0, 0);
                                *reinterpret_cast<uint4*>(vst + kKvHalf + r * 128 + 16 * c) = make_uint4(0, 0, 0, 0);
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(kBarVZero));
                    }
                }
                if (!ok && lane == 0) atomicOr(p.status, kDevErrTimeout);
            }
        } else if (warp == 1) {
            // ================= MMA issuer =================
            if (lane == 0) {
                constexpr uint32_t idS = umma_idesc_f16<kMmaBf16>(kTcRows, kTcKeys, false);
                constexpr uint32_t idPV = umma_idesc_f16<kMmaBf16>(kTcRows, kHeadDim, true);
                auto issue_s = [&](int x, int i) {
                    const uint32_t qbase = sbase + kOffQ + x * 2 * kQHalf;
                    const uint32_t kbase = sbase + kOffK + (i % kKStages) * kKvBytes;
#pragma unroll
                    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                        const uint64_t a = umma_desc_sw128(qbase + (kk >> 2) * kQHalf + (kk & 3) * 32, 16, 1024);
                        const uint64_t b = umma_desc_sw128(kbase + (kk >> 2) * kKvHalf + (kk & 3) * 32, 16, 1024);
                        umma_f16(tS(x), a, b, idS, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(kBarSFull + x));
                };
                // P.V over keys 64 half .. 64 half + 63 (half = 0, 1), or all 128 (half = -1)
                auto issue_pv = [&](int x, int j, int half) {
                    const uint32_t vbase = sbase + kOffV + (j % kVStages) * kKvBytes;
                    const int kk0 = half > 0 ? kTcKeys / 32 : 0;
                    const int kk1 = half == 0 ? kTcKeys / 32 : kTcKeys / 16;
#pragma unroll
                    for (int kk = 0; kk < kTcKeys / 16; ++kk) {
                        if (kk < kk0 || kk >= kk1) continue;
                        // V is MN-major: d-halves kKvHalf apart, 16 keys = 2 KiB
                        const uint64_t b = umma_desc_sw128(vbase + kk * 2048, kKvHalf, 1024);
                        umma_f16_ts(tO(x), tS(x) + 8 * kk, b, idPV, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                };
                // Fixed order: per step, P.V(i) of A and A's S(i+1) right behind it (it
                // reuses the columns P(i) sat in), then the same for B.  Tile A runs about
                // half a step ahead of B, so this is the order in which the inputs become
                // ready.
                const int na = tile_steps(0), nb = tile_steps(1), nmax = na > nb ? na : nb;
                auto wait = [&](uint32_t b, uint32_t par) -> bool {
                    if (ok && !mbar_wait_bounded(b, par, p.timeout_ns)) ok = false;
                    return ok;
                };
                auto poll = [&](uint32_t b, uint32_t par) -> bool {
                    if (ok && !mbar_poll_bounded(b, par, p.timeout_ns)) ok = false;
                    return ok;
                };
                if (wait(bar(kBarQFull), 0) && nmax > 0 && wait(bar(kBarKFull), 0)) {
                    tc_fence_after();
                    if (na > 0) issue_s(0, 0);
                    if (nb > 0) issue_s(1, 0);
                    umma_commit(bar(kBarKEmpty));
                }
                for (int i = 0; i < nmax && ok; ++i) {
                    const int sv = i % kVStages, sk = (i + 1) % kKStages;
                    if constexpr (!kFp8) {
                        // V_i and K_{i+1} are copied long before a softmax releases P(i):
                        // take them first, so that nothing stands between P and its products
                        if (!wait(bar(kBarVFull + sv), (i / kVStages) & 1) ||
                            (i == nsteps - 1 && !wait(bar(kBarVZero), 0)) ||
                            (i + 1 < nmax && !wait(bar(kBarKFull + sk), ((i + 1) / kKStages) & 1)))
                            break;
                    }
                    for (int x = 0; x < 2 && ok; ++x) {
                        if (i >= tile_steps(x)) continue;
                        if constexpr (!kFp8) {
                            // P.V of the first 64 keys while the softmax works on the rest
                            if (!poll(bar(kBarPHalf + x), i & 1)) break;
                            tc_fence_after();
                            issue_pv(x, i, 0);
                            if (!poll(bar(kBarPFull + x), i & 1)) break;
                            tc_fence_after();
                            issue_pv(x, i, 1);
                        } else {
                            // the converters widen K_{i+1} after V_i: K is taken after the P.V
                            if (!wait(bar(kBarPFull + x), i & 1) || !wait(bar(kBarVFull + sv), (i / kVStages) & 1)) break;
                            tc_fence_after();
                            issue_pv(x, i, -1);
                        }
                        if (i + 1 == tile_steps(x)) umma_commit(bar(kBarPvDone + x));
                        if (i + 1 < tile_steps(x)) {
                            if (kFp8 && !wait(bar(kBarKFull + sk), ((i + 1) / kKStages) & 1)) break;
                            tc_fence_after();
                            issue_s(x, i + 1);
                        }
                    }
                    if (!ok) break;
                    // every P.V(i) is issued: V_i is free; every S(i + 1): K_{i+1} is free
                    umma_commit(bar(kBarVEmpty + sv));
                    if (i + 1 < nmax) umma_commit(bar(kBarKEmpty + sk));
                }
                if (!ok) atomicOr(p.status, kDevErrTimeout);
            }
            __syncwarp();
        } else if (kFp8 && (warp == 2 || warp == 3)) {
            // ================= FP8 converters: warps 2 and 3 =================
            // A step's K (and its V) is two items of 64 keys; thread = one key row (128 d)
            // of an item.  Items are fetched two ahead, in the order K(i) 0, K(i) 1,
            // V(i) 0, V(i) 1, K(i+1) 0, ...
            const int krow = warp == 2 ? lane : 32 + lane;     // key within the item
            auto load_item = [&](const uint8_t* cache, int i, int u, uint4 (&x8)[8]) {
                const int key = (step0 + i) * kTcKeys + 64 * u + krow;
                if (i < nsteps && key <= pos_last_cta) {      // later keys get P = 0: store zeros
                    int phys = __ldg(bt + (key >> p.block_shift));
                    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
                        atomicOr(p.status, kDevErrRange);
                        phys = 0;
                    }
                    const size_t off = (((static_cast<size_t>(phys) * p.num_kv_heads + h) << p.block_shift) +
                                        (key & (p.block_size - 1))) * kHeadDim;
                    const uint4* src = reinterpret_cast<const uint4*>(cache + off);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x8[e] = __ldg(src + e);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) x8[e] = make_uint4(0, 0, 0, 0);
                }
            };
            auto widen_store = [&](uint8_t* stage, int u, const uint4 (&x8)[8]) {
                // 128 e4m3 codes -> exact f16, two d-halves, 128-byte swizzle
                const int row = 64 * u + krow;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t w[4] = {x8[e].x, x8[e].y, x8[e].z, x8[e].w};
                    uint32_t f[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        f[2 * k] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] & 0xffffu));
                        f[2 * k + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> 16));
                    }
                    uint8_t* dst = stage + (e >> 2) * kKvHalf;
                    *reinterpret_cast<uint4*>(dst + sw128_offset(row, 16 * (e & 3))) = make_uint4(f[0], f[1], f[2], f[3]);
                    *reinterpret_cast<uint4*>(dst + sw128_offset(row, 16 * (e & 3) + 8)) = make_uint4(f[4], f[5], f[6], f[7]);
                }
            };
            const uint8_t* kc = static_cast<const uint8_t*>(p.k_cache);
            const uint8_t* vc = static_cast<const uint8_t*>(p.v_cache);
            uint4 xa[8], xb[8];
            load_item(kc, 0, 0, xa);
            load_item(kc, 0, 1, xb);
            for (int i = 0; i < nsteps && ok; ++i) {
                const int sk = i % kKStages, sv = i % kVStages;
                if (i >= kKStages && !warp_wait(bar(kBarKEmpty + sk), ((i / kKStages) - 1) & 1, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                uint8_t* kdst = sm + kOffK + sk * kKvBytes;
                widen_store(kdst, 0, xa);
                load_item(vc, i, 0, xa);
                widen_store(kdst, 1, xb);
                load_item(vc, i, 1, xb);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarKFull + sk));
                if (i >= kVStages && !warp_wait(bar(kBarVEmpty + sv), ((i / kVStages) - 1) & 1, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                uint8_t* vdst = sm + kOffV + sv * kKvBytes;
                widen_store(vdst, 0, xa);
                load_item(kc, i + 1, 0, xa);
                widen_store(vdst, 1, xb);
                load_item(kc, i + 1, 1, xb);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarVFull + sv));
            }
            if (!ok && lane == 0) atomicOr(p.status, kDevErrTimeout);
        }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // ================= softmax: warps 4-7 tile A, 8-11 tile B; thread = one MMA row =================
        const int x = warp < 8 ? 0 : 1;
        const int quarter = warp & 3;                  // tensor-memory lanes 32 quarter .. + 31
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int steps = tile_steps(x);
        const int jf = x == 0 ? jf0 : jf1;
        const int jl = x == 0 ? jl0 : jl1;
        const int jq = r / G;
        const bool live = steps > 0 && r < QT * G && jf + jq <= jl;
        const int pos_first = qpos(jf);
        const int pos = live ? qpos(jf + jq) : qpos(jl);
        const size_t qrow = (static_cast<size_t>(q0 + (live ? jf + jq : jf0)) * p.num_q_heads + h * G +
                             (live ? r % G : 0)) * kHeadDim;
        // Q row -> shared memory (MMA input type), 128-byte swizzle, two d-halves; the
        // row's 16 loads all go out before the first store (one memory round trip)
        {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + qrow);
            uint8_t* qdst = sm + kOffQ + x * 2 * kQHalf;
            uint4 qv[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) qv[c] = live ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                uint4 v = qv[c];
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
        const float kscale = kFp8 ? __ldg(p.k_scale + h * p.scale_stride) : 1.0f;
        const float vscale = kFp8 ? __ldg(p.v_scale + h * p.scale_stride) : 1.0f;
        const float s_log2 = p.scale_log2 * kscale;
        const bool pos_scale = s_log2 >= 0.f;
        const uint32_t s_addr = tS(x) + lane_off;
        float m_used = -INFINITY, l = 0.f;
        for (int i = 0; i < steps && ok; ++i) {
            if (!warp_wait(bar(kBarSFull + x), i & 1, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int key0 = (step0 + i) * kTcKeys;
            const bool need_mask = key0 + kTcKeys - 1 > pos_first;
            const int lim = pos - key0;                 // columns > lim are masked
            // the whole row of S in registers: one tensor-memory round trip per step
            uint32_t sv[kTcKeys];
#pragma unroll
            for (int c = 0; c < kTcKeys / 32; ++c)
                tmem_ld32(s_addr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c));
            tmem_wait_ld();
            // row maximum of s * scale = max(s) * scale for scale >= 0, min(s) * scale
            // otherwise; four independent chains, masked columns only on diagonal steps
            float mx;
            if (!need_mask) {
                float e4[4];
                if (pos_scale) {
                    e4[0] = e4[1] = e4[2] = e4[3] = -INFINITY;
#pragma unroll
                    for (int e = 0; e < kTcKeys; e += 2)
                        e4[(e >> 1) & 3] = max3f(e4[(e >> 1) & 3], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
                    mx = fmaxf(fmaxf(e4[0], e4[1]), fmaxf(e4[2], e4[3])) * s_log2;
                } else {
                    e4[0] = e4[1] = e4[2] = e4[3] = INFINITY;
#pragma unroll
                    for (int e = 0; e < kTcKeys; e += 2)
                        e4[(e >> 1) & 3] = min3f(e4[(e >> 1) & 3], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
                    mx = fminf(fminf(e4[0], e4[1]), fminf(e4[2], e4[3])) * s_log2;
                }
            } else {
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < kTcKeys; ++e)
                    mx4[e & 3] = fmaxf(mx4[e & 3], e <= lim ? __uint_as_float(sv[e]) * s_log2 : -INFINITY);
                mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));   // -inf when every column is masked
            }
            const bool need = mx > m_used + kRescaleLog2;
            const bool resc = __any_sync(0xffffffffu, need);
            const float m_new = need ? fmaxf(m_used, mx) : m_used;
            const float alpha = ex2_approx(m_used - m_new);    // 0 on the first step, 1 when kept
            m_used = m_new;
            // O is final for P.V(i-1): S(i) was issued after it and completes after it.
            // Rescaled before any of P(i) is released, since P.V(i) accumulates into it.
            if (i >= 1 && resc) {
#pragma unroll 1
                for (int c = 0; c < kHeadDim / 32; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(tO(x) + lane_off + 32 * c, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                    tmem_st32(tO(x) + lane_off + 32 * c, ov);
                }
            }
            // p = 2^(s * scale - m) as the 16-bit A operand of P.V, written over the
            // columns of S (keys 32 c .. +31 -> columns 16 c .. +15)
            // (s * scale - m) and the running sums two columns per instruction (f32x2)
            uint64_t sum2[2] = {0ull, 0ull};
            const uint64_t scale2 = f2_pack(s_log2, s_log2);
            const uint64_t negm2 = f2_pack(-m_new, -m_new);
#pragma unroll
            for (int c = 0; c < kTcKeys / 32; ++c) {
                uint32_t pw[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int k = 32 * c + e;
                    float a0, a1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])), scale2, negm2), a0, a1);
                    float p0 = ex2_approx(a0);
                    float p1 = ex2_approx(a1);
                    if (need_mask) {
                        p0 = k <= lim ? p0 : 0.f;
                        p1 = k + 1 <= lim ? p1 : 0.f;
                    }
                    sum2[(e >> 1) & 1] = f2_add(sum2[(e >> 1) & 1], f2_pack(p0, p1));
                    pw[e >> 1] = pack2<kMmaBf16>(p0, p1);
                }
                tmem_st16(s_addr + 16 * c, pw);
                if (!kFp8 && c == kTcKeys / 64 - 1) {
                    // the first 64 keys' P (and any rescale of O) is in tensor memory
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kBarPHalf + x));
                }
            }
            tmem_wait_st();
            float s0, s1, s2, s3;
            f2_unpack(sum2[0], s0, s1);
            f2_unpack(sum2[1], s2, s3);
            l = l * alpha + ((s0 + s1) + (s2 + s3));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarPFull + x));
        }
        // ---- epilogue: O / l ----
        if (steps > 0) {
            if (ok && prefix && warp_wait(bar(kBarPvDone + x), 0, p.timeout_ns)) {
                // unnormalised rows and (max, sum) for the combine of the cascade decode
                tc_fence_after();
                // segment z of the prefix keys: its own rows of partials
                const size_t seg_rows = static_cast<size_t>(blockIdx.z) * p.num_seqs * p.num_q_heads;
                float* seg_o = blockIdx.z == 0 ? p.prefix_o : p.prefix_o_extra + (seg_rows - static_cast<size_t>(p.num_seqs) * p.num_q_heads) * kHeadDim;
                float* seg_ml = blockIdx.z == 0 ? p.prefix_ml : p.prefix_ml_extra + (seg_rows - static_cast<size_t>(p.num_seqs) * p.num_q_heads) * 2;
                float4* dst = reinterpret_cast<float4*>(seg_o + qrow);
#pragma unroll 1
                for (int c = 0; c < kHeadDim / 32; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(tO(x) + lane_off + 32 * c, ov);
                    tmem_wait_ld();
                    if (live) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[8 * c + e] = make_float4(__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                                                         __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3]));
                    }
                }
                if (live) {
                    seg_ml[(qrow / kHeadDim) * 2] = m_used;
                    seg_ml[(qrow / kHeadDim) * 2 + 1] = l;
                }
            } else if (ok && !prefix && warp_wait(bar(kBarPvDone + x), 0, p.timeout_ns)) {
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

size_t chunk_smem_bytes(CacheKind, int) {
    return 1024 + kOffBars + kBarBytes;
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
    cfg.gridDim = dim3(grid_x * p.num_kv_heads, 1, p.prefix_keys > 0 && p.prefix_splits > 1 ? p.prefix_splits : 1);
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
