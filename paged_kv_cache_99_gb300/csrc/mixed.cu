// Prefill chunks of a mixed batch for sm_103a.
//
// Problem ("Basics of LLM Inference and vLLM Internals", s.6 chunked prefill;
// "The Memory Trick Behind Fast LLM Serving", "Batching does not merge the
// conversations"): the query rows of all requests are flattened; a request with
// q_len > 1 new tokens is a prefill chunk whose row j sits at position
// seq_len - q_len + j and attends causally to its own cached tokens 0..pos,
// reached through its block table.
//
// Design: one CTA = one tile of consecutive queries of one chunk x all query
// heads of one KV head (64 MMA rows, query-major), so every K/V tile in shared
// memory serves the whole GQA group.  A producer warp walks the block table and
// issues bulk tensor copies (TMA, 128-byte swizzle) of 4 blocks (64 keys) per
// stage into a ring; four consumer warps compute S = Q K^T and O += P V with
// warp-level tensor-core MMAs and an online softmax, releasing each stage
// through an mbarrier.  The causal mask is applied only on the steps that cross
// the tile's first query position.  Tiles are scheduled heaviest first.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kChunkConsumers = 4;
constexpr int kChunkRows = kChunkConsumers * 16;    // MMA rows per CTA
constexpr int kStepBlocks = 4;                      // blocks (16 keys each) per stage
constexpr int kStepKeys = kStepBlocks * kBlockSize;

template <int Kind>
struct ChunkCfg {
    static constexpr bool kFp8 = Kind == kKindFp8;
    static constexpr int kTileBytes = kFp8 ? 2048 : 4096;
    static constexpr int kHalf = kStepBlocks * kTileBytes;         // K part of a stage
    static constexpr int kStageBytes = 2 * kHalf;
    static constexpr int kStages = kFp8 ? 4 : 3;
    static constexpr int kTileArea = kStages * kStageBytes;
    static constexpr int kBarBytes = 2 * kStages * 8;
};

}  // namespace

template <int Kind, bool QBf16>
__global__ void __launch_bounds__((kChunkConsumers + 1) * 32, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const ChunkParams p) {
    using Cfg = ChunkCfg<Kind>;
    constexpr bool kFp8 = Cfg::kFp8;
    constexpr bool kMmaBf16 = Kind == kKindBf16;
    constexpr int NS = Cfg::kStages;
    constexpr int TILE = Cfg::kTileBytes;

    extern __shared__ uint8_t smem_raw[];
    __shared__ int warp_tot[kChunkConsumers + 1];
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t tiles = (raw_base + 1023u) & ~1023u;
    uint8_t* aligned = smem_raw + (tiles - raw_base);
    const uint32_t full_bars = tiles + Cfg::kTileArea;
    const uint32_t empty_bars = full_bars + 8 * NS;
    int* cum = reinterpret_cast<int*>(aligned + Cfg::kTileArea + Cfg::kBarBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int st = 0; st < NS; ++st) {
            mbar_init(full_bars + 8 * st, 1);
            mbar_init(empty_bars + 8 * st, kChunkConsumers);
        }
        fence_barrier_init();
        tmap_prefetch(&kmap);
        tmap_prefetch(&vmap);
    }

    grid_dependency_wait();

    // ---- tiles per chunk sequence, exclusive scan -> cum ----
    const int B = p.num_seqs;
    const int QT = p.queries_per_tile;
    auto tiles_of = [&](int s) -> int {
        const int ql = p.query_start_loc[s + 1] - p.query_start_loc[s];
        return ql >= 2 ? (ql + QT - 1) / QT : 0;
    };
    {
        const int per = (B + blockDim.x - 1) / blockDim.x;
        const int beg = min(B, static_cast<int>(threadIdx.x) * per);
        const int end = min(B, beg + per);
        int local = 0;
        for (int s = beg; s < end; ++s) local += tiles_of(s);
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
            run += tiles_of(s);
        }
        if (threadIdx.x == blockDim.x - 1) cum[B] = run;
    }
    __syncthreads();
    grid_launch_dependents();

    const int R = cum[B];
    if (static_cast<int>(blockIdx.x) >= R) return;
    const int tau = R - 1 - static_cast<int>(blockIdx.x);   // heaviest tiles first
    int s = 0;
    {
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (cum[mid] <= tau) lo = mid; else hi = mid;
        }
        s = lo;
    }
    const int qt = tau - cum[s];
    const int h = blockIdx.y;
    const int G = p.group;
    const int q0 = p.query_start_loc[s];
    const int q_len = p.query_start_loc[s + 1] - q0;
    const int n = p.seq_lens[s];
    const int j_first = qt * QT;
    const int j_last = min(q_len, j_first + QT) - 1;
    const int pos_first = n - q_len + j_first;
    const int pos_last = n - q_len + j_last;
    if (pos_first < 0 || n > p.max_blocks * kBlockSize) {   // inconsistent lengths: nothing sensible to do
        if (threadIdx.x == 0) atomicOr(p.status, kDevErrRange);
        return;
    }
    const int nsteps = (pos_last + kStepKeys) / kStepKeys;
    const int nblocks = (pos_last + kBlockSize) / kBlockSize;

    if (warp == kChunkConsumers) {
        // ================= producer =================
        if (lane != 0) return;
        const int32_t* bt = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
        for (int k = 0; k < nsteps; ++k) {
            const int st = k % NS;
            if (k >= NS && !mbar_wait_bounded(empty_bars + 8 * st, ((k / NS) - 1) & 1, p.timeout_ns)) {
                atomicOr(p.status, kDevErrTimeout);
                return;
            }
            const int nb = min(kStepBlocks, nblocks - k * kStepBlocks);
            const uint32_t bar = full_bars + 8 * st;
            const uint32_t kdst = tiles + st * Cfg::kStageBytes;
            const uint32_t vdst = kdst + Cfg::kHalf;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nb) * 2 * TILE);
            for (int b = 0; b < nb; ++b) {
                int phys = __ldg(bt + k * kStepBlocks + b);
                if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
                    atomicOr(p.status, kDevErrRange);
                    phys = 0;
                }
                const int y = (phys * p.num_kv_heads + h) * kBlockSize;
                if constexpr (kFp8) {
                    tma_load_2d(kdst + b * TILE, &kmap, 0, y, bar);
                    tma_load_2d(vdst + b * TILE, &vmap, 0, y, bar);
                } else {
                    tma_load_2d(kdst + b * TILE, &kmap, 0, y, bar);
                    tma_load_2d(kdst + b * TILE + 2048, &kmap, 64, y, bar);
                    tma_load_2d(vdst + b * TILE, &vmap, 0, y, bar);
                    tma_load_2d(vdst + b * TILE + 2048, &vmap, 64, y, bar);
                }
            }
        }
        return;
    }

    // ================= consumers =================
    const int g8 = lane >> 2;
    const int t = lane & 3;
    const int mi = lane >> 3;
    const int r8 = lane & 7;
    // MMA rows of this thread: ra = 16 w + g8, rb = ra + 8; row r -> (query r / G, head r % G)
    const int ra = warp * 16 + g8, rb = ra + 8;
    const int rows_used = QT * G;
    const int ja = j_first + ra / G, jb = j_first + rb / G;
    const bool live_a = ra < rows_used && ja <= j_last;
    const bool live_b = rb < rows_used && jb <= j_last;
    const int pos_a = live_a ? n - q_len + ja : pos_last;
    const int pos_b = live_b ? n - q_len + jb : pos_last;
    const uint16_t* qa_row = static_cast<const uint16_t*>(p.q) +
                             (static_cast<size_t>(q0 + (live_a ? ja : j_first)) * p.num_q_heads + h * G + (live_a ? ra % G : 0)) * kHeadDim;
    const uint16_t* qb_row = static_cast<const uint16_t*>(p.q) +
                             (static_cast<size_t>(q0 + (live_b ? jb : j_first)) * p.num_q_heads + h * G + (live_b ? rb % G : 0)) * kHeadDim;

    uint32_t qa[8][4];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        if constexpr (!kFp8) {
            qa[kk][0] = live_a ? *reinterpret_cast<const uint32_t*>(qa_row + 16 * kk + 2 * t) : 0u;
            qa[kk][1] = live_b ? *reinterpret_cast<const uint32_t*>(qb_row + 16 * kk + 2 * t) : 0u;
            qa[kk][2] = live_a ? *reinterpret_cast<const uint32_t*>(qa_row + 16 * kk + 2 * t + 8) : 0u;
            qa[kk][3] = live_b ? *reinterpret_cast<const uint32_t*>(qb_row + 16 * kk + 2 * t + 8) : 0u;
        } else {
            // k-slots (2t, 2t+1) <-> d (16kk+4t, +1); (2t+8, 2t+9) <-> d (16kk+4t+2, +3)
            const uint2 xa = live_a ? *reinterpret_cast<const uint2*>(qa_row + 16 * kk + 4 * t) : make_uint2(0, 0);
            const uint2 xb = live_b ? *reinterpret_cast<const uint2*>(qb_row + 16 * kk + 4 * t) : make_uint2(0, 0);
            qa[kk][0] = pack2<false>(to_float<QBf16>(xa.x & 0xffff), to_float<QBf16>(xa.x >> 16));
            qa[kk][1] = pack2<false>(to_float<QBf16>(xb.x & 0xffff), to_float<QBf16>(xb.x >> 16));
            qa[kk][2] = pack2<false>(to_float<QBf16>(xa.y & 0xffff), to_float<QBf16>(xa.y >> 16));
            qa[kk][3] = pack2<false>(to_float<QBf16>(xb.y & 0xffff), to_float<QBf16>(xb.y >> 16));
        }
    }

    const float kscale = kFp8 ? __ldg(p.k_scale) : 1.0f;
    const float vscale = kFp8 ? __ldg(p.v_scale) : 1.0f;
    const float s_log2 = p.scale_log2 * kscale;
    const uint32_t kq_row = static_cast<uint32_t>(r8 + ((mi & 1) << 3));     // K/V rows for fp8 and V
    const uint32_t k16_row = static_cast<uint32_t>(r8 + ((mi >> 1) << 3));   // K rows, 16-bit

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;

    for (int k = 0; k < nsteps; ++k) {
        const int st = k % NS;
        const uint32_t bar = full_bars + 8 * st;
        const uint32_t parity = (k / NS) & 1;
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded(bar, parity, p.timeout_ns);
        ok = __shfl_sync(0xffffffffu, static_cast<int>(ok), 0) != 0;
        if (!ok) {
            if (lane == 0) atomicOr(p.status, kDevErrTimeout);
            return;
        }
        mbar_try_wait(bar, parity);
        const uint32_t kbase = tiles + st * Cfg::kStageBytes;
        const uint32_t vbase = kbase + Cfg::kHalf;
        const int key0 = k * kStepKeys;

        // ---- S = Q K^T over 64 keys: s[nt] covers keys key0 + 8 nt .. +7 ----
        float sc[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
        for (int b = 0; b < kStepBlocks; ++b) {
            const uint32_t kt = kbase + b * TILE;
            if constexpr (!kFp8) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t c = 2 * kk + (mi & 1);
                    const uint32_t addr = kt + ((c >> 3) << 11) + (k16_row << 7) + (((c & 7) ^ r8) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(addr, b0, b1, b2, b3);
                    mma16816<kMmaBf16>(sc[2 * b], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                    mma16816<kMmaBf16>(sc[2 * b + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
                }
            } else {
#pragma unroll
                for (int kq = 0; kq < 4; ++kq) {
                    const uint32_t c = 2 * kq + (mi >> 1);
                    const uint32_t addr = kt + (kq_row << 7) + ((c ^ r8) << 4);
                    uint32_t x0, x1, x2, x3;
                    ldsm_x4(addr, x0, x1, x2, x3);
                    const int k0 = 2 * kq, k1 = 2 * kq + 1;
                    mma16816<false>(sc[2 * b], qa[k0][0], qa[k0][1], qa[k0][2], qa[k0][3],
                                    e4m3x2_to_f16x2(x0 & 0xffff), e4m3x2_to_f16x2(x0 >> 16));
                    mma16816<false>(sc[2 * b + 1], qa[k0][0], qa[k0][1], qa[k0][2], qa[k0][3],
                                    e4m3x2_to_f16x2(x1 & 0xffff), e4m3x2_to_f16x2(x1 >> 16));
                    mma16816<false>(sc[2 * b], qa[k1][0], qa[k1][1], qa[k1][2], qa[k1][3],
                                    e4m3x2_to_f16x2(x2 & 0xffff), e4m3x2_to_f16x2(x2 >> 16));
                    mma16816<false>(sc[2 * b + 1], qa[k1][0], qa[k1][1], qa[k1][2], qa[k1][3],
                                    e4m3x2_to_f16x2(x3 & 0xffff), e4m3x2_to_f16x2(x3 >> 16));
                }
            }
        }

        // ---- scale, causal mask, online softmax (rows ra, rb) ----
        const bool need_mask = key0 + kStepKeys - 1 > pos_first;
        float xa = -INFINITY, xb = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int key = key0 + 8 * nt + 2 * t + e;
                float va = sc[nt][e] * s_log2, vb = sc[nt][2 + e] * s_log2;
                if (need_mask) {
                    if (key > pos_a) va = -INFINITY;
                    if (key > pos_b) vb = -INFINITY;
                }
                sc[nt][e] = va;
                sc[nt][2 + e] = vb;
                xa = fmaxf(xa, va);
                xb = fmaxf(xb, vb);
            }
        }
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 1));
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 2));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 1));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 2));
        const float na = fmaxf(ma, xa), nb = fmaxf(mb, xb);
        const float aa = exp2f(ma - na), ab = exp2f(mb - nb);
        ma = na;
        mb = nb;
        float sa = 0.f, sb = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            sc[nt][0] = exp2f(sc[nt][0] - na);
            sc[nt][1] = exp2f(sc[nt][1] - na);
            sc[nt][2] = exp2f(sc[nt][2] - nb);
            sc[nt][3] = exp2f(sc[nt][3] - nb);
            sa += sc[nt][0] + sc[nt][1];
            sb += sc[nt][2] + sc[nt][3];
        }
        la = la * aa + sa;
        lb = lb * ab + sb;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            o[i][0] *= aa;
            o[i][1] *= aa;
            o[i][2] *= ab;
            o[i][3] *= ab;
        }

        // ---- O += P V, one 16-key block at a time ----
#pragma unroll
        for (int b = 0; b < kStepBlocks; ++b) {
            const uint32_t pa0 = pack2<kMmaBf16>(sc[2 * b][0], sc[2 * b][1]);
            const uint32_t pa1 = pack2<kMmaBf16>(sc[2 * b][2], sc[2 * b][3]);
            const uint32_t pa2 = pack2<kMmaBf16>(sc[2 * b + 1][0], sc[2 * b + 1][1]);
            const uint32_t pa3 = pack2<kMmaBf16>(sc[2 * b + 1][2], sc[2 * b + 1][3]);
            // keys at or beyond the sequence end (or in blocks not loaded) hold no data
            const int valid = min(kBlockSize, n - (key0 + b * kBlockSize));
            if (valid <= 0) continue;
            uint32_t vm01 = 0xffffffffu, vm23 = 0xffffffffu;
            if (valid < kBlockSize) {
                vm01 = (2 * t < valid ? 0x0000ffffu : 0u) | (2 * t + 1 < valid ? 0xffff0000u : 0u);
                vm23 = (2 * t + 8 < valid ? 0x0000ffffu : 0u) | (2 * t + 9 < valid ? 0xffff0000u : 0u);
            }
            const uint32_t vt = vbase + b * TILE;
            if (key0 + b * kBlockSize > pos_last) continue;   // block not loaded
            if constexpr (!kFp8) {
#pragma unroll
                for (int dp = 0; dp < 8; ++dp) {
                    const uint32_t c = 2 * dp + (mi >> 1);
                    const uint32_t addr = vt + ((c >> 3) << 11) + (kq_row << 7) + (((c & 7) ^ r8) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(addr, b0, b1, b2, b3);
                    mma16816<kMmaBf16>(o[2 * dp], pa0, pa1, pa2, pa3, b0 & vm01, b1 & vm23);
                    mma16816<kMmaBf16>(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2 & vm01, b3 & vm23);
                }
            } else {
#pragma unroll
                for (int dq = 0; dq < 4; ++dq) {
                    const uint32_t c = 2 * dq + (mi >> 1);
                    const uint32_t addr = vt + (kq_row << 7) + ((c ^ r8) << 4);
                    uint32_t x0, x1, x2, x3;
                    ldsm_x4_t(addr, x0, x1, x2, x3);
                    const uint32_t e0 = prmt(x0, 0, 0x3120), e1 = prmt(x1, 0, 0x3120);
                    const uint32_t e2 = prmt(x2, 0, 0x3120), e3 = prmt(x3, 0, 0x3120);
                    // n-tile (chunk c, parity pi) = o[2c + pi]: columns d = 16c + 4t + pi, +2
                    const int c0 = 2 * dq, c1 = 2 * dq + 1;
                    mma16816<false>(o[2 * c0], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(e0 & 0xffff) & vm01,
                                    e4m3x2_to_f16x2(e1 & 0xffff) & vm23);
                    mma16816<false>(o[2 * c0 + 1], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(e0 >> 16) & vm01,
                                    e4m3x2_to_f16x2(e1 >> 16) & vm23);
                    mma16816<false>(o[2 * c1], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(e2 & 0xffff) & vm01,
                                    e4m3x2_to_f16x2(e3 & 0xffff) & vm23);
                    mma16816<false>(o[2 * c1 + 1], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(e2 >> 16) & vm01,
                                    e4m3x2_to_f16x2(e3 >> 16) & vm23);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bars + 8 * st);
    }

    // ---- normalise and store ----
    la += __shfl_xor_sync(0xffffffffu, la, 1);
    la += __shfl_xor_sync(0xffffffffu, la, 2);
    lb += __shfl_xor_sync(0xffffffffu, lb, 1);
    lb += __shfl_xor_sync(0xffffffffu, lb, 2);
    const float ia = vscale / la, ib = vscale / lb;
    uint16_t* oa = static_cast<uint16_t*>(p.out) +
                   (static_cast<size_t>(q0 + ja) * p.num_q_heads + h * G + ra % G) * kHeadDim;
    uint16_t* ob = static_cast<uint16_t*>(p.out) +
                   (static_cast<size_t>(q0 + jb) * p.num_q_heads + h * G + rb % G) * kHeadDim;
    if constexpr (!kFp8) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int d = 8 * nt + 2 * t;
            if (live_a)
                *reinterpret_cast<uint32_t*>(oa + d) = static_cast<uint32_t>(from_float<QBf16>(o[nt][0] * ia)) |
                                                       (static_cast<uint32_t>(from_float<QBf16>(o[nt][1] * ia)) << 16);
            if (live_b)
                *reinterpret_cast<uint32_t*>(ob + d) = static_cast<uint32_t>(from_float<QBf16>(o[nt][2] * ib)) |
                                                       (static_cast<uint32_t>(from_float<QBf16>(o[nt][3] * ib)) << 16);
        }
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int d = 16 * c + 4 * t;
            if (live_a) {
                uint2 w;
                w.x = static_cast<uint32_t>(from_float<QBf16>(o[2 * c][0] * ia)) |
                      (static_cast<uint32_t>(from_float<QBf16>(o[2 * c + 1][0] * ia)) << 16);
                w.y = static_cast<uint32_t>(from_float<QBf16>(o[2 * c][1] * ia)) |
                      (static_cast<uint32_t>(from_float<QBf16>(o[2 * c + 1][1] * ia)) << 16);
                *reinterpret_cast<uint2*>(oa + d) = w;
            }
            if (live_b) {
                uint2 w;
                w.x = static_cast<uint32_t>(from_float<QBf16>(o[2 * c][2] * ib)) |
                      (static_cast<uint32_t>(from_float<QBf16>(o[2 * c + 1][2] * ib)) << 16);
                w.y = static_cast<uint32_t>(from_float<QBf16>(o[2 * c][3] * ib)) |
                      (static_cast<uint32_t>(from_float<QBf16>(o[2 * c + 1][3] * ib)) << 16);
                *reinterpret_cast<uint2*>(ob + d) = w;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {
void* chunk_fn(CacheKind kind, bool q_bf16) {
    switch (kind) {
        case kKindBf16: return reinterpret_cast<void*>(&chunk_kernel<kKindBf16, true>);
        case kKindFp16: return reinterpret_cast<void*>(&chunk_kernel<kKindFp16, false>);
        case kKindFp8:
            return q_bf16 ? reinterpret_cast<void*>(&chunk_kernel<kKindFp8, true>)
                          : reinterpret_cast<void*>(&chunk_kernel<kKindFp8, false>);
    }
    return nullptr;
}
}  // namespace

size_t chunk_smem_bytes(CacheKind kind, int num_seqs) {
    size_t area = 0;
    switch (kind) {
        case kKindBf16: area = ChunkCfg<kKindBf16>::kTileArea + ChunkCfg<kKindBf16>::kBarBytes; break;
        case kKindFp16: area = ChunkCfg<kKindFp16>::kTileArea + ChunkCfg<kKindFp16>::kBarBytes; break;
        case kKindFp8: area = ChunkCfg<kKindFp8>::kTileArea + ChunkCfg<kKindFp8>::kBarBytes; break;
    }
    return 1024 + area + static_cast<size_t>(num_seqs + 1) * 4;
}

int chunk_rows() { return kChunkRows; }

cudaError_t chunk_prepare(CacheKind kind, bool q_bf16, size_t max_smem) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, chunk_fn(kind, q_bf16));
    if (e != cudaSuccess) return e;
    size_t want = chunk_smem_bytes(kind, kMaxSeqs);
    const size_t cap = max_smem > fa.sharedSizeBytes ? max_smem - fa.sharedSizeBytes : 0;
    if (want > cap) want = cap;
    return cudaFuncSetAttribute(chunk_fn(kind, q_bf16), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(want));
}

cudaError_t launch_chunk(CacheKind kind, bool q_bf16, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         const ChunkParams& p, int grid_x, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, p.num_kv_heads);
    cfg.blockDim = dim3((kChunkConsumers + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (kind) {
        case kKindBf16: return cudaLaunchKernelEx(&cfg, chunk_kernel<kKindBf16, true>, kmap, vmap, p);
        case kKindFp16: return cudaLaunchKernelEx(&cfg, chunk_kernel<kKindFp16, false>, kmap, vmap, p);
        case kKindFp8:
            return q_bf16 ? cudaLaunchKernelEx(&cfg, chunk_kernel<kKindFp8, true>, kmap, vmap, p)
                          : cudaLaunchKernelEx(&cfg, chunk_kernel<kKindFp8, false>, kmap, vmap, p);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pa
