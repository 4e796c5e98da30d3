// C ABI of the paged attention library: argument checks, workspace layout,
// tensor-map encoding and launches.  See include/pa.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "pa.h"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 1000ull * 1000ull * 1000ull;   // 1 s per wait

struct DeviceState {
    bool ready = false;
    int sms = 0;
    size_t max_smem_optin = 0;
    bool decode_prepared[3][2][2][2][2] = {};
    bool chunk_prepared[3][2] = {};
};

std::mutex g_mu;
std::map<int, DeviceState> g_devices;
std::map<std::tuple<int, int, int, int, int, size_t>, int> g_occupancy;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

thread_local char g_last_error[256] = "";
std::atomic<unsigned long long> g_launches{0};

pa_status fail(const char* what, cudaError_t e) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s (%d)", what, cudaGetErrorString(e), static_cast<int>(e));
    return PA_ERR_CUDA;
}

pa_status fail_msg(const char* what) {
    snprintf(g_last_error, sizeof g_last_error, "%s", what);
    return PA_ERR_CUDA;
}

pa_status cuda_status(cudaError_t e, const char* what) { return e == cudaSuccess ? PA_OK : fail(what, e); }

// Status of a kernel launch; a launch that was enqueued is counted.
pa_status launched(cudaError_t e, const char* what) {
    if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(e, what);
}

// Device attributes of the current device; nullptr on failure.
DeviceState* device_state(int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        fail("cudaGetDevice", e);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& st = g_devices[dev];
    if (!st.ready) {
        int sms = 0, optin = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) {
            fail("cudaDeviceGetAttribute", e);
            return nullptr;
        }
        st.sms = sms;
        st.max_smem_optin = static_cast<size_t>(optin);
        st.ready = true;
    }
    if (dev_out) *dev_out = dev;
    return &st;
}

bool encode_fn() {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_encode) return true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
        snprintf(g_last_error, sizeof g_last_error, "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled): %s, query %d",
                 cudaGetErrorString(e), static_cast<int>(q));
        return false;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

// Tensor map over a cache viewed as rows of 128 elements (one token of one KV
// head); boxes of min(block size, 16) rows, 128-byte swizzle.  16-bit caches are
// copied in two 64-element halves, FP8 caches in one 128-byte box.
pa_status encode_cache_map(CUtensorMap* map, const void* base, int num_blocks, int num_kv_heads, int block_size,
                           bool fp8) {
    if (!encode_fn()) return PA_ERR_CUDA;
    const cuuint64_t rows = static_cast<cuuint64_t>(num_blocks) * num_kv_heads * block_size;
    const cuuint64_t dims[2] = {kHeadDim, rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim) * (fp8 ? 1 : 2)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(fp8 ? 128 : 64),
                               static_cast<cuuint32_t>(block_size < kBlockSize ? block_size : kBlockSize)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Tokens per physical block: 8, 16 or 32 (the kernels work in 16-key units).
bool block_size_ok(int bs) { return bs == 8 || bs == 16 || bs == 32; }

int block_shift_of(int bs) { return bs == 8 ? 3 : (bs == 16 ? 4 : 5); }

bool is_fp8(pa_dtype d) { return d == PA_FP8_E4M3 || d == PA_FP8_E4M3_PER_HEAD; }

// FP8 scale stride: 0 for one scale per tensor, 1 for one per KV head
int scale_stride_of(pa_dtype d) { return d == PA_FP8_E4M3_PER_HEAD ? 1 : 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int head_groups_of(int num_q_heads, int num_kv_heads) {
    const int group = num_q_heads / num_kv_heads;
    return (group + kHeadsPerGroup - 1) / kHeadsPerGroup;
}

int max_workers(const DeviceState& st) { return st.sms * kMaxDecodeCtasPerSm * kDecodeWarps; }

// Checks shared by decode and mixed.
pa_status check_attention_args(const void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                               int num_blocks, float scale, pa_dtype q_dtype, pa_dtype cache_dtype,
                               const float* k_scale, const float* v_scale, const void* workspace) {
    if (head_dim != kHeadDim || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
    if (q_dtype != PA_BF16 && q_dtype != PA_FP16) return PA_ERR_UNSUPPORTED;
    if (cache_dtype != q_dtype && !is_fp8(cache_dtype)) return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_seqs > kMaxSeqs) return PA_ERR_INVALID_ARG;
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (num_blocks <= 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (!k_cache || !v_cache || !workspace) return PA_ERR_INVALID_ARG;
    // the per-sequence arrays of an empty batch may be empty (null)
    if (num_seqs > 0 && (!out || !q || !block_tables || !seq_lens)) return PA_ERR_INVALID_ARG;
    if (is_fp8(cache_dtype) && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(workspace, 256))
        return PA_ERR_INVALID_ARG;
    // tensor-map rows and flattened 16-key unit counts must fit in 32 bits
    const long long rows = static_cast<long long>(num_blocks) * num_kv_heads * block_size;
    const long long units = static_cast<long long>(num_seqs) * num_kv_heads * head_groups_of(num_q_heads, num_kv_heads);
    const long long per_seq = (static_cast<long long>(max_blocks_per_seq) * block_size + kBlockSize - 1) / kBlockSize;
    if (rows >= (1ll << 31) || units * per_seq >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

CacheKind kind_of(pa_dtype cache_dtype) {
    return is_fp8(cache_dtype) ? kKindFp8 : (cache_dtype == PA_FP16 ? kKindFp16 : kKindBf16);
}

pa_status decode_impl(void* out, const void* q, const int32_t* query_start_loc, const void* k_cache,
                      const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* seq_lens, int num_seqs, int num_q_heads, int num_kv_heads, float scale,
                      pa_dtype q_dtype, pa_dtype cache_dtype, const float* k_scale, const float* v_scale,
                      void* workspace, size_t workspace_bytes, int num_workers, int num_blocks, int block_size,
                      int total_rows, cudaStream_t stream, bool overlap_prior = false, bool cascade = false,
                      int first_block = 0, int prefix_splits = 1, const float* prefix_o_extra = nullptr,
                      const float* prefix_ml_extra = nullptr, const void* k_new = nullptr,
                      const void* v_new = nullptr, const int64_t* slots = nullptr) {
    int dev = 0;
    DeviceState* st = device_state(&dev);
    if (!st) return PA_ERR_CUDA;
    const CacheKind kind = kind_of(cache_dtype);
    const bool q_bf16 = q_dtype == PA_BF16;
    const bool append = slots != nullptr;
    // claimed pieces balance SMs that stream at different rates; they pay only where
    // workers' ranges are long (judged from the table width: the decode grid decides
    // from the lengths) and the warps keep HBM busy: FP8 warps, and 16-bit warps with
    // more than 4 query heads per unit, are bound by the latency of each block, not
    // by HBM, and lose more to the pieces than the balance gains.  A mixed batch's
    // decode grid starts beside the chunk grid, CTA by CTA, and keeps static ranges; a
    // cascade's takes the SMs the prefix grid leaves free from the start and claims
    // like a plain decode
    const int hg0 = head_groups_of(num_q_heads, num_kv_heads);
    const long long units_max = static_cast<long long>(num_seqs) * num_kv_heads * hg0;
    const long long per_unit_max = (static_cast<long long>(max_blocks_per_seq) * block_size + kBlockSize - 1) / kBlockSize;
    const long long t_max = units_max * per_unit_max;
    const int w_default = st->sms * kMaxDecodeCtasPerSm * kDecodeWarps;
    const int w_est = num_workers > 0 ? num_workers : w_default;
    const int unit_heads = num_q_heads / num_kv_heads < kHeadsPerGroup ? num_q_heads / num_kv_heads : kHeadsPerGroup;
    const bool dyn = query_start_loc == nullptr && kind != kKindFp8 && unit_heads <= 4 &&
                     t_max / w_est >= kMinPieceRange;
    // a cascade's suffix decode and a mixed batch's decode rows (16-bit caches) take
    // the two-stage ring and three CTAs per SM
    const bool narrow = kind != kKindFp8 && !append && (cascade || query_start_loc != nullptr);
    const size_t smem = decode_smem_bytes(kind, num_seqs, narrow);
    if (smem + 1024 > st->max_smem_optin) return PA_ERR_UNSUPPORTED;
    int ctas = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!st->decode_prepared[kind][q_bf16][append][dyn][narrow]) {
            cudaError_t e = decode_prepare(kind, q_bf16, append, dyn, narrow, st->max_smem_optin);
            if (e != cudaSuccess) return fail("cudaFuncSetAttribute(decode)", e);
            st->decode_prepared[kind][q_bf16][append][dyn][narrow] = true;
        }
        auto key = std::make_tuple(dev, static_cast<int>(kind), static_cast<int>(q_bf16), static_cast<int>(append),
                                   static_cast<int>(dyn) + 2 * static_cast<int>(narrow), smem);
        auto it = g_occupancy.find(key);
        if (it == g_occupancy.end()) {
            cudaError_t e = decode_occupancy(kind, q_bf16, append, dyn, narrow, smem, &ctas);
            if (e != cudaSuccess) return fail("cudaOccupancyMaxActiveBlocksPerMultiprocessor(decode)", e);
            if (ctas <= 0) return fail_msg("decode kernel does not fit on an SM");
            g_occupancy[key] = ctas;
        } else {
            ctas = it->second;
        }
    }
    const int cap = kind == kKindFp8 ? kMaxDecodeCtasPerSmFp8 : narrow ? kMaxDecodeCtasPerSmNarrow : kMaxDecodeCtasPerSm;
    ctas = ctas > cap ? cap : ctas;
    const int full = st->sms * ctas * kDecodeWarps;
    if (num_workers < 0 || num_workers > max_workers(*st)) return PA_ERR_INVALID_ARG;
    const int W = num_workers == 0 ? full : num_workers;
    const int hg = head_groups_of(num_q_heads, num_kv_heads);
    // one slot per static range, and as many for claimed pieces
    const WorkspaceLayout lay = decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads, hg, dyn ? 2 * W : W);
    if (workspace_bytes < lay.total) return PA_ERR_WORKSPACE;

    CUtensorMap kmap, vmap;
    pa_status s = encode_cache_map(&kmap, k_cache, num_blocks, num_kv_heads, block_size, kind == kKindFp8);
    if (s != PA_OK) return s;
    s = encode_cache_map(&vmap, v_cache, num_blocks, num_kv_heads, block_size, kind == kKindFp8);
    if (s != PA_OK) return s;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    DecodeParams p;
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.query_start_loc = query_start_loc;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.scale_stride = scale_stride_of(cache_dtype);
    p.status = reinterpret_cast<int*>(ws + lay.status_off);
    p.plan = reinterpret_cast<int*>(ws + lay.plan_off);
    p.ml = reinterpret_cast<float*>(ws + lay.ml_off);
    p.partial = reinterpret_cast<float4*>(ws + lay.partial_off);
    p.num_seqs = num_seqs;
    p.total_rows = total_rows;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = num_q_heads / num_kv_heads;
    p.head_groups = hg;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.block_shift = block_shift_of(block_size);
    p.num_workers = W;
    p.dyn256 = dyn ? kDynShare256 : 0;
    p.narrow = narrow ? 1 : 0;
    p.claim = reinterpret_cast<unsigned*>(ws + lay.status_off + 8);
    p.overlap_prior = overlap_prior ? 1 : 0;
    p.cascade = cascade ? 1 : 0;
    p.first_block = cascade ? first_block : 0;
    p.prefix_o = reinterpret_cast<const float*>(ws + lay.prefix_o_off);
    p.prefix_ml = reinterpret_cast<const float*>(ws + lay.prefix_ml_off);
    p.prefix_splits = prefix_splits;
    p.prefix_o_extra = prefix_o_extra;
    p.prefix_ml_extra = prefix_ml_extra;
    p.append = slots != nullptr ? 1 : 0;
    p.k_new = static_cast<const uint16_t*>(k_new);
    p.v_new = static_cast<const uint16_t*>(v_new);
    p.slots = slots;
    p.k_cache_w = const_cast<void*>(k_cache);
    p.v_cache_w = const_cast<void*>(v_cache);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.timeout_ns = kDefaultTimeoutNs;
    const int grid = (W + kDecodeWarps - 1) / kDecodeWarps;
    s = launched(launch_decode(kind, q_bf16, kmap, vmap, p, grid, smem, stream), "launch(decode)");
    if (s != PA_OK) return s;
    return launched(launch_combine(q_bf16, kind == kKindFp8, p, 2 * st->sms, stream), "launch(combine)");
}

pa_status chunk_impl(void* out, const void* q, const int32_t* query_start_loc, const void* k_cache,
                     const void* v_cache, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* seq_lens, int num_seqs, int total_q, int num_q_heads, int num_kv_heads,
                     int num_blocks, int block_size, float scale, pa_dtype q_dtype, pa_dtype cache_dtype,
                     const float* k_scale, const float* v_scale, void* workspace, cudaStream_t stream,
                     int prefix_units = 0, float* prefix_o = nullptr, float* prefix_ml = nullptr,
                     int prefix_splits = 1, int prefix_steps = 0, float* prefix_o_extra = nullptr,
                     float* prefix_ml_extra = nullptr) {
    DeviceState* st = device_state(nullptr);
    if (!st) return PA_ERR_CUDA;
    const CacheKind kind = kind_of(cache_dtype);
    const bool q_bf16 = q_dtype == PA_BF16;
    const int group = num_q_heads / num_kv_heads;
    const int qt = chunk_rows() / group;
    if (qt < 1) return PA_ERR_UNSUPPORTED;
    const size_t smem = chunk_smem_bytes(kind, num_seqs);
    if (smem + 1024 > st->max_smem_optin) return PA_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!st->chunk_prepared[kind][q_bf16]) {
            cudaError_t e = chunk_prepare(kind, q_bf16, st->max_smem_optin);
            if (e != cudaSuccess) return fail("cudaFuncSetAttribute(chunk)", e);
            st->chunk_prepared[kind][q_bf16] = true;
        }
    }
    const int per_cta = qt * chunk_tiles_per_cta();   // queries of one chunk per CTA
    // prefix mode: the queries are the sequences' decode rows, one tile pair per CTA
    const long long grid_x = prefix_units > 0 ? (num_seqs + per_cta - 1) / per_cta
                                               : static_cast<long long>(num_seqs) + (total_q + per_cta - 1) / per_cta;
    if (grid_x * num_kv_heads >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    ChunkParams p;
    p.out = out;
    p.q = q;
    p.query_start_loc = query_start_loc;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.scale_stride = scale_stride_of(cache_dtype);
    p.status = static_cast<int*>(workspace);
    p.num_seqs = num_seqs;
    p.total_rows = total_q;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = group;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.block_shift = block_shift_of(block_size);
    p.queries_per_tile = qt;
    p.prefix_keys = prefix_units * kBlockSize;
    p.prefix_o = prefix_o;
    p.prefix_ml = prefix_ml;
    p.prefix_splits = prefix_splits;
    p.prefix_steps = prefix_steps;
    p.prefix_o_extra = prefix_o_extra;
    p.prefix_ml_extra = prefix_ml_extra;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.timeout_ns = kDefaultTimeoutNs;
    return launched(launch_chunk(kind, q_bf16, kmap, vmap, p, static_cast<int>(grid_x), smem, stream),
                       "launch(chunk)");
}

}  // namespace

WorkspaceLayout decode_workspace_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_groups,
                                        int range_slots) {
    WorkspaceLayout l;
    const size_t units = static_cast<size_t>(num_seqs) * num_kv_heads * head_groups;
    // a range's partial of unit u sits in slot (range index + u)
    const size_t slots = units + static_cast<size_t>(range_slots);
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads;
    l.status_off = 0;
    l.plan_off = 256;
    // the shared-prefix partials sit before the worker slots: their place does not
    // depend on the worker count
    l.prefix_o_off = l.plan_off + round_up((static_cast<size_t>(num_seqs) + 1) * 4, 256);
    l.prefix_ml_off = l.prefix_o_off + round_up(rows * kHeadDim * sizeof(float), 256);
    l.ml_off = l.prefix_ml_off + round_up(rows * 2 * sizeof(float), 256);
    l.partial_off = l.ml_off + round_up(slots * 16 * 4, 256);
    l.total = l.partial_off + slots * 8 * 32 * sizeof(float4);
    return l;
}

// Extra prefix segments of a split shared prefix, after the base workspace:
// [splits - 1][rows][128] f32 partial rows, then [splits - 1][rows][2] (max, sum).
struct PrefixExtra {
    size_t o_off, ml_off, end;
};

PrefixExtra prefix_extra_layout(size_t base, size_t rows, int splits) {
    PrefixExtra e;
    e.o_off = round_up(base, 256);
    e.ml_off = round_up(e.o_off + static_cast<size_t>(splits - 1) * rows * kHeadDim * sizeof(float), 256);
    e.end = e.ml_off + static_cast<size_t>(splits - 1) * rows * 2 * sizeof(float);
    return e;
}

// ---------------------------------------------------------------------------
// Allocation-free decode: scratch in a fixed device array of this library.
// ---------------------------------------------------------------------------

// Scratch of pa_decode_noalloc.  Every GPU that loads the library holds these
// 16 MiB until the process exits.  In host code the name below only stands in
// for the device array; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[16u << 20];

namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;
std::map<int, void*> g_noalloc_address;   // device -> device address of g_noalloc_scratch

// Device address of the static scratch on the current device, looked up once per
// device (with that device current) and cached.
pa_status noalloc_scratch(void** out, DeviceState** st_out) {
    int dev = 0;
    DeviceState* st = device_state(&dev);
    if (!st) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_noalloc_address.find(dev);
    if (it == g_noalloc_address.end()) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr) return fail("cudaGetSymbolAddress(scratch)", e);
        it = g_noalloc_address.emplace(dev, ptr).first;
    }
    *out = it->second;
    *st_out = st;
    return PA_OK;
}

}  // namespace

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported parameters";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_TIMEOUT: return "device wait timed out";
        case PA_ERR_OUT_OF_RANGE: return "block-table entry outside the pool";
        case PA_ERR_WORKSPACE: return "workspace too small";
        default: return "unknown status";
    }
}

int pa_version(void) { return 101; }

unsigned long long pa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char* pa_last_error(void) { return g_last_error; }

pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, pa_dtype src_dtype, pa_dtype cache_dtype,
                               const float* k_scale, const float* v_scale, pa_stream_t stream) {
    if (head_dim != kHeadDim || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
    if (src_dtype != PA_BF16 && src_dtype != PA_FP16) return PA_ERR_UNSUPPORTED;
    if (cache_dtype != src_dtype && !is_fp8(cache_dtype)) return PA_ERR_UNSUPPORTED;
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (is_fp8(cache_dtype) && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    if (static_cast<long long>(num_tokens) * num_kv_heads >= (1ll << 34)) return PA_ERR_UNSUPPORTED;
    return launched(launch_reshape(k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, num_blocks,
                                      block_shift_of(block_size), src_dtype == PA_BF16, is_fp8(cache_dtype), k_scale, v_scale, scale_stride_of(cache_dtype),
                                      reinterpret_cast<cudaStream_t>(stream)),
                       "launch(reshape_and_cache)");
}

size_t pa_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim) {
    if (num_seqs < 0 || num_seqs > kMaxSeqs || head_dim != kHeadDim || num_kv_heads <= 0 || num_q_heads <= 0 ||
        num_q_heads % num_kv_heads != 0)
        return 0;
    DeviceState* st = device_state(nullptr);
    if (!st) return 0;
    // the most range slots a call takes: a two-stage 16-bit grid's workers (three
    // CTAs per SM) and as many claimed pieces (an FP8 grid's workers, or a plain
    // 16-bit grid's workers and pieces, take fewer)
    return decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_groups_of(num_q_heads, num_kv_heads),
                                   2 * st->sms * kMaxDecodeCtasPerSmNarrow * kDecodeWarps)
        .total;
}

size_t pa_workspace_size_shared_prefix(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim) {
    const size_t base = pa_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim);
    if (base == 0) return 0;
    return prefix_extra_layout(base, static_cast<size_t>(num_seqs) * num_q_heads, kMaxPrefixSplits).end;
}

int pa_default_workers(void) {
    DeviceState* st = device_state(nullptr);
    return st ? max_workers(*st) : 0;
}

pa_status pa_decode_ex(void* out, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                       float scale, pa_dtype q_dtype, pa_dtype cache_dtype, const float* k_scale,
                       const float* v_scale, void* workspace, size_t workspace_bytes, int num_workers,
                       pa_stream_t stream) {
    pa_status s = check_attention_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                       scale, q_dtype, cache_dtype, k_scale, v_scale, workspace);
    if (s != PA_OK) return s;
    if (num_seqs == 0) return PA_OK;
    return decode_impl(out, q, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                       num_q_heads, num_kv_heads, scale, q_dtype, cache_dtype, k_scale, v_scale, workspace,
                       workspace_bytes, num_workers, num_blocks, block_size, num_seqs,
                       reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                  int num_seqs, int prefix_blocks, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int num_blocks, float scale, pa_dtype q_dtype,
                                  pa_dtype cache_dtype, const float* k_scale, const float* v_scale,
                                  void* workspace, size_t workspace_bytes, pa_stream_t stream) {
    pa_status s = check_attention_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                       scale, q_dtype, cache_dtype, k_scale, v_scale, workspace);
    if (s != PA_OK) return s;
    if (prefix_blocks < 0 || prefix_blocks > max_blocks_per_seq) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (workspace_bytes < pa_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim)) return PA_ERR_WORKSPACE;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    DeviceState* st = device_state(nullptr);
    if (!st) return PA_ERR_CUDA;
    // the split runs at a 16-key boundary: with 8-token blocks an odd last shared
    // block goes to every sequence's own part
    const int prefix_units = static_cast<int>(static_cast<long long>(prefix_blocks) * block_size / kBlockSize);
    const size_t base = pa_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim);
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int splits = 1, steps = 0;
    long long pair_ctas = 0;
    if (prefix_units > 0) {
        // Key segments of the prefix (each leaves its own partial rows): only when the
        // prefix grid, 4 us or so per 128-key step of a CTA, would outlast the decode
        // of the private blocks (at 5 TB/s, their mean length taken as half the
        // table's private width: the lengths are on the device), and only as many as
        // keep the prefix grid on under half the SMs and fit the workspace.
        const int per_cta = (chunk_rows() / (num_q_heads / num_kv_heads)) * chunk_tiles_per_cta();
        pair_ctas = static_cast<long long>((num_seqs + per_cta - 1) / per_cta) * num_kv_heads;
        const int total_steps = (prefix_units * kBlockSize + 127) / 128;
        const long long suffix_tokens =
            static_cast<long long>(max_blocks_per_seq) * block_size - static_cast<long long>(prefix_units) * kBlockSize;
        const double suffix_bytes = static_cast<double>(num_seqs) * num_kv_heads * (suffix_tokens > 0 ? suffix_tokens : 0) *
                                    kHeadDim * 2 * (is_fp8(cache_dtype) ? 1 : 2);
        const double decode_us = 0.5 * suffix_bytes / 5.0e6;
        long long cap = (st->sms / 2) / pair_ctas;
        if (cap > total_steps) cap = total_steps;
        if (cap > kMaxPrefixSplits) cap = kMaxPrefixSplits;
        auto prefix_us = [&](int k) { return 4.0 * ((total_steps + k - 1) / k) + 6.0; };
        while (splits < cap && prefix_us(splits) > decode_us &&
               prefix_extra_layout(base, rows, splits + 1).end <= workspace_bytes)
            ++splits;
        steps = (total_steps + splits - 1) / splits;
        splits = (total_steps + steps - 1) / steps;     // every segment has at least one step
    }
    const PrefixExtra ex = prefix_extra_layout(base, rows, splits);
    float* o_extra = splits > 1 ? reinterpret_cast<float*>(ws + ex.o_off) : nullptr;
    float* ml_extra = splits > 1 ? reinterpret_cast<float*>(ws + ex.ml_off) : nullptr;
    if (prefix_units > 0) {
        // the shared prefix once, as a dense contraction of every decode row against its keys
        const CacheKind kind = kind_of(cache_dtype);
        CUtensorMap kmap, vmap;
        s = encode_cache_map(&kmap, k_cache, num_blocks, num_kv_heads, block_size, kind == kKindFp8);
        if (s != PA_OK) return s;
        s = encode_cache_map(&vmap, v_cache, num_blocks, num_kv_heads, block_size, kind == kKindFp8);
        if (s != PA_OK) return s;
        const WorkspaceLayout lay = decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads,
                                                            head_groups_of(num_q_heads, num_kv_heads), 0);
        s = chunk_impl(out, q, nullptr, k_cache, v_cache, kmap, vmap, block_tables, max_blocks_per_seq, seq_lens,
                       num_seqs, num_seqs, num_q_heads, num_kv_heads, num_blocks, block_size, scale, q_dtype,
                       cache_dtype, k_scale, v_scale, workspace, cs, prefix_units,
                       reinterpret_cast<float*>(ws + lay.prefix_o_off), reinterpret_cast<float*>(ws + lay.prefix_ml_off),
                       splits, splits > 1 ? steps : 0, o_extra, ml_extra);
        if (s != PA_OK) return s;
    }
    // the private suffixes stream beside the prefix grid, on the SMs it leaves free;
    // the combine merges both
    int workers = 0;
    if (prefix_units > 0 && pair_ctas * splits < st->sms / 2)
        workers = static_cast<int>(static_cast<long long>(max_workers(*st)) * (st->sms - pair_ctas * splits) / st->sms);
    return decode_impl(out, q, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                       num_q_heads, num_kv_heads, scale, q_dtype, cache_dtype, k_scale, v_scale, workspace,
                       workspace_bytes, workers, num_blocks, block_size, num_seqs, cs, prefix_units > 0, true,
                       prefix_units, splits, o_extra, ml_extra);
}

pa_status pa_decode_append_ex(void* out, const void* q, const void* k_new, const void* v_new,
                              const int64_t* slot_mapping, void* k_cache, void* v_cache, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int num_q_heads,
                              int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                              pa_dtype q_dtype, pa_dtype cache_dtype, const float* k_scale, const float* v_scale,
                              void* workspace, size_t workspace_bytes, int num_workers, pa_stream_t stream) {
    pa_status s = check_attention_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                       scale, q_dtype, cache_dtype, k_scale, v_scale, workspace);
    if (s != PA_OK) return s;
    if (!k_new || !v_new || !slot_mapping || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    return decode_impl(out, q, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                       num_q_heads, num_kv_heads, scale, q_dtype, cache_dtype, k_scale, v_scale, workspace,
                       workspace_bytes, num_workers, num_blocks, block_size, num_seqs,
                       reinterpret_cast<cudaStream_t>(stream), false, false, 0, 1, nullptr, nullptr, k_new, v_new,
                       slot_mapping);
}

pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                           const int64_t* slot_mapping, void* k_cache, void* v_cache, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                           pa_dtype q_dtype, pa_dtype cache_dtype, const float* k_scale, const float* v_scale,
                           void* workspace, size_t workspace_bytes, pa_stream_t stream) {
    return pa_decode_append_ex(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                               max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, num_blocks, scale, q_dtype, cache_dtype, k_scale, v_scale, workspace,
                               workspace_bytes, 0, stream);
}

pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                    pa_dtype q_dtype, pa_dtype cache_dtype, const float* k_scale, const float* v_scale,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream) {
    return pa_decode_ex(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, q_dtype, cache_dtype,
                        k_scale, v_scale, workspace, workspace_bytes, 0, stream);
}

pa_status pa_mixed(void* out, const void* q, const int32_t* query_start_loc, const void* k_cache,
                   const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                   int num_seqs, int total_q, int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
                   int block_size, int num_blocks, float scale, pa_dtype q_dtype, pa_dtype cache_dtype,
                   const float* k_scale, const float* v_scale, void* workspace, size_t workspace_bytes,
                   pa_stream_t stream) {
    pa_status s = check_attention_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                       scale, q_dtype, cache_dtype, k_scale, v_scale, workspace);
    if (s != PA_OK) return s;
    if ((num_seqs > 0 && !query_start_loc) || total_q < 0 || max_q_len < 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_q == 0) return PA_OK;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const bool chunks = max_q_len >= 2;
    if (chunks) {
        const CacheKind kind = kind_of(cache_dtype);
        CUtensorMap kmap, vmap;
        s = encode_cache_map(&kmap, k_cache, num_blocks, num_kv_heads, block_size, kind == kKindFp8);
        if (s != PA_OK) return s;
        s = encode_cache_map(&vmap, v_cache, num_blocks, num_kv_heads, block_size, kind == kKindFp8);
        if (s != PA_OK) return s;
        s = chunk_impl(out, q, query_start_loc, k_cache, v_cache, kmap, vmap, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                       total_q, num_q_heads, num_kv_heads, num_blocks, block_size, scale, q_dtype, cache_dtype, k_scale,
                       v_scale, workspace, cs);
        if (s != PA_OK) return s;
    }
    // the decode rows stream K/V while the chunk tiles keep the tensor cores busy: the
    // decode grid starts once every chunk CTA is resident and fills the SMs the
    // chunk grid leaves idle
    return decode_impl(out, q, query_start_loc, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                       num_seqs, num_q_heads, num_kv_heads, scale, q_dtype, cache_dtype, k_scale, v_scale,
                       workspace, workspace_bytes, 0, num_blocks, block_size, total_q, cs, chunks);
}

pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                            int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int num_blocks, float scale, pa_dtype q_dtype, pa_dtype cache_dtype,
                            const float* k_scale, const float* v_scale, pa_stream_t stream) {
    void* scratch = nullptr;
    DeviceState* st = nullptr;
    pa_status s = noalloc_scratch(&scratch, &st);
    if (s != PA_OK) return s;
    s = check_attention_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                             num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, q_dtype,
                             cache_dtype, k_scale, v_scale, scratch);
    if (s != PA_OK) return s;
    if (num_seqs == 0) return PA_OK;
    // the largest worker count this device can use bounds the scratch a call needs
    const size_t need = decode_workspace_layout(num_seqs, num_q_heads, num_kv_heads,
                                                head_groups_of(num_q_heads, num_kv_heads), 2 * max_workers(*st)).total;
    if (need > kNoAllocScratchBytes) {
        snprintf(g_last_error, sizeof g_last_error,
                 "pa_decode_noalloc: this batch needs %zu bytes of scratch; the static scratch holds %zu",
                 need, kNoAllocScratchBytes);
        return PA_ERR_WORKSPACE;
    }
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // the device status word must start at zero; the rest is written before it is read
    s = cuda_status(cudaMemsetAsync(scratch, 0, 256, cs), "cudaMemsetAsync(scratch status)");
    if (s != PA_OK) return s;
    return decode_impl(out, q, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                       num_q_heads, num_kv_heads, scale, q_dtype, cache_dtype, k_scale, v_scale, scratch,
                       kNoAllocScratchBytes, 0, num_blocks, block_size, num_seqs, cs);
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int num_pairs,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks, pa_dtype cache_dtype,
                         void* workspace, pa_stream_t stream) {
    if (num_pairs < 0 || num_kv_heads < 1 || num_blocks < 1) return PA_ERR_INVALID_ARG;
    if (head_dim != kHeadDim || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
    if (cache_dtype != PA_BF16 && cache_dtype != PA_FP16 && !is_fp8(cache_dtype)) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !src || !dst || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PA_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, 256)) return PA_ERR_INVALID_ARG;
    const size_t block_bytes = static_cast<size_t>(num_kv_heads) * block_size * kHeadDim *
                               (is_fp8(cache_dtype) ? 1 : 2);
    return launched(launch_copy_blocks(k_cache, v_cache, src, dst, num_pairs, num_blocks, block_bytes,
                                          static_cast<int*>(workspace), reinterpret_cast<cudaStream_t>(stream)),
                       "launch(copy_blocks)");
}

pa_status pa_read_device_status(void* workspace, pa_stream_t stream) {
    if (!workspace) return PA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int word = 0;
    cudaError_t e;
    if ((e = cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return fail("cudaMemcpyAsync(status)", e);
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail("cudaStreamSynchronize", e);
    if (word != 0) {
        if ((e = cudaMemsetAsync(workspace, 0, sizeof(int), s)) != cudaSuccess) return fail("cudaMemsetAsync", e);
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail("cudaStreamSynchronize", e);
    }
    if (word & kDevErrTimeout) return PA_ERR_TIMEOUT;
    if (word & kDevErrRange) return PA_ERR_OUT_OF_RANGE;
    return PA_OK;
}

pa_status pa_selftest_wait_timeout(void* workspace, size_t workspace_bytes, unsigned timeout_us,
                                   pa_stream_t stream) {
    if (!workspace || workspace_bytes < 256 || !aligned(workspace, 256)) return PA_ERR_INVALID_ARG;
    if (timeout_us == 0 || timeout_us > 10u * 1000u * 1000u) return PA_ERR_INVALID_ARG;
    return launched(launch_wait_selftest(static_cast<int*>(workspace), 1000ull * timeout_us,
                                            reinterpret_cast<cudaStream_t>(stream)),
                       "launch(reshape_and_cache)");
}

}  // extern "C"
