// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

enum CacheKind { kKindBf16 = 0, kKindFp16 = 1, kKindFp8 = 2 };

constexpr int kHeadDim = 128;
// Keys per MMA unit: the attention kernels walk the cache in 16-key units, whatever
// the physical block size (8, 16 or 32 tokens: half a unit, one, or two).
constexpr int kBlockSize = 16;
constexpr int kMaxSeqs = 8192;
constexpr int kDecodeWarps = 4;        // warps per decode CTA
constexpr int kMaxDecodeCtasPerSm = 2;     // 16-bit caches: their rings fill shared memory
// FP8 caches: four CTAs (three stages each) fill the register file.  An FP8 warp is
// bound by the latency of the work on each block, not by HBM, so more warps per SM
// stream faster; its ranges need no claimed pieces, so its 2x workers fit the same
// partial slots as the 16-bit grid's workers and pieces.
constexpr int kMaxDecodeCtasPerSmFp8 = 4;
// 16-bit caches in a cascade's suffix decode or a mixed batch's decode rows: a
// two-stage ring per warp and three CTAs per SM.  More warps hide the work on each
// block (those grids run beside another grid and their rows are short or come from
// L2); for a plain decode from HBM the deeper ring streams faster.  Their workers and
// pieces take at most 2 x SMs x 3 x 4 partial slots, which pa_workspace_size covers.
constexpr int kMaxDecodeCtasPerSmNarrow = 3;
// Decode work claimed at run time: this share (in 1/256) of the flattened blocks
// goes to pieces of at least kMinPiece blocks (more than a ring holds) when static
// ranges hold at least kMinPieceRange blocks; a claim is sent kClaimAhead blocks
// before the end of the range in hand.
constexpr int kDynShare256 = 26;
constexpr int kMinPiece = 8;
constexpr int kMinPieceRange = 48;
constexpr int kClaimAhead = 4;
constexpr int kHeadsPerGroup = 8;          // query heads handled by one decode unit (MMA N)
// Up to this many sequences the combine kernel finds a unit's place in the flattened
// order itself (before waiting for the decode grid); above it the decode grid
// publishes its block prefix in the workspace.
constexpr int kCombineScanSeqs = 1024;
// Most key segments a shared prefix is cut into (pa_workspace_size_shared_prefix
// holds this many partials per row).
constexpr int kMaxPrefixSplits = 16;

// Bits of the device-side status word (first word of the workspace).
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrRange = 2;

// Decode: one "unit" = (sequence, KV head, group of up to 8 query heads).  The
// cached blocks of all units are laid end to end and cut into ranges: equal
// static ones, one per worker (warp), then pieces the workers claim.  A unit
// covered by several ranges leaves partials in the slots (range r, unit u) ->
// r + u, unique because both indices only grow along the flattened order; the
// combine kernel merges them.
struct DecodeParams {
    void* out;
    const void* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* query_start_loc;   // non-null: mixed batch, only rows with q_len == 1
    const float* k_scale;
    const float* v_scale;
    int scale_stride;                 // FP8 scales: 0 one per tensor, 1 one per KV head
    int* status;                      // device status word
    int* plan;                        // [num_seqs + 1]: block prefix per sequence (large batches only)
    float* ml;                        // [slots][16]: running max (8 heads), sum (8 heads)
    float4* partial;                  // [slots][8][32]: unnormalised output fragments
    int num_seqs;
    int total_rows;                   // rows of q and out (num_seqs, or total_q of a mixed batch)
    int num_q_heads;
    int num_kv_heads;
    int group;                        // query heads per KV head
    int head_groups;                  // ceil(group / 8)
    int max_blocks;                   // block-table row length
    int num_blocks;                   // pool size
    int block_size;                   // tokens per physical block: 8, 16 or 32
    int block_shift;                  // log2(block_size)
    int num_workers;                  // warps taking part
    int dyn256;                       // share of the blocks in claimed pieces, in 1/256
    int narrow;                       // 16-bit cache, two-stage ring (three CTAs per SM)
    unsigned* claim;                  // [0] piece counter, [1] its value when this call began
    int overlap_prior;                // nonzero: the previous launch is this call's chunk kernel,
                                      // which started only after its own predecessors finished;
                                      // run beside it and wait for it only before exiting
    // Shared-prefix (cascade) decode: every table starts with the same first_block
    // physical blocks; the decode grid covers blocks first_block.. only and always
    // leaves partials, and the combine folds in the prefix partial of each row.
    int cascade;                      // nonzero: cascade mode
    int first_block;                  // shared leading 16-key units (cascade mode)
    const float* prefix_o;            // [num_seqs][num_q_heads][128]: unnormalised prefix output
    const float* prefix_ml;           // [num_seqs][num_q_heads][2]: its (max in log2 units, sum)
    int prefix_splits;                // prefix partials per row (key segments of the prefix)
    const float* prefix_o_extra;      // [prefix_splits - 1][num_seqs][num_q_heads][128]
    const float* prefix_ml_extra;     // [prefix_splits - 1][num_seqs][num_q_heads][2]
    // Slot write fused into the decode: the new token of sequence s (row s of k_new /
    // v_new, [num_seqs][num_kv_heads][128] in the query's 16-bit type) goes to slot
    // slots[s], which must be the slot of position seq_lens[s] - 1 (a negative slot
    // is padding); the warps that read the sequence's last 16 keys write it first.
    int append;
    const uint16_t* k_new;
    const uint16_t* v_new;
    const int64_t* slots;
    void* k_cache_w;
    void* v_cache_w;
    float scale_log2;                 // softmax scale * log2(e)
    unsigned long long timeout_ns;    // bound of every barrier wait
};

// Prefill chunk tiles of a mixed batch (causal, no split).
struct ChunkParams {
    void* out;
    const void* q;
    const void* k_cache;              // read directly by the FP8 path
    const void* v_cache;
    const int32_t* query_start_loc;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const float* k_scale;
    const float* v_scale;
    int scale_stride;                 // FP8 scales: 0 one per tensor, 1 one per KV head
    int* status;
    int num_seqs;
    int total_rows;                   // rows of q and out
    int num_q_heads;
    int num_kv_heads;
    int group;
    int max_blocks;
    int num_blocks;
    int block_size;                   // tokens per physical block: 8, 16 or 32
    int block_shift;                  // log2(block_size)
    int queries_per_tile;             // queries of one sequence per CTA tile
    // Prefix mode (prefix_keys > 0): the queries are the decode rows of all
    // sequences ([num_seqs][num_q_heads][128]), every one at position prefix_keys - 1,
    // the keys are the first prefix_keys tokens of sequence 0's table, and the
    // output is unnormalised: prefix_o (f32 rows) and prefix_ml (max, sum).
    // Split prefix: gridDim.z = prefix_splits CTAs per tile pair, segment z covering
    // steps [z prefix_steps, (z + 1) prefix_steps) of 128 keys; segment 0 writes
    // prefix_o / prefix_ml, segment z > 0 the (z - 1)-th block of prefix_o_extra /
    // prefix_ml_extra (same row layout).
    int prefix_keys;
    int prefix_splits;
    int prefix_steps;
    float* prefix_o;
    float* prefix_ml;
    float* prefix_o_extra;
    float* prefix_ml_extra;
    float scale_log2;
    unsigned long long timeout_ns;
};

struct WorkspaceLayout {
    size_t status_off;
    size_t plan_off;
    size_t ml_off;
    size_t partial_off;
    size_t prefix_o_off;              // shared-prefix partials: [num_seqs][num_q_heads][128] f32
    size_t prefix_ml_off;             // and [num_seqs][num_q_heads][2] f32
    size_t total;
};

// range_slots: partial slots besides one per unit (one per static range, plus one per
// claimed piece when pieces are on)
WorkspaceLayout decode_workspace_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_groups,
                                        int range_slots);

// Decode kernels: dynamic shared memory for num_seqs sequences.
// narrow: the 16-bit kernel with a two-stage ring per warp (three CTAs per SM)
size_t decode_smem_bytes(CacheKind kind, int num_seqs, bool narrow);
cudaError_t decode_prepare(CacheKind kind, bool q_bf16, bool append, bool dyn, bool narrow, size_t max_smem);
cudaError_t decode_occupancy(CacheKind kind, bool q_bf16, bool append, bool dyn, bool narrow, size_t smem,
                             int* ctas_per_sm);
cudaError_t launch_decode(CacheKind kind, bool q_bf16, const CUtensorMap& kmap,
                          const CUtensorMap& vmap, const DecodeParams& p, int grid, size_t smem,
                          cudaStream_t stream);
// Block copies (copy-on-write): dst[i] <- src[i] in both caches.
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int num_pairs,
                               int num_blocks, size_t block_bytes, int* status, cudaStream_t stream);

cudaError_t launch_combine(bool out_bf16, bool fp8_cache, const DecodeParams& p, int max_ctas,
                           cudaStream_t stream);

// Slot write.
cudaError_t launch_reshape(const void* k, const void* v, void* k_cache, void* v_cache,
                           const int64_t* slots, int num_tokens, int num_kv_heads, int num_blocks,
                           int block_shift, bool src_bf16, bool cache_fp8, const float* k_scale,
                           const float* v_scale, int scale_stride, cudaStream_t stream);

// Prefill chunks.
size_t chunk_smem_bytes(CacheKind kind, int num_seqs);
int chunk_rows();           // MMA rows of one query tile
int chunk_tiles_per_cta();  // query tiles one CTA processes
cudaError_t chunk_prepare(CacheKind kind, bool q_bf16, size_t max_smem);
cudaError_t launch_chunk(CacheKind kind, bool q_bf16, const CUtensorMap& kmap,
                         const CUtensorMap& vmap, const ChunkParams& p, int grid_x, size_t smem,
                         cudaStream_t stream);

// Bounded-wait self test.
cudaError_t launch_wait_selftest(int* status, unsigned long long timeout_ns, cudaStream_t stream);

}  // namespace pa
