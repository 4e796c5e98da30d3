/*
 * pa.h -- C ABI of the paged-KV-cache attention library (libpa.so), sm_103a.
 *
 * The operations follow the statement of the problem on three web pages:
 *   [P1] "Basics of LLM Inference and vLLM Internals: KV Cache, PagedAttention,
 *        and Scheduler" -- s.2 "KV Cache and Sizing Formulas", s.4 "PagedAttention
 *        and Block Management", s.6 "Chunked Prefill, Scheduler, and Preemption";
 *   [P2] drpranayjha.com (Red Hat AI Inference Server part) -- "How PagedAttention
 *        pages the KV cache";
 *   [P3] "The Memory Trick Behind Fast LLM Serving" -- "PagedAttention changes
 *        the shape of the problem", "Batching does not merge the conversations".
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory.   Every pointer argument named as "device" is caller-owned GPU memory
 *           of the current device; the library allocates no memory, keeps no
 *           state besides per-device attribute caches, and never synchronises
 *           the stream (except pa_read_device_status, which says so).
 * Streams.  Work is enqueued asynchronously on `stream` (NULL = legacy default
 *           stream).  pa_stream_t is the same handle as cudaStream_t.
 * Errors.   Host-checkable problems are reported before anything is launched:
 *           PA_ERR_INVALID_ARG (null pointer, negative count, misaligned buffer,
 *           H_q not a multiple of H_kv, ...; the per-sequence or per-token arrays
 *           of an empty batch may be null: such a call does nothing and returns
 *           PA_OK), PA_ERR_UNSUPPORTED (head_dim != 128,
 *           block_size not 8, 16 or 32, dtype pair not listed), PA_ERR_WORKSPACE (workspace
 *           too small).  A failed launch returns PA_ERR_CUDA.  Problems only the
 *           device can see (a block-table entry outside the pool, a bounded wait
 *           that ran out) are recorded in the workspace's status word and
 *           returned by pa_read_device_status; kernels never trap.
 * Shapes.   head_dim d = 128; block_size bs = 8, 16 (the default the pages
 *           use) or 32: larger blocks waste more of a sequence's last block,
 *           smaller ones cut the kernels' contiguous runs [P1 s.11, question 3].
 *           Cache layout is [num_blocks][num_kv_heads][bs][128] for both K and V,
 *           so one (block, KV head) tile is bs x 128 contiguous elements (4 KiB
 *           in bf16/fp16 and 2 KiB in FP8 at bs = 16).  A slot number is
 *           physical_block * bs + offset.
 * GQA.      Query head h reads KV head h / (num_q_heads / num_kv_heads):
 *           consecutive query heads form a group [P1 s.2].
 * FP8.      FP8-E4M3 ("fn": bias 7, max 448, no inf, NaN = S.1111.111) with
 *           float32 scales, separate for K and V, one per tensor (PA_FP8_E4M3) or
 *           one per KV head (PA_FP8_E4M3_PER_HEAD), read from device memory so
 *           that calls can be captured in CUDA graphs.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pa_stream_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,
    PA_ERR_UNSUPPORTED = 2,
    PA_ERR_CUDA = 3,
    PA_ERR_TIMEOUT = 4,        /* device: a bounded wait gave up */
    PA_ERR_OUT_OF_RANGE = 5,   /* device: a block-table entry outside [0, num_blocks) */
    PA_ERR_WORKSPACE = 6
} pa_status;

/*
 * Element types.  PA_FP8_E4M3 caches carry one float32 scale per tensor (k_scale,
 * v_scale point to one float each); PA_FP8_E4M3_PER_HEAD caches hold the same
 * e4m3 codes with one scale per KV head (k_scale, v_scale point to
 * num_kv_heads floats, head h's elements dequantised with scale[h]).  The pages
 * mention an FP8 KV cache [P1 s.7 "--kv-cache-dtype fp8"] but not its scaling;
 * per-head scales are this library's variant of it.
 */
typedef enum { PA_BF16 = 0, PA_FP16 = 1, PA_FP8_E4M3 = 2, PA_FP8_E4M3_PER_HEAD = 3 } pa_dtype;

/* Static description of a status code.  Never NULL. */
PA_API const char* pa_status_string(int status);

/* Library ABI version (major * 100 + minor). */
PA_API int pa_version(void);

/* Kernels this library has enqueued in this process (every entry point counts the
 * launches it makes; a launch into a stream being captured counts once, at
 * capture).  A caller can read it before and after a call to see how many kernels
 * the call launches. */
PA_API unsigned long long pa_kernel_launches(void);

/* Text of the last CUDA failure seen by a call of this thread that returned
 * PA_ERR_CUDA (which CUDA call failed and its error string); "" if none.  The
 * buffer is thread-local and valid until the next failing call. */
PA_API const char* pa_last_error(void);

/*
 * Slot write ("reshape_and_cache") [P1 s.4 block table; P3 "PagedAttention
 * changes the shape of the problem"].
 *
 * For every new token t in [0, num_tokens) with slot = slot_mapping[t] >= 0,
 * stores k[t][h][:] into k_cache[slot / bs][h][slot % bs][:] and v[t][h][:]
 * into v_cache at the same place, for every KV head h.  A negative slot is
 * padding and writes nothing.  A slot >= num_blocks * block_size is skipped (nothing is
 * written).  Two tokens with the same slot in one call: undefined which wins.
 *
 *   k, v           device, [num_tokens][num_kv_heads][128] of src_dtype (bf16|fp16)
 *   k_cache,v_cache device, [num_blocks][num_kv_heads][16][128] of cache_dtype,
 *                  16-byte aligned
 *   slot_mapping   device, int64 [num_tokens]
 *   cache_dtype    == src_dtype (bits copied unchanged), or PA_FP8_E4M3:
 *                  code = e4m3(fl32(x) / scale), the quotient rounded once to
 *                  binary32 (IEEE division), then round-to-nearest-even to E4M3 with
 *                  magnitudes above 448 clamped to 448; a NaN quotient ->
 *                  S.1111.111 with S the sign bit of the source element x; a zero
 *                  result keeps the quotient's sign [P1 s.2, s.7 "--kv-cache-dtype fp8"];
 *                  or PA_FP8_E4M3_PER_HEAD: the same with head h's scale[h].
 *   k_scale,v_scale device float32: one each (PA_FP8_E4M3) or num_kv_heads each
 *                  (PA_FP8_E4M3_PER_HEAD); required (non-NULL) iff FP8.
 * Bytes outside the written slots are never touched.
 */
PA_API pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, pa_dtype src_dtype,
                               pa_dtype cache_dtype, const float* k_scale, const float* v_scale,
                               pa_stream_t stream);

/*
 * Bytes of workspace pa_decode / pa_mixed need on the CURRENT device for
 * num_seqs sequences (the default worker count depends on the device's SM
 * count).  The workspace is caller-owned device memory, 256-byte aligned.  Its
 * first 256 bytes must be zero before the first call: they hold the device
 * status word (the first word, see pa_read_device_status) and the counter from
 * which decode warps claim the last pieces of work, which every call leaves
 * ready for the next.  The rest is scratch each call overwrites before reading
 * and needs no initialisation.  One workspace must not be used by two calls
 * that may overlap on the GPU.  Returns 0 for invalid arguments.
 */
PA_API size_t pa_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim);

/*
 * Bytes of workspace with which pa_decode_shared_prefix can cut the shared
 * prefix into as many key segments as it wants (up to 16 partials per query
 * row: num_seqs * num_q_heads * 520 bytes each beyond pa_workspace_size).
 * Same rules as pa_workspace_size.  Returns 0 for invalid arguments.
 */
PA_API size_t pa_workspace_size_shared_prefix(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim);

/* Default number of decode workers (warps) on the current device for a 16-bit
 * cache: two 4-warp CTAs per SM.  An FP8 cache defaults to twice as many (four
 * CTAs per SM: its warps are bound by the latency of the work on each block, not
 * by HBM); the 16-bit decode rows of pa_mixed and the private suffixes of
 * pa_decode_shared_prefix run three CTAs per SM (shorter rings: those grids run
 * beside another grid).  Explicit worker counts run from 1 to this value. */
PA_API int pa_default_workers(void);

/*
 * Decode attention over the paged cache [P1 s.2 "attention revisits the keys
 * and values of all preceding tokens", s.4 block table; P2 "How PagedAttention
 * pages the KV cache"].
 *
 * For every sequence s and query head h (KV head kh = h / G, G = H_q / H_kv):
 *   out[s][h][:] = softmax_t( scale * q[s][h] . K_s[t] ) . V_s[t],  t < seq_lens[s]
 * where token t of sequence s lives in physical block block_tables[s][t / 16],
 * offset t % 16, KV head kh.  seq_lens[s] counts every cached token, including
 * this step's own (write it with pa_reshape_and_cache first).  seq_lens[s] == 0
 * gives zeros.  Entries of block_tables past ceil(seq_lens[s] / 16) are never
 * read.  An entry that is read and lies outside [0, num_blocks) is replaced by
 * block 0 and recorded as PA_ERR_OUT_OF_RANGE in the workspace status word.
 *
 *   out            device, [num_seqs][num_q_heads][128] of q_dtype
 *   q              device, [num_seqs][num_q_heads][128], q_dtype bf16|fp16, 16-byte aligned
 *   k_cache,v_cache device, layout above; cache_dtype == q_dtype, PA_FP8_E4M3 or
 *                  PA_FP8_E4M3_PER_HEAD
 *   block_tables   device, int32 [num_seqs][max_blocks_per_seq]
 *   seq_lens       device, int32 [num_seqs]; each <= block_size * max_blocks_per_seq
 *   scale          softmax scale (e.g. 1/sqrt(128))
 *   k_scale,v_scale device float32 scalars, required iff cache is FP8 (dequant
 *                  is code * scale)
 *   workspace      see pa_workspace_size
 * num_seqs <= 8192.  The work is split evenly over the workers by cached
 * blocks; a sequence split across workers is merged by a log-sum-exp combine
 * launched behind the decode kernel on the same stream.  The result does not
 * depend on where blocks live.
 */
PA_API pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                    int num_blocks, float scale, pa_dtype q_dtype, pa_dtype cache_dtype,
                    const float* k_scale, const float* v_scale, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream);

/*
 * One decode step in one pass: pa_reshape_and_cache of each sequence's new token
 * followed by pa_decode, with the same results (the cache bytes bit for bit, the
 * outputs exactly) [P1 s.3: each step appends one token per running request and
 * attends over all of them; s.4 slot mapping].  The warps that read a sequence's
 * last 16 keys store its new token into the cache slot first, so the slot write
 * costs no separate launch.
 *
 *   k_new, v_new   device, [num_seqs][num_kv_heads][128] of q_dtype, 16-byte aligned
 *   slot_mapping   device, int64 [num_seqs]: slot_mapping[s] must be the slot of
 *                  position seq_lens[s] - 1 of sequence s (block
 *                  block_tables[s][(seq_lens[s] - 1) / block_size], offset
 *                  (seq_lens[s] - 1) % block_size), or negative (padding: nothing is
 *                  written).  Another slot, or a non-negative slot for an empty
 *                  sequence, is recorded as PA_ERR_OUT_OF_RANGE and not written.
 *   k_cache, v_cache written at those slots (FP8 with the pa_reshape_and_cache rule)
 * The block holding a new token must belong to its sequence alone (copy it first
 * when it is shared, see pa_pool_copy_on_write).  Other arguments as pa_decode.
 */
PA_API pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                                  const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                  int num_blocks, float scale, pa_dtype q_dtype, pa_dtype cache_dtype,
                                  const float* k_scale, const float* v_scale, void* workspace,
                                  size_t workspace_bytes, pa_stream_t stream);

/* pa_decode_append with an explicit worker count (1 .. pa_default_workers(); 0 =
 * the default), as pa_decode_ex is to pa_decode.  The cache bytes it writes do not
 * depend on the worker count; outputs agree with pa_decode_append to rounding.
 * With long ranges per worker (>= 48 16-key units, 16-bit cache, at most 4
 * query heads per KV head) the last ~10% of the work is handed out at run time
 * in pieces, so a small worker count is how a small batch reaches that path. */
PA_API pa_status pa_decode_append_ex(void* out, const void* q, const void* k_new, const void* v_new,
                                     const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int num_blocks, float scale,
                                     pa_dtype q_dtype, pa_dtype cache_dtype, const float* k_scale,
                                     const float* v_scale, void* workspace, size_t workspace_bytes,
                                     int num_workers, pa_stream_t stream);

/* pa_decode with an explicit worker count (1 .. pa_default_workers(); 0 = the
 * default).  Fewer workers means longer ranges per worker and fewer split
 * points; results agree with pa_decode to rounding. */
PA_API pa_status pa_decode_ex(void* out, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                       int head_dim, int block_size, int num_blocks, float scale,
                       pa_dtype q_dtype, pa_dtype cache_dtype, const float* k_scale,
                       const float* v_scale, void* workspace, size_t workspace_bytes,
                       int num_workers, pa_stream_t stream);

/*
 * Decode for a batch whose block tables share their leading blocks: the same
 * result as pa_decode, computed in cascade.  The pages describe requests that
 * start with the same prompt reusing the same full KV blocks, so that their
 * block tables point at the same physical blocks [P3 "Prefix caching is the
 * second win"; P1 s.4 block table, s.5 prefix caching]; they give no kernel for
 * it (the cascade split below is this library's).
 *
 * Precondition: for every sequence s, block_tables[s][j] == block_tables[0][j]
 * for j < prefix_blocks, and seq_lens[s] >= block_size * prefix_blocks.  A batch
 * that violates it is recorded as PA_ERR_OUT_OF_RANGE in the workspace status
 * word (its outputs are then unspecified).  The split between the shared part
 * and the private parts falls on a multiple of 16 keys: with 8-token blocks and
 * an odd prefix_blocks the last shared block is read with each sequence's
 * private blocks (and is not checked against the precondition).
 *
 * The prefix keys are read once for the whole batch: every decode row of every
 * sequence is contracted against them on the tensor cores as one dense tile
 * grid (one CTA per 256 query rows of a KV head and key segment), leaving an
 * unnormalised partial per row and segment; the private blocks after the
 * prefix stream through the decode kernel; the combine kernel merges all of
 * them by log-sum-exp.  The prefix is cut into key segments of whole 128-key
 * steps until its grid has about one CTA per SM, as far as the workspace
 * holds the extra partials; a prefix grid under half the SMs runs beside the
 * decode grid (which then takes the other SMs), a larger one runs first.
 * prefix_blocks == 0 reduces to pa_decode with every row merged by the
 * combine.
 *
 *   prefix_blocks  host, 0 <= prefix_blocks <= max_blocks_per_seq
 *   workspace      at least pa_workspace_size(num_seqs, num_q_heads,
 *                  num_kv_heads, head_dim) bytes (then the prefix is one
 *                  segment); pa_workspace_size_shared_prefix bytes allow
 *                  every split
 * Other arguments as pa_decode; results agree with pa_decode to rounding.
 */
PA_API pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* seq_lens, int num_seqs, int prefix_blocks,
                                  int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                  int num_blocks, float scale, pa_dtype q_dtype, pa_dtype cache_dtype,
                                  const float* k_scale, const float* v_scale, void* workspace,
                                  size_t workspace_bytes, pa_stream_t stream);

/*
 * Mixed batch: decode rows and prefill chunks in one flattened query array
 * [P3 "Batching does not merge the conversations"; P1 s.6 chunked prefill].
 *
 * Sequence s owns query rows query_start_loc[s] .. query_start_loc[s+1]-1
 * (q_len_s rows).  seq_lens[s] counts the cached tokens including this step's
 * q_len_s new ones, so row j of sequence s sits at position
 * pos = seq_lens[s] - q_len_s + j and attends causally to tokens 0 .. pos of its
 * own sequence only.  q_len_s == 1 is a decode row; q_len_s == 0 contributes
 * nothing.
 *
 *   out, q          device, [total_q][num_q_heads][128] of q_dtype
 *   query_start_loc device, int32 [num_seqs + 1], non-decreasing,
 *                   query_start_loc[0] == 0, query_start_loc[num_seqs] == total_q
 *   max_q_len       host upper bound of q_len_s (0 or 1: no prefill chunks, the
 *                   prefill kernel is not launched)
 * Other arguments as pa_decode.
 */
PA_API pa_status pa_mixed(void* out, const void* q, const int32_t* query_start_loc, const void* k_cache,
                   const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* seq_lens, int num_seqs, int total_q, int max_q_len,
                   int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   float scale, pa_dtype q_dtype, pa_dtype cache_dtype, const float* k_scale,
                   const float* v_scale, void* workspace, size_t workspace_bytes,
                   pa_stream_t stream);

/*
 * Decode without a caller-provided workspace (no counterpart on the pages; the
 * pages do not discuss memory ownership of the kernels).
 *
 * Same computation and arguments as pa_decode, minus the workspace.  It is for
 * callers that cannot allocate device memory themselves: a plugin or host
 * framework that hands over only input and output buffers, or a latency-critical
 * path where cudaMalloc / cudaFree (which may synchronise the device) are not
 * allowed.  The scratch lives in one static 16 MiB device array inside libpa.so;
 * every GPU that loads the library holds it until the process exits.  This call
 * allocates nothing and calls no allocating routine.
 *
 *  - Limit: the batch must fit the 16 MiB scratch.  With S = num_seqs,
 *    G = num_q_heads / num_kv_heads, W = pa_default_workers() (1216 on a 152-SM
 *    GB300), N = S * num_kv_heads * ceil(G / 8) + 2 W partial slots and R(x) = x
 *    rounded up to a multiple of 256, a call needs
 *        256 + R(4 (S + 1)) + R(512 S num_q_heads) + R(8 S num_q_heads)
 *            + R(64 N) + 4096 N
 *    bytes; the 2 W slots alone take about 10.1 MB on a 152-SM GB300.  There
 *    that allows at most 100 sequences with 64 query and 8 KV heads, 133 with
 *    32 and 8, 177 with 8 and 8, 457 with 12 and 2, 533 with 8 and 2.  Larger
 *    batches return PA_ERR_WORKSPACE with the sizes in pa_last_error().
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current and caches it; make that
 *    first call before any stream capture.
 *  - All calls share the one array, which keeps the previous call's contents;
 *    each call clears the part that must start at zero (the status word and
 *    the work counter at its head) on its stream.  Calls that may overlap on the GPU (other streams, other threads)
 *    race on the array and give undefined results: serialise them.
 *  - Device-side reports (PA_ERR_OUT_OF_RANGE for a bad block-table entry,
 *    PA_ERR_TIMEOUT) stay in the static array, where no caller can read them,
 *    and the next call clears them: this call cannot report them.  A caller
 *    that needs those checks must use pa_decode with a workspace and read it
 *    with pa_read_device_status.
 */
PA_API pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                   float scale, pa_dtype q_dtype, pa_dtype cache_dtype,
                                   const float* k_scale, const float* v_scale, pa_stream_t stream);

/*
 * Block copies for copy-on-write [P1 s.4: a physical block shared by several
 * block tables carries a reference count; a sequence about to write into a
 * shared block needs its own copy first].
 *
 * For i < num_pairs: block dst[i] <- block src[i], every KV head, in both
 * caches (layout as pa_decode).  The dst blocks must be distinct and none may be
 * a src block of the same call (the result is otherwise unspecified).  An id
 * outside [0, num_blocks) skips its pair and, when workspace is not NULL, is
 * recorded as PA_ERR_OUT_OF_RANGE in its status word.
 *
 *   src, dst        device, int32 [num_pairs]
 *   workspace       NULL, or a workspace whose status word records errors
 */
PA_API pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst,
                                int num_pairs, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                pa_dtype cache_dtype, void* workspace, pa_stream_t stream);

/*
 * Block pool (host memory, no GPU work) [P1 s.4 "PagedAttention and Block
 * Management", s.5 "Prefix Caching"; P3 "The block pool", "Prefix caching is the
 * second win"].
 *
 * A pool of num_blocks physical blocks of block_size tokens.  Block 0 is the
 * null block and is never handed out, so num_blocks - 1 are usable.  Free blocks
 * wait in one queue; allocation takes them from the front.  A block in use has
 * a reference count (one per block table holding it).  A full block of a prompt
 * is registered under a chained hash (the previous block's hash, its own
 * tokens, and extra_key at the root of the chain); when its count drops to zero
 * it keeps that content and goes to the back of the queue (a request's last
 * blocks ahead of its earlier ones), so later prompts with the same prefix can
 * reuse it until the front of the queue reaches it.  A block without registered
 * content goes to the front.  Hits are checked against the stored tokens.
 *
 * Functions return PA_ERR_INVALID_ARG for bad arguments (NULL pool, an id that
 * is not in use where one must be), PA_ERR_OUT_OF_RANGE when the queue holds
 * too few blocks (then nothing changes).  A pool serialises its own calls.
 */
typedef struct pa_block_pool pa_block_pool;

/* NULL for num_blocks < 2, block_size < 1 or no memory. */
PA_API pa_block_pool* pa_pool_create(int num_blocks, int block_size);
PA_API void pa_pool_destroy(pa_block_pool* pool);
/* Blocks in the free queue (with or without reusable content). */
PA_API int pa_pool_num_free(pa_block_pool* pool);
/* Blocks holding registered prompt content (in use or free). */
PA_API int pa_pool_num_cached(pa_block_pool* pool);
/* Reference count of a block (0 when free), -1 for an id outside the pool. */
PA_API int pa_pool_ref_count(pa_block_pool* pool, int block);
/* n blocks for new content (count 1; any content they held is dropped). */
PA_API pa_status pa_pool_allocate(pa_block_pool* pool, int n, int32_t* blocks);
/* One more reference to each block (another table aliases it). */
PA_API pa_status pa_pool_share(pa_block_pool* pool, const int32_t* blocks, int n);
/* One reference less to each block, given in table order; blocks reaching zero
 * enter the free queue as described above. */
PA_API pa_status pa_pool_free(pa_block_pool* pool, const int32_t* blocks, int n);
/* Blocks for a prompt of num_tokens tokens: ceil(num_tokens / block_size)
 * entries in `blocks`.  The longest run of leading full blocks whose content is
 * registered is reused (one more reference each), never including the block
 * that holds the last token; the rest are allocated, and their full blocks
 * registered.  *hit_tokens = block_size * reused blocks. */
PA_API pa_status pa_pool_allocate_prompt(pa_block_pool* pool, const int32_t* tokens, int num_tokens,
                                         uint64_t extra_key, int32_t* blocks, int* hit_tokens);
/* Copy-on-write: every blocks[i] with more than one reference is replaced by a
 * newly allocated block (the shared one loses a reference); the (old, new) pairs
 * go to src/dst (n entries each at most) for pa_copy_blocks, *num_copies of
 * them. */
PA_API pa_status pa_pool_copy_on_write(pa_block_pool* pool, int32_t* blocks, int n, int32_t* src, int32_t* dst,
                                       int* num_copies);

/*
 * Reads (and clears) the device-side status word of a workspace.  Synchronises
 * `stream`.  Returns PA_OK, PA_ERR_OUT_OF_RANGE or PA_ERR_TIMEOUT (the first
 * recorded, timeouts first), or PA_ERR_CUDA if the copy failed.
 */
PA_API pa_status pa_read_device_status(void* workspace, pa_stream_t stream);

/*
 * Self-test of the bounded waits: launches one warp that waits on a barrier
 * nothing will ever complete, with a limit of timeout_us microseconds; the wait
 * must give up and record PA_ERR_TIMEOUT in the workspace status word (read it
 * with pa_read_device_status).  Touches only the status word.
 */
PA_API pa_status pa_selftest_wait_timeout(void* workspace, size_t workspace_bytes, unsigned timeout_us,
                                   pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
