// Slot write ("reshape_and_cache") for sm_103a.
//
// Every new token's K and V vectors (one per KV head) go to the cache slot the
// slot mapping names: physical block slot / bs, offset slot % bs for blocks of
// bs = 8, 16 or 32 tokens ("Basics of LLM Inference and vLLM Internals", s.4: a
// block table maps logical blocks to physical blocks; the slot mapping is that
// table resolved per token).
//
// One warp per (token, KV head): lanes 0-15 move the 256-byte K row, lanes
// 16-31 the V row, 16 bytes per lane.  An FP8 cache stores
// e4m3(fl32(x) / scale): IEEE division, then round-to-nearest-even to E4M3 with
// saturation to +-448 (the hardware's satfinite conversion); a NaN quotient
// becomes S.1111.111 with the sign of the source element, and a result of
// magnitude zero keeps the sign of the quotient.
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

template <bool SrcBf16, bool Fp8>
__global__ void __launch_bounds__(256)
    reshape_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, void* k_cache,
                   void* v_cache, const int64_t* __restrict__ slots, int num_tokens, int num_kv_heads,
                   int num_blocks, int block_shift, const float* k_scale, const float* v_scale, int scale_stride) {
    grid_dependency_wait();
    grid_launch_dependents();
    const long long pair = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (pair >= static_cast<long long>(num_tokens) * num_kv_heads) return;
    const int tok = static_cast<int>(pair / num_kv_heads);
    const int h = static_cast<int>(pair % num_kv_heads);
    const long long slot = slots[tok];
    if (slot < 0 || slot >= (static_cast<long long>(num_blocks) << block_shift)) return;
    const int lane = threadIdx.x & 31;
    const bool is_v = lane >= 16;
    const int col = (lane & 15) * 8;
    const uint16_t* src = (is_v ? v : k) + (static_cast<size_t>(tok) * num_kv_heads + h) * kHeadDim + col;
    const size_t dst = (((static_cast<size_t>(slot >> block_shift) * num_kv_heads + h) << block_shift) +
                        static_cast<size_t>(slot & ((1 << block_shift) - 1))) * kHeadDim + col;
    const uint4 x = *reinterpret_cast<const uint4*>(src);
    if constexpr (!Fp8) {
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(is_v ? v_cache : k_cache) + dst) = x;
    } else {
        const float scale = __ldg((is_v ? v_scale : k_scale) + h * scale_stride);   // per tensor or per head
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t out[2];
#pragma unroll
        for (int i = 0; i < 2; ++i)
            out[i] = e4m3_pair<SrcBf16>(w[2 * i], scale) | (e4m3_pair<SrcBf16>(w[2 * i + 1], scale) << 16);
        *reinterpret_cast<uint2*>(static_cast<uint8_t*>(is_v ? v_cache : k_cache) + dst) = make_uint2(out[0], out[1]);
    }
}

}  // namespace

cudaError_t launch_reshape(const void* k, const void* v, void* k_cache, void* v_cache,
                           const int64_t* slots, int num_tokens, int num_kv_heads, int num_blocks,
                           int block_shift, bool src_bf16, bool cache_fp8, const float* k_scale,
                           const float* v_scale, int scale_stride, cudaStream_t stream) {
    const long long pairs = static_cast<long long>(num_tokens) * num_kv_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((pairs + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint16_t* kk = static_cast<const uint16_t*>(k);
    const uint16_t* vv = static_cast<const uint16_t*>(v);
    if (cache_fp8) {
        return src_bf16 ? cudaLaunchKernelEx(&cfg, reshape_kernel<true, true>, kk, vv, k_cache, v_cache, slots,
                                             num_tokens, num_kv_heads, num_blocks, block_shift, k_scale, v_scale,
                                             scale_stride)
                        : cudaLaunchKernelEx(&cfg, reshape_kernel<false, true>, kk, vv, k_cache, v_cache, slots,
                                             num_tokens, num_kv_heads, num_blocks, block_shift, k_scale, v_scale,
                                             scale_stride);
    }
    return cudaLaunchKernelEx(&cfg, reshape_kernel<true, false>, kk, vv, k_cache, v_cache, slots, num_tokens,
                              num_kv_heads, num_blocks, block_shift, k_scale, v_scale, scale_stride);
}

}  // namespace pa
