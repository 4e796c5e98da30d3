// Block copies for copy-on-write: dst[i] <- src[i], every KV head, K and V.
//
// Problem ("Basics of LLM Inference and vLLM Internals", s.4: physical blocks
// shared by several block tables carry a reference count): before a sequence
// writes a new token into a block it shares, it needs a private copy of that
// block.  The copy is pure data movement (HBM-bound): one CTA per (pair, cache),
// 16-byte vector loads and stores over the block's contiguous H_kv x 16 x 128
// elements.
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

__global__ void __launch_bounds__(256) copy_blocks_kernel(uint8_t* k_cache, uint8_t* v_cache, const int32_t* src,
                                                          const int32_t* dst, int num_blocks, size_t block_bytes,
                                                          int* status) {
    grid_dependency_wait();
    const int i = blockIdx.x;
    const int s = src[i], d = dst[i];
    if (static_cast<unsigned>(s) >= static_cast<unsigned>(num_blocks) ||
        static_cast<unsigned>(d) >= static_cast<unsigned>(num_blocks)) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && status) atomicOr(status, kDevErrRange);
        return;
    }
    uint8_t* cache = blockIdx.y == 0 ? k_cache : v_cache;
    const uint4* from = reinterpret_cast<const uint4*>(cache + static_cast<size_t>(s) * block_bytes);
    uint4* to = reinterpret_cast<uint4*>(cache + static_cast<size_t>(d) * block_bytes);
    const size_t n = block_bytes / 16;
    for (size_t e = threadIdx.x; e < n; e += blockDim.x) to[e] = __ldg(from + e);
    grid_launch_dependents();
}

}  // namespace

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int num_pairs,
                               int num_blocks, size_t block_bytes, int* status, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_pairs), 2);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, copy_blocks_kernel, static_cast<uint8_t*>(k_cache),
                              static_cast<uint8_t*>(v_cache), src, dst, num_blocks, block_bytes, status);
}

}  // namespace pa
