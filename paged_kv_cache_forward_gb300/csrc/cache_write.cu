// cache_write.cu -- scatter new tokens' K and V into the paged cache.
//
// The step before attention in a serving loop: the K and V rows computed for
// the new tokens are stored into the paged KV cache of the Triton unified-
// attention page (section "Why is switching the card so hard": the paged KV
// cache), token t going to page slot_mapping[t] / P, slot slot_mapping[t] % P.
// A negative slot is padding and writes nothing.  HBM-bound: every byte of
// k_new and v_new is read once and written once with 16-byte vector accesses;
// one CTA of 128 threads per token row pair, so the grid is the token count.
// A slot past the pool is recorded in the sticky error word and skipped.

#include <cuda_bf16.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) cache_write_kernel(const uint4* __restrict__ k_new,
                                                              const uint4* __restrict__ v_new,
                                                              const int64_t* __restrict__ slot_mapping,
                                                              uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                              int64_t num_slots, int row_chunks, int32_t* err) {
    const int64_t t = blockIdx.x;
    // The slot and the token's rows are loaded together (the rows do not depend
    // on the slot), so a CTA waits for one round trip before its stores, not two.
    const int64_t s = slot_mapping[t];
    const bool ok = s >= 0 && s < num_slots;  // s < 0: a token that is not cached
    if (s >= num_slots && threadIdx.x == 0) flag_error(err, kDevBadBlock);
    // a token row is row_chunks 16-byte chunks ([Hkv, D] bf16), contiguous in
    // both the new-token tensors and the cache (slot s is row s of the cache)
    const int64_t src = t * row_chunks, dst = s * row_chunks;
    for (int c = threadIdx.x; c < row_chunks; c += kThreads) {
        const uint4 kv = __ldcs(k_new + src + c);  // streamed: read once
        const uint4 vv = __ldcs(v_new + src + c);
        if (ok) {
            k_cache[dst + c] = kv;
            v_cache[dst + c] = vv;
        }
    }
}

}  // namespace

cudaError_t launch_cache_write(const void* k_new, const void* v_new, const int64_t* slot_mapping, void* k_cache,
                               void* v_cache, int64_t num_tokens, int64_t num_blocks, int32_t page_size,
                               int32_t num_kv_heads, int32_t head_dim, int32_t* err, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int row_chunks = num_kv_heads * head_dim / 8;
    return launch_kernel(cache_write_kernel, static_cast<unsigned>(num_tokens), kThreads, 0, stream, 1, false,
                         static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
                         static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_blocks * page_size,
                         row_chunks, err);
}

}  // namespace pa
