// cache_write.cu -- scatter new tokens' K and V into the paged cache.
//
// The step before attention in a serving loop: the K and V rows computed for
// the new tokens are stored into the paged KV cache of the Triton unified-
// attention page (section "Why is switching the card so hard": the paged KV
// cache), token t going to page slot_mapping[t] / P, slot slot_mapping[t] % P.
// A negative slot is padding and writes nothing.  HBM-bound: every byte of
// k_new and v_new is read once and written once with 16-byte vector accesses;
// one CTA of 128 threads per kTok tokens.  A slot past the pool is recorded in
// the sticky error word and skipped.

#include <cuda_bf16.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 128;
// Tokens per CTA: their slots and rows are all in flight together (the
// varlen prefill's 11273 tokens: 1 token 16.6 us, 2 tokens 15.6 us, 4 16.0 us,
// 8 16.7 us).
constexpr int kTok = 2;

__global__ void __launch_bounds__(kThreads) cache_write_kernel(const uint4* __restrict__ k_new,
                                                              const uint4* __restrict__ v_new,
                                                              const int64_t* __restrict__ slot_mapping,
                                                              uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                              int64_t num_tokens, int64_t num_slots, int row_chunks,
                                                              int32_t* err) {
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTok;
    int64_t s[kTok];
#pragma unroll
    for (int j = 0; j < kTok; ++j) s[j] = t0 + j < num_tokens ? slot_mapping[t0 + j] : -1;
    for (int c = threadIdx.x; c < row_chunks; c += kThreads) {
        uint4 kv[kTok], vv[kTok];
#pragma unroll
        for (int j = 0; j < kTok; ++j)
            if (t0 + j < num_tokens) {
                kv[j] = __ldcs(k_new + (t0 + j) * row_chunks + c);
                vv[j] = __ldcs(v_new + (t0 + j) * row_chunks + c);
            }
#pragma unroll
        for (int j = 0; j < kTok; ++j)
            if (s[j] >= 0 && s[j] < num_slots) {
                k_cache[s[j] * row_chunks + c] = kv[j];
                v_cache[s[j] * row_chunks + c] = vv[j];
            }
    }
    if (threadIdx.x == 0)
#pragma unroll
        for (int j = 0; j < kTok; ++j)
            if (s[j] >= num_slots) flag_error(err, kDevBadBlock);
}

}  // namespace

cudaError_t launch_cache_write(const void* k_new, const void* v_new, const int64_t* slot_mapping, void* k_cache,
                               void* v_cache, int64_t num_tokens, int64_t num_blocks, int32_t page_size,
                               int32_t num_kv_heads, int32_t head_dim, int32_t* err, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int row_chunks = num_kv_heads * head_dim / 8;
    return launch_kernel(cache_write_kernel, static_cast<unsigned>((num_tokens + kTok - 1) / kTok), kThreads, 0,
                         stream, 1, false, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                         slot_mapping, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_tokens,
                         num_blocks * page_size, row_chunks, err);
}

}  // namespace pa
