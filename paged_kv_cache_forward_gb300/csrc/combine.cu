// combine.cu -- log-sum-exp merge of split-KV partials.
//
// The last step of the "Parallel Tiled Softmax" item of the five-step list on the
// Triton unified-attention page ("What three things the IBM paper got right"):
// each split s of a decode row left an unnormalised O_s with its running max m_s
// (log2 units) and sum l_s.  The online-softmax recurrence of "The Flash
// Attention revolution" (GPU programming guide page) applied across splits gives
//     M = max_s m_s,  w_s = 2^(m_s - M),  out = (sum_s w_s O_s) / (sum_s w_s l_s).
// One warp per (sequence, query head); the max and the denominator are warp
// shuffle reductions, O is read with 16-byte vector loads.  Splits that saw no
// key do not exist (a split is only launched with work), so every m_s is finite.

#include <cuda_bf16.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kWarpsPerCta = 4;

template <int D>
__global__ void __launch_bounds__(kWarpsPerCta * 32) combine_lse_kernel(const Args a) {
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
    if (row >= static_cast<int64_t>(a.num_seqs) * a.num_q_heads) return;
    const int b = static_cast<int>(row / a.num_q_heads);
    const int hq = static_cast<int>(row % a.num_q_heads);
    const int q0 = a.query_start_loc[b];
    if (a.query_start_loc[b + 1] - q0 != 1) return;
    if (q0 < 0 || q0 >= a.num_tokens) return;  // flagged by the decode kernel
    const int L = min(a.seq_lens[b], a.max_pages * a.page_size);
    const int ns = (L + a.kv_chunk - 1) / a.kv_chunk;
    if (ns <= 1) return;  // the decode kernel wrote this row itself

    const int64_t slot0 = static_cast<int64_t>(b) * a.splits * a.num_q_heads + hq;  // split stride Hq
    const float* ml = a.ws_ml;
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, ml[(slot0 + static_cast<int64_t>(s) * a.num_q_heads) * 2]);
    M = warp_max(M);
    float den = 0.f;
    for (int s = lane; s < ns; s += 32) {
        const int64_t sl = slot0 + static_cast<int64_t>(s) * a.num_q_heads;
        den += fast_exp2(ml[sl * 2] - M) * ml[sl * 2 + 1];
    }
    den = warp_sum(den);

    constexpr int kPer = D / 32;  // 4 (D = 128) or 2 (D = 64) values per lane
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    for (int s = 0; s < ns; ++s) {
        const int64_t sl = slot0 + static_cast<int64_t>(s) * a.num_q_heads;
        const float w = fast_exp2(ml[sl * 2] - M);
        const float* os = a.ws_o + sl * D + lane * kPer;
        if constexpr (kPer == 4) {
            const float4 v = *reinterpret_cast<const float4*>(os);
            acc[0] += w * v.x;
            acc[1] += w * v.y;
            acc[2] += w * v.z;
            acc[3] += w * v.w;
        } else {
            const float2 v = *reinterpret_cast<const float2*>(os);
            acc[0] += w * v.x;
            acc[1] += w * v.y;
        }
    }
    const float inv = 1.f / den;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + (static_cast<int64_t>(q0) * a.num_q_heads + hq) * D +
                         lane * kPer;
#pragma unroll
    for (int i = 0; i < kPer; i += 2) {
        *reinterpret_cast<uint32_t*>(out + i) = pack_bf16(acc[i] * inv, acc[i + 1] * inv);
    }
}

}  // namespace

int64_t combine_ctas(const Args& a) {
    if (a.splits <= 1) return 0;
    const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
    return (rows + kWarpsPerCta - 1) / kWarpsPerCta;
}

cudaError_t launch_combine(const Args& a, cudaStream_t stream) {
    const int64_t ctas = combine_ctas(a);
    if (ctas == 0) return cudaSuccess;
    switch (a.head_dim) {
        case 64:
            combine_lse_kernel<64><<<static_cast<unsigned>(ctas), kWarpsPerCta * 32, 0, stream>>>(a);
            break;
        case 128:
            combine_lse_kernel<128><<<static_cast<unsigned>(ctas), kWarpsPerCta * 32, 0, stream>>>(a);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace pa
