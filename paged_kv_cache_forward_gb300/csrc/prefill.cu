// prefill.cu -- causal varlen chunked-prefill attention over the paged cache.
//
// One CTA owns (query tile, KV head h).  A tile packs TQ consecutive new tokens
// of one sequence times the G query heads that share h into 64 rows (the
// "Q-Block" item of the five-step list on the Triton unified-attention page,
// section "What three things the IBM paper got right"), row r = (token r / G,
// head h*G + r % G).  It walks the keys 0 .. (position of its last token) in
// tiles of 64 (4 pages), gathered through the block table by 16-byte cp.async
// into a double-buffered, XOR-swizzled shared-memory tile, and runs the
// FlashAttention-2 loop of "The Flash Attention revolution" / "Flash Attention
// in Triton" (GPU programming guide page): S = Q K^T, causal -inf mask
// (bottom-right aligned: token i of a sequence with L_b keys and n_b new tokens
// sits at p = L_b - n_b + i), online softmax in log2 units, O += P V, then
// O / l to bf16.  Each of the 4 warps owns 16 rows.
//
// The grid is static: ceil(T / TQ) + B tiles per KV head bound the tiles of any
// batch with these shapes.  Each CTA finds its (sequence, tile) by a prefix sum
// over the per-sequence tile counts; surplus CTAs and decode sequences (n_b = 1,
// handled by the decode kernel) exit at once.

#include <cuda_bf16.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsCta = 64;  // 16 rows per warp
constexpr int kKeys = 64;     // keys per KV tile
constexpr int kPage = 16;

template <int D>
struct PrefillTile {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kChunksPerRow = D / 8;
    static constexpr int kTileBytes = kKeys * kRowBytes;  // K or V
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kSmemBytes = 2 * kStageBytes + 64;
};

template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return r * PrefillTile<D>::kRowBytes + ((c ^ (r & 7)) << 4);
}

__device__ __forceinline__ int tiles_of(int n, int tq) { return n >= 2 ? (n + tq - 1) / tq : 0; }

template <int D>
__global__ void __launch_bounds__(kWarps * 32) prefill_mma_kernel(const Args a, int tq_tokens, int tiles_bound) {
    using Tile = PrefillTile<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    int* s_info = reinterpret_cast<int*>(smem + 2 * Tile::kStageBytes);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int tq = lane & 3;

    const int tile = blockIdx.x % tiles_bound;
    const int h = blockIdx.x / tiles_bound;

    // Find the sequence that owns global tile `tile` (warp 0 scans the batch).
    if (warp == 0) {
        int found_b = -1, found_t = 0, base = 0;
        for (int b0 = 0; b0 < a.num_seqs && found_b < 0; b0 += 32) {
            const int b = b0 + lane;
            const int cnt = b < a.num_seqs ? tiles_of(a.query_start_loc[b + 1] - a.query_start_loc[b], tq_tokens) : 0;
            int inc = cnt;  // inclusive scan over the warp
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += v;
            }
            const int excl = base + inc - cnt;
            const bool mine = cnt > 0 && tile >= excl && tile < excl + cnt;
            const unsigned m = __ballot_sync(0xffffffffu, mine);
            if (m) {
                const int src = __ffs(m) - 1;
                found_b = b0 + src;
                found_t = tile - __shfl_sync(0xffffffffu, excl, src);
            }
            base += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) {
            s_info[0] = found_b;
            s_info[1] = found_t;
        }
    }
    __syncthreads();
    const int b = s_info[0];
    if (b < 0) return;
    const int t_in_seq = s_info[1];

    const int q0 = a.query_start_loc[b];
    const int n = a.query_start_loc[b + 1] - q0;
    if (q0 < 0 || static_cast<int64_t>(q0) + n > a.num_tokens) {
        if (threadIdx.x == 0) flag_error(a.err, kDevBadQueryStart);
        return;
    }
    const int cap = a.max_pages * kPage;
    int L = a.seq_lens[b];
    if (L > cap) {
        flag_error(a.err, kDevSeqTooLong);
        L = cap;
    }
    const int G = a.group;
    const int i0 = t_in_seq * tq_tokens;               // first new token of the tile
    const int ntok = min(tq_tokens, n - i0);           // tokens in this tile
    const int prefix = L - n;                          // cached keys before the new ones
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    if (prefix < 0) {
        if (threadIdx.x == 0) flag_error(a.err, kDevQueryTooLong);
        for (int i = threadIdx.x; i < ntok * G * D; i += blockDim.x) {
            const int r = i / D;
            out[(static_cast<int64_t>(q0 + i0 + r / G) * a.num_q_heads + h * G + r % G) * D + i % D] =
                __float2bfloat16(0.f);
        }
        return;
    }
    const int kv_end = prefix + i0 + ntok;  // keys 0 .. kv_end-1 are visible to some row
    const int ntiles = (kv_end + kKeys - 1) / kKeys;

    // This thread's two rows (g and g + 8 of its warp): token and causal limit.
    const int r_lo = warp * 16 + g, r_hi = r_lo + 8;
    const bool v_lo = r_lo < ntok * G, v_hi = r_hi < ntok * G;
    const int p_lo = v_lo ? prefix + i0 + r_lo / G : -1;
    const int p_hi = v_hi ? prefix + i0 + r_hi / G : -1;
    const int p_min_warp = prefix + i0 + (warp * 16) / G;  // smallest limit among valid rows of the warp

    const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* q_lo = q + (static_cast<int64_t>(q0 + i0 + r_lo / G) * a.num_q_heads + h * G + r_lo % G) * D;
    const __nv_bfloat16* q_hi = q + (static_cast<int64_t>(q0 + i0 + r_hi / G) * a.num_q_heads + h * G + r_hi % G) * D;
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const int c = ks * 16 + 2 * tq;
        qa[ks][0] = v_lo ? *reinterpret_cast<const uint32_t*>(q_lo + c) : 0u;
        qa[ks][1] = v_hi ? *reinterpret_cast<const uint32_t*>(q_hi + c) : 0u;
        qa[ks][2] = v_lo ? *reinterpret_cast<const uint32_t*>(q_lo + c + 8) : 0u;
        qa[ks][3] = v_hi ? *reinterpret_cast<const uint32_t*>(q_hi + c + 8) : 0u;
    }

    const __nv_bfloat16* kc = reinterpret_cast<const __nv_bfloat16*>(a.k_cache);
    const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(a.v_cache);
    const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_pages;
    const uint32_t sbase = smem_u32(smem);

    auto issue = [&](int kt) {
        if (kt < ntiles) {
            const uint32_t st = sbase + (kt & 1) * Tile::kStageBytes;
            constexpr int kChunks = kKeys * Tile::kChunksPerRow;  // per K (or V) tile
#pragma unroll
            for (int i = 0; i < kChunks / (kWarps * 32); ++i) {
                const int c = threadIdx.x + kWarps * 32 * i;
                const int r = c / Tile::kChunksPerRow;  // key within the tile
                const int cc = c % Tile::kChunksPerRow;
                const int j = kt * kKeys + r;
                int page = 0;
                bool ok = j < L;
                if (ok) {
                    page = bt[j / kPage];
                    if (static_cast<uint32_t>(page) >= static_cast<uint64_t>(a.num_blocks)) {
                        flag_error(a.err, kDevBadBlock);
                        ok = false;
                        page = 0;
                    }
                }
                const int64_t off = ((static_cast<int64_t>(page) * kPage + (ok ? j % kPage : 0)) * a.num_kv_heads + h) * D +
                                    cc * 8;
                cp_async_16(st + swz<D>(r, cc), kc + off, ok ? 16 : 0);
                cp_async_16(st + Tile::kTileBytes + swz<D>(r, cc), vc + off, ok ? 16 : 0);
            }
        }
        cp_async_commit();
    };

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

    issue(0);
    for (int kt = 0; kt < ntiles; ++kt) {
        issue(kt + 1);
        cp_async_wait<1>();
        __syncthreads();
        const uint32_t sk = sbase + (kt & 1) * Tile::kStageBytes;
        const uint32_t sv = sk + Tile::kTileBytes;
        const int j0 = kt * kKeys;

        // Warp-uniform: skip the tile only if no row of this warp sees any of its keys.
        const bool warp_active = __any_sync(0xffffffffu, j0 <= max(p_lo, p_hi));
        if (warp_active) {
            float sc[kKeys / 8][4];
#pragma unroll
            for (int i = 0; i < kKeys / 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
            {
                const int mi = lane >> 3;
#pragma unroll
                for (int np = 0; np < kKeys / 16; ++np) {
                    const int key = np * 16 + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        uint32_t k0, k1, k2, k3;
                        ldmatrix_x4(sk + swz<D>(key, 2 * ks + (mi & 1)), k0, k1, k2, k3);
                        mma_bf16_16816(sc[2 * np], qa[ks], k0, k1);
                        mma_bf16_16816(sc[2 * np + 1], qa[ks], k2, k3);
                    }
                }
            }
            const bool need_mask = j0 + kKeys - 1 > p_min_warp;
#pragma unroll
            for (int nt = 0; nt < kKeys / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = j0 + nt * 8 + 2 * tq + (e & 1);
                    const int lim = e < 2 ? p_lo : p_hi;
                    const float x = sc[nt][e] * a.scale_log2;
                    sc[nt][e] = (!need_mask || j <= lim) ? x : -INFINITY;
                }
            float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < kKeys / 8; ++nt) {
                mx_lo = fmaxf(mx_lo, fmaxf(sc[nt][0], sc[nt][1]));
                mx_hi = fmaxf(mx_hi, fmaxf(sc[nt][2], sc[nt][3]));
            }
            mx_lo = quad_max(mx_lo);
            mx_hi = quad_max(mx_hi);
            const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
            const float mu_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
            const float mu_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
            const float al_lo = fast_exp2(m_lo - mu_lo), al_hi = fast_exp2(m_hi - mu_hi);
            m_lo = mn_lo;
            m_hi = mn_hi;
            l_lo *= al_lo;
            l_hi *= al_hi;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                o[i][0] *= al_lo;
                o[i][1] *= al_lo;
                o[i][2] *= al_hi;
                o[i][3] *= al_hi;
            }
            const int mi = lane >> 3;
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk) {
                uint32_t pa[4];
                pa[0] = pack_bf16(fast_exp2(sc[2 * kk][0] - mu_lo), fast_exp2(sc[2 * kk][1] - mu_lo));
                pa[1] = pack_bf16(fast_exp2(sc[2 * kk][2] - mu_hi), fast_exp2(sc[2 * kk][3] - mu_hi));
                pa[2] = pack_bf16(fast_exp2(sc[2 * kk + 1][0] - mu_lo), fast_exp2(sc[2 * kk + 1][1] - mu_lo));
                pa[3] = pack_bf16(fast_exp2(sc[2 * kk + 1][2] - mu_hi), fast_exp2(sc[2 * kk + 1][3] - mu_hi));
                l_lo += (bf16_lo(pa[0]) + bf16_hi(pa[0])) + (bf16_lo(pa[2]) + bf16_hi(pa[2]));
                l_hi += (bf16_lo(pa[1]) + bf16_hi(pa[1])) + (bf16_lo(pa[3]) + bf16_hi(pa[3]));
                const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
                for (int nd = 0; nd < D / 16; ++nd) {
                    uint32_t v0, v1, v2, v3;
                    ldmatrix_x4_trans(sv + swz<D>(key, 2 * nd + (mi >> 1)), v0, v1, v2, v3);
                    mma_bf16_16816(o[2 * nd], pa, v0, v1);
                    mma_bf16_16816(o[2 * nd + 1], pa, v2, v3);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    l_lo = quad_sum(l_lo);
    l_hi = quad_sum(l_hi);
    const float inv_lo = v_lo ? 1.f / l_lo : 0.f, inv_hi = v_hi ? 1.f / l_hi : 0.f;
    __nv_bfloat16* o_lo = out + (static_cast<int64_t>(q0 + i0 + r_lo / G) * a.num_q_heads + h * G + r_lo % G) * D;
    __nv_bfloat16* o_hi = out + (static_cast<int64_t>(q0 + i0 + r_hi / G) * a.num_q_heads + h * G + r_hi % G) * D;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        const int c = i * 8 + 2 * tq;
        if (v_lo) *reinterpret_cast<uint32_t*>(o_lo + c) = pack_bf16(o[i][0] * inv_lo, o[i][1] * inv_lo);
        if (v_hi) *reinterpret_cast<uint32_t*>(o_hi + c) = pack_bf16(o[i][2] * inv_hi, o[i][3] * inv_hi);
    }
}

int tokens_per_tile(int group) { return group <= kRowsCta ? kRowsCta / group : 0; }

int tiles_bound(const Args& a) {
    const int tq = tokens_per_tile(a.group);
    if (tq == 0) return 0;
    return static_cast<int>((a.num_tokens + tq - 1) / tq + a.num_seqs);
}

template <int D>
cudaError_t launch_prefill_d(const Args& a, cudaStream_t stream) {
    using Tile = PrefillTile<D>;
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configured[dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Tile::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured[dev & 63] = true;
    }
    const int64_t ctas = prefill_ctas(a);
    if (ctas == 0) return cudaSuccess;
    prefill_mma_kernel<D><<<static_cast<unsigned>(ctas), kWarps * 32, Tile::kSmemBytes, stream>>>(
        a, tokens_per_tile(a.group), tiles_bound(a));
    return cudaGetLastError();
}

}  // namespace

int64_t prefill_ctas(const Args& a) {
    if (a.num_tokens < 2) return 0;
    return static_cast<int64_t>(tiles_bound(a)) * a.num_kv_heads;
}

cudaError_t launch_prefill(const Args& a, cudaStream_t stream) {
    switch (a.head_dim) {
        case 64: return launch_prefill_d<64>(a, stream);
        case 128: return launch_prefill_d<128>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
