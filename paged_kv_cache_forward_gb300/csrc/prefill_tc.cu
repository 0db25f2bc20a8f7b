// prefill_tc.cu -- causal varlen chunked prefill on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), sm_103a.
//
// One CTA owns (query tile, KV head h).  The tile packs TQ = floor(128 / G)
// consecutive new tokens of one sequence times the G query heads sharing h into
// the M = 128 rows of one MMA tile, row r = (token r / G, head h*G + r % G): the
// "Q-Block" item of the five-step list on the Triton unified-attention page
// (section "What three things the IBM paper got right"), so each KV tile is
// loaded once for all G heads.  Keys are walked in tiles of 128 (8 pages) up to
// the tile's last causal position, with the FlashAttention recurrence of "The
// Flash Attention revolution" (GPU programming guide page): S = Q K^T, causal
// -inf mask bottom-right aligned ("Flash Attention in Triton"), online softmax,
// O += P V, out = O / l.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q once, then per KV tile the K page boxes and the
//               V page boxes (64 columns x 16 slots of one page and head, 128-byte
//               swizzle) into separate 3-stage K and V rings, so a K stage is
//               refilled as soon as its S MMA is done.  Block-table entries are
//               fetched one group of 4 tiles ahead.  The one page of V that holds
//               the sequence end is copied by plain loads with zero fill, so no
//               slot past seq_len reaches the MMA.
//   warp 1      allocates all 512 TMEM columns (S double buffer, O, P double
//               buffer); its lane 0 issues the MMAs: S(kt) = Q K(kt)^T (M=128,
//               N=128, K=D, both operands from shared memory) into TMEM, then
//               O += P(kt-1) V(kt-1) (A = P read from TMEM, B = V MN-major in shared
//               memory), so that the softmax of tile kt overlaps the MMAs.
//   warps 2-5   softmax, one thread per row (TMEM lane): load S from TMEM,
//               mask, running max in log2 units, P = 2^(x - m) as bf16 pairs
//               stored straight into TMEM.  The running max is only moved (and O
//               in TMEM rescaled) when the row max grows by more than 2^8; the
//               final O / l is exact either way.
// Every wait on an mbarrier is bounded (2 s); on timeout the CTA records
// kDevWaitTimeout, stops all roles, drains the MMAs it issued, frees TMEM and
// exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "tc_device.cuh"
#include "tmap.h"

namespace pa {
namespace {

constexpr int kThreads = 192;
constexpr int kM = 128;            // rows per tile
constexpr int kKeys = 128;         // keys per KV tile
constexpr int kPage = 16;
constexpr int kPagesPerTile = kKeys / kPage;
constexpr int kHalfBytes = 128 * 128;  // 128 rows x 128 B: one 64-column half of a tile
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256, kTmemP0 = 384, kTmemP1 = 448;
constexpr int kKStages = 3, kVStages = 3;
constexpr int kTilesPerGroup = 4;  // block-table prefetch: 4 tiles x 8 pages = one entry per lane

template <int D>
struct Smem {
    static constexpr int kHalves = D / 64;
    static constexpr int kTile = kHalves * kHalfBytes;  // one K or V tile (128 keys x D)
    static constexpr int kQ = 0;
    static constexpr int kK0 = kQ + kTile;
    static constexpr int kV0 = kK0 + kKStages * kTile;
    static constexpr int kBar = kV0 + kVStages * kTile;
    static constexpr int kNumBars = 22;
    static constexpr int kMisc = kBar + kNumBars * 8;  // tmem address, abort flag, tile info
    static constexpr int kBytes = kMisc + 64;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024
};

// barrier indices
enum Bar {
    kQFull = 0,
    kKFull0 = 1,     // [3]
    kKEmpty0 = 4,    // [3]
    kVFull0 = 7,     // [3]
    kVEmpty0 = 10,   // [3]
    kSFull0 = 13,    // [2]
    kSFree0 = 15,    // [2]
    kPFull0 = 17,    // [2]
    kPvDone0 = 19,   // [2]
    kDrain = 21,
};

// Tiles of a sequence with n new tokens (the decode path takes n <= qmax).
__device__ __forceinline__ int tiles_of(int n, int tq, int qmax) { return n > qmax ? (n + tq - 1) / tq : 0; }

// Bounded wait by every lane of a warp; the result is made warp-uniform so that a
// timeout can never leave some lanes at a warp-collective instruction alone.
__device__ __forceinline__ bool warp_wait(uint32_t addr, uint32_t parity, const volatile int* abort) {
    const bool ok = tc::mbar_wait(addr, parity, abort, kTimeoutNs);
    return __all_sync(0xffffffffu, ok);
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled half.
__device__ __forceinline__ uint32_t sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const Args a, int tq_tokens, int tiles_bound) {
    using S = Smem<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const sp = smem_raw + (base - raw);
    auto bar = [&](int i) { return base + S::kBar + 8 * i; };
    uint32_t* const s_tmem = reinterpret_cast<uint32_t*>(sp + S::kMisc);
    volatile int* const s_abort = reinterpret_cast<volatile int*>(sp + S::kMisc + 4);
    int* const s_info = reinterpret_cast<int*>(sp + S::kMisc + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tile = blockIdx.x % tiles_bound;
    const int h = blockIdx.x / tiles_bound;

    // ---- which sequence owns this tile (prefix sum of per-sequence tile counts)
    if (warp == 0) {
        int found_b = -1, found_t = 0, base_t = 0;
        for (int b0 = 0; b0 < a.num_seqs && found_b < 0; b0 += 32) {
            const int b = b0 + lane;
            const int cnt = b < a.num_seqs ? tiles_of(a.query_start_loc[b + 1] - a.query_start_loc[b], tq_tokens, a.decode_max_q) : 0;
            int inc = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += v;
            }
            const int excl = base_t + inc - cnt;
            const unsigned m = __ballot_sync(0xffffffffu, cnt > 0 && tile >= excl && tile < excl + cnt);
            if (m) {
                const int src = __ffs(m) - 1;
                found_b = b0 + src;
                found_t = tile - __shfl_sync(0xffffffffu, excl, src);
            }
            base_t += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) {
            s_info[0] = found_b;
            s_info[1] = found_t;
            *s_abort = 0;
        }
    }
    __syncthreads();
    const int b = s_info[0];
    if (b < 0) return;  // surplus CTA of the static grid (uniform for the block)
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
        if (threadIdx.x == 0) flag_error(a.err, kDevSeqTooLong);
        L = cap;
    }
    const int G = a.group;
    const int i0 = t_in_seq * tq_tokens;
    const int ntok = min(tq_tokens, n - i0);
    const int prefix = L - n;
    __nv_bfloat16* const out = reinterpret_cast<__nv_bfloat16*>(a.out);
    if (prefix < 0) {
        if (threadIdx.x == 0) flag_error(a.err, kDevQueryTooLong);
        for (int i = threadIdx.x; i < ntok * G * D; i += blockDim.x) {
            const int r = i / D;
            out[(static_cast<int64_t>(q0 + i0 + r / G) * a.num_q_heads + h * G + r % G) * D + i % D] =
                __float2bfloat16(0.f);
        }
        return;
    }
    const int kv_end = prefix + i0 + ntok;  // keys [0, kv_end) are visible to some row
    const int ntiles = (kv_end + kKeys - 1) / kKeys;
    const int last_page = (kv_end + kPage - 1) / kPage;  // pages [0, last_page) are read
    const int full_pages = L / kPage;                    // pages with no slot past L

    // ---- barriers and TMEM
    if (threadIdx.x == 0) {
        tc::mbar_init(bar(kQFull), 1);
        for (int i = 0; i < kKStages; ++i) {
            tc::mbar_init(bar(kKFull0 + i), 1);
            tc::mbar_init(bar(kKEmpty0 + i), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            tc::mbar_init(bar(kVFull0 + i), 1);
            tc::mbar_init(bar(kVEmpty0 + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(kSFull0 + i), 1);
            tc::mbar_init(bar(kSFree0 + i), 4);
            tc::mbar_init(bar(kPFull0 + i), 4);
            tc::mbar_init(bar(kPvDone0 + i), 1);
        }
        tc::mbar_init(bar(kDrain), 1);
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(base + S::kMisc, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *s_tmem;
    bool ok = true;

    if (warp == 0) {
        // ================================================= TMA producer
        if (lane == 0) {
            tc::prefetch_tmap(&tm_q);
            tc::prefetch_tmap(&tm_k);
            tc::prefetch_tmap(&tm_v);
            tc::mbar_arrive_expect_tx(bar(kQFull), S::kHalves * 64 * 2 * G * tq_tokens);
#pragma unroll
            for (int hf = 0; hf < S::kHalves; ++hf)
                tc::tma_load_3d(base + S::kQ + hf * kHalfBytes, &tm_q, bar(kQFull), hf * 64, h * G, q0 + i0);
        }
        const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_pages;
        // lane l holds the block-table entry of page (group * 32 + l); the next
        // group's entries are loaded while the current group is being used.
        auto load_group = [&](int grp) -> int {
            const int pg = grp * kTilesPerGroup * kPagesPerTile + lane;
            return pg < last_page ? bt[pg] : 0;
        };
        int cur_grp = load_group(0);
        int next_grp = load_group(1);
        const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(a.v_cache);
        for (int kt = 0; kt < ntiles; ++kt) {
            const int slot = kt % kTilesPerGroup;
            if (slot == 0 && kt > 0) {
                cur_grp = next_grp;
                next_grp = load_group(kt / kTilesPerGroup + 1);
            }
            const int p0 = kt * kPagesPerTile;
            const int np = min(kPagesPerTile, last_page - p0);
            const int nv = max(0, min(np, full_pages - p0));  // V pages by TMA
            int page = __shfl_sync(0xffffffffu, cur_grp, (slot * kPagesPerTile + lane) & 31);
            if (lane < np && static_cast<uint32_t>(page) >= static_cast<uint64_t>(a.num_blocks)) {
                flag_error(a.err, kDevBadBlock);
                page = 0;
            }
            // ---- K(kt)
            const int kst = kt % kKStages;
            if (kt >= kKStages && !warp_wait(bar(kKEmpty0 + kst), (kt / kKStages - 1) & 1, s_abort)) {
                ok = false;
                break;
            }
            const uint32_t sk = base + S::kK0 + kst * S::kTile;
            if (lane == 0) tc::mbar_arrive_expect_tx(bar(kKFull0 + kst), np * S::kHalves * 2048);
            __syncwarp();
            if (lane < np) {
#pragma unroll
                for (int hf = 0; hf < S::kHalves; ++hf)
                    tc::tma_load_4d(sk + hf * kHalfBytes + lane * 2048, &tm_k, bar(kKFull0 + kst), hf * 64, h, 0,
                                    page);
            }
            // ---- V(kt)
            const int vst = kt % kVStages;
            if (kt >= kVStages && !warp_wait(bar(kVEmpty0 + vst), (kt / kVStages - 1) & 1, s_abort)) {
                ok = false;
                break;
            }
            const uint32_t sv = base + S::kV0 + vst * S::kTile;
            if (nv < np) {
                // The page holding the sequence end: plain loads, slots >= L as zeros.
                const int pi = np - 1;
                const int pg = __shfl_sync(0xffffffffu, page, pi);
                for (int c = lane; c < kPage * (D / 8); c += 32) {
                    const int t = c / (D / 8), ch = c % (D / 8);
                    const int row = pi * kPage + t;
                    uint4 val = make_uint4(0u, 0u, 0u, 0u);
                    if ((p0 + pi) * kPage + t < L)
                        val = *reinterpret_cast<const uint4*>(
                            vc + ((static_cast<int64_t>(pg) * kPage + t) * a.num_kv_heads + h) * D + ch * 8);
                    const uint32_t dst = sv + (ch >> 3) * kHalfBytes + sw128(row, ch & 7);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(val.x), "r"(val.y),
                                 "r"(val.z), "r"(val.w)
                                 : "memory");
                }
                tc::fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_expect_tx(bar(kVFull0 + vst), nv * S::kHalves * 2048);
            __syncwarp();
            if (lane < nv) {
#pragma unroll
                for (int hf = 0; hf < S::kHalves; ++hf)
                    tc::tma_load_4d(sv + hf * kHalfBytes + lane * 2048, &tm_v, bar(kVFull0 + vst), hf * 64, h, 0,
                                    page);
            }
        }
        if (!ok && lane == 0) {
            *s_abort = 1;
            flag_error(a.err, kDevWaitTimeout);
        }
    } else if (warp == 1) {
        // ===================================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdQK = tc::idesc_bf16_f32(kM, kKeys, false, false);
            constexpr uint32_t kIdPV = tc::idesc_bf16_f32(kM, D, false, true);
            auto issue_pv = [&](int j) -> bool {
                if (!tc::mbar_wait(bar(kPFull0 + (j & 1)), (j >> 1) & 1, s_abort, kTimeoutNs)) return false;
                const int vst = j % kVStages;
                if (!tc::mbar_wait(bar(kVFull0 + vst), (j / kVStages) & 1, s_abort, kTimeoutNs)) return false;
                tc::tc_fence_after();
                const int npj = min(kPagesPerTile, last_page - j * kPagesPerTile);
                const uint32_t sv = base + S::kV0 + vst * S::kTile;
                const uint32_t pa = tmem + ((j & 1) ? kTmemP1 : kTmemP0);
                for (int ks = 0; ks < npj; ++ks) {  // one 16-key step per page; P: 8 columns per step
                    const uint64_t bd = tc::desc_sw128(sv + ks * 2048, kHalfBytes, 1024);
                    tc::mma_bf16_tmem_a(tmem + kTmemO, pa + ks * 8, bd, kIdPV, (j > 0 || ks > 0) ? 1u : 0u);
                }
                tc::mma_commit(bar(kPvDone0 + (j & 1)));
                tc::mma_commit(bar(kVEmpty0 + vst));
                return true;
            };
            ok = tc::mbar_wait(bar(kQFull), 0, s_abort, kTimeoutNs);
            tc::tc_fence_after();
            for (int kt = 0; kt < ntiles && ok; ++kt) {
                const int sb = kt & 1;
                const int kst = kt % kKStages;
                ok = tc::mbar_wait(bar(kKFull0 + kst), (kt / kKStages) & 1, s_abort, kTimeoutNs);
                if (ok && kt >= 2) ok = tc::mbar_wait(bar(kSFree0 + sb), ((kt >> 1) - 1) & 1, s_abort, kTimeoutNs);
                if (!ok) break;
                tc::tc_fence_after();
                const uint32_t sk = base + S::kK0 + kst * S::kTile;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
                    const uint64_t ad = tc::desc_sw128(base + S::kQ + off, 16, 1024);
                    const uint64_t bd = tc::desc_sw128(sk + off, 16, 1024);
                    tc::mma_bf16(tmem + (sb ? kTmemS1 : kTmemS0), ad, bd, kIdQK, ks > 0 ? 1u : 0u);
                }
                tc::mma_commit(bar(kSFull0 + sb));
                tc::mma_commit(bar(kKEmpty0 + kst));
                if (kt >= 1) ok = issue_pv(kt - 1);
            }
            if (ok) ok = issue_pv(ntiles - 1);
            if (!ok) {
                *s_abort = 1;
                flag_error(a.err, kDevWaitTimeout);
            }
            // drain: every MMA issued above has finished before TMEM is freed
            tc::mma_commit(bar(kDrain));
            tc::mbar_wait(bar(kDrain), 0, nullptr, kTimeoutNs);
        }
        __syncwarp();
    } else {
        // ======================================================== softmax
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // row == TMEM lane
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const bool valid = r < ntok * G;
        const int pos = valid ? prefix + i0 + r / G : -1;  // causal limit of this row
        const float c = a.scale_log2;
        float m_used = -INFINITY;  // running max, log2 units
        float lsum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // split to keep the adds independent
        for (int kt = 0; kt < ntiles; ++kt) {
            const int sb = kt & 1;
            if (!warp_wait(bar(kSFull0 + sb), (kt >> 1) & 1, s_abort)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            uint32_t sr[kKeys];
#pragma unroll
            for (int q = 0; q < kKeys / 32; ++q)
                tc::tmem_ld32(lane_addr + (sb ? kTmemS1 : kTmemS0) + q * 32,
                              *reinterpret_cast<uint32_t(*)[32]>(&sr[q * 32]));
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(kSFree0 + sb));

            const int j0 = kt * kKeys;
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
            const bool diag = __any_sync(0xffffffffu, j0 + kKeys - 1 > pos);
            if (diag) {
#pragma unroll
                for (int j = 0; j < kKeys; ++j) {
                    const float s = __uint_as_float(sr[j]);
                    const float v = (j0 + j <= pos) ? s : -INFINITY;
                    sr[j] = __float_as_uint(v);
                    mx8[j & 7] = fmaxf(mx8[j & 7], v);
                }
            } else {
#pragma unroll
                for (int j = 0; j < kKeys; ++j) mx8[j & 7] = fmaxf(mx8[j & 7], __uint_as_float(sr[j]));
            }
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            const float mnew = mx * c;  // scale > 0, so the max commutes with it
            if (kt == 0) {
                m_used = mnew;
            } else {
                const bool need = mnew > m_used + 8.f;
                if (__any_sync(0xffffffffu, need)) {
                    // O is final for tiles < kt once P V(kt-1) is done
                    if (!warp_wait(bar(kPvDone0 + ((kt - 1) & 1)), ((kt - 1) >> 1) & 1, s_abort)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const float alpha = need ? fast_exp2(m_used - mnew) : 1.f;
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        uint32_t o[32];
                        tc::tmem_ld32(lane_addr + kTmemO + q * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::tmem_st32(lane_addr + kTmemO + q * 32, o);
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) lsum[e] *= alpha;
                    if (need) m_used = mnew;
                }
            }
            const float mu = m_used == -INFINITY ? 0.f : m_used;
            // P buffer sb is free once P V(kt-2) is done
            if (kt >= 2 && !warp_wait(bar(kPvDone0 + sb), ((kt >> 1) - 1) & 1, s_abort)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            // P = 2^(s*c - m) as bf16 pairs; l sums the rounded values the MMA will use.
            const uint32_t pcol = lane_addr + (sb ? kTmemP1 : kTmemP0);
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int j = hlf * 64 + 2 * e;
                    const float x0 = fast_exp2(fmaf(__uint_as_float(sr[j]), c, -mu));
                    const float x1 = fast_exp2(fmaf(__uint_as_float(sr[j + 1]), c, -mu));
                    pk[e] = pack_bf16(x0, x1);
                    lsum[e & 7] += bf16_lo(pk[e]) + bf16_hi(pk[e]);
                }
                tc::tmem_st32(pcol + hlf * 32, pk);
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(kPFull0 + sb));
        }
        if (ok) ok = warp_wait(bar(kPvDone0 + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, s_abort);
        if (ok) {
            tc::tc_fence_after();
            const float l = ((lsum[0] + lsum[1]) + (lsum[2] + lsum[3])) + ((lsum[4] + lsum[5]) + (lsum[6] + lsum[7]));
            const float inv = valid ? 1.f / l : 0.f;
            __nv_bfloat16* orow =
                out + (static_cast<int64_t>(q0 + i0 + (valid ? r / G : 0)) * a.num_q_heads + h * G + r % G) * D;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tc::tmem_ld32(lane_addr + kTmemO + q * 32, o);
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 v;
                        v.x = pack_bf16(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                        v.y = pack_bf16(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                        v.z = pack_bf16(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                        v.w = pack_bf16(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + q * 32 + e) = v;
                    }
                }
            }
        } else if (lane == 0) {
            *s_abort = 1;
            flag_error(a.err, kDevWaitTimeout);
        }
    }

    // ---- teardown: every role is out of its loop; the MMA thread has drained.
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// --------------------------------------------------------------- host side
int tokens_per_tile(int group) { return group <= kM ? kM / group : 0; }

int tiles_bound(const Args& a) {
    const int tq = tokens_per_tile(a.group);
    if (tq == 0) return 0;
    return static_cast<int>((a.num_tokens + tq - 1) / tq + a.num_seqs);
}

template <int D>
cudaError_t launch_d(const Args& a, cudaStream_t stream) {
    using S = Smem<D>;
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configured[dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             S::kAlloc);
        if (e != cudaSuccess) return e;
        configured[dev & 63] = true;
    }
    const int64_t ctas = prefill_ctas(a);
    if (ctas == 0) return cudaSuccess;
    const int G = a.group, tq = tokens_per_tile(G);
    CUtensorMap tq_map, tk_map, tv_map;
    if (!encode_q_map(&tq_map, a.q, D, a.num_q_heads, a.num_tokens, G, tq) ||
        !encode_cache_map(&tk_map, a.k_cache, D, a.num_kv_heads, a.num_blocks) ||
        !encode_cache_map(&tv_map, a.v_cache, D, a.num_kv_heads, a.num_blocks))
        return cudaErrorInvalidValue;
    prefill_tc_kernel<D><<<static_cast<unsigned>(ctas), kThreads, S::kAlloc, stream>>>(tq_map, tk_map, tv_map, a, tq,
                                                                                       tiles_bound(a));
    return cudaGetLastError();
}

}  // namespace

int64_t prefill_ctas(const Args& a) {
    if (a.num_tokens < 2) return 0;
    return static_cast<int64_t>(tiles_bound(a)) * a.num_kv_heads;
}

cudaError_t launch_prefill(const Args& a, cudaStream_t stream) {
    switch (a.head_dim) {
        case 64: return launch_d<64>(a, stream);
        case 128: return launch_d<128>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
