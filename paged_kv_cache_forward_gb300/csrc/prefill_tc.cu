// prefill_tc.cu -- causal varlen chunked prefill on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), sm_103a.
//
// A work item is (a pair of query tiles, KV head h); one persistent CTA per SM
// takes items one after another (see prefill_tc_kernel).  A tile packs TQ =
// floor(128 / G) consecutive new tokens of one sequence times the G query heads
// sharing h into the M = 128 rows of one MMA tile, row r = (token r / G, head
// h*G + r % G): the "Q-Block" item of the five-step list on the Triton
// unified-attention page (section "What three things the IBM paper got right"),
// so each KV tile is loaded once for all G heads.  The two tiles of the pair (A:
// tokens [i0, i0 + TQ), B: the next TQ tokens) share every K and V tile in
// shared memory.  Keys are walked in tiles of 128 (8 pages) up to each tile's
// last causal position, with the FlashAttention recurrence of "The Flash
// Attention revolution" (GPU programming guide page): S = Q K^T, causal -inf
// mask bottom-right aligned ("Flash Attention in Triton"), online softmax,
// O += P V, out = O / l.
//
// Warp roles (640 threads at D <= 128, 384 at D = 256), each looping over the
// CTA's items:
//   warps 0, 2  TMA producers: warp 0 resolves the items and per item loads
//               both Q tiles and the K page boxes (64 columns x 16 slots of one
//               page and head, 128-byte swizzle) into the K ring; warp 2 the V
//               page boxes into the V ring, each running ahead on its own.
//               Block-table entries are fetched one group of 4 tiles ahead.
//               The one page of V that holds the sequence end is copied by
//               plain loads with zero fill, so no slot past seq_len reaches the
//               MMA.
//   warp 1      allocates all 512 TMEM columns (S and O of each tile); its lane 0
//               issues the MMAs in the order
//                   O_A += P_A(j) V(j),  S_A(j+1) = Q_A K(j+1)^T,
//                   O_B += P_B(j) V(j),  S_B(j+1) = Q_B K(j+1)^T,
//               so that while the softmax of one tile runs, the tensor cores work
//               on the other (ping-pong).  P is written as bf16 pairs over the
//               last 64 columns of its tile's S; the MMA that next overwrites S
//               is issued after the P V that reads it, and tcgen05 operations of
//               one thread execute in issue order.
//   (warp 3 idle)
//   softmax     one thread per row (TMEM lane).  At D <= 128 each tile's rows are
//               shared by two warps per lane quarter, 64 key columns each (warps
//               4-7 / 8-11: columns 0-63 of tile A / B, warps 12-15 / 16-19:
//               columns 64-127), which exchange their row maxima through shared
//               memory; at D = 256 warps 4-7 hold whole 128-column rows of the
//               single tile.  S is loaded from TMEM at once, masked, its max taken
//               in log2 units, and P = 2^(x - m) stored straight into TMEM as
//               bf16 with one wait; the normaliser l sums those same bf16
//               values.  The running max is only moved (and O in TMEM rescaled)
//               when the row max grows by more than 2^8; the final O / l is
//               exact either way.
// Every wait on an mbarrier is bounded (2 s); on timeout the CTA records
// kDevWaitTimeout, stops all roles, drains the MMAs it issued, frees TMEM and
// exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "tc_device.cuh"
#include "tmap.h"

namespace pa {
namespace {

constexpr int kWarpV = 2;  // the V producer
constexpr int kM = 128;            // rows per tile
constexpr int kKeys = 128;         // keys per KV tile
constexpr int kPage = 16;
constexpr int kPagesPerTile = kKeys / kPage;
constexpr int kHalfBytes = 128 * 128;  // 128 rows x 128 B: one 64-column half of a tile
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint32_t kTmemCols = 512;
// TMEM columns of tile x: S at 128 x (P over its last 64 columns), O at 256 + 128 x.
__device__ __forceinline__ uint32_t tmem_s(int x) { return x ? 128u : 0u; }
__device__ __forceinline__ uint32_t tmem_o(int x) { return x ? 384u : 256u; }
// Query tiles per CTA, ring depths, softmax warps and registers.
//  * D <= 128: a pair of query tiles per CTA (S and O of both in the 512 TMEM
//    columns), 2-stage K and V rings, and two softmax warps per TMEM lane
//    quarter of each tile, each taking 64 of the tile's 128 key columns (the
//    row max is exchanged through shared memory).  640 threads launch with 96
//    registers each; each softmax warp holds 64 S values within those, and
//    warpgroup 0 (producers, MMA issuer) drops to 88.
//  * D = 256: one tile's O alone takes 256 columns, so a CTA holds one tile, with
//    single-stage 64 KiB K and V rings (K(j+1) loads during the softmax and P V
//    of tile j, V(j+1) during S(j+1) and its softmax) and one softmax warp per
//    lane quarter holding the whole 128-column S row: 384 threads at 168
//    registers, 128 x 104 + 256 x 200 = 384 x 168 (warps 8-11 idle).
// The launcher checks the launch register count, so a split that does not fit
// is an error, not a wait in setmaxnreg.
template <int D>
struct Cfg {
    static constexpr int kTiles = D <= 128 ? 2 : 1;
    static constexpr int kKStages = D <= 128 ? 2 : 1;
    static constexpr int kVStages = D <= 128 ? 2 : 1;
    static constexpr int kColSplit = D <= 128 ? 2 : 1;  // softmax warps per lane quarter of a tile
    static constexpr int kThreads = D <= 128 ? 640 : 384;
    static constexpr uint32_t kRegsLaunch = D <= 128 ? 96 : 168;
    static constexpr uint32_t kRegsIssue = D <= 128 ? 88 : 104;
    static constexpr uint32_t kRegsSoftmax = D <= 128 ? 96 : 200;
    static_assert(128 * kRegsIssue + (kThreads - 128) * kRegsSoftmax <= kThreads * kRegsLaunch,
                  "register split above the launch");
};
constexpr int kMaxKStages = 3, kMaxVStages = 2;  // barrier slots
constexpr int kTilesPerGroup = 4;  // block-table prefetch: 4 tiles x 8 pages = one entry per lane
#ifndef PA_PREFILL_L2_PREFETCH
#define PA_PREFILL_L2_PREFETCH 2
#endif
constexpr int kPrefetchTiles = PA_PREFILL_L2_PREFETCH;  // K/V tiles ahead brought into L2 (0: none)
static_assert(kPrefetchTiles < kTilesPerGroup, "prefetched tiles must be in the current or next group");

template <int D>
struct Smem {
    static constexpr int kHalves = D / 64;
    static constexpr int kTile = kHalves * kHalfBytes;  // one Q, K or V tile (128 rows x D)
    static constexpr int kQ0 = 0;                       // Q_A, then Q_B
    static constexpr int kK0 = kQ0 + Cfg<D>::kTiles * kTile;
    static constexpr int kV0 = kK0 + Cfg<D>::kKStages * kTile;
    static constexpr int kBar = kV0 + Cfg<D>::kVStages * kTile;
    static constexpr int kNumBars = 23;
    static constexpr int kMisc = kBar + kNumBars * 8;  // tmem address, abort flag
    static constexpr int kItems = kMisc + 32;          // 2-slot item ring, 32 bytes a slot
    // row-max exchange of the two softmax warps of a lane quarter: [2 buffers]
    // [2 tiles][2 halves][128 rows] fp32, then the final l: [2 tiles][2 halves][128]
    static constexpr int kXMax = kItems + 64;
    static constexpr int kXL = kXMax + (Cfg<D>::kColSplit > 1 ? 2 * 2 * 2 * 128 * 4 : 0);
    static constexpr int kBytes = kXL + (Cfg<D>::kColSplit > 1 ? 2 * 2 * 128 * 4 : 0);
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024
    static_assert(kAlloc <= 227 * 1024, "shared memory above the per-CTA limit");
};

// barrier indices
enum Bar {
    kQFull = 0,
    kKFull0 = 1,    // [kMaxKStages = 3]
    kKEmpty0 = 4,   // [3]
    kVFull0 = 7,    // [kMaxVStages = 2]
    kVEmpty0 = 9,   // [2]
    kSFull0 = 11,   // [2] per tile: S(j) in TMEM
    kPFull0 = 13,   // [2] per tile: P(j) in TMEM (every softmax warp of the tile arrives)
    kODone0 = 15,   // [2] per tile: the tile's last O += P V of an item done
    kDrain = 17,
    kQEmpty = 18,      // the item's last S MMA has read Q
    kItemFull0 = 19,   // [2] item ring slot written
    kItemEmpty0 = 21,  // [2] item ring slot read by every role
};

// Tiles of a sequence with n new tokens (the decode path takes n <= qmax), and
// the work items (pairs of tiles, or single tiles at D = 256) they make per KV head.
__device__ __forceinline__ int tiles_of(int n, int tq, int qmax) { return n > qmax ? (n + tq - 1) / tq : 0; }
__device__ __forceinline__ int pairs_of(int n, int tq, int qmax, int tiles_per_item) {
    return (tiles_of(n, tq, qmax) + tiles_per_item - 1) / tiles_per_item;
}

// Register budget of the calling warpgroup (every warp of it executes the same one).
template <uint32_t N>
__device__ __forceinline__ void reg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void reg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N)); }

// Bounded wait by every lane of a warp; the result is made warp-uniform so that a
// timeout can never leave some lanes at a warp-collective instruction alone.
// (Polling from lane 0 alone and broadcasting was measured slower: 1096 -> 993
// TFLOP/s on the varlen prefill.)
__device__ __forceinline__ bool warp_wait(uint32_t addr, uint32_t parity, const volatile int* abort) {
    const bool ok = tc::mbar_wait(addr, parity, abort, kTimeoutNs);
    return __all_sync(0xffffffffu, ok);
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled half.
__device__ __forceinline__ uint32_t sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float2 unpack2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;\n" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

// acc += the two bf16 halves of v, widened (two mixed-precision adds): the
// normaliser l sums exactly the bf16-rounded P that the P V product consumes.
__device__ __forceinline__ void add_bf16_pair(uint64_t& acc, uint32_t v) {
    float a0, a1;
    unsigned short lo, hi;
    asm("mov.b64 {%0, %1}, %2;\n" : "=f"(a0), "=f"(a1) : "l"(acc));
    asm("mov.b32 {%0, %1}, %2;\n" : "=h"(lo), "=h"(hi) : "r"(v));
    asm("add.rn.f32.bf16 %0, %1, %0;\n" : "+f"(a0) : "h"(lo));
    asm("add.rn.f32.bf16 %0, %1, %0;\n" : "+f"(a1) : "h"(hi));
    asm("mov.b64 %0, {%1, %2};\n" : "=l"(acc) : "f"(a0), "f"(a1));
}

// (a0, a1) * (b, b) + (c, c) on the packed f32x2 FMA.
__device__ __forceinline__ void fma2(float& y0, float& y1, float a0, float a1, float b, float c) {
    uint64_t a, bb, cc, y;
    asm("mov.b64 %0, {%1, %2};\n" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %1};\n" : "=l"(bb) : "f"(b));
    asm("mov.b64 %0, {%1, %1};\n" : "=l"(cc) : "f"(c));
    asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(y) : "l"(a), "l"(bb), "l"(cc));
    asm("mov.b64 {%0, %1}, %2;\n" : "=f"(y0), "=f"(y1) : "l"(y));
}

// One S tile: D / 16 MMAs of K = 16 (the K steps walk the two 64-column halves
// of Q and K), accumulating from the second on.
template <int D>
__device__ __forceinline__ void issue_s_group(uint32_t d, uint64_t da, uint64_t db, uint32_t idesc) {
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t off = static_cast<uint64_t>((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4;
        tc::mma_bf16(d, da + off, db + off, idesc, ks > 0 ? 1u : 0u);
    }
}
// One P V step over the npj pages of a KV tile: A = P from TMEM (8 columns per
// 16 keys), B = V (one page of 16 keys per MMA, 2 KiB apart).
__device__ __forceinline__ void issue_pv_group(uint32_t d, uint32_t pa, uint64_t db, uint32_t idesc, int npj,
                                               bool first) {
#pragma unroll
    for (int ks = 0; ks < kPagesPerTile; ++ks)
        if (ks < npj) tc::mma_bf16_tmem_a(d, pa + ks * 8, db + ks * (2048 >> 4), idesc, (!first || ks > 0) ? 1u : 0u);
}

// A work item is (pair of query tiles, KV head).  Items are numbered pair-major:
// item w is pair w / Hkv of KV head w % Hkv, pairs counted over the sequences in
// order and, within a sequence, last pair first (it sees the most keys), so the
// items handed out last are the shortest of the last sequence.
struct Item {
    int b;   // sequence; -1: no item left
    int h;   // KV head
    int i0;  // first new token (within the sequence) of tile A
    int q0;  // first query row of the sequence
    int n;   // new tokens of the sequence
    int L;   // keys of the sequence (clamped to the block table's capacity)
    int pad[2];
};
enum ItemStatus { kItemEnd = 0, kItemOk = 1, kItemSkip = 2 };

// Resolves item w (warp-collective; every lane gets the same result).  An item
// whose metadata are inconsistent is settled here (error code; rows of a query
// longer than its sequence written as zeros) and reported as skipped.
template <int D, int kTiles>
__device__ ItemStatus resolve_item(const Args& a, int w, int tq_tokens, Item& it, int lane) {
    const int pidx = w / a.num_kv_heads;
    int found_b = -1, found_p = 0, base_t = 0, q0 = 0, n = 0;
    for (int b0 = 0; b0 < a.num_seqs && found_b < 0; b0 += 32) {
        const int b = b0 + lane;
        int s0 = 0, s1 = 0;
        if (b < a.num_seqs) {
            s0 = a.query_start_loc[b];
            s1 = a.query_start_loc[b + 1];
        }
        const int cnt = b < a.num_seqs ? pairs_of(s1 - s0, tq_tokens, a.decode_max_q, kTiles) : 0;
        int inc = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        const int excl = base_t + inc - cnt;
        const unsigned m = __ballot_sync(0xffffffffu, cnt > 0 && pidx >= excl && pidx < excl + cnt);
        if (m) {
            const int src = __ffs(m) - 1;
            found_b = b0 + src;
            found_p = __shfl_sync(0xffffffffu, excl + cnt - 1, src) - pidx;  // last pair first
            q0 = __shfl_sync(0xffffffffu, s0, src);
            n = __shfl_sync(0xffffffffu, s1 - s0, src);
        }
        base_t += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (found_b < 0) return kItemEnd;  // w is past the last item
    it.b = found_b;
    it.h = w - pidx * a.num_kv_heads;
    it.i0 = found_p * kTiles * tq_tokens;
    it.q0 = q0;
    it.n = n;
    if (q0 < 0 || static_cast<int64_t>(q0) + n > a.num_tokens) {
        if (lane == 0) flag_error(a.err, kDevBadQueryStart);
        return kItemSkip;
    }
    const int cap = a.max_pages * kPage;
    int L = a.seq_lens[found_b];
    if (L > cap) {
        if (lane == 0) flag_error(a.err, kDevSeqTooLong);
        L = cap;
    }
    it.L = L;
    if (L < n) {
        if (lane == 0) flag_error(a.err, kDevQueryTooLong);
        const int G = a.group;
        const int rows = min(kTiles * tq_tokens, n - it.i0) * G;
        __nv_bfloat16* const out = reinterpret_cast<__nv_bfloat16*>(a.out);
        for (int i = lane; i < rows * D; i += 32) {
            const int r = i / D;
            out[(static_cast<int64_t>(q0 + it.i0 + r / G) * a.num_q_heads + it.h * G + r % G) * D + i % D] =
                __float2bfloat16(0.f);
        }
        return kItemSkip;
    }
    return kItemOk;
}

// What every role derives from an item.
struct ItemShape {
    int ntok[2];     // new tokens of tile x
    int nkv[2];      // KV tiles up to tile x's last causal position
    int ntiles;      // KV tiles of the item
    int last_page;   // pages [0, last_page) are read
    int full_pages;  // pages with no slot past L
    int prefix;      // cached keys before the first new token
};
__device__ __forceinline__ ItemShape shape_of(const Item& it, int tq_tokens, int kTiles) {
    ItemShape s;
    s.prefix = it.L - it.n;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        s.ntok[x] = x < kTiles ? max(0, min(tq_tokens, it.n - (it.i0 + x * tq_tokens))) : 0;
        s.nkv[x] = s.ntok[x] > 0 ? (s.prefix + it.i0 + x * tq_tokens + s.ntok[x] + kKeys - 1) / kKeys : 0;
    }
    s.ntiles = max(s.nkv[0], s.nkv[1]);
    const int kv_end = s.prefix + it.i0 + s.ntok[0] + s.ntok[1];  // keys [0, kv_end) are visible to some row
    s.last_page = (kv_end + kPage - 1) / kPage;
    s.full_pages = it.L / kPage;
    return s;
}

// Persistent: one CTA per SM walks the items.  Warp 0 resolves the CTA's next
// item (its first is blockIdx.x, later ones come from an atomic counter in the
// workspace, so CTAs that finish early take more) and publishes it in a 2-slot
// ring of shared memory that every other role reads in the same order.  All ring
// and barrier positions run on across items, so the next item's Q, K and first
// S MMAs proceed while the softmax warps still finish the previous one.
template <int D>
__global__ void __launch_bounds__(Cfg<D>::kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const Args a, int tq_tokens) {
    using S = Smem<D>;
    constexpr int kTiles = Cfg<D>::kTiles, kKStages = Cfg<D>::kKStages, kVStages = Cfg<D>::kVStages;
    constexpr int kColSplit = Cfg<D>::kColSplit;
    constexpr uint32_t kRegsIssue = Cfg<D>::kRegsIssue, kRegsSoftmax = Cfg<D>::kRegsSoftmax;
    // setmaxnreg only where a budget differs from the launch's
    constexpr bool kDecRegs = kRegsIssue < Cfg<D>::kRegsLaunch, kIncRegs = kRegsSoftmax > Cfg<D>::kRegsLaunch;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const sp = smem_raw + (base - raw);
    auto bar = [&](int i) { return base + S::kBar + 8 * i; };
    uint32_t* const s_tmem = reinterpret_cast<uint32_t*>(sp + S::kMisc);
    volatile int* const s_abort = reinterpret_cast<volatile int*>(sp + S::kMisc + 4);
    Item* const s_items = reinterpret_cast<Item*>(sp + S::kItems);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.group;

    // ---- barriers and TMEM, once per CTA
    if (threadIdx.x == 0) {
        tc::mbar_init(bar(kQFull), 1);
        tc::mbar_init(bar(kQEmpty), 1);
        for (int i = 0; i < kMaxKStages; ++i) {
            tc::mbar_init(bar(kKFull0 + i), 1);
            tc::mbar_init(bar(kKEmpty0 + i), 1);
        }
        for (int i = 0; i < kMaxVStages; ++i) {
            tc::mbar_init(bar(kVFull0 + i), 1);
            tc::mbar_init(bar(kVEmpty0 + i), 1);
        }
        for (int x = 0; x < 2; ++x) {
            tc::mbar_init(bar(kSFull0 + x), 1);
            tc::mbar_init(bar(kPFull0 + x), 4 * kColSplit);
            tc::mbar_init(bar(kODone0 + x), 1);
            tc::mbar_init(bar(kItemFull0 + x), 1);
            // readers of an item: the MMA thread, the V producer, the softmax warps
            tc::mbar_init(bar(kItemEmpty0 + x), 2 + 4 * kTiles * kColSplit);
        }
        tc::mbar_init(bar(kDrain), 1);
        *s_abort = 0;
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

    if (warp == 0 || warp == kWarpV) {
        if constexpr (kDecRegs) reg_dec<kRegsIssue>();
        // ===================== scheduler + Q and K producer (warp 0), V producer (warp 2)
        const bool is_v = warp == kWarpV;
        if (lane == 0) {
            if (!is_v) {
                tc::prefetch_tmap(&tm_q);
                tc::prefetch_tmap(&tm_k);
            } else {
                tc::prefetch_tmap(&tm_v);
            }
        }
        const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(a.v_cache);
        const int stages = is_v ? kVStages : kKStages;
        const int full0 = is_v ? kVFull0 : kKFull0, empty0 = is_v ? kVEmpty0 : kKEmpty0;
        const uint32_t ring = base + (is_v ? S::kV0 : S::kK0);
        const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
        int w = blockIdx.x;  // warp 0: the item to resolve next
        uint32_t tc_n = 0;   // K or V tiles loaded so far (ring position)
        for (int it = 0;; ++it) {
            const int slot = it & 1;
            Item itm;
            if (!is_v) {
                ItemStatus st;
                while ((st = resolve_item<D, kTiles>(a, w, tq_tokens, itm, lane)) == kItemSkip) {
                    int wn = 0;
                    if (lane == 0) wn = static_cast<int>(gridDim.x) + atomicAdd(a.sched, 1);
                    w = __shfl_sync(0xffffffffu, wn, 0);
                }
                if (st == kItemEnd) itm.b = -1;
                if (it >= 2 && !warp_wait(bar(kItemEmpty0 + slot), ((it >> 1) - 1) & 1, s_abort)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    s_items[slot] = itm;
                    tc::mbar_arrive(bar(kItemFull0 + slot));
                }
                __syncwarp();
            } else {
                if (!warp_wait(bar(kItemFull0 + slot), (it >> 1) & 1, s_abort)) {
                    ok = false;
                    break;
                }
                itm = s_items[slot];
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(kItemEmpty0 + slot));
            }
            if (itm.b < 0) break;
            // warp 0: the number of the item after this one, fetched while this one loads
            int wn = 0;
            if (!is_v && lane == 0) wn = static_cast<int>(gridDim.x) + atomicAdd(a.sched, 1);
            const ItemShape sh = shape_of(itm, tq_tokens, kTiles);
            const int h = itm.h, L = itm.L;
            const int32_t* bt = a.block_table + static_cast<int64_t>(itm.b) * a.max_pages;
            // lane l holds the block-table entry of page (group * 32 + l); the next
            // group's entries are loaded while the current group is being used.
            auto load_group = [&](int grp) -> int {
                const int pg = grp * kTilesPerGroup * kPagesPerTile + lane;
                return pg < sh.last_page ? bt[pg] : 0;
            };
            int cur_grp = load_group(0);
            int next_grp = load_group(1);
            for (int kt = 0; kt < sh.ntiles; ++kt) {
                const int gslot = kt % kTilesPerGroup;
                if (gslot == 0 && kt > 0) {
                    cur_grp = next_grp;
                    next_grp = load_group(kt / kTilesPerGroup + 1);
                }
                const int p0 = kt * kPagesPerTile;
                const int np = min(kPagesPerTile, sh.last_page - p0);
                // pages by TMA: all of K; V up to the one holding the sequence end
                const int nt = is_v ? max(0, min(np, sh.full_pages - p0)) : np;
                int page = __shfl_sync(0xffffffffu, cur_grp, (gslot * kPagesPerTile + lane) & 31);
                if (lane < np && static_cast<uint32_t>(page) >= static_cast<uint64_t>(a.num_blocks)) {
                    flag_error(a.err, kDevBadBlock);
                    page = 0;
                }
                const int st = tc_n % stages;
                if (tc_n >= static_cast<uint32_t>(stages) &&
                    !warp_wait(bar(empty0 + st), (tc_n / stages - 1) & 1, s_abort)) {
                    ok = false;
                    break;
                }
                const uint32_t sd = ring + st * S::kTile;
                if (is_v && nt < np) {
                    // The V page holding the sequence end: plain loads, slots >= L as zeros.
                    const int pi = np - 1;
                    const int pg = __shfl_sync(0xffffffffu, page, pi);
                    for (int c = lane; c < kPage * (D / 8); c += 32) {
                        const int t = c / (D / 8), ch = c % (D / 8);
                        const int row = pi * kPage + t;
                        uint4 val = make_uint4(0u, 0u, 0u, 0u);
                        if ((p0 + pi) * kPage + t < L)
                            val = *reinterpret_cast<const uint4*>(
                                vc + ((static_cast<int64_t>(pg) * kPage + t) * a.num_kv_heads + h) * D + ch * 8);
                        const uint32_t dst = sd + (ch >> 3) * kHalfBytes + sw128(row, ch & 7);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(val.x), "r"(val.y),
                                     "r"(val.z), "r"(val.w)
                                     : "memory");
                    }
                    tc::fence_proxy_async_smem();
                }
                __syncwarp();
                // (tests only: CTA 0 withholds the K tile of its first item, so
                // that the MMA thread's wait for it runs out)
                const bool withhold = a.test_stall_prefill && !is_v && blockIdx.x == 0 && it == 0 && kt == 0;
                if (lane == 0 && !withhold) tc::mbar_arrive_expect_tx(bar(full0 + st), nt * S::kHalves * 2048);
                __syncwarp();
                if (lane < nt && !withhold) {
#pragma unroll
                    for (int hf = 0; hf < S::kHalves; ++hf)
                        tc::tma_load_4d(sd + hf * kHalfBytes + lane * 2048, tm, bar(full0 + st), hf * 64, h, 0, page);
                }
                ++tc_n;
                if (!is_v && kt == 0) {
                    // Q of this item (after its first K tile): once the previous
                    // item's last S MMA has read the Q buffer.
                    if (it > 0 && !warp_wait(bar(kQEmpty), (it - 1) & 1, s_abort)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        const int nq = sh.ntok[1] > 0 ? 2 : 1;
                        tc::mbar_arrive_expect_tx(bar(kQFull), nq * S::kHalves * 64 * 2 * G * tq_tokens);
                        for (int x = 0; x < nq; ++x)
#pragma unroll
                            for (int hf = 0; hf < S::kHalves; ++hf)
                                tc::tma_load_3d(base + S::kQ0 + x * S::kTile + hf * kHalfBytes, &tm_q, bar(kQFull),
                                                hf * 64, h * G, itm.q0 + itm.i0 + x * tq_tokens);
                    }
                    __syncwarp();
                }
                // L2 prefetch of the pages kPrefetchTiles tiles ahead, so that their
                // ring loads find them in L2 rather than in HBM.
                if (kPrefetchTiles > 0 && kt + kPrefetchTiles < sh.ntiles) {
                    const int kp = kt + kPrefetchTiles;
                    const int pp0 = kp * kPagesPerTile;
                    const int npp = min(kPagesPerTile, sh.last_page - pp0);
                    const int spg = kp % kTilesPerGroup;
                    // tile kp's entries: in this group, or (kp / 4 > kt / 4) in the next
                    const int src = (kp / kTilesPerGroup == kt / kTilesPerGroup) ? cur_grp : next_grp;
                    const int ppage = __shfl_sync(0xffffffffu, src, (spg * kPagesPerTile + lane) & 31);
                    if (lane < npp && static_cast<uint32_t>(ppage) < static_cast<uint64_t>(a.num_blocks)) {
#pragma unroll
                        for (int hf = 0; hf < S::kHalves; ++hf) tc::tma_prefetch_4d(tm, hf * 64, h, 0, ppage);
                    }
                }
            }
            if (!ok) break;
            if (!is_v) w = __shfl_sync(0xffffffffu, wn, 0);
        }
        if (!ok && lane == 0) {
            *s_abort = 1;
            flag_error(a.err, kDevWaitTimeout);
        }
    } else if (warp == 1) {
        // ===================================================== MMA issuer
        if constexpr (kDecRegs) reg_dec<kRegsIssue>();
        if (lane == 0) {
            constexpr uint32_t kIdQK = tc::idesc_bf16_f32(kM, kKeys, false, false);
            constexpr uint32_t kIdPV = tc::idesc_bf16_f32(kM, D, false, true);
            // Shared-memory descriptors, computed once: an MMA only adds a
            // constant to the start-address field (16-byte units; every operand
            // lies below 256 KiB, so the 14-bit field never carries).  Issuing
            // is the bottleneck of this thread (a tcgen05.mma costs tens of
            // cycles to issue), so nothing else is computed per MMA and the
            // groups are plain inline functions of register values.
            const uint64_t dq0 = tc::desc_sw128(base + S::kQ0, 16, 1024);
            const uint64_t dk0 = tc::desc_sw128(base + S::kK0, 16, 1024);
            const uint64_t dv0 = tc::desc_sw128(base + S::kV0, kHalfBytes, 1024);
            constexpr uint64_t kTileU = S::kTile >> 4;
            const uint32_t d_s0 = tmem + tmem_s(0), d_s1 = tmem + tmem_s(1);
            const uint32_t d_o0 = tmem + tmem_o(0), d_o1 = tmem + tmem_o(1);
            uint32_t kc = 0, vc = 0, pc0 = 0, pc1 = 0;  // K and V tiles, P tiles consumed so far
#define PA_ISSUE_S(x)                                                                                         \
    do {                                                                                                      \
        issue_s_group<D>((x) ? d_s1 : d_s0, dq0 + ((x) ? kTileU : 0), dk0 + (kc % kKStages) * kTileU, kIdQK); \
        tc::mma_commit(bar(kSFull0 + (x)));                                                                   \
    } while (0)
// (the caller has waited for P_x(jj))
#define PA_ISSUE_PV(x, jj)                                                                                  \
    do {                                                                                                    \
        tc::tc_fence_after();                                                                               \
        issue_pv_group((x) ? d_o1 : d_o0, ((x) ? d_s1 : d_s0) + 64, dv0 + (vc % kVStages) * kTileU, kIdPV,  \
                       min(kPagesPerTile, last_page - (jj) * kPagesPerTile), (jj) == 0);                    \
        if ((jj) == ((x) ? nkv1 : nkv0) - 1) tc::mma_commit(bar(kODone0 + (x)));                            \
    } while (0)
            for (int it = 0; ok; ++it) {
                const int slot = it & 1;
                if (!(ok = tc::mbar_wait(bar(kItemFull0 + slot), (it >> 1) & 1, s_abort, kTimeoutNs))) break;
                const Item itm = s_items[slot];
                tc::mbar_arrive(bar(kItemEmpty0 + slot));
                if (itm.b < 0) break;
                const ItemShape sh = shape_of(itm, tq_tokens, kTiles);
                const int nkv0 = sh.nkv[0], nkv1 = sh.nkv[1], ntiles = sh.ntiles, last_page = sh.last_page;
                if (!(ok = tc::mbar_wait(bar(kQFull), it & 1, s_abort, kTimeoutNs))) break;
                if (!(ok = tc::mbar_wait(bar(kKFull0 + kc % kKStages), (kc / kKStages) & 1, s_abort, kTimeoutNs)))
                    break;
                tc::tc_fence_after();
                // S(0) of both tiles.  The P V that read each tile's last P of the
                // previous item was issued before, and one thread's tcgen05
                // operations execute in issue order.
                if (nkv0 > 0) PA_ISSUE_S(0);
                if (nkv1 > 0) PA_ISSUE_S(1);
                tc::mma_commit(bar(kKEmpty0 + kc % kKStages));
                ++kc;
                if (ntiles == 1) tc::mma_commit(bar(kQEmpty));
                for (int j = 0; j < ntiles && ok; ++j) {
                    const bool nxt0 = j + 1 < nkv0, nxt1 = j + 1 < nkv1;
                    ok = tc::mbar_wait(bar(kVFull0 + vc % kVStages), (vc / kVStages) & 1, s_abort, kTimeoutNs);
                    if (!ok) break;
                    tc::tc_fence_after();
                    if (j < nkv0) {
                        // (P_A(0) of an item arrives after its softmax warps have
                        // read the previous item's O_A, which this P V overwrites)
                        if (!(ok = tc::mbar_wait(bar(kPFull0), pc0 & 1, s_abort, kTimeoutNs))) break;
                        ++pc0;
                        PA_ISSUE_PV(0, j);
                    }
                    if (nxt0 || nxt1) {
                        ok = tc::mbar_wait(bar(kKFull0 + kc % kKStages), (kc / kKStages) & 1, s_abort, kTimeoutNs);
                        if (!ok) break;
                        tc::tc_fence_after();
                    }
                    if (nxt0) PA_ISSUE_S(0);
                    if (j < nkv1) {
                        if (!(ok = tc::mbar_wait(bar(kPFull0 + 1), pc1 & 1, s_abort, kTimeoutNs))) break;
                        ++pc1;
                        PA_ISSUE_PV(1, j);
                    }
                    tc::mma_commit(bar(kVEmpty0 + vc % kVStages));
                    ++vc;
                    if (nxt1) PA_ISSUE_S(1);
                    if (nxt0 || nxt1) {
                        tc::mma_commit(bar(kKEmpty0 + kc % kKStages));
                        ++kc;
                        if (j + 2 == ntiles) tc::mma_commit(bar(kQEmpty));  // the item's last S MMAs
                    }
                }
            }
#undef PA_ISSUE_S
#undef PA_ISSUE_PV
            if (!ok) {
                *s_abort = 1;
                flag_error(a.err, kDevWaitTimeout);
            }
            // drain: every MMA issued above has finished before TMEM is freed
            tc::mma_commit(bar(kDrain));
            tc::mbar_wait(bar(kDrain), 0, nullptr, kTimeoutNs);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 4 + 4 * kTiles * kColSplit) {
        // ======================================================== softmax
        // Warp 4 + 4 t + q (t = tile, q = TMEM lane quarter) takes the tile's S
        // columns [0, kCols) and, with the column split, warp 4 + 8 + 4 t + q
        // takes [kCols, 128) of the same 32 rows; the two exchange their row
        // maxima (and at the end their sums l) through shared memory.
        if constexpr (kIncRegs) reg_inc<kRegsSoftmax>();
        constexpr int kCols = kKeys / kColSplit;  // S columns of this warp
        constexpr int kOCols = D / kColSplit;     // O columns this warp rescales and writes
        const int sw = warp - 4;
        const int x = (sw >> 2) & (kTiles - 1);   // tile: A or B
        const int half = sw >> 3;                 // column half (0 without the split)
        const int quarter = warp & 3;             // TMEM lanes 32 * (warp % 4) ..
        const int r = quarter * 32 + lane;        // row == TMEM lane
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t s_addr = lane_addr + tmem_s(x);
        const uint32_t my_s = s_addr + half * kCols;
        const uint32_t my_p = s_addr + 64 + half * (kCols / 2);  // key k -> column 64 + k / 2
        const uint32_t o_addr = lane_addr + tmem_o(x) + half * kOCols;
        float* const xmax = reinterpret_cast<float*>(sp + S::kXMax);  // [buf][tile][half][row]
        float* const xl = reinterpret_cast<float*>(sp + S::kXL);      // [tile][half][row]
        // The pair meets at a named barrier (1 + tile * 4 + quarter; 0 is
        // __syncthreads) after each of its bounded mbarrier waits, with a
        // reduction of the two warps' wait results: both continue, or both
        // leave (on a timeout or an abort seen by either), so neither can be
        // left waiting at the barrier for a partner that has gone.  The barrier
        // also publishes the values each warp wrote to shared memory before it.
        const int pair_bar = 1 + x * 4 + quarter;
        auto pair_and = [&](bool v) -> bool {
            if constexpr (kColSplit > 1) {
                uint32_t both;
                tc::tc_fence_before();
                asm volatile(
                    "{\n"
                    ".reg .pred p, q;\n"
                    "setp.ne.u32 p, %1, 0;\n"
                    "bar.red.and.pred q, %2, 64, p;\n"
                    "selp.u32 %0, 1, 0, q;\n"
                    "}\n"
                    : "=r"(both)
                    : "r"(static_cast<uint32_t>(v)), "r"(pair_bar)
                    : "memory");
                tc::tc_fence_after();
                return both != 0;
            } else {
                return v;
            }
        };
        const float c = a.scale_log2;
        uint32_t sc = 0, oc = 0;  // S tiles and finished O of this tile so far
        for (int it = 0; ok; ++it) {
            const int slot = it & 1;
            if (!pair_and(warp_wait(bar(kItemFull0 + slot), (it >> 1) & 1, s_abort))) {
                ok = false;
                break;
            }
            const Item itm = s_items[slot];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(kItemEmpty0 + slot));
            if (itm.b < 0) break;
            const ItemShape shp = shape_of(itm, tq_tokens, kTiles);
            const int nt = x ? shp.nkv[1] : shp.nkv[0];
            if (nt == 0) continue;
            const int t0 = itm.i0 + x * tq_tokens;  // first new token of this tile
            const bool valid = r < (x ? shp.ntok[1] : shp.ntok[0]) * G;
            const int pos = valid ? shp.prefix + t0 + r / G : -1;  // causal limit of this row
            float m_used = -INFINITY;  // running max, log2 units
            uint64_t lsum[2] = {0, 0};  // 4 independent partial sums, in f32x2 pairs (0 = +0.0f, +0.0f)
            for (int kt = 0; kt < nt; ++kt) {
                const bool s_ready = warp_wait(bar(kSFull0 + x), sc & 1, s_abort);
                if (kColSplit == 1 && !s_ready) {
                    ok = false;
                    break;
                }
                const int buf = sc & 1;
                ++sc;
                tc::tc_fence_after();
                const int j0 = kt * kKeys + half * kCols;  // key of this warp's first column
                const bool diag = __any_sync(0xffffffffu, j0 + kCols - 1 > pos);
                // This warp's S columns in one load and one wait.
                uint32_t sh[kCols];
                if constexpr (kCols == 128)
                    tc::tmem_ld128(my_s, sh);
                else
                    tc::tmem_ld64(my_s, sh);
                if (diag) {
#pragma unroll
                    for (int j = 0; j < kCols; ++j)
                        if (j0 + j > pos) sh[j] = __float_as_uint(-INFINITY);
                }
                float mx8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx8[e] = max3(__uint_as_float(sh[e]), __uint_as_float(sh[8 + e]),
                                                          __uint_as_float(sh[16 + e]));
#pragma unroll
                for (int j = 24; j < kCols - 8; j += 16)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        mx8[e] = max3(mx8[e], __uint_as_float(sh[j + e]), __uint_as_float(sh[j + 8 + e]));
#pragma unroll
                for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(mx8[e], __uint_as_float(sh[kCols - 8 + e]));
                float mx = max3(max3(mx8[0], mx8[1], mx8[2]), max3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
                if constexpr (kColSplit > 1) {
                    // the row max over both halves; both warps of the pair then
                    // take the same rescale decisions.  (Two buffers: a warp may
                    // write the next tile's max before its partner read this one.)
                    float* const xm = xmax + ((buf * 2 + x) * 2) * kM;
                    xm[half * kM + r] = mx;
                    if (!pair_and(s_ready)) {
                        ok = false;
                        break;
                    }
                    mx = fmaxf(mx, xm[(1 - half) * kM + r]);
                }
                const float mnew = mx * c;  // scale > 0, so the max commutes with it
                float alpha = 1.f;
                bool rescale = false;
                if (kt == 0) {
                    m_used = mnew;
                } else {
                    const bool need = mnew > m_used + 8.f;
                    if (__any_sync(0xffffffffu, need)) {
                        alpha = need ? fast_exp2(m_used - mnew) : 1.f;
                        rescale = true;
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float2 v = unpack2(lsum[e]);
                            asm("mov.b64 %0, {%1, %2};\n" : "=l"(lsum[e]) : "f"(v.x * alpha), "f"(v.y * alpha));
                        }
                        if (need) m_used = mnew;
                    }
                }
                const float nmu = m_used == -INFINITY ? 0.f : -m_used;
                // P = 2^(s*c - m) as bf16 pairs over the last 64 columns of S (key
                // k of the tile to column 64 + k / 2), 32 keys per store.  Every S
                // column of the tile is in the registers of one of the pair's
                // warps by now (the exchange above follows both loads), so any
                // column may be overwritten; the P V that read the previous P
                // finished before this S was written.  l sums the same bf16
                // values, so V rows all equal to c give c.
#pragma unroll
                for (int ch = 0; ch < kCols / 32; ++ch) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float y0, y1;
                        fma2(y0, y1, __uint_as_float(sh[32 * ch + 2 * e]), __uint_as_float(sh[32 * ch + 2 * e + 1]), c,
                             nmu);
                        const float x0 = fast_exp2(y0), x1 = fast_exp2(y1);
                        pk[e] = pack_bf16(x0, x1);
                        add_bf16_pair(lsum[e & 1], pk[e]);
                    }
                    tc::tmem_st16_async(my_p + 16 * ch, pk);
                }
                tc::tmem_wait_st();
                if (rescale) {
                    // O holds tiles < kt: P V(kt-1) was issued before S(kt), and
                    // the commit this warp waited for to read S(kt) completes only
                    // after every earlier MMA of the issuing thread; P V(kt) waits
                    // for this warp's arrival below.  Each warp of a pair rescales
                    // its own columns of O.
#pragma unroll
                    for (int q = 0; q < kOCols / 32; ++q) {
                        uint32_t o[32];
                        tc::tmem_ld32(o_addr + q * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::tmem_st32(o_addr + q * 32, o);
                    }
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(kPFull0 + x));
            }
            if (!ok) break;
            const bool o_ready = warp_wait(bar(kODone0 + x), oc & 1, s_abort);
            ++oc;
            tc::tc_fence_after();
            const float2 l0 = unpack2(lsum[0]), l1 = unpack2(lsum[1]);
            float l = (l0.x + l0.y) + (l1.x + l1.y);
            if constexpr (kColSplit > 1) {
                // l over both halves (the partner reads this slot before either
                // warp can write it again: the next item's max exchanges come
                // in between)
                xl[(x * 2 + half) * kM + r] = l;
            }
            if (!pair_and(o_ready)) {
                ok = false;
                break;
            }
            if constexpr (kColSplit > 1) l += xl[(x * 2 + 1 - half) * kM + r];
            const float inv = valid ? 1.f / l : 0.f;
            __nv_bfloat16* orow =
                reinterpret_cast<__nv_bfloat16*>(a.out) +
                (static_cast<int64_t>(itm.q0 + t0 + (valid ? r / G : 0)) * a.num_q_heads + itm.h * G + r % G) * D +
                half * kOCols;
#pragma unroll
            for (int q = 0; q < kOCols / 32; ++q) {
                uint32_t o[32];
                tc::tmem_ld32(o_addr + q * 32, o);
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
            // (O has been read out: the next item's first P V, which overwrites
            // O, waits for this warp's next P, arrived after this point.)
        }
        if (!ok && lane == 0) {
            *s_abort = 1;
            flag_error(a.err, kDevWaitTimeout);
        }
    } else if (warp < 4) {
        if constexpr (kDecRegs) reg_dec<kRegsIssue>();  // idle warp of warpgroup 0
    } else {
        if constexpr (kIncRegs) reg_inc<kRegsSoftmax>();  // idle softmax warps (one query tile per CTA)
    }

    // ---- teardown: every role is out of its loop; the MMA thread has drained.
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    // The last CTA to finish returns the item counters to zero for the next
    // launch (every CTA's last fetch precedes its arrival here).
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(a.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            __threadfence();
            atomicExch(a.sched, 0);
            atomicExch(a.sched + 1, 0);
        }
    }
}

// --------------------------------------------------------------- host side
int tokens_per_tile(int group) { return group <= kM ? kM / group : 0; }

// Upper bound on the tile pairs (single tiles at D = 256) of any batch with these
// shapes: sum over sequences of ceil(ceil(n_b / TQ) / k) = sum of
// ceil(n_b / (k TQ)) <= T / (k TQ) + B, with k tiles per pair.
int pairs_bound(const Args& a) {
    const int tq = tokens_per_tile(a.group);
    if (tq == 0) return 0;
    const int per_cta = a.head_dim <= 128 ? 2 : 1;  // Cfg<D>::kTiles
    return static_cast<int>(a.num_tokens / (per_cta * tq) + a.num_seqs);
}

template <int D>
cudaError_t launch_d(const Args& a, cudaStream_t stream) {
    using S = Smem<D>;
    // One-time set-up per device.  Host threads may race here; both then set
    // the same values, which is harmless, and the flags are atomic.
    static std::atomic<bool> configured[64];
    static std::atomic<int> sms[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configured[dev & 63].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             S::kAlloc);
        if (e != cudaSuccess) return e;
        // The warpgroups' register split must fit in what the CTA launches with,
        // or setmaxnreg.inc would wait for registers that never come.
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, prefill_tc_kernel<D>);
        if (e != cudaSuccess) return e;
        if (static_cast<uint32_t>(fa.numRegs) < Cfg<D>::kRegsLaunch) return cudaErrorInvalidConfiguration;
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        sms[dev & 63].store(n, std::memory_order_relaxed);
        configured[dev & 63].store(true, std::memory_order_release);
    }
    const int64_t items = prefill_ctas(a);
    if (items == 0) return cudaSuccess;
    // one persistent CTA per SM (at most one per item)
    const int nsm = sms[dev & 63].load(std::memory_order_relaxed);
    const int64_t ctas = items < nsm ? items : nsm;
    const int G = a.group, tq = tokens_per_tile(G);
    CUtensorMap tq_map, tk_map, tv_map;
    if (!encode_q_map(&tq_map, a.q, D, a.num_q_heads, a.num_tokens, G, tq) ||
        !encode_cache_map(&tk_map, a.k_cache, D, a.num_kv_heads, a.num_blocks) ||
        !encode_cache_map(&tv_map, a.v_cache, D, a.num_kv_heads, a.num_blocks))
        return cudaErrorInvalidValue;
    // (no programmatic dependent launch: back-to-back prefill calls gained
    // nothing measurable from it, and mixed batches, whose prefill kernel runs
    // beside the decode kernel, lost 2 %)
    return launch_kernel(prefill_tc_kernel<D>, static_cast<unsigned>(ctas), Cfg<D>::kThreads, S::kAlloc, stream, 1, false, tq_map,
                         tk_map, tv_map, a, tq);
}

}  // namespace

// Work items (tile pairs x KV heads) of the largest batch with these shapes.
int64_t prefill_ctas(const Args& a) {
    if (a.num_tokens < 2) return 0;
    return static_cast<int64_t>(pairs_bound(a)) * a.num_kv_heads;
}

cudaError_t launch_prefill(const Args& a, cudaStream_t stream) {
    switch (a.head_dim) {
        case 64: return launch_d<64>(a, stream);
        case 128: return launch_d<128>(a, stream);
        case 256: return launch_d<256>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
