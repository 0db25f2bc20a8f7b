// decode.cu -- GQA Q-block split-KV decode kernel.
//
// One CTA owns (sequence b, KV head h, row group rg, split s).  Its query rows
// are the G query heads sharing h times the n_b new tokens of b (n_b * G <= 16:
// a single decode token, or a few speculative-decoding tokens), row r = (token
// r / G, head h*G + r % G); with more than 16 heads per KV head, single-token
// sequences only, in row groups of 16 heads.  This is the "Q-Block" item of the
// five-step list on the Triton unified-attention page, section "What three things
// the IBM paper got right": query heads sharing a KV head are computed together,
// so each KV page is read once per KV head, not once per query head.  Split s
// covers keys [s*kv_chunk, min((s+1)*kv_chunk, L_b)) -- one tile of the
// "Parallel Tiled Softmax" item of the same list -- or, in cluster mode, every
// C-th page of the sequence starting at page s; each row is masked causally at
// its own position L_b - n_b + token.
//
// Inside the CTA, kWarps warps (4, 8 or 12) take its pages round-robin.  Each
// warp runs its own kStages-deep cp.async pipeline of 16-token pages of K and V
// (16-byte copies into an XOR-swizzled layout, so the ldmatrix fragment loads
// are bank-conflict free), computes S = Q K^T and O += P V with bf16 m16n8k16
// MMAs (the query rows padded to 16), and keeps an online softmax (running max
// m, sum l; the recurrence of "The Flash Attention revolution" on the GPU
// programming guide page) in the log2 domain.  At the end the warps' (m, l, O)
// are merged in shared memory; a sequence with one split writes bf16 out
// directly.  With several splits each CTA writes its unnormalised partial
// (O, m, l) to the workspace and takes a ticket from a per-(sequence, KV head,
// row group) counter; the CTA that draws the last ticket merges all splits by
// log-sum-exp (no CTA waits for another, so there is no spin and no second
// launch).  In cluster mode the C CTAs of (b, h, rg) form a thread-block
// cluster and merge in distributed shared memory instead.  The variant (warps,
// stages), the split size and the cluster size come from the offline table.
//
// HBM-bound: per CTA it streams its keys' D * 2 bytes each of K and as many of
// V, which is the whole algorithmic traffic of decode.  The contraction has only
// G rows (4 for Llama), too few for a tcgen05 tile; the warp MMAs keep the
// arithmetic well below the memory time.

#include <cuda_bf16.h>

#include <atomic>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// Warps per CTA and pipeline depth per warp are template parameters chosen per
// call (from the offline table): a warp keeps kStages - 1 pages in flight while
// it computes one, and the shared memory of a CTA (kStages pages of K and V per
// warp) sets how many CTAs share an SM.  Few long sequences want many warps per
// CTA (few splits, so a short merge); large batches want small CTAs.
constexpr int kPage = 16;
constexpr int kRows = 16;  // MMA M: query-head rows per CTA
constexpr int kMaxCluster = 16;  // CTAs of one (sequence, KV head, row group) in cluster mode

template <int D, int kWarps, int kStages>
struct DecodeTile {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kChunksPerRow = D / 8;                 // 16-byte chunks
    static constexpr int kPageBytes = kPage * kRowBytes;        // K (or V) of one page, one head
    static constexpr int kStageBytes = 2 * kPageBytes;          // K then V
    static constexpr int kWarpBytes = kStages * kStageBytes;
    static constexpr int kPipeBytes = kWarps * kWarpBytes;
    // merge area (over the pipeline, once it is drained): per warp O[16][D + 8]
    // fp32 (the padding makes the fragment stores bank-conflict free) + m[16] + l[16]
    static constexpr int kMS = D + 8;  // row stride of a warp's O
    static constexpr int kMergeWarpFloats = kRows * kMS + 2 * kRows;
    static constexpr int kMergeBytes = kWarps * kMergeWarpFloats * 4;
    static constexpr int kSmemBytes = kPipeBytes > kMergeBytes ? kPipeBytes : kMergeBytes;
    // Cluster mode only, after that: the partials the cluster's CTAs push to
    // this one, O[src][16][cols] (cols = ceil(D / C), so C * cols <= D + C - 1)
    // and (m, l)[src][16].  Separate from the pipeline, which may still be busy
    // when a faster peer pushes.
    static constexpr int kRecvOFloats = kRows * (D + kMaxCluster);
    static constexpr int kRecvBytes = (kRecvOFloats + kMaxCluster * kRows * 2) * 4;
};

// Byte offset of 16-byte chunk c of row r: chunks are XOR-permuted by r % 8.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return r * (D * 2) + ((c ^ (r & 7)) << 4);
}

// Partial-row index of (sequence b, split s, new token i, query head hq).
__device__ __forceinline__ int64_t partial_row(const Args& a, int b, int s, int i, int hq) {
    return ((static_cast<int64_t>(b) * a.splits + s) * a.decode_max_q + i) * a.num_q_heads + hq;
}

// Log-sum-exp merge of the nsplits partials of the CTA's rows (row r = token
// tok[r], query head head[r]) of sequence b (the last step of "Parallel Tiled
// Softmax"): M = max_s m_s, w_s = 2^(m_s - M), out = sum_s w_s O_s / sum_s w_s l_s.
// A split that saw no visible key of a row has m_s = -inf and weight 0.  The
// partials were written by other CTAs, so they are read with L2-coherent loads.
// A work item is (row, 4 columns).  When the CTA has at least two threads per
// item, lanes l and l + 16 of a warp share one item and take the even and the
// odd splits, then combine by a shuffle, so each thread waits for half as many
// loads.  A thread reads the (m, l) and O of kBatch of its splits per batch into
// one of two register buffers, the next batch's loads in flight while the
// current one is combined.
template <int D, int kBatch>
__device__ __forceinline__ void merge_splits(const Args& a, int b, const int* tok, const int* head, int rows,
                                             int nsplits, int q0) {
    const int64_t split_rows = static_cast<int64_t>(a.decode_max_q) * a.num_q_heads;  // rows per split
    const int64_t split_o = split_rows * D;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    constexpr int kGroups = D / 4;  // 4 consecutive columns per work item
    const int total = rows * kGroups;
    const bool two = static_cast<int>(blockDim.x) >= 2 * total;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per_warp = two ? 16 : 32;
    const int part = two ? lane >> 4 : 0;
    const int stride = two ? 2 : 1;
    const int nloc = (nsplits - part + stride - 1) / stride;  // splits part, part + stride, ...
    for (int base = warp * per_warp; base < total; base += (blockDim.x >> 5) * per_warp) {
        const int it = base + (two ? (lane & 15) : lane);
        const bool active = it < total;
        const int r = active ? it / kGroups : 0;
        const int d4 = active ? (it % kGroups) * 4 : 0;
        float M = -INFINITY, den = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (active) {
            const int64_t row = partial_row(a, b, 0, tok[r], head[r]);
            const float2* ml = reinterpret_cast<const float2*>(a.ws_ml) + row;  // (m, l) of split 0
            const float* os = a.ws_o + row * D + d4;
            auto load = [&](int j0, float2 (&mlv)[kBatch], float4 (&ov)[kBatch]) {
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    if (j0 + k < nloc) {
                        const int sp = part + stride * (j0 + k);
                        mlv[k] = __ldcg(ml + sp * split_rows);
                        ov[k] = __ldcg(reinterpret_cast<const float4*>(os + sp * split_o));
                    } else {
                        mlv[k] = make_float2(-INFINITY, 0.f);
                        ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            };
            auto combine = [&](const float2 (&mlv)[kBatch], const float4 (&ov)[kBatch]) {
                float Mn = M;
#pragma unroll
                for (int k = 0; k < kBatch; ++k) Mn = fmaxf(Mn, mlv[k].x);
                const float sc = M == -INFINITY ? 0.f : fast_exp2(M - Mn);  // earlier batches, rebased
                den *= sc;
                acc.x *= sc;
                acc.y *= sc;
                acc.z *= sc;
                acc.w *= sc;
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const float w = mlv[k].x == -INFINITY ? 0.f : fast_exp2(mlv[k].x - Mn);
                    den += w * mlv[k].y;
                    acc.x += w * ov[k].x;
                    acc.y += w * ov[k].y;
                    acc.z += w * ov[k].z;
                    acc.w += w * ov[k].w;
                }
                M = Mn;
            };
            float2 mla[kBatch], mlb[kBatch];
            float4 oa[kBatch], ob[kBatch];
            load(0, mla, oa);
            for (int j0 = 0; j0 < nloc; j0 += 2 * kBatch) {
                const bool second = j0 + kBatch < nloc;
                if (second) load(j0 + kBatch, mlb, ob);
                combine(mla, oa);
                if (j0 + 2 * kBatch < nloc) load(j0 + 2 * kBatch, mla, oa);
                if (second) combine(mlb, ob);
            }
        }
        if (two) {
            // the other half of the splits, from lane ^ 16 (every lane takes part)
            const float Mo = __shfl_xor_sync(0xffffffffu, M, 16);
            const float deno = __shfl_xor_sync(0xffffffffu, den, 16);
            float4 acco;
            acco.x = __shfl_xor_sync(0xffffffffu, acc.x, 16);
            acco.y = __shfl_xor_sync(0xffffffffu, acc.y, 16);
            acco.z = __shfl_xor_sync(0xffffffffu, acc.z, 16);
            acco.w = __shfl_xor_sync(0xffffffffu, acc.w, 16);
            const float Mn = fmaxf(M, Mo);
            const float w = M == -INFINITY ? 0.f : fast_exp2(M - Mn);
            const float wo = Mo == -INFINITY ? 0.f : fast_exp2(Mo - Mn);
            den = w * den + wo * deno;
            acc.x = w * acc.x + wo * acco.x;
            acc.y = w * acc.y + wo * acco.y;
            acc.z = w * acc.z + wo * acco.z;
            acc.w = w * acc.w + wo * acco.w;
        }
        if (active && part == 0) {
            const float inv = 1.f / den;
            uint2 packed;
            packed.x = pack_bf16(acc.x * inv, acc.y * inv);
            packed.y = pack_bf16(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(out + (static_cast<int64_t>(q0 + tok[r]) * a.num_q_heads + head[r]) * D + d4) =
                packed;
        }
    }
}

// A 32-bit global load issued where it is written (the asm is not moved past
// the branches that follow, so independent loads are in flight together).
__device__ __forceinline__ int ldg_s32(const int32_t* p) {
    int v;
    asm volatile("ld.global.nc.s32 %0, [%1];\n" : "=r"(v) : "l"(p));
    return v;
}

// Thread-block cluster helpers: the cluster's CTAs are resident together, so a
// cluster barrier always completes; ld.shared::cluster reads a peer CTA's
// shared memory at the same offset as `local` in this CTA.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// The two halves of a cluster barrier: arrive (relaxed: nothing to publish yet)
// early, wait just before the first access to a peer's shared memory, so that
// every peer has started by then.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory"); }
// Stores v into peer CTA `peer`'s shared memory at the offset of `local` here.
__device__ __forceinline__ void st_peer(float* local, uint32_t peer, float v) {
    uint32_t addr = smem_u32(local), remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(addr), "r"(peer));
    asm volatile("st.shared::cluster.f32 [%0], %1;\n" ::"r"(remote), "f"(v) : "memory");
}
__device__ __forceinline__ void st_peer4(float* local, uint32_t peer, float4 v) {
    uint32_t addr = smem_u32(local), remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(addr), "r"(peer));
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(remote), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_peer2(float* local, uint32_t peer, float x, float y) {
    uint32_t addr = smem_u32(local), remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(addr), "r"(peer));
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};\n" ::"r"(remote), "f"(x), "f"(y) : "memory");
}

// The keys of CTA split s of a sequence of L keys: its npages pages (the CTA's
// k-th page is p0 + pstep * k) hold keys below `end`; npages = 0: none.
__device__ __forceinline__ void split_pages(const Args& a, int s, int L, bool clustered, int& end, int& npages) {
    if (clustered) {
        const int pages_b = (L + kPage - 1) / kPage;
        end = L;
        npages = pages_b > s ? (pages_b - s + a.splits - 1) / a.splits : 0;  // 0: an empty CTA of the cluster
    } else {
        const int start = s * a.kv_chunk;
        end = min(L, start + a.kv_chunk);
        npages = start < L ? (end - start + kPage - 1) / kPage : 0;
    }
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}

// 4-warp CTAs are sized to share an SM three at a time (at most 170 registers),
// except at D = 256, whose O fragments alone take 128 registers a thread.
template <int D, int kWarps, int kStages>
__global__ void __launch_bounds__(kWarps * 32, (kWarps == 4 && D <= 128) ? 3 : 1)
    decode_splitkv_kernel(const Args a) {
    using Tile = DecodeTile<D, kWarps, kStages>;
    extern __shared__ __align__(128) uint8_t smem[];
    // Without early_metadata no memory is accessed before the previous kernel
    // on the stream has completed; with it, the metadata loads, the setup that
    // needs only them and the L2 prefetches come first (see
    // pa_options.early_metadata).
    const bool early = a.early_metadata != 0;
    if (!early) grid_dependency_wait();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;   // MMA group id: row g and g + 8
    const int tq = lane & 3;   // thread in quad: columns 2tq, 2tq + 1

    int64_t idx = blockIdx.x;
    const int s = static_cast<int>(idx % a.splits);
    idx /= a.splits;
    const int rg = static_cast<int>(idx % a.row_groups);
    idx /= a.row_groups;
    const int h = static_cast<int>(idx % a.num_kv_heads);
    const int b = static_cast<int>(idx / a.num_kv_heads);
    // Cluster mode: the a.splits == a.decode_cluster CTAs of (b, h, rg) form one
    // thread-block cluster, take the sequence's pages round-robin (CTA s: pages
    // s, s + C, s + 2C, ...) and merge through distributed shared memory.
    // Otherwise split s covers keys [s * kv_chunk, (s + 1) * kv_chunk) and the
    // splits merge through the workspace.  Either way the CTA's k-th page is
    // p0 + pstep * k, and its warp w takes k = w, w + kWarps, ...
    const bool clustered = a.decode_cluster > 1;
    const int p0 = clustered ? s : s * (a.kv_chunk / kPage);
    const int pstep = clustered ? a.splits : 1;

    // Every exit before the cluster barriers below depends on b alone, so the
    // CTAs of a cluster take it together.  The metadata loads and the first
    // block-table entries (the page set does not depend on the sequence length)
    // are issued together, before anything waits on them.
    const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_pages;
    int bt_cur = 0, bt_nxt = 0;
    {
        const int pe = clustered ? a.max_pages : min(a.max_pages, p0 + a.kv_chunk / kPage);
        const int i0 = p0 + pstep * (warp + kWarps * lane), i1 = i0 + pstep * 32 * kWarps;
        if (i0 < pe) bt_cur = ldg_s32(bt + i0);
        if (i1 < pe) bt_nxt = ldg_s32(bt + i1);
    }
    const int q0 = ldg_s32(a.query_start_loc + b);
    const int q1 = ldg_s32(a.query_start_loc + b + 1);
    int L = ldg_s32(a.seq_lens + b);
    // With early_metadata everything below that needs only the metadata runs
    // before the wait for the previous kernel; whatever writes or reads q or KV
    // waits for it first (wait_prev: a second wait returns at once), and so does
    // every exit, so that the next kernel is only scheduled once this one has
    // passed its wait.
    auto wait_prev = [&]() {
        if (early) grid_dependency_wait();
    };
    const int n = q1 - q0;
    if (n < 1 || n > a.decode_max_q) {  // empty, or the prefill kernel's
        wait_prev();
        return;
    }
    if (q0 < 0 || static_cast<int64_t>(q0) + n > a.num_tokens) {
        wait_prev();
        flag_error(a.err, kDevBadQueryStart);
        return;
    }
    const int cap = a.max_pages * kPage;
    if (L > cap) {
        wait_prev();
        flag_error(a.err, kDevSeqTooLong);
        L = cap;
    }
    // Rows of this CTA: r -> (new token, query head).
    const bool packed = a.row_groups == 1;  // tokens x G heads in one tile
    const int rows = packed ? n * a.group : min(kRows, a.group - rg * kRows);
    auto tok_of = [&](int r) { return packed ? r / a.group : 0; };
    auto head_of = [&](int r) { return packed ? h * a.group + r % a.group : h * a.group + rg * kRows + r; };
    __shared__ int s_tok[kRows], s_head[kRows];
    if (threadIdx.x < kRows) {  // for the merges below; read after later barriers
        s_tok[threadIdx.x] = tok_of(threadIdx.x);
        s_head[threadIdx.x] = head_of(threadIdx.x);
    }
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    if (L < n) {
        // A query must see at least itself; the caller broke the contract.
        wait_prev();
        if (s == 0) {
            flag_error(a.err, kDevQueryTooLong);
            for (int i = threadIdx.x; i < rows * D; i += blockDim.x)
                out[(static_cast<int64_t>(q0 + tok_of(i / D)) * a.num_q_heads + head_of(i / D)) * D + i % D] =
                    __float2bfloat16(0.f);
        }
        return;
    }
    // This CTA's pages (npages of them, page p0 + pstep * k for k < npages) hold
    // keys below `end`.
    int end, npages;
    split_pages(a, s, L, clustered, end, npages);
    if (!clustered && npages == 0) {  // past the end of the sequence
        wait_prev();
        return;
    }
    const int nsplits = clustered ? a.splits : (L + a.kv_chunk - 1) / a.kv_chunk;
    const int my_pages = warp < npages ? (npages - warp + kWarps - 1) / kWarps : 0;
    if (clustered) cluster_arrive_relaxed();  // waited for before the first push to a peer

    // Block-table entries of this warp's pages, 32 at a time in registers (lane l
    // holds the entry of the warp's page 32 * round + l), the next round loaded
    // ahead, so that the copies do not wait on them (the first two rounds were
    // loaded above).
    auto bt_entry = [&](int i) { return i < my_pages ? bt[p0 + pstep * (warp + kWarps * i)] : 0; };

    // Each of this thread's two rows (g, g + 8) has its own causal limit.
    const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* kc = reinterpret_cast<const __nv_bfloat16*>(a.k_cache);
    const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(a.v_cache);
    const bool row_lo = g < rows, row_hi = g + 8 < rows;
    const __nv_bfloat16* qg =
        q + (static_cast<int64_t>(q0 + (row_lo ? tok_of(g) : 0)) * a.num_q_heads + (row_lo ? head_of(g) : 0)) * D;
    const __nv_bfloat16* qg8 =
        q + (static_cast<int64_t>(q0 + (row_hi ? tok_of(g + 8) : 0)) * a.num_q_heads + (row_hi ? head_of(g + 8) : 0)) *
                D;
    const int lim_lo = L - n + (row_lo ? tok_of(g) : 0);      // last key row g may see
    const int lim_hi = L - n + (row_hi ? tok_of(g + 8) : 0);

    const uint32_t wbase = smem_u32(smem) + warp * Tile::kWarpBytes;
    const uint64_t policy = policy_evict_first();

    auto page_of = [&](int it) {  // every lane calls it with the same it
        if (it > 0 && (it & 31) == 0) {
            bt_cur = bt_nxt;
            bt_nxt = bt_entry(it + 32 + lane);
        }
        return __shfl_sync(0xffffffffu, bt_cur, it & 31);
    };
    // Issue the copies of this warp's it-th page into stage it % kStages; always
    // commit a group so that the wait count below stays uniform.
    auto issue = [&](int it) {
        if (it < my_pages) {
            const int lp = p0 + pstep * (warp + kWarps * it);
            const int page = page_of(it);
            const bool ok = static_cast<uint32_t>(page) < static_cast<uint64_t>(a.num_blocks);
            if (!ok) flag_error(a.err, kDevBadBlock);
            const int valid = ok ? min(kPage, end - lp * kPage) : 0;
            const uint32_t st = wbase + (it % kStages) * Tile::kStageBytes;
            const int64_t page_base = static_cast<int64_t>(ok ? page : 0) * kPage;
#pragma unroll
            for (int i = 0; i < Tile::kChunksPerRow / 2; ++i) {
                const int c = lane + 32 * i;
                const int r = c / Tile::kChunksPerRow;
                const int cc = c % Tile::kChunksPerRow;
                const int bytes = r < valid ? 16 : 0;
                const int64_t off = ((page_base + (r < valid ? r : 0)) * a.num_kv_heads + h) * D + cc * 8;
                cp_async_16_stream(st + swz<D>(r, cc), kc + off, bytes, policy);
                cp_async_16_stream(st + Tile::kPageBytes + swz<D>(r, cc), vc + off, bytes, policy);
            }
        }
        cp_async_commit();
    };

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY;  // running max (log2 units) of rows g, g+8
    float l_lo = 0.f, l_hi = 0.f;              // this thread's share of the running sums

    if (early) {
        // While the previous kernel finishes: warm L2 with the K and V rows of
        // this warp's first a.prefetch_pages pages (a prefetch reads nothing
        // into the SM, so a page that kernel writes is still read after it).
        constexpr int kLines = D / 64;  // 128-byte lines per row of one KV head
        for (int k = 0; k < a.prefetch_pages && k < my_pages; ++k) {  // (prefetch_pages <= 64)
            const int page = __shfl_sync(0xffffffffu, k < 32 ? bt_cur : bt_nxt, k & 31);
            const int valid = min(kPage, end - (p0 + pstep * (warp + kWarps * k)) * kPage);
            if (static_cast<uint32_t>(page) < static_cast<uint64_t>(a.num_blocks)) {
                for (int i = lane; i < valid * kLines; i += 32) {
                    const int64_t off =
                        ((static_cast<int64_t>(page) * kPage + i / kLines) * a.num_kv_heads + h) * D + (i % kLines) * 64;
                    prefetch_l2(kc + off);
                    prefetch_l2(vc + off);
                }
            }
        }
        grid_dependency_wait();
    }
    grid_launch_dependents();
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) issue(i);
    // Q fragments for all D/16 k-steps (rows >= `rows` zero), loaded after the
    // first pages' copies are issued: the copies wait for nothing else, and
    // the loads then overlap their latency.
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const int c = ks * 16 + 2 * tq;
        qa[ks][0] = row_lo ? *reinterpret_cast<const uint32_t*>(qg + c) : 0u;
        qa[ks][1] = row_hi ? *reinterpret_cast<const uint32_t*>(qg8 + c) : 0u;
        qa[ks][2] = row_lo ? *reinterpret_cast<const uint32_t*>(qg + c + 8) : 0u;
        qa[ks][3] = row_hi ? *reinterpret_cast<const uint32_t*>(qg8 + c + 8) : 0u;
    }

    for (int it = 0; it < my_pages; ++it) {
        issue(it + kStages - 1);
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const uint32_t sk = wbase + (it % kStages) * Tile::kStageBytes;
        const uint32_t sv = sk + Tile::kPageBytes;
        // S = Q K^T for the page's 16 tokens: two n-tiles of 8 tokens.
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            const int mi = lane >> 3;
            const int tok = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t k0, k1, k2, k3;
                ldmatrix_x4(sk + swz<D>(tok, 2 * ks + (mi & 1)), k0, k1, k2, k3);
                mma_bf16_16816(sc[0], qa[ks], k0, k1);
                mma_bf16_16816(sc[1], qa[ks], k2, k3);
            }
        }
        // Mask keys past the end of the split (only the sequence's last page is
        // partial) and move to log2 units.
        const int tok0 = (p0 + pstep * (warp + kWarps * it)) * kPage;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = tok0 + nt * 8 + 2 * tq + (e & 1);
                sc[nt][e] = (j < end && j <= (e < 2 ? lim_lo : lim_hi)) ? sc[nt][e] * a.scale_log2 : -INFINITY;
            }
        const float mx_lo = quad_max(fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1])));
        const float mx_hi = quad_max(fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3])));
        // The running max only moves when a row's max grows by more than 2^8
        // (log2 units), and only then are O and l rescaled; P <= 2^8 otherwise,
        // and the final O / l is the same.  The four threads of a row hold the
        // same max, so they take the same decision.
        const bool need_lo = mx_lo > m_lo + 8.f, need_hi = mx_hi > m_hi + 8.f;
        if (__any_sync(0xffffffffu, need_lo || need_hi)) {
            const float al_lo = need_lo ? fast_exp2(m_lo - mx_lo) : 1.f;  // 0 when m was -inf
            const float al_hi = need_hi ? fast_exp2(m_hi - mx_hi) : 1.f;
            if (need_lo) m_lo = mx_lo;
            if (need_hi) m_hi = mx_hi;
            l_lo *= al_lo;
            l_hi *= al_hi;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                o[i][0] *= al_lo;
                o[i][1] *= al_lo;
                o[i][2] *= al_hi;
                o[i][3] *= al_hi;
            }
        }
        const float mu_lo = m_lo == -INFINITY ? 0.f : m_lo;
        const float mu_hi = m_hi == -INFINITY ? 0.f : m_hi;

        // P in bf16 as the A operand of P V; the sums use the same rounded P.
        uint32_t pa[4];
        pa[0] = pack_bf16(fast_exp2(sc[0][0] - mu_lo), fast_exp2(sc[0][1] - mu_lo));
        pa[1] = pack_bf16(fast_exp2(sc[0][2] - mu_hi), fast_exp2(sc[0][3] - mu_hi));
        pa[2] = pack_bf16(fast_exp2(sc[1][0] - mu_lo), fast_exp2(sc[1][1] - mu_lo));
        pa[3] = pack_bf16(fast_exp2(sc[1][2] - mu_hi), fast_exp2(sc[1][3] - mu_hi));
        l_lo += (bf16_lo(pa[0]) + bf16_hi(pa[0])) + (bf16_lo(pa[2]) + bf16_hi(pa[2]));
        l_hi += (bf16_lo(pa[1]) + bf16_hi(pa[1])) + (bf16_lo(pa[3]) + bf16_hi(pa[3]));
        // O += P V: V rows are tokens, so the B fragments come from transposed loads.
        {
            const int mi = lane >> 3;
            const int tok = (mi & 1) * 8 + (lane & 7);
#pragma unroll
            for (int nd = 0; nd < D / 16; ++nd) {
                uint32_t v0, v1, v2, v3;
                ldmatrix_x4_trans(sv + swz<D>(tok, 2 * nd + (mi >> 1)), v0, v1, v2, v3);
                mma_bf16_16816(o[2 * nd], pa, v0, v1);
                mma_bf16_16816(o[2 * nd + 1], pa, v2, v3);
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();
    __syncthreads();

    // Merge the warps' partial softmax states in shared memory into this CTA's
    // (O, m, l) for each row r: M = max over the warps of m_w; each warp scales
    // its O_w and l_w by 2^(m_w - M) in registers (one exponential per row and
    // thread); O and l are the sums of the scaled partials.
    constexpr int kMS = Tile::kMS;
    constexpr int kM0 = kRows * kMS;  // m[16], then the scaled l[16], after the O rows
    float* mw = reinterpret_cast<float*>(smem) + warp * Tile::kMergeWarpFloats;
    const float* ms = reinterpret_cast<const float*>(smem);
    l_lo = quad_sum(l_lo);
    l_hi = quad_sum(l_hi);
    if (tq == 0) {
        mw[kM0 + g] = m_lo;
        mw[kM0 + g + 8] = m_hi;
    }
    __syncthreads();
    auto row_max = [&](int r) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ms[w * Tile::kMergeWarpFloats + kM0 + r]);
        return M;
    };
    {
        const float sc_lo = m_lo == -INFINITY ? 0.f : fast_exp2(m_lo - row_max(g));
        const float sc_hi = m_hi == -INFINITY ? 0.f : fast_exp2(m_hi - row_max(g + 8));
        if (row_lo) {
#pragma unroll
            for (int i = 0; i < D / 8; ++i)
                *reinterpret_cast<float2*>(mw + g * kMS + i * 8 + 2 * tq) =
                    make_float2(o[i][0] * sc_lo, o[i][1] * sc_lo);
        }
        if (row_hi) {  // (no lane of the CTA has one when rows <= 8)
#pragma unroll
            for (int i = 0; i < D / 8; ++i)
                *reinterpret_cast<float2*>(mw + (g + 8) * kMS + i * 8 + 2 * tq) =
                    make_float2(o[i][2] * sc_hi, o[i][3] * sc_hi);
        }
        if (tq == 0) {
            mw[kM0 + kRows + g] = l_lo * sc_lo;
            mw[kM0 + kRows + g + 8] = l_hi * sc_hi;
        }
    }
    __syncthreads();
    auto row_sum = [&](int r) {
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) l += ms[w * Tile::kMergeWarpFloats + kM0 + kRows + r];
        return l;
    };
    // Cluster mode: CTA c of the cluster owns columns [c * cols, (c + 1) * cols)
    // and receives every CTA's partial of them.
    const int C = a.splits;
    const int ccols = clustered ? (D + C - 1) / C : D;
    float* recv_o = reinterpret_cast<float*>(smem + Tile::kSmemBytes);  // [src][16][ccols]
    float* recv_ml = recv_o + Tile::kRecvOFloats;                        // [src][16][2]
    if (clustered) cluster_wait();  // every peer has started: its receive area exists
    // One item: row r, columns d .. d + 3.
    for (int i = threadIdx.x; i < rows * (D / 4); i += blockDim.x) {
        const int r = i / (D / 4), d = (i % (D / 4)) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float4 v = *reinterpret_cast<const float4*>(ms + w * Tile::kMergeWarpFloats + r * kMS + d);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const float av[4] = {acc.x, acc.y, acc.z, acc.w};
        if (clustered) {
            if (ccols % 4 == 0) {  // the 4 columns have one owner: one 16-byte push
                const int own = d / ccols;
                st_peer4(recv_o + (s * kRows + r) * ccols + (d - own * ccols), own, acc);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int own = (d + j) / ccols;
                    st_peer(recv_o + (s * kRows + r) * ccols + (d + j - own * ccols), own, av[j]);
                }
            }
            if (d == 0) {
                const float M = row_max(r), l = row_sum(r);
                for (int c = 0; c < C; ++c) st_peer2(recv_ml + (s * kRows + r) * 2, c, M, l);
            }
        } else if (nsplits == 1) {
            const float inv = 1.f / row_sum(r);
            uint2 packed;
            packed.x = pack_bf16(av[0] * inv, av[1] * inv);
            packed.y = pack_bf16(av[2] * inv, av[3] * inv);
            *reinterpret_cast<uint2*>(out + (static_cast<int64_t>(q0 + s_tok[r]) * a.num_q_heads + s_head[r]) * D +
                                      d) = packed;
        } else {
            const int64_t slot = partial_row(a, b, s, s_tok[r], s_head[r]);
            *reinterpret_cast<float4*>(a.ws_o + slot * D + d) = acc;
            if (d == 0) *reinterpret_cast<float2*>(a.ws_ml + slot * 2) = make_float2(row_max(r), row_sum(r));
        }
    }

    if (clustered) {
        // Every CTA of the cluster has pushed its partial of each column block to
        // the block's owner; after the barrier (release / acquire: the pushes are
        // visible) each CTA merges its own columns from its shared memory.  A CTA
        // with no keys pushed m = -inf and weight 0.  Nobody touches a peer's
        // shared memory after the barrier, so a CTA may exit when it is done.
        cluster_sync();
        __shared__ float s_w[kMaxCluster][kRows], s_inv[kRows];
        if (threadIdx.x < rows) {
            // (unrolled over the largest cluster, so that every load is in flight at once)
            const int r = threadIdx.x;
            float2 ml[kMaxCluster];
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c)
                ml[c] = c < C ? *reinterpret_cast<const float2*>(recv_ml + (c * kRows + r) * 2)
                              : make_float2(-INFINITY, 0.f);
            float M = -INFINITY;
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c) M = fmaxf(M, ml[c].x);
            float l = 0.f;
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c) {
                const float w = ml[c].x == -INFINITY ? 0.f : fast_exp2(ml[c].x - M);
                if (c < C) {
                    s_w[c][r] = w;
                    l += w * ml[c].y;
                }
            }
            s_inv[r] = 1.f / l;
        }
        __syncthreads();
        const int d0 = s * ccols;
        const int ncols = max(0, min(ccols, D - d0));
        if (ccols % 4 == 0) {  // (then ncols is a multiple of 4 too)
            const int q4 = ncols / 4;
            for (int i = threadIdx.x; i < rows * q4; i += blockDim.x) {
                const int r = i / q4, j = (i - r * q4) * 4;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c)
                    if (c < C) {
                        const float w = s_w[c][r];
                        const float4 v = *reinterpret_cast<const float4*>(recv_o + (c * kRows + r) * ccols + j);
                        acc.x += w * v.x;
                        acc.y += w * v.y;
                        acc.z += w * v.z;
                        acc.w += w * v.w;
                    }
                const float inv = s_inv[r];
                uint2 packed;
                packed.x = pack_bf16(acc.x * inv, acc.y * inv);
                packed.y = pack_bf16(acc.z * inv, acc.w * inv);
                *reinterpret_cast<uint2*>(out + (static_cast<int64_t>(q0 + s_tok[r]) * a.num_q_heads + s_head[r]) * D +
                                          d0 + j) = packed;
            }
        } else {
            for (int i = threadIdx.x; i < rows * ncols; i += blockDim.x) {
                const int r = i / ncols, j = i % ncols;
                float acc = 0.f;
                for (int c = 0; c < C; ++c) acc += s_w[c][r] * recv_o[(c * kRows + r) * ccols + j];
                out[(static_cast<int64_t>(q0 + s_tok[r]) * a.num_q_heads + s_head[r]) * D + d0 + j] =
                    __float2bfloat16(acc * s_inv[r]);
            }
        }
        return;
    }
    if (nsplits == 1) return;

    // Split merge through the workspace.  Each split CTA publishes its partial,
    // then takes a ticket; the one that draws the last ticket merges every split
    // of (b, h, rg) and resets the counter for the next call.  Nobody waits on
    // anybody.  The ticket is a release-acquire atomic of one thread after a
    // CTA barrier: release is cumulative, so it publishes the whole CTA's
    // partial, and the last CTA's acquire makes every partial visible to it
    // (its barrier passes that on to the other threads).
    __shared__ int s_last;
    __syncthreads();
    int32_t* counter = a.counters + (static_cast<int64_t>(b) * a.num_kv_heads + h) * a.row_groups + rg;
    if (threadIdx.x == 0) {
        int prev;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;\n" : "=r"(prev) : "l"(counter) : "memory");
        s_last = prev == nsplits - 1;
    }
    __syncthreads();
    if (!s_last) return;
    merge_splits<D, 8>(a, b, s_tok, s_head, rows, nsplits, q0);
    if (threadIdx.x == 0) *counter = 0;
}

template <int D, int kWarps, int kStages>
cudaError_t launch_decode_d(const Args& a, cudaStream_t stream) {
    using Tile = DecodeTile<D, kWarps, kStages>;
    auto kernel = decode_splitkv_kernel<D, kWarps, kStages>;
    // The attributes are set once per device.  Host threads may race here; both
    // then set the same values, which is harmless, and the flags are atomic.
    static std::atomic<bool> configured[64];
    static std::atomic<int> sms[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configured[dev & 63].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Tile::kSmemBytes + Tile::kRecvBytes);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        int n = 0;
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        sms[dev & 63].store(n, std::memory_order_relaxed);
        configured[dev & 63].store(true, std::memory_order_release);
    }
    const int64_t ctas = decode_ctas(a);
    if (ctas == 0) return cudaSuccess;
    const size_t smem = Tile::kSmemBytes + (a.decode_cluster > 1 ? Tile::kRecvBytes : 0);
    // programmatic dependent launch for grids of at most one CTA per SM (larger
    // grids would land unevenly on SMs still busy with the previous kernel)
    const bool pdl = ctas <= sms[dev & 63].load(std::memory_order_relaxed);
    // With early_metadata, a grid launched early prefetches about 256 KiB of
    // pages per CTA while the previous kernel finishes (on the 32k-key single
    // stream, 8 warps x 2 stages: 128 KiB 23.8 us a step, 256 KiB 22.8 us,
    // 512 KiB 23.7 us, every page 24.4 us).  A grid launched normally starts
    // at once, so there is nothing to overlap and it prefetches nothing.
    Args la = a;
    constexpr int kPrefetchPages = (256 << 10) / (kWarps * Tile::kStageBytes);
    static_assert(kPrefetchPages >= 1 && kPrefetchPages <= 64, "prefetch depth");
    la.prefetch_pages = (a.early_metadata && pdl) ? kPrefetchPages : 0;
    return launch_kernel(kernel, static_cast<unsigned>(ctas), kWarps * 32, smem, stream, a.decode_cluster, pdl, la);
}

template <int D>
cudaError_t launch_decode_variant(const Args& a, cudaStream_t stream) {
    if constexpr (D == 256) {  // 4-warp CTAs only: 128 KiB (2 stages) or 192 KiB (3) of pages
        switch (a.decode_warps * 16 + a.decode_stages) {
            case 4 * 16 + 2: return launch_decode_d<256, 4, 2>(a, stream);
            case 4 * 16 + 3: return launch_decode_d<256, 4, 3>(a, stream);
            default: return cudaErrorInvalidValue;
        }
    } else {
        switch (a.decode_warps * 16 + a.decode_stages) {
            case 4 * 16 + 2: return launch_decode_d<D, 4, 2>(a, stream);
            case 4 * 16 + 3: return launch_decode_d<D, 4, 3>(a, stream);
            case 4 * 16 + 4: return launch_decode_d<D, 4, 4>(a, stream);
            case 8 * 16 + 2: return launch_decode_d<D, 8, 2>(a, stream);
            case 8 * 16 + 3: return launch_decode_d<D, 8, 3>(a, stream);
            case 12 * 16 + 2: return launch_decode_d<D, 12, 2>(a, stream);
            default: return cudaErrorInvalidValue;
        }
    }
}

}  // namespace

bool decode_variant_supported(int head_dim, int warps, int stages) {
    if (head_dim == 256) return warps == 4 && (stages == 2 || stages == 3);
    return (warps == 4 && stages >= 2 && stages <= 4) || (warps == 8 && (stages == 2 || stages == 3)) ||
           (warps == 12 && stages == 2);
}

int64_t decode_ctas(const Args& a) {
    return static_cast<int64_t>(a.num_seqs) * a.num_kv_heads * a.row_groups * a.splits;
}

cudaError_t launch_decode(const Args& a, cudaStream_t stream) {
    switch (a.head_dim) {
        case 64: return launch_decode_variant<64>(a, stream);
        case 128: return launch_decode_variant<128>(a, stream);
        case 256: return launch_decode_variant<256>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
