// pa_internal.h -- what the C-ABI layer hands to the kernel launchers.
// Not installed; the public interface is include/pagedattn.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace pa {

// Device error codes written to the sticky error word (first one wins).
enum DeviceError : int32_t {
    kDevOk = 0,
    kDevBadBlock = 1,      // a block-table entry outside [0, num_blocks)
    kDevSeqTooLong = 2,    // seq_lens[b] > max_pages * page_size (clamped)
    kDevQueryTooLong = 3,  // query_start_loc gives n_b > seq_lens[b] (rows written as 0)
    kDevWaitTimeout = 4,   // a bounded wait in a kernel gave up
    kDevBadQueryStart = 5, // query_start_loc not within [0, T] or decreasing (rows skipped)
};

struct Args {
    const void* q;        // [T, Hq, D] bf16
    const void* k_cache;  // [NB, P, Hkv, D] bf16
    const void* v_cache;  // [NB, P, Hkv, D] bf16
    const int32_t* block_table;      // [B, max_pages]
    const int32_t* seq_lens;         // [B]
    const int32_t* query_start_loc;  // [B + 1]
    void* out;                       // [T, Hq, D] bf16
    float* ws_o;    // split partials: [B, splits, Hq, D] fp32 (unnormalised O)
    float* ws_ml;   // [B, splits, Hq, 2] fp32: running max (log2 domain) and sum
    int32_t* counters;  // split tickets [B, Hkv, row_groups]; zero between calls
    int32_t* err;   // sticky device error word
    int32_t* sched; // prefill item counters [2] (next item, finished CTAs); zero between calls
    int64_t num_tokens;
    int64_t num_blocks;
    int32_t num_seqs, num_q_heads, num_kv_heads, group, head_dim, page_size, max_pages;
    int32_t kv_chunk;    // tokens per split (multiple of the page size)
    int32_t splits;      // splits in the static decode grid
    int32_t row_groups;  // ceil(group / 16): 16 query-head rows per decode CTA
    int32_t decode_max_q;  // sequences with 1..decode_max_q new tokens take the decode path
    int32_t decode_stages; // cp.async pipeline depth per decode warp (pages)
    int32_t decode_warps;  // warps per decode CTA
    int32_t decode_cluster;  // > 1: the splits of a (sequence, KV head, row group) are one
                             // thread-block cluster of this many CTAs (== splits), merged
                             // through distributed shared memory; 1: merged through ws
    int32_t test_stall_prefill;  // tests only: see pa_options
    int32_t early_metadata;      // decode: metadata loads (and KV prefetch) before the PDL wait
    int32_t prefetch_pages;      // decode, set at launch: pages per warp prefetched before that wait
    float scale;         // softmax scale
    float scale_log2;    // scale * log2(e)
};

cudaError_t launch_decode(const Args& a, cudaStream_t stream);
cudaError_t launch_prefill(const Args& a, cudaStream_t stream);
cudaError_t launch_cache_write(const void* k_new, const void* v_new, const int64_t* slot_mapping, void* k_cache,
                               void* v_cache, int64_t num_tokens, int64_t num_blocks, int32_t page_size,
                               int32_t num_kv_heads, int32_t head_dim, int32_t* err, cudaStream_t stream);

// New tokens a sequence may have and still take the decode path: its query rows
// (tokens x the G heads of a KV head) must fit one 16-row MMA tile.  With more
// than 16 heads per KV head the decode path takes single-token queries only.
inline int32_t decode_max_q(int32_t group) { return group <= 16 ? 16 / group : 1; }

// Splits whose partials go through the workspace (none in cluster mode).
inline int32_t ws_splits(int32_t splits, int32_t decode_cluster) { return decode_cluster > 1 ? 1 : splits; }

// Byte offset, in the workspace header, of the prefill kernel's two item
// counters (zero before and after every call: the last CTA resets them).
constexpr int64_t kSchedOffset = 128;

// Workspace layout shared by pa_forward and pa_forward_noalloc: a 256-byte
// header (sticky error word at 0, prefill item counters at kSchedOffset), an
// area of split ticket counters (zero before and
// after every call: the last CTA of each ticket resets it), then the partials O
// and (m, l) of [B, splits, decode_max_q, Hq] rows.  The counter area never
// overlaps bytes that held partials: its size is a property of the buffer
// (counter_area_bytes, at least what the call needs), not of the call.
struct WorkspaceLayout {
    int64_t counters_off, counter_bytes, o_off, ml_off, bytes;
};
inline int64_t counter_bytes_needed(int64_t num_seqs, int32_t num_kv_heads, int32_t row_groups, int32_t splits) {
    const int64_t counters = splits > 1 ? num_seqs * num_kv_heads * row_groups : 0;
    return ((counters * 4 + 255) / 256) * 256;
}
inline WorkspaceLayout workspace_layout(int64_t num_seqs, int32_t num_q_heads, int32_t splits, int32_t head_dim,
                                        int32_t decode_max_q, int64_t counter_area_bytes) {
    WorkspaceLayout w{};
    const int64_t rows = splits > 1 ? num_seqs * splits * decode_max_q * num_q_heads : 0;
    w.counters_off = 256;
    w.counter_bytes = counter_area_bytes;
    w.o_off = w.counters_off + counter_area_bytes;
    w.ml_off = w.o_off + rows * head_dim * 4;
    w.bytes = w.ml_off + rows * 2 * 4;
    return w;
}

// Launches a kernel of this library, as 1-D thread-block clusters of `cluster`
// CTAs if cluster > 1.  With `pdl`, the launch allows programmatic dependent
// launch: the grid may be scheduled while the previous kernel on the stream is
// still finishing (once all of that kernel's CTAs have started and signalled),
// and the kernel's griddepcontrol.wait, before its first memory access, holds
// it until that kernel has completed and its writes are visible.  That hides
// the launch latency of back-to-back calls and changes no result.  Used only
// for grids that fit on the GPU in one wave, whose CTAs then land one per SM.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                          cudaStream_t stream, int cluster, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Programmatic dependent launch, device side.  grid_dependency_wait returns
// once the previous kernel on the stream has completed and its writes are
// visible (at once when the kernel was not launched with pdl).
// grid_launch_dependents lets the next kernel on the stream be scheduled; a
// kernel calls it only after its own wait, so that a kernel scheduled early
// runs beside its immediate predecessor alone, never beside an older one.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Sets the calling thread's pa_last_error() text.
void set_last_error(const char* msg);

// (warps per CTA, pipeline depth) pairs the decode kernel is built for:
// (4, 2..4), (8, 2..3), (12, 2); at head_dim 256 only (4, 2..3).
bool decode_variant_supported(int head_dim, int warps, int stages);

// Static grid sizes (functions of shapes only), shared with the planner; for
// the persistent prefill kernel, its work items (the grid is min(items, SMs)).
int64_t decode_ctas(const Args& a);
int64_t prefill_ctas(const Args& a);

}  // namespace pa
