// noalloc.cu -- pa_forward_noalloc: the forward pass with no memory allocation.
//
// pa_forward keeps its split-KV scratch in a buffer it allocates (cudaMalloc)
// on first use.  Some callers cannot let a library allocate: hosts whose device
// memory is entirely owned by their own allocator or budgeted up front
// (inference servers that give all free memory to their KV-cache pool, plugins
// inside another framework's memory manager), and latency-critical loops where
// an allocation's cost or failure at an arbitrary call is not acceptable.  This
// entry point uses instead a fixed scratch array that is part of the library's
// device image: a GPU holds it from the time the library's code is loaded there
// (at the latest, this entry point's first call on it) until the process exits,
// and no call allocates or frees anything.
//
// Limits and rules:
//  * The scratch holds kNoAllocScratchBytes (32 MiB).  A call whose split
//    partials do not fit (pa_plan(...).workspace_bytes larger than that) is
//    rejected with PA_ERR_UNSUPPORTED before anything is launched.
//  * All calls on a device share the one array and it keeps the last call's
//    contents.  Calls that overlap on the GPU (on different streams without
//    ordering between them) race on it; order them on one stream.
//  * The first call on a device looks up the array's device address with that
//    device current (cudaGetSymbolAddress) and caches it for the process; make
//    that first call before any stream capture, and do not reset the device
//    afterwards (the cached address would be stale).
//  * The sticky error word is the caller's device int32 if one is given (the
//    caller clears it), else a slot in the scratch that each call clears and
//    nothing reads back.
//  * Host threads may call it concurrently (the set-up is under a mutex).

#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "pa_internal.h"
#include "pagedattn.h"

namespace pa {
// (api.cpp) True if p is device or managed memory, false for host memory.
bool device_resident(const void* p);
}  // namespace pa

namespace {

constexpr int64_t kNoAllocScratchBytes = 32ll << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

pa_status report(pa_status st, const char* msg) {
    pa::set_last_error(msg);
    return st;
}

// Device address of the scratch array on the current device (set up once).
pa_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return report(PA_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices) return report(PA_ERR_UNSUPPORTED, "device ordinal above 63");
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
            return report(PA_ERR_CUDA, msg);
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" pa_status pa_forward_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        const int32_t* query_start_loc, void* out, float scale, const pa_dims* dims,
                                        int32_t* device_error, void* stream) {
    pa_plan_info info{};
    pa_status st = pa_plan(dims, nullptr, &info);  // validates dims, sets the error text on failure
    if (st != PA_OK) return st;
    if (dims->num_seqs == 0 || dims->num_tokens == 0) return PA_OK;
    if (info.workspace_bytes > kNoAllocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "pa_forward_noalloc: these shapes need %lld bytes of scratch; the fixed scratch holds %lld "
                 "(use pa_forward, or fewer sequences / a shorter max_pages)",
                 static_cast<long long>(info.workspace_bytes), static_cast<long long>(kNoAllocScratchBytes));
        return report(PA_ERR_UNSUPPORTED, msg);
    }
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !query_start_loc || !out)
        return report(PA_ERR_INVALID_ARG, "NULL data pointer");
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return report(PA_ERR_INVALID_ARG, "q, k_cache, v_cache and out must be 16-byte aligned");
    if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(query_start_loc, 4) ||
        !aligned(device_error, 4))
        return report(PA_ERR_INVALID_ARG, "int32 arguments must be 4-byte aligned");
    if (!(scale == scale)) return report(PA_ERR_INVALID_ARG, "scale is NaN");
    if (info.prefill_ctas > 0 && !pa::device_resident(q))
        return report(PA_ERR_INVALID_ARG, "q must be device memory when the dims allow prefill rows");

    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != PA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    pa::Args a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.query_start_loc = query_start_loc;
    a.out = out;
    a.num_tokens = dims->num_tokens;
    a.num_blocks = dims->num_blocks;
    a.num_seqs = dims->num_seqs;
    a.num_q_heads = dims->num_q_heads;
    a.num_kv_heads = dims->num_kv_heads;
    a.group = dims->num_q_heads / dims->num_kv_heads;
    a.head_dim = dims->head_dim;
    a.page_size = dims->page_size;
    a.max_pages = dims->max_pages;
    a.kv_chunk = info.kv_chunk;
    a.splits = info.splits;
    a.row_groups = (a.group + 15) / 16;
    a.decode_max_q = pa::decode_max_q(a.group);
    a.decode_stages = info.decode_stages;
    a.decode_warps = info.decode_warps;
    a.decode_cluster = info.decode_cluster > 1 ? info.decode_cluster : 1;
    a.scale = scale;
    a.scale_log2 = scale * 1.4426950408889634f;
    const pa::WorkspaceLayout wl =
        pa::workspace_layout(a.num_seqs, a.num_q_heads, pa::ws_splits(a.splits, a.decode_cluster), a.head_dim,
                             a.decode_max_q,
                             pa::counter_bytes_needed(a.num_seqs, a.num_kv_heads, a.row_groups,
                                                      pa::ws_splits(a.splits, a.decode_cluster)));
    unsigned char* const sb = static_cast<unsigned char*>(scratch);
    a.counters = reinterpret_cast<int32_t*>(sb + wl.counters_off);
    a.ws_o = reinterpret_cast<float*>(sb + wl.o_off);
    a.ws_ml = reinterpret_cast<float*>(sb + wl.ml_off);
    a.err = device_error ? device_error : static_cast<int32_t*>(scratch);
    a.sched = reinterpret_cast<int32_t*>(sb + pa::kSchedOffset);
    // The error word (unless the caller's), the prefill item counters and the
    // split ticket counters must start at zero: clear them in one memset (a
    // completed call leaves the counters zero, but the array is shared and the
    // last call may not have completed normally).  The partials are written
    // before they are read within one call, so they need no clearing.
    {
        const int64_t lo = device_error ? pa::kSchedOffset : 0;
        cudaError_t e = cudaMemsetAsync(sb + lo, 0, static_cast<size_t>(wl.o_off - lo), s);
        if (e != cudaSuccess) return report(PA_ERR_CUDA, "cudaMemsetAsync(error word and counters) failed");
    }
    cudaError_t e = pa::launch_decode(a, s);
    if (e == cudaSuccess) e = pa::launch_prefill(a, s);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "pa_forward_noalloc launch: %s", cudaGetErrorString(e));
        return report(PA_ERR_CUDA, msg);
    }
    return PA_OK;
}
