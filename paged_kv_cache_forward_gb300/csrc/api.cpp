// api.cpp -- the C ABI of libpagedattn (declared in include/pagedattn.h):
// host-side argument checks, the launch plan (split size from the tuned table),
// the per-(device, stream) workspace cache, and the kernel launches.

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "pa_internal.h"
#include "pagedattn.h"

namespace {

thread_local char g_last_error[512] = "";

pa_status fail(pa_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
pa_status fail(pa_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

pa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ---------------------------------------------------------------- split table
// Keys per split and decode kernel variant, picked from the head dim, the
// context bound (max_pages * page_size) and the number of decode units, as
// measured by the offline sweep (lut_gb300.inc).
struct LutEntry {
    int32_t head_dim;
    int32_t max_bound;  // applies when context bound <= max_bound
    int32_t max_units;  // ... and (sequences x KV heads x row groups) <= max_units
    int32_t kv_chunk;
    int32_t decode_stages;  // 0: the default depth
    int32_t decode_warps;   // 0: the default warps per CTA
    int32_t decode_cluster; // 0 or 1: splits merge through the workspace; else cluster size (= splits)
};
#include "lut_gb300.inc"

constexpr int32_t kDefaultDecodeStages = 2, kDefaultDecodeWarps = 4;
constexpr int32_t kMaxDecodeCluster = 16;  // largest thread-block cluster (non-portable size)

// The key is the head dim, the context bound and the number of independent
// (sequence, KV head, row group) units: the decode grid is units x splits, so a
// shape with the same units and bound needs the same split (an MQA batch of 8
// behaves like one Llama sequence with 8 KV heads).  Every built head dim has
// rows ending in a catch-all; a table without the head dim would fall back to
// its last row.
const LutEntry& table_entry(int32_t head_dim, int64_t bound, int64_t units, int32_t row_groups) {
    if (row_groups > 1)  // more than 16 query heads per KV head: the wide-group cells, if swept
        for (const LutEntry& e : kSplitTableWide)
            if (e.head_dim == head_dim && bound <= e.max_bound && units <= e.max_units) return e;
    for (const LutEntry& e : kSplitTable)
        if (e.head_dim == head_dim && bound <= e.max_bound && units <= e.max_units) return e;
    return kSplitTable[sizeof(kSplitTable) / sizeof(kSplitTable[0]) - 1];
}

// ----------------------------------------------------------------- validation
constexpr int64_t kMaxCtas = 0x7fffffffLL;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

pa_status check_dims(const pa_dims* d) {
    if (!d) return fail(PA_ERR_INVALID_ARG, "dims is NULL");
    if (d->num_tokens < 0 || d->num_seqs < 0) return fail(PA_ERR_INVALID_ARG, "negative num_tokens or num_seqs");
    if (d->num_q_heads <= 0 || d->num_kv_heads <= 0)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads and num_kv_heads must be positive");
    if (d->num_q_heads % d->num_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads (%d) is not a multiple of num_kv_heads (%d)", d->num_q_heads,
                    d->num_kv_heads);
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d not built (64, 128, 256)", d->head_dim);
    if (d->page_size != 16) return fail(PA_ERR_UNSUPPORTED, "page_size %d not built (16)", d->page_size);
    if (d->num_q_heads / d->num_kv_heads > 64)
        return fail(PA_ERR_UNSUPPORTED, "more than 64 query heads per KV head");
    if (d->num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "num_blocks must be positive");
    if (d->max_pages <= 0) return fail(PA_ERR_INVALID_ARG, "max_pages must be positive");
    if (static_cast<int64_t>(d->max_pages) * d->page_size > 0x7fffffffLL)
        return fail(PA_ERR_INVALID_ARG, "max_pages * page_size overflows int32");
    if (d->num_tokens > 0x7fffffffLL) return fail(PA_ERR_UNSUPPORTED, "more than 2^31-1 tokens");
    if (d->num_seqs > 0 && d->num_tokens == 0) return PA_OK;
    return PA_OK;
}

struct Plan {
    int32_t kv_chunk = 0, splits = 0, row_groups = 0;
    int64_t decode_ctas = 0, combine_ctas = 0, prefill_ctas = 0, ws_bytes = 0, counter_bytes = 0;
    int32_t launches = 0;
    pa::Args args{};
};

constexpr int64_t kErrWordBytes = 256;  // the sticky error word lives at the workspace start

pa_status make_plan(const pa_dims* d, const pa_options* o, Plan* p) {
    pa_status st = check_dims(d);
    if (st != PA_OK) return st;
    const int64_t bound = static_cast<int64_t>(d->max_pages) * d->page_size;
    const int32_t group0 = d->num_q_heads / d->num_kv_heads;
    const int32_t rgroups = (group0 + 15) / 16;
    const LutEntry& te =
        table_entry(d->head_dim, bound, static_cast<int64_t>(d->num_seqs) * d->num_kv_heads * rgroups, rgroups);
    int64_t chunk = (o && o->kv_chunk) ? o->kv_chunk : te.kv_chunk;
    if (chunk < d->page_size || chunk % d->page_size)
        return fail(PA_ERR_INVALID_ARG, "kv_chunk %lld must be a positive multiple of page_size",
                    static_cast<long long>(chunk));
    // the table's variant, unless the caller forces one (fully or in part)
    int32_t stages = te.decode_stages ? te.decode_stages : kDefaultDecodeStages;
    int32_t warps = te.decode_warps ? te.decode_warps : kDefaultDecodeWarps;
    if (!pa::decode_variant_supported(d->head_dim, warps, stages)) {
        // (only a table without rows for this head dim gets here)
        warps = kDefaultDecodeWarps;
        stages = kDefaultDecodeStages;
    }
    if (o && (o->decode_stages || o->decode_warps)) {
        stages = o->decode_stages ? o->decode_stages : kDefaultDecodeStages;
        warps = o->decode_warps ? o->decode_warps : kDefaultDecodeWarps;
    }
    if (!pa::decode_variant_supported(d->head_dim, warps, stages))
        return fail(PA_ERR_INVALID_ARG,
                    "decode variant (%d warps, %d stages) is not built for head_dim %d (128 and 64: (4, 2..4), "
                    "(8, 2..3), (12, 2); 256: (4, 2..3))",
                    warps, stages, d->head_dim);
    // cluster mode: the table's, unless the caller forces a split size or a cluster
    int32_t cluster = te.decode_cluster > 1 ? te.decode_cluster : 1;
    // The table's cells give one CTA at most 8192 * 128 / D keys of a sequence
    // (a sequence at the bound must not leave a few CTAs streaming after the
    // rest of the batch is done).  A bound beyond the swept ones can break that
    // for a cluster (bound / C keys per CTA): take static splits of that size.
    const int64_t max_keys = 8192LL * 128 / d->head_dim;
    if (cluster > 1 && !(o && (o->kv_chunk || o->decode_cluster)) && (bound + cluster - 1) / cluster > max_keys) {
        cluster = 1;
        chunk = max_keys;
    }
    if (o && (o->kv_chunk || o->decode_cluster)) cluster = o->decode_cluster > 1 ? o->decode_cluster : 1;
    if (o && o->kv_chunk && o->decode_cluster > 1)
        return fail(PA_ERR_INVALID_ARG, "kv_chunk and decode_cluster > 1 are exclusive (a cluster deals the pages round-robin)");
    if (o && (o->early_metadata < 0 || o->early_metadata > 1))
        return fail(PA_ERR_INVALID_ARG, "early_metadata %d is not 0 or 1", o->early_metadata);
    if (o && (o->launch_only < 0 || o->launch_only > 2))
        return fail(PA_ERR_INVALID_ARG, "launch_only %d is not 0, 1 or 2", o->launch_only);
    if (o && (o->decode_cluster < 0 || o->decode_cluster > kMaxDecodeCluster))
        return fail(PA_ERR_INVALID_ARG, "decode_cluster %d is not in 0..%d", o->decode_cluster, kMaxDecodeCluster);
    if (cluster > 1) {
        // keys per CTA of the longest possible sequence, its pages dealt
        // round-robin to `cluster` CTAs (reported; the kernel needs only the size)
        const int64_t pages = (bound + d->page_size - 1) / d->page_size;
        chunk = (pages + cluster - 1) / cluster * d->page_size;
    }
    if (chunk > bound) chunk = bound;
    const int32_t group = d->num_q_heads / d->num_kv_heads;
    pa::Args& a = p->args;
    a.num_tokens = d->num_tokens;
    a.num_blocks = d->num_blocks;
    a.num_seqs = d->num_seqs;
    a.num_q_heads = d->num_q_heads;
    a.num_kv_heads = d->num_kv_heads;
    a.group = group;
    a.head_dim = d->head_dim;
    a.page_size = d->page_size;
    a.max_pages = d->max_pages;
    a.kv_chunk = static_cast<int32_t>(chunk);
    a.splits = cluster > 1 ? cluster : static_cast<int32_t>((bound + chunk - 1) / chunk);
    a.decode_cluster = cluster;
    a.row_groups = (group + 15) / 16;
    a.decode_max_q = pa::decode_max_q(group);
    a.decode_stages = stages;
    a.decode_warps = warps;
    a.test_stall_prefill = o ? o->test_stall_prefill : 0;
    a.early_metadata = o ? o->early_metadata : 0;
    p->kv_chunk = a.kv_chunk;
    p->splits = a.splits;
    p->row_groups = a.row_groups;
    if (d->num_seqs == 0 || d->num_tokens == 0) {
        p->ws_bytes = 0;
        return PA_OK;
    }
    p->decode_ctas = pa::decode_ctas(a);
    p->combine_ctas = 0;  // the log-sum-exp merge runs inside the decode kernel
    p->prefill_ctas = pa::prefill_ctas(a);
    if (p->decode_ctas > kMaxCtas || p->prefill_ctas > kMaxCtas)
        return fail(PA_ERR_UNSUPPORTED, "launch grid above 2^31-1 CTAs; use a larger kv_chunk");
    p->launches = (p->decode_ctas > 0) + (p->prefill_ctas > 0);
    const int32_t wss = pa::ws_splits(a.splits, a.decode_cluster);
    p->counter_bytes = pa::counter_bytes_needed(d->num_seqs, d->num_kv_heads, a.row_groups, wss);
    p->ws_bytes =
        pa::workspace_layout(d->num_seqs, d->num_q_heads, wss, d->head_dim, a.decode_max_q, p->counter_bytes).bytes;
    return PA_OK;
}

// --------------------------------------------------------- workspace cache
struct Workspace {
    int device;
    cudaStream_t stream;
    void* ptr;
    int64_t bytes;
    int64_t counter_bytes;  // size of the counter area (fixed for the buffer's life)
};

std::mutex g_ws_mutex;
std::vector<Workspace> g_ws;       // live, one per (device, stream)
std::vector<Workspace> g_retired;  // outgrown buffers, kept for captured graphs

// A second stream per (device, stream) on which the prefill kernel of a mixed
// batch runs beside the decode kernel: forked from and joined back into the
// caller's stream by two events, so the call stays stream-ordered and a capture
// records the fork and the join.  The prefill kernel's CTAs then take the SMs
// that the decode kernel's last wave leaves idle.
struct SideStream {
    int device;
    cudaStream_t stream;  // the caller's
    cudaStream_t side;
    cudaEvent_t fork, join;
};
std::vector<SideStream> g_side;

// The side stream of (device, stream) into *out (a copy: the handles stay valid
// until pa_release_workspaces), created if allowed (never while the stream is
// capturing).  False if there is none.
bool get_side(cudaStream_t stream, bool may_create, SideStream* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    for (const SideStream& x : g_side)
        if (x.device == dev && x.stream == stream) {
            *out = x;
            return true;
        }
    if (!may_create) return false;
    SideStream n{dev, stream, nullptr, nullptr, nullptr};
    if (cudaStreamCreateWithFlags(&n.side, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming) != cudaSuccess) {
        if (n.fork) cudaEventDestroy(n.fork);
        cudaStreamDestroy(n.side);
        return false;
    }
    g_side.push_back(n);
    *out = n;
    return true;
}

// Returns the workspace of (device, stream) able to hold a call that needs a
// counter area of `counter_bytes` and `bytes` in all (at that counter size),
// growing it if allowed.  A new buffer is zeroed (error word and split counters
// start at 0) and keeps its counter area size for life, so partials never land
// on counter bytes.  *counter_area receives the buffer's counter area size.
pa_status get_workspace(cudaStream_t stream, int64_t bytes, int64_t counter_bytes, bool may_grow, void** out,
                        int64_t* counter_area) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    Workspace* w = nullptr;
    for (Workspace& x : g_ws)
        if (x.device == dev && x.stream == stream) w = &x;
    if (w && w->counter_bytes >= counter_bytes && w->bytes >= bytes + (w->counter_bytes - counter_bytes)) {
        *out = w->ptr;
        if (counter_area) *counter_area = w->counter_bytes;
        return PA_OK;
    }
    if (!may_grow)
        return fail(PA_ERR_NOT_PREPARED,
                    "workspace of %lld bytes needed while the stream is capturing; call pa_prepare first",
                    static_cast<long long>(bytes));
    // a new buffer: counter area at least as large as before, total at least as large
    const int64_t new_counters = w ? (w->counter_bytes > counter_bytes ? w->counter_bytes : counter_bytes) : counter_bytes;
    int64_t new_bytes = bytes + (new_counters - counter_bytes);
    if (w && w->bytes > new_bytes) new_bytes = w->bytes;
    bytes = new_bytes;
    void* p = nullptr;
    e = cudaMalloc(&p, static_cast<size_t>(bytes));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
    e = cudaMemsetAsync(p, 0, static_cast<size_t>(bytes), stream);
    if (e == cudaSuccess && w) {
        // carry the old sticky error over, then retire the old buffer
        e = cudaMemcpyAsync(p, w->ptr, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream);
    }
    if (e != cudaSuccess) {
        cudaFree(p);
        return cuda_fail(e, "workspace init");
    }
    if (w) {
        g_retired.push_back(*w);
        w->ptr = p;
        w->bytes = bytes;
        w->counter_bytes = new_counters;
    } else {
        g_ws.push_back(Workspace{dev, stream, p, bytes, new_counters});
    }
    *out = p;
    if (counter_area) *counter_area = new_counters;
    return PA_OK;
}

pa_status check_pointers(const void* q, const void* k, const void* v, const int32_t* bt, const int32_t* sl,
                         const int32_t* qsl, const void* out) {
    if (!q || !k || !v || !bt || !sl || !qsl || !out) return fail(PA_ERR_INVALID_ARG, "NULL data pointer");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return fail(PA_ERR_INVALID_ARG, "q, k_cache, v_cache and out must be 16-byte aligned");
    if (!aligned(bt, 4) || !aligned(sl, 4) || !aligned(qsl, 4))
        return fail(PA_ERR_INVALID_ARG, "block_table, seq_lens and query_start_loc must be 4-byte aligned");
    return PA_OK;
}

// Records a caller's timing event.  Inside stream capture the record must be an
// external one, so that replaying the graph records the event again.
pa_status record(void* ev, cudaStream_t s, bool capturing) {
    if (!ev) return PA_OK;
    cudaError_t e = cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), s,
                                             capturing ? cudaEventRecordExternal : cudaEventRecordDefault);
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "cudaEventRecord");
}

}  // namespace

namespace pa {
// Lets other translation units of the library report through pa_last_error().
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

// True if p is device (or managed) memory of the CUDA driver, false for host
// memory, mapped or not.  The prefill kernel reads q with tensor copies and needs
// the former; the decode kernel reads q and the metadata and writes out with
// plain loads and stores, which reach pinned host memory as well.
bool device_resident(const void* p) {
    // (a query, not stream work: allowed inside a capture in any capture mode)
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    cudaPointerAttributes at{};
    const cudaError_t e = cudaPointerGetAttributes(&at, p);
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) {
        cudaGetLastError();  // (the query's error is not sticky; clear it)
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}
}  // namespace pa

extern "C" {

pa_status pa_plan(const pa_dims* dims, const pa_options* opts, pa_plan_info* info) {
    if (!info) return fail(PA_ERR_INVALID_ARG, "info is NULL");
    Plan p;
    pa_status st = make_plan(dims, opts, &p);
    if (st != PA_OK) return st;
    info->kv_chunk = p.kv_chunk;
    info->splits = p.splits;
    info->decode_ctas = p.decode_ctas;
    info->combine_ctas = p.combine_ctas;
    info->prefill_ctas = p.prefill_ctas;
    info->workspace_bytes = p.ws_bytes;
    info->launches = p.launches;
    info->decode_stages = p.args.decode_stages;
    info->decode_warps = p.args.decode_warps;
    info->decode_cluster = p.args.decode_cluster;
    return PA_OK;
}

pa_status pa_prepare(const pa_dims* dims, const pa_options* opts, void* stream) {
    Plan p;
    pa_status st = make_plan(dims, opts, &p);
    if (st != PA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone) return fail(PA_ERR_INVALID_ARG, "pa_prepare called during capture");
    void* ws = nullptr;
    st = get_workspace(s, p.ws_bytes > kErrWordBytes ? p.ws_bytes : kErrWordBytes, p.counter_bytes, true, &ws,
                       nullptr);
    SideStream side;
    if (st == PA_OK && p.decode_ctas > 0 && p.prefill_ctas > 0) get_side(s, true, &side);
    return st;
}

pa_status pa_forward_ex(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                        const int32_t* seq_lens, const int32_t* query_start_loc, void* out, float scale,
                        const pa_dims* dims, const pa_options* opts, void* stream) {
    Plan p;
    pa_status st = make_plan(dims, opts, &p);
    if (st != PA_OK) return st;
    if (dims->num_seqs == 0 || dims->num_tokens == 0) return PA_OK;
    st = check_pointers(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, out);
    if (st != PA_OK) return st;
    if (!(scale == scale)) return fail(PA_ERR_INVALID_ARG, "scale is NaN");
    if (p.prefill_ctas > 0 && !pa::device_resident(q))
        return fail(PA_ERR_INVALID_ARG, "q must be device memory when the dims allow prefill rows");

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    void* ws = nullptr;
    int64_t counter_area = 0;
    st = get_workspace(s, p.ws_bytes, p.counter_bytes, cs == cudaStreamCaptureStatusNone, &ws, &counter_area);
    if (st != PA_OK) return st;

    pa::Args a = p.args;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.query_start_loc = query_start_loc;
    a.out = out;
    a.err = static_cast<int32_t*>(ws);
    a.sched = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + pa::kSchedOffset);
    const pa::WorkspaceLayout wl =
        pa::workspace_layout(a.num_seqs, a.num_q_heads, pa::ws_splits(a.splits, a.decode_cluster), a.head_dim,
                             a.decode_max_q, counter_area);
    a.counters = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + wl.counters_off);
    a.ws_o = reinterpret_cast<float*>(static_cast<char*>(ws) + wl.o_off);
    a.ws_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + wl.ml_off);
    a.scale = scale;
    a.scale_log2 = scale * 1.4426950408889634f;

    const bool capturing = cs != cudaStreamCaptureStatusNone;
    // Both kernels: the prefill one on the side stream, forked after everything
    // before this call on s and joined back before anything after it.  The two
    // kernels touch disjoint rows of out and disjoint workspace words.
    SideStream side{};
    const bool forked = p.decode_ctas > 0 && p.prefill_ctas > 0 && get_side(s, !capturing, &side);
    cudaStream_t ps = s;
    if (forked) {
        if ((e = cudaEventRecord(side.fork, s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(fork)");
        if ((e = cudaStreamWaitEvent(side.side, side.fork, 0)) != cudaSuccess)
            return cuda_fail(e, "cudaStreamWaitEvent(fork)");
        ps = side.side;
    }
    const int32_t only = opts ? opts->launch_only : 0;
    if (only != 2) {
        if ((st = record(opts ? opts->decode_start_event : nullptr, s, capturing)) != PA_OK) return st;
        if ((e = pa::launch_decode(a, s)) != cudaSuccess) return cuda_fail(e, "decode launch");
        if ((st = record(opts ? opts->decode_stop_event : nullptr, s, capturing)) != PA_OK) return st;
    }
    if (only != 1) {
        if ((st = record(opts ? opts->prefill_start_event : nullptr, ps, capturing)) != PA_OK) return st;
        if ((e = pa::launch_prefill(a, ps)) != cudaSuccess) return cuda_fail(e, "prefill launch");
        if ((st = record(opts ? opts->prefill_stop_event : nullptr, ps, capturing)) != PA_OK) return st;
    }
    if (forked) {
        if ((e = cudaEventRecord(side.join, ps)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(join)");
        if ((e = cudaStreamWaitEvent(s, side.join, 0)) != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(join)");
    }
    return PA_OK;
}

pa_status pa_forward(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                     const int32_t* seq_lens, const int32_t* query_start_loc, void* out, float scale,
                     const pa_dims* dims, void* stream) {
    return pa_forward_ex(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, out, scale, dims, nullptr,
                         stream);
}

pa_status pa_cache_write(const void* k_new, const void* v_new, const int64_t* slot_mapping, void* k_cache,
                         void* v_cache, const pa_cache_dims* d, void* stream) {
    if (!d) return fail(PA_ERR_INVALID_ARG, "dims is NULL");
    if (d->num_tokens < 0 || d->num_blocks <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 || d->page_size <= 0)
        return fail(PA_ERR_INVALID_ARG, "cache dims must be positive (num_tokens >= 0)");
    if ((static_cast<int64_t>(d->num_kv_heads) * d->head_dim) % 8)
        return fail(PA_ERR_UNSUPPORTED, "num_kv_heads * head_dim must be a multiple of 8");
    if (d->num_tokens > 0x7fffffffLL) return fail(PA_ERR_UNSUPPORTED, "more than 2^31-1 tokens");
    if (d->num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache)
        return fail(PA_ERR_INVALID_ARG, "NULL data pointer");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return fail(PA_ERR_INVALID_ARG, "k/v tensors must be 16-byte aligned and slot_mapping 8-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    void* ws = nullptr;
    pa_status st = get_workspace(s, kErrWordBytes, 0, cs == cudaStreamCaptureStatusNone, &ws, nullptr);
    if (st != PA_OK) return st;
    e = pa::launch_cache_write(k_new, v_new, slot_mapping, k_cache, v_cache, d->num_tokens, d->num_blocks,
                               d->page_size, d->num_kv_heads, d->head_dim, static_cast<int32_t*>(ws), s);
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "cache write launch");
}

pa_status pa_device_error(void* stream, int32_t* code) {
    if (!code) return fail(PA_ERR_INVALID_ARG, "code is NULL");
    *code = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* ws = nullptr;
    pa_status st = get_workspace(s, kErrWordBytes, 0, true, &ws, nullptr);
    if (st != PA_OK) return st;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int32_t v = 0;
    e = cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read error word");
    if (v) {
        const int32_t zero = 0;
        e = cudaMemcpy(ws, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clear error word");
    }
    *code = v;
    return PA_OK;
}

pa_status pa_release_workspaces(void) {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    int cur = 0;
    cudaGetDevice(&cur);
    pa_status st = PA_OK;
    auto drop = [&](std::vector<Workspace>& v) {
        for (Workspace& w : v) {
            cudaSetDevice(w.device);
            cudaError_t e = cudaFree(w.ptr);
            if (e != cudaSuccess && st == PA_OK) st = cuda_fail(e, "cudaFree(workspace)");
        }
        v.clear();
    };
    drop(g_ws);
    drop(g_retired);
    for (SideStream& x : g_side) {
        cudaSetDevice(x.device);
        cudaEventDestroy(x.fork);
        cudaEventDestroy(x.join);
        cudaStreamDestroy(x.side);
    }
    g_side.clear();
    cudaSetDevice(cur);
    return st;
}

const char* pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported configuration";
        case PA_ERR_NOT_PREPARED: return "workspace not prepared before capture";
        case PA_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

const char* pa_last_error(void) { return g_last_error; }

int32_t pa_version(void) { return 102; }

}  // extern "C"
