/*
 * pagedattn.h -- C ABI of libpagedattn, a unified paged-attention forward pass
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation.  For every sequence b of a batch and every new query token i
 * of it, and every query head h:
 *
 *     out[t, h, :] = softmax_j( scale * <q[t, h, :], K_b[j, h / G, :]> ) . V_b[j, h / G, :]
 *
 * over the keys j = 0 .. p that the token may see, where t = query_start_loc[b] + i,
 * p = seq_lens[b] - n_b + i (the n_b new tokens are the last n_b positions of
 * the sequence, so the causal mask is bottom-right aligned) and G = Hq / Hkv.
 * This is scaled dot-product attention as defined on the GPU programming guide
 * page ("From megabytes to megawatts: a full guide to high-performance LLM and
 * diffusion kernels with CUDA and Triton", section "Decomposing multi-head
 * attention (MHA)"), masked causally as in its section "Flash Attention in
 * Triton" (future tokens get -inf).  K_b and V_b are read through the block table
 * from a paged KV cache, and query heads that share a KV head are computed
 * together (Q-Block), as the Triton unified-attention page describes ("One line
 * of Triton code beats both NVIDIA and AMD ...", papers.ananclaw.com, section
 * "What three things the IBM paper got right", second item, the five-step list).
 * Decode (n_b = 1) and chunked-prefill (n_b > 1) sequences may be mixed in one
 * call.  Long key ranges are split across SMs and the partial results merged by
 * log-sum-exp ("Parallel Tiled Softmax", same list), using the online-softmax
 * recurrence of the guide's section "The Flash Attention revolution".
 *
 * Layouts (all row-major and contiguous; element counts, not bytes):
 *   q               [T, Hq, D]        bf16    T = query_start_loc[B]
 *   k_cache,v_cache [NB, P, Hkv, D]   bf16    token-major pages: the D values of
 *                                             one token of one KV head are
 *                                             contiguous
 *   block_table     [B, max_pages]    int32   logical page -> physical page
 *   seq_lens        [B]               int32   L_b: cached prefix + new tokens
 *   query_start_loc [B + 1]           int32   0 = qsl[0] <= qsl[1] <= ... = T
 *   out             [T, Hq, D]        bf16    written for every query row
 * Logical position j of sequence b is slot j % P of physical page
 * block_table[b][j / P].  Entries of block_table past a sequence's last page may
 * be loaded but are never used: they need not be valid block ids.
 *
 * Pointers.  Every data pointer is a DEVICE pointer on the current CUDA device
 * (the one the stream belongs to).  q, k_cache, v_cache and out must be 16-byte
 * aligned; the int32 arrays 4-byte aligned.  The caller owns all of them; the
 * library keeps none after a call returns.  One exception: when the dims allow
 * no prefill rows (pa_plan_info.prefill_ctas == 0), q, block_table, seq_lens,
 * query_start_loc and out may be pinned host memory that the device can address
 * (cudaHostAlloc / cudaHostRegister under unified addressing; a PyTorch
 * pin_memory tensor), because the decode kernel reads them and writes out with
 * plain loads and stores, which then cross the host link (NVLink-C2C on a
 * Grace-Blackwell node): a decode step with host inputs and outputs needs no
 * copies.  k_cache and v_cache are always device memory.  When the dims allow
 * prefill rows, q must be device (or managed) memory, since the prefill kernel
 * reads it with tensor copies; pa_forward and pa_forward_noalloc check this
 * (one pointer query, made only then) and return PA_ERR_INVALID_ARG otherwise.
 *
 * Streams and graphs.  Every call is asynchronous on the given stream
 * (a cudaStream_t passed as void*; NULL is the legacy default stream).  No call
 * of pa_forward reads device memory on the host or synchronises, and its launch
 * grids depend only on the pa_dims, so it can be captured in a CUDA graph and
 * replayed with new contents of the same buffers (the "static launch grid" and
 * "CUDA / HIP Graphs" items of the same five-step list).  When the dims allow
 * both decode and prefill rows, the prefill kernel runs on a second stream the
 * library keeps per (device, stream), forked from the given stream by an event
 * and joined back by another before the call returns: work enqueued on the
 * stream before the call happens before both kernels, work enqueued after it
 * after both, and a capture records the fork and the join (pa_prepare creates
 * that stream; a call captured without it launches both kernels on the given
 * stream, one after the other).  A decode grid of at most one CTA per SM is
 * launched with programmatic dependent launch: its CTAs may be scheduled while
 * the previous kernel on the stream finishes, but they wait for that kernel to
 * complete (griddepcontrol.wait) before any memory access, so the ordering
 * above holds.  Only after that wait does the decode kernel let the next kernel
 * on the stream be scheduled early, so a kernel that starts early never runs
 * beside anything but the one kernel immediately before it.  The one exception
 * is opt-in: with pa_options.early_metadata the decode kernel reads the
 * metadata (and prefetches its first KV pages into L2) before that wait.
 *
 * Scratch memory.  Splitting a long key range needs a workspace of
 * pa_plan(...).workspace_bytes bytes, which the library allocates and caches per
 * (device, stream).  It grows on demand outside graph capture; inside capture it
 * cannot, so call pa_prepare with the largest dims first.  Buffers are kept until
 * pa_release_workspaces, so graphs that captured them stay valid.
 *
 * Errors.  Functions return a pa_status and never abort or throw.  Argument
 * checks are done on the host before any launch; on failure nothing is
 * launched and pa_last_error() (per thread) says why.  Values that live on the
 * device (block ids, lengths) are the caller's contract; the kernels check them
 * anyway, never access memory outside the buffers because of them, and record
 * the first violation in a sticky per-stream error word (pa_device_error).
 */
#ifndef PAGEDATTN_H_
#define PAGEDATTN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* bad pointer, shape, alignment or option      */
    PA_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim, page size ...  */
    PA_ERR_NOT_PREPARED = 3,  /* workspace too small while the stream captures */
    PA_ERR_CUDA = 4,          /* a CUDA runtime call failed (see pa_last_error) */
} pa_status;

/* Shapes of one call.  head_dim must be 64, 128 or 256 and page_size 16; any
 * num_q_heads that is a multiple of num_kv_heads, at most 64 times it, is
 * accepted. */
typedef struct {
    int64_t num_tokens;    /* T: rows of q and out (= query_start_loc[B])        */
    int64_t num_blocks;    /* NB: pages in each of k_cache and v_cache           */
    int32_t num_seqs;      /* B                                                  */
    int32_t num_q_heads;   /* Hq                                                 */
    int32_t num_kv_heads;  /* Hkv                                                */
    int32_t head_dim;      /* D                                                  */
    int32_t page_size;     /* P                                                  */
    int32_t max_pages;     /* row length of block_table; max_pages * P bounds L_b */
} pa_dims;

/* Optional knobs, for tests and the offline sweep.  Zero-initialise. */
typedef struct {
    int32_t kv_chunk;  /* 0: from the tuned table; else keys per split (multiple
                          of page_size); a chunk >= max_pages * P means no split */
    int32_t decode_stages;  /* decode kernel variant: pipeline depth in pages per  */
    int32_t decode_warps;   /* warp, and warps per CTA.  Both 0: from the tuned
                               table; either set: that variant, the other field
                               defaulting to 2 stages / 4 warps.  Built variants
                               (warps, stages): (4, 2..4), (8, 2..3), (12, 2);
                               others are PA_ERR_INVALID_ARG.  Deeper pipelines
                               and more warps keep more bytes in flight per CTA
                               but fit fewer CTAs on an SM. */
    int32_t decode_cluster; /* 0: from the tuned table (unless kv_chunk is set);
                               1: splits of kv_chunk keys merged through the
                               workspace; 2..16: the pages of each (sequence, KV
                               head) are dealt round-robin to a thread-block
                               cluster of this many CTAs, merged in distributed
                               shared memory (kv_chunk must then be 0). */
    /* cudaEvent_t handles recorded on the stream immediately before and after
       the decode kernel and the prefill kernel (NULL: not recorded). */
    void* decode_start_event;
    void* decode_stop_event;
    void* prefill_start_event;
    void* prefill_stop_event;
    /* Tests only: nonzero makes the prefill kernel's first CTA withhold the K
       tile of its first work item, so that the wait for it runs out (after
       2 s) and the kernel takes its abort path: device error 4, the other
       roles stop, issued MMAs drain, TMEM is freed.  No memory is touched that
       a normal call would not touch; outputs of that CTA's item are left as
       they were. */
    int32_t test_stall_prefill;
    /* Timing and tests: 0 launches every kernel the batch needs; 1 only the
       decode kernel, 2 only the prefill kernel (rows of the other kind are then
       not written).  Other values are PA_ERR_INVALID_ARG. */
    int32_t launch_only;
    /* 1: the caller guarantees that block_table, seq_lens and query_start_loc
       are not written by the kernel immediately before this call on the stream
       (as in the attention layers of one decode step, which share the
       metadata).  Work enqueued before that kernel, host copies included, is
       finished by then if that kernel lets its successor be scheduled only
       after its own wait for its predecessor, as this library's kernels do; a
       kernel that does not use programmatic dependent launch lets it be
       scheduled only when it completes.  A decode kernel launched with programmatic
       dependent launch (see "Streams and graphs") then loads its metadata and
       block-table entries, and prefetches the first KV pages of each warp into
       L2, while that kernel is still finishing; q, the KV values it computes
       with, and every write still wait for it.  A prefetch only warms L2, so a
       KV page that kernel writes is still read after the write.  Breaking the
       guarantee gives wrong rows (a stale length or page id), never an access
       outside the buffers: page ids and lengths are bounds-checked as always.
       0: every access waits (the default).  Other values are
       PA_ERR_INVALID_ARG. */
    int32_t early_metadata;
} pa_options;

/* What a call with these dims launches (host-only; no device work). */
typedef struct {
    int32_t kv_chunk;         /* keys per split                                */
    int32_t splits;           /* splits of the longest possible sequence       */
    int64_t decode_ctas;      /* decode kernel grid                            */
    int64_t combine_ctas;     /* 0: the log-sum-exp merge of the splits runs in
                                 the decode kernel (last split CTA to finish) */
    int64_t prefill_ctas;     /* prefill work items (tile pairs x KV heads); its
                                 persistent kernel runs min(this, SMs) CTAs    */
    int64_t workspace_bytes;  /* scratch this call needs                       */
    int32_t launches;         /* kernels launched per pa_forward               */
    int32_t decode_stages;    /* decode pipeline depth (pages per warp)        */
    int32_t decode_warps;     /* warps per decode CTA                          */
    int32_t decode_cluster;   /* 1, or the CTAs per cluster (= splits)         */
} pa_plan_info;

/*
 * The forward pass.  Computes out for every query row of the batch (see the top
 * of this file).  scale multiplies the dot products (typically 1/sqrt(D)).
 * Returns PA_OK after enqueuing the kernels on stream; PA_ERR_* otherwise,
 * without launching anything.  Zero sequences or zero tokens is a no-op.
 */
pa_status pa_forward(const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_table, const int32_t* seq_lens,
                     const int32_t* query_start_loc, void* out, float scale,
                     const pa_dims* dims, void* stream);

/* pa_forward with options (opts may be NULL). */
pa_status pa_forward_ex(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_table, const int32_t* seq_lens,
                        const int32_t* query_start_loc, void* out, float scale,
                        const pa_dims* dims, const pa_options* opts, void* stream);

/* Fills *info with the launch plan for dims (host only).  The split size and the
 * decode kernel variant (warps, pipeline depth, cluster size) come from the
 * table an offline sweep produced, keyed on the context bound
 * (max_pages * page_size) and the decode units (sequences x KV heads x row
 * groups of 16 query heads): the "offline micro-benchmarks -> decision tree" of
 * the same page's third section, with no tuning at run time. */
pa_status pa_plan(const pa_dims* dims, const pa_options* opts, pa_plan_info* info);

/* Allocates (outside any capture) the workspace a pa_forward with these dims and
 * options needs on stream, and the side stream and events of a call with both
 * kernels, so that the call can then be captured. */
pa_status pa_prepare(const pa_dims* dims, const pa_options* opts, void* stream);

/* Synchronises stream, then returns the stream's sticky device error code in
 * *code (0 = none; 1 bad block id; 2 seq_len above max_pages * page_size;
 * 3 more new tokens than seq_len; 4 a bounded wait gave up; 5 query_start_loc
 * outside [0, num_tokens]) and clears it.  Rows the check skipped are not written. */
pa_status pa_device_error(void* stream, int32_t* code);

/* Frees every cached workspace on every device, and the side streams and
 * events.  No graph that captured a pa_forward may be replayed afterwards. */
pa_status pa_release_workspaces(void);

/* Static text for a status, and this thread's last error detail. */
const char* pa_status_string(pa_status status);
const char* pa_last_error(void);

/*
 * pa_forward without any allocation.  The pages this library follows have no
 * counterpart of this call.  It serves callers that cannot let a library
 * allocate device memory: hosts whose device memory is owned or budgeted up
 * front by their own allocator (an inference server that hands all free memory
 * to its KV-cache pool, a plugin living inside another framework's memory
 * manager), and latency-critical loops where an allocation's cost, or its
 * failure at an arbitrary call, is not acceptable.
 *
 * Same arguments and result as pa_forward (the same kernels with the same
 * launch plan, so the same output bits), plus device_error: a device int32
 * that receives the first device-side error code (as pa_device_error reports
 * them; the caller zeroes it), or NULL to discard the codes.  The split-KV
 * scratch is a fixed 32 MiB array in the library's device image instead of an
 * allocation; a GPU holds it from the time the library's code is loaded there
 * (at the latest this call's first use) until the process exits.  Shapes whose
 * pa_plan(...).workspace_bytes exceed 32 MiB are rejected with
 * PA_ERR_UNSUPPORTED before any launch.  Every call on a device shares that one
 * array, which keeps the last call's contents (each call clears the counters it
 * needs at zero, with a memset on the stream): calls that overlap on the GPU
 * (unordered streams) race, so order them on one stream.  Both kernels run on
 * the given stream, one after the other.  The first call on each device looks
 * up the array's device address with that device current (cudaGetSymbolAddress)
 * and keeps it for the life of the process; make that first call before any
 * stream capture, and do not reset the device (cudaDeviceReset) after it.  It
 * calls no cudaMalloc, cudaFree or allocating routine, and may be called from
 * several host threads.
 */
pa_status pa_forward_noalloc(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_table, const int32_t* seq_lens,
                             const int32_t* query_start_loc, void* out, float scale,
                             const pa_dims* dims, int32_t* device_error, void* stream);

/* Shapes of a paged KV-cache write. */
typedef struct {
    int64_t num_tokens;    /* T: rows of k_new, v_new and slot_mapping           */
    int64_t num_blocks;    /* NB: pages in each of k_cache and v_cache           */
    int32_t num_kv_heads;  /* Hkv                                                */
    int32_t head_dim;      /* D (Hkv * D must be a multiple of 8)                */
    int32_t page_size;     /* P                                                  */
    int32_t reserved;
} pa_cache_dims;

/*
 * Paged KV-cache write: the step that brings the new tokens' K and V into the
 * paged KV cache (the Triton unified-attention page, section "Why is switching
 * the card so hard": paged KV cache) before pa_forward reads them through the
 * block table.  For every token t with s = slot_mapping[t] >= 0, k_new[t] and
 * v_new[t] are copied to page s / P, slot s % P of k_cache and v_cache; a
 * negative slot is padding and writes nothing.
 *   k_new, v_new     [T, Hkv, D]      bf16, device, 16-byte aligned
 *   slot_mapping     [T]              int64, device, 8-byte aligned
 *   k_cache, v_cache [NB, P, Hkv, D]  bf16, device, 16-byte aligned (written)
 * Two tokens with the same slot race (the caller's contract).  A slot at or past
 * NB * P is not written and sets device error 1 (see pa_device_error).  Stream
 * ordered and graph-capturable (its error word lives in the stream's workspace,
 * so call pa_prepare, or any pa_forward, on the stream before capturing).
 */
pa_status pa_cache_write(const void* k_new, const void* v_new, const int64_t* slot_mapping, void* k_cache,
                         void* v_cache, const pa_cache_dims* dims, void* stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H_ */
