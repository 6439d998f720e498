/*
 * rpa.h -- C ABI of the GB300 ragged paged attention library (librpa.so).
 *
 * Ragged paged attention is the mixed prefill/decode grouped-query attention
 * of a serving engine, as defined by the "ragged_paged.zig" page (Cfg, run,
 * flashAttention):
 *
 *   queries of many sequences are packed raggedly into q[num_q_tokens, Hq, D];
 *   sequence s owns tokens [cu_q_lens[s], cu_q_lens[s+1]) and kv_lens[s] keys;
 *   its keys live in fixed-size pages of kv_pages[total_num_pages, page_size,
 *   2*Hkv, D] (combined head 2h = K of kv head h, 2h+1 = V of kv head h),
 *   logical page j of s being physical page page_indices[s, j].
 *
 *   Query token i of s sits at key position p = kv_len - q_len + i.  Query head
 *   qh reads kv head qh / (Hq/Hkv).  The logit of key j is
 *   sm_scale * <q, k_scale*K_j>, soft-capped as cap*tanh(x/cap) when a cap is
 *   set (before masking); key j is masked when j >= kv_len, when causal and
 *   j > p, or when p - sliding_window >= j.  The output is the softmax-weighted
 *   sum of v_scale*V_j, cast to the q dtype.
 *
 * Conventions for every entry point:
 *  - All functions return an RpaStatus code (0 = RPA_OK); no C++ exception
 *    crosses this boundary and no function aborts the process.
 *  - "device" pointers are CUDA global memory of the device that was current
 *    at rpa_create; "host" pointers are ordinary (ideally pinned) host memory.
 *  - The caller owns every tensor.  The handle owns only its workspace.
 *  - Work is enqueued on the given stream (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream) and is asynchronous unless stated.
 */
#ifndef RPA_H_
#define RPA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types ("ragged_paged.zig", Cfg.q_dtype / Cfg.kv_dtype).
 *   q (and o, which has q's type): bf16, f16 or f32.
 *   K/V: bf16, f16, fp8 e4m3fn, fp8 e5m2 or int8 (two's complement); the 8-bit
 *        types are usually paired with k_scale / v_scale.
 * The tensor cores take both operands of a product in one type: bf16 with bf16
 * K/V, f16 with every other K/V type.  K/V values convert exactly; q values
 * of another type are rounded to that type to nearest even (f32 q; f16 q with
 * bf16 K/V; bf16 q with f16 or 8-bit K/V), which the tolerance of the results
 * covers.  The page's other K/V types (f32, i32, i16) are not supported
 * (RPA_ERR_UNSUPPORTED). */
typedef enum RpaDtype {
    RPA_DT_BF16 = 0,
    RPA_DT_FP8_E4M3 = 1,
    RPA_DT_F16 = 2,
    RPA_DT_F32 = 3,       /* q only */
    RPA_DT_FP8_E5M2 = 4,  /* K/V only */
    RPA_DT_INT8 = 5       /* K/V only */
} RpaDtype;

typedef enum RpaStatus {
    RPA_OK = 0,
    RPA_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad configuration value */
    RPA_ERR_UNSUPPORTED = 2,    /* dtype (f32/i32/i16 K/V), head_dim not in {64,128,256}, Hq % Hkv != 0, group > 64,
                                   page_size not a multiple of 4, mask_value above -1e30 */
    RPA_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
    RPA_ERR_BAD_PAGE_INDEX = 4, /* device-detected: a used page id outside [0, total_num_pages) */
    RPA_ERR_BAD_LENGTHS = 5,    /* device-detected: kv_len > pages_per_seq*page_size, q_len > kv_len,
                                   cu_q_lens decreasing or past num_q_tokens, negative lengths */
    RPA_ERR_TIMEOUT = 6,        /* device-detected: a bounded wait gave up */
    RPA_ERR_NO_ALLOC_LIMIT = 7  /* rpa_forward_noalloc: the configuration's workspace exceeds
                                   the library's fixed 32 MiB scratch array */
} RpaStatus;

/* Kernel configuration: the shape fields and numeric knobs of the page's Cfg.
 * The block knobs (num_kv_pages_per_block, num_queries_per_block) are not
 * exposed: the library picks its own tiles. */
typedef struct RpaCfg {
    int64_t num_q_tokens;    /* rows of q and o */
    int64_t num_q_heads;     /* Hq */
    int64_t num_kv_heads;    /* Hkv; Hq % Hkv == 0 and Hq/Hkv <= 64 */
    int64_t head_dim;        /* D in {64, 128, 256} */
    int64_t total_num_pages; /* physical pages in kv_pages */
    int64_t page_size;       /* keys per page: a multiple of 4 (others give RPA_ERR_UNSUPPORTED) */
    int64_t max_num_seqs;    /* rows of kv_lens / page_indices; cu_q_lens has max_num_seqs+1 */
    int64_t pages_per_seq;   /* columns of page_indices */
    int64_t sliding_window;  /* used when has_sliding_window; must be >= 1 */
    int32_t q_dtype;         /* RpaDtype of q and o: BF16, F16 or F32 */
    int32_t kv_dtype;        /* RpaDtype of kv_pages: BF16, F16, FP8_E4M3, FP8_E5M2 or INT8 */
    float sm_scale;          /* logit scale, finite */
    float mask_value;        /* additive mask of the page (default -2.38197633e38); must be
                                <= -1e30 so that masked keys get weight exactly 0 */
    float soft_cap;          /* used when has_soft_cap; > 0 */
    float k_scale;           /* used when has_k_scale; K dequant factor */
    float v_scale;           /* used when has_v_scale; V dequant factor */
    int32_t has_soft_cap;
    int32_t has_k_scale;
    int32_t has_v_scale;
    int32_t is_causal;       /* 1 = causal (default of the page) */
    int32_t has_sliding_window;
    int32_t has_sinks;       /* 1: attention sinks, read from `sinks` */
    int32_t kv_layout;       /* RpaKvLayout: RPA_KV_SPLIT (the page's layout, default) or RPA_KV_LATENT */
    int32_t reserved;        /* set to 0 */
    int64_t v_head_dim;      /* RPA_KV_SPLIT: 0 or head_dim.  RPA_KV_LATENT: the width of V and o */
    const float* sinks;      /* when has_sinks: device, [num_q_heads] fp32, 4-byte aligned; the
                                sink logit of each query head (the "from_qwen_ops.rs" page,
                                flat_softmax_rows_at, `sinks`): it starts the row maximum and
                                exp(sink - max) joins the softmax denominator, carrying no
                                value.  It is a logit of the softmax as it stands (not scaled by
                                sm_scale, not soft-capped).  Read by every call on the handle
                                (or by the rpa_forward_noalloc call given this cfg): it must
                                stay valid while those calls run. */
} RpaCfg;

/* K/V page layouts.
 * RPA_KV_SPLIT:  kv_pages[total_num_pages, page_size, 2*Hkv, head_dim], combined
 *                head 2h = K of kv head h, 2h+1 = its V ("ragged_paged.zig").
 * RPA_KV_LATENT: latent attention over a paged latent cache (the
 *                "from_qwen_ops.rs" page, "The latent-attention family at
 *                whole-tile widths"): kv_pages[total_num_pages, page_size,
 *                Hkv, head_dim], one latent row per kv head and slot; K is the
 *                whole row and V its first v_head_dim elements, so q is
 *                [num_q_tokens, Hq, head_dim] and o [num_q_tokens, Hq,
 *                v_head_dim].  Supported: head_dim 576 with v_head_dim 512 (a
 *                512-wide latent and a 64-wide rope part), bf16 or f16 rows,
 *                page_size a multiple of 8, Hq/Hkv at most 16 or a multiple of
 *                16; any other choice gives RPA_ERR_UNSUPPORTED. */
typedef enum RpaKvLayout { RPA_KV_SPLIT = 0, RPA_KV_LATENT = 1 } RpaKvLayout;

typedef struct RpaHandle RpaHandle;

/* Fill *cfg with the page's defaults for the shape fields given: q/kv bf16,
 * mask_value -2.38197633e38, causal, no softcap, no scales, no window. */
void rpa_cfg_init(RpaCfg* cfg);

/* Check a configuration on the host only (no CUDA call).  Returns RPA_OK,
 * RPA_ERR_INVALID_ARG or RPA_ERR_UNSUPPORTED. */
int rpa_validate_cfg(const RpaCfg* cfg);

/* Validate cfg, then allocate the workspace (plan buffers and split-KV
 * partials, sized for the worst case of cfg) on the current device.
 * On success *out receives the handle; on failure *out is NULL. */
int rpa_create(const RpaCfg* cfg, RpaHandle** out);

/* One ragged paged attention call (the page's kernel call with inputs
 * kv_lens, page_indices, cu_q_lens, num_seqs, q, kv_pages and output o).
 *   q            device, [num_q_tokens, Hq, D] q_dtype, 16-byte aligned
 *   kv_pages     device, [total_num_pages, page_size, 2*Hkv, D] kv_dtype, 16-byte aligned
 *                ([total_num_pages, page_size, Hkv, D] for RPA_KV_LATENT)
 *   kv_lens      device, int32 [max_num_seqs]
 *   page_indices device, int32 [max_num_seqs, pages_per_seq], row-major
 *   cu_q_lens    device, int32 [max_num_seqs + 1]
 *   num_seqs     host scalar, 0 <= num_seqs <= max_num_seqs (the page passes it
 *                as a one-element array)
 *   o            device, [num_q_tokens, Hq, Dv] q_dtype (Dv = D, or v_head_dim for
 *                RPA_KV_LATENT), 16-byte aligned, written in
 *                full: rows of tokens outside [cu_q_lens[0], cu_q_lens[num_seqs])
 *                are written as 0
 *   stream       cudaStream_t as void*
 * Host-detectable errors return at once without enqueuing work.  Lengths and
 * page ids are checked on the device and set the status read by
 * rpa_get_status: bad lengths leave every row of o zero; a bad page id is
 * never dereferenced (its keys read as zero) and leaves the rows of the
 * sequences that use it unspecified.  Calls on one handle must be serialised
 * on the GPU (one stream, or ordered streams): they share the workspace.
 * The call may be captured into a CUDA graph (after one eager call, which
 * sets kernel attributes); the graph's replays read the buffers passed at
 * capture and must be serialised like calls. */
int rpa_forward(RpaHandle* h, const void* q, const void* kv_pages, const int32_t* kv_lens,
                const int32_t* page_indices, const int32_t* cu_q_lens, int32_t num_seqs,
                void* o, void* stream);

/* rpa_forward with the per-step inputs and the output in HOST memory: q,
 * kv_lens, page_indices and cu_q_lens are copied host->device into staging
 * buffers owned by the handle (allocated on first use), the call runs, and o
 * is copied back device->host, all on `stream`.  kv_pages stays a device
 * pointer (the paged cache is resident state).  The host buffers must stay
 * valid until the stream reaches the end of the call; pinned memory makes
 * the copies asynchronous. */
int rpa_forward_host(RpaHandle* h, const void* q_host, const void* kv_pages,
                     const int32_t* kv_lens_host, const int32_t* page_indices_host,
                     const int32_t* cu_q_lens_host, int32_t num_seqs, void* o_host,
                     void* stream);

/* Synchronise `stream` and return the device-side status of the last call
 * (RPA_OK, RPA_ERR_BAD_PAGE_INDEX, RPA_ERR_BAD_LENGTHS or RPA_ERR_TIMEOUT),
 * or RPA_ERR_CUDA if the synchronisation failed. */
int rpa_get_status(RpaHandle* h, void* stream);

/* Work plan of the last call, for tests and tooling.  Synchronises `stream`.
 * info (host, 16 int32) receives: [0] status, [1] decode items, [2] prefill
 * items, [3] split-KV combine entries, [4] decode chunk (keys), [5] decode
 * tile rows, [6] query tokens per prefill tile, [7] partial slots used, [8] planned
 * units, [9] 1 if units were sorted by cost, [10] decode CTAs given work, [11]
 * prefill CTAs given work, [12] SMs, [13] / [14] resident decode / prefill
 * CTAs per SM, [15] bit 0: decode and prefill ran concurrently, bit 1: decode units were
 * items of the prefill-side kernel (8-bit K/V on tensor memory, or the latent layout).  items (host, may be NULL)
 * receives up to max_items decode items followed by the prefill items, 8
 * int32 each: seq, kv head, first query token of the sequence's tile (local),
 * tokens in the tile, first key, end key, partial slot (-1 = direct write),
 * piece index. */
int rpa_read_plan(RpaHandle* h, int32_t* info, int32_t* items, int64_t max_items, void* stream);

/* Per-kernel timing for benchmarks.  After rpa_profile_begin(h, n) the next n
 * calls of rpa_forward on h record CUDA events around each of their four
 * kernels: planner, decode attention, prefill attention, combine.  Each kernel
 * is timed on the stream it runs on, from an event recorded just before its
 * launch (after any wait on the other stream) to one recorded just after it,
 * so that the two attention kernels are timed correctly also when they run at
 * once on two streams.  rpa_profile_read synchronises on those events and
 * writes, for each recorded call c < *n_calls, ms[4*c + k] = duration of
 * kernel k in milliseconds (a kernel with no work reads as its launch time);
 * ms holds max_calls*4 floats (host).  Profiling stops after n calls or at the
 * next rpa_profile_begin; the events are owned by h. */
int rpa_profile_begin(RpaHandle* h, int32_t max_calls);
int rpa_profile_read(RpaHandle* h, float* ms, int32_t max_calls, int32_t* n_calls);

/* Options of a handle (rpa_set_option).  Production code needs none of them;
 * the library reads no environment variable. */
typedef enum RpaOption {
    RPA_OPT_WAIT_TIMEOUT_MS = 1,   /* bound of every device-side wait, in ms (1 .. 3600000; default
                                      1000); a wait that runs out sets RPA_ERR_TIMEOUT */
    RPA_OPT_SERIAL = 2,            /* 1: run decode and prefill attention one after the other on the
                                      caller's stream instead of concurrently with an SM split
                                      (default 0; configurations without the split always run
                                      serially) */
    RPA_OPT_PREFILL_SMS = 3,       /* > 0: SMs given to prefill attention when both kernels have
                                      work and run concurrently (0 = the planner's model; tuning) */
    RPA_OPT_DECODE_SMS = 4,        /* > 0: SMs given to decode attention (0 = the planner's model) */
    RPA_OPT_PLAN_EARLY = 5,        /* 1: the caller guarantees that a call's kv_lens and cu_q_lens are
                                      complete when the call is enqueued (no kernel still writing them
                                      precedes it on the stream: host copies, or kernels that end before
                                      the call, satisfy this); the planner then reads and orders them
                                      while the kernel before it (typically the previous call's
                                      combine) still runs.  Default 0: it first waits for that kernel */
    RPA_OPT_TEST_STALL_PRODUCER = 100  /* test hook, 1: the decode kernel's copy warp issues nothing, so
                                      that its consumers' bounded waits run out (status
                                      RPA_ERR_TIMEOUT); the kernel still returns */
} RpaOption;

/* Set option `option` of h to `value` for the following calls.  Host only.
 * Returns RPA_OK, or RPA_ERR_INVALID_ARG for an unknown option or a value
 * outside its range (the option is then unchanged). */
int rpa_set_option(RpaHandle* h, int32_t option, int64_t value);

/* rpa_forward for callers that cannot allocate device memory.
 *
 * The method has no counterpart to this entry point (it is an API choice); it exists for callers
 * that may not call cudaMalloc/cudaFree where they run attention: serving
 * engines that hand all device memory to their own arena allocator, code
 * paths where an allocation's implicit device synchronisation is not
 * allowed, and plain-C hosts that have no allocator to give the library.
 *
 * It takes no handle: the configuration and tensors are those of rpa_create
 * plus rpa_forward, and the planner, attention and combine kernels are the
 * same.  Their workspace (plan, work items, split-KV partials) is carved from
 * one 32 MiB array in the library's own device memory, which every GPU that
 * loads the library holds until the process exits.  A configuration whose
 * worst-case workspace exceeds 32 MiB returns RPA_ERR_NO_ALLOC_LIMIT before
 * anything is enqueued.  Nothing here calls cudaMalloc, cudaFree or any other
 * allocating routine.
 *
 * The first call on each device (with that device current) looks up the
 * array's device address and sets kernel attributes; make that first call
 * before any stream capture.  Every call shares the one array and it keeps
 * the previous call's contents (the call clears what must start at zero), so
 * calls that overlap on the GPU -- on different streams, or from different
 * threads -- race and must be serialised by the caller.  The device-side
 * status is not reported by this entry point: bad lengths (o all zero), a bad
 * page id, and a device wait that ran out (after 1 s; o then unspecified)
 * still return RPA_OK. */
int rpa_forward_noalloc(const RpaCfg* cfg, const void* q, const void* kv_pages,
                        const int32_t* kv_lens, const int32_t* page_indices,
                        const int32_t* cu_q_lens, int32_t num_seqs, void* o, void* stream);

/* Free the workspace and the handle (synchronises the device first). NULL is ignored. */
void rpa_destroy(RpaHandle* h);

/* Static description of a status code. */
const char* rpa_strerror(int code);

/* ABI version of this header (major*100 + minor): 200. */
int rpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RPA_H_ */
