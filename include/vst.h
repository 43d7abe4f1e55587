/*
 * vst.h -- C ABI of libvst: incremental sliding-window KV attention on one GB300 (sm_103a).
 *
 * The operation. A streaming audio-LLM runs its attention layers incrementally: each new
 * chunk of frames (encoder) or each new token (decoder) attends, under a windowed-causal
 * mask keyed on absolute positions, to keys/values cached from earlier calls. The
 * definition followed here is the offline one: for a query at absolute position i and
 * query head h,
 *
 *     out = sum_j softmax_j( RoPE(q_i, i) . RoPE(k_j, j) / sqrt(D) ) v_j,
 *     over absolute positions j with 0 <= i - j < W, KV head h / (H / Hk),
 *
 * with NEOX (rotate-half) RoPE, theta = 1e6. Sources: "Voxtral Realtime -- incremental
 * streaming implementation plan", sections "SHIPPED" (Mechanism: encoder cache with
 * sliding_window=750 under a windowed-causal mask, decoder persistent sliding KV(8192)) and
 * "Unbounded length (shipped)" (1536-slot encoder ring, compaction that copies the last 750
 * frames to the front, feeds pushed in <= 512-frame batches, mask on absolute positions);
 * "Voxtral Realtime" family doc, "Architecture (summary)" (encoder: NEOX RoPE theta=1e6,
 * head dim 64, sliding window 750; decoder: GQA 32q/8kv, head dim 128, sliding 8192) and
 * Capability Validation, Streaming row, item (5) (decoder modulo ring: token cur writes
 * slot cur % n_ctx and the mask reveals [cur-8191, cur]; positions stay absolute).
 *
 * The shape of the API follows "Stateless modules and streaming contexts" (bunsen book),
 * sections "The principle: state is injected" and "The pattern": a config builds an
 * immutable module (here: the fixed RoPE cos/sin table), and each stream's cache context
 * is made by the caller and passed in on every call, so one module serves many streams and
 * a batch of streams can run through one launch.
 *
 * Conventions.
 *   - bf16 tensors are passed as device pointers (void*), row-major, 16-byte aligned.
 *     q / out: [rows][H][D]; k / v: [rows][Hk][D].
 *   - `stream` is a cudaStream_t passed as void*. Every call only enqueues work on it and
 *     returns; no call synchronises the device. Host-side state (positions, ring fill)
 *     advances when the call returns, so calls on one ctx must stay on one stream (or be
 *     ordered by the caller).
 *   - A ctx is used by one host thread at a time. Contexts are independent of each other.
 *   - Errors: argument and config errors return before anything is enqueued and leave the
 *     ctx unchanged. A CUDA error while enqueueing marks the ctx failed: later calls on it
 *     return VST_E_STATE until vst_ctx_reset.
 *   - Inputs must be finite. Ring slots that are never written are zeroed at create/reset.
 */
#ifndef VST_H
#define VST_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VST_API __attribute__((visibility("default")))
#else
#define VST_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VST_OK = 0,
    VST_E_INVAL = -1,       /* bad argument (null pointer, size, position past the table) */
    VST_E_UNSUPPORTED = -2, /* configuration the library has no kernel for */
    VST_E_CUDA = -3,        /* a CUDA runtime call failed */
    VST_E_STATE = -4,       /* ctx is failed (earlier CUDA error) or of the wrong kind */
    VST_E_TIMEOUT = -5,     /* a kernel gave up on a bounded wait (reported by vst_ctx_check) */
    VST_E_NOMEM = -6        /* caller memory too small, or cudaMalloc failed */
} vst_status;

typedef enum { VST_ENC = 1, VST_DEC = 2 } vst_kind;

/* Configuration of one attention layer's cache. The two shapes the pages give are
 *   encoder: kind VST_ENC, H = Hk = 20, D = 64, W = 750, ring 1536, max_batch 512
 *   decoder: kind VST_DEC, H = 32, Hk = 8, D = 128, W = 8192, ring 8192 (or any multiple
 *            of 128 >= W), max_batch 1
 * with rope_theta 1e6 and max_position 131072 (the decoder's position cap, family doc,
 * Streaming row, item (5)). Supported by the library: encoder D = 64 with H = Hk; decoder
 * D = 128 with H = 4 * Hk. Other values return VST_E_UNSUPPORTED from vst_module_create. */
typedef struct {
    int32_t kind;         /* vst_kind */
    int32_t n_heads;      /* H, query heads */
    int32_t n_kv_heads;   /* Hk, key/value heads; H % Hk == 0 */
    int32_t head_dim;     /* D */
    int32_t window;       /* W: the query at position p sees keys p-W+1 .. p */
    int32_t ring_slots;   /* R: cache rows per KV head */
    int32_t max_batch;    /* encoder: frames appended per internal batch (<= 512) */
    int32_t reserved;     /* must be 0 */
    int64_t max_position; /* absolute positions must stay below this (RoPE table length) */
    double rope_theta;    /* RoPE base */
} vst_config;

/* Fill *cfg with the pages' encoder (kind = VST_ENC) or decoder (VST_DEC) configuration. */
VST_API vst_status vst_config_default(int32_t kind, vst_config* cfg);

typedef struct vst_module vst_module; /* immutable: config + RoPE table on one device */
typedef struct vst_ctx vst_ctx;       /* one (stream, layer) cache */
typedef struct vst_offline vst_offline; /* scratch for batched whole-clip encoder attention */

/* Build the module on the current CUDA device: validates cfg, computes the RoPE cos/sin
 * table on the host in double precision (angle p * theta^(-2i/D)), rounds it to fp32 and
 * uploads it (device memory owned by the module, max_position * D * 4 bytes). Blocking. */
VST_API vst_status vst_module_create(const vst_config* cfg, vst_module** out);
VST_API vst_status vst_module_destroy(vst_module* m); /* all its contexts must be destroyed first */
VST_API vst_status vst_module_config(const vst_module* m, vst_config* cfg);

/* Device bytes one ctx of this module needs (rings + scratch), a multiple of 256. */
VST_API size_t vst_ctx_bytes(const vst_module* m);

/* Create a ctx. dev_mem: caller-owned device memory of at least vst_ctx_bytes(m) bytes,
 * 256-byte aligned, that must outlive the ctx; or NULL, and the library allocates it with
 * cudaMalloc and frees it in vst_ctx_destroy. The ring is zeroed on `stream`. */
VST_API vst_status vst_ctx_create(const vst_module* m, void* dev_mem, size_t bytes, void* stream,
                          vst_ctx** out);
/* Forget the stream (positions back to 0, ring empty, failure cleared) and zero the ring on
 * `stream`; memory is kept (streaming plan, "Per-hook behavior": stream_reset). */
VST_API vst_status vst_ctx_reset(vst_ctx* c, void* stream);
VST_API vst_status vst_ctx_destroy(vst_ctx* c);

typedef struct {
    int32_t kind;
    int32_t failed;         /* 1 after a CUDA error, until reset */
    int64_t n_kv;           /* encoder: ring rows in use, slots [0, n_kv) */
    int64_t abs_base;       /* encoder: absolute position held by slot 0 */
    int64_t abs_next;       /* absolute position of the next frame/token */
    int64_t n_compactions;  /* encoder compactions enqueued so far */
    void* k_ring;           /* device [Hk][R][D] bf16, RoPE already applied */
    void* v_ring;           /* device [Hk][R][D] bf16 */
} vst_ctx_info;
VST_API vst_status vst_ctx_info_get(const vst_ctx* c, vst_ctx_info* out);

/* Read the ctx's device error word (blocking: synchronises `stream`). Returns VST_OK, or
 * VST_E_TIMEOUT when a kernel of this ctx abandoned a bounded wait, and clears the word. */
VST_API vst_status vst_ctx_check(vst_ctx* c, void* stream);
/* Test helper for failure detection: one device wait of the kind every kernel uses for its
 * copies and MMAs (an mbarrier wait bounded to 2 s of %globaltimer time), recorded in this
 * ctx's error word. complete = 1: the wait is satisfied at once. complete = 0: nothing
 * completes it; it gives up after the limit, the kernel records a time-out and returns, and
 * the next vst_ctx_check reports VST_E_TIMEOUT (and clears it). Nothing faults, traps or
 * stays pending: the ctx remains usable. Enqueued on `stream`; VST_E_INVAL for a NULL ctx. */
VST_API vst_status vst_ctx_selftest_wait(vst_ctx* c, int32_t complete, void* stream);

/* ---- encoder chunk path (streaming plan, "SHIPPED" and "Unbounded length") -------------
 * Feed n_new >= 0 frames: q [n_new][H][D], k/v [n_new][Hk][D] -> out [n_new][H][D]. Frames
 * get absolute positions abs_next .. abs_next + n_new - 1. The feed is pushed in batches of
 * at most max_batch; before a batch that would not fit in the ring, the last W rows are
 * copied to the front (compaction); each batch's K (rotated) and V are appended at ring
 * rows [n_kv, n_kv + b), then every new frame attends to the window [p - W + 1, p]. The
 * output does not depend on how a stream is cut into feeds (bit for bit). */
VST_API vst_status vst_enc_feed(vst_ctx* c, const void* q, const void* k, const void* v, int32_t n_new,
                        void* out, void* stream);
/* The same for n_ctx contexts of one module in lockstep (one launch per kernel): tensors
 * are stacked per ctx, q [n_ctx][n_new][H][D], k/v [n_ctx][n_new][Hk][D], out like q. The
 * contexts must be distinct; their positions and ring fills may differ. */
VST_API vst_status vst_enc_feed_batch(vst_ctx* const* ctxs, int32_t n_ctx, const void* q, const void* k,
                              const void* v, int32_t n_new, void* out, void* stream);
/* Compact now, whatever the fill (keeps the last W rows); no-op when n_kv <= W. */
VST_API vst_status vst_ctx_compact(vst_ctx* c, void* stream);

/* Host-only: the launch shape of the chunk attention for one batch of `batch` frames over
 * n_ctx contexts of n_heads heads, whose widest window spans max_key_tiles key tiles of 128
 * absolute positions, when the GPU holds resident_ctas CTAs of the split shape at once (the
 * SMs the stream can use -- the device's, lowered by an MPS active-thread percentage in the
 * environment or by the stream's green context -- times the split shape's CTAs per SM).
 * *split = 0: the loop shape, one CTA per (ctx, head, 128-frame query tile), *grid_x query
 * tiles. *split = k > 0: the split shape, one CTA per (ctx, head, group of k key tiles),
 * *grid_x groups; chosen only for a single query tile when n_ctx x n_heads < resident_ctas,
 * with k the least that keeps the grid within resident_ctas: the shape's merging CTA waits
 * for the other CTAs of its (ctx, head), so they must all be resident together. Both shapes
 * give the same bits. VST_E_INVAL for non-positive sizes or NULL outputs. Needs no GPU. */
VST_API vst_status vst_enc_launch_shape(int32_t n_heads, int32_t n_ctx, int32_t batch, int32_t max_key_tiles,
                                        int64_t resident_ctas, int32_t* split, int32_t* grid_x);

/* Host-only: the schedule vst_enc_feed would enqueue for a ctx in state (n_kv, abs_base)
 * fed n_new frames. Writes up to max_steps entries: batch[i] frames appended in step i,
 * compact[i] = 1 if a compaction precedes it. Returns the step count in *n_steps and the
 * final state in *n_kv_out / *abs_base_out. Needs no GPU. */
VST_API vst_status vst_enc_plan(const vst_config* cfg, int64_t n_kv, int64_t abs_base, int32_t n_new,
                        int32_t* batch, int32_t* compact, int32_t max_steps, int32_t* n_steps,
                        int64_t* n_kv_out, int64_t* abs_base_out);

/* ---- batched offline encoder over whole clips ---------------------------------------------
 * The pages' batch path ("Voxtral Realtime" family doc, Capability Validation, Batch row,
 * item (1)): clips right-padded to one length T and stacked, one shared position range and
 * mask, each caller slicing its clip's real rows. Causal masks never let padding reach a
 * real row. Optionally with a right lookahead: the (left L, right R) sliding mask of
 * "Moonshine streaming forward map", Encoder table, per-layer sliding-window mask row.
 * Frame i of a clip sees frame j of the same clip iff 0 <= i - j < L or 0 < j - i < R.
 * With L = W and R = 0, row i is bit for bit what streaming the clip through
 * vst_enc_feed gives for frame i (same tiles, same order of folds).
 *
 * A plan holds the scratch for B clips of T frames: K' and V of each clip, [H][T][D] bf16,
 * plus one error word and two tensor maps per clip. vst_offline_bytes gives its size
 * (0 for a decoder module or B, T < 1). dev_mem: caller-owned device memory of at least
 * that size, 256-byte aligned, or NULL for library-owned memory. Creation uploads the
 * tensor maps (blocking). */
VST_API size_t vst_offline_bytes(const vst_module* m, int32_t B, int32_t T);
VST_API vst_status vst_offline_create(const vst_module* m, int32_t B, int32_t T, void* dev_mem, size_t bytes,
                                      vst_offline** out);
VST_API vst_status vst_offline_destroy(vst_offline* p);
/* q, k, v, out: [B][T][H][D] bf16 device pointers, 16-byte aligned (Hk = H for the
 * encoder). left >= 1, right >= 0. Two launches per 64 clips: RoPE of K into the scratch,
 * then the loop-shape attention over all query tiles. Asynchronous on `stream`; positions
 * run 0 .. T-1 in every clip. VST_E_INVAL on bad arguments (nothing enqueued). */
VST_API vst_status vst_enc_offline(vst_offline* p, const void* q, const void* k, const void* v, int32_t left,
                                   int32_t right, void* out, void* stream);
/* Synchronise `stream`; VST_E_TIMEOUT (and clear it) if a bounded wait in a kernel gave up. */
VST_API vst_status vst_offline_check(vst_offline* p, void* stream);

/* ---- decoder step path (family doc, Streaming row, item (5)) ---------------------------
 * One token per stream: for each of n_streams contexts (one module, distinct), token s is
 * at absolute position pos_s = abs_next of ctxs[s]; its K (rotated) and V go to ring slot
 * pos_s % R, then its query attends keys [max(0, pos_s - W + 1), pos_s].
 * q [n_streams][H][D], k/v [n_streams][Hk][D], out [n_streams][H][D]. */
VST_API vst_status vst_dec_step(vst_ctx* const* ctxs, int32_t n_streams, const void* q, const void* k,
                        const void* v, void* out, void* stream);
/* vst_dec_step for callers that cannot allocate device memory at call time. The paper
 * (the pages this library follows) has no counterpart: this is a deployment variant.
 * Some callers must not call cudaMalloc while they stream: a real-time audio thread that
 * may not block (cudaMalloc can synchronise the device and take milliseconds), or a
 * process whose device memory is owned by another allocator or fixed at start-up. This
 * call computes exactly what vst_dec_step computes, but its scratch (split partials and
 * merge counters) lives in one static device array of 4 MiB inside libvst, held on every
 * GPU that loads the library until the process exits; the call itself allocates nothing.
 *   - Limit: n_streams * per-stream scratch must fit in 4 MiB, where per-stream scratch is
 *     H*S*2*4 + H*S*D*4 + Hk*4 bytes (each part rounded up to 256) and S = splits per
 *     step, ceil((W-1)/512) + 1. For the pages' decoder (32 heads x 128, window 8192,
 *     S = 17) that is 14 streams per call. Larger calls return VST_E_INVAL, nothing
 *     enqueued.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call uses the same array and leaves its last contents there; each call clears
 *     the counters it needs (stream-ordered) before its launch. Two calls that overlap on
 *     the GPU (different streams, not ordered) race on the array: order them.
 * Arguments, layouts, ownership and errors are those of vst_dec_step. */
VST_API vst_status vst_dec_step_noalloc(vst_ctx* const* ctxs, int32_t n_streams, const void* q,
                                        const void* k, const void* v, void* out, void* stream);
/* Decoder prefill: n tokens of one decoder ctx at positions pos .. pos + n - 1, pos being
 * its abs_next. This is the prompt the stream driver prefills once before stepping
 * ("Voxtral Realtime -- incremental streaming implementation plan", SHIPPED / Mechanism and
 * the stream_feed hook; 39 tokens there, any n here). Output row i is, bit for bit, what
 * the i-th of n successive vst_dec_step calls (one token each) returns: token i's K
 * (rotated) and V go to ring slot p_i % R and its query attends keys
 * [max(0, p_i - W + 1), p_i].
 * q [n][H][D], k/v [n][Hk][D], out [n][H][D]: bf16 device pointers, 16-byte aligned.
 * Tokens go in chunks of up to 64 per attention launch, each chunk's rows appended to the
 * ring first. So a chunk stays below position R (nothing evicted yet) or spans at most
 * R - W + 1 tokens: one token per launch once a ring with R = W is full; a ring a little
 * larger than the window keeps chunks of 64 everywhere.
 * The first call allocates the ctx's prefill scratch: split partials for 64 tokens, about
 * 18 MB for the pages' decoder (cudaMalloc, blocking). vst_ctx_destroy frees it.
 * Errors: VST_E_INVAL for bad arguments or positions past max_position (nothing
 * enqueued); VST_E_NOMEM if the scratch cannot be allocated; otherwise as vst_dec_step. */
VST_API vst_status vst_dec_prefill(vst_ctx* c, const void* q, const void* k, const void* v, int32_t n,
                                   void* out, void* stream);
/* Append n tokens of K/V (no attention) at positions abs_next .. abs_next + n - 1 of one
 * decoder ctx: k/v [n][Hk][D]. Used to fill a cache. */
VST_API vst_status vst_dec_append(vst_ctx* c, const void* k, const void* v, int32_t n, void* stream);

/* ---- kernel timing (tracing) -------------------------------------------------------------
 * When enabled, every kernel launch of this library is bracketed by two CUDA events
 * recorded on the launching stream (the kernel-level analogue of the pages' per-component
 * stream timer, family doc, Streaming row, item (7)). Off by default; costs two event
 * records per launch when on. One device per process while enabled. */
typedef enum { VST_K_ROPE_APPEND = 0, VST_K_COMPACT = 1, VST_K_ENC_ATTN = 2, VST_K_DEC_STEP = 3,
               VST_K_COUNT = 4 } vst_kernel_id;
typedef struct {
    int32_t kernel;    /* vst_kernel_id */
    int32_t reserved;
    int64_t launches;  /* launches timed since the last read */
    double total_ms;   /* sum of their event-to-event durations */
} vst_prof_stat;
VST_API vst_status vst_prof_enable(int32_t on);
/* Wait for the recorded events, fill out[0 .. VST_K_COUNT-1] (one entry per kernel id) and
 * forget them. Blocking. */
VST_API vst_status vst_prof_read(vst_prof_stat* out, int32_t max);
/* Kernels launched by this library since it was loaded (always counted). */
VST_API int64_t vst_launch_count(void);
VST_API const char* vst_kernel_name(int32_t kernel);

VST_API const char* vst_status_str(vst_status s);
/* Library version, "major.minor.patch". */
VST_API const char* vst_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VST_H */
