// vst_api.cu -- host side of libvst: configuration checks, the module (RoPE table), the
// per-stream contexts and their bookkeeping, and the batched launchers (kernel e) that
// turn one API call over many contexts into one launch per kernel.
//
// Bookkeeping follows the streaming plan ("Voxtral Realtime -- incremental streaming
// implementation plan", "Unbounded length (shipped)"): the encoder ring holds rows
// [0, n_kv) = absolute frames [abs_base, abs_base + n_kv); a feed is pushed in batches of
// at most max_batch frames; a batch that would not fit first triggers a compaction that
// keeps the last W rows. All of it is known on the host, so no call ever waits for the GPU.
#include <algorithm>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "vst_internal.h"

namespace vst {
// selftest.cu: one bounded device wait recorded in `err` (satisfied at once if `complete`).
cudaError_t launch_wait_selftest(int* err, int complete, cudaStream_t s);
}  // namespace vst

using namespace vst;

struct vst_module {
    vst_config cfg;
    int device;
    int n_sms;     // SMs of the device (launch-shape choice)
    int sms_usable;    // n_sms, lowered to the share an MPS active-thread percentage leaves
    int split_per_sm;  // split-shape CTAs one SM holds at once (0: never use the split shape)
    float2* rope;  // device [max_position][D/2]
    int splits;    // scratch slots per head: decoder splits per step / encoder key tiles
    CUtensorMap* rope_map;  // device: tensor map over the rope table (128-row boxes)
};

struct vst_ctx {
    const vst_module* m;
    uint8_t* mem;
    bool owns;
    size_t bytes;
    __nv_bfloat16* k_ring;
    __nv_bfloat16* v_ring;
    float* part_ml;
    float* part_o;
    unsigned* counters;
    int* err;
    const CUtensorMap* tmap_k;
    const CUtensorMap* tmap_v;
    int64_t n_kv, abs_base, abs_next, n_compactions;
    int failed;
    CUtensorMap host_maps[2];
    uint8_t* pf_mem;  // decoder prefill scratch (library-owned, allocated on first use)
    size_t pf_bytes;
};

// Offline plan: scratch for B whole clips of T frames ([B][H][T][D] K' and V), the error
// word and one pair of tensor maps per clip, in caller-provided or library-owned memory.
struct vst_offline {
    const vst_module* m;
    uint8_t* mem;
    bool owns;
    size_t bytes;
    int32_t B, T;
    CUtensorMap* maps;  // device: [B][2] (K', V)
    int* err;
    __nv_bfloat16* k_scr;
    __nv_bfloat16* v_scr;
};

namespace {

struct Layout {
    size_t k_off, v_off, ml_off, o_off, total;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int dec_splits(const vst_config& c) { return (c.window - 1 + kDecSplit - 1) / kDecSplit + 1; }

// Key tiles (128 absolute positions each) met by a query tile of up to 128 rows: the keys
// span at most 127 + W positions, which cross at most ceil((127 + W) / 128) + 1 tiles.
int enc_split_tiles(const vst_config& c) { return (c.window + 127 + 127) / kEncTileN + 1; }

int scratch_slots(const vst_config& c) { return c.kind == VST_DEC ? dec_splits(c) : enc_split_tiles(c); }


Layout layout_of(const vst_config& c)
{
    Layout L{};
    const size_t ring = (size_t)c.n_kv_heads * c.ring_slots * c.head_dim * sizeof(__nv_bfloat16);
    L.k_off = kCtxHeaderBytes;
    L.v_off = align256(L.k_off + ring);
    size_t end = align256(L.v_off + ring);
    // partial softmax scratch: decoder one row per (head, split); encoder 128 rows per
    // (head, key tile)
    const size_t rows = c.kind == VST_DEC ? 1 : kEncTileM;
    const size_t S = (size_t)scratch_slots(c);
    L.ml_off = end;
    L.o_off = align256(L.ml_off + (size_t)c.n_heads * S * rows * 2 * sizeof(float));
    end = align256(L.o_off + (size_t)c.n_heads * S * rows * c.head_dim * sizeof(float));
    L.total = end;
    return L;
}

vst_status check_config(const vst_config* c)
{
    if (!c)
        return VST_E_INVAL;
    if (c->reserved != 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
        c->window <= 0 || c->ring_slots <= 0 || c->max_position <= 0 || !(c->rope_theta > 0.0) ||
        c->n_heads % c->n_kv_heads != 0)
        return VST_E_INVAL;
    if (c->kind == VST_ENC) {
        if (c->max_batch <= 0 || (long long)c->window + c->max_batch > c->ring_slots)
            return VST_E_INVAL;
        // kernels (a), (b), (d): head dim 64, one KV head per query head, a compaction plane
        // of at most 128 KB, batches of at most 512 frames.
        if (c->head_dim != 64 || c->n_heads != c->n_kv_heads || c->max_batch > 512 ||
            (long long)c->window * c->head_dim * 2 > 128 * 1024)
            return VST_E_UNSUPPORTED;
        return VST_OK;
    }
    if (c->kind == VST_DEC) {
        if (c->ring_slots < c->window)
            return VST_E_INVAL;
        // kernel (c): head dim 128, 4 query heads per KV head, ring a multiple of the tile,
        // at most 32 splits per step (window <= 31 * 512 + 1).
        if (c->head_dim != 128 || c->n_heads != 4 * c->n_kv_heads || c->ring_slots % kDecTile != 0 ||
            dec_splits(*c) > 32)
            return VST_E_UNSUPPORTED;
        return VST_OK;
    }
    return VST_E_INVAL;
}

// Switch to the module's device for the duration of a call, then restore.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess)
            ok = false;
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev)
            cudaSetDevice(prev);
    }
};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor map over a ring [Hk][R][D] bf16: box of 64 dims x 128 rows x 1 head, 128-B
// swizzle, zero fill outside the ring.
bool make_ring_map(CUtensorMap* map, void* base, const vst_config& c)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {(cuuint64_t)c.head_dim, (cuuint64_t)c.ring_slots, (cuuint64_t)c.n_kv_heads};
    const cuuint64_t strides[2] = {(cuuint64_t)c.head_dim * 2, (cuuint64_t)c.ring_slots * c.head_dim * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Tensor map over a launch's queries for the loop shape: rows of D bf16 at `base`, laid out
// [jobs][row stride `job_rows`][H][D]; dims {D, H, rows, jobs}, box {D, 1, 128, 1}, 128-B
// swizzle (the Q' operand layout), zero fill past the rows.
bool make_query_map(CUtensorMap* map, const void* base, int D, int H, int rows, int jobs, long long job_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)jobs};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)job_rows * H * D * 2};
    const cuuint32_t box[4] = {(cuuint32_t)D, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---- launch accounting and optional per-kernel event timing
std::atomic<long long> g_launches{0};
std::atomic<int> g_prof_on{0};
std::mutex g_prof_mu;
struct ProfRec {
    int kid;
    cudaEvent_t a, b;
};
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pooled_event()
{
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Launch one kernel through f(); count it, and time it when timing is on.
template <class F>
cudaError_t tracked(int kid, cudaStream_t s, F&& f)
{
    if (!g_prof_on.load(std::memory_order_relaxed)) {
        const cudaError_t e = f();
        if (e == cudaSuccess)
            g_launches.fetch_add(1, std::memory_order_relaxed);
        return e;
    }
    std::lock_guard<std::mutex> lk(g_prof_mu);
    ProfRec r{kid, pooled_event(), pooled_event()};
    // Under stream capture an event record becomes a graph node only with the external
    // flag; then every replay of the graph re-records it.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cap);
    const unsigned flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0u;
    cudaEventRecordWithFlags(r.a, s, flags);
    const cudaError_t e = f();
    cudaEventRecordWithFlags(r.b, s, flags);
    if (e == cudaSuccess) {
        g_launches.fetch_add(1, std::memory_order_relaxed);
        g_prof_recs.push_back(r);
    }
    return e;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// ---- programmatic dependent launch bookkeeping
// The contexts the most recent kernel of this library touched, per stream. A chunk
// attention or decode launch may request ring tiles before the previous kernel in the
// stream has finished only if that kernel touched none of its contexts (it cannot then be
// writing those rings). Any other producer in between -- a kernel of the caller, a memset
// -- starts only after our earlier kernels complete, so it cannot open a race.
std::mutex g_touch_mu;
std::unordered_map<cudaStream_t, std::vector<const vst_ctx*>> g_last_touch;

// Record that the next launch on s touches ctxs[0..n) and return whether it may start its
// ring loads early.
int record_touch(cudaStream_t s, const vst_ctx* const* ctxs, int n)
{
    std::lock_guard<std::mutex> lk(g_touch_mu);
    std::vector<const vst_ctx*>& prev = g_last_touch[s];
    int early = 1;
    for (const vst_ctx* p : prev)
        for (int i = 0; i < n && early; ++i)
            if (p == ctxs[i])
                early = 0;
    prev.assign(ctxs, ctxs + n);
    return early;
}

// ---- co-residency of the split shape
// The split shape's merger waits for the other CTAs of its (ctx, head), so a split-shape grid
// must be resident all at once. These give the SMs a launch on a stream can use.

// The device's SM count, lowered to the share that an MPS active-thread percentage set in
// the environment leaves this process (rounded down).
int mps_sm_limit(int n_sms)
{
    const char* e = std::getenv("CUDA_MPS_ACTIVE_THREAD_PERCENTAGE");
    if (!e)
        return n_sms;
    char* end = nullptr;
    const double pct = std::strtod(e, &end);
    if (end == e || !(pct > 0.0) || pct >= 100.0)
        return n_sms;
    return (int)std::floor(n_sms * pct / 100.0);
}

struct GreenFns {
    PFN_cuStreamGetGreenCtx_v12040 stream_ctx = nullptr;
    PFN_cuGreenCtxGetDevResource_v12040 resource = nullptr;
};

const GreenFns& green_fns()
{
    static GreenFns f;
    static std::once_flag once;
    std::call_once(once, [] {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuStreamGetGreenCtx", &a, 12040, cudaEnableDefault, &qa) ==
                cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuGreenCtxGetDevResource", &b, 12040, cudaEnableDefault, &qb) ==
                cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            f.stream_ctx = reinterpret_cast<PFN_cuStreamGetGreenCtx_v12040>(a);
            f.resource = reinterpret_cast<PFN_cuGreenCtxGetDevResource_v12040>(b);
        }
    });
    return f;
}

// SMs a launch on stream s can use: the module's usable count, or fewer when s belongs to a
// green context (that context's SM resource).
int stream_sms(const vst_module* m, cudaStream_t s)
{
    int sms = m->sms_usable;
    const GreenFns& f = green_fns();
    CUgreenCtx gc = nullptr;
    if (f.stream_ctx && f.stream_ctx(reinterpret_cast<CUstream>(s), &gc) == CUDA_SUCCESS && gc) {
        CUdevResource r;
        std::memset(&r, 0, sizeof r);
        if (f.resource(gc, &r, CU_DEV_RESOURCE_TYPE_SM) == CUDA_SUCCESS)
            sms = std::min(sms, (int)r.sm.smCount);
    }
    return sms;
}

// Launch shape of one batch of the chunk attention (the same bits either way). Loop shape
// (false): one CTA per (ctx, head, query tile), grid_x = query tiles. Split shape (true), for
// a batch of one query tile when n_ctx x n_heads CTAs would leave most SMs idle: one CTA per
// (ctx, head, group of per_cta consecutive key tiles), the groups just large enough that the
// grid has at most `resident` CTAs, all of which the GPU holds at once.
bool enc_shape(int n_heads, int n_ctx, int q_tiles, int max_tiles, long long resident, int* per_cta, int* grid_x)
{
    *per_cta = 0;
    *grid_x = q_tiles;
    if (q_tiles != 1 || max_tiles < 1 || (long long)n_ctx * n_heads >= resident)
        return false;
    int k = 1;
    while ((long long)n_ctx * n_heads * ((max_tiles + k - 1) / k) > resident)
        ++k;
    *per_cta = k;
    *grid_x = (max_tiles + k - 1) / k;
    return true;
}

// Zero the error word, counters and both rings (not the tensor maps).
cudaError_t clear_ctx(vst_ctx* c, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(c->mem, 0, 256, s);
    if (e != cudaSuccess)
        return e;
    const Layout L = layout_of(c->m->cfg);
    return cudaMemsetAsync(c->mem + L.k_off, 0, L.ml_off - L.k_off, s);
}

vst_status fail_all(vst_ctx* const* ctxs, int n)
{
    for (int i = 0; i < n; ++i)
        ctxs[i]->failed = 1;
    return VST_E_CUDA;
}

// Common checks for a call over n contexts of one kind.
vst_status check_ctxs(vst_ctx* const* ctxs, int n, int kind)
{
    if (!ctxs || n <= 0)
        return VST_E_INVAL;
    const vst_module* m = nullptr;
    for (int i = 0; i < n; ++i) {
        if (!ctxs[i])
            return VST_E_INVAL;
        if (i == 0)
            m = ctxs[0]->m;
        if (ctxs[i]->m != m)
            return VST_E_INVAL;
        if (ctxs[i]->m->cfg.kind != kind || ctxs[i]->failed)
            return VST_E_STATE;
    }
    // distinct contexts (small n in practice; quadratic check is cheap next to a launch)
    for (int i = 0; i < n; ++i)
        for (int j = i + 1; j < n; ++j)
            if (ctxs[i] == ctxs[j])
                return VST_E_INVAL;
    return VST_OK;
}

}  // namespace

extern "C" {

const char* vst_version(void) { return "0.1.0"; }

vst_status vst_prof_enable(int32_t on)
{
    g_prof_on.store(on ? 1 : 0);
    return VST_OK;
}

vst_status vst_prof_read(vst_prof_stat* out, int32_t max)
{
    if (!out || max < VST_K_COUNT)
        return VST_E_INVAL;
    for (int k = 0; k < VST_K_COUNT; ++k)
        out[k] = vst_prof_stat{k, 0, 0, 0.0};
    std::lock_guard<std::mutex> lk(g_prof_mu);
    vst_status st = VST_OK;
    for (const ProfRec& r : g_prof_recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
            st = VST_E_CUDA;
        out[r.kid].launches += 1;
        out[r.kid].total_ms += ms;
        g_event_pool.push_back(r.a);
        g_event_pool.push_back(r.b);
    }
    g_prof_recs.clear();
    return st;
}

int64_t vst_launch_count(void) { return g_launches.load(); }

const char* vst_kernel_name(int32_t kernel)
{
    switch (kernel) {
    case VST_K_ROPE_APPEND: return "rope_append_kernel";
    case VST_K_COMPACT: return "compact_kernel";
    case VST_K_ENC_ATTN: return "enc_attn_kernel";
    case VST_K_DEC_STEP: return "dec_step_kernel";
    }
    return "unknown";
}

const char* vst_status_str(vst_status s)
{
    switch (s) {
    case VST_OK: return "ok";
    case VST_E_INVAL: return "invalid argument";
    case VST_E_UNSUPPORTED: return "unsupported configuration";
    case VST_E_CUDA: return "CUDA error";
    case VST_E_STATE: return "context failed or of the wrong kind";
    case VST_E_TIMEOUT: return "kernel wait timed out";
    case VST_E_NOMEM: return "out of memory";
    }
    return "unknown status";
}

vst_status vst_config_default(int32_t kind, vst_config* cfg)
{
    if (!cfg)
        return VST_E_INVAL;
    std::memset(cfg, 0, sizeof *cfg);
    cfg->kind = kind;
    cfg->rope_theta = 1.0e6;
    cfg->max_position = 131072;
    if (kind == VST_ENC) {
        cfg->n_heads = 20;
        cfg->n_kv_heads = 20;
        cfg->head_dim = 64;
        cfg->window = 750;
        cfg->ring_slots = 1536;
        cfg->max_batch = 512;
        return VST_OK;
    }
    if (kind == VST_DEC) {
        cfg->n_heads = 32;
        cfg->n_kv_heads = 8;
        cfg->head_dim = 128;
        cfg->window = 8192;
        cfg->ring_slots = 8192;
        cfg->max_batch = 1;
        return VST_OK;
    }
    return VST_E_INVAL;
}

vst_status vst_module_create(const vst_config* cfg, vst_module** out)
{
    if (!out)
        return VST_E_INVAL;
    *out = nullptr;
    vst_status st = check_config(cfg);
    if (st != VST_OK)
        return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return VST_E_CUDA;
    const int half = cfg->head_dim / 2;
    const size_t n = (size_t)cfg->max_position * half;
    // RoPE table: (cos, sin) of p * theta^(-2i/D), computed in double, stored as fp32.
    std::vector<double> freq(half);
    for (int i = 0; i < half; ++i)
        freq[i] = std::pow(cfg->rope_theta, -2.0 * i / cfg->head_dim);
    std::vector<float2> table;
    try {
        table.resize(n);
    } catch (const std::bad_alloc&) {
        return VST_E_NOMEM;
    }
    for (int64_t p = 0; p < cfg->max_position; ++p)
        for (int i = 0; i < half; ++i) {
            const double a = (double)p * freq[i];
            table[(size_t)p * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
        }
    vst_module* m = new (std::nothrow) vst_module();
    if (!m)
        return VST_E_NOMEM;
    m->cfg = *cfg;
    m->device = dev;
    m->splits = scratch_slots(*cfg);
    if (cudaDeviceGetAttribute(&m->n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || m->n_sms <= 0)
        m->n_sms = 148;
    m->sms_usable = mps_sm_limit(m->n_sms);
    if (cfg->kind != VST_ENC || enc_attn_split_blocks_per_sm(&m->split_per_sm) != cudaSuccess)
        m->split_per_sm = 0;
    if (cudaMalloc(&m->rope, n * sizeof(float2)) != cudaSuccess) {
        delete m;
        return VST_E_NOMEM;
    }
    if (cudaMemcpy(m->rope, table.data(), n * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(m->rope);
        delete m;
        return VST_E_CUDA;
    }
    // the encoder's loop shape fetches 128 rows of the table at a time by TMA
    if (cfg->kind == VST_ENC) {
        CUtensorMap host;
        auto fn = encode_fn();
        const cuuint64_t dims[2] = {(cuuint64_t)cfg->head_dim, (cuuint64_t)cfg->max_position};
        const cuuint64_t strides[1] = {(cuuint64_t)cfg->head_dim * sizeof(float)};
        const cuuint32_t box[2] = {(cuuint32_t)cfg->head_dim, 128};
        const cuuint32_t estr[2] = {1, 1};
        void* dmap = nullptr;
        if (!fn || fn(&host, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, m->rope, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
            cudaMalloc(&dmap, sizeof(CUtensorMap)) != cudaSuccess ||
            cudaMemcpy(dmap, &host, sizeof(CUtensorMap), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaFree(dmap);
            cudaFree(m->rope);
            delete m;
            return VST_E_UNSUPPORTED;
        }
        m->rope_map = static_cast<CUtensorMap*>(dmap);
    }
    *out = m;
    return VST_OK;
}

vst_status vst_module_destroy(vst_module* m)
{
    if (!m)
        return VST_E_INVAL;
    DeviceGuard g(m->device);
    cudaFree(m->rope);
    cudaFree(m->rope_map);
    delete m;
    return VST_OK;
}

vst_status vst_module_config(const vst_module* m, vst_config* cfg)
{
    if (!m || !cfg)
        return VST_E_INVAL;
    *cfg = m->cfg;
    return VST_OK;
}

size_t vst_ctx_bytes(const vst_module* m)
{
    return m ? layout_of(m->cfg).total : 0;
}

vst_status vst_ctx_create(const vst_module* m, void* dev_mem, size_t bytes, void* stream, vst_ctx** out)
{
    if (!m || !out)
        return VST_E_INVAL;
    *out = nullptr;
    const Layout L = layout_of(m->cfg);
    if (dev_mem && (bytes < L.total || ((uintptr_t)dev_mem & 255u)))
        return dev_mem && bytes < L.total ? VST_E_NOMEM : VST_E_INVAL;
    DeviceGuard g(m->device);
    if (!g.ok)
        return VST_E_CUDA;
    vst_ctx* c = new (std::nothrow) vst_ctx();
    if (!c)
        return VST_E_NOMEM;
    c->m = m;
    c->owns = dev_mem == nullptr;
    c->bytes = L.total;
    if (c->owns) {
        if (cudaMalloc(&dev_mem, L.total) != cudaSuccess) {
            delete c;
            return VST_E_NOMEM;
        }
    }
    c->mem = static_cast<uint8_t*>(dev_mem);
    c->err = reinterpret_cast<int*>(c->mem + kErrOffset);
    c->counters = reinterpret_cast<unsigned*>(c->mem + kCounterOffset);
    c->tmap_k = reinterpret_cast<const CUtensorMap*>(c->mem + kTmapOffset);
    c->tmap_v = reinterpret_cast<const CUtensorMap*>(c->mem + kTmapOffset + sizeof(CUtensorMap));
    c->k_ring = reinterpret_cast<__nv_bfloat16*>(c->mem + L.k_off);
    c->v_ring = reinterpret_cast<__nv_bfloat16*>(c->mem + L.v_off);
    c->part_ml = reinterpret_cast<float*>(c->mem + L.ml_off);
    c->part_o = reinterpret_cast<float*>(c->mem + L.o_off);
    bool ok = make_ring_map(&c->host_maps[0], c->k_ring, m->cfg) && make_ring_map(&c->host_maps[1], c->v_ring, m->cfg);
    cudaStream_t s = as_stream(stream);
    if (ok)
        ok = cudaMemcpyAsync(c->mem + kTmapOffset, c->host_maps, sizeof c->host_maps, cudaMemcpyHostToDevice, s) ==
                 cudaSuccess &&
             clear_ctx(c, s) == cudaSuccess;
    if (!ok) {
        if (c->owns)
            cudaFree(c->mem);
        delete c;
        return VST_E_CUDA;
    }
    *out = c;
    return VST_OK;
}

vst_status vst_ctx_reset(vst_ctx* c, void* stream)
{
    if (!c)
        return VST_E_INVAL;
    DeviceGuard g(c->m->device);
    c->n_kv = c->abs_base = c->abs_next = c->n_compactions = 0;
    c->failed = 0;
    if (clear_ctx(c, as_stream(stream)) != cudaSuccess ||
        (c->pf_mem && cudaMemsetAsync(c->pf_mem, 0, c->pf_bytes, as_stream(stream)) != cudaSuccess)) {
        c->failed = 1;
        return VST_E_CUDA;
    }
    return VST_OK;
}

vst_status vst_ctx_destroy(vst_ctx* c)
{
    if (!c)
        return VST_E_INVAL;
    {
        DeviceGuard g(c->m->device);
        if (c->owns)
            cudaFree(c->mem);
        if (c->pf_mem)
            cudaFree(c->pf_mem);
    }
    delete c;
    return VST_OK;
}

vst_status vst_ctx_info_get(const vst_ctx* c, vst_ctx_info* out)
{
    if (!c || !out)
        return VST_E_INVAL;
    out->kind = c->m->cfg.kind;
    out->failed = c->failed;
    out->n_kv = c->n_kv;
    out->abs_base = c->abs_base;
    out->abs_next = c->abs_next;
    out->n_compactions = c->n_compactions;
    out->k_ring = c->k_ring;
    out->v_ring = c->v_ring;
    return VST_OK;
}

vst_status vst_ctx_check(vst_ctx* c, void* stream)
{
    if (!c)
        return VST_E_INVAL;
    DeviceGuard g(c->m->device);
    int host_err = 0;
    cudaStream_t s = as_stream(stream);
    if (cudaMemcpyAsync(&host_err, c->err, sizeof host_err, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return VST_E_CUDA;
    if (host_err != 0) {
        // Clear the error word and, for good measure, the merge counters (every CTA counts
        // itself in even when it gives up, so they should read zero already once the
        // launches have ended, which the synchronisation above ensures).
        cudaMemsetAsync(c->mem, 0, kTmapOffset, s);
        if (c->pf_mem)
            cudaMemsetAsync(c->pf_mem, 0, c->pf_bytes, s);
        return VST_E_TIMEOUT;
    }
    return VST_OK;
}

vst_status vst_ctx_selftest_wait(vst_ctx* c, int32_t complete, void* stream)
{
    if (!c)
        return VST_E_INVAL;
    DeviceGuard g(c->m->device);
    if (!g.ok || launch_wait_selftest(c->err, complete ? 1 : 0, as_stream(stream)) != cudaSuccess)
        return VST_E_CUDA;
    return VST_OK;
}

vst_status vst_enc_plan(const vst_config* cfg, int64_t n_kv, int64_t abs_base, int32_t n_new, int32_t* batch,
                        int32_t* compact, int32_t max_steps, int32_t* n_steps, int64_t* n_kv_out,
                        int64_t* abs_base_out)
{
    if (!cfg || cfg->kind != VST_ENC || n_new < 0 || n_kv < 0 || n_kv > cfg->ring_slots || !n_steps)
        return VST_E_INVAL;
    const vst_status st = check_config(cfg);
    if (st != VST_OK)
        return st;
    int32_t k = 0;
    for (int32_t off = 0; off < n_new;) {
        const int32_t b = n_new - off < cfg->max_batch ? n_new - off : cfg->max_batch;
        int32_t comp = 0;
        if (n_kv + b > cfg->ring_slots) {
            const int64_t keep = n_kv < cfg->window ? n_kv : cfg->window;
            abs_base += n_kv - keep;
            n_kv = keep;
            comp = 1;
        }
        if (k < max_steps) {
            if (batch)
                batch[k] = b;
            if (compact)
                compact[k] = comp;
        }
        ++k;
        n_kv += b;
        off += b;
    }
    *n_steps = k;
    if (n_kv_out)
        *n_kv_out = n_kv;
    if (abs_base_out)
        *abs_base_out = abs_base;
    return VST_OK;
}

vst_status vst_enc_launch_shape(int32_t n_heads, int32_t n_ctx, int32_t batch, int32_t max_key_tiles,
                                int64_t resident_ctas, int32_t* split, int32_t* grid_x)
{
    if (n_heads <= 0 || n_ctx <= 0 || batch <= 0 || max_key_tiles <= 0 || resident_ctas < 0 || !split || !grid_x)
        return VST_E_INVAL;
    int per_cta = 0, gx = 0;
    enc_shape(n_heads, n_ctx, (batch + kEncTileM - 1) / kEncTileM, max_key_tiles, resident_ctas, &per_cta, &gx);
    *split = per_cta;
    *grid_x = gx;
    return VST_OK;
}

vst_status vst_enc_feed_batch(vst_ctx* const* ctxs, int32_t n_ctx, const void* q, const void* k, const void* v,
                              int32_t n_new, void* out, void* stream)
{
    vst_status st = check_ctxs(ctxs, n_ctx, VST_ENC);
    if (st != VST_OK)
        return st;
    if (n_new < 0)
        return VST_E_INVAL;
    if (n_new == 0)
        return VST_OK;
    if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return VST_E_INVAL;
    const vst_module* m = ctxs[0]->m;
    const vst_config& cfg = m->cfg;
    for (int i = 0; i < n_ctx; ++i)
        if (ctxs[i]->abs_next + n_new > cfg.max_position)
            return VST_E_INVAL;
    DeviceGuard g(m->device);
    if (!g.ok)
        return fail_all(ctxs, n_ctx);
    cudaStream_t s = as_stream(stream);
    const int H = cfg.n_heads, Hk = cfg.n_kv_heads, D = cfg.head_dim;
    const auto* qb = static_cast<const __nv_bfloat16*>(q);
    const auto* kb = static_cast<const __nv_bfloat16*>(k);
    const auto* vb = static_cast<const __nv_bfloat16*>(v);
    auto* ob = static_cast<__nv_bfloat16*>(out);

    const CompactCommon cc{Hk, cfg.ring_slots, D, cfg.window};
    EncAttnCommon ec{m->rope, 0, H, cfg.window, cfg.ring_slots, 0, m->splits, 0, 0,
                     (float)(1.4426950408889634 / std::sqrt((double)D))};
    ec.tmap_rope = m->rope_map;
    CompactJob cj[kMaxJobs];
    const vst_ctx* cctx[kMaxJobs];
    EncAttnJob ej[kMaxJobs];

    for (int32_t off = 0; off < n_new;) {
        const int32_t b = n_new - off < cfg.max_batch ? n_new - off : cfg.max_batch;
        const int q_tiles = (b + kEncTileM - 1) / kEncTileM;
        for (int c0 = 0; c0 < n_ctx; c0 += kMaxJobs) {
            const int nj = n_ctx - c0 < kMaxJobs ? n_ctx - c0 : kMaxJobs;
            int ncj = 0;
            for (int i = 0; i < nj; ++i) {
                vst_ctx* c = ctxs[c0 + i];
                if (c->n_kv + b > cfg.ring_slots) {
                    const int64_t keep = c->n_kv < cfg.window ? c->n_kv : cfg.window;
                    cctx[ncj] = c;
                    cj[ncj++] = CompactJob{c->k_ring, c->v_ring, c->n_kv - keep};
                    c->abs_base += c->n_kv - keep;
                    c->n_kv = keep;
                    c->n_compactions += 1;
                }
            }
            if (ncj > 0) {
                CompactCommon cc2 = cc;
                cc2.early = record_touch(s, cctx, ncj);
                if (tracked(VST_K_COMPACT, s, [&] { return launch_compact(cc2, cj, ncj, s); }) != cudaSuccess)
                    return fail_all(ctxs, n_ctx);
            }
            // Launch shape, same bits either way (enc_shape): the loop shape when it fills the
            // GPU, else the split shape with a grid the stream's SMs hold at once.
            const long long resident = q_tiles == 1 ? (long long)stream_sms(m, s) * m->split_per_sm : 0;
            const bool split_candidate = q_tiles == 1 && (long long)nj * H < resident;
            int max_tiles = 0;
            for (int i = 0; i < nj; ++i) {
                vst_ctx* c = ctxs[c0 + i];
                const long long row = (long long)(c0 + i) * n_new + off;
                ej[i] = EncAttnJob{qb + row * H * D, kb + row * Hk * D, vb + row * Hk * D, ob + row * H * D,
                                   c->k_ring, c->v_ring, c->tmap_k, c->tmap_v, c->part_ml, c->part_o,
                                   c->counters, c->err, c->abs_next, c->abs_base, c->n_kv, i};
                if (split_candidate) {
                    const long long lo = c->abs_next - cfg.window + 1 > 0 ? c->abs_next - cfg.window + 1 : 0;
                    const int tiles = (int)((c->abs_next + b - 1) / kEncTileN - lo / kEncTileN + 1);
                    max_tiles = tiles > max_tiles ? tiles : max_tiles;
                }
            }
            int per_cta = 0, grid_x = q_tiles;
            const bool split = enc_shape(H, nj, q_tiles, max_tiles, resident, &per_cta, &grid_x);
            if (!split) {
                // Loop shape: the batch's K' and V rows go to the ring first (kernel a), so
                // that every key tile of the attention arrives whole by TMA.
                const AppendCommon ac{m->rope, b, Hk, D, cfg.ring_slots, 0};
                AppendJob aj[kMaxJobs];
                for (int i = 0; i < nj; ++i) {
                    const vst_ctx* c = ctxs[c0 + i];
                    const long long row = (long long)(c0 + i) * n_new + off;
                    aj[i] = AppendJob{kb + row * Hk * D, vb + row * Hk * D, c->k_ring, c->v_ring, c->abs_next, c->n_kv};
                }
                record_touch(s, ctxs + c0, nj);
                if (tracked(VST_K_ROPE_APPEND, s, [&] { return launch_rope_append(ac, aj, nj, s); }) != cudaSuccess)
                    return fail_all(ctxs, n_ctx);
            }
            EncAttnCommon e2 = ec;
            e2.n_rows = b;
            e2.split = per_cta;
            e2.appended = split ? 0 : 1;
            if (!split && !make_query_map(&e2.tmap_q, qb + ((long long)c0 * n_new + off) * H * D, D, H, b, nj, n_new))
                return fail_all(ctxs, n_ctx);
            e2.lpt = (long long)H * nj <= m->n_sms;
            e2.early = record_touch(s, ctxs + c0, nj);
            if (tracked(VST_K_ENC_ATTN, s, [&] {
                    return split ? launch_enc_attn_split(e2, ej, nj, grid_x, s) : launch_enc_attn(e2, ej, nj, grid_x, s);
                }) != cudaSuccess)
                return fail_all(ctxs, n_ctx);
            for (int i = 0; i < nj; ++i) {
                ctxs[c0 + i]->n_kv += b;
                ctxs[c0 + i]->abs_next += b;
            }
        }
        off += b;
    }
    return VST_OK;
}

vst_status vst_enc_feed(vst_ctx* c, const void* q, const void* k, const void* v, int32_t n_new, void* out,
                        void* stream)
{
    return vst_enc_feed_batch(&c, 1, q, k, v, n_new, out, stream);
}

vst_status vst_ctx_compact(vst_ctx* c, void* stream)
{
    vst_ctx* cs[1] = {c};
    vst_status st = check_ctxs(cs, 1, VST_ENC);
    if (st != VST_OK)
        return st;
    const vst_config& cfg = c->m->cfg;
    if (c->n_kv <= cfg.window)
        return VST_OK;
    DeviceGuard g(c->m->device);
    CompactCommon cc{cfg.n_kv_heads, cfg.ring_slots, cfg.head_dim, cfg.window};
    const CompactJob cj{c->k_ring, c->v_ring, c->n_kv - cfg.window};
    cudaStream_t s = as_stream(stream);
    cc.early = record_touch(s, cs, 1);
    if (tracked(VST_K_COMPACT, s, [&] { return launch_compact(cc, &cj, 1, s); }) != cudaSuccess)
        return fail_all(cs, 1);
    c->abs_base += c->n_kv - cfg.window;
    c->n_kv = cfg.window;
    c->n_compactions += 1;
    return VST_OK;
}

vst_status vst_dec_step(vst_ctx* const* ctxs, int32_t n_streams, const void* q, const void* k, const void* v,
                        void* out, void* stream)
{
    vst_status st = check_ctxs(ctxs, n_streams, VST_DEC);
    if (st != VST_OK)
        return st;
    if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return VST_E_INVAL;
    const vst_module* m = ctxs[0]->m;
    const vst_config& cfg = m->cfg;
    for (int i = 0; i < n_streams; ++i)
        if (ctxs[i]->abs_next >= cfg.max_position)
            return VST_E_INVAL;
    DeviceGuard g(m->device);
    if (!g.ok)
        return fail_all(ctxs, n_streams);
    cudaStream_t s = as_stream(stream);
    const int H = cfg.n_heads, Hk = cfg.n_kv_heads, D = cfg.head_dim;
    const auto* qb = static_cast<const __nv_bfloat16*>(q);
    const auto* kb = static_cast<const __nv_bfloat16*>(k);
    const auto* vb = static_cast<const __nv_bfloat16*>(v);
    auto* ob = static_cast<__nv_bfloat16*>(out);
    const DecCommon dc0{m->rope, 0, Hk, cfg.ring_slots, cfg.window, m->splits, 0,
                        (float)(1.4426950408889634 / std::sqrt((double)D))};
    DecJob jobs[kMaxJobs];
    for (int c0 = 0; c0 < n_streams; c0 += kMaxJobs) {
        const int nj = n_streams - c0 < kMaxJobs ? n_streams - c0 : kMaxJobs;
        int work = 0;
        for (int i = 0; i < nj; ++i) {
            vst_ctx* c = ctxs[c0 + i];
            const long long si = c0 + i;
            const long long pos = c->abs_next;
            const long long lo = pos - cfg.window + 1 > 0 ? pos - cfg.window + 1 : 0;
            const int sig0 = (int)(lo / kDecSplit);
            const int nsp = (int)(pos / kDecSplit) - sig0 + 1;
            jobs[i] = DecJob{qb + si * H * D, kb + si * Hk * D, vb + si * Hk * D, ob + si * H * D,
                             c->k_ring, c->v_ring, c->tmap_k, c->tmap_v, c->part_ml, c->part_o,
                             c->counters, c->err, pos, sig0, nsp, work, 0};
            work += nsp;
        }
        DecCommon dc = dc0;
        dc.n_jobs = nj;
        dc.early = record_touch(s, ctxs + c0, nj);
        if (tracked(VST_K_DEC_STEP, s, [&] { return launch_dec_step(dc, jobs, nj, work, s); }) != cudaSuccess)
            return fail_all(ctxs, n_streams);
        for (int i = 0; i < nj; ++i)
            ctxs[c0 + i]->abs_next += 1;
    }
    return VST_OK;
}

// ---- batched offline encoder over whole clips ------------------------------------------

size_t vst_offline_bytes(const vst_module* m, int32_t B, int32_t T)
{
    if (!m || m->cfg.kind != VST_ENC || B < 1 || T < 1)
        return 0;
    const vst_config& c = m->cfg;
    const size_t scr = align256((size_t)B * c.n_kv_heads * T * c.head_dim * sizeof(__nv_bfloat16));
    return align256((size_t)B * 2 * sizeof(CUtensorMap)) + 256 + 2 * scr;
}

vst_status vst_offline_create(const vst_module* m, int32_t B, int32_t T, void* dev_mem, size_t bytes,
                              vst_offline** out)
{
    if (!out)
        return VST_E_INVAL;
    *out = nullptr;
    if (!m || m->cfg.kind != VST_ENC || B < 1 || T < 1 || T > m->cfg.max_position)
        return VST_E_INVAL;
    const vst_config& cfg = m->cfg;
    const size_t need = vst_offline_bytes(m, B, T);
    if (dev_mem && (bytes < need || ((uintptr_t)dev_mem & 255u)))
        return VST_E_INVAL;
    DeviceGuard g(m->device);
    if (!g.ok)
        return VST_E_CUDA;
    vst_offline* p = new (std::nothrow) vst_offline();
    if (!p)
        return VST_E_NOMEM;
    p->m = m;
    p->B = B;
    p->T = T;
    p->bytes = need;
    if (dev_mem) {
        p->mem = static_cast<uint8_t*>(dev_mem);
        p->owns = false;
    } else {
        void* mem = nullptr;
        if (cudaMalloc(&mem, need) != cudaSuccess) {
            delete p;
            return VST_E_NOMEM;
        }
        p->mem = static_cast<uint8_t*>(mem);
        p->owns = true;
    }
    const size_t maps_bytes = align256((size_t)B * 2 * sizeof(CUtensorMap));
    const size_t scr = align256((size_t)B * cfg.n_kv_heads * T * cfg.head_dim * sizeof(__nv_bfloat16));
    p->maps = reinterpret_cast<CUtensorMap*>(p->mem);
    p->err = reinterpret_cast<int*>(p->mem + maps_bytes);
    p->k_scr = reinterpret_cast<__nv_bfloat16*>(p->mem + maps_bytes + 256);
    p->v_scr = reinterpret_cast<__nv_bfloat16*>(p->mem + maps_bytes + 256 + scr);
    // clip b's K' and V: [H][T][D] each, maps over them as over a ring of T slots
    vst_config mc = cfg;
    mc.ring_slots = T;
    std::vector<CUtensorMap> host(2 * (size_t)B);
    bool ok = true;
    const size_t per_clip = (size_t)cfg.n_kv_heads * T * cfg.head_dim;
    for (int b = 0; b < B && ok; ++b)
        ok = make_ring_map(&host[2 * b], p->k_scr + b * per_clip, mc) &&
             make_ring_map(&host[2 * b + 1], p->v_scr + b * per_clip, mc);
    if (!ok || cudaMemcpy(p->maps, host.data(), host.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(p->err, 0, 256) != cudaSuccess) {
        if (p->owns)
            cudaFree(p->mem);
        delete p;
        return ok ? VST_E_CUDA : VST_E_UNSUPPORTED;
    }
    *out = p;
    return VST_OK;
}

vst_status vst_offline_destroy(vst_offline* p)
{
    if (!p)
        return VST_E_INVAL;
    if (p->owns) {
        DeviceGuard g(p->m->device);
        cudaFree(p->mem);
    }
    delete p;
    return VST_OK;
}

vst_status vst_enc_offline(vst_offline* p, const void* q, const void* k, const void* v, int32_t left, int32_t right,
                           void* out, void* stream)
{
    if (!p || !q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return VST_E_INVAL;
    if (left < 1 || right < 0)
        return VST_E_INVAL;
    const vst_module* m = p->m;
    const vst_config& cfg = m->cfg;
    DeviceGuard g(m->device);
    if (!g.ok)
        return VST_E_CUDA;
    cudaStream_t s = as_stream(stream);
    const int H = cfg.n_heads, Hk = cfg.n_kv_heads, D = cfg.head_dim;
    const int32_t T = p->T;
    const auto* qb = static_cast<const __nv_bfloat16*>(q);
    const auto* kb = static_cast<const __nv_bfloat16*>(k);
    const auto* vb = static_cast<const __nv_bfloat16*>(v);
    auto* ob = static_cast<__nv_bfloat16*>(out);
    const size_t per_clip = (size_t)Hk * T * D;
    for (int32_t b0 = 0; b0 < p->B; b0 += kMaxJobs) {
        const int nj = p->B - b0 < kMaxJobs ? p->B - b0 : kMaxJobs;
        // K' (rotated at positions 0 .. T-1) and V of each clip into its [H][T][D] scratch
        const AppendCommon ac{m->rope, T, Hk, D, T, 0};
        AppendJob aj[kMaxJobs];
        EncAttnJob ej[kMaxJobs];
        for (int i = 0; i < nj; ++i) {
            const long long row = (long long)(b0 + i) * T;
            __nv_bfloat16* ks = p->k_scr + (b0 + i) * per_clip;
            __nv_bfloat16* vs = p->v_scr + (b0 + i) * per_clip;
            aj[i] = AppendJob{kb + row * Hk * D, vb + row * Hk * D, ks, vs, 0, 0};
            ej[i] = EncAttnJob{qb + row * H * D, kb + row * Hk * D, vb + row * Hk * D, ob + row * H * D, ks, vs,
                               p->maps + 2 * (b0 + i), p->maps + 2 * (b0 + i) + 1, nullptr, nullptr, nullptr, p->err,
                               0, 0, 0, i};
        }
        if (tracked(VST_K_ROPE_APPEND, s, [&] { return launch_rope_append(ac, aj, nj, s); }) != cudaSuccess)
            return VST_E_CUDA;
        // one loop-shape launch over every query tile of every clip; mask [i - left + 1, i + right - 1]
        EncAttnCommon ec{m->rope, T, H, left, T, 0, 0, 0, 1, (float)(1.4426950408889634 / std::sqrt((double)D)),
                         right > 0 ? right - 1 : 0, H * nj <= m->n_sms ? 1 : 0, m->rope_map};
        if (!make_query_map(&ec.tmap_q, qb + (long long)b0 * T * H * D, D, H, T, nj, T))
            return VST_E_UNSUPPORTED;
        const int grid_x = (T + kEncTileN - 1) / kEncTileN;
        if (tracked(VST_K_ENC_ATTN, s, [&] { return launch_enc_attn(ec, ej, nj, grid_x, s); }) != cudaSuccess)
            return VST_E_CUDA;
    }
    return VST_OK;
}

vst_status vst_offline_check(vst_offline* p, void* stream)
{
    if (!p)
        return VST_E_INVAL;
    DeviceGuard g(p->m->device);
    int err = 0;
    cudaStream_t s = as_stream(stream);
    if (cudaMemcpyAsync(&err, p->err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return VST_E_CUDA;
    if (err != 0) {
        cudaMemsetAsync(p->err, 0, sizeof(int), s);
        return VST_E_TIMEOUT;
    }
    return VST_OK;
}

vst_status vst_dec_prefill(vst_ctx* c, const void* q, const void* k, const void* v, int32_t n, void* out,
                           void* stream)
{
    vst_ctx* cs[1] = {c};
    vst_status st = check_ctxs(cs, 1, VST_DEC);
    if (st != VST_OK)
        return st;
    if (n < 0)
        return VST_E_INVAL;
    if (n == 0)
        return VST_OK;
    if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return VST_E_INVAL;
    const vst_module* m = c->m;
    const vst_config& cfg = m->cfg;
    if (c->abs_next + n > cfg.max_position)
        return VST_E_INVAL;
    DeviceGuard g(m->device);
    if (!g.ok)
        return fail_all(cs, 1);
    const int H = cfg.n_heads, Hk = cfg.n_kv_heads, D = cfg.head_dim;
    const long long R = cfg.ring_slots, W = cfg.window;
    // per token of a chunk: m, l [H][S][2] and o [H][S][D] floats, then Hk merge counters
    const size_t ml_bytes = align256((size_t)H * m->splits * 2 * sizeof(float));
    const size_t o_bytes = align256((size_t)H * m->splits * D * sizeof(float));
    const size_t cnt_bytes = align256((size_t)Hk * sizeof(unsigned));
    const size_t per_token = ml_bytes + o_bytes + cnt_bytes;
    if (!c->pf_mem) {
        const size_t bytes = (size_t)kPrefillChunk * per_token;
        void* mem = nullptr;
        if (cudaMalloc(&mem, bytes) != cudaSuccess)
            return VST_E_NOMEM;
        if (cudaMemset(mem, 0, bytes) != cudaSuccess) {  // the merge counters start at zero
            cudaFree(mem);
            return VST_E_CUDA;
        }
        c->pf_mem = static_cast<uint8_t*>(mem);
        c->pf_bytes = bytes;
    }
    cudaStream_t s = as_stream(stream);
    const auto* qb = static_cast<const __nv_bfloat16*>(q);
    const auto* kb = static_cast<const __nv_bfloat16*>(k);
    const auto* vb = static_cast<const __nv_bfloat16*>(v);
    auto* ob = static_cast<__nv_bfloat16*>(out);
    const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    DecJob jobs[kPrefillChunk];
    for (int32_t off = 0; off < n;) {
        const long long pos0 = c->abs_next;
        // Chunk length. The chunk's rows are appended first, then each token attends from the
        // ring. Token j's row evicts key p_j - R, which an earlier token i of the chunk still
        // sees when p_j - R >= p_i - W + 1. So a chunk either stays below position R (nothing
        // is evicted) or spans at most R - W + 1 tokens; with R = W that is one token.
        long long len = n - off < kPrefillChunk ? n - off : kPrefillChunk;
        if (pos0 + len > R) {
            const long long lim = std::max(R - W + 1, R - pos0);
            len = std::max(1LL, std::min(len, lim));
        }
        const AppendCommon ac{m->rope, (int)len, Hk, D, (int)R, 1};
        const AppendJob aj{kb + (long long)off * Hk * D, vb + (long long)off * Hk * D, c->k_ring, c->v_ring, pos0, 0};
        record_touch(s, cs, 1);
        if (tracked(VST_K_ROPE_APPEND, s, [&] { return launch_rope_append(ac, &aj, 1, s); }) != cudaSuccess)
            return fail_all(cs, 1);
        int work = 0;
        for (int i = 0; i < (int)len; ++i) {
            const long long pos = pos0 + i;
            const long long lo = pos - W + 1 > 0 ? pos - W + 1 : 0;
            const int sig0 = (int)(lo / kDecSplit);
            const int nsp = (int)(pos / kDecSplit) - sig0 + 1;
            uint8_t* base = c->pf_mem + (size_t)i * per_token;
            const long long t = off + i;
            jobs[i] = DecJob{qb + t * H * D, kb + t * Hk * D, vb + t * Hk * D, ob + t * H * D, c->k_ring, c->v_ring,
                             c->tmap_k, c->tmap_v, reinterpret_cast<float*>(base),
                             reinterpret_cast<float*>(base + ml_bytes), reinterpret_cast<unsigned*>(base + ml_bytes + o_bytes),
                             c->err, pos, sig0, nsp, work, 0};
            work += nsp;
        }
        DecCommon dc{m->rope, (int)len, Hk, (int)R, (int)W, m->splits, 0, scale_log2, 1};
        dc.early = record_touch(s, cs, 1);  // 0: the append just wrote this ring
        if (tracked(VST_K_DEC_STEP, s, [&] { return launch_dec_step(dc, jobs, (int)len, work, s); }) != cudaSuccess)
            return fail_all(cs, 1);
        c->abs_next += len;
        off += (int32_t)len;
    }
    return VST_OK;
}

vst_status vst_dec_append(vst_ctx* c, const void* k, const void* v, int32_t n, void* stream)
{
    vst_ctx* cs[1] = {c};
    vst_status st = check_ctxs(cs, 1, VST_DEC);
    if (st != VST_OK)
        return st;
    if (n < 0)
        return VST_E_INVAL;
    if (n == 0)
        return VST_OK;
    if (!k || !v || !aligned16(k) || !aligned16(v))
        return VST_E_INVAL;
    const vst_config& cfg = c->m->cfg;
    if (c->abs_next + n > cfg.max_position)
        return VST_E_INVAL;
    DeviceGuard g(c->m->device);
    const auto* kb = static_cast<const __nv_bfloat16*>(k);
    const auto* vb = static_cast<const __nv_bfloat16*>(v);
    const int Hk = cfg.n_kv_heads, D = cfg.head_dim;
    // At most R rows per launch so that no two rows of one launch share a slot.
    for (int32_t off = 0; off < n; off += cfg.ring_slots) {
        const int32_t rows = n - off < cfg.ring_slots ? n - off : cfg.ring_slots;
        const AppendCommon ac{c->m->rope, rows, Hk, D, cfg.ring_slots, 1};
        const AppendJob aj{kb + (long long)off * Hk * D, vb + (long long)off * Hk * D, c->k_ring, c->v_ring,
                           c->abs_next, 0};
        cudaStream_t s = as_stream(stream);
        record_touch(s, cs, 1);
        if (tracked(VST_K_ROPE_APPEND, s, [&] { return launch_rope_append(ac, &aj, 1, s); }) != cudaSuccess)
            return fail_all(cs, 1);
        c->abs_next += rows;
    }
    return VST_OK;
}

}  // extern "C"

// ---- decoder step without allocation ---------------------------------------------------
// Same computation as vst_dec_step, but the per-call scratch (split partials and the merge
// counters) comes from one file-scope device array instead of the contexts' memory, so the
// call itself allocates nothing. The array is fixed at kNoAllocScratchBytes; its device
// address is looked up once per device with cudaGetSymbolAddress (in host code the symbol
// is only a stand-in, not a device address).
namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB per device, held until exit
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

// Device address of the scratch array on device `dev` (looked up on first use).
cudaError_t noalloc_scratch(int dev, unsigned char** out)
{
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = static_cast<unsigned char*>(g_noalloc_ptr[dev]);
    return cudaSuccess;
}

}  // namespace

extern "C" {

vst_status vst_dec_step_noalloc(vst_ctx* const* ctxs, int32_t n_streams, const void* q, const void* k, const void* v,
                                void* out, void* stream)
{
    vst_status st = check_ctxs(ctxs, n_streams, VST_DEC);
    if (st != VST_OK)
        return st;
    if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return VST_E_INVAL;
    const vst_module* m = ctxs[0]->m;
    const vst_config& cfg = m->cfg;
    for (int i = 0; i < n_streams; ++i)
        if (ctxs[i]->abs_next >= cfg.max_position)
            return VST_E_INVAL;
    const int H = cfg.n_heads, Hk = cfg.n_kv_heads, D = cfg.head_dim;
    // per stream: m, l [H][S][2] and o [H][S][D] floats, then Hk counters (256-B aligned)
    const size_t ml_bytes = align256((size_t)H * m->splits * 2 * sizeof(float));
    const size_t o_bytes = align256((size_t)H * m->splits * D * sizeof(float));
    const size_t cnt_bytes = align256((size_t)Hk * sizeof(unsigned));
    const size_t per_stream = ml_bytes + o_bytes + cnt_bytes;
    if ((size_t)n_streams * per_stream > kNoAllocScratchBytes || n_streams > kMaxJobs)
        return VST_E_INVAL;  // more streams than the fixed scratch holds
    DeviceGuard g(m->device);
    if (!g.ok)
        return fail_all(ctxs, n_streams);
    unsigned char* scratch = nullptr;
    if (noalloc_scratch(m->device, &scratch) != cudaSuccess)
        return fail_all(ctxs, n_streams);
    cudaStream_t s = as_stream(stream);
    const auto* qb = static_cast<const __nv_bfloat16*>(q);
    const auto* kb = static_cast<const __nv_bfloat16*>(k);
    const auto* vb = static_cast<const __nv_bfloat16*>(v);
    auto* ob = static_cast<__nv_bfloat16*>(out);
    DecCommon dc{m->rope, n_streams, Hk, cfg.ring_slots, cfg.window, m->splits, 0,
                 (float)(1.4426950408889634 / std::sqrt((double)D))};
    DecJob jobs[kMaxJobs];
    int work = 0;
    for (int i = 0; i < n_streams; ++i) {
        vst_ctx* c = ctxs[i];
        unsigned char* base = scratch + (size_t)i * per_stream;
        const long long pos = c->abs_next;
        const long long lo = pos - cfg.window + 1 > 0 ? pos - cfg.window + 1 : 0;
        const int sig0 = (int)(lo / kDecSplit);
        const int nsp = (int)(pos / kDecSplit) - sig0 + 1;
        jobs[i] = DecJob{qb + (long long)i * H * D, kb + (long long)i * Hk * D, vb + (long long)i * Hk * D,
                         ob + (long long)i * H * D, c->k_ring, c->v_ring, c->tmap_k, c->tmap_v,
                         reinterpret_cast<float*>(base), reinterpret_cast<float*>(base + ml_bytes),
                         reinterpret_cast<unsigned*>(base + ml_bytes + o_bytes), c->err, pos, sig0, nsp, work, 0};
        work += nsp;
    }
    // The merge counters must start at zero; the kernel re-arms them, but the array is
    // shared by every call, so clear this call's counters first (stream-ordered).
    for (int i = 0; i < n_streams; ++i)
        if (cudaMemsetAsync(scratch + (size_t)i * per_stream + ml_bytes + o_bytes, 0, cnt_bytes, s) != cudaSuccess)
            return fail_all(ctxs, n_streams);
    record_touch(s, ctxs, n_streams);  // dc.early stays 0: this launch follows the memsets
    if (tracked(VST_K_DEC_STEP, s, [&] { return launch_dec_step(dc, jobs, n_streams, work, s); }) != cudaSuccess)
        return fail_all(ctxs, n_streams);
    for (int i = 0; i < n_streams; ++i)
        ctxs[i]->abs_next += 1;
    return VST_OK;
}

}  // extern "C"
