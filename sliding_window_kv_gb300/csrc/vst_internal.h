// vst_internal.h -- structures shared by the host API (vst_api.cu) and the kernels.
//
// Device memory of one ctx is one block:
//   [0, 256)          header: error word (int32 at 0), merge counters (uint32 at 64, one per
//                     KV head, decoder only)
//   [256, 512)        two CUtensorMap (128 B each, 64-B aligned): K ring, V ring
//   [512, ...)        K ring [Hk][R][D] bf16, then V ring [Hk][R][D] bf16
//   then              partial softmax state per (query head, split or key tile): m, l
//                     [H][S][(128)][2] fp32 and o [H][S][(128)][D] fp32; decoder: S splits
//                     per step, one query row each; encoder: S key tiles of 128 rows (split
//                     launch shape of the chunk attention)
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

#include "../../include/vst.h"

namespace vst {

constexpr int kCtxHeaderBytes = 512;
constexpr int kErrOffset = 0;
constexpr int kCounterOffset = 64;
constexpr int kTmapOffset = 256;

// Decoder: keys are processed in tiles of kDecTile absolute positions and reduced into one
// partial per split of kDecSplit absolute positions (the ring must be a multiple of a tile).
constexpr int kDecTile = 128;
constexpr int kDecSplit = 512;
// Encoder attention tiles: 128 queries x 128 keys (absolute-position aligned). A query tile
// of up to 128 rows meets at most enc_split_tiles(W) key tiles.
constexpr int kEncTileM = 128;
constexpr int kEncTileN = 128;

constexpr int kMaxJobs = 64;  // contexts per launch
constexpr int kPrefillChunk = kMaxJobs;  // decoder prefill: tokens per attention launch (one job each)

// Error codes written into the ctx error word by kernels.
constexpr int kErrTimeout = 1;

struct AppendJob {
    const __nv_bfloat16* k;  // [n_rows][Hk][D] input
    const __nv_bfloat16* v;
    __nv_bfloat16* k_ring;   // [Hk][R][D]
    __nv_bfloat16* v_ring;
    long long pos0;          // absolute position of input row 0
    long long slot0;         // ring slot of row 0 (contiguous mode)
};

struct AppendCommon {
    const float2* rope;      // [max_position][D/2] (cos, sin)
    int n_rows, Hk, D, R;
    int modulo;              // 1: slot = position % R (decoder); 0: slot0 + row (encoder)
};

struct CompactJob {
    __nv_bfloat16* k_ring;
    __nv_bfloat16* v_ring;
    long long src_row;       // rows [src_row, src_row + keep) move to [0, keep)
};

struct CompactCommon {
    int Hk, R, D, keep;
    int split;  // CTAs per (K|V, head) plane; set by the launcher
    int early;  // 1: the previous kernel in the stream touched none of these rings
};
constexpr int kCompactSplit = 2;  // CTAs per plane when no job's move overlaps itself

struct EncAttnJob {
    const __nv_bfloat16* q;  // [n_rows][H][D] input rows of this batch
    const __nv_bfloat16* k;  // [n_rows][H][D] (encoder: Hk = H), not rotated yet
    const __nv_bfloat16* v;
    __nv_bfloat16* out;      // [n_rows][H][D]
    __nv_bfloat16* k_ring;   // [H][R][D]: the batch's rows go to slots slot0 + row
    __nv_bfloat16* v_ring;
    const CUtensorMap* tmap_k;  // over the K ring, dims {D, R, Hk}, box {64, 128, 1}, SW128
    const CUtensorMap* tmap_v;
    float* part_ml;          // split mode scratch: [H][split_tiles][128][2] (m_t, l_t)
    float* part_o;           // split mode scratch: [H][split_tiles][4 quarters][128][D / 4]
    unsigned* counters;      // split mode: [H] CTAs of each head that have published their partials
    int* err;
    long long pos0;          // absolute position of row 0
    long long abs_base;      // absolute position held by ring slot 0
    long long slot0;         // ring slot of row 0 (n_kv before the batch)
    int q_z;                 // loop shape: this job's index in tmap_q's outer dimension
};

struct EncAttnCommon {
    const float2* rope;
    int n_rows, H, W, R;
    int split;               // 0: loop mode; k > 0: split mode, k key tiles per CTA
    int split_tiles;         // scratch tiles per head
    int early;               // 1: ring loads may start before the previous kernel completes
    int appended;            // 1: the batch's K'/V rows are already in the ring (loop shape)
    float scale_log2;        // log2(e) / sqrt(D)
    int right;               // keys after the query that the mask shows (loop shape; 0: causal)
    int lpt;                 // loop shape: launch the last query tiles of every (context, head) first
    const CUtensorMap* tmap_rope;  // loop shape: over the (cos, sin) table, fp32 {D, positions}, box {D, 128}
    CUtensorMap tmap_q;      // loop shape: over this launch's queries {D, H, rows, jobs}, box {D, 1, 128, 1}, SW128
};

struct DecJob {
    const __nv_bfloat16* q;  // [H][D] this stream's query
    const __nv_bfloat16* k;  // [Hk][D] this step's key (not rotated yet)
    const __nv_bfloat16* v;  // [Hk][D]
    __nv_bfloat16* out;      // [H][D]
    __nv_bfloat16* k_ring;
    __nv_bfloat16* v_ring;
    const CUtensorMap* tmap_k;  // dims {D, R, Hk}, box {64, 128, 1}, SW128
    const CUtensorMap* tmap_v;
    float* part_ml;          // [H][S][2]
    float* part_o;           // [H][S][D]
    unsigned* counters;      // [Hk]
    int* err;
    long long pos;           // absolute position of this step's token
    int sigma0;              // first split (absolute block index) of this step
    int n_splits;
    int work_begin;          // first work item (blockIdx.x) of this job
    int pad;
};

struct DecCommon {
    const float2* rope;
    int n_jobs, Hk, R, W, S;
    int early;               // 1: ring loads may start before the previous kernel completes
    float scale_log2;
    int appended;            // 1: every job's K'/V row is already in the ring (prefill chunks)
};

// Kernel parameters: the common block plus up to J jobs, passed by value. Launchers pick
// the smallest J that holds the jobs so one-context launches stay small.
template <class Common, class Job, int J>
struct KParams {
    Common c;
    Job jobs[J];
};

// Kernel launchers (one per kernel file). They only enqueue; errors are returned as
// cudaError_t from cudaGetLastError.
// n_jobs <= kMaxJobs.
cudaError_t launch_rope_append(const AppendCommon& c, const AppendJob* jobs, int n_jobs,
                               cudaStream_t s);
cudaError_t launch_compact(const CompactCommon& c, const CompactJob* jobs, int n_jobs,
                           cudaStream_t s);
cudaError_t launch_enc_attn(const EncAttnCommon& c, const EncAttnJob* jobs, int n_jobs, int grid_x,
                            cudaStream_t s);
cudaError_t launch_enc_attn_split(const EncAttnCommon& c, const EncAttnJob* jobs, int n_jobs, int grid_x,
                            cudaStream_t s);
cudaError_t launch_dec_step(const DecCommon& c, const DecJob* jobs, int n_jobs, int total_work,
                            cudaStream_t s);
// CTAs of the split shape that one SM holds at once (0 on error); the split shape's merger
// waits for the other CTAs of its grid, so its grid must fit the SMs at this occupancy.
cudaError_t enc_attn_split_blocks_per_sm(int* n);

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current device, once per
// device: `done` (one per kernel instantiation, bit d for device d < 64) records where it is
// set. Safe from several host threads: a first call racing another sets the same attribute
// twice, which the runtime allows.
template <class Kernel>
cudaError_t smem_limit_once(std::atomic<unsigned long long>& done, Kernel kernel, int bytes)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && ((done.load(std::memory_order_acquire) >> dev) & 1ull))
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev < 64)
        done.fetch_or(1ull << dev, std::memory_order_release);
    return e;
}

// Launch with programmatic stream serialization: the kernel may start while the previous
// kernel in the stream is finishing; it runs griddep_wait() before touching anything that
// kernel may produce or consume. Every kernel of the library releases its dependents
// (griddep_launch_dependents) only after its own griddep_wait has returned, so when a
// launch starts, every kernel before its immediate predecessor has completed: what it
// does before its wait overlaps that one predecessor and nothing earlier.
template <class Kernel, class Params>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const Params& p)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Copy jobs into a KParams<J> with the smallest J in {1, 8, 64} that fits and call
// f(params) with it.
template <class Common, class Job, class F>
cudaError_t with_params(const Common& c, const Job* jobs, int n_jobs, F&& f)
{
    if (n_jobs <= 1) {
        KParams<Common, Job, 1> p;
        p.c = c;
        p.jobs[0] = jobs[0];
        return f(p);
    }
    if (n_jobs <= 8) {
        KParams<Common, Job, 8> p;
        p.c = c;
        for (int i = 0; i < n_jobs; ++i) p.jobs[i] = jobs[i];
        return f(p);
    }
    KParams<Common, Job, kMaxJobs> p;
    p.c = c;
    for (int i = 0; i < n_jobs; ++i) p.jobs[i] = jobs[i];
    return f(p);
}

}  // namespace vst
