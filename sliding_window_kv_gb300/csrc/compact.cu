// compact.cu -- kernel (d): ring compaction.
//
// Streaming plan, "Unbounded length (shipped)": periodic compaction copies the last 750
// frames to the front of the 1536-slot ring so memory stays constant for any stream
// length; slot 0 then holds absolute frame abs_base + (n_kv - 750).
//
// The move ring[s] <- ring[src + s], s in [0, keep), overlaps itself whenever src < keep.
// When some job's move does, one CTA owns each (context, K|V plane, KV head) plane: every
// thread first loads its share of the source rows into registers, the CTA synchronises, and
// only then does any thread store. When no job's move overlaps (src >= keep, the usual
// case), each plane is split by rows over `split` CTAs: source and destination rows are then
// disjoint, so no CTA can overwrite rows that another still reads. Planes are disjoint, so
// no two planes share bytes either.
//
// Launched with programmatic dependent launch; the next kernel may start its prologue at
// once (every kernel of the library waits for its predecessor before touching a ring). The
// copy waits for the previous kernel in the stream, which may still read this ring, unless
// the host says that kernel touched none of these rings (early): the copy then runs beside
// the previous kernel's tail, and the wait comes after it, so that this grid still completes
// only after its predecessor (whatever follows in the stream may rely on that order).
#include "common.cuh"
#include "ptx.cuh"
#include "vst_internal.h"

namespace vst {

constexpr int kCompactThreads = 512;
constexpr int kCompactVecPerThread = 16;  // 16 x 16 B per thread: planes up to 128 KB

// This CTA's rows: every thread loads its share into registers, the CTA synchronises, then
// every thread stores.
__device__ __forceinline__ void copy_plane(const uint4* src, uint4* dst, int n_vec)
{
    uint4 r[kCompactVecPerThread];
#pragma unroll
    for (int i = 0; i < kCompactVecPerThread; ++i) {
        const int e = threadIdx.x + i * kCompactThreads;
        if (e < n_vec)
            r[i] = src[e];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kCompactVecPerThread; ++i) {
        const int e = threadIdx.x + i * kCompactThreads;
        if (e < n_vec)
            dst[e] = r[i];
    }
}

template <int J>
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const __grid_constant__ KParams<CompactCommon, CompactJob, J> p)
{
    const CompactCommon& c = p.c;
    const CompactJob& job = p.jobs[blockIdx.y];
    // The next kernel is released only once the wait has returned, so that when it starts,
    // every kernel before this one has completed (what its own early loads rely on).
    if (!c.early) {
        griddep_wait();
        griddep_launch_dependents();
    }
    const int plane = blockIdx.x / c.split;  // 0 .. 2*Hk-1: K heads then V heads
    const int part = blockIdx.x % c.split;
    const int head = plane % c.Hk;
    const int rows_per = (c.keep + c.split - 1) / c.split;
    const int row_lo = part * rows_per, row_hi = min(c.keep, row_lo + rows_per);
    if (row_lo < row_hi) {
        __nv_bfloat16* ring = plane < c.Hk ? job.k_ring : job.v_ring;
        const long long row_elems = c.D;
        uint4* dst = reinterpret_cast<uint4*>(ring + ((long long)head * c.R + row_lo) * row_elems);
        const uint4* src =
            reinterpret_cast<const uint4*>(ring + ((long long)head * c.R + job.src_row + row_lo) * row_elems);
        copy_plane(src, dst, (int)((row_hi - row_lo) * row_elems * 2 / 16));
    }
    if (c.early) {
        griddep_wait();
        griddep_launch_dependents();
    }
}

cudaError_t launch_compact(const CompactCommon& c0, const CompactJob* jobs, int n_jobs, cudaStream_t s)
{
    if (n_jobs == 0)
        return cudaSuccess;
    if ((long long)c0.keep * c0.D * 2 > 16LL * kCompactThreads * kCompactVecPerThread)
        return cudaErrorInvalidValue;
    CompactCommon c = c0;
    c.split = kCompactSplit;
    for (int i = 0; i < n_jobs; ++i)
        if (jobs[i].src_row < c.keep)
            c.split = 1;  // the move overlaps itself: one CTA reads a whole plane before writing
    const dim3 grid((unsigned)(2 * c.Hk * c.split), (unsigned)n_jobs);
    return with_params(c, jobs, n_jobs, [&](const auto& p) {
        return launch_pdl(compact_kernel<sizeof(p.jobs) / sizeof(p.jobs[0])>, grid, dim3(kCompactThreads), 0, s, p);
    });
}

}  // namespace vst
