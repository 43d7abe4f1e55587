// compact.cu -- kernel (d): ring compaction.
//
// Streaming plan, "Unbounded length (shipped)": periodic compaction copies the last 750
// frames to the front of the 1536-slot ring so memory stays constant for any stream
// length; slot 0 then holds absolute frame abs_base + (n_kv - 750).
//
// The move ring[s] <- ring[src + s], s in [0, keep), overlaps itself whenever src < keep.
// One CTA owns one (context, K|V plane, KV head) plane: every thread first loads its
// share of the source rows into registers, the CTA synchronises, and only then does any
// thread store. Planes are disjoint, so no two CTAs touch the same bytes.
#include "common.cuh"
#include "vst_internal.h"

namespace vst {

constexpr int kCompactThreads = 512;
constexpr int kCompactVecPerThread = 16;  // 16 x 16 B per thread: planes up to 128 KB

template <int J>
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const __grid_constant__ KParams<CompactCommon, CompactJob, J> p)
{
    const CompactCommon& c = p.c;
    const CompactJob& job = p.jobs[blockIdx.y];
    const int plane = blockIdx.x;  // 0 .. 2*Hk-1: K heads then V heads
    const int head = plane % c.Hk;
    __nv_bfloat16* ring = plane < c.Hk ? job.k_ring : job.v_ring;
    const long long row_elems = c.D;
    uint4* dst = reinterpret_cast<uint4*>(ring + (long long)head * c.R * row_elems);
    const uint4* src = reinterpret_cast<const uint4*>(ring + ((long long)head * c.R + job.src_row) * row_elems);
    const int n_vec = (int)(c.keep * row_elems * 2 / 16);

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

cudaError_t launch_compact(const CompactCommon& c, const CompactJob* jobs, int n_jobs, cudaStream_t s)
{
    if (n_jobs == 0)
        return cudaSuccess;
    if ((long long)c.keep * c.D * 2 > 16LL * kCompactThreads * kCompactVecPerThread)
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(2 * c.Hk), (unsigned)n_jobs);
    return with_params(c, jobs, n_jobs, [&](const auto& p) {
        compact_kernel<sizeof(p.jobs) / sizeof(p.jobs[0])><<<grid, kCompactThreads, 0, s>>>(p);
        return cudaGetLastError();
    });
}

}  // namespace vst
