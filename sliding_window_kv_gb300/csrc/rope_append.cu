// rope_append.cu -- kernel (a): rotate new keys at their absolute positions and append
// K' and V to the ring.
//
// Streaming plan ("Voxtral Realtime -- incremental streaming implementation plan"),
// SHIPPED/Mechanism: the chunk's K/V are written at cache rows [n_kv_before, n_kv_total);
// "Chunk alignment": RoPE at absolute positions. Decoder (family doc, Streaming row,
// item (5)): token cur writes slot cur % n_ctx.
//
// One thread owns 8 elements of the first half of a head vector and the 8 matching
// elements of the second half (the NEOX pairs), so every load and store is a 16-byte
// vector and the (cos, sin) table row is read once per pair.
#include "common.cuh"
#include "ptx.cuh"
#include "vst_internal.h"

namespace vst {

template <int J>
__global__ void __launch_bounds__(256) rope_append_kernel(const __grid_constant__ KParams<AppendCommon, AppendJob, J> p)
{
    const AppendCommon& c = p.c;
    const AppendJob& job = p.jobs[blockIdx.y];
    // Programmatic dependent launch: the previous kernel may still read the rows this one
    // overwrites, so wait for it; the next kernel waits for this one before it reads them.
    griddep_wait();
    griddep_launch_dependents();
    const int half = c.D / 2;
    const int per_vec = half / 8;  // threads per head vector
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total = (long long)c.n_rows * c.Hk * per_vec;
    if (idx >= total)
        return;
    const int part = (int)(idx % per_vec);
    const long long rh = idx / per_vec;  // row * Hk + head
    const int head = (int)(rh % c.Hk);
    const long long row = rh / c.Hk;
    const long long pos = job.pos0 + row;
    const long long slot = c.modulo ? (pos % c.R) : (job.slot0 + row);

    const int i0 = part * 8;
    const __nv_bfloat16* kin = job.k + rh * c.D;
    const __nv_bfloat16* vin = job.v + rh * c.D;
    const uint4 k1 = *reinterpret_cast<const uint4*>(kin + i0);
    const uint4 k2 = *reinterpret_cast<const uint4*>(kin + i0 + half);
    const uint4 v1 = *reinterpret_cast<const uint4*>(vin + i0);
    const uint4 v2 = *reinterpret_cast<const uint4*>(vin + i0 + half);
    const float2* cs = c.rope + pos * half + i0;

    const uint32_t a[4] = {k1.x, k1.y, k1.z, k1.w};
    const uint32_t b[4] = {k2.x, k2.y, k2.z, k2.w};
    uint32_t ya[4], yb[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float y1a, y2a, y1b, y2b;
        rope_pair(bf16lo(a[w]), bf16lo(b[w]), cs[2 * w], y1a, y2a);
        rope_pair(bf16hi(a[w]), bf16hi(b[w]), cs[2 * w + 1], y1b, y2b);
        ya[w] = pack_bf16(y1a, y1b);
        yb[w] = pack_bf16(y2a, y2b);
    }
    const long long base = ((long long)head * c.R + slot) * c.D;
    *reinterpret_cast<uint4*>(job.k_ring + base + i0) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
    *reinterpret_cast<uint4*>(job.k_ring + base + i0 + half) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
    *reinterpret_cast<uint4*>(job.v_ring + base + i0) = v1;
    *reinterpret_cast<uint4*>(job.v_ring + base + i0 + half) = v2;
}

cudaError_t launch_rope_append(const AppendCommon& c, const AppendJob* jobs, int n_jobs,
                               cudaStream_t s)
{
    const long long total = (long long)c.n_rows * c.Hk * (c.D / 16);
    if (total == 0 || n_jobs == 0)
        return cudaSuccess;
    const int threads = 256;
    const dim3 grid((unsigned)((total + threads - 1) / threads), (unsigned)n_jobs);
    return with_params(c, jobs, n_jobs, [&](const auto& p) {
        return launch_pdl(rope_append_kernel<sizeof(p.jobs) / sizeof(p.jobs[0])>, grid, dim3(threads), 0, s, p);
    });
}

}  // namespace vst
