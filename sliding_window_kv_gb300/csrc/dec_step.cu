// dec_step.cu -- kernel (c) with kernel (a)'s decoder half fused in: one decoder step for a
// batch of streams against their sliding KV rings.
//
// Family doc "Voxtral Realtime", Architecture (summary): decoder GQA 32q/8kv, head dim 128,
// sliding window 8192, NEOX RoPE theta=1e6. Capability Validation, Streaming row, item (5):
// token cur writes slot cur % n_ctx (evicting cur-8192), the step mask reveals
// [cur-8191, cur], positions stay absolute.
//
// Work item: one CTA per (stream, KV head, split), a split being the 128 absolute positions
// [128*sigma, 128*sigma + 128); the splits of a step are those that meet
// [max(0, pos-W+1), pos]. Each CTA
//   1. TMA-loads the split's K and V rows (slots 128*sigma mod R, 2 x 64-dim boxes each,
//      128-B swizzle) -- 64 KB per CTA, all in flight at once;
//   2. meanwhile rotates the 4 query heads of its group (fp32, scaled to log2 units) and,
//      if the split holds pos, rotates the new key: that row of the smem tile is replaced
//      by K'/V of this step and the same bytes are stored to ring slot pos % R;
//   3. scores: one thread per key, 4 heads; masked keys get -inf;
//   4. split-local softmax (max and sum by warp shuffles, then across the 4 warps in fixed
//      order) and P.V (two key halves, combined in fixed order);
//   5. writes its partial (m, l, o) and bumps a per-(stream, KV head) counter; the CTA that
//      finishes last folds all partials of its group in ascending split order and writes
//      the output, then re-arms the counter.
// The fold order depends only on absolute positions, so a stream's output is the same bits
// whether it runs alone or in a batch, and whatever the ring size.
#include "common.cuh"
#include "ptx.cuh"
#include "vst_internal.h"

namespace vst {

namespace {

constexpr int kThreads = 128;
constexpr int kD = 128;
constexpr int kG = 4;                      // query heads per KV head
constexpr uint32_t kBox = 128u * 128u;     // 128 keys x 64 dims x 2 B
constexpr uint32_t kOffK0 = 0;
constexpr uint32_t kOffK1 = kBox;
constexpr uint32_t kOffV0 = 2 * kBox;
constexpr uint32_t kOffV1 = 3 * kBox;
constexpr uint32_t kOffQ = 4 * kBox;               // float [4][128]
constexpr uint32_t kOffP = kOffQ + kG * kD * 4;    // float [4][128]
constexpr uint32_t kOffRed = kOffP + kG * kD * 4;  // float [64][8]
constexpr uint32_t kOffNew = kOffRed + 64 * 8 * 4; // bf16 K'[128], V[128]
constexpr uint32_t kOffWarp = kOffNew + 512;       // float [4 warps][4 heads] x 2
constexpr uint32_t kOffBar = kOffWarp + 2 * 16 * 4;
constexpr uint32_t kSmemBytes = kOffBar + 64 + 1024;

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x = __fadd_rn(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    return x;
}

}  // namespace

template <int J>
__global__ void __launch_bounds__(kThreads)
    dec_step_kernel(const __grid_constant__ KParams<DecCommon, DecJob, J> p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_last;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    float* sq = reinterpret_cast<float*>(smem + kOffQ);
    float* sp = reinterpret_cast<float*>(smem + kOffP);
    float* sred = reinterpret_cast<float*>(smem + kOffRed);
    __nv_bfloat16* snew = reinterpret_cast<__nv_bfloat16*>(smem + kOffNew);
    float* swarp = reinterpret_cast<float*>(smem + kOffWarp);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    const uint32_t bar = smem_u32(&bars[0]);

    const DecCommon& c = p.c;
    const int item = blockIdx.x;
    int j = 0;
    while (j + 1 < c.n_jobs && p.jobs[j + 1].work_begin <= item)
        ++j;
    const DecJob& job = p.jobs[j];
    const int g = blockIdx.y;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int sl = item - job.work_begin;          // split index within this step
    const long long key0 = (long long)(job.sigma0 + sl) * kDecSplit;
    const long long pos = job.pos;
    const long long lo = max(0LL, pos - c.W + 1);
    const int slot0 = (int)(key0 % c.R);
    const bool newest = pos >= key0 && pos < key0 + kDecSplit;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        tmap_acquire(job.tmap_k);
        tmap_acquire(job.tmap_v);
        mbar_arrive_expect_tx(bar, 4 * kBox);
        tma_load_3d(smem_u32(smem + kOffK0), job.tmap_k, bar, 0, slot0, g);
        tma_load_3d(smem_u32(smem + kOffK1), job.tmap_k, bar, 64, slot0, g);
        tma_load_3d(smem_u32(smem + kOffV0), job.tmap_v, bar, 0, slot0, g);
        tma_load_3d(smem_u32(smem + kOffV1), job.tmap_v, bar, 64, slot0, g);
    }

    // ---- rotate the 4 query heads of group g (fp32, then scaled to log2 units)
    {
        const int hh = warp;  // one warp per query head
        const __nv_bfloat16* q = job.q + (long long)(g * kG + hh) * kD;
        const float2* cs = c.rope + pos * (kD / 2);
        const uint32_t a = *reinterpret_cast<const uint32_t*>(q + 2 * lane);
        const uint32_t b = *reinterpret_cast<const uint32_t*>(q + 64 + 2 * lane);
        float y1, y2, y3, y4;
        rope_pair(bf16lo(a), bf16lo(b), cs[2 * lane], y1, y2);
        rope_pair(bf16hi(a), bf16hi(b), cs[2 * lane + 1], y3, y4);
        sq[hh * kD + 2 * lane] = __fmul_rn(y1, c.scale_log2);
        sq[hh * kD + 2 * lane + 1] = __fmul_rn(y3, c.scale_log2);
        sq[hh * kD + 64 + 2 * lane] = __fmul_rn(y2, c.scale_log2);
        sq[hh * kD + 64 + 2 * lane + 1] = __fmul_rn(y4, c.scale_log2);
    }
    // ---- the new key (rotated) and value of this step, if this split holds pos
    if (newest && warp == 0) {
        const __nv_bfloat16* k = job.k + (long long)g * kD;
        const __nv_bfloat16* v = job.v + (long long)g * kD;
        const float2* cs = c.rope + pos * (kD / 2);
        const uint32_t a = *reinterpret_cast<const uint32_t*>(k + 2 * lane);
        const uint32_t b = *reinterpret_cast<const uint32_t*>(k + 64 + 2 * lane);
        float y1, y2, y3, y4;
        rope_pair(bf16lo(a), bf16lo(b), cs[2 * lane], y1, y2);
        rope_pair(bf16hi(a), bf16hi(b), cs[2 * lane + 1], y3, y4);
        reinterpret_cast<uint32_t*>(snew)[lane] = pack_bf16(y1, y3);
        reinterpret_cast<uint32_t*>(snew)[32 + lane] = pack_bf16(y2, y4);
        reinterpret_cast<uint32_t*>(snew + kD)[lane] = *reinterpret_cast<const uint32_t*>(v + 2 * lane);
        reinterpret_cast<uint32_t*>(snew + kD)[32 + lane] = *reinterpret_cast<const uint32_t*>(v + 64 + 2 * lane);
    }
    __syncthreads();
    const bool loaded = mbar_wait(bar, 0);
    if (newest && tid < 16) {
        // chunk tid of the 256-byte row: dims [8*tid, 8*tid+8)
        const int rr = (int)(pos - key0);
        const int half = tid >> 3, ch = tid & 7;
        const uint4 kw = reinterpret_cast<const uint4*>(snew)[tid];
        const uint4 vw = reinterpret_cast<const uint4*>(snew + kD)[tid];
        *reinterpret_cast<uint4*>(smem + (half ? kOffK1 : kOffK0) + sw128_offset(rr, ch)) = kw;
        *reinterpret_cast<uint4*>(smem + (half ? kOffV1 : kOffV0) + sw128_offset(rr, ch)) = vw;
        const long long gofs = ((long long)g * c.R + pos % c.R) * kD + 8 * tid;
        *reinterpret_cast<uint4*>(job.k_ring + gofs) = kw;
        *reinterpret_cast<uint4*>(job.v_ring + gofs) = vw;
    }
    if (__syncthreads_or(!loaded)) {
        if (tid == 0)
            atomicExch(job.err, kErrTimeout);
    }

    // ---- scores: thread tid owns key key0 + tid
    const long long kp = key0 + tid;
    const bool valid = kp >= lo && kp <= pos && loaded;
    float s[kG] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int cidx = 0; cidx < 16; ++cidx) {
        const uint8_t* kt = smem + ((cidx >> 3) ? kOffK1 : kOffK0);
        const uint4 kw = *reinterpret_cast<const uint4*>(kt + sw128_offset(tid, cidx & 7));
        const float kf[8] = {bf16lo(kw.x), bf16hi(kw.x), bf16lo(kw.y), bf16hi(kw.y),
                             bf16lo(kw.z), bf16hi(kw.z), bf16lo(kw.w), bf16hi(kw.w)};
#pragma unroll
        for (int hh = 0; hh < kG; ++hh) {
            const float4 qa = reinterpret_cast<const float4*>(sq + hh * kD + 8 * cidx)[0];
            const float4 qb = reinterpret_cast<const float4*>(sq + hh * kD + 8 * cidx)[1];
            float acc = s[hh];
            acc = __fmaf_rn(qa.x, kf[0], acc);
            acc = __fmaf_rn(qa.y, kf[1], acc);
            acc = __fmaf_rn(qa.z, kf[2], acc);
            acc = __fmaf_rn(qa.w, kf[3], acc);
            acc = __fmaf_rn(qb.x, kf[4], acc);
            acc = __fmaf_rn(qb.y, kf[5], acc);
            acc = __fmaf_rn(qb.z, kf[6], acc);
            acc = __fmaf_rn(qb.w, kf[7], acc);
            s[hh] = acc;
        }
    }
#pragma unroll
    for (int hh = 0; hh < kG; ++hh)
        if (!valid)
            s[hh] = -INFINITY;

    // ---- split-local softmax per head
#pragma unroll
    for (int hh = 0; hh < kG; ++hh) {
        const float wm = warp_max(s[hh]);
        if (lane == 0)
            swarp[warp * kG + hh] = wm;
    }
    __syncthreads();
    float mh[kG], lh[kG];
#pragma unroll
    for (int hh = 0; hh < kG; ++hh) {
        float m = swarp[hh];
        for (int w = 1; w < 4; ++w)
            m = fmaxf(m, swarp[w * kG + hh]);
        mh[hh] = m;
        const float pv = valid ? ex2(__fsub_rn(s[hh], m)) : 0.f;
        sp[hh * kD + tid] = pv;
        const float ws = warp_sum(pv);
        if (lane == 0)
            swarp[16 + warp * kG + hh] = ws;
    }
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < kG; ++hh) {
        float l = swarp[16 + hh];
        for (int w = 1; w < 4; ++w)
            l = __fadd_rn(l, swarp[16 + w * kG + hh]);
        lh[hh] = l;
    }

    // ---- P.V: thread -> dims (2dp, 2dp+1), keys [64kh, 64kh+64)
    const int dp = tid & 63, kh = tid >> 6;
    const int d = 2 * dp;
    const uint8_t* vt = smem + ((d >> 6) ? kOffV1 : kOffV0);
    const int ch = (d & 63) >> 3;
    const int within = (d & 7) * 2;
    float acc[kG][2];
#pragma unroll
    for (int hh = 0; hh < kG; ++hh)
        acc[hh][0] = acc[hh][1] = 0.f;
#pragma unroll 8
    for (int kk = 0; kk < 64; ++kk) {
        const int key = 64 * kh + kk;
        const uint32_t vw = *reinterpret_cast<const uint32_t*>(vt + sw128_offset(key, ch) + within);
        const float v0 = bf16lo(vw), v1 = bf16hi(vw);
#pragma unroll
        for (int hh = 0; hh < kG; ++hh) {
            const float pp = sp[hh * kD + key];
            acc[hh][0] = __fmaf_rn(pp, v0, acc[hh][0]);
            acc[hh][1] = __fmaf_rn(pp, v1, acc[hh][1]);
        }
    }
    if (kh == 1) {
#pragma unroll
        for (int hh = 0; hh < kG; ++hh) {
            sred[dp * 8 + 2 * hh] = acc[hh][0];
            sred[dp * 8 + 2 * hh + 1] = acc[hh][1];
        }
    }
    __syncthreads();
    if (kh == 0) {
#pragma unroll
        for (int hh = 0; hh < kG; ++hh) {
            const float o0 = __fadd_rn(acc[hh][0], sred[dp * 8 + 2 * hh]);
            const float o1 = __fadd_rn(acc[hh][1], sred[dp * 8 + 2 * hh + 1]);
            const int hq = g * kG + hh;
            *reinterpret_cast<float2*>(job.part_o + ((long long)hq * c.S + sl) * kD + d) = make_float2(o0, o1);
        }
    }
    if (tid < kG) {
        const int hq = g * kG + tid;
        *reinterpret_cast<float2*>(job.part_ml + ((long long)hq * c.S + sl) * 2) = make_float2(mh[tid], lh[tid]);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(job.counters + g, 1u);
        s_last = (prev == (unsigned)(job.n_splits - 1));
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();

    // ---- last CTA of (stream, g): fold the splits in ascending order
    {
        const int hh = warp;
        const int hq = g * kG + hh;
        const int d4 = lane * 4;
        float m = -INFINITY, l = 0.f;
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        for (int sj = 0; sj < job.n_splits; ++sj) {
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(job.part_ml + ((long long)hq * c.S + sj) * 2));
            const float4 oj = __ldcg(reinterpret_cast<const float4*>(job.part_o + ((long long)hq * c.S + sj) * kD + d4));
            const float mn = fmaxf(m, ml.x);
            const float a = ex2(__fsub_rn(m, mn));
            const float b = ex2(__fsub_rn(ml.x, mn));
            l = __fmaf_rn(l, a, __fmul_rn(ml.y, b));
            o[0] = __fmaf_rn(o[0], a, __fmul_rn(oj.x, b));
            o[1] = __fmaf_rn(o[1], a, __fmul_rn(oj.y, b));
            o[2] = __fmaf_rn(o[2], a, __fmul_rn(oj.z, b));
            o[3] = __fmaf_rn(o[3], a, __fmul_rn(oj.w, b));
            m = mn;
        }
        const uint32_t w0 = pack_bf16(__fdiv_rn(o[0], l), __fdiv_rn(o[1], l));
        const uint32_t w1 = pack_bf16(__fdiv_rn(o[2], l), __fdiv_rn(o[3], l));
        *reinterpret_cast<uint2*>(job.out + (long long)hq * kD + d4) = make_uint2(w0, w1);
    }
    if (tid == 0)
        job.counters[g] = 0u;
}

template <int J>
static cudaError_t launch_dec_j(const KParams<DecCommon, DecJob, J>& p, int total_work, cudaStream_t s)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(dec_step_kernel<J>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess)
            return e;
        configured[dev] = 1;
    }
    const dim3 grid((unsigned)total_work, (unsigned)p.c.Hk);
    dec_step_kernel<J><<<grid, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_dec_step(const DecCommon& c, const DecJob* jobs, int n_jobs, int total_work,
                            cudaStream_t s)
{
    if (n_jobs == 0 || total_work == 0)
        return cudaSuccess;
    return with_params(c, jobs, n_jobs, [&](const auto& p) {
        return launch_dec_j<sizeof(p.jobs) / sizeof(p.jobs[0])>(p, total_work, s);
    });
}

}  // namespace vst
