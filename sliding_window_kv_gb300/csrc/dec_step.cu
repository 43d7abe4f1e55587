// dec_step.cu -- kernel (c) with kernel (a)'s decoder half fused in: one decoder step for a
// batch of streams against their sliding KV rings.
//
// Family doc "Voxtral Realtime", Architecture (summary): decoder GQA 32q/8kv, head dim 128,
// sliding window 8192, NEOX RoPE theta=1e6. Capability Validation, Streaming row, item (5):
// token cur writes slot cur % n_ctx (evicting cur-8192), the step mask reveals
// [cur-8191, cur], positions stay absolute.
//
// Work item: one CTA per (stream, KV head g, split), a split being the 512 absolute
// positions [512*sigma, 512*sigma + 512) -- four key tiles of 128 -- cut to the step's
// window [max(0, pos-W+1), pos]. The CTA streams its tiles through a two-stage TMA ring
// (K and V of a tile, 64 KB per stage, 128-B swizzle, slots 128*tau mod R) and for each tile:
//   S^T = K Q'^T     tcgen05.mma M=128 keys, N=16 (the 4 query heads of the group, zero
//                    padded), K=128 dims; A = K tile (K-major), B = Q' (K-major); in TMEM
//   softmax          one key per thread (TMEM lane); per head: tile max and sum by warp
//                    shuffles then across the 4 warps in fixed order; P^T -> smem (bf16)
//   O^T = V^T P^T    tcgen05.mma M=128 dims, N=16, K=128 keys; A = V tile read as
//                    MN-major (dims contiguous), B = P^T (K-major); in TMEM
//   fold             thread d folds (m_t, l_t, O_t[d]) of the 4 heads into registers.
// The query heads are rotated in the prologue; if the split holds pos, the new key is
// rotated too, patched into its tile row in shared memory, and stored (K', V) to ring slot
// pos % R by this CTA. Each CTA writes its split's (m, l, o) per head; the last CTA of
// (stream, g) folds the splits in ascending order and writes the output. Tiles and splits
// are fixed by absolute position, so a stream's output is the same bits alone or in a
// batch, and whatever the ring size.
#include "common.cuh"
#include "ptx.cuh"
#include "vst_internal.h"

namespace vst {

namespace {

constexpr int kThreads = 128;
constexpr int kD = 128;
constexpr int kG = 4;                       // query heads per KV head
constexpr int kTile = kDecTile;             // keys per tile
constexpr int kTilesPerSplit = kDecSplit / kTile;
constexpr uint32_t kBox = 128u * 128u;      // 128 keys x 64 dims x 2 B
constexpr uint32_t kStage = 4 * kBox;       // K lo, K hi, V lo, V hi
constexpr uint32_t kOffQ = 2 * kStage;      // Q' [16 rows][128 dims]: 2 blocks of 2 KB
constexpr uint32_t kOffP = kOffQ + 4096;    // P^T [16 rows][128 keys]: 2 blocks of 2 KB
constexpr uint32_t kOffNew = kOffP + 4096;  // new K' row, new V row (bf16 x 128 each)
constexpr uint32_t kOffRed = kOffNew + 512; // float [2][4 warps][4 heads]
constexpr uint32_t kOffBar = kOffRed + 128;
constexpr uint32_t kSmemBytes = kOffBar + 64 + 1024;
constexpr uint32_t kTmemCols = 32;          // S^T in [0,16), O^T in [16,32)

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 16, false, false);
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 16, true, false);

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

// Fold a tile-local (or split-local) softmax state into a running one (one value of o).
__device__ __forceinline__ void fold1(float& m, float& l, float& o, float mt, float lt, float ot)
{
    const float mn = fmaxf(m, mt);
    const float a = ex2(__fsub_rn(m, mn));
    const float b = ex2(__fsub_rn(mt, mn));
    l = __fmaf_rn(l, a, __fmul_rn(lt, b));
    o = __fmaf_rn(o, a, __fmul_rn(ot, b));
    m = mn;
}

__device__ __forceinline__ uint32_t sw16(int row, int col)
{
    // byte offset of element col (0..127) of row `row` in a [16][128] bf16 K-major operand
    // stored as two 64-column blocks of 2 KB
    return (uint32_t)((col >> 6) * 2048) + sw128_offset(row, (col & 63) >> 3) + (uint32_t)((col & 7) * 2);
}

}  // namespace

template <int J>
__global__ void __launch_bounds__(kThreads, 1)
    dec_step_kernel(const __grid_constant__ KParams<DecCommon, DecJob, J> p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    __shared__ int s_last;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sP = smem + kOffP;
    __nv_bfloat16* snew = reinterpret_cast<__nv_bfloat16*>(smem + kOffNew);
    float* sred = reinterpret_cast<float*>(smem + kOffRed);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    const uint32_t bar_full0 = smem_u32(&bars[0]);
    const uint32_t bar_full1 = smem_u32(&bars[1]);
    const uint32_t bar_m = smem_u32(&bars[2]);

    const DecCommon& c = p.c;
    const int item = blockIdx.x;
    int j = 0;
    while (j + 1 < c.n_jobs && p.jobs[j + 1].work_begin <= item)
        ++j;
    const DecJob& job = p.jobs[j];
    const int g = blockIdx.y;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int sl = item - job.work_begin;  // split index within this step
    const long long pos = job.pos;
    const long long lo = max(0LL, pos - c.W + 1);
    const long long sig = job.sigma0 + sl;
    const long long tau_lo = max(sig * kTilesPerSplit, lo / kTile);
    const long long tau_hi = min(sig * kTilesPerSplit + kTilesPerSplit - 1, pos / kTile);
    const int n_tiles = (int)(tau_hi - tau_lo + 1);
    const long long tau_new = pos / kTile;  // tile holding this step's key

    auto issue_tile = [&](int i) {
        const int st = i & 1;
        const uint32_t base = smem_u32(smem) + st * kStage;
        const uint32_t bar = st ? bar_full1 : bar_full0;
        const int slot = (int)(((tau_lo + i) * kTile) % c.R);
        mbar_arrive_expect_tx(bar, kStage);
        tma_load_3d(base, job.tmap_k, bar, 0, slot, g);
        tma_load_3d(base + kBox, job.tmap_k, bar, 64, slot, g);
        tma_load_3d(base + 2 * kBox, job.tmap_v, bar, 0, slot, g);
        tma_load_3d(base + 3 * kBox, job.tmap_v, bar, 64, slot, g);
    };

    if (tid == 0) {
        mbar_init(bar_full0, 1);
        mbar_init(bar_full1, 1);
        mbar_init(bar_m, 1);
        fence_mbar_init();
        tmap_acquire(job.tmap_k);
        tmap_acquire(job.tmap_v);
        issue_tile(0);
        if (n_tiles > 1)
            issue_tile(1);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }

    // ---- Q' (4 rotated heads, bf16) and zero padding rows 4..15 of Q' and P^T
    for (int e = tid; e < 12 * 16; e += kThreads) {  // 12 rows x 16 chunks of zeros, both tiles
        const int row = 4 + e / 16, ch = e % 16;
        const uint32_t off = (uint32_t)((ch >> 3) * 2048) + sw128_offset(row, ch & 7);
        *reinterpret_cast<uint4*>(sQ + off) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sP + off) = make_uint4(0, 0, 0, 0);
    }
    {
        const int hh = warp;  // one warp per query head, lane owns pairs (2l, 2l+1)
        const __nv_bfloat16* q = job.q + (long long)(g * kG + hh) * kD;
        const float2* cs = c.rope + pos * (kD / 2);
        const uint32_t a = *reinterpret_cast<const uint32_t*>(q + 2 * lane);
        const uint32_t b = *reinterpret_cast<const uint32_t*>(q + 64 + 2 * lane);
        float y1, y2, y3, y4;
        rope_pair(bf16lo(a), bf16lo(b), cs[2 * lane], y1, y2);
        rope_pair(bf16hi(a), bf16hi(b), cs[2 * lane + 1], y3, y4);
        *reinterpret_cast<uint32_t*>(sQ + sw16(hh, 2 * lane)) = pack_bf16(y1, y3);
        *reinterpret_cast<uint32_t*>(sQ + sw16(hh, 64 + 2 * lane)) = pack_bf16(y2, y4);
    }
    const bool has_new = tau_new >= tau_lo && tau_new <= tau_hi;
    if (has_new && warp == 0) {
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
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    // running state: thread tid owns dimension d = tid of the 4 heads
    float m[kG], l[kG], o[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
        o[h] = 0.f;
    }
    int fail = 0, aborted = 0;
    uint32_t ph_m = 0;
    int issued = n_tiles < 2 ? n_tiles : 2;  // tiles whose loads thread 0 has issued
    int consumed = 0;                       // tiles whose loads have landed

    for (int i = 0; i < n_tiles; ++i) {
        const long long tau = tau_lo + i;
        const int st = i & 1;
        uint8_t* sK = smem + st * kStage;
        uint8_t* sV = sK + 2 * kBox;
        if (!mbar_wait(st ? bar_full1 : bar_full0, (uint32_t)((i >> 1) & 1)))
            fail = 1;
        else
            consumed = i + 1;
        if (!fail && has_new && tau == tau_new && tid < 16) {
            // chunk tid of the new 256-byte row: dims [8*tid, 8*tid+8)
            const int rr = (int)(pos - tau * kTile);
            const int half = tid >> 3, ch = tid & 7;
            const uint4 kw = reinterpret_cast<const uint4*>(snew)[tid];
            const uint4 vw = reinterpret_cast<const uint4*>(snew + kD)[tid];
            *reinterpret_cast<uint4*>(sK + half * kBox + sw128_offset(rr, ch)) = kw;
            *reinterpret_cast<uint4*>(sV + half * kBox + sw128_offset(rr, ch)) = vw;
            const long long gofs = ((long long)g * c.R + pos % c.R) * kD + 8 * tid;
            *reinterpret_cast<uint4*>(job.k_ring + gofs) = kw;
            *reinterpret_cast<uint4*>(job.v_ring + gofs) = vw;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(fail)) {
            aborted = 1;
            break;
        }
        tc_fence_after();

        // ---- S^T = K Q'^T
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = smem_desc_sw128(smem_u32(sK) + (kk >> 2) * kBox + 32 * (kk & 3), 16, 1024);
                const uint64_t bd = smem_desc_sw128(smem_u32(sQ) + (kk >> 2) * 2048 + 32 * (kk & 3), 16, 1024);
                mma_bf16_ss(tmem + 0, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar_m);
        }
        if (!mbar_wait(bar_m, ph_m))
            fail = 1;
        ph_m ^= 1;
        tc_fence_after();

        // ---- tile softmax: thread tid owns key 128*tau + tid
        uint32_t sv[32];
        tmem_ld_32x32b_x32(tmem + lane_base, sv);
        tmem_ld_wait();
        const long long kp = tau * kTile + tid;
        const bool valid = kp >= lo && kp <= pos;
        float sc[kG];
#pragma unroll
        for (int h = 0; h < kG; ++h) {
            sc[h] = valid ? __fmul_rn(__uint_as_float(sv[h]), c.scale_log2) : -INFINITY;
            const float wm = warp_max(sc[h]);
            if (lane == 0)
                sred[warp * kG + h] = wm;
        }
        __syncthreads();
        float mt[kG], pv[kG];
#pragma unroll
        for (int h = 0; h < kG; ++h) {
            mt[h] = fmaxf(fmaxf(sred[h], sred[kG + h]), fmaxf(sred[2 * kG + h], sred[3 * kG + h]));
            pv[h] = valid ? ex2(__fsub_rn(sc[h], mt[h])) : 0.f;
            const float ws = warp_sum(pv[h]);
            if (lane == 0)
                sred[16 + warp * kG + h] = ws;
        }
#pragma unroll
        for (int h = 0; h < kG; ++h)
            *reinterpret_cast<__nv_bfloat16*>(sP + sw16(h, tid)) = __float2bfloat16_rn(pv[h]);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        float lt[kG];
#pragma unroll
        for (int h = 0; h < kG; ++h)
            lt[h] = __fadd_rn(__fadd_rn(sred[16 + h], sred[16 + kG + h]),
                              __fadd_rn(sred[16 + 2 * kG + h], sred[16 + 3 * kG + h]));

        // ---- O^T = V^T P^T
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = smem_desc_sw128(smem_u32(sV) + 2048 * kk, kBox, 1024);
                const uint64_t bd = smem_desc_sw128(smem_u32(sP) + (kk >> 2) * 2048 + 32 * (kk & 3), 16, 1024);
                mma_bf16_ss(tmem + 16, ad, bd, kIdescO, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar_m);
        }
        if (!mbar_wait(bar_m, ph_m))
            fail = 1;
        ph_m ^= 1;
        tc_fence_after();
        if (tid == 0 && !fail && i + 2 < n_tiles) {  // this stage is free: fetch tile i + 2
            issue_tile(i + 2);
            issued = i + 3;
        }
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tmem + lane_base, ov);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < kG; ++h)
            fold1(m[h], l[h], o[h], mt[h], lt[h], __uint_as_float(ov[16 + h]));
        tc_fence_before();
        if (__syncthreads_or(fail)) {
            aborted = 1;
            break;
        }
        tc_fence_after();
    }

    if (aborted) {
        if (tid == 0) {
            // A bounded wait gave up: record it, let copies still in flight land, release TMEM.
            atomicExch(job.err, kErrTimeout);
            for (int k = consumed; k < issued; ++k)
                mbar_wait((k & 1) ? bar_full1 : bar_full0, (uint32_t)((k >> 1) & 1));
        }
    } else {
        // ---- this split's partial; the last CTA of (stream, g) folds all splits in order
#pragma unroll
        for (int h = 0; h < kG; ++h)
            job.part_o[((long long)(g * kG + h) * c.S + sl) * kD + tid] = o[h];
        if (tid < kG)
            *reinterpret_cast<float2*>(job.part_ml + ((long long)(g * kG + tid) * c.S + sl) * 2) =
                make_float2(m[tid], l[tid]);
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const unsigned prev = atomicAdd(job.counters + g, 1u);
            s_last = prev == (unsigned)(job.n_splits - 1);
        }
        __syncthreads();
        if (s_last) {
            __threadfence();
            const int hh = warp;
            const int hq = g * kG + hh;
            const int d4 = lane * 4;
            float mm = -INFINITY, ll = 0.f;
            float oo[4] = {0.f, 0.f, 0.f, 0.f};
            const float* pml = job.part_ml + (long long)hq * c.S * 2;
            const float* po = job.part_o + (long long)hq * c.S * kD + d4;
            for (int s0 = 0; s0 < job.n_splits; s0 += 8) {
                float2 ml[8];
                float4 ov4[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (s0 + u < job.n_splits) {
                        ml[u] = __ldcg(reinterpret_cast<const float2*>(pml + (s0 + u) * 2));
                        ov4[u] = __ldcg(reinterpret_cast<const float4*>(po + (long long)(s0 + u) * kD));
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (s0 + u < job.n_splits) {
                        float m0 = mm, l0 = ll;
                        fold1(m0, l0, oo[0], ml[u].x, ml[u].y, ov4[u].x);
                        float m1 = mm, l1 = ll;
                        fold1(m1, l1, oo[1], ml[u].x, ml[u].y, ov4[u].y);
                        float m2 = mm, l2 = ll;
                        fold1(m2, l2, oo[2], ml[u].x, ml[u].y, ov4[u].z);
                        fold1(mm, ll, oo[3], ml[u].x, ml[u].y, ov4[u].w);
                    }
                }
            }
            const uint32_t w0 = pack_bf16(__fdiv_rn(oo[0], ll), __fdiv_rn(oo[1], ll));
            const uint32_t w1 = pack_bf16(__fdiv_rn(oo[2], ll), __fdiv_rn(oo[3], ll));
            *reinterpret_cast<uint2*>(job.out + (long long)hq * kD + d4) = make_uint2(w0, w1);
            if (tid == 0)
                job.counters[g] = 0u;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
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
