// enc_attn.cu -- kernel (b): windowed-causal chunk attention against the encoder ring.
//
// Streaming plan ("Voxtral Realtime -- incremental streaming implementation plan"):
// SHIPPED/Mechanism -- mha_cached reads cache rows [0, n_kv_total) under a windowed-causal
// mask; "Unbounded length" -- the mask uses absolute positions (slot 0 holds frame
// abs_base); "Risk / notes" -- the chunk attention is a multi-query prefill against <= 750
// cached keys. Frame i attends to [i-749, i] ("RECOMMENDED implementation").
//
// Work item: one CTA per (context, head, 128-query tile of the batch). Keys are visited in
// tiles of 128 ABSOLUTE positions [128t, 128t+128), loaded by TMA from ring slots
// 128t - abs_base (rows outside the ring read as zero). Per tile:
//   S  = Q' K'^T       tcgen05.mma, M=128 N=128 K=64, A/B K-major bf16 in smem, D in TMEM
//   softmax            each thread owns one query row (TMEM lane); tile-local max m_t,
//                      p = 2^(s*log2e/sqrt(D) - m_t), l_t = sum p; P -> smem as bf16
//   O_t = P V          tcgen05.mma, M=128 N=64 K=128, A = P (K-major), B = V (MN-major)
//   fold               (m, l, o) <- merge((m, l, o), (m_t, l_t, O_t)) in registers
// A tile with no visible key for a row is skipped for that row (an exact no-op). Because
// tiles are fixed by absolute position and are folded in ascending order, a row's result
// depends only on its own window, never on how the stream was cut into feeds or when the
// ring was compacted.
//
// The query is rotated here, in the prologue (fp32 math, rounded to bf16 as the MMA
// operand); keys arrive already rotated in the ring (kernel a).
#include "common.cuh"
#include "ptx.cuh"
#include "vst_internal.h"

namespace vst {

namespace {

constexpr int kThreads = 128;
constexpr int kD = 64;
constexpr uint32_t kTileBytes = 128u * 128u;  // 128 rows x 128 B
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kTileBytes;
constexpr uint32_t kOffP = kOffV + kTileBytes;       // two 64-key blocks
constexpr uint32_t kOffBar = kOffP + 2 * kTileBytes;
constexpr uint32_t kSmemBytes = kOffBar + 64 + 1024;  // + slack to align the base to 1024
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmS = 0;    // S tile: columns [0, 128)
constexpr uint32_t kTmO = 128;  // O tile: columns [128, 192)

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 64, false, true);

}  // namespace

template <int J>
__global__ void __launch_bounds__(kThreads, 1)
    enc_attn_kernel(const __grid_constant__ KParams<EncAttnCommon, EncAttnJob, J> p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sK = smem + kOffK;
    uint8_t* sV = smem + kOffV;
    uint8_t* sP = smem + kOffP;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    const uint32_t bar_k = smem_u32(&bars[0]);
    const uint32_t bar_v = smem_u32(&bars[1]);
    const uint32_t bar_m = smem_u32(&bars[2]);

    const EncAttnCommon& c = p.c;
    const EncAttnJob& job = p.jobs[blockIdx.z];
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int row0 = blockIdx.x * 128;
    const int nrows = min(128, c.n_rows - row0);
    const long long p_first = job.pos0 + row0;
    const long long p_last = p_first + nrows - 1;
    const long long key_lo = max(0LL, p_first - c.W + 1);
    const long long t_begin = key_lo / 128;
    const long long t_end = p_last / 128;

    if (tid == 0) {
        mbar_init(bar_k, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_m, 1);
        fence_mbar_init();
        tmap_acquire(job.tmap_k);
        tmap_acquire(job.tmap_v);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }

    // ---- rotate this thread's query row into sQ (bf16, K-major, 128-B swizzle)
    const int r = tid;
    const long long pq = p_first + r;
    if (r < nrows) {
        const __nv_bfloat16* qrow = job.q + ((long long)(row0 + r) * c.H + h) * kD;
        const float2* cs = c.rope + pq * (kD / 2);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            const uint4 a = *reinterpret_cast<const uint4*>(qrow + 8 * ch);
            const uint4 b = *reinterpret_cast<const uint4*>(qrow + 32 + 8 * ch);
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
            const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
            uint32_t ya[4], yb[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                float y1a, y2a, y1b, y2b;
                rope_pair(bf16lo(aw[w]), bf16lo(bw[w]), cs[8 * ch + 2 * w], y1a, y2a);
                rope_pair(bf16hi(aw[w]), bf16hi(bw[w]), cs[8 * ch + 2 * w + 1], y1b, y2b);
                ya[w] = pack_bf16(y1a, y1b);
                yb[w] = pack_bf16(y2a, y2b);
            }
            *reinterpret_cast<uint4*>(sQ + sw128_offset(r, ch)) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
            *reinterpret_cast<uint4*>(sQ + sw128_offset(r, 4 + ch)) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
        }
    } else {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(sQ + sw128_offset(r, ch)) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    bool pend_k = false, pend_v = false;
    if (tid == 0) {
        const int slot = (int)(t_begin * 128 - job.abs_base);
        mbar_arrive_expect_tx(bar_k, kTileBytes);
        tma_load_3d(smem_u32(sK), job.tmap_k, bar_k, 0, slot, h);
        mbar_arrive_expect_tx(bar_v, kTileBytes);
        tma_load_3d(smem_u32(sV), job.tmap_v, bar_v, 0, slot, h);
        pend_k = pend_v = true;
    }

    float o[kD];
#pragma unroll
    for (int d = 0; d < kD; ++d)
        o[d] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t ph_k = 0, ph_v = 0, ph_m = 0;
    bool aborted = false;

    for (long long t = t_begin; t <= t_end; ++t) {
        int fail = 0;
        // ---- S = Q K^T
        if (tid == 0) {
            if (mbar_wait(bar_k, ph_k)) {
                pend_k = false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = smem_desc_sw128(smem_u32(sQ) + 32 * kk, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(smem_u32(sK) + 32 * kk, 16, 1024);
                    mma_bf16_ss(tmem + kTmS, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar_m);
            } else {
                fail = 1;
            }
        }
        ph_k ^= 1;
        if (!fail && !mbar_wait(bar_m, ph_m))
            fail = 1;
        ph_m ^= 1;
        tc_fence_after();
        if (tid == 0 && !fail && t < t_end) {
            const int slot = (int)((t + 1) * 128 - job.abs_base);
            mbar_arrive_expect_tx(bar_k, kTileBytes);
            tma_load_3d(smem_u32(sK), job.tmap_k, bar_k, 0, slot, h);
            pend_k = true;
        }

        // ---- tile-local softmax of row r (scores in log2 units)
        const long long kbase = t * 128;
        const long long lo_c = (r < nrows) ? (pq - c.W + 1 - kbase) : 1000;
        const long long hi_c = (r < nrows) ? (pq - kbase) : -1;
        float mt = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem + lane_base + kTmS + cc * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int col = cc * 32 + j;
                if (col >= lo_c && col <= hi_c)
                    mt = fmaxf(mt, __fmul_rn(__uint_as_float(v[j]), c.scale_log2));
            }
        }
        float lt = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem + lane_base + kTmS + cc * 32, v);
            tmem_ld_wait();
            float pv[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int col = cc * 32 + j;
                const bool ok = col >= lo_c && col <= hi_c;
                pv[j] = ok ? ex2(__fsub_rn(__fmul_rn(__uint_as_float(v[j]), c.scale_log2), mt)) : 0.f;
                lt = __fadd_rn(lt, pv[j]);
            }
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                const uint4 w = make_uint4(pack_bf16(pv[8 * qd + 0], pv[8 * qd + 1]),
                                           pack_bf16(pv[8 * qd + 2], pv[8 * qd + 3]),
                                           pack_bf16(pv[8 * qd + 4], pv[8 * qd + 5]),
                                           pack_bf16(pv[8 * qd + 6], pv[8 * qd + 7]));
                *reinterpret_cast<uint4*>(sP + (cc >> 1) * kTileBytes + sw128_offset(r, (cc & 1) * 4 + qd)) = w;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(fail)) {
            aborted = true;
            break;
        }
        tc_fence_after();

        // ---- O_t = P V
        if (tid == 0) {
            if (mbar_wait(bar_v, ph_v)) {
                pend_v = false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = smem_desc_sw128(smem_u32(sP) + (kk >> 2) * kTileBytes + 32 * (kk & 3), 16, 1024);
                    const uint64_t bd = smem_desc_sw128(smem_u32(sV) + 2048 * kk, kTileBytes, 1024);
                    mma_bf16_ss(tmem + kTmO, ad, bd, kIdescO, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar_m);
            } else {
                fail = 1;
            }
        }
        ph_v ^= 1;
        if (!fail && !mbar_wait(bar_m, ph_m))
            fail = 1;
        ph_m ^= 1;
        tc_fence_after();
        if (tid == 0 && !fail && t < t_end) {
            const int slot = (int)((t + 1) * 128 - job.abs_base);
            mbar_arrive_expect_tx(bar_v, kTileBytes);
            tma_load_3d(smem_u32(sV), job.tmap_v, bar_v, 0, slot, h);
            pend_v = true;
        }

        // ---- fold the tile into the running state (skipped when the row saw no key)
        uint32_t ov[64];
        tmem_ld_32x32b_x32(tmem + lane_base + kTmO, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
        tmem_ld_32x32b_x32(tmem + lane_base + kTmO + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
        tmem_ld_wait();
        if (mt != -INFINITY) {
            const float mn = fmaxf(m_run, mt);
            const float a = ex2(__fsub_rn(m_run, mn));
            const float b = ex2(__fsub_rn(mt, mn));
            l_run = __fmaf_rn(l_run, a, __fmul_rn(lt, b));
#pragma unroll
            for (int d = 0; d < kD; ++d)
                o[d] = __fmaf_rn(o[d], a, __fmul_rn(__uint_as_float(ov[d]), b));
            m_run = mn;
        }
        tc_fence_before();
        if (__syncthreads_or(fail)) {
            aborted = true;
            break;
        }
        tc_fence_after();
    }

    if (!aborted) {
        if (r < nrows) {
            __nv_bfloat16* orow = job.out + ((long long)(row0 + r) * c.H + h) * kD;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16(__fdiv_rn(o[8 * ch + 2 * e], l_run), __fdiv_rn(o[8 * ch + 2 * e + 1], l_run));
                *reinterpret_cast<uint4*>(orow + 8 * ch) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    } else if (tid == 0) {
        // A bounded wait gave up: record it, let copies still in flight land, then release
        // TMEM and leave.
        atomicExch(job.err, kErrTimeout);
        if (pend_k)
            mbar_wait(bar_k, ph_k);
        if (pend_v)
            mbar_wait(bar_v, ph_v);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int J>
static cudaError_t launch_enc_attn_j(const KParams<EncAttnCommon, EncAttnJob, J>& p, int n_jobs,
                                     cudaStream_t s)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(enc_attn_kernel<J>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess)
            return e;
        configured[dev] = 1;
    }
    const dim3 grid((unsigned)((p.c.n_rows + 127) / 128), (unsigned)p.c.H, (unsigned)n_jobs);
    enc_attn_kernel<J><<<grid, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_enc_attn(const EncAttnCommon& c, const EncAttnJob* jobs, int n_jobs, cudaStream_t s)
{
    if (n_jobs == 0 || c.n_rows == 0)
        return cudaSuccess;
    return with_params(c, jobs, n_jobs, [&](const auto& p) {
        return launch_enc_attn_j<sizeof(p.jobs) / sizeof(p.jobs[0])>(p, n_jobs, s);
    });
}

}  // namespace vst
