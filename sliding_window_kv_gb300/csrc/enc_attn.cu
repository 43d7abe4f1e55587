// enc_attn.cu -- kernel (b) with the encoder half of kernel (a) fused in: windowed-causal
// chunk attention against the encoder ring, for one batch of new frames per context.
//
// Streaming plan ("Voxtral Realtime -- incremental streaming implementation plan"):
// SHIPPED/Mechanism -- mha_cached writes the chunk's K/V at cache rows
// [n_kv_before, n_kv_total) and reads [0, n_kv_total) under a windowed-causal mask;
// "Unbounded length" -- the mask uses absolute positions (slot 0 holds frame abs_base);
// "Chunk alignment" -- RoPE at absolute positions; "Risk / notes" -- the chunk attention is a
// multi-query prefill against <= 750 cached keys. Frame i attends to [i-749, i]
// ("RECOMMENDED implementation").
//
// Keys are visited in tiles of 128 ABSOLUTE positions [128t, 128t+128), loaded whole by
// TMA from ring slots 128t - abs_base (rows outside the ring read as zero): the batch's own
// rows were rotated and appended to the ring by kernel (a) (rope_append.cu) just before
// this launch. Per tile:
//   S   = Q' K'^T      tcgen05.mma M=128 N=128 K=64, A/B K-major bf16 in smem, D in TMEM
//   softmax            tile-local max m_t, p = 2^(s*log2e/sqrt(D) - m_t), l_t = sum p;
//                      P -> smem as bf16
//   O_t = P V          tcgen05.mma M=128 N=64 K=128, A = P (K-major), B = V (MN-major)
//   fold               (m, l, o) <- fold((m, l, o), (m_t, l_t, O_t)), ascending t
// A tile where a row sees no key is skipped for that row (exact no-op).
//
// Threads: 256 per CTA, two CTAs per SM. Query row r (TMEM lane r) is shared by the two
// threads (r, half), one in each group of four warps: thread (r, half) owns score quarters
// 2 half and 2 half + 1 (columns [64 half, 64 half + 64)), output dims [32 half, 32 half
// + 32) and RoPE pairs [16 half, 16 half + 16). Row max and row sum are combined from the
// two halves through shared memory, (Q0 + Q1) + (Q2 + Q3) (enc_common.cuh).
//
// Launch shape (loop): one CTA per (context, head, 128-query tile) folds its key tiles in
// registers. The split shape for a single query tile (enc_attn_split.cu) gives the same
// bits: tiles are fixed by absolute position and folded in ascending order, and every
// row's arithmetic comes from enc_common.cuh -- so a row's result depends only on its own
// window, never on how the stream was cut into feeds, on when the ring was compacted, or
// on the launch shape.
#include "common.cuh"
#include "enc_common.cuh"
#include "ptx.cuh"
#include "vst_internal.h"

namespace vst {

namespace {

constexpr int kThreads = 256;
constexpr int kD = 64;
constexpr int kDh = kD / 2;                            // output dims per thread
constexpr uint32_t kTileBytes = 128u * 128u;           // 128 rows x 128 B
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kTileBytes;
constexpr uint32_t kOffP = kOffV + kTileBytes;         // two 64-key blocks
constexpr uint32_t kOffRed = kOffP + 2 * kTileBytes;   // float [2][2 halves][128]: row max / sum halves
constexpr uint32_t kOffBar = kOffRed + 2 * 2 * 128 * 4;
constexpr uint32_t kSmemBytes = kOffBar + 64 + 1024;   // + slack to align the base to 1024
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmS = 0;    // S tile: columns [0, 128)
constexpr uint32_t kTmO = 128;  // O tile: columns [128, 192)

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 64, false, true);

}  // namespace

template <int J>
__global__ void __launch_bounds__(kThreads, 2)
    enc_attn_kernel(const __grid_constant__ KParams<EncAttnCommon, EncAttnJob, J> p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    const EncAttnCommon& c = p.c;
    const EncAttnJob& job = p.jobs[blockIdx.z];
    const int h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = 32 * (warp & 3) + lane;  // TMEM lane = query row of this thread
    const int half = warp >> 2;            // half of the row
    const int row0 = (int)blockIdx.x * 128;
    const int nrows = min(128, c.n_rows - row0);
    const long long p_first = job.pos0 + row0;
    const long long t_lo = max(0LL, p_first - c.W + 1) / 128;
    const long long t_hi = (p_first + nrows - 1) / 128;

    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sK = smem + kOffK;
    uint8_t* sV = smem + kOffV;
    uint8_t* sP = smem + kOffP;
    float* red_m = reinterpret_cast<float*>(smem + kOffRed);  // [2 halves][128]
    float* red_l = red_m + 2 * 128;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    const uint32_t bar_k = smem_u32(&bars[0]), bar_v = smem_u32(&bars[1]), bar_m = smem_u32(&bars[2]);

    // Prologue. The first ring tiles may be requested before the previous kernel in the
    // stream has finished when the host says that kernel did not touch this ring (early);
    // everything else waits for it.
    auto issue_k = [&](long long t) {
        mbar_arrive_expect_tx(bar_k, kTileBytes);
        tma_load_3d(smem_u32(sK), job.tmap_k, bar_k, 0, (int)(t * 128 - job.abs_base), h);
    };
    auto issue_v = [&](long long t) {
        mbar_arrive_expect_tx(bar_v, kTileBytes);
        tma_load_3d(smem_u32(sV), job.tmap_v, bar_v, 0, (int)(t * 128 - job.abs_base), h);
    };
    if (tid == 0) {
        mbar_init(bar_k, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_m, 1);
        fence_mbar_init();
        tmap_acquire(job.tmap_k);
        tmap_acquire(job.tmap_v);
        if (c.early) {
            issue_k(t_lo);
            issue_v(t_lo);
        }
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    griddep_wait();
    if (tid == 0 && !c.early) {
        issue_k(t_lo);
        issue_v(t_lo);
    }
    __syncwarp();

    // ---- this thread's half of query row r, rotated, into sQ
    const long long pq = p_first + r;
    const bool row_real = r < nrows;
    if (row_real) {
        const __nv_bfloat16* qrow = job.q + ((long long)(row0 + r) * c.H + h) * kD;
        enc::rotate_quarter(qrow, c.rope + pq * (kD / 2), sQ, r, 2 * half);
        enc::rotate_quarter(qrow, c.rope + pq * (kD / 2), sQ, r, 2 * half + 1);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)  // chunks {q, 4 + q} of quarters q = 2 half, 2 half + 1
            *reinterpret_cast<uint4*>(sQ + sw128_offset(r, (e >> 1) * 4 + 2 * half + (e & 1))) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();  // Q' (generic stores) before the MMAs read it
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    float o[kDh];
#pragma unroll
    for (int d = 0; d < kDh; ++d)
        o[d] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t ph_k = 0, ph_v = 0, ph_m = 0;
    bool pend_k = tid == 0, pend_v = tid == 0;
    int fail = 0, aborted = 0;

    for (long long t = t_lo; t <= t_hi; ++t) {
        // ---- K of tile t in smem, then S = Q K^T
        if (!mbar_wait(bar_k, ph_k))
            fail = 1;
        ph_k ^= 1;
        if (tid == 0)
            pend_k = false;
        tc_fence_before();
        if (__syncthreads_or(fail)) {
            aborted = 1;
            break;
        }
        tc_fence_after();
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(tmem + kTmS, smem_desc_sw128(smem_u32(sQ) + 32 * kk, 16, 1024),
                            smem_desc_sw128(smem_u32(sK) + 32 * kk, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
            mma_commit(bar_m);
        }
        __syncwarp();
        if (!mbar_wait(bar_m, ph_m))
            fail = 1;
        ph_m ^= 1;
        tc_fence_after();
        if (tid == 0 && !fail && t < t_hi) {  // K buffer is free: fetch the next tile's K
            issue_k(t + 1);
            pend_k = true;
        }
        __syncwarp();

        // ---- tile-local softmax of this thread's half of row r
        int lo = 1, hi = 0;  // visible columns of row r in this tile; empty unless r is real
        if (row_real) {
            lo = (int)max(-1LL, min(128LL, pq - c.W + 1 - t * 128));
            hi = (int)max(-1LL, min(128LL, pq - t * 128));
        }
        // both quarters of this half-row in one TMEM round trip, kept for the exp pass
        uint32_t sa[32], sb[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kTmS + 64 * half, sa);
        tmem_ld_32x32b_x32(tmem + lane_base + kTmS + 64 * half + 32, sb);
        tmem_ld_wait();
        const float mh = fmaxf(enc::quarter_max(sa, 64 * half, lo, hi), enc::quarter_max(sb, 64 * half + 32, lo, hi));
        red_m[half * 128 + r] = mh;
        __syncthreads();
        const float mt = __fmul_rn(fmaxf(red_m[r], red_m[128 + r]), c.scale_log2);  // -inf: row sees nothing
        const float la = enc::quarter_exp(sa, 64 * half, lo, hi, c.scale_log2, -mt, sP, r);
        const float lb = enc::quarter_exp(sb, 64 * half + 32, lo, hi, c.scale_log2, -mt, sP, r);
        red_l[half * 128 + r] = __fadd_rn(la, lb);

        // ---- V of tile t in smem, then O_t = P V
        if (!mbar_wait(bar_v, ph_v))
            fail = 1;
        ph_v ^= 1;
        if (tid == 0)
            pend_v = false;
        fence_proxy_async_smem();  // P (generic stores) before the MMA reads it
        tc_fence_before();
        if (__syncthreads_or(fail)) {
            aborted = 1;
            break;
        }
        tc_fence_after();
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ss(tmem + kTmO,
                            smem_desc_sw128(smem_u32(sP) + (kk >> 2) * kTileBytes + 32 * (kk & 3), 16, 1024),
                            smem_desc_sw128(smem_u32(sV) + 2048 * kk, kTileBytes, 1024), kIdescO, kk > 0 ? 1u : 0u);
            mma_commit(bar_m);
        }
        __syncwarp();
        const float lt = __fadd_rn(red_l[r], red_l[128 + r]);
        if (!mbar_wait(bar_m, ph_m))
            fail = 1;
        ph_m ^= 1;
        tc_fence_after();
        if (tid == 0 && !fail && t < t_hi) {  // V buffer is free: fetch the next tile's V
            issue_v(t + 1);
            pend_v = true;
        }
        __syncwarp();

        // ---- O_t of this thread's dims, folded into the running state
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kTmO + kDh * half, ov);
        tmem_ld_wait();
        if (mt != -INFINITY) {
            float ot[kDh];
#pragma unroll
            for (int d = 0; d < kDh; ++d)
                ot[d] = __uint_as_float(ov[d]);
            enc::fold_tile<kDh>(m_run, l_run, o, mt, lt, ot);
        }
        tc_fence_before();
    }

    griddep_launch_dependents();
    if (aborted && tid == 0) {
        // A bounded wait gave up: record it and let copies still in flight land.
        atomicExch(job.err, kErrTimeout);
        if (pend_k)
            mbar_wait(bar_k, ph_k);
        if (pend_v)
            mbar_wait(bar_v, ph_v);
    }
    if (!aborted && row_real)
        enc::store_out<kDh>(job.out + ((long long)(row0 + r) * c.H + h) * kD, o, l_run, kDh * half);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int J>
static cudaError_t launch_enc_attn_j(const KParams<EncAttnCommon, EncAttnJob, J>& p, int n_jobs, int grid_x,
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
    const dim3 grid((unsigned)grid_x, (unsigned)p.c.H, (unsigned)n_jobs);
    return launch_pdl(enc_attn_kernel<J>, grid, dim3(kThreads), kSmemBytes, s, p);
}

cudaError_t launch_enc_attn(const EncAttnCommon& c, const EncAttnJob* jobs, int n_jobs, int grid_x, cudaStream_t s)
{
    if (n_jobs == 0 || c.n_rows == 0)
        return cudaSuccess;
    if (c.split || !c.appended)
        return cudaErrorInvalidValue;  // split shape: launch_enc_attn_split; rows appended first
    return with_params(c, jobs, n_jobs, [&](const auto& p) {
        return launch_enc_attn_j<sizeof(p.jobs) / sizeof(p.jobs[0])>(p, n_jobs, grid_x, s);
    });
}

}  // namespace vst
