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
// window [max(0, pos-W+1), pos]. Each key tile (K and V, 32 KB each, two 64-dim boxes with
// 128-B swizzle, ring slots 128*tau mod R) arrives by TMA. Per tile:
//   S^T = K Q'^T     tcgen05.mma M=128 keys, N=16 (the 4 query heads of the group, zero
//                    padded), K=128 dims; A = K tile (K-major), B = Q' (K-major); TMEM
//   softmax          512 threads: thread (head h, key k) holds one score; per head the
//                    tile max and sum go through warp shuffles and the head's 4 warps
//                    (fixed order); P^T -> smem (bf16)
//   O^T = V^T P^T    tcgen05.mma M=128 dims, N=16, K=128 keys; A = V tile read as
//                    MN-major (dims contiguous), B = P^T (K-major); TMEM
//   fold             thread (head h, dim d) folds (m_t, l_t, O_t[h][d]) into registers.
// Pipeline: one K buffer and two V buffers per CTA and two CTAs per SM, so that one CTA's
// prologue and merge overlap another's streaming (also across launches: the next launch's
// CTAs share the SM while this one finishes). The next K is fetched as soon as S^T is
// done; V runs two tiles ahead (V of tile i + 2 as soon as O^T of tile i is done); S^T
// alternates between two TMEM buffers.
// The query heads are rotated in the prologue; if the split holds pos, the new key is
// rotated too, patched into its tile row in shared memory, and stored (K', V) to ring slot
// pos % R by this CTA. A prefill chunk (several tokens of one stream, one job each) has its
// rows appended to the ring before the launch, so there every key comes from the ring. Each CTA writes its split's (m, l, o) per head; the last CTA of
// (stream, g) folds the splits in ascending order and writes the output. Tiles and splits
// are fixed by absolute position, so a stream's output is the same bits alone or in a
// batch, with either pipeline, and whatever the ring size.
#include "common.cuh"
#include "ptx.cuh"
#include "vst_internal.h"

namespace vst {

namespace {

constexpr int kThreads = 512;
constexpr int kD = 128;
constexpr int kG = 4;                       // query heads per KV head
constexpr int kTile = kDecTile;             // keys per tile
constexpr int kTilesPerSplit = kDecSplit / kTile;
constexpr uint32_t kBox = 128u * 128u;      // 128 keys x 64 dims x 2 B
constexpr uint32_t kStage = 6 * kBox;       // K lo, K hi, then two V buffers (lo, hi)
constexpr uint32_t kTmemCols = 64;          // S^T buffers at [0,16) and [16,32); O^T at [32,48)
constexpr uint32_t kTmO = 32;
// Split partials loaded per round of the last CTA's fold: 17, the splits of a full 8192
// window, so that one round trip fetches them all.
constexpr int kMergeGroup = 17;

struct Layout {
    static constexpr uint32_t kOffQ = kStage;           // Q' [16 rows][128 dims]: 2 blocks of 2 KB
    static constexpr uint32_t kOffP = kOffQ + 4096;     // P^T [16 rows][128 keys]: 2 blocks of 2 KB
    static constexpr uint32_t kOffNew = kOffP + 4096;   // new K' row, new V row (bf16 x 128 each)
    static constexpr uint32_t kOffRed = kOffNew + 512;  // float [2][4 heads][4 warps]; merge coefficients
    static constexpr uint32_t kOffBar = kOffRed + 4 * 32 * 3 * 4;  // 6 mbarriers
    static constexpr uint32_t kSmemBytes = kOffBar + 128 + 1024;
};

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

// Barrier over the 4 warps (128 threads) of one head group.
__device__ __forceinline__ void head_sync(int hh)
{
    __syncwarp();  // .aligned: the whole warp executes it together
    asm volatile("bar.sync %0, 128;" ::"r"(1 + hh) : "memory");
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
__global__ void __launch_bounds__(kThreads, 2)
    dec_step_kernel(const __grid_constant__ KParams<DecCommon, DecJob, J> p)
{
    using L = Layout;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    __shared__ int s_last;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sQ = smem + L::kOffQ;
    uint8_t* sP = smem + L::kOffP;
    __nv_bfloat16* snew = reinterpret_cast<__nv_bfloat16*>(smem + L::kOffNew);
    float* red_m = reinterpret_cast<float*>(smem + L::kOffRed);  // [4 heads][4 warps]
    float* red_l = red_m + 16;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
    // bars: K landed, V buffer 0 landed, S^T done [2], O^T done, V buffer 1 landed
    const uint32_t bar_k = smem_u32(&bars[0]);
    auto bar_v = [&](int i) { return smem_u32(&bars[(i & 1) ? 5 : 1]); };  // V of tile i
    auto bar_s = [&](int b) { return smem_u32(&bars[2 + b]); };
    const uint32_t bar_o = smem_u32(&bars[4]);

    const DecCommon& c = p.c;
    const int item = blockIdx.x;
    int j = 0;
    while (j + 1 < c.n_jobs && p.jobs[j + 1].work_begin <= item)
        ++j;
    const DecJob& job = p.jobs[j];
    const int g = blockIdx.y;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int hh = warp >> 2;                 // query head of the group owned by this thread
    const int row = 32 * (warp & 3) + lane;   // TMEM lane: key of the tile (S), dim (O)
    const int sl = item - job.work_begin;     // split index within this step
    const long long pos = job.pos;
    const long long lo = max(0LL, pos - c.W + 1);
    const long long sig = job.sigma0 + sl;
    const long long tau_lo = max(sig * kTilesPerSplit, lo / kTile);
    const long long tau_hi = min(sig * kTilesPerSplit + kTilesPerSplit - 1, pos / kTile);
    const int n_tiles = (int)(tau_hi - tau_lo + 1);
    const long long tau_new = pos / kTile;  // tile holding this step's key
    // This CTA rotates, patches in and stores the step's key unless the row is already in
    // the ring (a prefill chunk, appended before the launch).
    const bool has_new = !c.appended && tau_new >= tau_lo && tau_new <= tau_hi;

    uint8_t* const sK = smem;  // K tile: two 64-dim boxes
    auto sV = [&](int i) { return smem + (2 + 2 * (i & 1)) * kBox; };  // V of tile i: two buffers
    auto parity = [&](int i) { return (uint32_t)(i & 1); };
    auto slot_of = [&](int i) { return (int)(((tau_lo + i) * kTile) % c.R); };
    int k_issued = 0, v_issued = 0;  // tiles requested so far, in order (thread 0)
    auto issue_k = [&](int i) {
        k_issued = i + 1;
        const uint32_t dst = smem_u32(sK);
        mbar_arrive_expect_tx(bar_k, 2 * kBox);
        tma_load_3d(dst, job.tmap_k, bar_k, 0, slot_of(i), g);
        tma_load_3d(dst + kBox, job.tmap_k, bar_k, 64, slot_of(i), g);
    };
    auto issue_v = [&](int i) {
        v_issued = i + 1;
        const uint32_t dst = smem_u32(sV(i));
        mbar_arrive_expect_tx(bar_v(i), 2 * kBox);
        tma_load_3d(dst, job.tmap_v, bar_v(i), 0, slot_of(i), g);
        tma_load_3d(dst + kBox, job.tmap_v, bar_v(i), 64, slot_of(i), g);
    };
    auto issue_first = [&]() {  // every split has at least one tile
        issue_k(0);
        issue_v(0);
        if (n_tiles > 1)
            issue_v(1);
    };

    // Prologue. The first ring tiles may be requested before the previous kernel in the
    // stream has finished when the host says that kernel did not touch this ring (early);
    // everything else waits for it.
    if (tid == 0) {
        for (int b = 0; b < 6; ++b)
            mbar_init(smem_u32(&bars[b]), 1);
        fence_mbar_init();
        tmap_acquire(job.tmap_k);
        tmap_acquire(job.tmap_v);
        if (c.early)
            issue_first();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    // What the prologue of a decoder step reads right after the wait -- the group's four query
    // heads, the (cos, sin) row of pos and, if this CTA stores the step's key, its K and V
    // rows -- is pulled into L2 now, so that those loads hit L2. (A prefill chunk's launch
    // follows its own append, which the prefetches would only compete with.)
    if (!c.appended) {
        if (tid == 32) {
            prefetch_l2(job.q + (long long)g * kG * kD, kG * kD * 2);
        } else if (tid == 64) {
            prefetch_l2(c.rope + pos * (kD / 2), kD * 4);
        } else if (tid == 96 && has_new) {
            prefetch_l2(job.k + (long long)g * kD, kD * 2);
            prefetch_l2(job.v + (long long)g * kD, kD * 2);
        }
    }
    griddep_wait();
    if (tid == 0 && !c.early)
        issue_first();

    // ---- Q' (4 rotated heads, bf16), the new K'/V row, zero padding rows 4..15
    if (tid < 256) {
        const int h = tid >> 6, i = tid & 63;  // pair (i, i + 64) of head h
        const __nv_bfloat16* q = job.q + (long long)(g * kG + h) * kD;
        float y1, y2;
        rope_pair(__bfloat162float(q[i]), __bfloat162float(q[i + 64]), c.rope[pos * (kD / 2) + i], y1, y2);
        *reinterpret_cast<__nv_bfloat16*>(sQ + sw16(h, i)) = __float2bfloat16_rn(y1);
        *reinterpret_cast<__nv_bfloat16*>(sQ + sw16(h, i + 64)) = __float2bfloat16_rn(y2);
    } else if (tid < 320) {
        if (has_new) {
            const int i = tid - 256;
            const __nv_bfloat16* k = job.k + (long long)g * kD;
            const __nv_bfloat16* v = job.v + (long long)g * kD;
            float y1, y2;
            rope_pair(__bfloat162float(k[i]), __bfloat162float(k[i + 64]), c.rope[pos * (kD / 2) + i], y1, y2);
            snew[i] = __float2bfloat16_rn(y1);
            snew[i + 64] = __float2bfloat16_rn(y2);
            snew[kD + i] = v[i];
            snew[kD + i + 64] = v[i + 64];
        }
    } else {
        for (int e = tid - 320; e < 12 * 16; e += kThreads - 320) {  // 12 rows x 16 chunks
            const int r = 4 + e / 16, ch = e % 16;
            const uint32_t off = (uint32_t)((ch >> 3) * 2048) + sw128_offset(r, ch & 7);
            *reinterpret_cast<uint4*>(sQ + off) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(sP + off) = make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int rr_new = (int)(pos - tau_new * kTile);  // row of the new key in its tile

    // Warp 0: wait for tile i's K, patch the new key in if it is there, and (the elected lane)
    // issue S^T for it into S buffer i & 1. Returns false if the wait gave up.
    const uint32_t elect = warp == 0 ? elect_one_sync() : 0u;
    auto prepare_and_issue_s = [&](int i) -> bool {
        bool ok = mbar_wait(bar_k, parity(i));
        if (ok && has_new && tau_lo + i == tau_new && lane < 16) {
            const uint4 kw = reinterpret_cast<const uint4*>(snew)[lane];  // dims [8 lane, 8 lane + 8)
            *reinterpret_cast<uint4*>(sK + (lane >> 3) * kBox + sw128_offset(rr_new, lane & 7)) = kw;
            *reinterpret_cast<uint4*>(job.k_ring + ((long long)g * c.R + pos % c.R) * kD + 8 * lane) = kw;
            fence_proxy_async_smem();
        }
        __syncwarp();
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (ok) {  // the whole warp, converged; the elected lane issues
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = smem_desc_sw128(smem_u32(sK) + (kk >> 2) * kBox + 32 * (kk & 3), 16, 1024);
                const uint64_t bd = smem_desc_sw128(smem_u32(sQ) + (kk >> 2) * 2048 + 32 * (kk & 3), 16, 1024);
                mma_bf16_ss_if(tmem + 16 * (i & 1), ad, bd, kIdescS, kk > 0 ? 1u : 0u, elect);
            }
            mma_commit_if(bar_s(i & 1), elect);
        }
        return ok;
    };

    // running state of (head hh, dim row)
    float m = -INFINITY, l = 0.f, o = 0.f;
    int fail = 0, aborted = 0;
    uint32_t ph_o = 0;

    for (int i = 0; i < n_tiles; ++i) {
        // ---- S^T of tile i (issued by warp 0 alone: the other warps wait for its completion;
        // if warp 0 gives up, they give up on that wait and the barrier below ends the loop)
        if (warp == 0 && !prepare_and_issue_s(i))
            fail = 1;
        if (!fail && !mbar_wait(bar_s(i & 1), (uint32_t)((i >> 1) & 1)))
            fail = 1;
        tc_fence_after();
        if (tid == 0 && !fail && i + 1 < n_tiles)
            issue_k(i + 1);  // the K buffer is free once S^T of tile i is done
        const uint32_t sv = tmem_ld_32x32b_x1(tmem + lane_base + 16 * (i & 1) + hh);  // head hh's column
        tmem_ld_wait();

        // ---- softmax of head hh over the tile's 128 keys (thread: key `row`)
        const long long kp = (tau_lo + i) * kTile + row;
        const bool valid = kp >= lo && kp <= pos;
        const float sc = valid ? __fmul_rn(__uint_as_float(sv), c.scale_log2) : -INFINITY;
        const float wm = warp_max(sc);
        if (lane == 0)
            red_m[hh * 4 + (warp & 3)] = wm;
        head_sync(hh);
        const float mt = fmaxf(fmaxf(red_m[hh * 4], red_m[hh * 4 + 1]), fmaxf(red_m[hh * 4 + 2], red_m[hh * 4 + 3]));
        const float pv = valid ? ex2(__fsub_rn(sc, mt)) : 0.f;
        *reinterpret_cast<__nv_bfloat16*>(sP + sw16(hh, row)) = __float2bfloat16_rn(pv);
        const float ws = warp_sum(pv);
        if (lane == 0)
            red_l[hh * 4 + (warp & 3)] = ws;

        // ---- V of tile i (new value patched in), then O^T = V^T P^T
        if (!mbar_wait(bar_v(i), (uint32_t)((i >> 1) & 1)))
            fail = 1;
        if (!fail && has_new && tau_lo + i == tau_new && tid < 16) {
            const uint4 vw = reinterpret_cast<const uint4*>(snew + kD)[tid];
            *reinterpret_cast<uint4*>(sV(i) + (tid >> 3) * kBox + sw128_offset(rr_new, tid & 7)) = vw;
            *reinterpret_cast<uint4*>(job.v_ring + ((long long)g * c.R + pos % c.R) * kD + 8 * tid) = vw;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(fail)) {
            aborted = 1;
            break;
        }
        tc_fence_after();
        const float lt = __fadd_rn(__fadd_rn(red_l[hh * 4], red_l[hh * 4 + 1]), __fadd_rn(red_l[hh * 4 + 2], red_l[hh * 4 + 3]));
        if (warp == 0) {  // converged after the barrier; the elected lane issues
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = smem_desc_sw128(smem_u32(sV(i)) + 2048 * kk, kBox, 1024);
                const uint64_t bd = smem_desc_sw128(smem_u32(sP) + (kk >> 2) * 2048 + 32 * (kk & 3), 16, 1024);
                mma_bf16_ss_if(tmem + kTmO, ad, bd, kIdescO, kk > 0 ? 1u : 0u, elect);
            }
            mma_commit_if(bar_o, elect);
        }
        if (!mbar_wait(bar_o, ph_o))
            fail = 1;
        ph_o ^= 1;
        tc_fence_after();
        if (tid == 0 && !fail && i + 2 < n_tiles)
            issue_v(i + 2);  // tile i's V buffer is free once O^T of tile i is done
        const uint32_t ov = tmem_ld_32x32b_x1(tmem + lane_base + kTmO + hh);
        tmem_ld_wait();
        fold1(m, l, o, mt, lt, __uint_as_float(ov));
        tc_fence_before();
    }

    griddep_launch_dependents();
    if (aborted && tid == 0) {
        // A bounded wait gave up: record it and give copies in flight a bounded chance to
        // land. The CTA still counts itself in below, so that the merge counter of (stream, g)
        // ends this launch at zero like any other: the launch's output is undefined (the
        // error word says so), the next launch's is not.
        atomicExch(job.err, kErrTimeout);
        if (k_issued > 0)  // tile i's K is the i-th completion of the K barrier
            mbar_wait(bar_k, parity(k_issued - 1));
        for (int i = v_issued - 2 < 0 ? 0 : v_issued - 2; i < v_issued; ++i)  // the last V of each buffer
            mbar_wait(bar_v(i), (uint32_t)((i >> 1) & 1));
    }
    {
        // ---- this split's partial; the last CTA of (stream, g) folds all splits in order.
        // The CTA barrier orders every thread's partial before thread 0's counter update
        // (acquire-release), which also makes the other CTAs' partials visible to the last CTA.
        const int hq = g * kG + hh;
        if (!aborted) {
            job.part_o[((long long)hq * c.S + sl) * kD + row] = o;
            if ((warp & 3) == 0 && lane == 0)
                *reinterpret_cast<float2*>(job.part_ml + ((long long)hq * c.S + sl) * 2) = make_float2(m, l);
        }
        __syncthreads();
        if (tid == 0) {
            const unsigned prev = atom_add_acq_rel_gpu(job.counters + g, 1u);
            s_last = prev == (unsigned)(job.n_splits - 1);
        }
        __syncthreads();
        if (s_last) {
            // The fold of split u is (m, l, o) <- (max(m, m_u), l a_u + l_u b_u, o a_u + o_u b_u)
            // with a_u = 2^(m - max), b_u = 2^(m_u - max): the coefficients depend on the
            // head only, so the head's first warp computes them once (the running max is an
            // exact prefix max), and every thread replays the same FMA chain for its dim.
            const int ns = job.n_splits;
            float* coef = red_m;  // [4 heads][32 splits][a, b, l_u]: reuses the reduction area
            // this dim's partials of the first kMergeGroup splits: in flight while the coefficients
            // are computed
            const float* po = job.part_o + (long long)hq * c.S * kD + row;
            float ov0[kMergeGroup];
#pragma unroll
            for (int u = 0; u < kMergeGroup; ++u)
                ov0[u] = u < ns ? __ldcg(po + (long long)u * kD) : 0.f;
            if ((warp & 3) == 0) {
                float2 mlv = make_float2(-INFINITY, 0.f);
                if (lane < ns)
                    mlv = __ldcg(reinterpret_cast<const float2*>(job.part_ml + ((long long)hq * c.S + lane) * 2));
                float mpre = mlv.x;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float t = __shfl_up_sync(0xFFFFFFFFu, mpre, off);
                    if (lane >= off)
                        mpre = fmaxf(mpre, t);
                }
                float mprev = __shfl_up_sync(0xFFFFFFFFu, mpre, 1);
                if (lane == 0)
                    mprev = -INFINITY;
                coef[(hh * 32 + lane) * 3 + 0] = ex2(__fsub_rn(mprev, mpre));
                coef[(hh * 32 + lane) * 3 + 1] = ex2(__fsub_rn(mlv.x, mpre));
                coef[(hh * 32 + lane) * 3 + 2] = mlv.y;
            }
            head_sync(hh);
            const float* cf = coef + hh * 32 * 3;
            float oo = 0.f, ll = 0.f;
            for (int u0 = 0; u0 < ns; u0 += kMergeGroup) {
                float ov[kMergeGroup];
#pragma unroll
                for (int u = 0; u < kMergeGroup; ++u)
                    ov[u] = u0 == 0 ? ov0[u] : (u0 + u < ns ? __ldcg(po + (long long)(u0 + u) * kD) : 0.f);
#pragma unroll
                for (int u = 0; u < kMergeGroup; ++u) {
                    if (u0 + u < ns) {
                        const float a = cf[(u0 + u) * 3], b = cf[(u0 + u) * 3 + 1], lu = cf[(u0 + u) * 3 + 2];
                        ll = __fmaf_rn(ll, a, __fmul_rn(lu, b));
                        oo = __fmaf_rn(oo, a, __fmul_rn(ov[u], b));
                    }
                }
            }
            job.out[(long long)hq * kD + row] = __float2bfloat16_rn(__fdiv_rn(oo, ll));
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
    static std::atomic<unsigned long long> configured{0};
    const uint32_t smem = Layout::kSmemBytes;
    const cudaError_t e = smem_limit_once(configured, dec_step_kernel<J>, (int)smem);
    if (e != cudaSuccess)
        return e;
    const dim3 grid((unsigned)total_work, (unsigned)p.c.Hk);
    return launch_pdl(dec_step_kernel<J>, grid, dim3(kThreads), smem, s, p);
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
