// enc_attn_split.cu -- kernel (b), split launch shape for small batches: windowed-causal
// chunk attention against the encoder ring, with the encoder half of kernel (a) fused in.
//
// Streaming plan ("Voxtral Realtime -- incremental streaming implementation plan"):
// SHIPPED/Mechanism -- mha_cached writes the chunk's K/V at cache rows
// [n_kv_before, n_kv_total) and reads [0, n_kv_total) under a windowed-causal mask;
// "Unbounded length" -- the mask uses absolute positions (slot 0 holds frame abs_base);
// "Chunk alignment" -- RoPE at absolute positions; "Risk / notes" -- the chunk attention is a
// multi-query prefill against <= 750 cached keys. Frame i attends to [i-749, i]
// ("RECOMMENDED implementation").
//
// Keys are visited in tiles of 128 ABSOLUTE positions [128t, 128t+128), loaded by TMA from
// ring slots 128t - abs_base (rows outside the ring read as zero). Rows of a tile that
// belong to this batch (positions >= pos0) are not in the ring yet: every CTA that loads
// such a tile rotates those keys itself from the input and patches them into shared
// memory; the CTA whose query tile holds a new row also stores it (K rotated, V) to ring
// slot n_kv_before + row. Per tile:
//   S   = Q' K'^T      tcgen05.mma M=128 N=128 K=64, A/B K-major bf16 in smem, D in TMEM
//   softmax            tile-local max m_t, p = 2^(s*log2e/sqrt(D) - m_t), l_t = sum p;
//                      P -> TMEM as bf16 pairs, over the S columns already read
//   O_t = P V          tcgen05.mma M=128 N=64 K=128, A = P from TMEM, B = V (MN-major smem)
//   fold               (m, l, o) <- fold((m, l, o), (m_t, l_t, O_t)), ascending t
// A tile where a row sees no key is skipped for that row (exact no-op).
//
// Threads: 512 per CTA. Query row r (TMEM lane r) is shared by the four threads
// (r, q), q = 0..3, one in each group of four warps: thread (r, q) owns score columns
// [32q, 32q+32), output dims [16q, 16q+16) and RoPE pairs [8q, 8q+8). Row max and row sum
// are combined from the four quarters through shared memory, (Q0 + Q1) + (Q2 + Q3).
//
// Launch shape (split): for a batch of a single query tile, one CTA per (context, head,
// group of `split` consecutive key tiles), with groups just large enough that every CTA
// starts in the first wave. The CTA of the last group (the merger) folds every tile of the
// (context, head) in ascending order, with the fold of enc_common.cuh. The others write
// each tile's (m_t, l_t, O_t) to scratch and count themselves in with one releasing
// increment; the merger keeps its own last tile in shared memory and waits (bounded) for
// the count, so its handoff costs one acquiring poll and no fence. The first tile's new rows are rotated and stored to the ring in the
// prologue, so their global loads overlap those of the queries. The loop shape
// (enc_attn.cu) gives the same bits: tiles are fixed by absolute position, folded in
// ascending order, and every row's arithmetic comes from enc_common.cuh.
#include "common.cuh"
#include "enc_common.cuh"
#include "ptx.cuh"
#include "vst_internal.h"

namespace vst {

namespace {

constexpr int kThreads = 512;
constexpr int kD = 64;
constexpr int kDq = kD / 4;                   // output dims per thread
constexpr uint32_t kTileBytes = 128u * 128u;  // 128 rows x 128 B
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kTileBytes;
constexpr uint32_t kOffP = kOffV + kTileBytes;       // the merger's own tile partial: O as [row][64] floats
constexpr uint32_t kOffRed = kOffP + 2 * kTileBytes; // float [2][4][128]: row max / row sum quarters
constexpr uint32_t kOffKn = kOffRed + 2 * 4 * 128 * 4; // split mode: new rows of the first key tile,
constexpr uint32_t kOffVn = kOffKn + kTileBytes;       // K rotated and V, staged in the prologue
constexpr uint32_t kOffBar = kOffVn + kTileBytes;
constexpr uint32_t kSmemBytes = kOffBar + 64 + 1024;  // + slack to align the base to 1024
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmS = 0;    // S tile: columns [0, 128)
constexpr uint32_t kTmO = 128;  // O tile: columns [128, 192)

constexpr int kMergeGroup = 8;  // tile partials loaded together by the merger

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 64, false, true);

using enc::quarter_max;
using enc::rotate_quarter;

struct Cta {
    uint8_t *sQ, *sK, *sV, *sP, *sKn, *sVn;
    float *red_m, *red_l;  // [4][128]
    uint32_t bar_k, bar_v, bar_m;
    uint32_t tmem, lane_base;
    int tid, warp, r, q;
};

// New rows of key tile t (positions >= pos0) are not in the ring yet: thread (r, q) replaces
// its quarter of row r of the smem tile with K' = RoPE(k) (is_k) or V from the input; the
// CTA whose query tile owns the row also stores that quarter to ring slot slot0 + row.
__device__ __forceinline__ void patch_new_row(const Cta& s, const EncAttnCommon& c, const EncAttnJob& job, int h,
                                              long long t, int own_lo, int own_hi, bool is_k)
{
    const long long p = t * 128 + s.r;
    const long long i = p - job.pos0;  // batch row
    if (i < 0 || i >= c.n_rows)
        return;
    uint8_t* tile = is_k ? s.sK : s.sV;
    int ch0, ch1;
    if (is_k) {
        rotate_quarter(job.k + (i * c.H + h) * kD, c.rope + p * (kD / 2), tile, s.r, s.q);
        ch0 = s.q;
        ch1 = 4 + s.q;
    } else {
        const __nv_bfloat16* vrow = job.v + (i * c.H + h) * kD;
        ch0 = 2 * s.q;
        ch1 = 2 * s.q + 1;
        *reinterpret_cast<uint4*>(tile + sw128_offset(s.r, ch0)) = *reinterpret_cast<const uint4*>(vrow + 8 * ch0);
        *reinterpret_cast<uint4*>(tile + sw128_offset(s.r, ch1)) = *reinterpret_cast<const uint4*>(vrow + 8 * ch1);
    }
    if (i >= own_lo && i < own_hi) {
        __nv_bfloat16* ring = (is_k ? job.k_ring : job.v_ring) + ((long long)h * c.R + (job.slot0 + i)) * kD;
        *reinterpret_cast<uint4*>(ring + 8 * ch0) = *reinterpret_cast<const uint4*>(tile + sw128_offset(s.r, ch0));
        *reinterpret_cast<uint4*>(ring + 8 * ch1) = *reinterpret_cast<const uint4*>(tile + sw128_offset(s.r, ch1));
    }
}

// Split mode prologue: thread (r, q) rotates its quarter of new row r of key tile t (if that
// row is new) into the staging tiles and stores it to the ring, so that the global loads of
// the new rows overlap those of the queries; returns whether row r of tile t is new.
__device__ __forceinline__ bool stage_new_row(const Cta& s, const EncAttnCommon& c, const EncAttnJob& job, int h,
                                              long long t)
{
    const long long p = t * 128 + s.r;
    const long long i = p - job.pos0;  // batch row
    if (i < 0 || i >= c.n_rows)
        return false;
    rotate_quarter(job.k + (i * c.H + h) * kD, c.rope + p * (kD / 2), s.sKn, s.r, s.q);
    const __nv_bfloat16* vrow = job.v + (i * c.H + h) * kD;
    const uint4 v0 = *reinterpret_cast<const uint4*>(vrow + 16 * s.q);
    const uint4 v1 = *reinterpret_cast<const uint4*>(vrow + 16 * s.q + 8);
    *reinterpret_cast<uint4*>(s.sVn + sw128_offset(s.r, 2 * s.q)) = v0;
    *reinterpret_cast<uint4*>(s.sVn + sw128_offset(s.r, 2 * s.q + 1)) = v1;
    __nv_bfloat16* kring = job.k_ring + ((long long)h * c.R + (job.slot0 + i)) * kD;
    __nv_bfloat16* vring = job.v_ring + ((long long)h * c.R + (job.slot0 + i)) * kD;
    *reinterpret_cast<uint4*>(kring + 8 * s.q) = *reinterpret_cast<const uint4*>(s.sKn + sw128_offset(s.r, s.q));
    *reinterpret_cast<uint4*>(kring + 32 + 8 * s.q) =
        *reinterpret_cast<const uint4*>(s.sKn + sw128_offset(s.r, 4 + s.q));
    *reinterpret_cast<uint4*>(vring + 16 * s.q) = v0;
    *reinterpret_cast<uint4*>(vring + 16 * s.q + 8) = v1;
    return true;
}

// Copy this thread's chunks of a staged row into the loaded tile.
__device__ __forceinline__ void unstage_row(const Cta& s, bool is_k)
{
    const int ch0 = is_k ? s.q : 2 * s.q, ch1 = is_k ? 4 + s.q : 2 * s.q + 1;
    const uint8_t* src = is_k ? s.sKn : s.sVn;
    uint8_t* dst = is_k ? s.sK : s.sV;
    *reinterpret_cast<uint4*>(dst + sw128_offset(s.r, ch0)) = *reinterpret_cast<const uint4*>(src + sw128_offset(s.r, ch0));
    *reinterpret_cast<uint4*>(dst + sw128_offset(s.r, ch1)) = *reinterpret_cast<const uint4*>(src + sw128_offset(s.r, ch1));
}

// Issued by the whole of warp 0 (converged); the elected lane `e` executes the MMAs.
__device__ __forceinline__ void issue_s_mma(const Cta& s, uint32_t e)
{
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = smem_desc_sw128(smem_u32(s.sQ) + 32 * kk, 16, 1024);
        const uint64_t bd = smem_desc_sw128(smem_u32(s.sK) + 32 * kk, 16, 1024);
        mma_bf16_ss_if(s.tmem + kTmS, ad, bd, kIdescS, kk > 0 ? 1u : 0u, e);
    }
    mma_commit_if(s.bar_m, e);
}

// O = P V: A = P from tensor memory (keys [32 q, 32 q + 32) as bf16 pairs in columns
// [32 q, 32 q + 16), written by the threads of quarter q over scores they have read; 16 keys
// per eight columns), B = V (MN-major shared memory, 16 keys per K step).
__device__ __forceinline__ void issue_o_mma(const Cta& s, uint32_t e)
{
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a = s.tmem + kTmS + 32u * (kk >> 1) + 8u * (kk & 1);
        const uint64_t bd = smem_desc_sw128(smem_u32(s.sV) + 2048 * kk, kTileBytes, 1024);
        mma_bf16_ts_if(s.tmem + kTmO, a, bd, kIdescO, kk > 0 ? 1u : 0u, e);
    }
    mma_commit_if(s.bar_m, e);
}

}  // namespace

template <int J>
__global__ void __launch_bounds__(kThreads, 1)
    enc_attn_split_kernel(const __grid_constant__ KParams<EncAttnCommon, EncAttnJob, J> p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    __shared__ int s_last;
    const EncAttnCommon& c = p.c;
    const EncAttnJob& job = p.jobs[blockIdx.z];
    const int h = blockIdx.y;
    const int row0 = 0;  // a single query tile
    const int nrows = min(128, c.n_rows - row0);
    const long long p_first = job.pos0 + row0;
    const long long p_last = p_first + nrows - 1;
    const long long t_lo = max(0LL, p_first - c.W + 1) / 128;
    const long long t_hi = p_last / 128;
    const long long t_begin = t_lo + (long long)blockIdx.x * c.split;
    const long long t_end = min(t_begin + c.split - 1, t_hi);
    if (t_begin > t_hi)
        return;  // this job has fewer tiles than the grid

    Cta s;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    s.sQ = smem + kOffQ;
    s.sK = smem + kOffK;
    s.sV = smem + kOffV;
    s.sP = smem + kOffP;
    s.sKn = smem + kOffKn;
    s.sVn = smem + kOffVn;
    s.red_m = reinterpret_cast<float*>(smem + kOffRed);
    s.red_l = s.red_m + 4 * 128;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    s.bar_k = smem_u32(&bars[0]);
    s.bar_v = smem_u32(&bars[1]);
    s.bar_m = smem_u32(&bars[2]);
    s.tid = threadIdx.x;
    s.warp = s.tid >> 5;
    s.r = 32 * (s.warp & 3) + (s.tid & 31);  // TMEM lane = query row of this thread
    s.q = s.warp >> 2;                       // quarter of the row

    // Prologue. The first ring tiles may be requested before the previous kernel in the
    // stream has finished when the host says that kernel did not touch this ring (early);
    // everything else waits for it.
    auto issue_first_tile = [&]() {
        const int slot = (int)(t_begin * 128 - job.abs_base);
        mbar_arrive_expect_tx(s.bar_k, kTileBytes);
        tma_load_3d(smem_u32(s.sK), job.tmap_k, s.bar_k, 0, slot, h);
        mbar_arrive_expect_tx(s.bar_v, kTileBytes);
        tma_load_3d(smem_u32(s.sV), job.tmap_v, s.bar_v, 0, slot, h);
    };
    if (s.tid == 0) {
        mbar_init(s.bar_k, 1);
        mbar_init(s.bar_v, 1);
        mbar_init(s.bar_m, 1);
        fence_mbar_init();
        tmap_acquire(job.tmap_k);
        tmap_acquire(job.tmap_v);
        if (c.early)
            issue_first_tile();
    }
    if (s.warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    // What the prologue reads right after the wait -- row r's query and (cos, sin) row and,
    // if row r of the first key tile is new, its K and V -- is pulled into L2 now, one
    // 128- or 256-byte prefetch per thread, so that those loads hit L2.
    {
        const long long i = t_begin * 128 + s.r - job.pos0;  // batch row at row r of the first tile
        if (s.q == 0 && s.r < nrows)
            prefetch_l2(job.q + ((long long)(row0 + s.r) * c.H + h) * kD, kD * 2);
        else if (s.q == 1 && s.r < nrows)
            prefetch_l2(c.rope + (p_first + s.r) * (kD / 2), kD * 4);
        else if (s.q >= 2 && i >= 0 && i < c.n_rows)
            prefetch_l2((s.q == 2 ? job.k : job.v) + (i * c.H + h) * kD, kD * 2);
    }
    griddep_wait();
    if (s.tid == 0 && !c.early)
        issue_first_tile();

    // ---- this thread's quarter of query row r, rotated, into sQ
    const int r = s.r;
    const long long pq = p_first + r;
    if (r < nrows) {
        rotate_quarter(job.q + ((long long)(row0 + r) * c.H + h) * kD, c.rope + pq * (kD / 2), s.sQ, r, s.q);
    } else {
        *reinterpret_cast<uint4*>(s.sQ + sw128_offset(r, s.q)) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(s.sQ + sw128_offset(r, 4 + s.q)) = make_uint4(0, 0, 0, 0);
    }
    // the first key tile's new rows are rotated and stored to the ring now
    const bool staged = (t_begin + 1) * 128 > job.pos0 && stage_new_row(s, c, job, h, t_begin);
    // (the loop's first CTA barrier publishes these shared-memory writes and the TMEM address)
    s.lane_base = (uint32_t)((s.warp & 3) * 32) << 16;

    uint32_t ph_k = 0, ph_v = 0, ph_m = 0;
    bool pend_k = s.tid == 0, pend_v = s.tid == 0;
    // The CTA of the last key tiles (the merger) folds every tile of (job, head); the others
    // publish their tile partials to scratch and count themselves in.
    const long long others = (t_hi - t_lo) / c.split;
    const bool merger = (long long)blockIdx.x == others;
    const uint32_t elect = s.warp == 0 ? elect_one_sync() : 0u;  // lane of warp 0 that issues MMAs
    int fail = 0, aborted = 0;

    for (long long t = t_begin; t <= t_end; ++t) {
        const bool has_new = (t + 1) * 128 > job.pos0;
        // ---- K of tile t in smem (new rows patched in), then S = Q K^T
        if (!mbar_wait(s.bar_k, ph_k))
            fail = 1;
        ph_k ^= 1;
        if (s.tid == 0)
            pend_k = false;
        if (!fail && has_new) {
            if (t == t_begin) {
                if (staged)
                    unstage_row(s, true);
            } else {
                patch_new_row(s, c, job, h, t, row0, row0 + nrows, true);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        const int any_fail = __syncthreads_or(fail);
        s.tmem = s_tmem;
        if (any_fail) {
            aborted = 1;
            break;
        }
        tc_fence_after();
        if (s.warp == 0)
            issue_s_mma(s, elect);
        if (!mbar_wait(s.bar_m, ph_m))
            fail = 1;
        ph_m ^= 1;
        tc_fence_after();
        if (s.tid == 0 && !fail && t < t_end) {  // K buffer is free: fetch the next tile's K
            mbar_arrive_expect_tx(s.bar_k, kTileBytes);
            tma_load_3d(smem_u32(s.sK), job.tmap_k, s.bar_k, 0, (int)((t + 1) * 128 - job.abs_base), h);
            pend_k = true;
        }

        // ---- tile-local softmax: this thread's 32 columns of row r
        const long long kbase = t * 128;
        int lo = 1, hi = 0;  // visible columns of row r in this tile; empty unless r is real
        if (r < nrows) {
            lo = (int)max(-1LL, min(128LL, pq - c.W + 1 - kbase));
            hi = (int)max(-1LL, min(128LL, pq - kbase));
        }
        const int c0 = 32 * s.q;
        uint32_t sv[32];
        tmem_ld_32x32b_x32(s.tmem + s.lane_base + kTmS + c0, sv);
        tmem_ld_wait();
        const uint32_t vmask = enc::visible_mask(c0, lo, hi);
        s.red_m[s.q * 128 + r] = quarter_max(sv, vmask);
        // the four warps that hold rows [32 (warp & 3), +32) meet on their own barrier
        __syncwarp();
        asm volatile("bar.sync %0, 128;" ::"r"(1 + (s.warp & 3)) : "memory");
        const float mraw = fmaxf(fmaxf(s.red_m[r], s.red_m[128 + r]), fmaxf(s.red_m[256 + r], s.red_m[384 + r]));
        const float mt = __fmul_rn(mraw, c.scale_log2);  // -inf when the row sees nothing here
        {
            // P over this thread's scores already read, four columns at a time
            const uint32_t tm_q = s.tmem + s.lane_base + kTmS + c0;
            s.red_l[s.q * 128 + r] = enc::quarter_exp_to(
                sv, vmask, c.scale_log2, -mt, [&](int qd, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
                    tmem_st_32x32b_x4(tm_q + 4 * qd, w0, w1, w2, w3);
                });
            tmem_st_wait();
        }

        // ---- V of tile t in smem (new rows patched in), then O_t = P V
        if (!mbar_wait(s.bar_v, ph_v))
            fail = 1;
        ph_v ^= 1;
        if (s.tid == 0)
            pend_v = false;
        if (!fail && has_new) {
            if (t == t_begin) {
                if (staged)
                    unstage_row(s, false);
            } else {
                patch_new_row(s, c, job, h, t, row0, row0 + nrows, false);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(fail)) {
            aborted = 1;
            break;
        }
        tc_fence_after();
        if (s.warp == 0)
            issue_o_mma(s, elect);
        const float lt = __fadd_rn(__fadd_rn(s.red_l[r], s.red_l[128 + r]), __fadd_rn(s.red_l[256 + r], s.red_l[384 + r]));
        if (!mbar_wait(s.bar_m, ph_m))
            fail = 1;
        ph_m ^= 1;
        tc_fence_after();
        if (s.tid == 0 && !fail && t < t_end) {  // V buffer is free: fetch the next tile's V
            mbar_arrive_expect_tx(s.bar_v, kTileBytes);
            tma_load_3d(smem_u32(s.sV), job.tmap_v, s.bar_v, 0, (int)((t + 1) * 128 - job.abs_base), h);
            pend_v = true;
        }

        float ot[kDq];
        {
            uint32_t ov[16];
            tmem_ld_32x32b_x16(s.tmem + s.lane_base + kTmO + kDq * s.q, ov);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < kDq; ++j)
                ot[j] = __uint_as_float(ov[j]);
        }
        if (r < nrows) {
            if (merger && t == t_hi) {
                // the merger's own last tile stays in shared memory: O as [row][64] floats in
                // the P buffer (the PV MMA that read it has completed), (m_t, l_t) per row in
                // the row-max area (last read before the barrier after V landed)
                float* lo_o = reinterpret_cast<float*>(s.sP) + r * kD + kDq * s.q;
#pragma unroll
                for (int d = 0; d < kDq; d += 4)
                    *reinterpret_cast<float4*>(lo_o + d) = make_float4(ot[d], ot[d + 1], ot[d + 2], ot[d + 3]);
                if (s.q == 0)
                    reinterpret_cast<float2*>(s.red_m)[r] = make_float2(mt, lt);
            } else {
                // tile partial of (row r, quarter q) -> scratch [h][tile][q][row][16]: a warp's
                // 32 rows of one quarter are 2 KB contiguous; only rows of the batch are kept
                const long long slot_t = (long long)h * c.split_tiles + (t - t_lo);
                float* po = job.part_o + ((slot_t * 4 + s.q) * 128 + r) * kDq;
#pragma unroll
                for (int d = 0; d < kDq; d += 4)
                    *reinterpret_cast<float4*>(po + d) = make_float4(ot[d], ot[d + 1], ot[d + 2], ot[d + 3]);
                if (s.q == 0)
                    *reinterpret_cast<float2*>(job.part_ml + (slot_t * 128 + r) * 2) = make_float2(mt, lt);
            }
        }
        tc_fence_before();
        if (__syncthreads_or(fail)) {
            aborted = 1;
            break;
        }
        tc_fence_after();
    }

    griddep_launch_dependents();
    if (aborted && s.tid == 0) {
        // A bounded wait gave up: record it and let copies still in flight land. The CTA
        // still takes part in the handoff below, so that the merger does not wait out its
        // own limit, then releases TMEM and leaves.
        atomicExch(job.err, kErrTimeout);
        if (pend_k)
            mbar_wait(s.bar_k, ph_k);
        if (pend_v)
            mbar_wait(s.bar_v, ph_v);
    }
    if (!merger) {
        // The CTA barrier that ended the last tile orders every thread's partials before
        // thread 0's releasing increment (cumulative), which the merger acquires. (After a
        // failure the partials do not matter; the count still does.)
        if (s.tid == 0)
            red_add_release_gpu(job.counters + h, 1u);
    } else {
        if (t_end > t_begin) {
            __threadfence();  // this CTA's own earlier tile partials, read back from scratch below
            __syncthreads();
        }
        if (s.tid == 0) {
            // Wait until the other CTAs of (job, head) have counted themselves in, then re-arm
            // the counter for the next launch by taking their counts back out: a CTA that
            // arrives after the wait gave up still adds its one, so the counter is zero when
            // the grid ends either way. The barrier after it passes what thread 0 acquired on
            // to the readers.
            const bool all_in = wait_count(job.counters + h, (unsigned)others);
            atomicSub(job.counters + h, (unsigned)others);
            if (!all_in)
                atomicExch(job.err, kErrTimeout);
            s_last = all_in && !aborted;
        }
        __syncthreads();
        if (s_last) {
            // All threads of the CTA share the merge: item (row, g) folds dims [8g, 8g+8) of
            // a row over the tiles in ascending order, in groups of up to kMergeGroup tiles
            // whose loads are all issued before their folds. The last tile is this CTA's own,
            // from shared memory.
            const int nt = (int)(t_hi - t_lo + 1);
            const float* pml0 = job.part_ml + (long long)h * c.split_tiles * 128 * 2;
            const float* po0 = job.part_o + (long long)h * c.split_tiles * 128 * kD;
            const float* own_o = reinterpret_cast<const float*>(s.sP);
            const float2* own_ml = reinterpret_cast<const float2*>(s.red_m);
            for (int it = s.tid; it < nrows * 8; it += kThreads) {
                const int row = it >> 3, g = it & 7;  // dims [8g, 8g+8): quarter g / 2, half g % 2
                float m = -INFINITY, l = 0.f, om[8];
#pragma unroll
                for (int d = 0; d < 8; ++d)
                    om[d] = 0.f;
                for (int g0 = 0; g0 < nt; g0 += kMergeGroup) {
                    const int ng = min(kMergeGroup, nt - g0);
                    float2 ml[kMergeGroup];
                    float4 xa[kMergeGroup], xb[kMergeGroup];
#pragma unroll
                    for (int u = 0; u < kMergeGroup; ++u) {
                        ml[u] = make_float2(-INFINITY, 0.f);
                        xa[u] = xb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        const long long tile = g0 + u;
                        if (u < ng && tile == nt - 1) {
                            ml[u] = own_ml[row];
                            const float4* src = reinterpret_cast<const float4*>(own_o + row * kD + 8 * g);
                            xa[u] = src[0];
                            xb[u] = src[1];
                        } else if (u < ng) {
                            ml[u] = __ldcg(reinterpret_cast<const float2*>(pml0 + (tile * 128 + row) * 2));
                            const float* src = po0 + ((tile * 4 + (g >> 1)) * 128 + row) * kDq + 8 * (g & 1);
                            xa[u] = __ldcg(reinterpret_cast<const float4*>(src));
                            xb[u] = __ldcg(reinterpret_cast<const float4*>(src + 4));
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kMergeGroup; ++u) {
                        const float ot[8] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w, xb[u].x, xb[u].y, xb[u].z, xb[u].w};
                        enc::fold_tile_if<8>(ml[u].x != -INFINITY, m, l, om, ml[u].x, ml[u].y, ot);
                    }
                }
                enc::store_out<8>(job.out + ((long long)(row0 + row) * c.H + h) * kD, om, l, 8 * g);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (s.warp == 0) {
        tc_fence_after();
        tmem_dealloc(s.tmem, kTmemCols);
    }
}

template <int J>
static cudaError_t launch_enc_attn_split_j(const KParams<EncAttnCommon, EncAttnJob, J>& p, int n_jobs, int grid_x,
                                     cudaStream_t s)
{
    static std::atomic<unsigned long long> configured{0};
    const cudaError_t e = smem_limit_once(configured, enc_attn_split_kernel<J>, (int)kSmemBytes);
    if (e != cudaSuccess)
        return e;
    const dim3 grid((unsigned)grid_x, (unsigned)p.c.H, (unsigned)n_jobs);
    return launch_pdl(enc_attn_split_kernel<J>, grid, dim3(kThreads), kSmemBytes, s, p);
}

template <int J>
static cudaError_t split_blocks_per_sm_j(int* n)
{
    static std::atomic<unsigned long long> configured{0};
    const cudaError_t e = smem_limit_once(configured, enc_attn_split_kernel<J>, (int)kSmemBytes);
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, enc_attn_split_kernel<J>, kThreads, kSmemBytes);
}

cudaError_t enc_attn_split_blocks_per_sm(int* n)
{
    // the least over the job-table sizes a launch may use
    int a = 0, b = 0, d = 0;
    cudaError_t e = split_blocks_per_sm_j<1>(&a);
    if (e == cudaSuccess)
        e = split_blocks_per_sm_j<8>(&b);
    if (e == cudaSuccess)
        e = split_blocks_per_sm_j<kMaxJobs>(&d);
    *n = e == cudaSuccess ? min(a, min(b, d)) : 0;
    return e;
}

cudaError_t launch_enc_attn_split(const EncAttnCommon& c, const EncAttnJob* jobs, int n_jobs, int grid_x, cudaStream_t s)
{
    if (n_jobs == 0 || c.n_rows == 0)
        return cudaSuccess;
    if (c.right != 0)
        return cudaErrorInvalidValue;  // the split shape serves the streaming (causal) mask only
    return with_params(c, jobs, n_jobs, [&](const auto& p) {
        return launch_enc_attn_split_j<sizeof(p.jobs) / sizeof(p.jobs[0])>(p, n_jobs, grid_x, s);
    });
}

}  // namespace vst
