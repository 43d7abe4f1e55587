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
// With a right lookahead (offline clips, "Moonshine streaming forward map", Encoder table,
// per-layer sliding-window mask row), frame i also sees [i+1, i+right] of the batch, right
// being EncAttnCommon::right (the host passes the mask's R - 1: "0 < j - i < R"); right is 0
// on the streaming path.
//
// Keys are visited in tiles of 128 ABSOLUTE positions [128t, 128t+128), loaded whole by
// TMA from ring slots 128t - abs_base (rows outside the ring read as zero): the batch's own
// rows were rotated and appended to the ring by kernel (a) (rope_append.cu) just before
// this launch. Per tile:
//   S   = Q' K'^T      tcgen05.mma M=128 N=128 K=64, A/B K-major bf16 in smem, D in TMEM
//   softmax            tile-local max m_t, p = 2^(s*log2e/sqrt(D) - m_t), l_t = sum p;
//                      P -> TMEM as bf16 pairs, over the S columns already read
//   O_t = P V          tcgen05.mma M=128 N=32 K=128 per 32 output dims, A = P from TMEM,
//                      B = V (MN-major smem)
//   fold               (m, l, o) <- fold((m, l, o), (m_t, l_t, O_t)), ascending t
// A tile where a row sees no key is skipped for that row (exact no-op).
//
// Threads: 288 per CTA, two CTAs per SM. Eight softmax warps: query row r (TMEM lane r) is
// shared by the two threads (r, half), one in each group of four warps; thread (r, half)
// owns score columns [64 half, 64 half + 64), output dims [32 half, 32 half + 32) and RoPE
// pairs [16 half, 16 half + 16). Row max and row sum are combined from the two halves
// through shared memory, (Q0 + Q1) + (Q2 + Q3) (enc_common.cuh). One control warp issues
// the TMA loads and the MMAs (converged, through its elected lane).
//
// Tensor memory: two 128-column buffers; tile t uses buffer (t - t_lo) & 1, whose columns
// [64 half, 64 half + 64) belong to thread (r, half): they first hold its 64 scores of S_t,
// then its 64 probabilities P_t as bf16 pairs in [64 half, 64 half + 32) (each written over
// scores the thread has already read) and output dims [32 half, 32 half + 32) of O_t in
// [64 half + 32, 64 half + 64), so no thread writes columns another still reads. Per tile,
// each softmax thread takes the row max of S_t, then folds O_{t-1} (PV_{t-1} ran meanwhile;
// the fold frees the other buffer for S_{t+1}), then takes the exps and writes P_t.
//
// Launch shape (loop): one CTA per (context, head, 128-query tile) folds its key tiles in
// registers. The split shape for a single query tile (enc_attn_split.cu) gives the same
// bits: tiles are fixed by absolute position and folded in ascending order, every row's
// arithmetic comes from enc_common.cuh, and both shapes' P V products read the same bf16 P
// values from tensor memory (as two N = 32 products here, one N = 64 product there).
#include "common.cuh"
#include "enc_common.cuh"
#include "ptx.cuh"
#include "vst_internal.h"

namespace vst {

namespace {

constexpr int kSoftmaxThreads = 256;               // warps 0-7: two threads per query row
constexpr int kThreads = kSoftmaxThreads + 32;     // warp 8: TMA and MMA issue
constexpr int kD = 64;
constexpr int kDh = kD / 2;                        // output dims per thread
constexpr uint32_t kTileBytes = 128u * 128u;       // 128 rows x 128 B
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;     // two K buffers
constexpr uint32_t kOffV = kOffK + 2 * kTileBytes;
constexpr uint32_t kOffCs = kOffV + kTileBytes;    // (cos, sin) rows of the queries: 128 x 256 B; once
                                                   // Q' is rotated, its first 16 KB are V buffer 1
constexpr uint32_t kOffRedM = kOffCs + 2 * kTileBytes;  // float [2 tile parities][2 halves][128]
constexpr uint32_t kOffRedL = kOffRedM + 2 * 2 * 128 * 4;
constexpr uint32_t kOffBar = kOffRedL + 2 * 2 * 128 * 4;
constexpr int kNumBars = 14;
constexpr uint32_t kSmemBytes = kOffBar + 8 * kNumBars + 1024;  // + slack to align the base to 1024
constexpr uint32_t kTmemCols = 256;  // two 128-column buffers (S_t, then P_t and O_t)
constexpr uint32_t kTmO = 32;        // output dims [32 h, 32 h + 32) at columns 64 h + kTmO of a buffer

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 32, false, true);

// mbarriers (index = bit in the phase and pending masks)
constexpr int kBarK = 0;      // 0, 1: K buffer landed (TMA)
constexpr int kBarV = 2;      // V buffer 0 landed (TMA); buffer 1: kBarV1
constexpr int kBarS = 3;      // 3, 4: S in TMEM buffer ready (MMA commit)
constexpr int kBarO = 5;      // 5, 6: O in TMEM buffer ready (MMA commit)
constexpr int kBarFree = 7;   // 7, 8: O in TMEM buffer read by all eight softmax warps
constexpr int kBarP = 9;      // 9, 10: P keys [64 half, 64 half + 64) written by the four warps of that half
constexpr int kBarQ = 11;     // Q' written by all eight softmax warps
constexpr int kBarQin = 12;   // raw queries and their (cos, sin) rows landed (TMA)
constexpr int kBarV1 = 13;    // V buffer 1 landed (TMA)
constexpr uint32_t kQinBytes = kTileBytes + 128u * kD * 4u;  // 128 query rows + 128 table rows

}  // namespace

// Two CTAs per SM: nine warps each, so one SM sub-partition holds five warps, which caps a
// thread at 96 registers (5 x 32 x 96 of its 16,384).
template <int J>
__global__ void __launch_bounds__(kThreads, 2)
    enc_attn_kernel(const __grid_constant__ KParams<EncAttnCommon, EncAttnJob, J> p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    const EncAttnCommon& c = p.c;
    // Launch order. Plain: query tile fastest, so the query tiles of a (context, head), which
    // share most of their key tiles, run side by side and read them once into L2. With lpt
    // (set when all the (context, head) pairs of the launch fit on the GPU at once, so that
    // neighbouring query tiles still run together): the query tile slowest and the last one
    // first, so that the first query tiles of a clip, which see fewer key tiles, come last and
    // leave a shorter tail.
    unsigned qi = blockIdx.x, hi = blockIdx.y, zi = blockIdx.z;
    if (c.lpt) {
        const unsigned n_hz = gridDim.y * gridDim.z;
        const unsigned lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        qi = gridDim.x - 1 - lin / n_hz;
        hi = (lin % n_hz) % gridDim.y;
        zi = (lin % n_hz) / gridDim.y;
    }
    const EncAttnJob& job = p.jobs[zi];
    const int h = (int)hi;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = (int)qi * 128;
    const int nrows = min(128, c.n_rows - row0);
    const long long p_first = job.pos0 + row0;
    const long long key_last = job.pos0 + c.n_rows - 1;  // last key of the batch
    const long long t_lo = max(0LL, p_first - c.W + 1) / 128;
    const long long t_hi = min(p_first + nrows - 1 + c.right, key_last) / 128;

    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sCs = smem + kOffCs;
    float* red_m = reinterpret_cast<float*>(smem + kOffRedM);  // [parity][half][128]
    float* red_l = reinterpret_cast<float*>(smem + kOffRedL);
    const uint32_t bar0 = smem_u32(smem + kOffBar);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    if (warp == 8) {
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < kNumBars; ++i)
                mbar_init(bar(i), i == kBarP || i == kBarP + 1 ? 4u : (i >= kBarFree && i <= kBarQ) ? 8u : 1u);
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    int aborted = 0;

    if (warp == 8) {
        // ================= control warp: TMA loads and MMA issue =================
        // Key tile t uses TMEM, K and V buffers (t - t_lo) & 1. For tile t:
        //   K_{t+1} landed, O_{t-1} read by every softmax warp -> S_{t+1} = Q' K_{t+1}^T
        //   S_t done -> fetch K_{t+2} into the buffer K_t used
        //   V_t landed, P_t keys [0, 64) written -> first four K steps of O_t dims [0, 32) = P_t V_t
        //   (A from TMEM); P_t keys [64, 128) written -> the last four, then all eight of dims
        //   [32, 64) (their accumulator overlays the scores of keys [96, 128))
        //   O_t done -> fetch V_{t+2} into the buffer V_t used
        // The whole warp runs this code; the elected lane alone issues copies and MMAs.
        const uint32_t e = elect_one_sync();
        uint32_t ph = 0, pend = 0;  // pend: copies and MMAs started and not yet seen complete
        int fail = 0;
        auto wait = [&](int i) {  // the same answer in every lane
            const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(i), (ph >> i) & 1u));
            if (ok) {
                ph ^= 1u << i;
                pend &= ~(1u << i);
            }
            return ok;
        };
        auto issue_k = [&](long long t) {
            const int kb = (int)((t - t_lo) & 1);
            if (e) {
                mbar_arrive_expect_tx(bar(kBarK + kb), kTileBytes);
                tma_load_3d(smem_u32(smem + kOffK) + kb * kTileBytes, job.tmap_k, bar(kBarK + kb), 0,
                            (int)(t * 128 - job.abs_base), h);
            }
            pend |= 1u << (kBarK + kb);
        };
        auto v_buf = [&](long long t) { return smem_u32(smem + (((t - t_lo) & 1) ? kOffCs : kOffV)); };
        auto v_bar = [&](long long t) { return ((t - t_lo) & 1) ? kBarV1 : kBarV; };
        auto issue_v = [&](long long t) {
            if (e) {
                mbar_arrive_expect_tx(bar(v_bar(t)), kTileBytes);
                tma_load_3d(v_buf(t), job.tmap_v, bar(v_bar(t)), 0, (int)(t * 128 - job.abs_base), h);
            }
            pend |= 1u << v_bar(t);
        };
        auto issue_s = [&](long long t) {
            const int b = (int)((t - t_lo) & 1);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss_if(tmem + 128u * b, smem_desc_sw128(smem_u32(sQ) + 32 * kk, 16, 1024),
                               smem_desc_sw128(smem_u32(smem + kOffK) + b * kTileBytes + 32 * kk, 16, 1024), kIdescS,
                               kk > 0 ? 1u : 0u, e);
            mma_commit_if(bar(kBarS + b), e);
            pend |= 1u << (kBarS + b);
        };
        // K steps [k0, k1) (keys [16 k0, 16 k1)) of output dims [32 nh, 32 nh + 32): A = P_t, whose
        // keys [64 kh, 64 kh + 64) sit in columns [64 kh, 64 kh + 32) of the buffer, 16 keys per
        // eight columns; B = V_t's dims [32 nh, 32 nh + 32) (64 bytes into each row)
        auto issue_pv = [&](long long t, int nh, int kh) {  // K steps [4 kh, 4 kh + 4)
            const uint32_t tb = tmem + 128u * (uint32_t)((t - t_lo) & 1);
            const uint64_t vd = smem_desc_sw128(v_buf(t) + 8192 * kh + 64 * nh, kTileBytes, 1024);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)  // the descriptor's address field counts 16-byte units
                mma_bf16_ts_if(tb + 64u * nh + kTmO, tb + 64u * kh + 8u * k4, vd + (uint64_t)(128 * k4), kIdescO,
                               kh > 0 || k4 > 0 ? 1u : 0u, e);
        };
        auto issue_first = [&]() {
            issue_k(t_lo);
            if (t_lo < t_hi)
                issue_k(t_lo + 1);
            issue_v(t_lo);
        };

        // The first ring tiles may be requested before the previous kernel in the stream has
        // finished when the host says that kernel did not touch this ring (early). The rows of
        // the constant (cos, sin) table go at once, the queries once the previous kernel is done.
        if (e) {
            tmap_acquire(job.tmap_k);
            tmap_acquire(job.tmap_v);
            tmap_acquire(c.tmap_rope);
            mbar_arrive_expect_tx(bar(kBarQin), kQinBytes);
            tma_load_2d(smem_u32(sCs), c.tmap_rope, bar(kBarQin), 0, (int)p_first);
        }
        pend |= 1u << kBarQin;  // waited by the softmax warps; here only after a failure
        if (c.early)
            issue_first();
        griddep_wait();
        if (e)
            tma_load_4d(smem_u32(sQ), &c.tmap_q, bar(kBarQin), 0, h, row0, job.q_z);
        if (!c.early)
            issue_first();
        if (!wait(kBarQ) || !wait(kBarK)) {
            fail = 1;
        } else {
            issue_s(t_lo);
            if (t_lo < t_hi)
                issue_v(t_lo + 1);  // the (cos, sin) rows are no longer needed
        }

        for (long long t = t_lo; !fail && t <= t_hi; ++t) {
            const int b = (int)((t - t_lo) & 1), nb = b ^ 1;
            if (t < t_hi) {
                if (!wait(kBarK + nb) || (t > t_lo && !wait(kBarFree + nb))) {
                    fail = 1;
                    break;
                }
                tc_fence_after();
                issue_s(t + 1);
            }
            if (t + 2 <= t_hi) {
                if (!wait(kBarS + b)) {
                    fail = 1;
                    break;
                }
                issue_k(t + 2);
            }
            if (!wait(v_bar(t)) || !wait(kBarP)) {
                fail = 1;
                break;
            }
            tc_fence_after();
            issue_pv(t, 0, 0);
            if (!wait(kBarP + 1)) {
                fail = 1;
                break;
            }
            tc_fence_after();
            issue_pv(t, 0, 1);
            issue_pv(t, 1, 0);
            issue_pv(t, 1, 1);
            mma_commit_if(bar(kBarO + b), e);
            pend |= 1u << (kBarO + b);
            if (t + 2 <= t_hi) {
                if (!wait(kBarO + b)) {
                    fail = 1;
                    break;
                }
                issue_v(t + 2);
            }
        }
        if (fail) {
            // A bounded wait gave up: record it and let copies and MMAs in flight land.
            if (e)
                atomicExch(job.err, kErrTimeout);
#pragma unroll
            for (int i = 0; i < kBarFree; ++i)
                if ((pend >> i) & 1u)
                    mbar_wait(bar(i), (ph >> i) & 1u);
            if ((pend >> kBarV1) & 1u)
                mbar_wait(bar(kBarV1), (ph >> kBarV1) & 1u);
            mbar_wait(bar(kBarQin), 0);
        }
        __syncwarp();
        griddep_launch_dependents();
    } else {
        // ================= softmax warps: two threads per query row =================
        // Thread (r, half) owns score columns [64 half, 64 half + 64), output dims
        // [32 half, 32 half + 32) and RoPE pairs [16 half, 16 half + 16) of query row r.
        const int r = 32 * (warp & 3) + lane;  // TMEM lane = query row of this thread
        const int half = warp >> 2;
        const int pair_bar = 1 + (warp & 3);   // named barrier of warps w and w + 4 (the same rows)
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const bool row_real = r < nrows;
        // keys relative to the query tile's first position: the batch's last key, and the first
        // key of the current tile
        const int kl = (int)(key_last - p_first);
        int rel = (int)(t_lo * 128 - p_first);

        griddep_wait();
        // Raw query row r (zero past the batch) and its (cos, sin) row landed by TMA: rotate
        // this thread's two quarters in place.
        int qfail = mbar_wait(bar(kBarQin), 0) ? 0 : 1;
        if (!qfail) {
            const float2* cs = reinterpret_cast<const float2*>(sCs + r * (kD * 4));
            enc::rotate_quarter_in_place(sQ, cs, r, 2 * half);
            enc::rotate_quarter_in_place(sQ, cs, r, 2 * half + 1);
        }
        fence_proxy_async_smem();  // Q' (generic stores) before the MMAs read it
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar(kBarQ));

        float o[kDh];
#pragma unroll
        for (int d = 0; d < kDh; ++d)
            o[d] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;
        float mt_prev = -INFINITY;  // tile-local max of the previous tile, folded one tile late
        float l_prev = 0.f;         // this thread's half of the previous tile's sum
        int fail = qfail;
        const int n_t = (int)(t_hi - t_lo + 1);
        // o <- fold(o, O_i) for tile i of the CTA, in TMEM buffer i & 1, with m_t = mt and
        // l_t = l_prev + the partner's half (ordered before this read by a pair barrier; the
        // sum is the same in either order)
        auto fold_from = [&](int i, float mt) {
            const int b = i & 1;
            if (!mbar_wait(bar(kBarO + b), (uint32_t)((i >> 1) & 1)))
                fail = 1;
            tc_fence_after();
            const float lt = __fadd_rn(l_prev, red_l[(b * 2 + (half ^ 1)) * 128 + r]);
            // in two groups of 16 dims (the same operations per dim as one group of 32)
            const enc::FoldCoef f = enc::fold_coef(m_run, mt);
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                uint32_t ov[16];
                tmem_ld_32x32b_x16(tmem + 128u * b + lane_base + 64 * half + kTmO + 16 * g, ov);
                tmem_ld_wait();
                if (mt != -INFINITY) {
                    float ot[16];
#pragma unroll
                    for (int d = 0; d < 16; ++d)
                        ot[d] = __uint_as_float(ov[d]);
                    enc::fold_apply<16>(o + 16 * g, ot, f);
                }
            }
            if (mt != -INFINITY)
                enc::fold_finish(m_run, l_run, lt, f);
        };

        for (int i = 0; i < n_t; ++i, rel += 128) {
            const int b = i & 1;

            // ---- S_i: this thread's 64 columns of row r, as two quarters of 32
            if (!mbar_wait(bar(kBarS + b), (uint32_t)((i >> 1) & 1)))
                fail = 1;
            tc_fence_after();
            const uint32_t tm_s = tmem + 128u * b + lane_base + 64 * half;  // this thread's columns
            // Every column visible to every row of the CTA (the same answer in all threads):
            // no per-column masks.
            const bool interior = nrows == 128 && rel >= 128 - c.W && min(c.right, kl) - rel >= 127;
            uint32_t mask0 = 0xffffffffu, mask1 = 0xffffffffu;
            if (!interior) {
                int lo = 1, hi = 0;  // visible columns of row r in this tile; empty unless r is real
                if (row_real) {
                    lo = max(-1, min(128, r - c.W + 1 - rel));
                    hi = max(-1, min(128, min(r + c.right, kl) - rel));
                }
                mask0 = enc::visible_mask(64 * half, lo, hi);
                mask1 = enc::visible_mask(64 * half + 32, lo, hi);
            }

            // ---- tile-local row max of row r, one quarter at a time
            float mh;
            {
                uint32_t sv[32];
                tmem_ld_32x32b_x32(tm_s, sv);
                tmem_ld_wait();
                mh = interior ? enc::quarter_max_all(sv) : enc::quarter_max(sv, mask0);
                tmem_ld_32x32b_x32(tm_s + 32, sv);
                tmem_ld_wait();
                mh = fmaxf(mh, interior ? enc::quarter_max_all(sv) : enc::quarter_max(sv, mask1));
            }
            red_m[(b * 2 + half) * 128 + r] = mh;
            if (bar_sync_or(pair_bar, 64, fail)) {  // also orders the partner's l of the previous tile
                aborted = 1;
                break;
            }
            // the two halves' maxima (exact, so the same in either order)
            const float mt = __fmul_rn(fmaxf(mh, red_m[(b * 2 + (half ^ 1)) * 128 + r]), c.scale_log2);

            // ---- fold of the previous tile (its PV ran while this tile's max was taken); frees its
            // buffer for S_{i+1}
            if (i > 0) {
                fold_from(i - 1, mt_prev);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(kBarFree + (b ^ 1)));
            }

            // ---- tile-local exps, quarter by quarter (S_i read again); P_i over this thread's
            // scores already read
            float l0, l1;
            {
                auto st0 = [&](int qd, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
                    tmem_st_32x32b_x4(tm_s + 4 * qd, w0, w1, w2, w3);
                };
                auto st1 = [&](int qd, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
                    tmem_st_32x32b_x4(tm_s + 16 + 4 * qd, w0, w1, w2, w3);
                };
                uint32_t sv[32];
                tmem_ld_32x32b_x32(tm_s, sv);
                tmem_ld_wait();
                l0 = interior ? enc::quarter_exp_core<false>(sv, mask0, c.scale_log2, -mt, st0)
                              : enc::quarter_exp_to(sv, mask0, c.scale_log2, -mt, st0);
                tmem_ld_32x32b_x32(tm_s + 32, sv);
                tmem_ld_wait();
                l1 = interior ? enc::quarter_exp_core<false>(sv, mask1, c.scale_log2, -mt, st1)
                              : enc::quarter_exp_to(sv, mask1, c.scale_log2, -mt, st1);
            }
            l_prev = __fadd_rn(l0, l1);
            red_l[(b * 2 + half) * 128 + r] = l_prev;
            tmem_st_wait();
            tc_fence_before();  // P_i written (and S_i read) before the MMAs use the columns
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(kBarP + half));
            mt_prev = mt;
        }
        // ---- fold of the last tile
        if (!aborted && bar_sync_or(pair_bar, 64, fail))  // orders the partner's l of the last tile
            aborted = 1;
        if (!aborted) {
            fold_from(n_t - 1, mt_prev);
            if (bar_sync_or(pair_bar, 64, fail))
                aborted = 1;
        }
        if (aborted && lane == 0)
            atomicExch(job.err, kErrTimeout);
        griddep_launch_dependents();
        if (!aborted && row_real)
            enc::store_out<kDh>(job.out + ((long long)(row0 + r) * c.H + h) * kD, o, l_run, kDh * half);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int J>
static cudaError_t launch_enc_attn_j(const KParams<EncAttnCommon, EncAttnJob, J>& p, int n_jobs, int grid_x,
                                     cudaStream_t s)
{
    static std::atomic<unsigned long long> configured{0};
    const cudaError_t e = smem_limit_once(configured, enc_attn_kernel<J>, (int)kSmemBytes);
    if (e != cudaSuccess)
        return e;
    const dim3 grid((unsigned)grid_x, (unsigned)p.c.H, (unsigned)n_jobs);
    return launch_pdl(enc_attn_kernel<J>, grid, dim3(kThreads), kSmemBytes, s, p);
}

cudaError_t launch_enc_attn(const EncAttnCommon& c, const EncAttnJob* jobs, int n_jobs, int grid_x, cudaStream_t s)
{
    if (n_jobs == 0 || c.n_rows == 0)
        return cudaSuccess;
    if (c.split || !c.appended || c.right < 0)
        return cudaErrorInvalidValue;  // split shape: launch_enc_attn_split; rows appended first
    return with_params(c, jobs, n_jobs, [&](const auto& p) {
        return launch_enc_attn_j<sizeof(p.jobs) / sizeof(p.jobs[0])>(p, n_jobs, grid_x, s);
    });
}

}  // namespace vst
