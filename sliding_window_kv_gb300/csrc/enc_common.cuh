// enc_common.cuh -- the per-row arithmetic of the chunk attention, shared by every launch
// shape of it (enc_attn.cu). Each shape splits a 128-column score row
// over a different number of threads, but all of them call these functions on the same
// 32-column quarters in the same order, so every shape produces the same bits.
//
// Row softmax of one 128-key tile, for a row whose visible columns are [lo, hi]:
//   quarter max    max over the quarter's visible columns (exact in any order)
//   row max        max of the 4 quarter maxima (exact in any order), m_t = max * log2e/sqrt(D)
//   quarter sum    p = 2^(s * log2e/sqrt(D) - m_t) over the quarter (0 where not visible),
//                  accumulated into 4 interleaved partial sums, combined (l0+l1)+(l2+l3)
//   row sum        l_t = (Q0 + Q1) + (Q2 + Q3)
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace vst {
namespace enc {

constexpr int kD = 64;
constexpr uint32_t kTileBytes = 128u * 128u;  // 128 rows x 128 B

// Visible columns of the quarter [c0, c0 + 32) as a bit mask: bit j is set iff column
// c0 + j lies in [lo, hi]. One mask and a select per column compile to straight-line code
// (a per-column range test with an early-out does not).
__device__ __forceinline__ uint32_t visible_mask(int c0, int lo, int hi)
{
    const int a = min(max(lo - c0, 0), 32), b = min(max(hi - c0 + 1, 0), 32);
    const uint32_t below_b = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
    const uint32_t below_a = a >= 32 ? 0xffffffffu : ((1u << a) - 1u);
    return below_b & ~below_a;
}

// Three-input maximum (one instruction); exact, so any grouping gives the same value.
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Max over the 32 values of x: four interleaved partial maxima of eight values each.
__device__ __forceinline__ float max32(const float (&x)[32])
{
    float m4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float a = max3(x[k], x[k + 4], x[k + 8]);
        const float b = max3(a, x[k + 12], x[k + 16]);
        const float d = max3(b, x[k + 20], x[k + 24]);
        m4[k] = fmaxf(d, x[k + 28]);
    }
    return fmaxf(max3(m4[0], m4[1], m4[2]), m4[3]);
}

// Max over the visible columns (bit j of `mask` for column j) of a quarter held in sv.
// Called by whole warps: the branch between the all-visible path and the per-column selects
// is taken for the whole warp at once (the selects give the same value when every bit is set).
__device__ __forceinline__ float quarter_max(const uint32_t* sv, uint32_t mask)
{
    if (__all_sync(0xffffffffu, mask == 0u))
        return -INFINITY;
    float x[32];
    if (__all_sync(0xffffffffu, mask == 0xffffffffu)) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            x[j] = __uint_as_float(sv[j]);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            x[j] = (mask >> j) & 1u ? __uint_as_float(sv[j]) : -INFINITY;
    }
    return max32(x);
}

// Max over a quarter whose 32 columns are all visible for the whole warp.
__device__ __forceinline__ float quarter_max_all(const uint32_t* sv)
{
    float x[32];
#pragma unroll
    for (int j = 0; j < 32; ++j)
        x[j] = __uint_as_float(sv[j]);
    return max32(x);
}

// Probabilities of a quarter (32 columns, neg = -m_t) as bf16 pairs handed to
// `sink(qd, w0, w1, w2, w3)` eight columns at a time: w_i holds columns 8 qd + 2i (low half)
// and 8 qd + 2i + 1; returns the quarter sum. Columns are taken in ascending order. With
// kSel, a column whose bit in `mask` is clear is 0; without, every column is visible.
template <bool kSel, class Sink>
__device__ __forceinline__ float quarter_exp_core(const uint32_t* sv, uint32_t mask, float scale_log2, float neg,
                                                  Sink&& sink)
{
    // Paired fp32 operations (__ffma2_rn, __fadd2_rn) round each lane exactly as the scalar
    // operation does; l01 and l23 hold the partial sums (l0, l1) and (l2, l3).
    float2 l01 = make_float2(0.f, 0.f), l23 = make_float2(0.f, 0.f);
    const float2 sc2 = make_float2(scale_log2, scale_log2), ng2 = make_float2(neg, neg);
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
        float pv[8];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const int j = 8 * qd + e;
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])), sc2, ng2);
            pv[e] = ex2(x.x);
            pv[e + 1] = ex2(x.y);
            if (kSel) {
                pv[e] = (mask >> j) & 1u ? pv[e] : 0.f;
                pv[e + 1] = (mask >> (j + 1)) & 1u ? pv[e + 1] : 0.f;
            }
        }
        l01 = __fadd2_rn(l01, make_float2(pv[0], pv[1]));
        l23 = __fadd2_rn(l23, make_float2(pv[2], pv[3]));
        l01 = __fadd2_rn(l01, make_float2(pv[4], pv[5]));
        l23 = __fadd2_rn(l23, make_float2(pv[6], pv[7]));
        sink(qd, pack_bf16(pv[0], pv[1]), pack_bf16(pv[2], pv[3]), pack_bf16(pv[4], pv[5]), pack_bf16(pv[6], pv[7]));
    }
    return __fadd_rn(__fadd_rn(l01.x, l01.y), __fadd_rn(l23.x, l23.y));
}

// The same with the visible columns in `mask` (bit j for column j; a hidden column is 0).
// Called by whole warps: the branches between nothing visible, everything visible and the
// per-column selects are taken warp by warp (the selects give the same values when every
// bit is set).
template <class Sink>
__device__ __forceinline__ float quarter_exp_to(const uint32_t* sv, uint32_t mask, float scale_log2, float neg,
                                                Sink&& sink)
{
    if (__all_sync(0xffffffffu, mask == 0u)) {  // nothing visible: P = 0 and the sum is 0
#pragma unroll
        for (int qd = 0; qd < 4; ++qd)
            sink(qd, 0u, 0u, 0u, 0u);
        return 0.f;
    }
    if (__all_sync(0xffffffffu, mask == 0xffffffffu))
        return quarter_exp_core<false>(sv, mask, scale_log2, neg, sink);
    return quarter_exp_core<true>(sv, mask, scale_log2, neg, sink);
}

// Merge of a tile-local softmax state (mt, lt, ot) into a running state (m, l, o):
//   mn = max(m, mt), a = 2^(m - mn), b = 2^(mt - mn), l <- l a + lt b, o <- o a + ot b.
struct FoldCoef {
    float a, b, mn;
};

__device__ __forceinline__ FoldCoef fold_coef(float m, float mt)
{
    const float mn = fmaxf(m, mt);
    return FoldCoef{ex2(__fsub_rn(m, mn)), ex2(__fsub_rn(mt, mn)), mn};
}

// o <- o a + ot b for N dims (the same element-wise operations for any split of the dims).
template <int N>
__device__ __forceinline__ void fold_apply(float* o, const float* ot, const FoldCoef& f)
{
    static_assert(N % 2 == 0, "dims in pairs");
    const float2 a2 = make_float2(f.a, f.a), b2 = make_float2(f.b, f.b);
#pragma unroll
    for (int d = 0; d < N; d += 2) {
        const float2 r = __ffma2_rn(make_float2(o[d], o[d + 1]), a2, __fmul2_rn(make_float2(ot[d], ot[d + 1]), b2));
        o[d] = r.x;
        o[d + 1] = r.y;
    }
}

__device__ __forceinline__ void fold_finish(float& m, float& l, float lt, const FoldCoef& f)
{
    l = __fmaf_rn(l, f.a, __fmul_rn(lt, f.b));
    m = f.mn;
}

template <int N>
__device__ __forceinline__ void fold_tile(float& m, float& l, float* o, float mt, float lt, const float* ot)
{
    const FoldCoef f = fold_coef(m, mt);
    fold_apply<N>(o, ot, f);
    fold_finish(m, l, lt, f);
}

// fold_tile when `seen`, else no change; branch-free (the skipped fold's values, which may
// be NaN when both maxima are -inf, are computed and discarded by a select).
template <int N>
__device__ __forceinline__ void fold_tile_if(bool seen, float& m, float& l, float* o, float mt, float lt,
                                             const float* ot)
{
    const FoldCoef f = fold_coef(m, mt);
#pragma unroll
    for (int d = 0; d < N; ++d) {
        const float on = __fmaf_rn(o[d], f.a, __fmul_rn(ot[d], f.b));
        o[d] = seen ? on : o[d];
    }
    const float ln = __fmaf_rn(l, f.a, __fmul_rn(lt, f.b));
    l = seen ? ln : l;
    m = seen ? f.mn : m;
}

// NEOX rotation of pairs [8q, 8q+8) of a 64-value head row: a holds elements [8q, 8q+8),
// b elements [32+8q, 32+8q+8) (bf16), cs the row's 32 (cos, sin) pairs; ya, yb the results.
__device__ __forceinline__ void rotate_chunks(const uint4 a, const uint4 b, const float2* cs, int q, uint4& ya,
                                              uint4& yb)
{
    const float4* cs4 = reinterpret_cast<const float4*>(cs + 8 * q);  // 8 (cos, sin) pairs, 16-B aligned
    const float4 c01 = cs4[0], c23 = cs4[1], c45 = cs4[2], c67 = cs4[3];
    const float2 cw[8] = {{c01.x, c01.y}, {c01.z, c01.w}, {c23.x, c23.y}, {c23.z, c23.w},
                          {c45.x, c45.y}, {c45.z, c45.w}, {c67.x, c67.y}, {c67.z, c67.w}};
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
    uint32_t ra[4], rb[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float y1a, y2a, y1b, y2b;
        rope_pair(bf16lo(aw[w]), bf16lo(bw[w]), cw[2 * w], y1a, y2a);
        rope_pair(bf16hi(aw[w]), bf16hi(bw[w]), cw[2 * w + 1], y1b, y2b);
        ra[w] = pack_bf16(y1a, y1b);
        rb[w] = pack_bf16(y2a, y2b);
    }
    ya = make_uint4(ra[0], ra[1], ra[2], ra[3]);
    yb = make_uint4(rb[0], rb[1], rb[2], rb[3]);
}

// Rotate pairs [8q, 8q+8) of a 64-value head row (NEOX: element i pairs with i + 32) at the
// angle table row cs, and write them as chunks q and 4 + q of a swizzled 128-byte row.
__device__ __forceinline__ void rotate_quarter(const __nv_bfloat16* src, const float2* cs, uint8_t* tile, int row,
                                               int q)
{
    const uint4 a = *reinterpret_cast<const uint4*>(src + 8 * q);
    const uint4 b = *reinterpret_cast<const uint4*>(src + 32 + 8 * q);
    uint4 ya, yb;
    rotate_chunks(a, b, cs, q, ya, yb);
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, q)) = ya;
    *reinterpret_cast<uint4*>(tile + sw128_offset(row, 4 + q)) = yb;
}

// The same rotation in place, for a row already in the swizzled tile (landed there by TMA).
__device__ __forceinline__ void rotate_quarter_in_place(uint8_t* tile, const float2* cs, int row, int q)
{
    uint4* pa = reinterpret_cast<uint4*>(tile + sw128_offset(row, q));
    uint4* pb = reinterpret_cast<uint4*>(tile + sw128_offset(row, 4 + q));
    uint4 ya, yb;
    rotate_chunks(*pa, *pb, cs, q, ya, yb);
    *pa = ya;
    *pb = yb;
}

// Store N consecutive output dims starting at dim d0 of an output row: o * (1 / l) as bf16
// (one correctly rounded reciprocal per row, then a multiply per dim).
template <int N>
__device__ __forceinline__ void store_out(__nv_bfloat16* orow, const float* o, float l, int d0)
{
    const float inv = __frcp_rn(l);
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int c = 0; c < N / 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 y = __fmul2_rn(make_float2(o[8 * c + 2 * e], o[8 * c + 2 * e + 1]), inv2);
            w[e] = pack_bf16(y.x, y.y);
        }
        *reinterpret_cast<uint4*>(orow + d0 + 8 * c) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace enc
}  // namespace vst
