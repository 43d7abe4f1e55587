/*
 * vst_oracle.c -- fp64 CPU oracle for incremental sliding-window KV attention.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the CPU-baseline
 * leg of the benchmark load or call this file. The product path (the CUDA library under
 * sliding_window_kv_gb300/) never does, and the two share no code, headers or tables.
 *
 * What it computes. The streaming method is a throughput device whose numerics equal the
 * offline whole-clip computation ("Voxtral Realtime -- incremental streaming
 * implementation plan", section "Why offline == streaming" and verification item 1). So
 * this oracle is the plain offline definition, in double precision, with an explicit
 * window mask, no ring, no chunking and no online softmax:
 *
 *   out[i][h] = sum_j softmax_j( RoPE(q[i][h], i) . RoPE(k[j][g], j) / sqrt(D) ) v[j][g]
 *               over absolute positions j with 0 <= i - j < W,  g = h / (H / Hk).
 *
 *   - Window W keys including self: frame i attends [i-749, i] for the encoder
 *     (streaming plan, "RECOMMENDED implementation" bullets), and decoder step `cur`
 *     reveals [cur-8191, cur] ("Voxtral Realtime" family doc, Capability Validation table,
 *     Streaming row, item (5)). The moonshine forward map states the same rule as
 *     mask = 0 iff q-k in [0, L) (Encoder table, per-layer sliding-window mask).
 *   - NEOX (rotate-half) RoPE with theta = 1e6 at absolute positions (family doc,
 *     "Architecture (summary)", Encoder and Decoder bullets; streaming plan, "Chunk
 *     alignment": "RoPE at absolute positions"). NEOX pairs element i with i + D/2; the
 *     moonshine forward map contrasts it with the GPT-J interleaved pairing (2i, 2i+1).
 *   - Frequencies f_i = theta^(-2i/D), i in [0, D/2): the standard rotary definition; the
 *     pages name the variant and theta but do not print the formula.
 *   - Softmax scale 1/sqrt(D): not stated on the pages; the plainest reading (standard
 *     scaled dot-product attention).
 *   - GQA: query head h reads KV head h / (H/Hk) (contiguous groups). The family doc gives
 *     only "GQA 32q/8kv"; contiguous grouping is the plainest reading.
 *
 * The encoder ring bookkeeping (vst_oracle_ring_feed) restates the pages' ring rules:
 * contiguous appends at rows [n_kv_before, n_kv_total), feeds pushed in batches of at most
 * 512, and compaction that copies the last 750 frames to the front (streaming plan,
 * "Unbounded length (shipped)"). When to compact is not fixed by the pages; the reading
 * taken is "just before a batch that would not fit", which gives the ~20 compactions the
 * family doc reports for ~15300 frames fed in small chunks (Streaming row, item (4)).
 *
 * Every function is pinned by tests/test_oracle.py against closed forms, textbook routines,
 * brute force and the pages' invariants.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* bf16 is the upper half of an IEEE binary32: widen the bit pattern, then convert. */
double vst_oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Widen n bf16 values to double. */
void vst_oracle_bf16_to_double_n(const uint16_t* x, long long n, double* y)
{
    for (long long i = 0; i < n; ++i)
        y[i] = vst_oracle_bf16_to_double(x[i]);
}

/* NEOX rotary embedding of one head vector x[D] at absolute position p:
 *   for i < D/2, a = p * theta^(-2i/D):
 *     y[i]       = x[i] cos a - x[i+D/2] sin a
 *     y[i+D/2]   = x[i+D/2] cos a + x[i] sin a
 * (y = x cos a + rotate_half(x) sin a, rotate_half(x) = (-x2, x1)). */
void vst_oracle_rope(const double* x, int D, double theta, long long p, double* y)
{
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double f = pow(theta, -2.0 * (double)i / (double)D);
        double a = (double)p * f;
        double c = cos(a), s = sin(a);
        double x1 = x[i], x2 = x[i + half];
        y[i] = x1 * c - x2 * s;
        y[i + half] = x2 * c + x1 * s;
    }
}

/* Rotate every head vector of a [n_rows][n_heads][D] bf16 tensor; row r sits at absolute
 * position pos0 + r. Output is double, same layout. */
void vst_oracle_rope_rows(const uint16_t* x, long long n_rows, int n_heads, int D,
                          double theta, long long pos0, double* y)
{
    double tmp[1024];
    for (long long r = 0; r < n_rows; ++r)
        for (int h = 0; h < n_heads; ++h) {
            const uint16_t* xv = x + (r * n_heads + h) * (long long)D;
            for (int d = 0; d < D; ++d)
                tmp[d] = vst_oracle_bf16_to_double(xv[d]);
            vst_oracle_rope(tmp, D, theta, pos0 + r, y + (r * n_heads + h) * (long long)D);
        }
}

/* One output row i (all H heads) over the keys j in [j0, j1] of a clip, offline definition:
 * out[h] = sum_j softmax_j(qr[i][h] . kr[j][g] / sqrt(D)) v[j][g], KV head g = h / (H / Hk),
 * the maximum score subtracted before exp. Layouts as vst_oracle_attend. */
static void attend_span(const double* qr, const double* kr, const double* v, int H, int Hk, int D,
                        long long i, long long j0, long long j1, double* out_row)
{
    int group = H / Hk;
    double scale = 1.0 / sqrt((double)D);
    for (int h = 0; h < H; ++h) {
        int g = h / group;
        const double* qi = qr + (i * H + h) * (long long)D;
        double* o = out_row + (long long)h * D;
        /* scores and their maximum */
        double m = -INFINITY;
        for (long long j = j0; j <= j1; ++j) {
            const double* kj = kr + (j * Hk + g) * (long long)D;
            double s = 0.0;
            for (int d = 0; d < D; ++d)
                s += qi[d] * kj[d];
            s *= scale;
            if (s > m)
                m = s;
        }
        /* softmax-weighted sum of values */
        double z = 0.0;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        for (long long j = j0; j <= j1; ++j) {
            const double* kj = kr + (j * Hk + g) * (long long)D;
            const double* vj = v + (j * Hk + g) * (long long)D;
            double s = 0.0;
            for (int d = 0; d < D; ++d)
                s += qi[d] * kj[d];
            double w = exp(s * scale - m);
            z += w;
            for (int d = 0; d < D; ++d)
                o[d] += w * vj[d];
        }
        for (int d = 0; d < D; ++d)
            o[d] /= z;
    }
}

/* Windowed-causal attention, offline definition, for rows i in [row_begin, row_end) of a
 * clip of T rows (row t = absolute position base + t; only differences matter here, RoPE
 * is already applied by the caller).
 *   qr  [T][H][D]   rotated queries (double)
 *   kr  [T][Hk][D]  rotated keys (double)
 *   v   [T][Hk][D]  values (double)
 *   out [row_end - row_begin][H][D]
 * Row i of head h attends keys j with 0 <= i - j < W, KV head g = h / (H / Hk). */
void vst_oracle_attend(const double* qr, const double* kr, const double* v, long long T,
                       int H, int Hk, int D, long long W, long long row_begin, long long row_end,
                       double* out)
{
    for (long long i = row_begin; i < row_end && i < T; ++i) {
        long long j0 = i - W + 1;
        if (j0 < 0)
            j0 = 0;
        attend_span(qr, kr, v, H, Hk, D, i, j0, i, out + (i - row_begin) * H * (long long)D);
    }
}

/* Sliding attention with a left window and a right lookahead, offline definition ("Moonshine
 * streaming forward map", Encoder table, per-layer sliding-window mask row): query i sees key
 * j of the same clip iff 0 <= i - j < L or 0 < j - i < R, for j in [0, T). So the visible
 * keys are [i - L + 1, i + R - 1], clipped to the clip; L = W, R = 0 is the windowed-causal
 * mask of vst_oracle_attend. Arguments as vst_oracle_attend. */
void vst_oracle_attend_lr(const double* qr, const double* kr, const double* v, long long T,
                          int H, int Hk, int D, long long L, long long R, long long row_begin,
                          long long row_end, double* out)
{
    for (long long i = row_begin; i < row_end && i < T; ++i) {
        long long lo = i - L + 1;
        long long hi = R > 0 ? i + R - 1 : i;
        if (lo < 0)
            lo = 0;
        if (hi > T - 1)
            hi = T - 1;
        attend_span(qr, kr, v, H, Hk, D, i, lo, hi, out + (i - row_begin) * H * (long long)D);
    }
}

/* Encoder ring bookkeeping as the pages state it. */
typedef struct {
    long long n_kv;          /* rows of the ring in use: slots [0, n_kv) */
    long long abs_base;      /* absolute frame index held by slot 0 */
    long long abs_next;      /* absolute index of the next frame to be fed */
    long long n_compactions; /* compactions performed so far */
} vst_oracle_ring_state;

/* Feed n_new frames: push them in batches of at most max_batch; before a batch that would
 * not fit in ring_slots, keep the last `keep` rows by moving them to the front. */
void vst_oracle_ring_feed(vst_oracle_ring_state* st, long long n_new, long long ring_slots,
                          long long keep, long long max_batch)
{
    while (n_new > 0) {
        long long b = n_new < max_batch ? n_new : max_batch;
        if (st->n_kv + b > ring_slots) {
            long long kept = st->n_kv < keep ? st->n_kv : keep;
            st->abs_base += st->n_kv - kept;
            st->n_kv = kept;
            st->n_compactions += 1;
        }
        st->n_kv += b;
        st->abs_next += b;
        n_new -= b;
    }
}
