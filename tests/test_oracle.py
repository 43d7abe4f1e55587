"""Pins for the fp64 oracle (CPU only).

The oracle is trusted only because these tests tie it to things other than itself:
IEEE bit patterns, closed forms, a library routine (torch scaled-dot-product attention),
an independent complex-number formulation of the rotation, brute force on tiny inputs, the
invariants the pages state (chunking is not observable, frame i depends on [i-749, i]
alone, a clip shorter than the window equals plain causal attention), and ring schedules
derived by hand from the pages' rules. ``test_mutants_are_caught`` plants plausible
mistakes in a copy of the oracle and checks that each one fails at least one pin.
"""
import ctypes
import math
import os
import random
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from sliding_window_kv_gb300 import synth

THETA = 1.0e6


def _bits(t):
    return synth.bits(t)


def _randn_bits(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return _bits(torch.randn(*shape, generator=g).to(torch.bfloat16))


def _rope_complex(x, pos, theta=THETA):
    """Independent formulation: pair (x_i, x_{i+D/2}) as the complex number x_i + i x_{i+D/2}
    and multiply by exp(i * pos * theta^(-2i/D))."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    freq = theta ** (-2.0 * np.arange(half) / D)
    pos = np.asarray(pos, dtype=np.float64)
    ang = pos.reshape(pos.shape + (1,) * (x.ndim - 1 - pos.ndim) + (1,)) * freq
    z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * ang)
    return np.concatenate([z.real, z.imag], axis=-1)


def _bruteforce(qb, kb, vb, W, pos0=0):
    """Full T x T score matrix with an explicit -inf mask and softmax by definition."""
    q = oracle.bf16_to_double(qb)
    k = oracle.bf16_to_double(kb)
    v = oracle.bf16_to_double(vb)
    T, H, D = q.shape
    Hk = k.shape[1]
    pos = np.arange(T) + pos0
    qr = _rope_complex(q, pos[:, None])
    kr = _rope_complex(k, pos[:, None])
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    allowed = (i - j >= 0) & (i - j < W)
    out = np.zeros((T, H, D))
    for h in range(H):
        g = h // (H // Hk)
        S = qr[:, h] @ kr[:, g].T / math.sqrt(D)
        S = np.where(allowed, S, -np.inf)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        out[:, h] = P @ v[:, g]
    return out


# ---------------------------------------------------------------- bf16 widening (IEEE)

def check_bf16():
    cases = {0x0000: 0.0, 0x3F80: 1.0, 0xC000: -2.0, 0x3F00: 0.5, 0x4049: 3.140625,
             0x0001: 2.0 ** -133, 0x7F7F: 3.3895313892515355e38, 0x8000: -0.0}
    bits = np.array(list(cases), dtype=np.uint16)
    got = oracle.bf16_to_double(bits)
    for b, g in zip(bits, got):
        assert g == cases[int(b)], (hex(b), g)


def test_bf16_widening():
    check_bf16()


# ---------------------------------------------------------------- RoPE

def check_rope_identity_at_zero():
    x = np.random.default_rng(0).standard_normal(64)
    assert np.array_equal(oracle.rope(x, 0), x)


def check_rope_neox_pairs():
    """NEOX rotates the pairs (i, i + D/2): each pair keeps its norm. The GPT-J interleaved
    pairing (2i, 2i+1) would not preserve these pair norms."""
    rng = np.random.default_rng(1)
    for D in (8, 64, 128):
        x = rng.standard_normal(D)
        y = oracle.rope(x, 977)
        h = D // 2
        assert np.allclose(x[:h] ** 2 + x[h:] ** 2, y[:h] ** 2 + y[h:] ** 2, rtol=1e-13, atol=0)


def check_rope_unit_vectors():
    """e_0 turns by exactly p radians (f_0 = theta^0 = 1) towards +e_{D/2}; e_1 of an
    8-dim head turns into e_5 (NEOX), never into e_0 (GPT-J would pair 0 and 1)."""
    D = 64
    e0 = np.zeros(D)
    e0[0] = 1.0
    y = oracle.rope(e0, 1)
    assert y[0] == pytest.approx(math.cos(1.0), abs=1e-15)
    assert y[32] == pytest.approx(math.sin(1.0), abs=1e-15)
    assert np.count_nonzero(y) == 2
    e1 = np.zeros(8)
    e1[1] = 1.0
    y = oracle.rope(e1, 1)
    f1 = THETA ** (-2.0 / 8)
    assert y[0] == 0.0 and y[1] == pytest.approx(math.cos(f1), abs=1e-15)
    assert y[5] == pytest.approx(math.sin(f1), abs=1e-15)


def check_rope_frequencies():
    """The angle of pair i at position p is p * theta^(-2i/D): consecutive pairs differ by
    the constant ratio theta^(-2/D), and the slowest pair runs at theta^(-(D-2)/D)."""
    for D in (64, 128):
        p = 3
        angles = []
        for i in range(D // 2):
            e = np.zeros(D)
            e[i] = 1.0
            y = oracle.rope(e, p)
            angles.append(math.atan2(y[i + D // 2], y[i]))
        angles = np.array(angles)
        assert angles[0] == pytest.approx(3.0 - 2 * math.pi * 0, abs=1e-12)
        with np.errstate(divide="ignore", invalid="ignore"):  # a wrong pairing gives zero angles
            ratios = angles[2:] / angles[1:-1]
        assert np.allclose(ratios, THETA ** (-2.0 / D), rtol=1e-9)
        assert angles[-1] == pytest.approx(p * THETA ** (-(D - 2.0) / D), rel=1e-12)


def check_rope_group():
    """Rotations compose and invert; the score depends on positions only through m - n."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal(128)
    k = rng.standard_normal(128)
    a, b = 1234, 5678
    assert np.allclose(oracle.rope(oracle.rope(x, a), b), oracle.rope(x, a + b), atol=1e-11)
    assert np.allclose(oracle.rope(oracle.rope(x, a), -a), x, atol=1e-12)
    s1 = oracle.rope(x, 700) @ oracle.rope(k, 650)
    s2 = oracle.rope(x, 100700) @ oracle.rope(k, 100650)
    assert s1 == pytest.approx(s2, abs=1e-9)


def check_rope_rows_matches_complex_form():
    xb = _randn_bits((9, 3, 64), 3)
    got = oracle.rope_rows(xb, pos0=4000)
    want = _rope_complex(oracle.bf16_to_double(xb), (np.arange(9) + 4000)[:, None])
    assert np.allclose(got, want, atol=1e-12)


@pytest.mark.parametrize("check", [check_rope_identity_at_zero, check_rope_neox_pairs,
                                   check_rope_unit_vectors, check_rope_frequencies,
                                   check_rope_group, check_rope_rows_matches_complex_form])
def test_rope(check):
    check()


# ---------------------------------------------------------------- attention

def check_bruteforce_tiny():
    for (T, H, Hk, D, W, pos0, seed) in [(12, 2, 1, 4, 3, 0, 10), (16, 4, 2, 64, 5, 0, 11),
                                         (16, 2, 2, 4, 1, 7, 12), (9, 4, 1, 8, 16, 100, 13)]:
        qb = _randn_bits((T, H, D), seed)
        kb = _randn_bits((T, Hk, D), seed + 100)
        vb = _randn_bits((T, Hk, D), seed + 200)
        got = oracle.attention(qb, kb, vb, W, pos0=pos0)
        want = _bruteforce(qb, kb, vb, W, pos0=pos0)
        assert np.allclose(got, want, atol=1e-12, rtol=0), (T, H, Hk, D, W)


def check_long_window_is_causal_sdpa():
    """W >= T: windowed attention is plain causal attention (torch's SDPA, scale 1/sqrt(D))."""
    T, H, D = 40, 2, 16
    qb, kb, vb = (_randn_bits((T, H, D), s) for s in (20, 21, 22))
    got = oracle.attention(qb, kb, vb, window=T + 5)
    pos = np.arange(T)[:, None]
    qr = torch.from_numpy(_rope_complex(oracle.bf16_to_double(qb), pos)).permute(1, 0, 2)
    kr = torch.from_numpy(_rope_complex(oracle.bf16_to_double(kb), pos)).permute(1, 0, 2)
    vv = torch.from_numpy(oracle.bf16_to_double(vb)).permute(1, 0, 2)
    want = torch.nn.functional.scaled_dot_product_attention(qr, kr, vv, is_causal=True)
    assert np.allclose(got, want.permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)


def check_jfk_clip_no_trim(page_constants):
    """A 748-frame clip under the 750 window never trims: windowed == unwindowed."""
    T = page_constants["jfk_frames"]
    W = page_constants["enc_window"]
    qb, kb, vb = (_randn_bits((T, 1, 64), s) for s in (30, 31, 32))
    a = oracle.attention(qb, kb, vb, window=W)
    b = oracle.attention(qb, kb, vb, window=10 ** 9)
    assert np.array_equal(a, b)


def check_window_one_returns_v():
    T, H, D = 20, 4, 8
    qb, kb, vb = (_randn_bits((T, H, D), s) for s in (40, 41, 42))
    out = oracle.attention(qb, kb, vb, window=1)
    assert np.array_equal(out, oracle.bf16_to_double(vb))


def check_zero_query_gives_window_mean():
    """q = 0 makes every score 0, so row i is the plain mean of v over [max(0,i-W+1), i]:
    the count min(W, i+1) pins both window edges."""
    T, H, D = 1000, 2, 4
    vb = _randn_bits((T, H, D), 50)
    kb = _randn_bits((T, H, D), 51)
    qb = np.zeros((T, H, D), dtype=np.uint16)
    v = oracle.bf16_to_double(vb)
    for W in (1, 3, 750):
        out = oracle.attention(qb, kb, vb, window=W)
        for i in (0, 1, 2, 5, W - 2, W - 1, W, W + 1, 999):
            if i < 0 or i >= T:
                continue
            j0 = max(0, i - W + 1)
            assert np.allclose(out[i], v[j0:i + 1].mean(axis=0), atol=1e-13), (W, i)


def check_decoder_window_8192():
    """Decoder step cur sees [cur-8191, cur]: with q = 0 the row is the mean over that span."""
    T, D = 8200, 4
    vb = _randn_bits((T, 1, D), 60)
    kb = _randn_bits((T, 1, D), 61)
    q = np.zeros((T, 4, D), dtype=np.uint16)
    v = oracle.bf16_to_double(vb)
    qr = oracle.rope_rows(q)
    kr = oracle.rope_rows(kb)
    out = oracle.attend(qr, kr, v, window=8192, rows=(8189, 8200))
    for i in range(8189, 8200):
        j0 = max(0, i - 8191)
        for h in range(4):
            assert np.allclose(out[i - 8189, h], v[j0:i + 1, 0].mean(axis=0), atol=1e-13), i


def check_gqa_groups():
    """32 query heads over 8 KV heads: head h reads KV head h // 4."""
    T, H, Hk, D = 6, 32, 8, 4
    v = np.zeros((T, Hk, D), dtype=np.float32)
    for g in range(Hk):
        v[:, g, :] = g + 1
    vb = _bits(torch.from_numpy(v).to(torch.bfloat16))
    kb = _randn_bits((T, Hk, D), 70)
    qb = _randn_bits((T, H, D), 71)
    out = oracle.attention(qb, kb, vb, window=4)
    for h in range(H):
        assert np.allclose(out[:, h, :], h // 4 + 1, atol=1e-12), h


def check_position_shift_invariance():
    """Scores depend on i - j only, so moving every position by a constant leaves the output
    unchanged: this pins that queries and keys are keyed on the same absolute positions."""
    T, H, D = 64, 2, 64
    qb, kb, vb = (_randn_bits((T, H, D), s) for s in (80, 81, 82))
    a = oracle.attention(qb, kb, vb, window=20, pos0=0)
    b = oracle.attention(qb, kb, vb, window=20, pos0=12345)
    assert np.allclose(a, b, atol=1e-9)
    assert not np.allclose(oracle.rope_rows(qb, 0), oracle.rope_rows(qb, 12345))


def check_window_locality():
    """Frame i depends on frames [i-W+1, i] alone (the bounded-window re-encode argument):
    a row computed from that slice equals the whole-clip row, bit for bit."""
    T, H, D, W = 300, 2, 64, 50
    qb, kb, vb = (_randn_bits((T, H, D), s) for s in (90, 91, 92))
    full = oracle.attention(qb, kb, vb, window=W)
    for i in (0, 10, 49, 50, 51, 200, 299):
        j0 = max(0, i - W + 1)
        row = oracle.attention_row(qb[i], kb[j0:i + 1], vb[j0:i + 1], i, W)
        assert np.array_equal(row, full[i]), i


def check_chunking_not_observable():
    """Feeding in chunks equals one call: each chunk is computed from the prefix alone."""
    T, H, D, W = 400, 2, 64, 64
    qb, kb, vb = (_randn_bits((T, H, D), s) for s in (100, 101, 102))
    whole = oracle.attention(qb, kb, vb, window=W)
    rng = random.Random(5)
    for _ in range(3):
        out = []
        t = 0
        while t < T:
            n = min(T - t, rng.choice([1, 7, 50, 100, 512]))
            e = t + n
            out.append(oracle.attention(qb[:e], kb[:e], vb[:e], window=W, rows=(t, e)))
            t = e
        assert np.array_equal(np.concatenate(out), whole)


# ---- (left, right) mask: "Moonshine streaming forward map", Encoder table, per-layer
# sliding-window mask row: mask[q, k] = 0 iff (q - k in [0, L)) or (k - q in (0, R)).

def _bruteforce_lr(qb, kb, vb, L, R, pos0=0):
    """Full T x T score matrix with the pages' (L, R) mask written out, softmax by definition."""
    q = oracle.bf16_to_double(qb)
    k = oracle.bf16_to_double(kb)
    v = oracle.bf16_to_double(vb)
    T, H, D = q.shape
    Hk = k.shape[1]
    pos = np.arange(T) + pos0
    qr = _rope_complex(q, pos[:, None])
    kr = _rope_complex(k, pos[:, None])
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    allowed = ((i - j >= 0) & (i - j < L)) | ((j - i > 0) & (j - i < R))
    out = np.zeros((T, H, D))
    for h in range(H):
        g = h // (H // Hk)
        S = qr[:, h] @ kr[:, g].T / math.sqrt(D)
        S = np.where(allowed, S, -np.inf)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        out[:, h] = P @ v[:, g]
    return out


def check_lr_bruteforce_tiny():
    for (T, H, Hk, D, L, R, pos0) in [(9, 2, 2, 8, 3, 2, 0), (12, 4, 2, 8, 16, 4, 5), (11, 2, 1, 16, 1, 3, 0),
                                      (10, 2, 2, 8, 4, 0, 7), (7, 2, 2, 8, 2, 9, 0)]:
        qb, kb, vb = (_randn_bits(s, seed) for s, seed in (((T, H, D), 110), ((T, Hk, D), 111), ((T, Hk, D), 112)))
        got = oracle.attention_lr(qb, kb, vb, L, R, pos0=pos0)
        want = _bruteforce_lr(qb, kb, vb, L, R, pos0=pos0)
        assert np.allclose(got, want, atol=1e-12, rtol=0), (T, L, R)


def check_lr_bidirectional_is_sdpa():
    """L and R past the clip: every row sees the whole clip, which is torch's unmasked SDPA."""
    T, H, D = 30, 2, 16
    qb, kb, vb = (_randn_bits((T, H, D), s) for s in (120, 121, 122))
    got = oracle.attention_lr(qb, kb, vb, T + 3, T + 3)
    pos = np.arange(T)[:, None]
    qr = torch.from_numpy(_rope_complex(oracle.bf16_to_double(qb), pos)).permute(1, 0, 2)
    kr = torch.from_numpy(_rope_complex(oracle.bf16_to_double(kb), pos)).permute(1, 0, 2)
    vv = torch.from_numpy(oracle.bf16_to_double(vb)).permute(1, 0, 2)
    want = torch.nn.functional.scaled_dot_product_attention(qr, kr, vv)
    assert np.allclose(got, want.permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)


def check_lr_zero_query_span_mean():
    """q = 0: row i is the plain mean of v over [max(0, i-L+1), min(T-1, i+R-1)], which pins
    both edges of the span (R = 0 and R = 1 both mean no lookahead)."""
    T, H, D = 60, 2, 4
    vb = _randn_bits((T, H, D), 130)
    kb = _randn_bits((T, H, D), 131)
    qb = np.zeros((T, H, D), dtype=np.uint16)
    v = oracle.bf16_to_double(vb)
    for L, R in ((16, 4), (16, 0), (16, 1), (1, 1), (5, 7)):
        out = oracle.attention_lr(qb, kb, vb, L, R)
        for i in (0, 1, 3, 15, 16, 30, 56, 57, 58, 59):
            j0, j1 = max(0, i - L + 1), min(T - 1, i + max(R - 1, 0))
            assert np.allclose(out[i], v[j0:j1 + 1].mean(axis=0), atol=1e-13), (L, R, i)


def check_lr_causal_case_is_windowed_attention():
    """R = 0 is the windowed-causal mask with W = L: the same bits as `attention`."""
    T, H, D = 80, 2, 64
    qb, kb, vb = (_randn_bits((T, H, D), s) for s in (140, 141, 142))
    for L in (1, 7, 80, 200):
        assert np.array_equal(oracle.attention_lr(qb, kb, vb, L, 0), oracle.attention(qb, kb, vb, window=L))


def check_lr_window_locality():
    """A row computed from its own span alone, [i - L + 1, i + R - 1] cut out of the clip and
    placed at its absolute positions, equals the whole-clip row bit for bit (the offline
    parity tests sample rows this way)."""
    T, H, D = 200, 2, 16
    qb, kb, vb = (_randn_bits((T, H, D), s) for s in (150, 151, 152))
    for L, R in ((16, 4), (150, 4), (1, 1), (40, 0)):
        whole = oracle.attention_lr(qb, kb, vb, L, R)
        for i in (0, 1, 15, 16, 100, 149, 150, 196, 199):
            a0, a1 = max(0, i - L + 1), min(T, i + max(R, 1))
            row = oracle.attention_lr(qb[a0:a1], kb[a0:a1], vb[a0:a1], L, R, pos0=a0, rows=(i - a0, i - a0 + 1))[0]
            assert np.array_equal(row, whole[i]), (L, R, i)


ATTENTION_CHECKS = [check_bruteforce_tiny, check_long_window_is_causal_sdpa,
                    check_window_one_returns_v, check_zero_query_gives_window_mean,
                    check_decoder_window_8192, check_gqa_groups, check_position_shift_invariance,
                    check_window_locality, check_chunking_not_observable, check_lr_bruteforce_tiny,
                    check_lr_bidirectional_is_sdpa, check_lr_zero_query_span_mean,
                    check_lr_causal_case_is_windowed_attention, check_lr_window_locality]


@pytest.mark.parametrize("check", ATTENTION_CHECKS)
def test_attention(check):
    check()


def test_jfk_clip_no_trim(page_constants):
    check_jfk_clip_no_trim(page_constants)


# ---------------------------------------------------------------- ring bookkeeping

def check_ring_schedules():
    # 10 feeds of 100: 1000 <= 1536 frames, so the ring never compacts.
    st = oracle.RingState()
    for _ in range(10):
        st.feed(100)
    assert (st.n_kv, st.abs_base, st.n_compactions) == (1000, 0, 0)
    # 88 feeds of 50 then 16 (the whole-earth length 4416): the ring reaches 1500 after
    # feed 30, feed 31 would make 1550 > 1536, so it keeps 750 and appends (800); every 15
    # feeds after that it is full again: compactions before feeds 31, 46, 61, 76.
    st = oracle.RingState()
    seen = []
    for f in range(1, 90):
        before = st.n_compactions
        st.feed(50 if f <= 88 else 16)
        if st.n_compactions != before:
            seen.append(f)
    assert seen == [31, 46, 61, 76]
    assert (st.n_kv, st.abs_base, st.abs_next) == (1416, 3000, 4416)
    # One feed of 2000 goes in as 512, 512, 512, 464: the ring fills to exactly 1536, then
    # the last batch needs room: keep 750 (abs_base 786) and append 464.
    st = oracle.RingState().feed(2000)
    assert (st.n_kv, st.abs_base, st.n_compactions) == (1214, 786, 1)


def check_ring_dots_full(page_constants):
    """~15300 frames fed in 24..48-frame pieces compact about 20 times."""
    rng = random.Random(7)
    st = oracle.RingState()
    total = 0
    while total < page_constants["dots_full_frames"]:
        n = rng.randint(24, 48)
        st.feed(n)
        total += n
        assert st.abs_next == st.abs_base + st.n_kv == total
        assert st.n_kv <= page_constants["enc_ring_slots"]
    assert 15 <= st.n_compactions <= 25


def check_ring_keeps_window():
    """After any feed the ring still holds the 749 frames before the newest one."""
    rng = random.Random(8)
    st = oracle.RingState()
    for _ in range(400):
        st.feed(rng.choice([1, 3, 50, 100, 511, 512, 513, 1500]))
        assert st.abs_base <= max(0, st.abs_next - 750)


def test_ring_schedules():
    check_ring_schedules()
    check_ring_keeps_window()


def test_ring_dots_full(page_constants):
    check_ring_dots_full(page_constants)


def test_page_constants_fixture(page_constants):
    c = page_constants
    assert c["enc_d_model"] // c["enc_head_dim"] == c["enc_heads"] == 20
    assert c["dec_q_heads"] % c["dec_kv_heads"] == 0
    assert c["enc_keep"] == c["enc_window"]
    assert c["enc_keep"] + c["enc_max_batch"] <= c["enc_ring_slots"]
    assert c["dec_window"] - 1 == c["dec_first_visible_offset"]
    assert c["dec_evicted_offset"] == c["dec_window"]


# ---------------------------------------------------------------- planted mistakes

MUTANTS = {
    "rope_sign": ("y[i] = x1 * c - x2 * s;", "y[i] = x1 * c + x2 * s;"),
    "rope_pairing": ("double x1 = x[i], x2 = x[i + half];",
                     "double x1 = x[2 * i], x2 = x[2 * i + 1];"),
    "rope_freq": ("pow(theta, -2.0 * (double)i / (double)D)", "pow(theta, -1.0 * (double)i / (double)D)"),
    "window_off_by_one": ("long long j0 = i - W + 1;", "long long j0 = i - W;"),
    "scale": ("double scale = 1.0 / sqrt((double)D);", "double scale = 1.0 / (double)D;"),
    "gqa_interleaved": ("int g = h / group;", "int g = h % Hk;"),
    "value_row": ("const double* vj = v + (j * Hk + g) * (long long)D;",
                  "const double* vj = v + (i * Hk + g) * (long long)D;"),
    "ring_trigger": ("if (st->n_kv + b > ring_slots) {", "if (st->n_kv + b >= ring_slots) {"),
    "ring_keep": ("st->abs_base += st->n_kv - kept;", "st->abs_base += st->n_kv - kept + 1;"),
    "bf16_shift": ("((uint32_t)b) << 16;", "((uint32_t)b) << 15;"),
    "lr_right_edge": ("long long hi = R > 0 ? i + R - 1 : i;", "long long hi = R > 0 ? i + R : i;"),
    "lr_left_edge": ("long long lo = i - L + 1;", "long long lo = i - L;"),
    "lr_clip_end": ("            hi = T - 1;", "            hi = T - 2;"),
}


def _all_pins(consts):
    checks = ([check_bf16, check_rope_identity_at_zero, check_rope_neox_pairs,
               check_rope_unit_vectors, check_rope_frequencies, check_rope_group,
               check_rope_rows_matches_complex_form, check_ring_schedules, check_ring_keeps_window,
               lambda: check_ring_dots_full(consts)] + ATTENTION_CHECKS)
    failed = 0
    for c in checks:
        try:
            c()
        except AssertionError:
            failed += 1
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(name, page_constants):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, "mutation site missing: %s" % old
    d = tempfile.mkdtemp()
    try:
        c = os.path.join(d, "m.c")
        so = os.path.join(d, "m.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o", so, c, "-lm"])
        saved = oracle._load()
        oracle._lib = oracle._bind(ctypes.CDLL(so))
        try:
            assert _all_pins(page_constants) > 0, "mutant %s passed every pin" % name
        finally:
            oracle._lib = saved
    finally:
        shutil.rmtree(d)


def test_unmutated_oracle_passes_every_pin(page_constants):
    assert _all_pins(page_constants) == 0
