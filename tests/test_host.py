"""CPU-only checks of the C ABI: the library loads without a GPU, exports exactly what
include/vst.h declares, the binding declares the same names, and the host logic (config
validation, the encoder feed schedule) behaves as the pages' rules say. No compute call."""
import ctypes
import os
import random
import re

import pytest

import oracle
from sliding_window_kv_gb300 import vst

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "vst.h")).read()
    return sorted(set(re.findall(r"^VST_API\s+[\w\s\*]+?\b(vst_\w+)\s*\(", src, flags=re.M)))


def test_library_loads_and_exports_header(page_constants):
    L = vst.lib()
    names = header_functions()
    assert len(names) >= 18
    for n in names:
        assert hasattr(L, n), n
    assert sorted(vst.EXPORTS) == names


def test_version_and_status_strings():
    assert re.match(r"^\d+\.\d+\.\d+$", vst.version())
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert vst.status_str(s)


def test_default_configs_match_pages(page_constants):
    c = page_constants
    e = vst.config_default(vst.ENC)
    assert (e.n_heads, e.n_kv_heads, e.head_dim, e.window, e.ring_slots, e.max_batch) == (
        c["enc_heads"], c["enc_heads"], c["enc_head_dim"], c["enc_window"], c["enc_ring_slots"], c["enc_max_batch"])
    d = vst.config_default(vst.DEC)
    assert (d.n_heads, d.n_kv_heads, d.head_dim, d.window) == (
        c["dec_q_heads"], c["dec_kv_heads"], c["dec_head_dim"], c["dec_window"])
    assert e.rope_theta == d.rope_theta == c["rope_theta"]
    assert d.max_position == c["max_position"]


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 32, vst.E_UNSUPPORTED), ("window", 0, vst.E_INVAL), ("ring_slots", 1000, vst.E_INVAL),
    ("n_kv_heads", 3, vst.E_INVAL), ("reserved", 1, vst.E_INVAL), ("max_batch", 1024, vst.E_INVAL),
    ("rope_theta", -1.0, vst.E_INVAL), ("kind", 7, vst.E_INVAL)])
def test_bad_encoder_configs_rejected_before_cuda(field, value, status):
    c = vst.config_default(vst.ENC)
    setattr(c, field, value)
    h = ctypes.c_void_p()
    assert vst.lib().vst_module_create(ctypes.byref(c), ctypes.byref(h)) == status
    assert not h.value


def test_batch_over_512_unsupported():
    c = vst.config_default(vst.ENC)
    c.ring_slots, c.max_batch = 4096, 1024
    h = ctypes.c_void_p()
    assert vst.lib().vst_module_create(ctypes.byref(c), ctypes.byref(h)) == vst.E_UNSUPPORTED


def test_bad_decoder_configs_rejected_before_cuda():
    for field, value, status in [("n_heads", 16, vst.E_UNSUPPORTED), ("ring_slots", 8000, vst.E_INVAL),
                                 ("ring_slots", 8192 + 64, vst.E_UNSUPPORTED), ("head_dim", 64, vst.E_UNSUPPORTED)]:
        c = vst.config_default(vst.DEC)
        setattr(c, field, value)
        h = ctypes.c_void_p()
        assert vst.lib().vst_module_create(ctypes.byref(c), ctypes.byref(h)) == status, (field, value)


def test_null_arguments_rejected():
    L = vst.lib()
    assert L.vst_enc_feed(None, None, None, None, 1, None, None) == vst.E_INVAL
    assert L.vst_dec_step(None, 1, None, None, None, None, None) == vst.E_INVAL
    assert L.vst_ctx_reset(None, None) == vst.E_INVAL
    assert L.vst_ctx_compact(None, None) == vst.E_INVAL
    assert L.vst_ctx_bytes(None) == 0


def test_enc_plan_matches_oracle_ring():
    """The schedule vst_enc_feed enqueues equals the oracle's ring bookkeeping (bit-exact
    integer work), for random feed sizes including 0, 1 and more than a batch."""
    cfg = vst.config_default(vst.ENC)
    rng = random.Random(11)
    for trial in range(20):
        st = oracle.RingState()
        n_kv, base = 0, 0
        for _ in range(200):
            n = rng.choice([0, 1, 3, 24, 48, 50, 100, 511, 512, 513, 1024, 2000])
            steps, n_kv, base = vst.enc_plan(cfg, n_kv, base, n)
            before = st.n_compactions
            st.feed(n)
            assert (n_kv, base) == (st.n_kv, st.abs_base)
            assert sum(b for b, _ in steps) == n
            assert all(0 < b <= 512 for b, _ in steps)
            assert sum(c for _, c in steps) == st.n_compactions - before


def test_enc_plan_hand_cases():
    cfg = vst.config_default(vst.ENC)
    steps, n_kv, base = vst.enc_plan(cfg, 0, 0, 2000)
    assert steps == [(512, 0), (512, 0), (512, 0), (464, 1)] and (n_kv, base) == (1214, 786)
    steps, n_kv, base = vst.enc_plan(cfg, 1500, 0, 50)
    assert steps == [(50, 1)] and (n_kv, base) == (800, 750)
    steps, n_kv, base = vst.enc_plan(cfg, 1486, 0, 50)
    assert steps == [(50, 0)] and (n_kv, base) == (1536, 0)


class _FakeCudaTensor:
    """Stands in for a CUDA tensor in the binding's checks (no GPU here)."""

    def __init__(self, n, dtype=None, cuda=True, contiguous=True):
        import torch
        self.n, self.dtype, self.is_cuda, self.contig = n, dtype or torch.bfloat16, cuda, contiguous

    def numel(self):
        return self.n

    def is_contiguous(self):
        return self.contig

    def data_ptr(self):
        return 0x1000


def test_binding_refuses_short_tensors():
    """The binding checks every tensor against the rows the call reads or writes before it
    reaches the library (whose pointers carry no size), and refuses anything but contiguous
    bf16 CUDA tensors."""
    import torch
    cfg = vst.config_default(vst.ENC)
    rows, hd = 10, cfg.n_heads * cfg.head_dim
    hkd = cfg.n_kv_heads * cfg.head_dim
    full, full_kv = _FakeCudaTensor(rows * hd), _FakeCudaTensor(rows * hkd)
    assert vst._io(cfg, rows, full, full_kv, full_kv, full) == (0x1000,) * 4
    assert vst._io(cfg, rows, None, 5, full_kv, None) == (0, 5, 0x1000, 0)  # None and raw pointers pass
    for i, n in enumerate((rows * hd, rows * hkd, rows * hkd, rows * hd)):
        for b in (_FakeCudaTensor(n - 1), _FakeCudaTensor(n, dtype=torch.float16), _FakeCudaTensor(n, cuda=False),
                  _FakeCudaTensor(n, contiguous=False), torch.empty(n, dtype=torch.bfloat16)):
            args = [full, full_kv, full_kv, full]
            args[i] = b
            with pytest.raises(ValueError):
                vst._io(cfg, rows, *args)
    short = _FakeCudaTensor(1)
    assert vst._io(None, rows, short, short, short, short) == (0x1000,) * 4  # unknown ctx: no size to check


def test_split_shape_grid_fits_the_resident_ctas():
    """The split shape of the chunk attention has a CTA that waits for the other CTAs of its
    (ctx, head), so its grid must be resident at once: checked with faked SM counts (a full
    GB300 at one split CTA per SM, an MPS share, a small green context, no occupancy)."""
    shape = vst.enc_launch_shape
    # one stream of 20 heads, a 50-frame feed: 7 or 8 key tiles of the 750 window
    assert shape(20, 1, 50, 7, 152) == (1, 7)     # 140 CTAs fit 152 SMs
    assert shape(20, 1, 50, 8, 152) == (2, 4)     # 160 do not: pairs of tiles, 80 CTAs
    assert shape(20, 1, 50, 7, 76) == (3, 3)      # half the SMs (MPS 50 %): 60 CTAs
    assert shape(20, 1, 50, 7, 20) == (0, 1)      # one CTA per head would not leave room: loop shape
    assert shape(20, 1, 50, 7, 0) == (0, 1)       # no split CTA fits an SM: loop shape
    assert shape(20, 1, 129, 8, 152) == (0, 2)    # two query tiles: loop shape
    assert shape(20, 8, 100, 8, 152) == (0, 1)    # 160 (ctx, head) pairs fill the GPU: loop shape
    rng = random.Random(7)
    for _ in range(3000):
        H, n, b, t = rng.randint(1, 32), rng.randint(1, 64), rng.randint(1, 512), rng.randint(1, 9)
        res = rng.choice([0, 1, 8, 20, 76, 100, 152, 304, rng.randint(0, 400)])
        k, gx = shape(H, n, b, t, res)
        if k == 0:
            assert gx == (b + 127) // 128
            assert b > 128 or n * H >= res
        else:
            assert b <= 128 and n * H < res
            assert gx == -(-t // k)
            assert n * H * gx <= res                              # the whole grid is resident
            assert k == 1 or n * H * -(-t // (k - 1)) > res       # and k is the least that fits
    for bad in [(0, 1, 50, 7, 152), (20, 0, 50, 7, 152), (20, 1, 0, 7, 152), (20, 1, 50, 0, 152),
                (20, 1, 50, 7, -1)]:
        with pytest.raises(vst.VstError) as e:
            shape(*bad)
        assert e.value.status == vst.E_INVAL
