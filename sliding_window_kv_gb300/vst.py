"""Thin ctypes binding of libvst (include/vst.h), same names without the ``vst_`` prefix.

Argument marshalling only: every step of the attention path runs in the CUDA kernels of
libvst.so. Tensors are torch bf16 CUDA tensors (contiguous); their data pointers and the
current CUDA stream are passed through. There is no fallback: if libvst.so is missing or
fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libvst.so")

OK, E_INVAL, E_UNSUPPORTED, E_CUDA, E_STATE, E_TIMEOUT, E_NOMEM = 0, -1, -2, -3, -4, -5, -6
ENC, DEC = 1, 2


class VstError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s (%d)" % (what, status_str(status), status))
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("window", ctypes.c_int32), ("ring_slots", ctypes.c_int32),
                ("max_batch", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("max_position", ctypes.c_int64), ("rope_theta", ctypes.c_double)]


class CtxInfo(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("failed", ctypes.c_int32), ("n_kv", ctypes.c_int64),
                ("abs_base", ctypes.c_int64), ("abs_next", ctypes.c_int64),
                ("n_compactions", ctypes.c_int64), ("k_ring", ctypes.c_void_p), ("v_ring", ctypes.c_void_p)]


class ProfStat(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("reserved", ctypes.c_int32), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


K_ROPE_APPEND, K_COMPACT, K_ENC_ATTN, K_DEC_STEP, K_COUNT = 0, 1, 2, 3, 4

EXPORTS = ["vst_config_default", "vst_module_create", "vst_module_destroy", "vst_module_config",
           "vst_ctx_bytes", "vst_ctx_create", "vst_ctx_reset", "vst_ctx_destroy", "vst_ctx_info_get",
           "vst_ctx_check", "vst_ctx_selftest_wait", "vst_enc_feed", "vst_enc_feed_batch", "vst_ctx_compact", "vst_enc_plan",
           "vst_enc_launch_shape",
           "vst_offline_bytes", "vst_offline_create", "vst_offline_destroy", "vst_enc_offline", "vst_offline_check",
           "vst_dec_step", "vst_dec_step_noalloc", "vst_dec_prefill", "vst_dec_append", "vst_prof_enable", "vst_prof_read", "vst_launch_count",
           "vst_kernel_name", "vst_status_str", "vst_version"]

_lib = None


def lib():
    """Load libvst.so (raises if it is missing: there is no other implementation)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libvst.so is not built (run __graft_entry__.build()): %s" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        PP = ctypes.POINTER(ctypes.c_void_p)
        sig = {
            "vst_config_default": ([I32, ctypes.POINTER(Config)], I32),
            "vst_module_create": ([ctypes.POINTER(Config), PP], I32),
            "vst_module_destroy": ([P], I32),
            "vst_module_config": ([P, ctypes.POINTER(Config)], I32),
            "vst_ctx_bytes": ([P], SZ),
            "vst_ctx_create": ([P, P, SZ, P, PP], I32),
            "vst_ctx_reset": ([P, P], I32),
            "vst_ctx_destroy": ([P], I32),
            "vst_ctx_info_get": ([P, ctypes.POINTER(CtxInfo)], I32),
            "vst_ctx_check": ([P, P], I32),
            "vst_ctx_selftest_wait": ([P, I32, P], I32),
            "vst_enc_feed": ([P, P, P, P, I32, P, P], I32),
            "vst_enc_feed_batch": ([PP, I32, P, P, P, I32, P, P], I32),
            "vst_ctx_compact": ([P, P], I32),
            "vst_enc_plan": ([ctypes.POINTER(Config), I64, I64, I32, ctypes.POINTER(I32), ctypes.POINTER(I32), I32,
                              ctypes.POINTER(I32), ctypes.POINTER(I64), ctypes.POINTER(I64)], I32),
            "vst_enc_launch_shape": ([I32, I32, I32, I32, I64, ctypes.POINTER(I32), ctypes.POINTER(I32)], I32),
            "vst_dec_step": ([PP, I32, P, P, P, P, P], I32),
            "vst_dec_step_noalloc": ([PP, I32, P, P, P, P, P], I32),
            "vst_dec_prefill": ([P, P, P, P, I32, P, P], I32),
            "vst_offline_bytes": ([P, I32, I32], SZ),
            "vst_offline_create": ([P, I32, I32, P, SZ, PP], I32),
            "vst_offline_destroy": ([P], I32),
            "vst_enc_offline": ([P, P, P, P, I32, I32, P, P], I32),
            "vst_offline_check": ([P, P], I32),
            "vst_dec_append": ([P, P, P, I32, P], I32),
            "vst_prof_enable": ([I32], I32),
            "vst_prof_read": ([ctypes.POINTER(ProfStat), I32], I32),
            "vst_launch_count": ([], I64),
            "vst_kernel_name": ([I32], ctypes.c_char_p),
            "vst_status_str": ([I32], ctypes.c_char_p),
            "vst_version": ([], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def status_str(s: int) -> str:
    return lib().vst_status_str(s).decode()


def version() -> str:
    return lib().vst_version().decode()


def _check(s: int, what: str):
    if s != OK:
        raise VstError(s, what)


_torch = None
_raw_stream = None  # (getter of the current stream's handle for a device index, current device index)


def _t():
    global _torch
    if _torch is None:
        import torch
        _torch = torch
    return _torch


def _p(t, n_elems: int, name: str, bf16) -> int:
    """Data pointer of a contiguous bf16 CUDA tensor holding at least n_elems elements; a raw
    integer pointer passes through (the caller's responsibility) and None gives 0."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if t.dtype is not bf16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s: expected a contiguous bf16 CUDA tensor" % name)
    if t.numel() < n_elems:
        raise ValueError("%s: %d elements, the call needs %d" % (name, t.numel(), n_elems))
    return t.data_ptr()


def _ptr(t) -> int:
    return _p(t, 0, "tensor", _t().bfloat16)


# ctx handle -> its module's config, for the size checks below (filled by ctx_create)
_ctx_cfg: dict = {}


def _io(cfg, rows: int, q, k, v, out):
    """Pointers of q, k, v and out after the checks of _p: q and out hold `rows` rows of
    [H][D], k and v `rows` rows of [Hk][D] (sizes unchecked when the config is unknown)."""
    bf16 = _t().bfloat16
    hq = hk = 0
    if cfg is not None:
        hq = rows * cfg.n_heads * cfg.head_dim
        hk = rows * cfg.n_kv_heads * cfg.head_dim
    return _p(q, hq, "q", bf16), _p(k, hk, "k", bf16), _p(v, hk, "v", bf16), _p(out, hq, "out", bf16)


def _stream(stream) -> int:
    """Handle of `stream` (a torch stream or a raw handle); None: torch's current stream on
    the current device."""
    global _raw_stream
    if stream is None:
        torch = _t()
        if _raw_stream is None:
            h = torch.cuda.current_stream().cuda_stream  # also initialises CUDA
            get = getattr(torch._C, "_cuda_getCurrentRawStream", None)
            dev = getattr(torch._C, "_cuda_getDevice", None)
            _raw_stream = (get, dev) if get is not None and dev is not None else False
            return h
        if _raw_stream:
            return _raw_stream[0](_raw_stream[1]())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def config_default(kind: int) -> Config:
    c = Config()
    _check(lib().vst_config_default(kind, ctypes.byref(c)), "vst_config_default")
    return c


def module_create(cfg: Config) -> int:
    h = ctypes.c_void_p()
    _check(lib().vst_module_create(ctypes.byref(cfg), ctypes.byref(h)), "vst_module_create")
    return h.value


def module_destroy(m: int):
    _check(lib().vst_module_destroy(m), "vst_module_destroy")


def module_config(m: int) -> Config:
    c = Config()
    _check(lib().vst_module_config(m, ctypes.byref(c)), "vst_module_config")
    return c


def ctx_bytes(m: int) -> int:
    return lib().vst_ctx_bytes(m)


def ctx_create(m: int, dev_mem: int = 0, nbytes: int = 0, stream=None) -> int:
    h = ctypes.c_void_p()
    _check(lib().vst_ctx_create(m, dev_mem or None, nbytes, _stream(stream), ctypes.byref(h)), "vst_ctx_create")
    _ctx_cfg[h.value] = module_config(m)
    return h.value


def ctx_reset(c: int, stream=None):
    _check(lib().vst_ctx_reset(c, _stream(stream)), "vst_ctx_reset")


def ctx_destroy(c: int):
    _check(lib().vst_ctx_destroy(c), "vst_ctx_destroy")
    _ctx_cfg.pop(c, None)


def ctx_info_get(c: int) -> CtxInfo:
    i = CtxInfo()
    _check(lib().vst_ctx_info_get(c, ctypes.byref(i)), "vst_ctx_info_get")
    return i


def ctx_check(c: int, stream=None) -> int:
    return lib().vst_ctx_check(c, _stream(stream))


def ctx_selftest_wait(c: int, complete: bool, stream=None):
    _check(lib().vst_ctx_selftest_wait(c, 1 if complete else 0, _stream(stream)), "vst_ctx_selftest_wait")


def enc_feed(c: int, q, k, v, out, stream=None, n_new: int | None = None):
    n = q.shape[0] if n_new is None else n_new
    pq, pk, pv, po = _io(_ctx_cfg.get(c), n, q, k, v, out)
    _check(lib().vst_enc_feed(c, pq, pk, pv, n, po, _stream(stream)), "vst_enc_feed")


def _handles(ctxs):
    arr = (ctypes.c_void_p * len(ctxs))(*ctxs)
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def enc_feed_batch(ctxs, q, k, v, out, n_new: int, stream=None):
    h, keep = _handles(ctxs)
    pq, pk, pv, po = _io(_ctx_cfg.get(ctxs[0]) if ctxs else None, len(ctxs) * n_new, q, k, v, out)
    _check(lib().vst_enc_feed_batch(h, len(ctxs), pq, pk, pv, n_new, po, _stream(stream)),
           "vst_enc_feed_batch")


def ctx_compact(c: int, stream=None):
    _check(lib().vst_ctx_compact(c, _stream(stream)), "vst_ctx_compact")


def enc_plan(cfg: Config, n_kv: int, abs_base: int, n_new: int, max_steps: int = 4096):
    batch = (ctypes.c_int32 * max_steps)()
    comp = (ctypes.c_int32 * max_steps)()
    n = ctypes.c_int32()
    nk = ctypes.c_int64()
    ab = ctypes.c_int64()
    _check(lib().vst_enc_plan(ctypes.byref(cfg), n_kv, abs_base, n_new, batch, comp, max_steps, ctypes.byref(n),
                              ctypes.byref(nk), ctypes.byref(ab)), "vst_enc_plan")
    k = min(n.value, max_steps)
    return [(batch[i], comp[i]) for i in range(k)], nk.value, ab.value


def enc_launch_shape(n_heads: int, n_ctx: int, batch: int, max_key_tiles: int, resident_ctas: int):
    """(split, grid_x) of the chunk attention's launch: split = 0 for the loop shape, else key
    tiles per CTA of the split shape (host-only; see vst_enc_launch_shape)."""
    sp = ctypes.c_int32()
    gx = ctypes.c_int32()
    _check(lib().vst_enc_launch_shape(n_heads, n_ctx, batch, max_key_tiles, resident_ctas, ctypes.byref(sp),
                                      ctypes.byref(gx)), "vst_enc_launch_shape")
    return sp.value, gx.value


def dec_step(ctxs, q, k, v, out, stream=None):
    h, keep = _handles(ctxs)
    pq, pk, pv, po = _io(_ctx_cfg.get(ctxs[0]) if ctxs else None, len(ctxs), q, k, v, out)
    _check(lib().vst_dec_step(h, len(ctxs), pq, pk, pv, po, _stream(stream)),
           "vst_dec_step")


def dec_step_noalloc(ctxs, q, k, v, out, stream=None):
    """vst_dec_step with its scratch in the library's static device array (no allocation)."""
    h, keep = _handles(ctxs)
    pq, pk, pv, po = _io(_ctx_cfg.get(ctxs[0]) if ctxs else None, len(ctxs), q, k, v, out)
    _check(lib().vst_dec_step_noalloc(h, len(ctxs), pq, pk, pv, po, _stream(stream)),
           "vst_dec_step_noalloc")


def dec_prefill(c: int, q, k, v, out, n: int | None = None, stream=None):
    """vst_dec_prefill: n tokens of one decoder ctx, q/out [n][H][D], k/v [n][Hk][D]."""
    n = q.shape[0] if n is None else n
    pq, pk, pv, po = _io(_ctx_cfg.get(c), n, q, k, v, out)
    _check(lib().vst_dec_prefill(c, pq, pk, pv, n, po, _stream(stream)), "vst_dec_prefill")


class Offline:
    """Owning wrapper: vst_offline_create / vst_offline_destroy (library-owned scratch)."""

    def __init__(self, module: "Module", B: int, T: int):
        out = ctypes.c_void_p()
        _check(lib().vst_offline_create(module.handle, B, T, None, 0, ctypes.byref(out)), "vst_offline_create")
        self.handle, self.B, self.T, self.cfg = out.value, B, T, module.cfg

    def run(self, q, k, v, out, left: int, right: int = 0, stream=None):
        """vst_enc_offline: q, k, v, out [B][T][H][D]."""
        pq, pk, pv, po = _io(self.cfg, self.B * self.T, q, k, v, out)
        _check(lib().vst_enc_offline(self.handle, pq, pk, pv, left, right, po, _stream(stream)), "vst_enc_offline")

    def check(self, stream=None) -> int:
        return lib().vst_offline_check(self.handle, _stream(stream))

    def close(self):
        if self.handle:
            lib().vst_offline_destroy(self.handle)
            self.handle = None


def offline_bytes(module_handle: int, B: int, T: int) -> int:
    return lib().vst_offline_bytes(module_handle, B, T)


def dec_append(c: int, k, v, n: int | None = None, stream=None):
    n = k.shape[0] if n is None else n
    _, pk, pv, _ = _io(_ctx_cfg.get(c), n, None, k, v, None)
    _check(lib().vst_dec_append(c, pk, pv, n, _stream(stream)), "vst_dec_append")


class Module:
    """Owning wrapper: vst_module_create / vst_module_destroy."""

    def __init__(self, cfg_or_kind):
        self.cfg = config_default(cfg_or_kind) if isinstance(cfg_or_kind, int) else cfg_or_kind
        self.handle = module_create(self.cfg)

    def close(self):
        if self.handle:
            module_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Ctx:
    """Owning wrapper: vst_ctx_create (library-allocated memory) / vst_ctx_destroy."""

    def __init__(self, module: Module, stream=None):
        self.module = module
        self.handle = ctx_create(module.handle, 0, 0, stream)

    def info(self) -> CtxInfo:
        return ctx_info_get(self.handle)

    def close(self):
        if self.handle:
            ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def prof_enable(on: bool):
    _check(lib().vst_prof_enable(1 if on else 0), "vst_prof_enable")


def prof_read() -> dict:
    """{kernel name: (launches, total_ms)} for the launches timed since the last read."""
    arr = (ProfStat * K_COUNT)()
    _check(lib().vst_prof_read(arr, K_COUNT), "vst_prof_read")
    return {kernel_name(a.kernel): (a.launches, a.total_ms) for a in arr}


def launch_count() -> int:
    return lib().vst_launch_count()


def kernel_name(k: int) -> str:
    return lib().vst_kernel_name(k).decode()
