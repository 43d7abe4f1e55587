"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle side.

This module holds none of the attention arithmetic. It only draws bf16 values that are
approximately N(0, 1), as a pure function of (seed, tensor id, element index), so that:

* the GPU side can generate tens of GB directly in device memory, and
* the oracle side can regenerate any slice (say the 750 frames in front of a sampled row)
  on the CPU, bit for bit, without the two ever exchanging data.

Construction. A 32-bit integer mixer (the xor-shift-multiply hash with multiplier
0x45d9f3b, applied twice, published by Thomas Mueller) hashes the element index together
with a per-tensor key. Every intermediate stays below 2**63, so int64 tensor arithmetic is
exact on any device. The low 16 bits pick an entry of a 65536-entry table holding
bf16(Phi^-1((u + 0.5) / 65536)), the standard-normal quantiles at the cell centres, so the
values follow N(0, 1) up to 16-bit quantisation and bf16 rounding. The table is computed
in float64 with ``torch.special.ndtri`` and rounded once to bf16.
"""
from __future__ import annotations

import functools

import torch

_M32 = 0xFFFFFFFF
_MULT = 0x45D9F3B


def _mix32(x: torch.Tensor) -> torch.Tensor:
    """32-bit mixer on int64 tensors holding values in [0, 2**32)."""
    x = ((x >> 16) ^ x) * _MULT & _M32
    x = ((x >> 16) ^ x) * _MULT & _M32
    return (x >> 16) ^ x


def _mix32_int(x: int) -> int:
    x &= _M32
    x = (((x >> 16) ^ x) * _MULT) & _M32
    x = (((x >> 16) ^ x) * _MULT) & _M32
    return (x >> 16) ^ x


def tensor_key(seed: int, *ids: int) -> int:
    """Fold a seed and a tuple of small integer ids into one 32-bit key."""
    k = _mix32_int(seed * 0x9E37 + 0x1234567)
    for i in ids:
        k = _mix32_int(k ^ _mix32_int(int(i) + 0x51ED27))
    return k


@functools.lru_cache(maxsize=None)
def _normal_table_cpu() -> torch.Tensor:
    u = (torch.arange(65536, dtype=torch.float64) + 0.5) / 65536.0
    return torch.special.ndtri(u).to(torch.bfloat16)


_tables: dict = {}


def _normal_table(device) -> torch.Tensor:
    dev = torch.device(device)
    t = _tables.get(dev)
    if t is None:
        t = _normal_table_cpu().to(dev)
        _tables[dev] = t
    return t


def bf16_normal(key: int, start: int, shape, device="cpu") -> torch.Tensor:
    """bf16 values ~N(0,1) for elements start .. start+numel-1 of the stream named by key."""
    n = 1
    for s in shape:
        n *= int(s)
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    lo = idx & _M32
    hi = idx >> 32
    h = _mix32(lo ^ _mix32(hi ^ key))
    return _normal_table(device)[h & 0xFFFF].reshape(tuple(shape))


def frames(key: int, frame_begin: int, n_frames: int, n_heads: int, head_dim: int,
           device="cpu") -> torch.Tensor:
    """Frames [frame_begin, frame_begin + n_frames) of a [frames][heads][head_dim] sequence."""
    per = n_heads * head_dim
    return bf16_normal(key, frame_begin * per, (n_frames, n_heads, head_dim), device)


def uniform_int(key: int, n: int, lo: int, hi: int) -> list[int]:
    """n integers uniform in [lo, hi] (inclusive), from the same counter hash."""
    idx = torch.arange(n, dtype=torch.int64)
    h = _mix32(idx ^ key)
    span = hi - lo + 1
    return [lo + int(x) % span for x in h.tolist()]


def bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (what the oracle takes)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
