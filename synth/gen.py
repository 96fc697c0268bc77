"""Counter-based seeded normal generator shared by both sides of every test.

This module holds no arithmetic of the attention method: it only turns
(seed, tensor id, element index) into a reproducible number, so that the
CUDA library and the fp64 oracle can be fed the very same inputs.

Definition (the only thing both sides rely on):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): ``out(key, n) = mix(key + (n + 1) * GAMMA)`` with
  ``mix(z) = z3`` where ``z1 = (z ^ (z >> 30)) * C1``,
  ``z2 = (z1 ^ (z1 >> 27)) * C2``, ``z3 = z2 ^ (z2 >> 31)``, all mod 2**64.
* ``key(seed, tensor_id) = mix(((seed << 32) + tensor_id + 1) * GAMMA)``.
* Element ``i`` of a tensor draws two words ``out(key, 2i)`` and
  ``out(key, 2i + 1)``, maps each to ``u = (w >> 11) * 2**-53 + 2**-54``
  (a uniform in the open interval (0, 1)), and takes the cosine branch of the
  Box-Muller transform (Box and Muller, 1958):
  ``z = sqrt(-2 ln u1) * cos(2 pi u2)``, in float64.
* The stored value is ``z * sigma`` rounded to float32 (round to nearest
  even) and, for bfloat16 tensors, rounded once more from float32 to
  bfloat16 (round to nearest even).

The same torch code runs on the CPU (inputs for the oracle) and on a CUDA
device (large inputs such as the prefill hidden states).  Integer arithmetic
is done in int64 with two's-complement wrap-around, which equals the uint64
arithmetic of the definition; right shifts are made logical by masking.
"""
from __future__ import annotations

import torch

GAMMA = 0x9E3779B97F4A7C15
C1 = 0xBF58476D1CE4E5B9
C2 = 0x94D049BB133111EB
_U64 = 1 << 64


def _s64(x: int) -> int:
    """Reinterpret an unsigned 64-bit integer as a signed int64 value."""
    x &= _U64 - 1
    return x - _U64 if x >= (1 << 63) else x


def _mix_int(z: int) -> int:
    z &= _U64 - 1
    z = ((z ^ (z >> 30)) * C1) & (_U64 - 1)
    z = ((z ^ (z >> 27)) * C2) & (_U64 - 1)
    return z ^ (z >> 31)


def stream_key(seed: int, tensor_id: int) -> int:
    """Per-tensor SplitMix64 key, as an unsigned Python int."""
    return _mix_int((((seed << 32) + tensor_id + 1) * GAMMA) & (_U64 - 1))


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 lanes (torch's >> is arithmetic)."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _s64(C1)
    z = (z ^ _lsr(z, 27)) * _s64(C2)
    return z ^ _lsr(z, 31)


def _uniform(words: torch.Tensor) -> torch.Tensor:
    return _lsr(words, 11).to(torch.float64) * (2.0 ** -53) + 2.0 ** -54


def normal_f64(seed: int, tensor_id: int, start: int, count: int,
               device="cpu") -> torch.Tensor:
    """Standard normals for element indices start .. start+count-1 (float64)."""
    key = _s64(stream_key(seed, tensor_id))
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    n1 = idx * 2 + 1                       # (n + 1) for n = 2i
    w1 = _mix(n1 * _s64(GAMMA) + key)
    w2 = _mix((n1 + 1) * _s64(GAMMA) + key)
    u1 = _uniform(w1)
    u2 = _uniform(w2)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * torch.pi) * u2)


def fill(seed: int, tensor_id: int, shape, sigma: float, dtype: torch.dtype,
         device="cpu", start: int = 0, chunk: int = 1 << 24) -> torch.Tensor:
    """Tensor of ``shape`` whose flat element k is element ``start + k``.

    ``dtype`` is torch.float32 or torch.bfloat16.  Generation is chunked so
    that the int64/float64 temporaries stay small.
    """
    numel = 1
    for s in shape:
        numel *= int(s)
    out = torch.empty(numel, dtype=dtype, device=device)
    for off in range(0, numel, chunk):
        n = min(chunk, numel - off)
        z = normal_f64(seed, tensor_id, start + off, n, device=device)
        v = (z * sigma).to(torch.float32)
        out[off:off + n] = v.to(dtype)
    return out.view(*shape)


def bf16_bits_from_f32(x: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even float32 -> bfloat16, as raw 16-bit patterns.

    Written out with integer operations so that a test can check torch's
    own conversion (used by ``fill``) against the definition.
    """
    b = x.to(torch.float32).contiguous().view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    lsb = (b >> 16) & 1
    r = (b + 0x7FFF + lsb) >> 16
    return (r & 0xFFFF).to(torch.int32)
