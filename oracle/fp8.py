"""E4M3 latent-cache rows: the codec and the row quantiser of the FP8 cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and
the benchmark's CPU-baseline leg may import this module.  The CUDA library
never imports, links or calls it, and shares no code with it.

Sources:
  [DS-report] page "DeepSeek 系列模型技术深度解读", section "FP8 混合精度训练"
              (DeepSeek-V3): the forward pass runs the attention GEMMs in
              FP8 while precision-sensitive parts stay in BF16.
  [OFP8]      the OCP 8-bit floating point specification, format E4M3:
              1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no
              infinities; exponent and mantissa all ones is NaN, so the
              largest finite magnitude is 1.75 * 2^8 = 448; exponent field 0
              holds the subnormals m/8 * 2^-6.

Readings (the pages give no scaling scheme for a cached row; each is a
stated assumption):
  * the 512 latent values c^KV of a row are stored as E4M3 codes with one
    fp32 scale s per row; a code stands for s * E4M3(code);
  * s = amax / 448 with amax = max |c_i| over the row, and the code of c_i
    is E4M3 of c_i * (448 / amax), rounded to nearest with ties to even and
    saturated at +-448; an all-zero row has s = 1 and all codes 0;
  * the decision is taken in fp32 on the row as it is produced in bf16
    (the value rounded to nearest-even bf16 from fp32): the two quotients
    448 / amax and amax / 448 and the product c_i * (448 / amax) are each
    rounded to fp32 -- the arithmetic the kernels use;
  * the 64 RoPE-key values k^R stay in bf16 and are stored divided by s
    (bf16 of fp32(k^R / s)), so that the score's latent and RoPE parts share
    one scale; a stored value stands for s * stored.
The dequantised row [s * E4M3(codes) ; s * stored k^R] is what the FP8 cache
holds; the decode over it is ``oracle.mla.decode_explicit`` unchanged.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Values of E4M3 codes (uint8 array) per [OFP8]; NaN for the NaN codes."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = m / 8.0 * 2.0 ** -6
    v = np.where(e == 0, sub, normal)
    v = np.where((e == 15) & ((c & 0x7) == 7), np.nan, v)
    return sign * v


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes of finite values x: nearest, ties to even, saturating.

    A magnitude below 2^-6 is a subnormal m * 2^-9 (m = 0..7; m = 8 carries
    into the smallest normal); above, x = (1 + f) 2^e with the mantissa
    f * 8 rounded to an integer (8 carries into the next binade); a
    magnitude past 448 gives 448.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    sign = np.where(np.signbit(x), 0x80, 0)
    out = np.zeros(x.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    m_sub = np.rint(a / 2.0 ** -9)            # ties to even; 8 -> code 0x08
    out = np.where(sub, m_sub, out)
    mant, ex = np.frexp(np.where(sub, 1.0, a))   # a = mant * 2^ex, mant in [0.5, 1)
    e = ex - 1                                    # a = (2 mant) * 2^e
    m = np.rint((2.0 * mant - 1.0) * 8.0)
    carry = m == 8
    e = np.where(carry, e + 1, e)
    m = np.where(carry, 0, m)
    code_n = ((e + 7) << 3) | m.astype(np.int64)
    code_n = np.minimum(code_n, 0x7E)           # saturate at 448 (0x7F is NaN)
    big = a >= E4M3_MAX
    out = np.where(sub, out, code_n)
    out = np.where(big, 0x7E, out)
    return (out.astype(np.int64) | sign).astype(np.uint8)


def bf16_round(x) -> np.ndarray:
    """fp32 -> bf16 (round to nearest, ties to even) of finite values, as
    float32 values."""
    f = np.asarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def quantize_rows(rows: np.ndarray, d_latent: int) -> dict:
    """FP8 cache rows of ``rows`` [N, d_latent + d_R] (float64, the exact
    rows), per the readings above.  Returns the stored parts (codes uint8
    [N, d_latent], scale float32 [N], kr bf16 values as float32 [N, d_R])
    and the dequantised rows ``deq`` [N, d_latent + d_R] (float64)."""
    rows = np.asarray(rows, dtype=np.float64)
    c = bf16_round(rows[:, :d_latent].astype(np.float32))
    kr = bf16_round(rows[:, d_latent:].astype(np.float32))
    amax = np.max(np.abs(c), axis=1)
    zero = amax == 0
    safe = np.where(zero, np.float32(1.0), amax).astype(np.float32)
    scale = np.where(zero, np.float32(1.0), safe / np.float32(E4M3_MAX)).astype(np.float32)
    inv = np.where(zero, np.float32(1.0), np.float32(E4M3_MAX) / safe).astype(np.float32)
    x = (c * inv[:, None]).astype(np.float32)
    codes = e4m3_encode(x)
    kr_s = bf16_round((kr / scale[:, None]).astype(np.float32))
    deq = np.concatenate([scale[:, None].astype(np.float64) * e4m3_decode(codes),
                          scale[:, None].astype(np.float64) * kr_s.astype(np.float64)], axis=1)
    return {"codes": codes, "scale": scale, "kr": kr_s, "deq": deq}
