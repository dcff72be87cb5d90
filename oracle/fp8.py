"""FP8 (E4M3, "fn" variant) KV cache: oracle encode/decode and cache write.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Sources: "vllm/v1/attention/backends/flash_attn.py" (kv_cache_dtype "fp8" /
"fp8_e4m3" views the cache as float8_e4m3fn; the same per-tensor scalars
layer._k_scale / layer._v_scale go to reshape_and_cache_flash and, as
k_descale / v_descale, to the attention call; with an fp8 cache the query
goes through scaled_fp8_quant(query, layer._q_scale) and the call gets
q_descale = layer._q_scale) and the FlashInfer backend page
(_trtllm_prefill_attn_kvfp8_dequant: value = fp8 * k_scale;
get_xqa_bmm1_scale: the logit scale times q_scale and k_scale).

Readings: the cache write stores code = e4m3(x / scale), the quotient taken
in float32 and rounded to the nearest E4M3 value (ties to even code),
saturating at +-448; a cached code reads back as decode(code) * scale.  The
query quantization is the same map with the query's scale (a static
per-tensor scale: the pages always pass one), and a query code reads back
as decode(code) * q_scale.

E4M3 "fn" per its definition: 1 sign bit, 4 exponent bits (bias 7),
3 mantissa bits; exponent 0 holds subnormals m/8 * 2^-6; the all-ones code
S.1111.111 is NaN; there is no infinity; the largest finite value is 448.
"""
from __future__ import annotations

import numpy as np


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of uint8 E4M3 codes (NaN for the NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6,
                   (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


_POS_CODES = np.arange(0, 127, dtype=np.uint8)          # +0 .. 448
_POS_VALS = e4m3_decode(_POS_CODES)


def e4m3_encode(x) -> np.ndarray:
    """Round values to E4M3 codes: nearest finite value, ties to the even
    code, saturating at +-448; NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    idx = np.searchsorted(_POS_VALS, a)            # first value >= a
    idx = np.clip(idx, 1, len(_POS_VALS) - 1)
    lo, hi = _POS_VALS[idx - 1], _POS_VALS[idx]
    take_hi = (a - lo > hi - a) | ((a - lo == hi - a) & (idx % 2 == 0))
    code = np.where(take_hi, idx, idx - 1).astype(np.int64)
    code = np.where(a >= _POS_VALS[-1], 126, code)          # saturate
    code = np.where(a == 0, 0, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize_ref(x, scale) -> np.ndarray:
    """E4M3 codes of x / scale, the quotient computed in float32."""
    q = np.asarray(x, dtype=np.float32) / np.float32(scale)
    return e4m3_encode(q.astype(np.float64))


def reshape_and_cache_fp8_ref(key, value, key_cache, value_cache,
                              slot_mapping, k_scale, v_scale):
    """Like reshape_and_cache_ref, storing E4M3 codes (uint8 caches)."""
    block_size = key_cache.shape[1]
    for t in range(len(slot_mapping)):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        blk, off = divmod(s, block_size)
        key_cache[blk, off] = quantize_ref(key[t], k_scale)
        value_cache[blk, off] = quantize_ref(value[t], v_scale)


def scaled_fp8_quant_ref(x, scale) -> np.ndarray:
    """Static per-tensor quantization of a [tokens, heads * head_size] (or
    any-shaped) array: E4M3 codes of x / scale, elementwise as quantize_ref,
    in x's shape."""
    x = np.asarray(x, dtype=np.float32)
    return quantize_ref(x, scale).reshape(x.shape)


def dequantize_ref(codes, scale) -> np.ndarray:
    """float64 values of E4M3 codes read back with a per-tensor scale:
    decode(code) * scale, the scale as the float32 the device holds."""
    return e4m3_decode(codes) * np.float64(np.float32(scale))
