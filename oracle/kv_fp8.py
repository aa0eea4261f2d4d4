"""FP8 (E4M3) key / value cache with one scale per (kv head, 128-token page)
(oracle side).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Source: "EAGLE-2: Feature-Level Speculative Decoding Guide", production
section (serving engines keep the KV cache in a shared pool for high
concurrency).  The pages give no number format for that cache; the reading
built here (each part a reading, stated once):

* element format: E4M3 -- 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
  bits; exponent field 0 holds the subnormals m * 2^-9; the all-ones code
  S.1111.111 is not a number and there is no infinity, so the largest finite
  magnitude is 1.75 * 2^8 = 448;
* scaling: the stored code of element x of page p of kv head h is E4M3(x /
  s[h][p]) rounded to nearest (ties to even mantissa), saturated to +-448;
  its value is decode(code) * s[h][p].  A page is 128 consecutive tokens of
  one kv head (all head_dim columns); the scale is the page's largest
  magnitude / 448 (how the cache's writer picks it; the attention only
  consumes codes and scales);
* the tree's own keys and values are not cached yet when the tree is
  verified: they stay bf16.

The attention over such a cache is the ordinary definition
(``tree_attention``) on the decoded values.
"""

import numpy as np

from .tree_attn import tree_attention

E4M3_MAX = 448.0
PAGE = 128


def e4m3_decode(codes):
    """uint8 codes -> float64 values (NaN for the S.1111.111 codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = sign * (1.0 + m / 8.0) * np.exp2(e - 7.0)
    sub = sign * (m / 8.0) * np.exp2(-6.0)
    v = np.where(e == 0, sub, normal)
    return np.where((e == 0xF) & (m == 0x7), np.nan, v)


def _finite_table():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    return codes, e4m3_decode(codes)


def e4m3_encode(x):
    """float values -> uint8 codes: nearest finite E4M3 value, ties to the
    even mantissa (the code with mantissa bit 0 clear), magnitudes beyond 448
    saturated to 448, the sign kept (a negative value that rounds to zero
    gives -0).  Written as a search over the 254 finite codes so that
    it follows the definition of rounding directly."""
    x = np.asarray(x, dtype=np.float64)
    codes, vals = _finite_table()
    pos = codes[(codes & 0x80) == 0]
    pv = e4m3_decode(pos)
    order = np.argsort(pv)
    pos, pv = pos[order], pv[order]          # 0, 2^-9, ..., 448 ascending
    mag = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(pv, mag, side="left"), 0, len(pv) - 1)
    lo = np.clip(hi - 1, 0, len(pv) - 1)
    d_hi = np.abs(pv[hi] - mag)
    d_lo = np.abs(mag - pv[lo])
    take_lo = (d_lo < d_hi) | ((d_lo == d_hi) & ((pos[lo] & 1) == 0))
    code = np.where(take_lo, pos[lo], pos[hi]).astype(np.uint8)
    return np.where(x < 0, code | 0x80, code).astype(np.uint8)


def page_scales(x, page=PAGE):
    """x [Hkv, S, d] -> scales [Hkv, ceil(S / page)]: each page's largest
    magnitude / 448 (a page of zeros gets 1)."""
    x = np.asarray(x, dtype=np.float64)
    hkv, S, _ = x.shape
    n = (S + page - 1) // page
    out = np.ones((hkv, n), dtype=np.float64)
    for p in range(n):
        amax = np.abs(x[:, p * page:(p + 1) * page]).max(axis=(1, 2))
        out[:, p] = np.where(amax > 0, amax / E4M3_MAX, 1.0)
    return out


def quantize_cache(x, scales, page=PAGE):
    """x [Hkv, S, d], scales [Hkv, pages] -> uint8 codes [Hkv, S, d]."""
    x = np.asarray(x, dtype=np.float64)
    s = np.repeat(np.asarray(scales, dtype=np.float64), page, axis=1)[:, : x.shape[1]]
    return e4m3_encode(x / s[:, :, None])


def dequantize_cache(codes, scales, page=PAGE):
    """uint8 codes [Hkv, S, d], scales [Hkv, pages] -> float64 [Hkv, S, d]."""
    codes = np.asarray(codes)
    s = np.repeat(np.asarray(scales, dtype=np.float64), page, axis=1)[:, : codes.shape[1]]
    return e4m3_decode(codes) * s[:, :, None]


def tree_attention_fp8(q, k_codes, k_scales, v_codes, v_scales, tree_k, tree_v, mask,
                       prefix_len, scale=None, heads=None, page=PAGE):
    """Tree attention over an E4M3 prefix cache (decode, then the definition);
    tree keys / values as given (bf16 values widened by the caller)."""
    k = dequantize_cache(np.asarray(k_codes)[:, :prefix_len], k_scales, page)
    v = dequantize_cache(np.asarray(v_codes)[:, :prefix_len], v_scales, page)
    return tree_attention(q, k, v, tree_k, tree_v, mask, prefix_len, scale=scale, heads=heads)
