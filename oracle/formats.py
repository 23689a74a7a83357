"""KV storage formats and the int4 cold codec, written out from their definitions.

TEST INFRASTRUCTURE: see the package docstring for who may import this.

* KvFormat {f32, f16, q8_0} — "KV Cache Design — cells, format, sessions",
  section 3 ("The storage format is a gate, never a guess").
  - f32: the row is stored as is.
  - f16: IEEE binary16, round to nearest even.
  - q8_0: groups of 32 values; one f16 scale d = amax/127 followed by 32
    int8 codes q = round-ties-even(x/d) (the page's store quantiser:
    "amax/127, f16 scale, round-ties-even"). A cell is a whole number of
    Q8_0 blocks rounded up to whole f32 words.
* int4 cold blocks — "Tiered KV cache — architecture", section "The
  three-tier model": per block one f32 scale followed by ceil(n/2) packed
  int4 nibbles.

Readings where the pages leave a step open:
  - q8_0 block byte layout: {f16 d (little endian); int8 q[32]} = 34 bytes;
    head h of a row owns blocks [h*d/32, (h+1)*d/32); the row is zero-padded
    to a multiple of 4 bytes.
  - q8_0 codes divide by the float32 d32 = amax/127 (IEEE division), not by
    the f16-rounded scale; codes are clamped to [-127, 127]; amax == 0 gives
    d = 0 and all codes 0.
  - int4: scale = amax/7 in float32, q = clamp(rint(x/scale), -8, 7),
    nibble = q + 8, element 2j in the low nibble of byte j and 2j+1 in the
    high nibble; amax == 0 gives scale 0 and every nibble 8. The block's
    elements are in pool order [slot][head][dim]. Dequantisation rounds the
    float32 product scale*(n-8) once more to the pool's type.
"""
from __future__ import annotations

import numpy as np

FORMATS = ("f32", "f16", "q8_0")
Q8_GROUP = 32
Q8_BLOCK_BYTES = 34


def row_bytes(fmt: str, n_kv_heads: int, head_dim: int) -> int:
    """Bytes of one cell (one token's K or V for all KV heads)."""
    n = n_kv_heads * head_dim
    if fmt == "f32":
        return 4 * n
    if fmt == "f16":
        return 2 * n
    if fmt == "q8_0":
        if head_dim % Q8_GROUP:
            raise ValueError("q8_0 needs head_dim % 32 == 0")
        raw = (n // Q8_GROUP) * Q8_BLOCK_BYTES
        return -(-raw // 4) * 4
    raise ValueError(f"unknown KV format {fmt!r}")


def to_f16(x) -> np.ndarray:
    """float32 -> binary16, round to nearest even (numpy's conversion)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16)


def q8_0_quantize_groups(x: np.ndarray):
    """Quantise float32 values in groups of 32.

    x: float32 [..., 32]. Returns (d16 float16 [...], q int8 [..., 32]).
    """
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] == Q8_GROUP
    amax = np.max(np.abs(x), axis=-1)
    d32 = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(d32 == 0, np.float32(1.0), d32).astype(np.float32)
    ratio = (x / safe[..., None]).astype(np.float32)
    q = np.rint(ratio)
    q = np.clip(q, -127, 127)
    q = np.where((d32 == 0)[..., None], 0, q).astype(np.int8)
    return to_f16(d32), q


def encode_rows(fmt: str, x: np.ndarray, n_kv_heads: int, head_dim: int) -> np.ndarray:
    """Store float32 rows [n_rows][n_kv_heads*head_dim] in `fmt` cells.

    Returns uint8 [n_rows][row_bytes(fmt, ...)].
    """
    x = np.asarray(x, dtype=np.float32)
    n_rows, n = x.shape
    assert n == n_kv_heads * head_dim
    rb = row_bytes(fmt, n_kv_heads, head_dim)
    if fmt == "f32":
        return x.copy().view(np.uint8).reshape(n_rows, rb)
    if fmt == "f16":
        return to_f16(x).view(np.uint8).reshape(n_rows, rb)
    d16, q = q8_0_quantize_groups(x.reshape(n_rows, n // Q8_GROUP, Q8_GROUP))
    blocks = np.zeros((n_rows, n // Q8_GROUP, Q8_BLOCK_BYTES), dtype=np.uint8)
    blocks[:, :, 0:2] = d16.astype("<f2").view(np.uint8).reshape(n_rows, n // Q8_GROUP, 2)
    blocks[:, :, 2:] = q.view(np.uint8)
    out = np.zeros((n_rows, rb), dtype=np.uint8)
    out[:, : blocks.shape[1] * Q8_BLOCK_BYTES] = blocks.reshape(n_rows, -1)
    return out


def decode_rows(fmt: str, cells: np.ndarray, n_kv_heads: int, head_dim: int) -> np.ndarray:
    """Read `fmt` cells back as float64 [n_rows][n_kv_heads*head_dim].

    q8_0 values are d*q with d the stored f16 scale: an 11-bit by 8-bit
    significand product, exact in float64 (and in float32).
    """
    cells = np.ascontiguousarray(cells, dtype=np.uint8)
    n_rows = cells.shape[0]
    n = n_kv_heads * head_dim
    if fmt == "f32":
        return cells.view("<f4").reshape(n_rows, n).astype(np.float64)
    if fmt == "f16":
        return cells.view("<f2").reshape(n_rows, n).astype(np.float64)
    g = n // Q8_GROUP
    blocks = cells[:, : g * Q8_BLOCK_BYTES].reshape(n_rows, g, Q8_BLOCK_BYTES)
    d = np.ascontiguousarray(blocks[:, :, 0:2]).view("<f2").reshape(n_rows, g).astype(np.float64)
    q = np.ascontiguousarray(blocks[:, :, 2:]).view(np.int8).astype(np.float64)
    return (d[:, :, None] * q).reshape(n_rows, n)


def int4_quantize_block(x: np.ndarray):
    """Quantise one block's values (any float type, flattened in pool order).

    Returns (scale float32, nibbles uint8 [ceil(n/2)]).
    """
    x = np.asarray(x).astype(np.float32).ravel()
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    scale = np.float32(amax / np.float32(7.0))
    if scale == 0:
        q = np.zeros(x.size, dtype=np.int64)
    else:
        q = np.clip(np.rint((x / scale).astype(np.float32)), -8, 7).astype(np.int64)
    nib = (q + 8).astype(np.uint8)
    if nib.size % 2:
        nib = np.concatenate([nib, np.zeros(1, dtype=np.uint8)])
    packed = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    return scale, packed


def int4_dequantize_block(scale, nibbles: np.ndarray, n: int, fmt: str) -> np.ndarray:
    """Inverse of int4_quantize_block: values scale*(nibble-8), rounded to
    float32 and then to the pool type `fmt` ('f16' or 'f32')."""
    nibbles = np.asarray(nibbles, dtype=np.uint8)
    nib = np.empty(2 * nibbles.size, dtype=np.int64)
    nib[0::2] = nibbles & 0xF
    nib[1::2] = nibbles >> 4
    vals = (np.float32(scale) * (nib[:n] - 8).astype(np.float32)).astype(np.float32)
    if fmt == "f16":
        return to_f16(vals)
    if fmt == "f32":
        return vals
    raise ValueError("int4 cold blocks hold f16 or f32 pools")
