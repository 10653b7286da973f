"""Plain CPU oracle for the KV-cache append step (bf16 copy, or fp8 e4m3fn
quantisation with a per-token, per-kv-head scale).

TEST INFRASTRUCTURE. Only the tests, the smoke check of the package entry
module and the benchmark's CPU-baseline leg may import or call this module.
It shares no code with the CUDA path and imports nothing from it.

What is computed (the definition, written out): the T new tokens of
sequence b take the logical positions C_b, ..., C_b + T - 1 after the C_b
tokens it already caches (C_b = context_lens[b], clamped to
[0, max_blocks_per_seq * P]); position j lives in slot j % P of page
block_tables[b, j // P]. For every new token t and kv head g the K row
k_new[b, t, g, :] (and the V row likewise) is written to that slot:

  * bf16 cache: the row as it is.
  * fp8 cache: with x the row widened exactly to float32,
        amax  = max_d |x_d|
        scale = amax / 448            (float32 division, round to nearest even;
                                       1 when amax = 0)
        y_d   = x_d / scale           (float32 division, round to nearest even)
        code_d = e4m3fn(y_d)          (nearest e4m3fn value, ties to the even
                                       code, magnitudes past 448 saturate to 448)
    and scale goes to k_scale[page, slot, g] (v_scale likewise).

Positions at or past max_blocks_per_seq * P, and page ids outside
[0, num_pages), are not written. Nothing else of the caches changes.

Sources. Paged KV caches with per-sequence block tables, and scratch storage
for the draft tokens, are the problem of the ROCm blog page "Implementing a
High-Performance Custom Diffusion Attention Kernel with FlyDSL" (introduction
item 1). The fp8 format (OCP e4m3fn codes, symmetric per-token scale) is the
MSLK pull request "[ROCm] Add FlyDSL paged-attention decode backend (dense +
fp8) with benchmark" (Kernels; Other changes: OCP rather than fnuz), whose
review thread asks that scales be computed when the cache is written. The
scale amax / 448 per token and kv head is the stated reading of "symmetric
per-token scale" (448 is the largest finite e4m3fn magnitude).

Every parity pin of this module lives in tests/test_oracle_append.py.
"""

from __future__ import annotations

import numpy as np

from .pa_oracle import e4m3fn_table

E4M3FN_MAX = 448.0

# Non-negative finite e4m3fn values in code order (codes 0x00..0x7E); the
# values increase with the code.
_POS_VALUES = e4m3fn_table()[:0x7F]


def e4m3fn_encode(y: np.ndarray) -> np.ndarray:
    """float32 values -> OCP e4m3fn codes (uint8): the nearest finite value,
    ties to the code with an even mantissa, |y| >= 448 saturates to +-448,
    the sign of zero is kept, NaN gives S.1111.111."""
    y = np.asarray(y, dtype=np.float32)
    a = np.abs(y.astype(np.float64)).ravel()
    sign = np.signbit(y).ravel().astype(np.uint8) << 7
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo).astype(np.uint8)
    mag = np.where(a >= E4M3FN_MAX, np.uint8(0x7E), mag)
    mag = np.where(np.isnan(a), np.uint8(0x7F), mag)
    return (mag | sign).reshape(y.shape)


def quantise_rows(x_bits: np.ndarray):
    """bf16 rows (uint16 bit patterns, [..., D]) -> (codes uint8 [..., D],
    scales float32 [...]) as defined in the module docstring."""
    x = (np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3FN_MAX), np.float32(1.0)).astype(np.float32)
    y = (x / scale[..., None]).astype(np.float32)
    return e4m3fn_encode(y), scale


def append(caches: dict, k_new_bits: np.ndarray, v_new_bits: np.ndarray, block_tables: np.ndarray,
           context_lens: np.ndarray, page_size: int) -> dict:
    """Returns copies of the caches with the new tokens appended.

    caches: {"k_cache", "v_cache"} [num_pages, P, Hkv, D] as uint16 (bf16
    bits) or uint8 (e4m3fn codes); for fp8 also {"k_scale", "v_scale"}
    [num_pages, P, Hkv] float32. k_new_bits, v_new_bits [B, T, Hkv, D]
    uint16 (bf16 bits)."""
    out = {n: np.array(a, copy=True) for n, a in caches.items()}
    fp8 = out["k_cache"].dtype == np.uint8
    B, T = k_new_bits.shape[:2]
    num_pages = out["k_cache"].shape[0]
    cap = block_tables.shape[1] * page_size
    for b in range(B):
        c = int(min(max(int(context_lens[b]), 0), cap))
        for t in range(T):
            j = c + t
            if j >= cap:
                continue
            page = int(block_tables[b, j // page_size])
            if not 0 <= page < num_pages:
                continue
            slot = j % page_size
            for name, rows in (("k", k_new_bits), ("v", v_new_bits)):
                if fp8:
                    codes, scale = quantise_rows(rows[b, t])
                    out[name + "_cache"][page, slot] = codes
                    out[name + "_scale"][page, slot] = scale
                else:
                    out[name + "_cache"][page, slot] = rows[b, t]
    return out
