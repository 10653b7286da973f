"""Plain fp64 CPU oracle for paged-KV decode attention.

TEST INFRASTRUCTURE. Only the tests, the smoke check of the package entry
module and the benchmark's CPU-baseline leg may import or call this module.
It shares no code with the CUDA path and imports nothing from it.

What is computed (the definition, written out):
for every sequence b, query token t and query head h, with kv head
g = floor(h / G), G = Hq / Hkv,

    keys   J = { paged token j : 0 <= j < C_b }  (+ the T draft-block scratch
             tokens of (b, g) in the TiDAR mode)
    k_j    = k_cache[block_tables[b, j // P], j % P, g, :]   (v_j likewise)
    s_j    = scale * <q[b, t, h, :], k_j>
    m      = max_j s_j,   l = sum_j exp(s_j - m)
    out    = sum_j exp(s_j - m) v_j / l
    lse    = m + ln l                     (natural log, scale included)

An empty key set gives out = 0 and lse = -inf.

Sources. The problem (paged KV caches plus scratch storage for draft tokens,
FlashAttention-style softmax with split-K, and the log-sum-exp as the
quantity to compare) is stated on the ROCm blog page "Implementing a
High-Performance Custom Diffusion Attention Kernel with FlyDSL"
(introduction items 1 and 3; "Debug Systematically"). The fp8 KV format
(OCP e4m3fn codes with a symmetric per-token scale) and the split-K partial
combine are from the MSLK pull request "[ROCm] Add FlyDSL paged-attention
decode backend (dense + fp8) with benchmark" (sections Kernels and Other
changes). Readings of what the pages leave open:
  * GQA: query head h uses kv head floor(h * Hkv / Hq) (contiguous groups).
  * lse is the natural log and includes the softmax scale.
  * Tokens at or past C_b are never keys; block-table entries past
    ceil(C_b / P) are never read.
  * fp8: x = value(code) * scale[page, slot, head]; the value of a code is
    the OCP e4m3fn definition (bias 7, no infinities, S.1111.111 is NaN).
  * f16 format (the MSLK pull request's dense path is "f16/bf16"): q, the
    caches and the scratch are IEEE binary16, widened exactly.
  * Draft-block mode: every draft token attends to the whole paged prefix
    and to all T scratch tokens of its sequence (no mask inside the block).
    With a draft-block size bs (inputs["draft_block"]), draft token t sees
    scratch token t' only if floor(t' / bs) <= floor(t / bs): the first
    min(T, (floor(t / bs) + 1) * bs) scratch tokens. bs = 1 is causal,
    bs >= T the unmasked mode.
  * Split-K (used to check the combine): split s of sequence b holds pages
    [s * pps, min((s + 1) * pps, n_b)) with pps = ceil(n_b / S) and
    n_b = ceil(C_b / P); the draft-block scratch tokens belong to split S-1.
    Combine: M = max_s lse_s, w_s = exp(lse_s - M),
    out = sum_s w_s out_s / sum_s w_s, lse = M + ln sum_s w_s; splits with
    lse = -inf weigh 0.

Every parity pin of this module lives in tests/test_oracle.py.
"""

from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np


# ---------------------------------------------------------------------------
# Exact widening of the stored formats to float64
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly: a bf16 value is the
    float32 whose upper 16 bits are the pattern and whose lower 16 are 0."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns (uint16) -> float64, exactly (1 sign, 5
    exponent bits with bias 15, 10 mantissa bits; exponent 0 subnormal)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def widen16(bits: np.ndarray, kv_format: str) -> np.ndarray:
    """16-bit rows of q (and of the 16-bit caches) to float64: f16 in the f16
    format, bf16 otherwise (the fp8 format keeps a bf16 q)."""
    return f16_bits_to_f64(bits) if kv_format == "f16" else bf16_bits_to_f64(bits)


def e4m3fn_value(code: int) -> float:
    """Value of one OCP e4m3fn code: 1 sign bit, 4 exponent bits (bias 7),
    3 mantissa bits; exponent 0 is subnormal (2^-6 * m/8); the pattern
    S.1111.111 is NaN; there are no infinities."""
    s = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * math.ldexp(m / 8.0, -6)
    return s * math.ldexp(1.0 + m / 8.0, e - 7)


def e4m3fn_table() -> np.ndarray:
    """The 256 e4m3fn code values as float64."""
    return np.array([e4m3fn_value(c) for c in range(256)], dtype=np.float64)


_E4M3FN = e4m3fn_table()


# ---------------------------------------------------------------------------
# Keys and values of one (sequence, kv head)
# ---------------------------------------------------------------------------

def _paged_rows(cache: np.ndarray, scales: Optional[np.ndarray], kv_format: str,
                bt_row: np.ndarray, ctx: int, page_size: int, g: int) -> np.ndarray:
    """The ctx logical rows of kv head g, read page by page through the
    block table, widened to float64: row j comes from physical page
    bt_row[j // P], slot j % P."""
    D = cache.shape[-1]
    out = np.empty((ctx, D), dtype=np.float64)
    for j in range(0, ctx, page_size):
        page = int(bt_row[j // page_size])
        n = min(page_size, ctx - j)
        raw = cache[page, :n, g, :]
        if kv_format in ("bf16", "f16"):
            out[j:j + n] = widen16(raw, kv_format)
        elif kv_format == "fp8":
            out[j:j + n] = _E4M3FN[raw] * scales[page, :n, g].astype(np.float64)[:, None]
        else:
            raise ValueError(kv_format)
    return out


def visible_scratch(inputs: dict, t: int) -> int:
    """How many scratch tokens (a prefix of the draft block) draft token t
    sees: all T, or min(T, (floor(t / bs) + 1) * bs) with a block size bs."""
    T = inputs["k_scratch"].shape[1]
    bs = inputs.get("draft_block")
    if bs is None:
        return T
    return min(T, (t // int(bs) + 1) * int(bs))


def keys_values(inputs: dict, b: int, g: int, page_range: Optional[Tuple[int, int]] = None,
                with_scratch: bool = True, scratch_count: Optional[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Keys and values (float64, [N, D]) of sequence b, kv head g: the paged
    tokens (all of them, or those of the pages in page_range), then the
    draft-block scratch tokens (all, or the first scratch_count) when present
    and with_scratch is set."""
    P = inputs["k_cache"].shape[1]
    ctx = max(0, int(inputs["context_lens"][b]))
    kv_format = inputs["kv_format"]
    first, last = 0, ctx
    if page_range is not None:
        first = min(ctx, page_range[0] * P)
        last = min(ctx, page_range[1] * P)
    bt_row = inputs["block_tables"][b]
    ks = _paged_rows(inputs["k_cache"], inputs.get("k_scale"), kv_format, bt_row, ctx, P, g)[first:last]
    vs = _paged_rows(inputs["v_cache"], inputs.get("v_scale"), kv_format, bt_row, ctx, P, g)[first:last]
    if with_scratch and inputs.get("k_scratch") is not None:
        n = inputs["k_scratch"].shape[1] if scratch_count is None else scratch_count
        ks = np.concatenate([ks, widen16(inputs["k_scratch"][b, :n, g, :], kv_format)], axis=0)
        vs = np.concatenate([vs, widen16(inputs["v_scratch"][b, :n, g, :], kv_format)], axis=0)
    return ks, vs


def _by_key_set(inputs: dict, sel):
    """Groups query rows (t, h) by the scratch tokens their draft token sees
    (one group without a scratch block): {scratch count or None: rows}."""
    groups = {}
    for (t, h) in sel:
        n = visible_scratch(inputs, t) if inputs.get("k_scratch") is not None else None
        groups.setdefault(n, []).append((t, h))
    return groups


# ---------------------------------------------------------------------------
# Softmax attention of a few query rows over one key set
# ---------------------------------------------------------------------------

def attend(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float):
    """out[r] = softmax_j(scale * q_r . k_j) @ V and lse[r] = ln sum_j exp(scale * q_r . k_j),
    evaluated as m + ln sum exp(s - m). No keys: out 0, lse -inf."""
    R, D = q_rows.shape
    if keys.shape[0] == 0:
        return np.zeros((R, values.shape[1]), dtype=np.float64), np.full(R, -np.inf)
    s = scale * (q_rows @ keys.T)                 # [R, N]
    m = s.max(axis=1, keepdims=True)              # [R, 1]
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    out = (e @ values) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


# ---------------------------------------------------------------------------
# Public oracle entry points
# ---------------------------------------------------------------------------

def as_oracle_inputs(bits: dict, kv_format: str) -> dict:
    """Bundle raw-bit numpy arrays (bf16 as uint16, fp8 as uint8) for the oracle."""
    d = dict(bits)
    d["kv_format"] = kv_format
    return d


def decode(inputs: dict, scale: float,
           rows: Optional[Iterable[Tuple[int, int, int]]] = None):
    """Full decode: out [B, T, Hq, D] and lse [B, T, Hq] in float64.

    With rows = [(b, t, h), ...] only those rows are computed; the others
    stay NaN (used to check single outputs of very large problems)."""
    q = inputs["q"]
    B, T, Hq, D = q.shape
    Hkv = inputs["k_cache"].shape[2]
    G = Hq // Hkv
    out = np.full((B, T, Hq, D), np.nan)
    lse = np.full((B, T, Hq), np.nan)
    want = None
    if rows is not None:
        want = {}
        for (b, t, h) in rows:
            want.setdefault((b, h * Hkv // Hq), []).append((t, h))
    units = want.keys() if want is not None else [(b, g) for b in range(B) for g in range(Hkv)]
    for (b, g) in units:
        if want is None:
            sel = [(t, h) for t in range(T) for h in range(g * G, (g + 1) * G)]
        else:
            sel = want[(b, g)]
        for n, group in _by_key_set(inputs, sel).items():
            keys, values = keys_values(inputs, b, g, scratch_count=n)
            q_rows = np.stack([widen16(q[b, t, h], inputs["kv_format"]) for (t, h) in group])
            o, l = attend(q_rows, keys, values, scale)
            for i, (t, h) in enumerate(group):
                out[b, t, h] = o[i]
                lse[b, t, h] = l[i]
    return out, lse


def split_page_ranges(n_pages: int, num_splits: int):
    """Page ranges [a, b) of the S splits of a sequence with n_pages pages."""
    pps = -(-n_pages // num_splits) if n_pages > 0 else 0
    ranges = []
    for s in range(num_splits):
        a = min(n_pages, s * pps)
        ranges.append((a, min(n_pages, a + pps) if pps else a))
    return ranges


def decode_split(inputs: dict, scale: float, num_splits: int):
    """Split-K partials: part_out [B, T, Hq, S, D] (each normalised over its
    own keys) and part_lse [B, T, Hq, S]."""
    q = inputs["q"]
    B, T, Hq, D = q.shape
    P = inputs["k_cache"].shape[1]
    Hkv = inputs["k_cache"].shape[2]
    G = Hq // Hkv
    S = num_splits
    part_out = np.zeros((B, T, Hq, S, D))
    part_lse = np.full((B, T, Hq, S), -np.inf)
    for b in range(B):
        ctx = max(0, int(inputs["context_lens"][b]))
        n_pages = -(-ctx // P)
        for s, (a, e) in enumerate(split_page_ranges(n_pages, S)):
            for g in range(Hkv):
                sel = [(t, h) for t in range(T) for h in range(g * G, (g + 1) * G)]
                for n, group in _by_key_set(inputs, sel).items():
                    keys, values = keys_values(inputs, b, g, page_range=(a, e),
                                               with_scratch=(s == S - 1), scratch_count=n)
                    q_rows = np.stack([widen16(q[b, t, h], inputs["kv_format"]) for (t, h) in group])
                    o, l = attend(q_rows, keys, values, scale)
                    for i, (t, h) in enumerate(group):
                        part_out[b, t, h, s] = o[i]
                        part_lse[b, t, h, s] = l[i]
    return part_out, part_lse


def combine(part_out: np.ndarray, part_lse: np.ndarray):
    """LSE-weighted combine of split partials along the split axis
    (part_out [..., S, D], part_lse [..., S]) -> out [..., D], lse [...]."""
    M = part_lse.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(M)
    Msafe = np.where(empty, 0.0, M)
    w = np.where(np.isfinite(part_lse), np.exp(part_lse - Msafe), 0.0)
    L = w.sum(axis=-1, keepdims=True)
    Lsafe = np.where(L > 0, L, 1.0)
    out = (w[..., None] * part_out).sum(axis=-2) / Lsafe
    lse = np.where(empty, -np.inf, Msafe + np.log(Lsafe))[..., 0]
    out = np.where(empty, 0.0, out)
    return out, lse
