"""Seeded synthetic inputs for paged-KV decode attention.

This module is shared by the tests, the benchmark and the oracle checks. It
draws random numbers and lays them out; it holds none of the attention
arithmetic. The workloads follow the statement of the problem on the ROCm
blog page "Implementing a High-Performance Custom Diffusion Attention Kernel
with FlyDSL" (introduction, item 1: paged KV caches plus scratch storage for
speculatively generated draft tokens) and the MSLK pull request "[ROCm] Add
FlyDSL paged-attention decode backend (dense + fp8) with benchmark" (Kernels:
dense bf16 and native fp8 e4m3fn KV with a symmetric per-token scale).

Layouts (all row-major, contiguous):
    q            [B, T, Hq, D]           bf16
    k/v cache    [num_pages, P, Hkv, D]  bf16, or e4m3fn codes as uint8
    k/v scale    [num_pages, P, Hkv]     float32 (fp8 only)
    block_tables [B, max_blocks]         int32, -1 where unused
    context_lens [B]                     int32
    k/v scratch  [B, T, Hkv, D]          bf16 (draft-block mode only)

Random streams: every tensor has its own stream id, and large tensors are
filled in chunks of whole pages, each chunk from its own generator seeded by
(seed, stream id, chunk index). The data are therefore a pure function of
the seed, independent of the number of threads used to make them.
"""

from __future__ import annotations

import dataclasses
import math
import os
import threading
from typing import Optional, Sequence

import numpy as np
import torch

E4M3FN_MAX = 448.0

_STREAM_CTX = 1
_STREAM_PERM = 2
_STREAM_Q = 3
_STREAM_K = 4
_STREAM_V = 5
_STREAM_KS = 6
_STREAM_VS = 7
_STREAM_KNEW = 8
_STREAM_VNEW = 9

# Elements per generator chunk (whole pages are kept together).
_CHUNK_ELEMS = 1 << 22


@dataclasses.dataclass(frozen=True)
class DecodeSpec:
    """Shape and value recipe of one decode workload."""

    name: str
    batch: int
    q_tokens: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    # Either explicit context lengths, or an inclusive uniform range.
    context_lens: Optional[Sequence[int]] = None
    ctx_range: Optional[tuple] = None
    kv_format: str = "bf16"  # "bf16", "f16" (q, caches and out in f16) or "fp8"
    draft_scratch: bool = False  # TiDAR draft block: contiguous scratch KV
    pool_pages: Optional[int] = None  # None: exactly the pages in use
    max_blocks_per_seq: Optional[int] = None  # None: from the largest context
    seed: int = 0
    draft_block: Optional[int] = None  # block-masked draft: token t sees the scratch blocks up to its own

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


# The five workloads of the decode engine (sizes from the problem statement).
SPECS = {
    "tiny": DecodeSpec("tiny", batch=2, q_tokens=1, num_q_heads=4, num_kv_heads=1,
                       head_dim=64, page_size=16, context_lens=(37, 100),
                       pool_pages=16, seed=0),
    "gqa": DecodeSpec("gqa", batch=32, q_tokens=1, num_q_heads=32, num_kv_heads=8,
                      head_dim=128, page_size=16, ctx_range=(512, 8192),
                      max_blocks_per_seq=8192 // 16, seed=1),
    "long": DecodeSpec("long", batch=4, q_tokens=1, num_q_heads=64, num_kv_heads=8,
                       head_dim=128, page_size=64, context_lens=(131072,) * 4, seed=2),
    "fp8": DecodeSpec("fp8", batch=64, q_tokens=1, num_q_heads=32, num_kv_heads=2,
                      head_dim=256, page_size=16, ctx_range=(1024, 16384),
                      kv_format="fp8", max_blocks_per_seq=16384 // 16, seed=3),
    "tidar": DecodeSpec("tidar", batch=16, q_tokens=8, num_q_heads=32, num_kv_heads=8,
                        head_dim=128, page_size=16, ctx_range=(2048, 8192),
                        draft_scratch=True, max_blocks_per_seq=8192 // 16, seed=4),
    # The GQA geometry in f16, and in bf16 with head dims 64 and 256.
    "gqa_f16": DecodeSpec("gqa_f16", batch=32, q_tokens=1, num_q_heads=32, num_kv_heads=8,
                          head_dim=128, page_size=16, ctx_range=(512, 8192), kv_format="f16",
                          max_blocks_per_seq=8192 // 16, seed=9),
    "gqa_d64": DecodeSpec("gqa_d64", batch=32, q_tokens=1, num_q_heads=32, num_kv_heads=8,
                          head_dim=64, page_size=16, ctx_range=(512, 8192),
                          max_blocks_per_seq=8192 // 16, seed=10),
    "gqa_d256": DecodeSpec("gqa_d256", batch=32, q_tokens=1, num_q_heads=32, num_kv_heads=8,
                           head_dim=256, page_size=16, ctx_range=(512, 8192),
                           max_blocks_per_seq=8192 // 16, seed=11),
    # Draft-block variants: the TiDAR workload with a causal draft, and a
    # 16-token draft (64 query rows per kv head) in blocks of 4.
    "tidar_causal": DecodeSpec("tidar_causal", batch=16, q_tokens=8, num_q_heads=32, num_kv_heads=8,
                               head_dim=128, page_size=16, ctx_range=(2048, 8192), draft_scratch=True,
                               max_blocks_per_seq=8192 // 16, seed=4, draft_block=1),
    "tidar_long": DecodeSpec("tidar_long", batch=16, q_tokens=16, num_q_heads=32, num_kv_heads=8,
                             head_dim=128, page_size=16, ctx_range=(2048, 8192), draft_scratch=True,
                             max_blocks_per_seq=8192 // 16, seed=8, draft_block=4),
}


@dataclasses.dataclass
class DecodeInputs:
    """Host (CPU) tensors of one decode problem."""

    spec: DecodeSpec
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None
    k_scratch: Optional[torch.Tensor] = None
    v_scratch: Optional[torch.Tensor] = None

    @property
    def scale(self) -> float:
        return self.spec.scale

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def tensors(self):
        names = ["q", "k_cache", "v_cache", "block_tables", "context_lens",
                 "k_scale", "v_scale", "k_scratch", "v_scratch"]
        return {n: getattr(self, n) for n in names if getattr(self, n) is not None}

    def to(self, device, non_blocking: bool = False) -> "DecodeInputs":
        moved = {n: t.to(device, non_blocking=non_blocking) for n, t in self.tensors().items()}
        return dataclasses.replace(self, **moved)

    def pin_memory(self) -> "DecodeInputs":
        return dataclasses.replace(self, **{n: t.pin_memory() for n, t in self.tensors().items()})

    # Raw-bit numpy views for the oracle (bf16 as uint16, fp8 as uint8).
    def numpy_bits(self):
        def bits(t):
            if t is None:
                return None
            if t.dtype in (torch.bfloat16, torch.float16):
                return t.contiguous().view(torch.int16).numpy().view(np.uint16)
            return t.contiguous().numpy()
        return {n: bits(t) for n, t in self.tensors().items()}


def _rng(seed: int, stream: int, chunk: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, chunk])))


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _parallel(fn, n: int) -> None:
    """Run fn(i) for i in range(n) on a few threads (numpy releases the GIL)."""
    nt = min(_threads(), n)
    if nt <= 1:
        for i in range(n):
            fn(i)
        return
    err = []

    def worker(w):
        try:
            for i in range(w, n, nt):
                fn(i)
        except BaseException as e:  # surfaced below
            err.append(e)

    ths = [threading.Thread(target=worker, args=(w,)) for w in range(nt)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    if err:
        raise err[0]


def _normal_bf16(shape, seed: int, stream: int, rows_per_chunk: int, dtype=torch.bfloat16) -> torch.Tensor:
    """N(0,1) float32 draws rounded to bf16 (or f16) by round to nearest even, chunked on dim 0."""
    out = torch.empty(shape, dtype=dtype)
    n0 = shape[0]
    nchunks = max(1, -(-n0 // rows_per_chunk))
    row_elems = int(np.prod(shape[1:])) if len(shape) > 1 else 1

    def fill(c):
        r0, r1 = c * rows_per_chunk, min(n0, (c + 1) * rows_per_chunk)
        buf = np.empty((r1 - r0) * row_elems, dtype=np.float32)
        _rng(seed, stream, c).standard_normal(out=buf, dtype=np.float32)
        out[r0:r1] = torch.from_numpy(buf).view((r1 - r0,) + tuple(shape[1:])).to(dtype)

    _parallel(fill, nchunks)
    return out


def _normal_fp8(shape, seed: int, stream: int, rows_per_chunk: int):
    """N(0,1) float32 draws quantised to e4m3fn with a symmetric scale per
    (page, token, kv head): scale = amax over D / 448 (fp32), code = RNE of
    clamp(x / scale, -448, 448). An all-zero vector gets scale 1."""
    codes = torch.empty(shape, dtype=torch.uint8)
    scales = torch.empty(shape[:-1], dtype=torch.float32)
    n0 = shape[0]
    nchunks = max(1, -(-n0 // rows_per_chunk))
    row_elems = int(np.prod(shape[1:]))

    def fill(c):
        r0, r1 = c * rows_per_chunk, min(n0, (c + 1) * rows_per_chunk)
        buf = np.empty((r1 - r0) * row_elems, dtype=np.float32)
        _rng(seed, stream, c).standard_normal(out=buf, dtype=np.float32)
        x = torch.from_numpy(buf).view((r1 - r0,) + tuple(shape[1:]))
        amax = x.abs().amax(dim=-1)
        s = torch.where(amax > 0, amax / E4M3FN_MAX, torch.ones_like(amax))
        y = torch.clamp(x / s.unsqueeze(-1), -E4M3FN_MAX, E4M3FN_MAX)
        codes[r0:r1] = y.to(torch.float8_e4m3fn).view(torch.uint8)
        scales[r0:r1] = s

    _parallel(fill, nchunks)
    return codes, scales


def draw_context_lens(spec: DecodeSpec) -> np.ndarray:
    if spec.context_lens is not None:
        lens = np.asarray(spec.context_lens, dtype=np.int64)
        assert lens.shape == (spec.batch,)
        return lens
    lo, hi = spec.ctx_range
    return _rng(spec.seed, _STREAM_CTX).integers(lo, hi, size=spec.batch, endpoint=True)


def make_inputs(spec: DecodeSpec, poison: bool = False) -> DecodeInputs:
    """Build the host tensors of one decode problem.

    Pages are drawn from a pool through a seeded random permutation: the
    sequences take consecutive slices of the permuted page ids, in batch
    order. With poison=True every value that must never be read is set to
    NaN (unused pool pages, and slots past the context end inside the last
    page of each sequence, including their fp8 scales) and unused
    block-table entries are set to INT32_MAX instead of -1.
    """
    B, T, Hq, Hkv, D, P = (spec.batch, spec.q_tokens, spec.num_q_heads,
                           spec.num_kv_heads, spec.head_dim, spec.page_size)
    assert Hq % Hkv == 0
    lens = draw_context_lens(spec)
    npages = [(int(c) + P - 1) // P for c in lens]
    used = int(sum(npages))
    pool = spec.pool_pages if spec.pool_pages is not None else max(used, 1)
    assert pool >= used, "page pool smaller than the pages in use"
    max_blocks = spec.max_blocks_per_seq if spec.max_blocks_per_seq is not None else max(1, max(npages))
    assert max_blocks >= max(npages)

    perm = _rng(spec.seed, _STREAM_PERM).permutation(pool).astype(np.int64)
    bt = np.full((B, max_blocks), np.iinfo(np.int32).max if poison else -1, dtype=np.int64)
    off = 0
    for b in range(B):
        bt[b, :npages[b]] = perm[off:off + npages[b]]
        off += npages[b]

    page_elems = P * Hkv * D
    rows_per_chunk = max(1, _CHUNK_ELEMS // page_elems)
    t16 = torch.float16 if spec.kv_format == "f16" else torch.bfloat16  # q, 16-bit caches, scratch
    q = _normal_bf16((B, T, Hq, D), spec.seed, _STREAM_Q, max(1, _CHUNK_ELEMS // (T * Hq * D)), t16)
    k_scale = v_scale = None
    if spec.kv_format in ("bf16", "f16"):
        k = _normal_bf16((pool, P, Hkv, D), spec.seed, _STREAM_K, rows_per_chunk, t16)
        v = _normal_bf16((pool, P, Hkv, D), spec.seed, _STREAM_V, rows_per_chunk, t16)
    elif spec.kv_format == "fp8":
        k, k_scale = _normal_fp8((pool, P, Hkv, D), spec.seed, _STREAM_K, rows_per_chunk)
        v, v_scale = _normal_fp8((pool, P, Hkv, D), spec.seed, _STREAM_V, rows_per_chunk)
    else:
        raise ValueError(f"unknown kv_format {spec.kv_format!r}")

    k_scr = v_scr = None
    if spec.draft_scratch:
        k_scr = _normal_bf16((B, T, Hkv, D), spec.seed, _STREAM_KS, B, t16)
        v_scr = _normal_bf16((B, T, Hkv, D), spec.seed, _STREAM_VS, B, t16)

    if poison:
        _poison(k, v, k_scale, v_scale, bt, lens, npages, pool, P)

    return DecodeInputs(
        spec=spec, q=q, k_cache=k, v_cache=v,
        block_tables=torch.from_numpy(bt.astype(np.int32)),
        context_lens=torch.from_numpy(np.asarray(lens, dtype=np.int32)),
        k_scale=k_scale, v_scale=v_scale, k_scratch=k_scr, v_scratch=v_scr)


def _poison(k, v, k_scale, v_scale, bt, lens, npages, pool, P):
    in_use = np.zeros(pool, dtype=bool)
    for b in range(len(lens)):
        in_use[bt[b, :npages[b]]] = True
    unused = torch.from_numpy(np.nonzero(~in_use)[0])

    def nan_fill(t, idx, slot0=None):
        if t.dtype in (torch.bfloat16, torch.float16):
            val = float("nan")
        elif t.dtype == torch.uint8:
            val = 0x7F  # e4m3fn NaN
        else:
            val = float("nan")
        if slot0 is None:
            t[idx] = val
        else:
            t[idx, slot0:] = val

    for t in (k, v, k_scale, v_scale):
        if t is not None and len(unused):
            nan_fill(t, unused)
    for b in range(len(lens)):
        c = int(lens[b])
        if npages[b] and c % P:
            last = int(bt[b, npages[b] - 1])
            for t in (k, v, k_scale, v_scale):
                if t is not None:
                    nan_fill(t, last, c % P)


def custom_spec(name="custom", **kw) -> DecodeSpec:
    """A DecodeSpec for ad-hoc shapes (tests)."""
    return DecodeSpec(name=name, **kw)


# ---------------------------------------------------------------------------
# KV-cache append (the step before a decode)
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class AppendSpec:
    """Shape and value recipe of one KV-cache append: B sequences that cache
    C_b tokens each receive T new tokens (K and V rows N(0,1) in bf16, or in
    f16 for an f16 cache)."""

    name: str
    batch: int
    new_tokens: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    context_lens: Optional[Sequence[int]] = None
    ctx_range: Optional[tuple] = None
    kv_format: str = "bf16"
    pool_pages: Optional[int] = None
    max_blocks_per_seq: Optional[int] = None
    seed: int = 0


# Append workloads: a prefill chunk of 512 tokens per sequence in the GQA
# geometry (bf16) and in the fp8 geometry, and one decode step (T = 1).
APPEND_SPECS = {
    "append": AppendSpec("append", batch=64, new_tokens=512, num_kv_heads=8, head_dim=128, page_size=16,
                         ctx_range=(0, 4096), max_blocks_per_seq=(4096 + 512) // 16, seed=5),
    "append_fp8": AppendSpec("append_fp8", batch=64, new_tokens=512, num_kv_heads=2, head_dim=256, page_size=16,
                             ctx_range=(0, 8192), kv_format="fp8", max_blocks_per_seq=(8192 + 512) // 16, seed=6),
    "append_step": AppendSpec("append_step", batch=32, new_tokens=1, num_kv_heads=8, head_dim=128, page_size=16,
                              ctx_range=(512, 8192), max_blocks_per_seq=8192 // 16 + 1, seed=7),
}


@dataclasses.dataclass
class AppendInputs:
    """Host (CPU) tensors of one append problem. The caches hold earlier
    contents everywhere (the slots the append overwrites included); the
    block tables cover C_b + T tokens of every sequence."""

    spec: AppendSpec
    k_new: torch.Tensor
    v_new: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None

    def tensors(self):
        names = ["k_new", "v_new", "block_tables", "context_lens", "k_cache", "v_cache", "k_scale", "v_scale"]
        return {n: getattr(self, n) for n in names if getattr(self, n) is not None}

    def to(self, device, non_blocking: bool = False) -> "AppendInputs":
        moved = {n: t.to(device, non_blocking=non_blocking) for n, t in self.tensors().items()}
        return dataclasses.replace(self, **moved)

    def clone(self) -> "AppendInputs":
        return dataclasses.replace(self, **{n: t.clone() for n, t in self.tensors().items()})

    def numpy_bits(self):
        return DecodeInputs.numpy_bits(self)


def make_append_inputs(spec: AppendSpec) -> AppendInputs:
    """Pool, block tables and earlier cache contents as for a decode over
    C_b + T tokens (make_inputs), then context_lens = C_b and the new rows."""
    B, T, Hkv, D = spec.batch, spec.new_tokens, spec.num_kv_heads, spec.head_dim
    lens = draw_context_lens(spec)
    base = make_inputs(DecodeSpec(
        name=spec.name, batch=B, q_tokens=1, num_q_heads=Hkv, num_kv_heads=Hkv, head_dim=D,
        page_size=spec.page_size, context_lens=tuple(int(c) + T for c in lens), kv_format=spec.kv_format,
        pool_pages=spec.pool_pages, max_blocks_per_seq=spec.max_blocks_per_seq, seed=spec.seed))
    rows = max(1, _CHUNK_ELEMS // (T * Hkv * D))
    t16 = torch.float16 if spec.kv_format == "f16" else torch.bfloat16  # new rows: the cache's type (fp8: bf16)
    return AppendInputs(
        spec=spec,
        k_new=_normal_bf16((B, T, Hkv, D), spec.seed, _STREAM_KNEW, rows, t16),
        v_new=_normal_bf16((B, T, Hkv, D), spec.seed, _STREAM_VNEW, rows, t16),
        block_tables=base.block_tables,
        context_lens=torch.from_numpy(np.asarray(lens, dtype=np.int32)),
        k_cache=base.k_cache, v_cache=base.v_cache, k_scale=base.k_scale, v_scale=base.v_scale)

