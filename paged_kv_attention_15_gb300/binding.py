"""ctypes binding of libpadecode.so (include/pa_decode.h).

Argument marshalling only: torch supplies device memory and the current
stream; every step of the computation runs in the library's CUDA kernels.
The library is loaded on first use; if it is missing the call raises, there
is no other implementation to fall back to.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpadecode.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "pa_decode.h")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = range(5)


class PaShape(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("q_tokens", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
    ]


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None

_P = ctypes.c_void_p
_DECODE_TAIL = [ctypes.POINTER(PaShape), ctypes.c_float, _P, _P, ctypes.c_int32, _P, ctypes.c_size_t, _P]
_SIGNATURES = {
    "pa_decode_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(PaShape), ctypes.c_int32]),
    "pa_decode_choose_splits": (ctypes.c_int32, [ctypes.POINTER(PaShape), ctypes.c_int32]),
    "pa_decode": (ctypes.c_int, [_P, _P, _P, _P, _P] + _DECODE_TAIL),
    "pa_decode_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P] + _DECODE_TAIL),
    "pa_decode_f16": (ctypes.c_int, [_P, _P, _P, _P, _P] + _DECODE_TAIL),
    "pa_decode_tidar": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P] + _DECODE_TAIL),
    "pa_decode_tidar_masked": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(PaShape), ctypes.c_float,
                                              ctypes.c_int32, _P, _P, ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "pa_decode_reduce": (ctypes.c_int, [_P, _P, ctypes.c_int32, ctypes.POINTER(PaShape), _P, _P, _P]),
    "pa_decode_reduce_f16": (ctypes.c_int, [_P, _P, ctypes.c_int32, ctypes.POINTER(PaShape), _P, _P, _P]),
    "pa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pa_kv_append": (ctypes.c_int, [_P, _P, _P, _P, ctypes.POINTER(PaShape), _P, _P, _P]),
    "pa_kv_append_fp8": (ctypes.c_int, [_P, _P, _P, _P, ctypes.POINTER(PaShape), _P, _P, _P, _P, _P]),
    "pa_decode_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32)]),
    "pa_decode_profile_events": (ctypes.c_int, [_P, _P]),
    "pa_decode_set_kernel_path": (ctypes.c_int, [ctypes.c_int32]),
    "pa_decode_set_combine": (ctypes.c_int, [ctypes.c_int32]),
    "pa_decode_kernel_for": (ctypes.c_int32, [ctypes.POINTER(PaShape), ctypes.c_int32]),
    "pa_decode_heads_per_unit": (ctypes.c_int32, [ctypes.POINTER(PaShape), ctypes.c_int32]),
    "pa_decode_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.POINTER(PaShape), ctypes.c_float, _P, _P,
                                         ctypes.c_int32, _P]),
}


def header_functions() -> list:
    """Names of the functions include/pa_decode.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with paged_kv_attention_15_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PaError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_shape(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor) -> PaShape:
    B, T, Hq, D = q.shape
    num_pages, P, Hkv, Dk = k_cache.shape
    if Dk != D:
        raise ValueError("q and k_cache head_dim differ")
    return PaShape(B, T, Hq, Hkv, D, P, num_pages, block_tables.shape[1])


def workspace_size(shape: PaShape, num_splits: int) -> int:
    return int(lib().pa_decode_workspace_size(ctypes.byref(shape), int(num_splits)))


def choose_splits(shape: PaShape, fp8: bool = False) -> int:
    """What num_splits=0 resolves to: 0 for the balanced schedule, else the
    explicit split count; -1 for an unsupported shape or no device."""
    return int(lib().pa_decode_choose_splits(ctypes.byref(shape), int(bool(fp8))))


def _need_contig(**tensors):
    for name, t in tensors.items():
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
           context_lens: torch.Tensor, scale: float, *, k_scale: Optional[torch.Tensor] = None,
           v_scale: Optional[torch.Tensor] = None, k_scratch: Optional[torch.Tensor] = None,
           v_scratch: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
           lse: Optional[torch.Tensor] = None, num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
           want_lse: bool = True, stream=None, draft_block: Optional[int] = None
           ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Paged decode through pa_decode / pa_decode_fp8 / pa_decode_tidar /
    pa_decode_tidar_masked.

    The fp8 entry point is used when k_cache is uint8 (e4m3fn codes, with
    k_scale/v_scale); pa_decode_f16 when q is float16 (f16 caches and out);
    the draft-block entry point when k_scratch is given,
    its block-masked form when draft_block is given too. out, lse and the
    workspace are allocated here when not passed in."""
    _need_contig(q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables, context_lens=context_lens,
                 k_scale=k_scale, v_scale=v_scale, k_scratch=k_scratch, v_scratch=v_scratch, out=out, lse=lse)
    shape = make_shape(q, k_cache, block_tables)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    need = workspace_size(shape, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if k_scratch is not None and q.dtype != torch.bfloat16:
        raise ValueError("the draft-block entry points take bf16 q, caches and scratch")
    L = lib()
    tail = (ctypes.byref(shape), float(scale), _ptr(out), _ptr(lse), int(num_splits), _ptr(workspace), ws_bytes,
            _stream(stream))
    if k_cache.dtype == torch.uint8:
        st = L.pa_decode_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                             _ptr(block_tables), _ptr(context_lens), *tail)
        _check(st, "pa_decode_fp8")
    elif k_scratch is not None and draft_block is not None:
        st = L.pa_decode_tidar_masked(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scratch), _ptr(v_scratch),
                                      _ptr(block_tables), _ptr(context_lens), ctypes.byref(shape), float(scale),
                                      int(draft_block), _ptr(out), _ptr(lse), int(num_splits), _ptr(workspace),
                                      ws_bytes, _stream(stream))
        _check(st, "pa_decode_tidar_masked")
    elif k_scratch is not None:
        st = L.pa_decode_tidar(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scratch), _ptr(v_scratch),
                               _ptr(block_tables), _ptr(context_lens), *tail)
        _check(st, "pa_decode_tidar")
    elif q.dtype == torch.float16:
        st = L.pa_decode_f16(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), *tail)
        _check(st, "pa_decode_f16")
    else:
        st = L.pa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), *tail)
        _check(st, "pa_decode")
    return out, lse


def decode_inputs(inp, **kw):
    """decode() on a DecodeInputs bundle already on the device (its spec's
    draft_block selects the block-masked draft entry point)."""
    if inp.spec.draft_block is not None and "draft_block" not in kw:
        kw["draft_block"] = inp.spec.draft_block
    return decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale,
                  k_scale=inp.k_scale, v_scale=inp.v_scale, k_scratch=inp.k_scratch, v_scratch=inp.v_scratch,
                  **kw)


def kv_append(k_new: torch.Tensor, v_new: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
              k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: Optional[torch.Tensor] = None,
              v_scale: Optional[torch.Tensor] = None, stream=None) -> None:
    """Appends k_new/v_new [B, T, Hkv, D] (bf16, or f16 into f16 caches) at
    positions context_lens[b] + t through pa_kv_append, or pa_kv_append_fp8
    when the caches are uint8 (e4m3fn codes; k_scale/v_scale [num_pages, P,
    Hkv] fp32 are written)."""
    _need_contig(k_new=k_new, v_new=v_new, block_tables=block_tables, context_lens=context_lens,
                 k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale)
    want = torch.bfloat16 if k_cache.dtype == torch.uint8 else k_cache.dtype
    if k_new.dtype != want or v_new.dtype != want or v_cache.dtype != k_cache.dtype:
        raise TypeError(f"kv_append: new rows must be {want} for a {k_cache.dtype} cache")
    B, T, Hkv, D = k_new.shape
    shape = PaShape(B, T, Hkv, Hkv, D, k_cache.shape[1], k_cache.shape[0], block_tables.shape[1])
    args = [_ptr(k_new), _ptr(v_new), _ptr(block_tables), _ptr(context_lens), ctypes.byref(shape),
            _ptr(k_cache), _ptr(v_cache)]
    if k_cache.dtype == torch.uint8:
        st = lib().pa_kv_append_fp8(*args, _ptr(k_scale), _ptr(v_scale), _stream(stream))
        _check(st, "pa_kv_append_fp8")
    else:
        st = lib().pa_kv_append(*args, _stream(stream))
        _check(st, "pa_kv_append")


def split_workspace_views(workspace: torch.Tensor, B: int, T: int, Hq: int, S: int, D: int):
    """part_out [B,T,Hq,S,D] and part_lse [B,T,Hq,S] inside an explicit-split workspace."""
    rows = B * T * Hq * S
    off = (rows * D * 4 + 255) // 256 * 256
    flat = workspace.view(torch.uint8)
    part_out = flat[: rows * D * 4].view(torch.float32).view(B, T, Hq, S, D)
    part_lse = flat[off: off + rows * 4].view(torch.float32).view(B, T, Hq, S)
    return part_out, part_lse


def decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                   context_lens: torch.Tensor, scale: float, *, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, num_splits: int = 0, stream=None):
    """pa_decode_noalloc: bf16 paged decode whose split-K scratch is the
    library's static device array (no workspace argument)."""
    _need_contig(q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables, context_lens=context_lens,
                 out=out, lse=lse)
    shape = make_shape(q, k_cache, block_tables)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    st = lib().pa_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
                                 ctypes.byref(shape), float(scale), _ptr(out), _ptr(lse), int(num_splits),
                                 _stream(stream))
    _check(st, "pa_decode_noalloc")
    return out, lse


def decode_reduce(part_out: torch.Tensor, part_lse: torch.Tensor, *, out: Optional[torch.Tensor] = None,
                  lse: Optional[torch.Tensor] = None, stream=None, out_dtype=torch.bfloat16):
    """pa_decode_reduce (bf16 out) or pa_decode_reduce_f16 (out_dtype
    torch.float16): combine part_out [B,T,Hq,S,D] by part_lse [B,T,Hq,S]."""
    _need_contig(part_out=part_out, part_lse=part_lse)
    B, T, Hq, S, D = part_out.shape
    shape = PaShape(B, T, Hq, 1, D, 16, 1, 1)
    if out is None:
        out = torch.empty((B, T, Hq, D), dtype=out_dtype, device=part_out.device)
    if lse is None:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=part_out.device)
    if out.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("out must be bf16 or f16")
    name = "pa_decode_reduce_f16" if out.dtype == torch.float16 else "pa_decode_reduce"
    st = getattr(lib(), name)(_ptr(part_out), _ptr(part_lse), S, ctypes.byref(shape), _ptr(out), _ptr(lse),
                              _stream(stream))
    _check(st, name)
    return out, lse


def arm_profile_events(start_event, split_done_event) -> None:
    """Record the two torch.cuda.Event objects around the split kernel of the
    calling thread's next decode call (see pa_decode_profile_events)."""
    _check(lib().pa_decode_profile_events(start_event.cuda_event, split_done_event.cuda_event),
           "pa_decode_profile_events")


def device_error() -> int:
    """Reads and clears the kernels' error flags on the current device (synchronous)."""
    v = ctypes.c_int32(0)
    _check(lib().pa_decode_device_error(ctypes.byref(v)), "pa_decode_device_error")
    return int(v.value)


# Decode kernels: automatic, the warp-level MMA kernel, the token-major
# tcgen05 kernel, the query-row-major tcgen05 kernel (16-bit, 64-row units).
KERNEL_AUTO, KERNEL_WARP_MMA, KERNEL_TCGEN05, KERNEL_TCGEN05_QROW, KERNEL_WARP_PAIR = 0, 1, 2, 3, 4
_FORMATS = {"bf16": 0, "fp8": 1, "f16": 2, "draft": 3}


def set_kernel_path(path: int) -> None:
    """Process-wide kernel choice: KERNEL_AUTO, KERNEL_WARP_MMA, KERNEL_TCGEN05,
    KERNEL_TCGEN05_QROW or KERNEL_WARP_PAIR (see pa_decode_set_kernel_path)."""
    _check(lib().pa_decode_set_kernel_path(int(path)), "pa_decode_set_kernel_path")


COMBINE_SEPARATE, COMBINE_FUSED = 0, 1


def set_combine(mode: int) -> None:
    """Process-wide split-K combine of the balanced schedule: COMBINE_SEPARATE
    or COMBINE_FUSED (see pa_decode_set_combine)."""
    _check(lib().pa_decode_set_combine(int(mode)), "pa_decode_set_combine")


def kernel_for(shape: PaShape, fmt: str) -> int:
    """The kernel (KERNEL_WARP_MMA, KERNEL_TCGEN05, KERNEL_TCGEN05_QROW or KERNEL_WARP_PAIR) a
    decode of this shape and format ('bf16', 'fp8', 'f16', 'draft') runs;
    -1 if unsupported."""
    return int(lib().pa_decode_kernel_for(ctypes.byref(shape), _FORMATS[fmt]))


def kernel_for_inputs(inp) -> int:
    """kernel_for() of a DecodeInputs bundle."""
    s = inp.spec
    fmt = "draft" if s.draft_scratch else s.kv_format
    return kernel_for(make_shape(inp.q, inp.k_cache, inp.block_tables), fmt)


def heads_per_unit(shape: PaShape, fmt: str) -> int:
    """kv heads per work unit of a decode of this shape and format ('bf16',
    'fp8', 'f16', 'draft'); -1 if unsupported."""
    return int(lib().pa_decode_heads_per_unit(ctypes.byref(shape), _FORMATS[fmt]))


def heads_per_unit_inputs(inp) -> int:
    """heads_per_unit() of a DecodeInputs bundle."""
    s = inp.spec
    fmt = "draft" if s.draft_scratch else s.kv_format
    return heads_per_unit(make_shape(inp.q, inp.k_cache, inp.block_tables), fmt)
