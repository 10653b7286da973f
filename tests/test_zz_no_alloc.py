"""pa_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (they get only input and output pointers, or must
not call cudaMalloc on their path). Its split-K scratch is a static array of
the library, so its results must equal pa_decode's with a caller workspace,
call after call, although the array keeps the previous call's contents.

This file is collected last on purpose: if it fails, a run that stops at
the first failure has already run every other test."""

import ctypes

import numpy as np
import pytest
import torch

from paged_kv_attention_15_gb300 import binding as pb
from paged_kv_attention_15_gb300 import inputs as gen

TOL = 1e-2  # bf16 output tolerance used by the parity tests
LSE_TOL = 1e-3


def _spec(seed, **kw):
    base = dict(batch=12, q_tokens=1, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                ctx_range=(1, 3000), max_blocks_per_seq=3000 // 16 + 1, seed=seed)
    base.update(kw)
    return gen.custom_spec(**base)


def _close(a, b, tol):
    a = a.float().cpu().double().numpy()
    b = b.float().cpu().double().numpy()
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin)
    assert np.all(np.abs(a[fin] - b[fin]) <= tol + tol * np.abs(b[fin]))


@pytest.mark.gpu
@pytest.mark.parametrize("num_splits", [0, 3])
def test_noalloc_matches_pa_decode_on_consecutive_calls(num_splits):
    torch.cuda.set_device(0)
    for seed in (31, 32):  # two calls in a row; the scratch keeps the first call's partials
        dev = gen.make_inputs(_spec(seed)).to("cuda")
        ref_out, ref_lse = pb.decode_inputs(dev, num_splits=num_splits)
        out, lse = pb.decode_noalloc(dev.q, dev.k_cache, dev.v_cache, dev.block_tables, dev.context_lens,
                                     dev.scale, num_splits=num_splits)
        torch.cuda.synchronize()
        assert pb.device_error() == 0
        _close(out, ref_out, TOL)
        _close(lse, ref_lse, LSE_TOL)


@pytest.mark.gpu
def test_noalloc_rejects_partials_beyond_the_static_scratch():
    torch.cuda.set_device(0)
    # 64 sequences x 32 heads x 1024 splits x 129 floats: far above the limit.
    # Real buffers of the declared shape (zero lengths, valid page ids), so
    # that even a call that wrongly went ahead would only compute.
    B, T, Hq, Hkv, D, P, pages = 64, 1, 32, 8, 128, 16, 1024
    shape = pb.PaShape(B, T, Hq, Hkv, D, P, pages, pages)
    assert pb.workspace_size(shape, 1024) > (8 << 20)
    q = torch.zeros(B, T, Hq, D, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(pages, P, Hkv, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    bt = torch.zeros(B, pages, dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 7.0)
    st = pb.lib().pa_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), lens.data_ptr(),
                                    ctypes.byref(shape), 0.1, out.data_ptr(), None, 1024, None)
    assert st == pb.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a rejected call must leave out untouched"
