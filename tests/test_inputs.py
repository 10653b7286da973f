"""The seeded generator: shapes, structure and determinism of the workloads."""

import numpy as np
import torch

from paged_kv_attention_15_gb300 import inputs as gen


def test_tiny_workload_structure():
    inp = gen.make_inputs(gen.SPECS["tiny"])
    assert tuple(inp.q.shape) == (2, 1, 4, 64) and inp.q.dtype == torch.bfloat16
    assert tuple(inp.k_cache.shape) == (16, 16, 1, 64)
    assert inp.context_lens.tolist() == [37, 100]
    bt = inp.block_tables.numpy()
    assert bt.shape == (2, 7)
    used = np.concatenate([bt[0, :3], bt[1, :7]])
    assert len(set(used.tolist())) == 10 and used.min() >= 0 and used.max() < 16
    assert np.all(bt[0, 3:] == -1)


def test_deterministic_and_thread_independent(monkeypatch):
    spec = gen.custom_spec(batch=4, q_tokens=1, num_q_heads=4, num_kv_heads=2, head_dim=64,
                           page_size=16, ctx_range=(1, 300), seed=7)
    a = gen.make_inputs(spec)
    monkeypatch.setattr(gen, "_threads", lambda: 1)
    b = gen.make_inputs(spec)

    def raw(t):
        return t.view(torch.int16) if t.dtype == torch.bfloat16 else t

    for n, t in a.tensors().items():
        assert torch.equal(raw(t), raw(b.tensors()[n])), n


def test_context_ranges_and_page_pool():
    for name in ("gqa", "fp8", "tidar"):
        spec = gen.SPECS[name]
        lens = gen.draw_context_lens(spec)
        lo, hi = spec.ctx_range
        assert lens.shape == (spec.batch,) and lens.min() >= lo and lens.max() <= hi
        assert spec.max_blocks_per_seq * spec.page_size >= hi


def test_fp8_codes_and_scales():
    spec = gen.custom_spec(batch=2, q_tokens=1, num_q_heads=4, num_kv_heads=2, head_dim=64,
                           page_size=16, context_lens=(20, 40), kv_format="fp8", seed=3)
    inp = gen.make_inputs(spec)
    assert inp.k_cache.dtype == torch.uint8 and inp.k_scale.dtype == torch.float32
    vals = inp.k_cache.view(torch.float8_e4m3fn).float()
    assert torch.isfinite(vals).all()
    # Every (page, slot, head) vector reaches +-448 somewhere (symmetric amax scale).
    assert torch.all(vals.abs().amax(-1) == 448.0)


def test_poison_marks_only_unread_values():
    spec = gen.custom_spec(batch=2, q_tokens=1, num_q_heads=2, num_kv_heads=1, head_dim=32,
                           page_size=16, context_lens=(20, 16), pool_pages=6, seed=1)
    inp = gen.make_inputs(spec, poison=True)
    bt = inp.block_tables
    assert bt[0, 2:].eq(2**31 - 1).all() and bt[1, 1:].eq(2**31 - 1).all()
    last = int(bt[0, 1])
    assert torch.isnan(inp.k_cache[last, 4:].float()).all()
    assert not torch.isnan(inp.k_cache[last, :4].float()).any()
    used = {int(bt[0, 0]), int(bt[0, 1]), int(bt[1, 0])}
    for p in range(6):
        assert torch.isnan(inp.v_cache[p].float()).any() == (p not in used or p == last)
