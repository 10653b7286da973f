"""The split-K combine fused into the warp-level split kernel
(pa_decode_set_combine(1)): the last CTA to finish a piece of a (sequence,
kv head group) unit combines the unit's pieces. Compared, through the C ABI,
with the fp64 oracle at the tolerance of test_gpu_parity.py, and with the
separate combine kernel. The single-token 16-bit shapes run the fused path
(D 64, 128, 256, f16, units over one to about a hundred CTAs, empty CTA
shares); fp8 and the draft-block shapes on the eight-warp instances keep the
separate combine in this mode and are checked as well."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_15_gb300 import binding as pb
from paged_kv_attention_15_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

LSE_TOL = 1e-3


@pytest.fixture(autouse=True)
def fused_combine():
    pb.set_combine(pb.COMBINE_FUSED)
    yield
    pb.set_combine(pb.COMBINE_SEPARATE)


def tol_of(s):
    return 2e-2 if s.kv_format == "fp8" else 1e-2


def ora(inp):
    oi = oracle.as_oracle_inputs(inp.numpy_bits(), inp.spec.kv_format)
    if inp.spec.draft_block is not None:
        oi["draft_block"] = inp.spec.draft_block
    return oi


def run(inp, dev=None):
    dev = dev if dev is not None else inp.to("cuda")
    assert pb.kernel_for_inputs(dev) in (pb.KERNEL_WARP_MMA, pb.KERNEL_WARP_PAIR)  # (fp8: the paired-role kernel)
    out, lse = pb.decode_inputs(dev, num_splits=0)
    torch.cuda.synchronize()
    assert pb.device_error() == 0
    return out.float().cpu().double().numpy(), lse.cpu().double().numpy()


def check(out, lse, ref_out, ref_lse, tol, rows=None):
    if rows is not None:
        idx = tuple(np.array(rows).T)
        out, lse, ref_out, ref_lse = out[idx], lse[idx], ref_out[idx], ref_lse[idx]
    assert np.all(np.isfinite(out)), "non-finite output"
    excess = np.abs(out - ref_out) - (tol + tol * np.abs(ref_out))
    assert excess.max() <= 0, f"out: max excess {excess.max():.3g}"
    inf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), inf), "lse -inf pattern differs"
    d = np.abs(lse[~inf] - ref_lse[~inf])
    assert d.size == 0 or d.max() <= LSE_TOL, f"lse: {d.max():.3g}"


def spec(**kw):
    base = dict(batch=4, q_tokens=1, num_q_heads=16, num_kv_heads=4, head_dim=128, page_size=16,
                context_lens=(1, 100, 16, 333), seed=51)
    base.update(kw)
    return gen.custom_spec(**base)


CASES = [
    dict(),                                                          # fewer pages than CTAs: empty shares
    dict(batch=6, ctx_range=(500, 3000), context_lens=None, pool_pages=1200),   # units over 2-4 CTAs
    dict(batch=2, context_lens=(20000, 7), pool_pages=1300, max_blocks_per_seq=1250),  # one unit over ~100 CTAs
    dict(num_q_heads=32, num_kv_heads=2, head_dim=256, kv_format="fp8", batch=5, ctx_range=(300, 4000),
         context_lens=None, pool_pages=1400),      # fp8: the separate combine in either mode
    dict(kv_format="f16", batch=6, ctx_range=(200, 2500), context_lens=None, pool_pages=1000),
    dict(head_dim=64, batch=6, ctx_range=(200, 2500), context_lens=None, pool_pages=1000),
    dict(head_dim=256, batch=4, ctx_range=(500, 2500), context_lens=None, pool_pages=700),
    dict(q_tokens=8, num_q_heads=8, num_kv_heads=2, draft_scratch=True, batch=5, ctx_range=(100, 3000),
         context_lens=None, pool_pages=1000),
    dict(q_tokens=8, num_q_heads=8, num_kv_heads=2, draft_scratch=True, draft_block=2, batch=4,
         context_lens=(0, 700, 1500, 9), pool_pages=400),
    dict(q_tokens=16, num_q_heads=8, num_kv_heads=2, draft_scratch=True, draft_block=4, batch=3,
         context_lens=(2000, 33, 900), pool_pages=300),
    dict(num_q_heads=64, num_kv_heads=1, batch=3, context_lens=(0, 1000, 4000), pool_pages=400),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_fused_combine_matches_the_oracle(case):
    inp = gen.make_inputs(spec(**case))
    ref_out, ref_lse = oracle.decode(ora(inp), inp.scale)
    check(*run(inp), ref_out, ref_lse, tol_of(inp.spec))


def test_fused_equals_separate_combine_within_rounding():
    inp = gen.make_inputs(spec(batch=6, ctx_range=(500, 3000), context_lens=None, pool_pages=1200))
    dev = inp.to("cuda")
    a = run(inp, dev)
    pb.set_combine(pb.COMBINE_SEPARATE)
    b = run(inp, dev)
    pb.set_combine(pb.COMBINE_FUSED)
    assert np.abs(a[0] - b[0]).max() <= 1e-2 and np.abs(a[1] - b[1]).max() <= 1e-4


def test_counters_stay_usable_across_calls_and_graph_replay():
    """The memset and the counters' wrap-around keep calls independent: the
    same call twice, then a captured graph replayed on new inputs, equal
    eager calls."""
    common = dict(batch=6, ctx_range=(1, 2500), context_lens=None, pool_pages=1000, max_blocks_per_seq=157)
    inp = gen.make_inputs(spec(**common))
    other = gen.make_inputs(spec(**common, seed=77))
    dev = inp.to("cuda")
    shp = pb.make_shape(dev.q, dev.k_cache, dev.block_tables)
    ws = torch.empty(pb.workspace_size(shp, 0), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev.q)
    lse = torch.empty(dev.q.shape[:3], dtype=torch.float32, device="cuda")
    pb.decode_inputs(dev, out=out, lse=lse, workspace=ws)
    first = (out.clone(), lse.clone())
    pb.decode_inputs(dev, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, first[0]) and torch.equal(lse, first[1])
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pb.decode_inputs(dev, out=out, lse=lse, workspace=ws)
    for name, t in other.tensors().items():
        getattr(dev, name).copy_(t)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    eager = pb.decode_inputs(other.to("cuda"), num_splits=0)
    torch.cuda.synchronize()
    assert torch.equal(out, eager[0]) and torch.equal(lse, eager[1])
    ref_out, ref_lse = oracle.decode(ora(other), other.scale)
    check(out.float().cpu().double().numpy(), lse.cpu().double().numpy(), ref_out, ref_lse, 1e-2)


def test_full_size_workloads_on_sampled_rows():
    for name in ("gqa", "tidar"):
        inp = gen.make_inputs(gen.SPECS[name])
        out, lse = run(inp)
        rng = np.random.default_rng(3)
        s = inp.spec
        rows = sorted({(int(rng.integers(s.batch)), int(rng.integers(s.q_tokens)), int(rng.integers(s.num_q_heads)))
                       for _ in range(48)})
        ref_out, ref_lse = oracle.decode(ora(inp), inp.scale, rows=rows)
        check(out, lse, ref_out, ref_lse, 1e-2, rows=rows)
