"""The query-row-major tcgen05 kernel (M = 64 query rows, scores and output
in tensor memory, K and V read by the tensor cores where the copies landed)
against the fp64 oracle, through the C ABI.

Every case forces that kernel (pa_decode_set_kernel_path(3)) and checks that
the library reports it for the shape, so a silent fall-back to another
kernel cannot pass. The bar is the one of test_gpu_parity.py:
|gpu - oracle| <= 1e-2 + 1e-2 |oracle| on out and |lse_gpu - lse_oracle| <=
1e-3.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_15_gb300 import binding as pb
from paged_kv_attention_15_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(autouse=True)
def qrow_path():
    pb.set_kernel_path(pb.KERNEL_TCGEN05_QROW)
    yield
    pb.set_kernel_path(pb.KERNEL_AUTO)


def ora(inp):
    oi = oracle.as_oracle_inputs(inp.numpy_bits(), inp.spec.kv_format)
    if inp.spec.draft_block is not None:
        oi["draft_block"] = inp.spec.draft_block
    return oi


def run(inp, num_splits, dev=None):
    dev = dev if dev is not None else inp.to("cuda")
    assert pb.kernel_for_inputs(dev) == pb.KERNEL_TCGEN05_QROW, "shape not on the query-row tcgen05 kernel"
    out, lse = pb.decode_inputs(dev, num_splits=num_splits)
    torch.cuda.synchronize()
    assert pb.device_error() == 0
    return out.float().cpu().double().numpy(), lse.cpu().double().numpy()


def check(out, lse, ref_out, ref_lse, rows=None):
    if rows is not None:
        idx = tuple(np.array(rows).T)
        out, lse, ref_out, ref_lse = out[idx], lse[idx], ref_out[idx], ref_lse[idx]
    assert np.all(np.isfinite(out)), "non-finite output"
    excess = np.abs(out - ref_out) - (TOL + TOL * np.abs(ref_out))
    assert excess.max() <= 0, f"out: max excess {excess.max():.3g}, max abs err {np.abs(out - ref_out).max():.3g}"
    inf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), inf), "lse -inf pattern differs"
    d = np.abs(lse[~inf] - ref_lse[~inf])
    assert d.size == 0 or d.max() <= LSE_TOL, f"lse: {d.max():.3g}"


def full(inp, num_splits):
    ref_out, ref_lse = oracle.decode(ora(inp), inp.scale)
    check(*run(inp, num_splits), ref_out, ref_lse)


def spec(**kw):
    # the TiDAR geometry: 8 draft tokens x 4 query heads = 32 rows per kv head
    base = dict(batch=4, q_tokens=8, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                context_lens=(1, 100, 16, 333), kv_format="bf16", draft_scratch=True, seed=43)
    base.update(kw)
    return gen.custom_spec(**base)


CASES = [
    dict(),                                                              # draft block, two kv heads per unit
    dict(draft_block=1),                                                 # causal draft
    dict(draft_block=3, context_lens=(0, 17, 64, 200)),                  # block-masked draft, empty prefix
    dict(context_lens=(15, 16, 17, 33)),                                 # partial last pages
    dict(page_size=32, context_lens=(31, 32, 65, 300)),                  # one 32-row box per stage
    dict(page_size=64, context_lens=(64, 1, 700, 65)),                   # stages inside one page
    dict(num_q_heads=16, num_kv_heads=4, batch=3, context_lens=(5, 400, 77)),  # two head groups
    dict(q_tokens=16, num_q_heads=8, num_kv_heads=2, draft_block=4),     # 64 rows per kv head, one head per unit
    dict(q_tokens=16, num_q_heads=8, num_kv_heads=2, draft_block=4, page_size=64,
         context_lens=(64, 129, 3, 500)),
    dict(q_tokens=4, num_q_heads=16, num_kv_heads=2),                    # 4 draft tokens x 8 heads
    dict(draft_scratch=False, q_tokens=1, num_q_heads=64, num_kv_heads=2),  # no draft: G = 32
    dict(draft_scratch=False, q_tokens=1, num_q_heads=64, num_kv_heads=1,
         context_lens=(0, 1000, 64, 63)),                                # G = 64, an empty sequence
    dict(draft_scratch=False, q_tokens=1, num_q_heads=64, num_kv_heads=2, kv_format="f16"),
    dict(draft_scratch=False, q_tokens=2, num_q_heads=32, num_kv_heads=2, kv_format="f16",
         page_size=32),
    dict(batch=9, ctx_range=(1, 2000), context_lens=None, pool_pages=1400),
    # 128-row units: four kv heads of 32 rows, one 16-token page box per stage
    dict(num_q_heads=16, num_kv_heads=4, context_lens=(15, 16, 17, 333)),
    dict(num_q_heads=32, num_kv_heads=8, draft_block=1, context_lens=(0, 100, 31, 700)),
    dict(num_q_heads=16, num_kv_heads=4, draft_block=3, page_size=32, context_lens=(33, 64, 1, 300)),
    dict(num_q_heads=16, num_kv_heads=4, page_size=64, context_lens=(64, 65, 129, 2)),
    dict(q_tokens=4, num_q_heads=32, num_kv_heads=4),                    # 4 draft tokens x 8 heads
    dict(draft_scratch=False, q_tokens=1, num_q_heads=128, num_kv_heads=4, context_lens=(0, 9, 400, 1000)),
    dict(draft_scratch=False, q_tokens=2, num_q_heads=64, num_kv_heads=4, kv_format="f16"),
    dict(batch=7, num_q_heads=32, num_kv_heads=8, ctx_range=(1, 1500), context_lens=None, pool_pages=800),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_qrow(case, num_splits):
    full(gen.make_inputs(spec(**case)), num_splits)


@pytest.mark.parametrize("q_scale", [4.0, 16.0])
def test_spread_scores_rescale_the_output(q_scale):
    """Scores spread over many log2 units: running maxima move past the
    slack in later stages, so the output in tensor memory is rescaled."""
    inp = gen.make_inputs(spec(context_lens=(700, 33, 1, 260)))
    q = (inp.q.float() * q_scale).to(inp.q.dtype)
    full(dataclasses.replace(inp, q=q), 0)
    full(dataclasses.replace(inp, q=q), 3)


def test_nan_poison_past_the_context():
    """Cache slots past every context end hold NaN: their scores are masked
    and their value rows are zeroed before the product reads them."""
    for kw in (dict(), dict(q_tokens=16, draft_block=4), dict(draft_scratch=False, q_tokens=1, num_q_heads=64),
               dict(num_q_heads=16, num_kv_heads=4)):
        inp = gen.make_inputs(spec(context_lens=(5, 17, 64, 99), **kw), poison=True)
        full(inp, 0)
        full(inp, 3)


def test_page_relabelling_is_bit_exact():
    inp = gen.make_inputs(spec(context_lens=(300, 17, 64, 900)))
    a = run(inp, 0)
    n = inp.k_cache.shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(5))
    inv = torch.argsort(perm)
    relab = dataclasses.replace(inp, k_cache=inp.k_cache[inv], v_cache=inp.v_cache[inv],
                                block_tables=torch.where(inp.block_tables >= 0, perm[inp.block_tables.long()].int(),
                                                         inp.block_tables))
    b = run(relab, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_matches_the_warp_mma_kernel():
    """The query-row kernel and the warp-level kernel agree within rounding."""
    for case in (dict(), dict(q_tokens=16, draft_block=4), dict(draft_scratch=False, q_tokens=1, num_q_heads=64),
                 dict(num_q_heads=32, num_kv_heads=8)):
        inp = gen.make_inputs(spec(**case))
        dev = inp.to("cuda")
        a = run(inp, 0, dev=dev)
        pb.set_kernel_path(pb.KERNEL_WARP_MMA)
        assert pb.kernel_for_inputs(dev) == pb.KERNEL_WARP_MMA
        out, lse = pb.decode_inputs(dev, num_splits=0)
        torch.cuda.synchronize()
        pb.set_kernel_path(pb.KERNEL_TCGEN05_QROW)
        b = (out.float().cpu().double().numpy(), lse.cpu().double().numpy())
        assert np.abs(a[0] - b[0]).max() <= 2 * TOL and np.abs(a[1] - b[1]).max() <= LSE_TOL


@pytest.mark.parametrize("name", ["tidar", "tidar_causal", "tidar_long"])
def test_full_size_workload(name):
    """The full-size draft workloads on the query-row kernel: every row of
    the TiDAR workload, sampled rows of the other two."""
    inp = gen.make_inputs(gen.SPECS[name])
    out, lse = run(inp, 0)
    rows = None
    if name != "tidar":
        rng = np.random.default_rng(11)
        s = inp.spec
        rows = sorted({(int(rng.integers(s.batch)), int(rng.integers(s.q_tokens)), int(rng.integers(s.num_q_heads)))
                       for _ in range(64)})
    ref_out, ref_lse = oracle.decode(ora(inp), inp.scale, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows)


def test_graph_capture_replays_like_eager():
    common = dict(batch=6, ctx_range=(1, 900), context_lens=None, pool_pages=500, max_blocks_per_seq=57)
    inp = gen.make_inputs(spec(**common))
    other = gen.make_inputs(spec(**common, seed=99))
    dev = inp.to("cuda")
    assert pb.kernel_for_inputs(dev) == pb.KERNEL_TCGEN05_QROW
    shp = pb.make_shape(dev.q, dev.k_cache, dev.block_tables)
    ws = torch.empty(pb.workspace_size(shp, 0), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev.q)
    lse = torch.empty(dev.q.shape[:3], dtype=torch.float32, device="cuda")
    pb.decode_inputs(dev, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pb.decode_inputs(dev, out=out, lse=lse, workspace=ws)
    for name, t in other.tensors().items():
        getattr(dev, name).copy_(t)
    g.replay()
    torch.cuda.synchronize()
    eager = pb.decode_inputs(other.to("cuda"), num_splits=0)
    torch.cuda.synchronize()
    assert torch.equal(out, eager[0]) and torch.equal(lse, eager[1])


def test_workspace_sized_under_the_default_selection_fits():
    """pa_decode_workspace_size(shape, 0) is the largest plan over every
    kernel selection: a workspace sized while the automatic choice is set
    serves a call on this kernel."""
    inp = gen.make_inputs(spec(**dict(batch=6, ctx_range=(1, 900), context_lens=None, pool_pages=500, max_blocks_per_seq=57)))
    dev = inp.to("cuda")
    shp = pb.make_shape(dev.q, dev.k_cache, dev.block_tables)
    pb.set_kernel_path(pb.KERNEL_AUTO)
    size = pb.workspace_size(shp, 0)
    pb.set_kernel_path(pb.KERNEL_TCGEN05_QROW)
    assert pb.kernel_for_inputs(dev) == pb.KERNEL_TCGEN05_QROW
    assert pb.workspace_size(shp, 0) == size
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    ref_out, ref_lse = oracle.decode(ora(inp), inp.scale)
    out, lse = pb.decode_inputs(dev, workspace=ws)
    torch.cuda.synchronize()
    assert pb.device_error() == 0
    check(out.float().cpu().double().numpy(), lse.cpu().double().numpy(), ref_out, ref_lse)
