"""The tcgen05 split kernel (token-major MMAs, scores and output in tensor
memory) against the fp64 oracle, through the C ABI.

Every case forces the tcgen05 path (pa_decode_set_kernel_path(2)) and
checks that the library reports that kernel for the shape, so a silent
fall-back to the warp-level kernel cannot pass. The bar is the one of
test_gpu_parity.py: |gpu - oracle| <= tol + tol |oracle| on out (tol 1e-2
for 16-bit caches, 2e-2 for fp8) and |lse_gpu - lse_oracle| <= 1e-3.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_15_gb300 import binding as pb
from paged_kv_attention_15_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

LSE_TOL = 1e-3


@pytest.fixture(autouse=True)
def tcgen05_path():
    pb.set_kernel_path(pb.KERNEL_TCGEN05)
    yield
    pb.set_kernel_path(pb.KERNEL_AUTO)


def tol_of(spec):
    return 2e-2 if spec.kv_format == "fp8" else 1e-2


def ora(inp):
    oi = oracle.as_oracle_inputs(inp.numpy_bits(), inp.spec.kv_format)
    if inp.spec.draft_block is not None:
        oi["draft_block"] = inp.spec.draft_block
    return oi


def run(inp, num_splits, dev=None):
    dev = dev if dev is not None else inp.to("cuda")
    assert pb.kernel_for_inputs(dev) == pb.KERNEL_TCGEN05, "shape not on the tcgen05 kernel"
    out, lse = pb.decode_inputs(dev, num_splits=num_splits)
    torch.cuda.synchronize()
    assert pb.device_error() == 0
    return out.float().cpu().double().numpy(), lse.cpu().double().numpy()


def check(out, lse, ref_out, ref_lse, tol, rows=None):
    if rows is not None:
        idx = tuple(np.array(rows).T)
        out, lse, ref_out, ref_lse = out[idx], lse[idx], ref_out[idx], ref_lse[idx]
    assert np.all(np.isfinite(out)), "non-finite output"
    excess = np.abs(out - ref_out) - (tol + tol * np.abs(ref_out))
    assert excess.max() <= 0, f"out: max excess {excess.max():.3g}, max abs err {np.abs(out - ref_out).max():.3g}"
    inf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), inf), "lse -inf pattern differs"
    d = np.abs(lse[~inf] - ref_lse[~inf])
    assert d.size == 0 or d.max() <= LSE_TOL, f"lse: {d.max():.3g}"


def full(inp, num_splits):
    ref_out, ref_lse = oracle.decode(ora(inp), inp.scale)
    check(*run(inp, num_splits), ref_out, ref_lse, tol_of(inp.spec))


def spec(**kw):
    base = dict(batch=4, q_tokens=1, num_q_heads=32, num_kv_heads=2, head_dim=256, page_size=16,
                context_lens=(1, 100, 16, 333), kv_format="fp8", seed=41)
    base.update(kw)
    return gen.custom_spec(**base)


# ------------------------------------------------------------------ fp8
FP8_CASES = [
    dict(),                                                         # the fp8 workload's geometry, ragged
    dict(context_lens=(64, 65, 128, 1000)),                         # stage boundaries (64 tokens)
    dict(head_dim=128, num_q_heads=16, num_kv_heads=1),             # D 128, one head per unit
    dict(head_dim=128, num_q_heads=64, num_kv_heads=4),             # D 128, four heads per unit
    dict(num_q_heads=16, num_kv_heads=1, context_lens=(0, 5, 700, 31)),  # empty sequence
    dict(page_size=32, context_lens=(33, 64, 200, 7)),
    dict(page_size=64, context_lens=(64, 1, 700, 65)),
    dict(page_size=128, context_lens=(300, 127, 128, 129)),          # one page holds more than a stage
    dict(page_size=256, context_lens=(600, 255, 1, 257)),
    dict(q_tokens=2, num_q_heads=16, num_kv_heads=2),                # G 8 x T 2 = 16 rows
    dict(num_q_heads=64, num_kv_heads=2),                            # 32 rows per kv head
    dict(batch=9, ctx_range=(1, 2000), context_lens=None, pool_pages=1200),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=[str(i) for i in range(len(FP8_CASES))])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_fp8(case, num_splits):
    full(gen.make_inputs(spec(**case)), num_splits)


# -------------------------------------------------------------- 16-bit
B16_CASES = [
    dict(kv_format="bf16", head_dim=128, num_q_heads=32, num_kv_heads=2),                 # G 16
    dict(kv_format="bf16", head_dim=128, num_q_heads=32, num_kv_heads=1),                 # G 32
    dict(kv_format="f16", head_dim=128, num_q_heads=32, num_kv_heads=2),
    dict(kv_format="bf16", head_dim=128, num_q_heads=64, num_kv_heads=4, page_size=64,
         context_lens=(64, 65, 900, 0)),
    dict(kv_format="bf16", head_dim=128, q_tokens=8, num_q_heads=8, num_kv_heads=2,
         draft_scratch=True),                                                              # draft block, 32 rows
    dict(kv_format="bf16", head_dim=128, q_tokens=8, num_q_heads=8, num_kv_heads=2,
         draft_scratch=True, draft_block=1),                                               # causal draft
    dict(kv_format="bf16", head_dim=128, q_tokens=8, num_q_heads=8, num_kv_heads=2,
         draft_scratch=True, draft_block=3, context_lens=(0, 17, 64, 200)),               # block-masked, empty prefix
    dict(kv_format="bf16", head_dim=128, q_tokens=4, num_q_heads=16, num_kv_heads=4,
         draft_scratch=True, page_size=32),                                                # 16 rows, 4 heads per unit
]


@pytest.mark.parametrize("case", B16_CASES, ids=[str(i) for i in range(len(B16_CASES))])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_16bit(case, num_splits):
    full(gen.make_inputs(spec(**case)), num_splits)


@pytest.mark.parametrize("q_scale", [4.0, 16.0])
@pytest.mark.parametrize("kv_format", ["bf16", "fp8"])
def test_spread_scores_rescale_the_output(kv_format, q_scale):
    """Scores spread over many log2 units: running maxima move past the
    slack in later stages, so the output in tensor memory is rescaled."""
    D = 128
    inp = gen.make_inputs(spec(kv_format=kv_format, head_dim=D, num_q_heads=16, num_kv_heads=1,
                               context_lens=(700, 33, 1, 260)))
    q = (inp.q.float() * q_scale).to(inp.q.dtype)
    full(dataclasses.replace(inp, q=q), 0)
    full(dataclasses.replace(inp, q=q), 3)


def test_nan_poison_past_the_context():
    """Cache slots past every context end hold NaN (fp8: the NaN code):
    they are never keys, and the zeroed value rows keep the products finite."""
    for fmt in ("fp8", "bf16"):
        inp = gen.make_inputs(spec(kv_format=fmt, head_dim=128, num_q_heads=32, num_kv_heads=2,
                                   context_lens=(5, 17, 64, 99)), poison=True)
        full(inp, 0)


def test_page_relabelling_is_bit_exact():
    inp = gen.make_inputs(spec())
    a = run(inp, 0)
    n = inp.k_cache.shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(5))
    inv = torch.argsort(perm)
    relab = dataclasses.replace(inp, k_cache=inp.k_cache[inv], v_cache=inp.v_cache[inv],
                                k_scale=inp.k_scale[inv], v_scale=inp.v_scale[inv],
                                block_tables=torch.where(inp.block_tables >= 0, perm[inp.block_tables.long()].int(),
                                                         inp.block_tables))
    b = run(relab, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_matches_the_warp_mma_kernel():
    """The two split kernels agree within rounding on the same inputs."""
    for case in (dict(), dict(kv_format="bf16", head_dim=128, q_tokens=8, num_q_heads=8, num_kv_heads=2,
                              draft_scratch=True)):
        inp = gen.make_inputs(spec(**case))
        dev = inp.to("cuda")
        a = run(inp, 0, dev=dev)
        pb.set_kernel_path(pb.KERNEL_WARP_MMA)
        assert pb.kernel_for_inputs(dev) == pb.KERNEL_WARP_MMA
        out, lse = pb.decode_inputs(dev, num_splits=0)
        torch.cuda.synchronize()
        pb.set_kernel_path(pb.KERNEL_TCGEN05)
        b = (out.float().cpu().double().numpy(), lse.cpu().double().numpy())
        tol = 2 * tol_of(inp.spec)
        assert np.abs(a[0] - b[0]).max() <= tol and np.abs(a[1] - b[1]).max() <= LSE_TOL


@pytest.mark.parametrize("name", ["fp8", "tidar", "tidar_causal"])
def test_full_size_workload(name):
    """The full-size workloads on the tcgen05 kernel, every row (fp8,
    tidar) or sampled rows (the causal draft)."""
    inp = gen.make_inputs(gen.SPECS[name])
    out, lse = run(inp, 0)
    rows = None
    if name == "tidar_causal":
        rng = np.random.default_rng(7)
        s = inp.spec
        rows = sorted({(int(rng.integers(s.batch)), int(rng.integers(s.q_tokens)), int(rng.integers(s.num_q_heads)))
                       for _ in range(64)})
    ref_out, ref_lse = oracle.decode(ora(inp), inp.scale, rows=rows)
    check(out, lse, ref_out, ref_lse, tol_of(inp.spec), rows=rows)


def test_graph_capture_replays_like_eager():
    common = dict(batch=6, ctx_range=(1, 900), context_lens=None, pool_pages=500, max_blocks_per_seq=57)
    inp = gen.make_inputs(spec(**common))
    other = gen.make_inputs(spec(**common, seed=99))
    dev = inp.to("cuda")
    assert pb.kernel_for_inputs(dev) == pb.KERNEL_TCGEN05
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
    pb.set_kernel_path(pb.KERNEL_TCGEN05)
    assert pb.kernel_for_inputs(dev) == pb.KERNEL_TCGEN05
    assert pb.workspace_size(shp, 0) == size
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    ref_out, ref_lse = oracle.decode(ora(inp), inp.scale)
    out, lse = pb.decode_inputs(dev, workspace=ws)
    torch.cuda.synchronize()
    assert pb.device_error() == 0
    check(out.float().cpu().double().numpy(), lse.cpu().double().numpy(), ref_out, ref_lse, tol_of(inp.spec))
