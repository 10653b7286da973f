"""The split kernel with paired consumer roles (an S warp computing scores,
softmax and the P operand, two PV warps holding the output; messages through
shared memory) against the fp64 oracle, through the C ABI.

Every case forces that kernel (pa_decode_set_kernel_path(4)) and checks that
the library reports it for the shape, so a silent fall-back to another
kernel cannot pass. The bars are those of test_gpu_parity.py:
|gpu - oracle| <= tol + tol |oracle| on out, tol = 2e-2 for fp8 KV and 1e-2
for 16-bit KV, and |lse_gpu - lse_oracle| <= 1e-3.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_15_gb300 import binding as pb
from paged_kv_attention_15_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

TOL = 2e-2
LSE_TOL = 1e-3


@pytest.fixture(autouse=True)
def pair_path():
    pb.set_kernel_path(pb.KERNEL_WARP_PAIR)
    yield
    pb.set_kernel_path(pb.KERNEL_AUTO)


def ora(inp):
    return oracle.as_oracle_inputs(inp.numpy_bits(), inp.spec.kv_format)


def run(inp, num_splits, dev=None):
    dev = dev if dev is not None else inp.to("cuda")
    assert pb.kernel_for_inputs(dev) == pb.KERNEL_WARP_PAIR, "shape not on the paired-role kernel"
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
    base = dict(batch=4, q_tokens=1, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                context_lens=(1, 100, 16, 333), kv_format="fp8", seed=47)
    base.update(kw)
    return gen.custom_spec(**base)


CASES = [
    dict(),                                                              # G 4, two kv heads per unit
    dict(head_dim=256, num_q_heads=16, num_kv_heads=1),                  # one full row tile
    dict(head_dim=256, num_q_heads=32, num_kv_heads=2, page_size=64, context_lens=(64, 1, 700, 65)),
    dict(num_q_heads=24, num_kv_heads=1),                                # two row tiles
    dict(num_q_heads=16, num_kv_heads=8, context_lens=(0, 5, 900, 31)),  # empty sequence
    # the fp8 workload's geometry (two kv heads per unit, 32-token slices on alternate stages), ragged
    dict(head_dim=256, num_q_heads=32, num_kv_heads=2, context_lens=(1, 17, 33, 500)),
    dict(num_q_heads=16, num_kv_heads=16, context_lens=(3, 77, 300, 0)),  # more than 8 kv heads
    dict(head_dim=256, num_q_heads=24, num_kv_heads=12, page_size=32),
    dict(q_tokens=4, num_q_heads=8, num_kv_heads=2),                     # 16 rows of 4 tokens
    dict(q_tokens=3, num_q_heads=10, num_kv_heads=2, head_dim=256),      # 15 rows, odd group
    dict(page_size=128, context_lens=(300, 127, 128, 129)),
    dict(page_size=256, context_lens=(600, 255, 1, 257), head_dim=256, num_q_heads=32, num_kv_heads=2),
    dict(batch=9, ctx_range=(1, 2000), context_lens=None, pool_pages=1400, head_dim=256, num_q_heads=32,
         num_kv_heads=2),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_pair(case, num_splits):
    full(gen.make_inputs(spec(**case)), num_splits)


@pytest.mark.parametrize("q_scale", [4.0, 16.0])
def test_spread_scores_move_the_running_max(q_scale):
    """Scores spread over many log2 units: the S warp's running max moves in
    later stages and the PV warp rescales the output it holds."""
    inp = gen.make_inputs(spec(head_dim=256, num_q_heads=32, num_kv_heads=2, context_lens=(700, 33, 1, 260)))
    q = (inp.q.float() * q_scale).to(inp.q.dtype)
    full(dataclasses.replace(inp, q=q), 0)
    full(dataclasses.replace(inp, q=q), 3)


def test_unread_values_are_never_read():
    """NaN in unused pages, in slots past the context end and in their fp8
    scales change nothing."""
    for kw in (dict(), dict(head_dim=256, num_q_heads=32, num_kv_heads=2)):
        s = spec(context_lens=(5, 100, 33, 250), pool_pages=60, **kw)
        clean, dirty = gen.make_inputs(s), gen.make_inputs(s, poison=True)
        for ns in (0, 2):
            a = run(clean, ns)
            b = run(dirty, ns)
            assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        full(dirty, 0)


def test_page_relabelling_is_bit_exact():
    inp = gen.make_inputs(spec(head_dim=256, num_q_heads=32, num_kv_heads=2, context_lens=(300, 17, 64, 900)))
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


def test_matches_the_single_role_kernel():
    """Same slices and arithmetic as the single-role warp-level kernel except
    the running max, which may lag by the 16-bit paths' slack on stages with
    small value scales (the single-role fp8 kernel keeps the exact max): the
    two agree within rounding."""
    for case in (dict(), dict(head_dim=256, num_q_heads=32, num_kv_heads=2, context_lens=(1, 17, 333, 2000)),
                 dict(num_q_heads=24, num_kv_heads=1)):
        inp = gen.make_inputs(spec(**case))
        dev = inp.to("cuda")
        for ns in (0, 3):
            a = run(inp, ns, dev=dev)
            pb.set_kernel_path(pb.KERNEL_WARP_MMA)
            assert pb.kernel_for_inputs(dev) == pb.KERNEL_WARP_MMA
            out, lse = pb.decode_inputs(dev, num_splits=ns)
            torch.cuda.synchronize()
            pb.set_kernel_path(pb.KERNEL_WARP_PAIR)
            assert np.abs(a[0] - out.float().cpu().double().numpy()).max() <= 2e-2
            assert np.abs(a[1] - lse.cpu().double().numpy()).max() <= LSE_TOL


def test_full_size_fp8_workload():
    """Every output row of the full-size fp8 workload, in the launch
    configuration the benchmark times (num_splits = 0)."""
    inp = gen.make_inputs(gen.SPECS["fp8"])
    out, lse = run(inp, 0)
    ref_out, ref_lse = oracle.decode(ora(inp), inp.scale)
    check(out, lse, ref_out, ref_lse)


def draft_spec(**kw):
    # the TiDAR geometry: 8 draft tokens x 4 query heads = 32 rows per kv head
    base = dict(batch=4, q_tokens=8, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                context_lens=(1, 100, 16, 333), kv_format="bf16", draft_scratch=True, seed=53)
    base.update(kw)
    return gen.custom_spec(**base)


DRAFT_CASES = [
    dict(),                                                              # two kv heads of 32 rows per unit
    dict(draft_block=1),                                                 # causal draft
    dict(draft_block=3, context_lens=(0, 17, 64, 200)),                  # block-masked draft, empty prefix
    dict(context_lens=(15, 16, 17, 33)),                                 # partial last pages
    dict(page_size=32, context_lens=(31, 32, 65, 300)),
    dict(page_size=64, context_lens=(64, 1, 700, 65)),
    dict(num_q_heads=16, num_kv_heads=4, batch=3, context_lens=(5, 400, 77)),  # two head groups
    dict(q_tokens=16, num_q_heads=8, num_kv_heads=2, draft_block=4),     # 64 rows of one kv head, 64-token slices
    dict(q_tokens=16, num_q_heads=8, num_kv_heads=2, draft_block=4, page_size=64, context_lens=(64, 129, 3, 500)),
    dict(q_tokens=4, num_q_heads=16, num_kv_heads=2),                    # 4 draft tokens x 8 heads
    dict(draft_scratch=False, q_tokens=1, num_q_heads=64, num_kv_heads=2),  # no draft: G = 32
    dict(draft_scratch=False, q_tokens=1, num_q_heads=64, num_kv_heads=1, context_lens=(0, 1000, 64, 63)),
    dict(draft_scratch=False, q_tokens=1, num_q_heads=64, num_kv_heads=2, kv_format="f16"),
    dict(batch=9, ctx_range=(1, 2000), context_lens=None, pool_pages=1400),
]


def draft_full(inp, num_splits):
    oi = ora(inp)
    if inp.spec.draft_block is not None:
        oi["draft_block"] = inp.spec.draft_block
    ref_out, ref_lse = oracle.decode(oi, inp.scale)
    tol = 1e-2
    out, lse = run(inp, num_splits)
    assert np.all(np.isfinite(out)), "non-finite output"
    excess = np.abs(out - ref_out) - (tol + tol * np.abs(ref_out))
    assert excess.max() <= 0, f"out: max excess {excess.max():.3g}"
    inf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), inf), "lse -inf pattern differs"
    d = np.abs(lse[~inf] - ref_lse[~inf])
    assert d.size == 0 or d.max() <= LSE_TOL, f"lse: {d.max():.3g}"


@pytest.mark.parametrize("case", DRAFT_CASES, ids=[str(i) for i in range(len(DRAFT_CASES))])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_pair_16bit_draft_geometry(case, num_splits):
    """16-bit caches on the paired-role kernel: units of 64 query rows (four
    row tiles, one pair each), slices of the whole stage (32 or 64 tokens),
    draft-block scratch and masks."""
    draft_full(gen.make_inputs(draft_spec(**case)), num_splits)


def test_pair_16bit_matches_the_single_role_kernel():
    """The single-role kernel slices these stages differently (two warps per
    row tile), so the two agree within rounding, not bit for bit."""
    for case in (dict(), dict(q_tokens=16, draft_block=4), dict(draft_scratch=False, q_tokens=1, num_q_heads=64)):
        inp = gen.make_inputs(draft_spec(**case))
        dev = inp.to("cuda")
        for ns in (0, 3):
            a = run(inp, ns, dev=dev)
            pb.set_kernel_path(pb.KERNEL_WARP_MMA)
            out, lse = pb.decode_inputs(dev, num_splits=ns)
            torch.cuda.synchronize()
            pb.set_kernel_path(pb.KERNEL_WARP_PAIR)
            assert np.abs(a[0] - out.float().cpu().double().numpy()).max() <= 2e-2
            assert np.abs(a[1] - lse.cpu().double().numpy()).max() <= LSE_TOL


def test_graph_capture_replays_like_eager():
    common = dict(batch=6, ctx_range=(1, 900), context_lens=None, pool_pages=500, max_blocks_per_seq=57,
                  head_dim=256, num_q_heads=32, num_kv_heads=2)
    inp = gen.make_inputs(spec(**common))
    other = gen.make_inputs(spec(**common, seed=99))
    dev = inp.to("cuda")
    assert pb.kernel_for_inputs(dev) == pb.KERNEL_WARP_PAIR
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
        if t is not None:
            getattr(dev, name).copy_(t)
    g.replay()
    torch.cuda.synchronize()
    eager = pb.decode_inputs(other.to("cuda"), num_splits=0)
    torch.cuda.synchronize()
    assert torch.equal(out, eager[0]) and torch.equal(lse, eager[1])
