"""GPU path (through the C ABI) against the fp64 oracle.

Bar: |gpu - oracle| <= tol + tol * |oracle| elementwise on out, with
tol = 1e-2 for bf16 KV and 2e-2 for fp8 KV, and |lse_gpu - lse_oracle| <= 1e-3
(lse = -inf exactly where the oracle's is). Inputs are the seeded synthetic
workloads; the full-size ones are checked on sampled rows the oracle
computes one by one, in the launch configuration the benchmark times
(num_splits = 0).
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


def tol_of(spec):
    return 2e-2 if spec.kv_format == "fp8" else 1e-2


def ora_inputs(inp):
    oi = oracle.as_oracle_inputs(inp.numpy_bits(), inp.spec.kv_format)
    if inp.spec.draft_block is not None:
        oi["draft_block"] = inp.spec.draft_block
    return oi


def gpu_decode(inp, num_splits=0, dev=None, **kw):
    dev = dev if dev is not None else inp.to("cuda")
    out, lse = pb.decode_inputs(dev, num_splits=num_splits, **kw)
    torch.cuda.synchronize()
    assert pb.device_error() == 0
    return out, lse


def to_np(out, lse):
    return out.float().cpu().double().numpy(), lse.cpu().double().numpy()


def assert_match(out, lse, ref_out, ref_lse, tol, rows=None):
    if rows is not None:
        idx = tuple(np.array(rows).T)
        out, lse, ref_out, ref_lse = out[idx], lse[idx], ref_out[idx], ref_lse[idx]
    assert np.all(np.isfinite(out)), "non-finite output"
    excess = np.abs(out - ref_out) - (tol + tol * np.abs(ref_out))
    assert excess.max() <= 0, f"out mismatch: max excess {excess.max():.3g}, max abs err {np.abs(out - ref_out).max():.3g}"
    inf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), inf), "lse -inf pattern differs"
    d = np.abs(lse[~inf] - ref_lse[~inf])
    assert d.size == 0 or d.max() <= LSE_TOL, f"lse mismatch: {d.max():.3g}"


def check_full(inp, num_splits):
    ref_out, ref_lse = oracle.decode(ora_inputs(inp), inp.scale)
    out, lse = to_np(*gpu_decode(inp, num_splits))
    assert_match(out, lse, ref_out, ref_lse, tol_of(inp.spec))


# --------------------------------------------------------------------- tiny
@pytest.mark.parametrize("num_splits", [1, 3, 0])
def test_tiny_workload(num_splits):
    check_full(gen.make_inputs(gen.SPECS["tiny"]), num_splits)


# ------------------------------------------------------------ shape sweeps
def spec(**kw):
    base = dict(batch=4, q_tokens=1, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                context_lens=(1, 100, 16, 333), seed=21)
    base.update(kw)
    return gen.custom_spec(**base)


SWEEP = [
    dict(),
    dict(head_dim=64),
    dict(head_dim=256),
    dict(page_size=32),
    dict(page_size=64, context_lens=(64, 65, 200, 1)),
    dict(page_size=128, context_lens=(300, 127, 128, 129)),
    dict(page_size=256, context_lens=(600, 255, 1, 257)),
    dict(num_q_heads=16, num_kv_heads=1),                       # G 16: one full row tile
    dict(num_q_heads=32, num_kv_heads=1, head_dim=64),          # G 32: two row tiles
    dict(num_q_heads=4, num_kv_heads=4),                        # MHA
    dict(q_tokens=4, num_q_heads=8, num_kv_heads=2),            # 16 rows
    dict(q_tokens=3, num_q_heads=10, num_kv_heads=2),           # 15 rows, odd group
    dict(context_lens=(0, 37, 0, 500)),                         # empty sequences
    dict(batch=9, ctx_range=(1, 700), context_lens=None, pool_pages=400),
    # head-group units: 4 kv heads x 8 rows in two row tiles; 4 x 16 rows in
    # four row tiles; 4 x (2 tokens x 2 heads) in one tile
    dict(num_q_heads=32, num_kv_heads=4),
    dict(num_q_heads=64, num_kv_heads=4),
    dict(q_tokens=2, num_q_heads=8, num_kv_heads=4),
]


@pytest.mark.parametrize("case", SWEEP, ids=[str(i) for i in range(len(SWEEP))])
@pytest.mark.parametrize("num_splits", [0, 1, 3, 17])
def test_bf16_sweep(case, num_splits):
    check_full(gen.make_inputs(spec(**case)), num_splits)


FP8_SWEEP = [
    dict(kv_format="fp8"),
    dict(kv_format="fp8", head_dim=256, num_q_heads=16, num_kv_heads=1),
    dict(kv_format="fp8", head_dim=256, num_q_heads=32, num_kv_heads=2, page_size=64, context_lens=(64, 1, 700, 65)),
    dict(kv_format="fp8", num_q_heads=24, num_kv_heads=1),       # two row tiles
    dict(kv_format="fp8", num_q_heads=16, num_kv_heads=8, context_lens=(0, 5, 900, 31)),
    # the fp8 workload's geometry (two kv heads per unit, slices of 32 tokens on alternate stages), ragged
    dict(kv_format="fp8", head_dim=256, num_q_heads=32, num_kv_heads=2, context_lens=(1, 17, 33, 500)),
    dict(kv_format="fp8", num_q_heads=16, num_kv_heads=16, context_lens=(3, 77, 300, 0)),   # more than 8 kv heads
    dict(kv_format="fp8", head_dim=256, num_q_heads=24, num_kv_heads=12, page_size=32),
]


@pytest.mark.parametrize("case", FP8_SWEEP, ids=[str(i) for i in range(len(FP8_SWEEP))])
@pytest.mark.parametrize("num_splits", [0, 1, 4])
def test_fp8_sweep(case, num_splits):
    check_full(gen.make_inputs(spec(**case)), num_splits)


# Block tables 64 pages wide: the host charges the weights only to calls
# whose page bound gives every SM several pages.
ITEM_WEIGHT_CASES = [
    dict(batch=40, ctx_range=(1, 48), context_lens=None, pool_pages=200, max_blocks_per_seq=64),  # 1-3 pages each
    dict(batch=40, ctx_range=(1, 48), context_lens=None, pool_pages=200, max_blocks_per_seq=64,
         kv_format="fp8"),                                                                       # paired kernel
    dict(batch=24, ctx_range=(0, 40), context_lens=None, pool_pages=120, max_blocks_per_seq=64, q_tokens=8,
         draft_scratch=True),
    dict(batch=7, context_lens=(1, 0, 17, 2, 33, 0, 5), num_q_heads=16, num_kv_heads=8, pool_pages=40,
         max_blocks_per_seq=400),
]


@pytest.mark.parametrize("case", ITEM_WEIGHT_CASES, ids=[str(i) for i in range(len(ITEM_WEIGHT_CASES))])
@pytest.mark.parametrize("combine", [pb.COMBINE_SEPARATE, pb.COMBINE_FUSED])
def test_balanced_schedule_item_weights(case, combine):
    """The balanced schedule charges each (sequence, head group) unit a few
    virtual pages ahead of its keys: with many short sequences, CTA shares
    start, end or lie wholly inside those pages (empty pieces), and the
    combined rows still match the oracle."""
    inp = gen.make_inputs(spec(**case))
    pb.set_combine(combine)
    try:
        check_full(inp, 0)
    finally:
        pb.set_combine(pb.COMBINE_SEPARATE)


FP8_SCALE_CASES = [
    dict(),
    dict(head_dim=256, num_q_heads=32, num_kv_heads=2, context_lens=(1, 40, 700, 2000)),
    dict(num_q_heads=24, num_kv_heads=1, context_lens=(90, 1000, 3, 257)),
]


@pytest.mark.parametrize("case", FP8_SCALE_CASES, ids=[str(i) for i in range(len(FP8_SCALE_CASES))])
@pytest.mark.parametrize("num_splits", [0, 1])
def test_fp8_query_and_value_scale_ranges(case, num_splits):
    """fp8 KV with query rows of very different magnitudes (each row times
    2^k, k in [-12, 3]), value scales that grow along every sequence (times
    2^(8 i / n), i the token, n the context length) and spread inside every
    stage (times a random 2^[-3, 3]), and key scales times 2^[-2, 2]: the
    scaled probabilities span far more than the e4m3 range, and every output
    element still meets the bar (a P operand of fewer than f16's eleven
    significant bits, or one whose range follows the stage's largest scale,
    misses it on elements near zero in rows of large outputs)."""
    inp = gen.make_inputs(spec(kv_format="fp8", **case))
    rng = np.random.default_rng(99)
    k = rng.integers(-12, 4, size=inp.q.shape[:-1])
    inp.q = (inp.q.float() * torch.from_numpy(np.exp2(k)).float()[..., None]).to(torch.bfloat16)
    bt = inp.block_tables.numpy()
    lens = inp.context_lens.numpy()
    P = inp.spec.page_size
    vs = inp.v_scale.clone()
    for b in range(bt.shape[0]):
        for i in range(int(lens[b])):
            page = int(bt[b, i // P])
            vs[page, i % P] *= float(2.0 ** np.floor(8 * i / max(1, int(lens[b]))))
    vs *= torch.from_numpy(np.exp2(rng.integers(-3, 4, size=vs.shape))).float()
    inp.v_scale = vs
    inp.k_scale = inp.k_scale * torch.from_numpy(np.exp2(rng.integers(-2, 3, size=inp.k_scale.shape))).float()
    check_full(inp, num_splits)


@pytest.mark.parametrize("q_scale", [4.0, 16.0])
@pytest.mark.parametrize("kv_format", ["bf16", "f16", "fp8"])
def test_spread_scores_move_the_running_max(kv_format, q_scale):
    """Queries scaled up so that scores spread over many log2 units: the
    running row max moves often, by less and by more than the 16-bit paths'
    slack before a rescale, and the result still matches the oracle."""
    inp = gen.make_inputs(spec(kv_format=kv_format, num_q_heads=16, num_kv_heads=1, head_dim=128,
                               context_lens=(700, 33, 1, 260)))
    q = (inp.q.float() * q_scale).to(inp.q.dtype)
    check_full(dataclasses.replace(inp, q=q), 0)
    check_full(dataclasses.replace(inp, q=q), 3)


F16_SWEEP = [
    dict(kv_format="f16"),
    dict(kv_format="f16", head_dim=64, num_q_heads=32, num_kv_heads=1),
    dict(kv_format="f16", head_dim=256, q_tokens=2, num_q_heads=16, num_kv_heads=4, page_size=64,
         context_lens=(64, 1, 700, 65)),
    dict(kv_format="f16", q_tokens=16, num_q_heads=8, num_kv_heads=2, context_lens=(0, 40, 129, 16)),
]


@pytest.mark.parametrize("case", F16_SWEEP, ids=[str(i) for i in range(len(F16_SWEEP))])
@pytest.mark.parametrize("num_splits", [0, 1, 4])
def test_f16_sweep(case, num_splits):
    check_full(gen.make_inputs(spec(**case)), num_splits)


# Head dim 64, G T = 4, kv heads a multiple of 8, 16-token pages: units of
# eight kv heads (two row tiles, four warps per tile, one head each), whose
# 16-row page box is 16 KB (with larger pages fewer heads fill a 16 KB box).
# Ragged lengths, several head groups per sequence, G x T as 4 x 1, 2 x 2
# and 1 x 4, a draft block of 2 tokens.
EIGHT_HEADS = [
    dict(head_dim=64, num_q_heads=32, num_kv_heads=8),
    dict(head_dim=64, num_q_heads=64, num_kv_heads=16, context_lens=(0, 17, 300, 1)),
    dict(head_dim=64, q_tokens=2, num_q_heads=16, num_kv_heads=8, context_lens=(63, 64, 1, 400)),
    dict(head_dim=64, q_tokens=4, num_q_heads=8, num_kv_heads=8, context_lens=(600, 255, 16, 257)),
    dict(head_dim=64, num_q_heads=32, num_kv_heads=8, batch=9, ctx_range=(0, 500), context_lens=None,
         pool_pages=400),
    dict(head_dim=64, q_tokens=2, num_q_heads=16, num_kv_heads=8, draft_scratch=True,
         context_lens=(0, 16, 33, 250)),
]


@pytest.mark.parametrize("kv_format", ["bf16", "f16"])
@pytest.mark.parametrize("case", EIGHT_HEADS, ids=[str(i) for i in range(len(EIGHT_HEADS))])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_units_of_eight_kv_heads(case, kv_format, num_splits):
    inp = gen.make_inputs(spec(kv_format=kv_format, **case))
    if inp.spec.draft_scratch and kv_format != "bf16":
        pytest.skip("the draft scratch path takes bf16")
    assert pb.heads_per_unit_inputs(inp) == 8
    check_full(inp, num_splits)


@pytest.mark.parametrize("combine", [pb.COMBINE_SEPARATE, pb.COMBINE_FUSED])
def test_units_of_eight_kv_heads_under_both_combines(combine):
    inp = gen.make_inputs(spec(head_dim=64, num_q_heads=32, num_kv_heads=8, batch=6, ctx_range=(1, 900),
                               context_lens=None, pool_pages=300))
    assert pb.heads_per_unit_inputs(inp) == 8
    pb.set_combine(combine)
    try:
        check_full(inp, 0)
    finally:
        pb.set_combine(pb.COMBINE_SEPARATE)


TIDAR_SWEEP = [
    dict(draft_scratch=True, q_tokens=8, num_q_heads=8, num_kv_heads=2),
    dict(draft_scratch=True, q_tokens=4, num_q_heads=4, num_kv_heads=1, context_lens=(0, 16, 17, 250)),
    dict(draft_scratch=True, q_tokens=2, num_q_heads=16, num_kv_heads=2, head_dim=64, page_size=64,
         context_lens=(63, 64, 1, 400)),
]


@pytest.mark.parametrize("case", TIDAR_SWEEP, ids=[str(i) for i in range(len(TIDAR_SWEEP))])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_tidar_sweep(case, num_splits):
    check_full(gen.make_inputs(spec(**case)), num_splits)


MASKED = [
    (dict(draft_scratch=True, q_tokens=8, num_q_heads=8, num_kv_heads=2), 1),
    (dict(draft_scratch=True, q_tokens=8, num_q_heads=8, num_kv_heads=2), 3),
    (dict(draft_scratch=True, q_tokens=8, num_q_heads=8, num_kv_heads=2), 4),
    (dict(draft_scratch=True, q_tokens=5, num_q_heads=4, num_kv_heads=1, context_lens=(0, 16, 17, 250)), 2),
    # long draft blocks: 64 rows of one kv head in four row tiles
    (dict(draft_scratch=True, q_tokens=16, num_q_heads=8, num_kv_heads=2), 1),
    (dict(draft_scratch=True, q_tokens=16, num_q_heads=8, num_kv_heads=2), 4),
    (dict(draft_scratch=True, q_tokens=16, num_q_heads=8, num_kv_heads=2), 16),
    (dict(draft_scratch=True, q_tokens=12, num_q_heads=8, num_kv_heads=2, context_lens=(3, 0, 100, 64)), 5),
    (dict(draft_scratch=True, q_tokens=32, num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=64,
          context_lens=(63, 64, 1, 400)), 8),
]


@pytest.mark.parametrize("case,bs", MASKED, ids=[str(i) for i in range(len(MASKED))])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_block_masked_draft_sweep(case, bs, num_splits):
    inp = gen.make_inputs(spec(**case))
    ref_out, ref_lse = oracle.decode(dict(ora_inputs(inp), draft_block=bs), inp.scale)
    out, lse = to_np(*gpu_decode(inp, num_splits, draft_block=bs))
    assert_match(out, lse, ref_out, ref_lse, tol_of(inp.spec))


LONG_ROWS = [
    dict(num_q_heads=64, num_kv_heads=1),                          # G 64
    dict(q_tokens=10, num_q_heads=16, num_kv_heads=4),             # 40 rows, padded to four tiles
    dict(q_tokens=16, num_q_heads=8, num_kv_heads=2, head_dim=64),
    dict(draft_scratch=True, q_tokens=16, num_q_heads=8, num_kv_heads=2),  # unmasked long draft
]


# Shapes whose units could hold 128 query rows (4 kv heads x 32 rows, 2 x 64):
# the units stay at 64 rows (four tiles; measured faster per call than
# 128-row units, whose larger page boxes leave more partials to combine)
EIGHT_TILES = [
    (dict(draft_scratch=True, q_tokens=8, num_q_heads=16, num_kv_heads=4), None),
    (dict(draft_scratch=True, q_tokens=8, num_q_heads=16, num_kv_heads=4, context_lens=(0, 31, 260, 16)), 3),
    (dict(draft_scratch=True, q_tokens=16, num_q_heads=8, num_kv_heads=4), 4),
    (dict(q_tokens=4, num_q_heads=32, num_kv_heads=4), None),
    (dict(draft_scratch=True, q_tokens=8, num_q_heads=32, num_kv_heads=8), 1),
    (dict(kv_format="f16", q_tokens=4, num_q_heads=32, num_kv_heads=4), None),
    (dict(draft_scratch=True, q_tokens=16, num_q_heads=16, num_kv_heads=4), 4),      # 2 heads x 64 rows
    (dict(draft_scratch=True, q_tokens=16, num_q_heads=16, num_kv_heads=4, page_size=32,
          context_lens=(32, 33, 1, 500)), 4),
    (dict(draft_scratch=True, q_tokens=8, num_q_heads=16, num_kv_heads=4, page_size=64,
          context_lens=(64, 65, 2, 700)), 2),
    (dict(q_tokens=1, num_q_heads=128, num_kv_heads=4, context_lens=(0, 7, 129, 1000)), None),  # G 32, no draft
]


@pytest.mark.parametrize("case,bs", EIGHT_TILES, ids=[str(i) for i in range(len(EIGHT_TILES))])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_units_of_up_to_four_row_tiles(case, bs, num_splits):
    inp = gen.make_inputs(spec(**case))
    oi = ora_inputs(inp)
    kw = {}
    if bs is not None:
        oi["draft_block"] = bs
        kw["draft_block"] = bs
    ref_out, ref_lse = oracle.decode(oi, inp.scale)
    out, lse = to_np(*gpu_decode(inp, num_splits, **kw))
    assert_match(out, lse, ref_out, ref_lse, tol_of(inp.spec))


@pytest.mark.parametrize("case", LONG_ROWS, ids=[str(i) for i in range(len(LONG_ROWS))])
@pytest.mark.parametrize("num_splits", [0, 1, 5])
def test_more_than_32_rows_per_kv_head(case, num_splits):
    check_full(gen.make_inputs(spec(**case)), num_splits)


# --------------------------------------------------------------- robustness
@pytest.mark.parametrize("kv_format", ["bf16", "fp8"])
@pytest.mark.parametrize("num_splits", [0, 2])
def test_unread_values_are_never_read(kv_format, num_splits):
    """NaN in unused pages, in slots past the context end and in their fp8
    scales, and INT32_MAX in unused block-table entries change nothing."""
    s = spec(kv_format=kv_format, context_lens=(5, 100, 33, 250), pool_pages=60)
    clean = gen.make_inputs(s)
    dirty = gen.make_inputs(s, poison=True)
    a = gpu_decode(clean, num_splits)
    b = gpu_decode(dirty, num_splits)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    check_full(dirty, num_splits)


@pytest.mark.parametrize("kv_format", ["bf16", "fp8"])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_out_of_range_page_ids_read_zeros(kv_format, num_splits):
    """Block-table entries outside [0, num_pages) inside the context act as
    pages of zero keys and values (the copy engine fills out-of-range boxes):
    the result equals the oracle's on a pool with one extra all-zero page
    (fp8: zero codes, scale 1) that those entries point to."""
    s = spec(kv_format=kv_format, context_lens=(100, 40, 250, 17), pool_pages=60)
    inp = gen.make_inputs(s)
    n = inp.num_pages
    bad = inp.block_tables.clone()
    bad[0, 2] = n + 3
    bad[2, 0] = -1
    bad[2, 9] = n
    gpu_in = dataclasses.replace(inp, block_tables=bad)
    ref = dataclasses.replace(inp)
    ref.k_cache = torch.cat([inp.k_cache, torch.zeros_like(inp.k_cache[:1])])
    ref.v_cache = torch.cat([inp.v_cache, torch.zeros_like(inp.v_cache[:1])])
    if kv_format == "fp8":
        ref.k_scale = torch.cat([inp.k_scale, torch.ones_like(inp.k_scale[:1])])
        ref.v_scale = torch.cat([inp.v_scale, torch.ones_like(inp.v_scale[:1])])
    fixed = bad.clone()
    fixed[(bad < 0) | (bad >= n)] = n
    fixed[inp.block_tables < 0] = inp.block_tables[inp.block_tables < 0]
    ref.block_tables = fixed
    ref_out, ref_lse = oracle.decode(ora_inputs(ref), inp.scale)
    out, lse = to_np(*gpu_decode(gpu_in, num_splits))
    assert_match(out, lse, ref_out, ref_lse, tol_of(s))


@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_page_relabelling_is_bit_exact(num_splits):
    inp = gen.make_inputs(spec(pool_pages=80, context_lens=(300, 7, 129, 64)))
    perm = torch.randperm(80, generator=torch.Generator().manual_seed(5))
    moved = dataclasses.replace(inp)
    moved.k_cache = torch.empty_like(inp.k_cache)
    moved.v_cache = torch.empty_like(inp.v_cache)
    moved.k_cache[perm] = inp.k_cache
    moved.v_cache[perm] = inp.v_cache
    bt = inp.block_tables.clone()
    valid = bt >= 0
    bt[valid] = perm[bt[valid].long()].to(torch.int32)
    moved.block_tables = bt
    a = gpu_decode(inp, num_splits)
    b = gpu_decode(moved, num_splits)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("S", [2, 5, 40])
def test_explicit_split_partials_match_oracle(S):
    """The per-split partials (an intermediate the pages suggest checking:
    the log-sum-exp) against the oracle's split variant."""
    inp = gen.make_inputs(spec(context_lens=(1, 100, 16, 333)))
    dev = inp.to("cuda")
    shp = pb.make_shape(dev.q, dev.k_cache, dev.block_tables)
    ws = torch.zeros(pb.workspace_size(shp, S), dtype=torch.uint8, device="cuda")
    gpu_decode(inp, S, dev=dev, workspace=ws)
    B, T, Hq, D = inp.q.shape
    po, pl = pb.split_workspace_views(ws, B, T, Hq, S, D)
    ref_po, ref_pl = oracle.decode_split(ora_inputs(inp), inp.scale, S)
    pl = pl.double().cpu().numpy()
    po = po.double().cpu().numpy()
    inf = np.isneginf(ref_pl)
    assert np.array_equal(np.isneginf(pl), inf)
    assert np.abs(pl[~inf] - ref_pl[~inf]).max() <= LSE_TOL
    fin = ~inf
    assert np.abs(po[fin] - ref_po[fin]).max() <= 1e-2 * (1 + np.abs(ref_po[fin]).max())


def test_reduce_entry_point_against_oracle_combine():
    rng = np.random.default_rng(9)
    B, T, Hq, S, D = 3, 2, 4, 7, 128
    po = rng.standard_normal((B, T, Hq, S, D)).astype(np.float32)
    pl = (rng.standard_normal((B, T, Hq, S)) * 3).astype(np.float32)
    pl[0, 0, 0, :] = -np.inf          # all splits empty
    pl[1, 1, 2, ::2] = -np.inf        # some empty
    ref_o, ref_l = oracle.combine(po.astype(np.float64), pl.astype(np.float64))
    out, lse = pb.decode_reduce(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda())
    torch.cuda.synchronize()
    o, l = to_np(out, lse)
    assert_match(o, l, ref_o, ref_l, 1e-2)


@pytest.mark.parametrize("D", [64, 256, 320, 1024])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_reduce_entry_point_head_dims_and_f16(D, out_dtype):
    """The standalone combine for head dims up to 1024 (rows wider than one
    warp's 256 columns are combined in chunks), with bf16 or f16 out."""
    rng = np.random.default_rng(D)
    B, T, Hq, S = 2, 1, 3, 5
    po = rng.standard_normal((B, T, Hq, S, D)).astype(np.float32)
    pl = (rng.standard_normal((B, T, Hq, S)) * 3).astype(np.float32)
    pl[1, 0, 1, 1:] = -np.inf
    ref_o, ref_l = oracle.combine(po.astype(np.float64), pl.astype(np.float64))
    out = torch.full((B, T, Hq, D), 5.0, dtype=out_dtype, device="cuda")
    out, lse = pb.decode_reduce(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), out=out)
    torch.cuda.synchronize()
    assert out.dtype == out_dtype
    assert_match(*to_np(out, lse), ref_o, ref_l, 1e-2)


def test_reduce_propagates_a_nan_split():
    """A split whose lse is NaN (work cut short) makes its row NaN; the other
    rows are unaffected."""
    rng = np.random.default_rng(3)
    B, T, Hq, S, D = 2, 1, 2, 4, 128
    po = rng.standard_normal((B, T, Hq, S, D)).astype(np.float32)
    pl = rng.standard_normal((B, T, Hq, S)).astype(np.float32)
    pl[0, 0, 1, 2] = np.nan
    po[0, 0, 1, 2] = np.nan
    out, lse = pb.decode_reduce(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda())
    torch.cuda.synchronize()
    o, l = to_np(out, lse)
    assert np.all(np.isnan(o[0, 0, 1])) and np.isnan(l[0, 0, 1])
    mask = np.ones((B, T, Hq), dtype=bool)
    mask[0, 0, 1] = False
    ref_o, ref_l = oracle.combine(po.astype(np.float64), pl.astype(np.float64))
    assert np.all(np.abs(o[mask] - ref_o[mask]) <= 1e-2 + 1e-2 * np.abs(ref_o[mask]))
    assert np.all(np.abs(l[mask] - ref_l[mask]) <= LSE_TOL)


def test_split_counts_beyond_pages_and_single_page():
    inp = gen.make_inputs(spec(context_lens=(16, 1, 17, 40)))
    for S in (1, 2, 3, 4, 9, 100):
        check_full(inp, S)


@pytest.mark.parametrize("kv_format", ["bf16", "fp8"])
def test_auto_splits_fall_back_to_explicit_splits_for_many_sequences(kv_format):
    """num_splits=0 runs the balanced schedule while the per-sequence table
    fits in shared memory; for 12000 sequences (8 bytes of table each, more
    than any instance has room for) it resolves to the explicit split count
    pa_decode_choose_splits reports, bit for bit."""
    small = gen.make_inputs(spec(kv_format=kv_format))
    assert pb.choose_splits(pb.make_shape(small.q, small.k_cache, small.block_tables), kv_format == "fp8") == 0
    s = spec(kv_format=kv_format, batch=12000, context_lens=None, ctx_range=(1, 40), pool_pages=36000)
    inp = gen.make_inputs(s)
    shp = pb.make_shape(inp.q, inp.k_cache, inp.block_tables)
    S = pb.choose_splits(shp, kv_format == "fp8")
    assert S >= 1
    # the size for num_splits = 0 covers every decode entry point's plan
    assert pb.workspace_size(shp, 0) >= pb.workspace_size(shp, S)
    dev = inp.to("cuda")
    a = gpu_decode(inp, 0, dev=dev)
    b = gpu_decode(inp, S, dev=dev)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    ref_out, ref_lse = oracle.decode(ora_inputs(inp), inp.scale)
    assert_match(*to_np(*a), ref_out, ref_lse, tol_of(s))


# ----------------------------------------------------- full-size workloads
def sample_rows(inp, n, seed):
    s = inp.spec
    rng = np.random.default_rng(seed)
    rows = {(0, 0, 0), (s.batch - 1, s.q_tokens - 1, s.num_q_heads - 1)}
    # every query token of one whole kv-head group
    b = int(rng.integers(s.batch))
    g = int(rng.integers(s.num_kv_heads))
    for t in range(s.q_tokens):
        for h in range(g * s.group, (g + 1) * s.group):
            rows.add((b, t, h))
    while len(rows) < n:
        rows.add((int(rng.integers(s.batch)), int(rng.integers(s.q_tokens)), int(rng.integers(s.num_q_heads))))
    return sorted(rows)


# The five workloads of the problem statement are compared on every output
# row (the oracle takes a few seconds each); the extension workloads on
# sampled rows.
FULL_ROWS = ("tiny", "gqa", "long", "fp8", "tidar")


@pytest.mark.parametrize("name", ["tiny", "gqa", "long", "fp8", "tidar", "tidar_causal", "tidar_long", "gqa_f16",
                                  "gqa_d64", "gqa_d256"])
def test_full_size_workload(name):
    inp = gen.make_inputs(gen.SPECS[name])
    out, lse = gpu_decode(inp, 0)
    out_np, lse_np = to_np(out, lse)
    assert np.all(np.isfinite(out_np)) and np.all(np.isfinite(lse_np))
    rows = None if name in FULL_ROWS else sample_rows(inp, 48, seed=len(name))
    ref_out, ref_lse = oracle.decode(ora_inputs(inp), inp.scale, rows=rows)
    assert_match(out_np, lse_np, ref_out, ref_lse, tol_of(inp.spec), rows=rows)
    # Explicit splits agree with the balanced launch at full size as well.
    out2, lse2 = to_np(*gpu_decode(inp, 7))
    assert np.abs(lse2 - lse_np).max() <= LSE_TOL
    assert np.abs(out2 - out_np).max() <= 2 * tol_of(inp.spec)


# ------------------------------------------------------------ graph capture
def test_graph_capture_replays_like_eager():
    """Captured into a CUDA graph, then inputs rewritten in place and the
    graph replayed: identical bits to an eager call on the new inputs."""
    common = dict(batch=6, ctx_range=(1, 900), context_lens=None, pool_pages=500, max_blocks_per_seq=57)
    inp = gen.make_inputs(spec(**common))
    other = gen.make_inputs(spec(**common, seed=99))
    dev = inp.to("cuda")
    shp = pb.make_shape(dev.q, dev.k_cache, dev.block_tables)
    ws = torch.empty(pb.workspace_size(shp, 0), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev.q)
    lse = torch.empty(dev.q.shape[:3], dtype=torch.float32, device="cuda")
    pb.decode_inputs(dev, out=out, lse=lse, workspace=ws)  # first call outside capture
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
    got = (out.clone(), lse.clone())
    eager = gpu_decode(other, 0)
    assert torch.equal(got[0], eager[0]) and torch.equal(got[1], eager[1])
    ref_out, ref_lse = oracle.decode(ora_inputs(other), other.scale)
    assert_match(*to_np(*got), ref_out, ref_lse, 1e-2)


# ----------------------------------------------------------- random shapes
def random_case(rng):
    """A small problem drawn from every supported axis at once."""
    kv_format = str(rng.choice(["bf16", "bf16", "fp8", "f16"]))
    D = int(rng.choice([128, 256] if kv_format == "fp8" else [64, 128, 256]))
    Hkv = int(rng.choice([1, 2, 4, 8, 16] if kv_format == "fp8" else [1, 2, 3, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    tidar = kv_format == "bf16" and rng.random() < 0.3
    T = int(rng.integers(1, max(2, min(8, 32 // G)) + 1))
    while G * T > 32:
        T -= 1
    P = int(rng.choice([16, 32, 64, 128, 256]))
    B = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.integers(0, 600, B)]
    if rng.random() < 0.3:
        lens[0] = 0
    case = dict(batch=B, q_tokens=T, num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=P,
                context_lens=tuple(lens), kv_format=kv_format, draft_scratch=tidar,
                seed=int(rng.integers(1 << 30)))
    if tidar and rng.random() < 0.5:
        case["draft_block"] = int(rng.integers(1, T + 1))
    return case, int(rng.choice([0, 0, 1, 2, 5]))


@pytest.mark.parametrize("i", range(60))
def test_random_shapes(i):
    case, num_splits = random_case(np.random.default_rng(1000 + i))
    inp = gen.make_inputs(spec(**case))
    oi = ora_inputs(inp)
    ref_out, ref_lse = oracle.decode(oi, inp.scale)
    out, lse = to_np(*gpu_decode(inp, num_splits))
    assert_match(out, lse, ref_out, ref_lse, tol_of(inp.spec))
