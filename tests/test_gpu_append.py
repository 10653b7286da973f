"""GPU KV-cache append (pa_kv_append / pa_kv_append_fp8, through the C ABI)
against the CPU oracle: the written caches (and fp8 scales) must equal the
oracle's bit for bit, since the append copies 16-bit rows (bf16, or f16 into
f16 caches) and takes every fp8 rounding decision in float32 exactly as the
oracle does."""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle import kv_append as ka
from paged_kv_attention_15_gb300 import binding as pb
from paged_kv_attention_15_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


def spec(**kw):
    base = dict(batch=4, new_tokens=5, num_kv_heads=2, head_dim=128, page_size=16,
                context_lens=(0, 13, 31, 100), seed=31)
    base.update(kw)
    return gen.AppendSpec(name="custom", **base)


def gpu_append(inp):
    dev = inp.to("cuda")
    pb.kv_append(dev.k_new, dev.v_new, dev.block_tables, dev.context_lens, dev.k_cache, dev.v_cache,
                 k_scale=dev.k_scale, v_scale=dev.v_scale)
    torch.cuda.synchronize()
    return dev


def oracle_append(inp, rows=None):
    bits = inp.numpy_bits()
    caches = {n: bits[n] for n in ("k_cache", "v_cache", "k_scale", "v_scale") if n in bits}
    bt, ctx, kn, vn = bits["block_tables"], bits["context_lens"], bits["k_new"], bits["v_new"]
    if rows is not None:
        bt, ctx, kn, vn = bt[rows], ctx[rows], kn[rows], vn[rows]
    return ka.append(caches, kn, vn, bt, ctx, inp.spec.page_size)


def bits_of(t):
    t = t.cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy().view(np.uint32)
    return t.numpy()


def assert_caches_equal(dev, ref, pages=None):
    for name in ("k_cache", "v_cache", "k_scale", "v_scale"):
        if name not in ref:
            continue
        got = bits_of(getattr(dev, name))
        want = ref[name].view(np.uint32) if ref[name].dtype == np.float32 else ref[name]
        if pages is not None:
            got, want = got[pages], want[pages]
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{name}: {len(bad)} elements differ, first at {bad[0].tolist()}"


CASES = [
    dict(),
    dict(head_dim=64, new_tokens=1),
    dict(head_dim=256, new_tokens=17, page_size=64, context_lens=(63, 64, 0, 130)),
    dict(new_tokens=40, num_kv_heads=1, context_lens=(5, 0, 16, 1)),
    dict(num_kv_heads=8, new_tokens=3, page_size=256, context_lens=(255, 0, 256, 700)),
    dict(batch=9, ctx_range=(0, 300), context_lens=None, new_tokens=7, num_kv_heads=4),
]


@pytest.mark.parametrize("kv_format", ["bf16", "f16", "fp8"])
@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_append_matches_oracle_bit_exact(case, kv_format):
    inp = gen.make_append_inputs(spec(kv_format=kv_format, **case))
    assert_caches_equal(gpu_append(inp), oracle_append(inp))


# Calls with at least a wave of resident warps' worth of tasks (2 B T of
# them): 16-bit rows of one or two 32-piece rounds take several tasks per
# warp step, whose payload loads all go out before their slot lookups.
MANY_TASKS = [
    dict(batch=16, new_tokens=256, num_kv_heads=2, head_dim=128, context_lens=None, ctx_range=(0, 300)),
    dict(batch=16, new_tokens=256, num_kv_heads=4, head_dim=128, context_lens=None, ctx_range=(0, 300)),
    dict(batch=16, new_tokens=256, num_kv_heads=3, head_dim=64, page_size=32, context_lens=None,
         ctx_range=(0, 300)),
    dict(batch=16, new_tokens=256, num_kv_heads=1, head_dim=256, context_lens=None, ctx_range=(0, 300)),
]


@pytest.mark.parametrize("kv_format", ["bf16", "f16", "fp8"])
@pytest.mark.parametrize("case", MANY_TASKS, ids=[str(i) for i in range(len(MANY_TASKS))])
def test_append_of_many_tasks_bit_exact(case, kv_format):
    inp = gen.make_append_inputs(spec(kv_format=kv_format, **case))
    assert_caches_equal(gpu_append(inp), oracle_append(inp))


@pytest.mark.parametrize("kv_format", ["bf16", "f16", "fp8"])
def test_many_task_calls_skip_bad_slots(kv_format):
    """Several tasks per warp step, some of them skipped: tokens past the
    block table's capacity (two sequences whose lengths leave room for only
    10 and 1 of their 256 new tokens) and page ids outside the pool
    (negative, or past its end)."""
    inp = gen.make_append_inputs(spec(kv_format=kv_format, batch=16, new_tokens=256, num_kv_heads=2,
                                      context_lens=None, ctx_range=(0, 300)))
    bt = inp.block_tables.clone()
    n, cap = inp.k_cache.shape[0], bt.shape[1] * 16
    bt[1, 3] = n + 11
    bt[5, 0] = -1
    bt[9, 7:12] = -7
    bt[14, bt.shape[1] - 1] = n
    lens = inp.context_lens.clone()
    lens[3] = cap - 10
    lens[8] = cap - 1
    inp = dataclasses.replace(inp, block_tables=bt, context_lens=lens)
    before = inp.clone()
    assert_caches_equal(gpu_append(inp), oracle_append(before))


@pytest.mark.parametrize("kv_format", ["bf16", "f16", "fp8"])
def test_positions_past_capacity_and_bad_pages_are_skipped(kv_format):
    inp = gen.make_append_inputs(spec(kv_format=kv_format, new_tokens=6, context_lens=(40, 42, 0, 3),
                                      max_blocks_per_seq=3))
    bt = inp.block_tables.clone()
    bt[2, 0] = inp.k_cache.shape[0] + 7
    bt[3, 0] = -5
    inp = dataclasses.replace(inp, block_tables=bt, context_lens=torch.tensor([40, 44, 0, 3], dtype=torch.int32))
    before = inp.clone()
    dev = gpu_append(inp)
    ref = oracle_append(before)
    assert_caches_equal(dev, ref)


def test_fp8_rows_of_the_hand_derived_examples():
    """The worked examples of tests/golden (padded with zeros, which change
    neither amax nor any code) come out of the GPU quantiser exactly."""
    from test_oracle_append import read_golden

    examples = list(read_golden())
    n = len(examples)
    inp = gen.make_append_inputs(spec(kv_format="fp8", batch=1, new_tokens=n, num_kv_heads=1, head_dim=64,
                                      context_lens=(0,)))
    rows = np.zeros((1, n, 1, 64), dtype=np.float32)
    for i, (x, _, _) in enumerate(examples):
        rows[0, i, 0, :len(x)] = x
    newk = torch.from_numpy(rows).to(torch.bfloat16)
    inp = dataclasses.replace(inp, k_new=newk, v_new=-newk)
    dev = gpu_append(inp)
    bt = inp.block_tables[0].tolist()
    for i, (x, scale, codes) in enumerate(examples):
        page, slot = bt[i // 16], i % 16
        got = dev.k_cache[page, slot, 0].cpu().numpy()
        assert got[:len(x)].tolist() == codes, (i, [hex(c) for c in got[:len(x)]])
        assert np.all(got[len(x):] == 0)
        assert float(dev.k_scale[page, slot, 0]) == scale
        negated = dev.v_cache[page, slot, 0].cpu().numpy()[:len(x)]
        assert negated.tolist() == [c ^ 0x80 for c in codes]  # -x: same magnitudes, flipped signs


@pytest.mark.parametrize("head_dim", [64, 128, 256])
def test_fp8_quantiser_stress_bit_exact(head_dim):
    """Millions of values over every binade (rows scaled by 2^-100 .. 2^60,
    single dominant elements, exact e4m3 midpoints times the scale, zeros of
    both signs): every code and scale equals the oracle's."""
    B, T, Hkv = 16, 64, 4
    rng = np.random.default_rng(head_dim)
    x = rng.standard_normal((B, T, Hkv, head_dim)) * 2.0 ** rng.integers(-60, 60, (B, T, Hkv, 1))
    x[:, 4::7] *= 2.0 ** -40                       # rows far below 2^-60
    x[:, ::7, :, 1:] *= 1e-3                     # one dominant element per row
    x[:, 1::7] = 0.0
    x[:, 2::7, :, ::2] = -0.0
    tab = oracle.e4m3fn_table()
    fin = np.unique(np.abs(tab[~np.isnan(tab)]))
    mids = (fin[:-1] + fin[1:]) / 2               # ties of the e4m3 rounding at scale 1 ...
    sel = x[:, 3::7]
    sel[..., 0] = 448.0
    sel[..., 1:] = rng.choice(np.concatenate([mids, -mids, fin]), sel[..., 1:].shape)
    x[:, 3::7] = sel                               # ... and amax 448, so scale = 1 exactly
    newk = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    inp = gen.make_append_inputs(spec(kv_format="fp8", batch=B, new_tokens=T, num_kv_heads=Hkv,
                                      head_dim=head_dim, context_lens=None, ctx_range=(0, 50)))
    inp = dataclasses.replace(inp, k_new=newk, v_new=-newk)
    assert_caches_equal(gpu_append(inp), oracle_append(inp))


@pytest.mark.parametrize("kv_format", ["bf16", "f16", "fp8"])
def test_decode_after_append_matches_oracle(kv_format):
    """Append T tokens on the GPU, then decode over C_b + T tokens: the result
    equals the oracle's decode of the oracle-appended cache."""
    inp = gen.make_append_inputs(spec(kv_format=kv_format, num_kv_heads=2, new_tokens=9,
                                      context_lens=(7, 16, 40, 0)))
    dev = gpu_append(inp)
    ref = oracle_append(inp)
    B, T, Hkv, D = inp.k_new.shape
    Hq = 4 * Hkv
    q = torch.randn(B, 1, Hq, D, generator=torch.Generator().manual_seed(3)).to(
        torch.float16 if kv_format == "f16" else torch.bfloat16)
    ctx = inp.context_lens + T
    out, lse = pb.decode(q.cuda(), dev.k_cache, dev.v_cache, dev.block_tables, ctx.cuda(), D ** -0.5,
                         k_scale=dev.k_scale, v_scale=dev.v_scale)
    torch.cuda.synchronize()
    oi = oracle.as_oracle_inputs(dict(q=q.view(torch.int16).numpy().view(np.uint16), k_cache=ref["k_cache"],
                                      v_cache=ref["v_cache"], k_scale=ref.get("k_scale"),
                                      v_scale=ref.get("v_scale"), block_tables=inp.block_tables.numpy(),
                                      context_lens=ctx.numpy()), kv_format)
    ref_out, ref_lse = oracle.decode(oi, D ** -0.5)
    tol = 2e-2 if kv_format == "fp8" else 1e-2
    got = out.float().cpu().double().numpy()
    assert np.all(np.abs(got - ref_out) <= tol + tol * np.abs(ref_out))
    assert np.abs(lse.cpu().double().numpy() - ref_lse).max() <= 1e-3


@pytest.mark.parametrize("name", list(gen.APPEND_SPECS))
def test_full_size_append_sampled(name):
    """The full workload on the GPU; the pages of four sampled sequences
    (every sequence owns its pages) equal the oracle's append of those."""
    inp = gen.make_append_inputs(gen.APPEND_SPECS[name])
    rows = sorted({0, inp.spec.batch - 1} | set(np.random.default_rng(1).choice(inp.spec.batch, 2).tolist()))
    ref = oracle_append(inp, rows=rows)
    dev = gpu_append(inp)
    bt = inp.block_tables[rows].numpy()
    pages = np.unique(bt[bt >= 0])
    assert_caches_equal(dev, ref, pages=pages)


def test_graph_replay_of_append_writes_the_same():
    inp = gen.make_append_inputs(spec(kv_format="fp8", new_tokens=33))
    ref = oracle_append(inp)
    dev = inp.to("cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pb.kv_append(dev.k_new, dev.v_new, dev.block_tables, dev.context_lens, dev.k_cache, dev.v_cache,
                     k_scale=dev.k_scale, v_scale=dev.v_scale, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert_caches_equal(dev, ref)
