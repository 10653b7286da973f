"""Pins of the fp64 oracle against things other than itself.

Each test ties the oracle to a library routine (torch scaled-dot-product
attention and logsumexp on de-paged keys, torch's float8_e4m3fn and bfloat16
conversions), to an invariant of the method (page relabelling, split-K
combine, GQA as MHA with repeated kv heads, draft block as extra pages), to a
closed form, or to the OCP e4m3fn table. A plausible slip in the oracle (a
wrong page or slot index, a wrong head group, a dropped scale, a transposed
product, a wrong combine weight) fails at least one of them; test_planted_*
plant such slips in a copy of the oracle and check that.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import pa_oracle
from paged_kv_attention_15_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def ora_inputs(inp):
    return oracle.as_oracle_inputs(inp.numpy_bits(), inp.spec.kv_format)


def small_spec(**kw):
    base = dict(batch=3, q_tokens=1, num_q_heads=8, num_kv_heads=2, head_dim=32,
                page_size=16, context_lens=(37, 1, 100), seed=11)
    base.update(kw)
    return gen.custom_spec(**base)


# ---------------------------------------------------------------------------
# Library routine: torch SDPA over keys de-paged with torch indexing
# ---------------------------------------------------------------------------

def torch_reference(inp):
    """Dense attention with torch on keys gathered by whole-page indexing."""
    s = inp.spec
    out = torch.zeros(s.batch, s.q_tokens, s.num_q_heads, s.head_dim, dtype=torch.float64)
    lse = torch.full((s.batch, s.q_tokens, s.num_q_heads), -math.inf, dtype=torch.float64)
    for b in range(s.batch):
        c = int(inp.context_lens[b])
        n = -(-c // s.page_size)
        pages = inp.block_tables[b, :n].long()
        if s.kv_format == "fp8":
            kd = inp.k_cache[pages].view(torch.float8_e4m3fn).to(torch.float64) * inp.k_scale[pages].double()[..., None]
            vd = inp.v_cache[pages].view(torch.float8_e4m3fn).to(torch.float64) * inp.v_scale[pages].double()[..., None]
        else:
            kd = inp.k_cache[pages].to(torch.float64)
            vd = inp.v_cache[pages].to(torch.float64)
        K = kd.reshape(n * s.page_size, s.num_kv_heads, s.head_dim)[:c]
        V = vd.reshape(n * s.page_size, s.num_kv_heads, s.head_dim)[:c]
        if inp.k_scratch is not None:
            K = torch.cat([K, inp.k_scratch[b].to(torch.float64)], 0)
            V = torch.cat([V, inp.v_scratch[b].to(torch.float64)], 0)
        if K.shape[0] == 0:
            continue
        q = inp.q[b].to(torch.float64).transpose(0, 1)  # [Hq, T, D]
        Kh = K.transpose(0, 1).repeat_interleave(s.group, dim=0)  # [Hq, N, D]
        Vh = V.transpose(0, 1).repeat_interleave(s.group, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(q[None], Kh[None], Vh[None], scale=s.scale)[0]
        out[b] = o.transpose(0, 1)
        lse[b] = torch.logsumexp(s.scale * q @ Kh.transpose(1, 2), dim=-1).transpose(0, 1)
    return out.numpy(), lse.numpy()


CASES = [
    dict(),                                                    # GQA 4, ragged, ctx 1
    dict(num_q_heads=4, num_kv_heads=4),                       # MHA
    dict(num_q_heads=8, num_kv_heads=1, head_dim=64),          # MQA
    dict(q_tokens=3, page_size=32, context_lens=(64, 65, 5)),  # several query tokens
    dict(kv_format="fp8", head_dim=64),                        # fp8 codes + scales
    dict(draft_scratch=True, q_tokens=4, context_lens=(20, 0, 33)),  # draft block, empty prefix
    dict(pool_pages=20, context_lens=(0, 17, 64)),             # empty context, spare pages
    dict(kv_format="f16", q_tokens=2),                         # f16 q, caches and out
    dict(kv_format="f16", draft_scratch=True, q_tokens=3),     # f16 draft block
]


@pytest.mark.parametrize("case", CASES)
def test_matches_torch_sdpa(case):
    inp = gen.make_inputs(small_spec(**case))
    out, lse = oracle.decode(ora_inputs(inp), inp.scale)
    ref_out, ref_lse = torch_reference(inp)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_row_subset_matches_full():
    inp = gen.make_inputs(small_spec())
    oi = ora_inputs(inp)
    out, lse = oracle.decode(oi, inp.scale)
    rows = [(0, 0, 3), (2, 0, 7), (1, 0, 0)]
    sub_out, sub_lse = oracle.decode(oi, inp.scale, rows=rows)
    for r in rows:  # BLAS may order a 1-row product differently: fp64 rounding only
        np.testing.assert_allclose(sub_out[r], out[r], rtol=0, atol=1e-14)
        assert abs(sub_lse[r] - lse[r]) < 1e-14
    assert np.isnan(sub_lse[0, 0, 0])


# ---------------------------------------------------------------------------
# Stored-format widening
# ---------------------------------------------------------------------------

def test_bf16_widening_matches_torch():
    x = torch.randn(4096, dtype=torch.float32).to(torch.bfloat16)
    x[:4] = torch.tensor([0.0, -0.0, float("inf"), 1e-40])
    bits = x.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(bits), x.to(torch.float64).numpy())


def test_f16_widening_matches_torch():
    x = torch.randn(4096, dtype=torch.float32).to(torch.float16)
    x[:5] = torch.tensor([0.0, -0.0, float("inf"), 6e-8, 65504.0])
    bits = x.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.f16_bits_to_f64(bits), x.to(torch.float64).numpy())


def test_e4m3fn_table_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    tab = oracle.e4m3fn_table()
    assert np.array_equal(np.isnan(tab), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(tab[ok], ref[ok])
    assert np.isnan(tab).sum() == 2


def test_e4m3fn_golden_ocp_values():
    tab = oracle.e4m3fn_table()
    n = 0
    with open(os.path.join(GOLDEN, "e4m3fn_ocp_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            code, val = line.split()
            code, val = int(code, 16), float(val)
            if math.isnan(val):
                assert math.isnan(tab[code])
            else:
                assert tab[code] == val and math.copysign(1, tab[code]) == math.copysign(1, val)
            n += 1
    assert n >= 15


def test_fp8_quantiser_round_trip_bound():
    """Generator codes decoded by the oracle are within half an e4m3 step
    (relative 2^-4 for normals, absolute scale * 2^-10 for subnormals) of
    the fp32 values they came from."""
    spec = small_spec(kv_format="fp8", head_dim=64, pool_pages=4, context_lens=(16, 16, 16))
    codes, scales = gen._normal_fp8((4, 16, 2, 64), seed=5, stream=4, rows_per_chunk=4)
    buf = np.empty(4 * 16 * 2 * 64, dtype=np.float32)
    gen._rng(5, 4, 0).standard_normal(out=buf, dtype=np.float32)
    x = buf.reshape(4, 16, 2, 64).astype(np.float64)
    xhat = oracle.e4m3fn_table()[codes.numpy()] * scales.numpy().astype(np.float64)[..., None]
    s = scales.numpy().astype(np.float64)[..., None]
    bound = np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(x - xhat) <= bound)
    # The largest magnitude of each vector maps to about 448 * scale.
    amax_idx = np.abs(x).argmax(axis=-1)
    top = np.take_along_axis(np.abs(xhat), amax_idx[..., None], -1)[..., 0]
    np.testing.assert_allclose(top, 448 * s[..., 0], rtol=2 ** -4)
    del spec


# ---------------------------------------------------------------------------
# Invariants of the method
# ---------------------------------------------------------------------------

def relabel_pages(oi, rng):
    """Move every physical page p to slot perm[p] and rewrite the block table."""
    pool = oi["k_cache"].shape[0]
    perm = rng.permutation(pool)
    out = dict(oi)
    for name in ("k_cache", "v_cache", "k_scale", "v_scale"):
        if oi.get(name) is not None:
            moved = np.empty_like(oi[name])
            moved[perm] = oi[name]
            out[name] = moved
    bt = oi["block_tables"].copy()
    valid = (bt >= 0) & (bt < pool)
    bt[valid] = perm[bt[valid]]
    out["block_tables"] = bt
    return out


@pytest.mark.parametrize("case", [dict(), dict(kv_format="fp8", head_dim=64),
                                  dict(draft_scratch=True, q_tokens=2)])
def test_page_relabelling_is_bit_exact(case):
    inp = gen.make_inputs(small_spec(pool_pages=24, **case))
    oi = ora_inputs(inp)
    out, lse = oracle.decode(oi, inp.scale)
    out2, lse2 = oracle.decode(relabel_pages(oi, np.random.default_rng(3)), inp.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("case", [dict(), dict(draft_scratch=True, q_tokens=2),
                                  dict(kv_format="fp8", head_dim=64)])
def test_split_combine_equals_unsplit(case):
    inp = gen.make_inputs(small_spec(**case))
    oi = ora_inputs(inp)
    out, lse = oracle.decode(oi, inp.scale)
    nmax = max(-(-int(c) // inp.spec.page_size) for c in inp.context_lens)
    for S in (1, 2, 3, 5, nmax, nmax + 3):
        po, pl = oracle.decode_split(oi, inp.scale, S)
        o2, l2 = oracle.combine(po, pl)
        np.testing.assert_allclose(o2, out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l2, lse, rtol=0, atol=1e-12)


def test_split_ranges_cover_pages_once():
    for n in range(0, 40):
        for S in range(1, 12):
            r = oracle.split_page_ranges(n, S)
            assert len(r) == S
            covered = [p for (a, b) in r for p in range(a, b)]
            assert covered == list(range(n))


def test_combine_all_empty_gives_zero_and_minus_inf():
    po = np.random.default_rng(0).standard_normal((2, 3, 4))
    pl = np.full((2, 3), -np.inf)
    o, l = oracle.combine(po, pl)
    assert np.all(o == 0) and np.all(l == -np.inf)


def test_gqa_equals_mha_with_repeated_kv_heads():
    inp = gen.make_inputs(small_spec(num_q_heads=8, num_kv_heads=2))
    oi = ora_inputs(inp)
    out, lse = oracle.decode(oi, inp.scale)
    mha = dict(oi)
    for name in ("k_cache", "v_cache"):
        mha[name] = np.repeat(oi[name], 4, axis=2)
    out2, lse2 = oracle.decode(mha, inp.scale)
    # Each MHA head is a 1-row product: equal up to fp64 rounding order.
    np.testing.assert_allclose(out, out2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-14)
    # A wrong head mapping (h % Hkv) would pair head 1 with kv head 1.
    K0 = oracle.keys_values(oi, 0, 0)[0]
    q1 = oracle.bf16_bits_to_f64(oi["q"][0, 0, 1])
    ref = np.log(np.exp(inp.scale * K0 @ q1).sum())
    assert abs(lse[0, 0, 1] - ref) < 1e-12


def test_draft_block_equals_extra_pages():
    """Scratch tokens attended like extra paged tokens appended to the sequence."""
    spec = small_spec(draft_scratch=True, q_tokens=4, page_size=16, context_lens=(32, 16, 48))
    inp = gen.make_inputs(spec)
    oi = ora_inputs(inp)
    out, lse = oracle.decode(oi, inp.scale)
    B, T, Hkv, D, P = 3, 4, 2, 32, 16
    pool = oi["k_cache"].shape[0]
    k = np.concatenate([oi["k_cache"], np.zeros((B, P, Hkv, D), np.uint16)], 0)
    v = np.concatenate([oi["v_cache"], np.zeros((B, P, Hkv, D), np.uint16)], 0)
    bt = np.concatenate([oi["block_tables"], np.full((B, 1), -1, np.int32)], 1)
    ctx = oi["context_lens"].copy()
    for b in range(B):
        k[pool + b, :T] = oi["k_scratch"][b]
        v[pool + b, :T] = oi["v_scratch"][b]
        bt[b, ctx[b] // P] = pool + b
        ctx[b] += T
    plain = dict(oi, k_cache=k, v_cache=v, block_tables=bt, context_lens=ctx,
                 k_scratch=None, v_scratch=None)
    out2, lse2 = oracle.decode(plain, inp.scale)
    np.testing.assert_allclose(out, out2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-13)


def masked_by_extra_tokens(oi, scale, bs):
    """Draft token t of a block-masked draft block computed as a plain decode
    (no scratch) whose sequence carries, after its prefix, the scratch
    tokens that t may see, appended as extra paged tokens."""
    B, T, Hq, D = oi["q"].shape
    P = oi["k_cache"].shape[1]
    Hkv = oi["k_cache"].shape[2]
    out = np.full((B, T, Hq, D), np.nan)
    lse = np.full((B, T, Hq), np.nan)
    for t in range(T):
        n = T if bs is None else min(T, (t // bs + 1) * bs)
        pool = oi["k_cache"].shape[0]
        k = np.concatenate([oi["k_cache"], np.zeros((B, P, Hkv, D), np.uint16)], 0)
        v = np.concatenate([oi["v_cache"], np.zeros((B, P, Hkv, D), np.uint16)], 0)
        bt = np.concatenate([oi["block_tables"], np.full((B, 1), -1, np.int32)], 1)
        ctx = oi["context_lens"].copy()
        for b in range(B):
            assert ctx[b] % P == 0  # the extra tokens start a fresh page
            k[pool + b, :n] = oi["k_scratch"][b, :n]
            v[pool + b, :n] = oi["v_scratch"][b, :n]
            bt[b, ctx[b] // P] = pool + b
            ctx[b] += n
        plain = dict(oi, q=oi["q"][:, t:t + 1], k_cache=k, v_cache=v, block_tables=bt, context_lens=ctx,
                     k_scratch=None, v_scratch=None, draft_block=None)
        o, l = oracle.decode(plain, scale)
        out[:, t], lse[:, t] = o[:, 0], l[:, 0]
    return out, lse


@pytest.mark.parametrize("bs", [1, 2, 3, 5, 8])
def test_block_masked_draft_equals_extra_tokens(bs):
    """Causal (bs 1) and block-causal draft blocks: token t sees the first
    min(T, (t // bs + 1) * bs) scratch tokens; bs >= T is the unmasked mode."""
    spec = small_spec(draft_scratch=True, q_tokens=5, page_size=16, context_lens=(32, 0, 48))
    inp = gen.make_inputs(spec)
    oi = dict(ora_inputs(inp), draft_block=bs)
    out, lse = oracle.decode(oi, inp.scale)
    out2, lse2 = masked_by_extra_tokens(oi, inp.scale, bs)
    np.testing.assert_allclose(out, out2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-13)
    if bs >= 5:
        ref, ref_lse = oracle.decode(ora_inputs(inp), inp.scale)
        np.testing.assert_array_equal(out, ref)
    # the split variant keeps the mask on the last split
    po, pl = oracle.decode_split(oi, inp.scale, 3)
    co, cl = oracle.combine(po, pl)
    np.testing.assert_allclose(co, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(cl, lse, rtol=0, atol=1e-12)


def test_planted_mask_slip_is_caught(monkeypatch):
    """Seeing one scratch token too many fails the extra-token pin."""
    orig = pa_oracle.visible_scratch
    monkeypatch.setattr(pa_oracle, "visible_scratch", lambda inputs, t: min(orig(inputs, t) + 1,
                                                                             inputs["k_scratch"].shape[1]))
    with pytest.raises(AssertionError):
        test_block_masked_draft_equals_extra_tokens(1)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def _bits(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def tiny_problem(q, keys, values, scale, page_size=1, reverse_pages=True):
    """One sequence, one head; keys/values [N, D] exactly representable in bf16.
    Pages are stored in reverse physical order to exercise the table."""
    q = np.asarray(q, np.float32)
    keys = np.asarray(keys, np.float32)
    values = np.asarray(values, np.float32)
    N, D = keys.shape
    n = -(-N // page_size)
    kc = np.zeros((n, page_size, 1, D), np.float32)
    vc = np.zeros((n, page_size, 1, D), np.float32)
    order = list(range(n))[::-1] if reverse_pages else list(range(n))
    for j in range(N):
        kc[order[j // page_size], j % page_size, 0] = keys[j]
        vc[order[j // page_size], j % page_size, 0] = values[j]
    oi = dict(q=_bits(q.reshape(1, 1, 1, D)), k_cache=_bits(kc), v_cache=_bits(vc),
              block_tables=np.array([order], np.int32), context_lens=np.array([N], np.int32),
              kv_format="bf16")
    out, lse = oracle.decode(oi, scale)
    return out[0, 0, 0], lse[0, 0, 0]


def test_two_keys_closed_form():
    # s = (0, 1): weights 1/(1+e), e/(1+e); one-hot values give them back.
    out, lse = tiny_problem([1, 0], [[0, 0], [1, 0]], [[1, 0], [0, 1]], scale=1.0)
    e = math.e
    assert abs(out[0] - 1 / (1 + e)) < 1e-15 and abs(out[1] - e / (1 + e)) < 1e-15
    assert abs(lse - math.log(1 + e)) < 1e-15


def test_single_key():
    rng = np.random.default_rng(1)
    q, k, v = (rng.standard_normal(8).astype(np.float32) for _ in range(3))
    qb, kb, vb = (oracle.bf16_bits_to_f64(_bits(x)) for x in (q, k, v))
    out, lse = tiny_problem(q, [k], [v], scale=0.3)
    np.testing.assert_array_equal(out, vb)
    assert abs(lse - 0.3 * float(qb @ kb)) < 1e-14


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(8), rng.standard_normal(8)
    V = rng.standard_normal((37, 8))
    out, lse = tiny_problem(q, [k] * 37, V, scale=0.25, page_size=16)
    vb = oracle.bf16_bits_to_f64(_bits(V))
    np.testing.assert_allclose(out, vb.mean(0), rtol=0, atol=1e-14)
    s = 0.25 * float(oracle.bf16_bits_to_f64(_bits(q)) @ oracle.bf16_bits_to_f64(_bits(k)))
    assert abs(lse - (s + math.log(37))) < 1e-13


def test_zero_query_gives_mean_and_log_count():
    rng = np.random.default_rng(3)
    K, V = rng.standard_normal((50, 16)), rng.standard_normal((50, 16))
    out, lse = tiny_problem(np.zeros(16), K, V, scale=0.7, page_size=16)
    np.testing.assert_allclose(out, oracle.bf16_bits_to_f64(_bits(V)).mean(0), rtol=0, atol=1e-14)
    assert abs(lse - math.log(50)) < 1e-14


def test_constant_values_pass_through():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((29, 16))
    out, _ = tiny_problem(rng.standard_normal(16), K, np.full((29, 16), 1.5), scale=0.5, page_size=16)
    np.testing.assert_allclose(out, 1.5, rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(5)
    K = rng.standard_normal((40, 16)) * 0.1
    V = rng.standard_normal((40, 16))
    q = np.zeros(16)
    q[0] = 8.0
    K[17, 0] = 8.0  # score 64 * scale vs ~ +-0.8 * scale for the others
    out, _ = tiny_problem(q, K, V, scale=1.0, page_size=16)
    np.testing.assert_allclose(out, oracle.bf16_bits_to_f64(_bits(V[17])), rtol=0, atol=1e-20 + 1e-24)


def test_one_hot_values_give_probabilities_summing_to_one():
    rng = np.random.default_rng(6)
    N = 16
    out, _ = tiny_problem(rng.standard_normal(N), rng.standard_normal((N, N)), np.eye(N),
                          scale=0.5, page_size=16)
    assert abs(out.sum() - 1.0) < 1e-14 and np.all(out > 0)


# ---------------------------------------------------------------------------
# Planted slips: a wrong oracle fails the pins above
# ---------------------------------------------------------------------------

def test_planted_wrong_slot_index_is_caught(monkeypatch):
    inp = gen.make_inputs(small_spec())
    ref_out, _ = torch_reference(inp)
    orig = pa_oracle._paged_rows

    def slipped(cache, scales, kv_format, bt_row, ctx, page_size, g):
        # Reads pages in the reverse logical order.
        n = -(-ctx // page_size)
        return orig(cache, scales, kv_format, bt_row[:n][::-1].copy(), ctx, page_size, g)

    monkeypatch.setattr(pa_oracle, "_paged_rows", slipped)
    out, _ = oracle.decode(ora_inputs(inp), inp.scale)
    assert np.abs(out - ref_out).max() > 1e-3


def test_planted_dropped_scale_is_caught(monkeypatch):
    inp = gen.make_inputs(small_spec(kv_format="fp8", head_dim=64))
    ref_out, ref_lse = torch_reference(inp)
    oi = ora_inputs(inp)
    oi["k_scale"] = np.ones_like(oi["k_scale"])
    _, lse = oracle.decode(oi, inp.scale)
    assert np.abs(lse - ref_lse).max() > 1e-3


def test_planted_wrong_combine_weight_is_caught(monkeypatch):
    inp = gen.make_inputs(small_spec())
    oi = ora_inputs(inp)
    out, _ = oracle.decode(oi, inp.scale)
    po, pl = oracle.decode_split(oi, inp.scale, 3)
    # Averaging partials without LSE weights is wrong whenever splits differ.
    wrong = np.nanmean(np.where(np.isfinite(pl)[..., None], po, np.nan), axis=-2)
    assert np.nanmax(np.abs(wrong - out)) > 1e-3
