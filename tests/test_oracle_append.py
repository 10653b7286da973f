"""Pins of the KV-cache append oracle (CPU only): the e4m3fn encoder against
brute force over all codes and against torch's float8 conversion, the
quantiser against hand-derived examples, and the append against what a
later read of the cache through the block table must return."""

import os

import numpy as np
import pytest
import torch

import oracle
from oracle import kv_append as ka

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TABLE = oracle.e4m3fn_table()


def bf16_bits(x):
    """float values (exact in bf16) -> uint16 bit patterns."""
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def brute_force_encode(y):
    """Nearest finite e4m3fn value of y's sign by exhaustive search; among
    equally near codes the one with an even mantissa (even code)."""
    out = np.empty(len(y), dtype=np.uint8)
    for i, v in enumerate(np.asarray(y, dtype=np.float32).astype(np.float64)):
        neg = bool(np.signbit(v))
        best, bestd = None, None
        for c in range(256):
            if np.isnan(TABLE[c]) or bool(c >> 7) != neg:
                continue
            d = abs(TABLE[c] - v)
            if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
                best, bestd = c, d
        out[i] = best
    return out


def sample_y(rng, n):
    """Float32 magnitudes spanning every binade, the subnormals, exact
    code values, midpoints between neighbouring codes, and past 448."""
    finite = TABLE[~np.isnan(TABLE)]
    pos = np.unique(finite[finite >= 0])
    mids = (pos[:-1] + pos[1:]) / 2
    parts = [
        rng.uniform(-470, 470, n),
        rng.standard_normal(n) * 10.0 ** rng.uniform(-4, 2, n),
        pos, -pos, mids, -mids,
        np.nextafter(mids, 0), np.nextafter(mids, 1000),
        [448.0, 449.0, 463.9, 464.0, 465.0, 1e6, -500.0, 0.0, -0.0],
    ]
    return np.concatenate([np.asarray(p, dtype=np.float64) for p in parts]).astype(np.float32)


def test_encode_equals_brute_force_nearest_even():
    y = sample_y(np.random.default_rng(0), 400)
    np.testing.assert_array_equal(ka.e4m3fn_encode(y), brute_force_encode(y))


def test_encode_equals_torch_conversion_within_range():
    y = sample_y(np.random.default_rng(1), 4000)
    y = y[np.abs(y) <= 448]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ka.e4m3fn_encode(y), ref)


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if not np.isnan(TABLE[c])], dtype=np.uint8)
    np.testing.assert_array_equal(ka.e4m3fn_encode(TABLE[codes].astype(np.float32)), codes)


def read_golden():
    with open(os.path.join(GOLDEN, "e4m3fn_quantise_examples.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            xs, sc, cs = (part.strip() for part in line.split(";"))
            x = [float.fromhex(v) if "0x" in v else float(v) for v in (s.strip() for s in xs.split(","))]
            yield x, float.fromhex(sc), [int(c, 16) for c in cs.split()]


def test_quantise_hand_derived_examples():
    n = 0
    for x, scale, codes in read_golden():
        got_codes, got_scale = ka.quantise_rows(bf16_bits(x))
        assert float(got_scale) == scale, (x, float(got_scale).hex())
        assert got_codes.tolist() == codes, (x, [hex(c) for c in got_codes])
        n += 1
    assert n == 5


def test_quantise_bound_and_amax_code():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((64, 8, 128)) * rng.uniform(0.01, 100, (64, 8, 1))).astype(np.float32)
    bits = bf16_bits(x)
    xb = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes, scale = ka.quantise_rows(bits)
    s = scale.astype(np.float64)[..., None]
    xhat = TABLE[codes] * s
    # half an e4m3 step: 2^-4 relative for normals, 2^-10 * scale absolute below 2^-6 * scale
    bound = np.maximum(np.abs(xb) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(xb - xhat) <= bound)
    top = np.take_along_axis(codes, np.abs(xb).argmax(-1)[..., None], -1)[..., 0]
    assert np.all(top & 0x7F == 0x7E)
    np.testing.assert_array_equal(scale, (np.abs(xb).max(-1).astype(np.float32) / np.float32(448)))


# ---------------------------------------------------------------------------
# Append
# ---------------------------------------------------------------------------

def make_case(rng, kv_format, B=3, T=5, Hkv=2, D=64, P=16, pool=40, ctx=(0, 13, 31), max_blocks=3):
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    perm = rng.permutation(pool)
    k = 0
    for b in range(B):
        need = min(max_blocks, -(-(ctx[b] + T) // P))
        bt[b, :need] = perm[k:k + need]
        k += need
    caches = {}
    if kv_format == "fp8":
        caches["k_cache"] = rng.integers(0, 256, (pool, P, Hkv, D)).astype(np.uint8)
        caches["v_cache"] = rng.integers(0, 256, (pool, P, Hkv, D)).astype(np.uint8)
        caches["k_scale"] = rng.uniform(0.1, 1, (pool, P, Hkv)).astype(np.float32)
        caches["v_scale"] = rng.uniform(0.1, 1, (pool, P, Hkv)).astype(np.float32)
    else:
        caches["k_cache"] = bf16_bits(rng.standard_normal((pool, P, Hkv, D)))
        caches["v_cache"] = bf16_bits(rng.standard_normal((pool, P, Hkv, D)))
    k_new = bf16_bits(rng.standard_normal((B, T, Hkv, D)))
    v_new = bf16_bits(rng.standard_normal((B, T, Hkv, D)))
    return caches, k_new, v_new, bt, np.asarray(ctx, dtype=np.int32), P


@pytest.mark.parametrize("kv_format", ["bf16", "fp8"])
def test_append_lands_where_the_block_table_reads(kv_format):
    rng = np.random.default_rng(3)
    caches, k_new, v_new, bt, ctx, P = make_case(rng, kv_format)
    out = ka.append(caches, k_new, v_new, bt, ctx, P)
    written = np.zeros(caches["k_cache"].shape[:3], dtype=bool)
    for b in range(bt.shape[0]):
        for t in range(k_new.shape[1]):
            j = ctx[b] + t
            page, slot = bt[b, j // P], j % P
            written[page, slot] = True
            for name, new in (("k", k_new), ("v", v_new)):
                if kv_format == "fp8":
                    x = (new[b, t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                    xhat = TABLE[out[name + "_cache"][page, slot]] * out[name + "_scale"][page, slot][:, None]
                    s = out[name + "_scale"][page, slot][:, None].astype(np.float64)
                    assert np.all(np.abs(x - xhat) <= np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-6))
                else:
                    np.testing.assert_array_equal(out[name + "_cache"][page, slot], new[b, t])
    # nothing else changed
    for name in out:
        np.testing.assert_array_equal(out[name][~written], caches[name][~written])


def test_append_skips_positions_past_capacity_and_bad_pages():
    rng = np.random.default_rng(4)
    caches, k_new, v_new, bt, ctx, P = make_case(rng, "bf16", ctx=(40, 44, 0), T=6)
    bt[2, 0] = 10_000  # outside the pool
    out = ka.append(caches, k_new, v_new, bt, ctx, P)
    # sequence 0: positions 40..45 -> 40..47 fit (capacity 48): all 6 written
    np.testing.assert_array_equal(out["k_cache"][bt[0, 2], 8:14], k_new[0])
    # sequence 1: positions 44..49 -> only 44..47 written
    np.testing.assert_array_equal(out["k_cache"][bt[1, 2], 12:16], k_new[1, :4])
    # sequence 2 writes nothing (bad page); total writes = 10 rows per tensor
    changed = np.any(out["k_cache"] != caches["k_cache"], axis=(-1, -2))
    assert changed.sum() == 10


def test_planted_slot_slip_is_caught(monkeypatch):
    """An append that writes one slot too far fails the landing pin."""
    rng = np.random.default_rng(3)
    caches, k_new, v_new, bt, ctx, P = make_case(rng, "bf16")
    orig = ka.append

    def slipped(caches, k_new_bits, v_new_bits, block_tables, context_lens, page_size):
        return orig(caches, k_new_bits, v_new_bits, block_tables, np.asarray(context_lens) + 1, page_size)

    monkeypatch.setattr(ka, "append", slipped)
    with pytest.raises(AssertionError):
        test_append_lands_where_the_block_table_reads("bf16")


def test_planted_rounding_slip_is_caught(monkeypatch):
    """Round-half-up instead of ties-to-even fails the hand-derived examples."""
    def half_up(y):
        y = np.asarray(y, dtype=np.float32)
        a = np.abs(y.astype(np.float64))
        vals = ka._POS_VALUES
        hi = np.clip(np.searchsorted(vals, a), 0, 0x7E)
        lo = np.clip(hi - 1, 0, 0x7E)
        mag = np.where(vals[hi] - a <= a - vals[lo], hi, lo).astype(np.uint8)
        mag = np.where(a >= 448, np.uint8(0x7E), mag)
        return (mag | (np.signbit(y).astype(np.uint8) << 7)).reshape(y.shape)

    monkeypatch.setattr(ka, "e4m3fn_encode", half_up)
    with pytest.raises(AssertionError):
        test_quantise_hand_derived_examples()
