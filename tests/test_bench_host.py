"""Host-side pieces of bench.py: the algorithmic byte count (the GB/s
numerator) and the reference arm's JSON line (the oracle on host cores)."""

import io
import json
from contextlib import redirect_stdout

import bench
from paged_kv_attention_15_gb300 import inputs as gen


def test_algorithmic_bytes_by_hand():
    spec = gen.custom_spec(batch=2, q_tokens=1, num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16,
                           context_lens=(37, 100), seed=1)
    inp = gen.make_inputs(spec)
    kv = 2 * (37 + 100) * 2 * 64 * 2          # K and V rows of valid tokens, 2 kv heads, bf16
    table = (3 + 7) * 4                        # block-table entries in use
    rows = 2 * 1 * 4
    qo = rows * 64 * 2 * 2 + rows * 4 + 2 * 4  # q, out, lse, context_lens
    assert bench.algorithmic_bytes(inp) == kv + table + qo


def test_algorithmic_bytes_fp8_and_scratch():
    spec = gen.custom_spec(batch=1, q_tokens=2, num_q_heads=2, num_kv_heads=1, head_dim=128, page_size=16,
                           context_lens=(20,), kv_format="fp8", seed=1)
    inp = gen.make_inputs(spec)
    expect = 2 * 20 * 128 * 1 + 2 * 20 * 4 + 2 * 4 + (4 * 128 * 2 * 2 + 4 * 4 + 4)
    assert bench.algorithmic_bytes(inp) == expect
    spec = gen.custom_spec(batch=1, q_tokens=2, num_q_heads=2, num_kv_heads=1, head_dim=64, page_size=16,
                           context_lens=(20,), draft_scratch=True, seed=1)
    inp = gen.make_inputs(spec)
    expect = 2 * 20 * 64 * 2 + 2 * 4 + (4 * 64 * 2 * 2 + 4 * 4 + 4) + 2 * 2 * 64 * 2
    assert bench.algorithmic_bytes(inp) == expect


def test_unit_bytes_sum_to_call_bytes():
    spec = gen.SPECS["tiny"]
    inp = gen.make_inputs(spec)
    total = sum(bench.unit_bytes(spec, int(c)) for c in inp.context_lens for _ in range(spec.num_kv_heads))
    assert total + spec.batch * 4 == bench.algorithmic_bytes(inp)


def test_reference_arm_prints_the_contract_line():
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "3",
                         "--reference-seconds", "0.5"])
    assert rc == 0
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["metric"] == bench.METRIC and line["steps"] == 2 and line["warmup"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["nproc"] >= 1 and line["cpu_baseline"]["threads_per_process"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_append_sample_on_own_pages_matches_whole_pool():
    """The CPU-baseline sampler gives the append oracle one sequence's pages
    with a renumbered block table: the rows it writes equal those of the
    oracle's append over the whole pool."""
    import numpy as np

    from oracle import kv_append as ka

    spec = gen.AppendSpec("t", batch=3, new_tokens=20, num_kv_heads=2, head_dim=64, page_size=16,
                          context_lens=(5, 30, 0), kv_format="fp8", seed=3)
    host = gen.make_append_inputs(spec)
    bits = host.numpy_bits()
    names = ("k_cache", "v_cache", "k_scale", "v_scale")
    full = ka.append({n: bits[n] for n in names}, bits["k_new"], bits["v_new"], bits["block_tables"],
                     bits["context_lens"], 16)
    for b in range(3):
        row = bits["block_tables"][b:b + 1]
        pages = row[row >= 0]
        local = np.where(row >= 0, np.cumsum(row >= 0, axis=1) - 1, -1).astype(np.int32)
        own = ka.append({n: bits[n][pages] for n in names}, bits["k_new"][b:b + 1], bits["v_new"][b:b + 1], local,
                        bits["context_lens"][b:b + 1], 16)
        for n in names:
            np.testing.assert_array_equal(own[n], full[n][pages])
    secs, nbytes, desc = bench.append_oracle_run(host, 0.5)
    assert secs > 0 and nbytes > 0 and "sequence" in desc


def test_append_bytes_by_hand():
    spec = gen.AppendSpec("t", batch=2, new_tokens=20, num_kv_heads=2, head_dim=64, page_size=16,
                          context_lens=(5, 30), seed=3)
    host = gen.make_append_inputs(spec)
    rows = 2 * 20 * 2 * 2                       # (token, kv head) rows of K and V
    pages = ((5 + 19) // 16 - 5 // 16 + 1) + ((30 + 19) // 16 - 30 // 16 + 1)  # 2 + 3 table entries
    assert bench.append_bytes(host) == rows * (2 * 64 + 2 * 64) + pages * 4 + 2 * 4
    fp8 = gen.make_append_inputs(gen.AppendSpec("t", batch=2, new_tokens=20, num_kv_heads=2, head_dim=128,
                                                page_size=16, context_lens=(5, 30), kv_format="fp8", seed=3))
    assert bench.append_bytes(fp8) == rows * (2 * 128 + 128 + 4) + pages * 4 + 2 * 4


def test_all_cores_oracle_pool_covers_every_unit_once():
    """The all-cores CPU baseline: two spawned processes share the workload
    through shared memory and split its units; with a large budget they do
    every unit exactly once, so their bytes equal the one-core run's."""
    spec = gen.custom_spec(batch=3, q_tokens=1, num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16,
                           context_lens=(37, 100, 5), seed=2)
    inp = gen.make_inputs(spec)
    per_key = bench.oracle_seconds_per_key(inp)
    s1, b1, _ = bench.oracle_sample_run(inp, 60.0, per_key=per_key)
    pool = bench.OraclePool(inp, 2)
    try:
        wall, b2, desc = pool.run(60.0, per_key)
    finally:
        pool.close()
    assert b2 == b1 == sum(bench.unit_bytes(spec, c) for c in (37, 100, 5) for _ in range(2))
    assert wall > 0 and "6 (sequence, kv head) unit(s)" in desc and "2 processes" in desc
