"""Several host threads calling the library at once, each on its own CUDA
stream, from a fresh process (so that they also race on the library's
one-time set-up per device): every result equals the same call made alone,
bit for bit."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import threading
import torch
from paged_kv_attention_15_gb300 import binding as pb
from paged_kv_attention_15_gb300 import inputs as gen

specs = [
    gen.custom_spec(batch=5, q_tokens=1, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                    ctx_range=(1, 900), seed=41),
    gen.custom_spec(batch=4, q_tokens=1, num_q_heads=32, num_kv_heads=2, head_dim=256, page_size=16,
                    ctx_range=(1, 900), kv_format="fp8", seed=42),
    gen.custom_spec(batch=3, q_tokens=8, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                    ctx_range=(0, 500), draft_scratch=True, draft_block=2, seed=43),
    gen.custom_spec(batch=4, q_tokens=2, num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=64,
                    ctx_range=(1, 900), kv_format="f16", seed=44),
]
inputs = [gen.make_inputs(s).to("cuda") for s in specs]
app = gen.make_append_inputs(gen.AppendSpec("t", batch=6, new_tokens=9, num_kv_heads=2, head_dim=128,
                                            page_size=16, ctx_range=(0, 300), kv_format="fp8", seed=45))
app_a, app_b = app.to("cuda"), app.to("cuda")
torch.cuda.synchronize()

results = [None] * (len(inputs) + 1)
start = threading.Barrier(len(inputs) + 1)

def decode_worker(i):
    st = torch.cuda.Stream()
    start.wait()
    with torch.cuda.stream(st):
        for _ in range(3):
            out, lse = pb.decode_inputs(inputs[i], stream=st)
    st.synchronize()
    results[i] = (out.clone(), lse.clone())

def append_worker():
    st = torch.cuda.Stream()
    start.wait()
    with torch.cuda.stream(st):
        pb.kv_append(app_a.k_new, app_a.v_new, app_a.block_tables, app_a.context_lens, app_a.k_cache,
                     app_a.v_cache, k_scale=app_a.k_scale, v_scale=app_a.v_scale, stream=st)
    st.synchronize()

threads = [threading.Thread(target=decode_worker, args=(i,)) for i in range(len(inputs))]
threads.append(threading.Thread(target=append_worker))
for t in threads:
    t.start()
for t in threads:
    t.join()

for i, inp in enumerate(inputs):
    out, lse = pb.decode_inputs(inp)
    torch.cuda.synchronize()
    assert torch.equal(out, results[i][0]) and torch.equal(lse, results[i][1]), f"decode {i} differs"
pb.kv_append(app_b.k_new, app_b.v_new, app_b.block_tables, app_b.context_lens, app_b.k_cache, app_b.v_cache,
             k_scale=app_b.k_scale, v_scale=app_b.v_scale)
torch.cuda.synchronize()
for n in ("k_cache", "v_cache", "k_scale", "v_scale"):
    assert torch.equal(getattr(app_a, n), getattr(app_b, n)), f"append {n} differs"
assert pb.device_error() == 0
print("threads ok")
"""


def test_concurrent_host_threads_match_single_calls():
    res = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "threads ok" in res.stdout
