"""The C-ABI library: it builds, loads, exports every function the header
declares, and rejects bad arguments before touching the GPU."""

import ctypes
import os

import pytest

from paged_kv_attention_15_gb300 import binding as pb
from paged_kv_attention_15_gb300 import build as pbuild


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pb.LIB_PATH):
        pbuild.build()
    return pb.lib()


def shape(**kw):
    base = dict(batch=2, q_tokens=1, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                num_pages=64, max_blocks_per_seq=8)
    base.update(kw)
    return pb.PaShape(*[base[f] for f, _ in pb.PaShape._fields_])


FAKE = 1 << 20  # an aligned, never dereferenced address


def call_decode(lib, s, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, scale=0.1, out=FAKE, lse=None, splits=1, ws=None, wsb=0)
    a.update(kw)
    return lib.pa_decode(a["q"], a["k"], a["v"], a["bt"], a["cl"], ctypes.byref(s), a["scale"], a["out"],
                         a["lse"], a["splits"], a["ws"], a["wsb"], None)


def test_exports_every_declared_function(lib):
    names = pb.header_functions()
    assert {"pa_decode", "pa_decode_fp8", "pa_decode_reduce", "pa_decode_tidar"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(pb._SIGNATURES) == set(names)


def test_status_strings(lib):
    for st in range(5):
        assert pb.status_string(st)
    assert pb.status_string(99) == "unknown status"


def test_shape_validation_before_any_launch(lib):
    assert call_decode(lib, shape(num_q_heads=6, num_kv_heads=4)) == pb.PA_ERR_INVALID_ARG
    assert call_decode(lib, shape(head_dim=96)) == pb.PA_ERR_UNSUPPORTED
    assert call_decode(lib, shape(page_size=8)) == pb.PA_ERR_UNSUPPORTED
    assert call_decode(lib, shape(page_size=48)) == pb.PA_ERR_UNSUPPORTED
    assert call_decode(lib, shape(num_q_heads=128, num_kv_heads=1)) == pb.PA_ERR_UNSUPPORTED  # 128 rows
    assert call_decode(lib, shape(num_q_heads=64, num_kv_heads=1, head_dim=256)) == pb.PA_ERR_UNSUPPORTED
    assert call_decode(lib, shape(q_tokens=0)) == pb.PA_ERR_INVALID_ARG
    assert call_decode(lib, shape(num_pages=0)) == pb.PA_ERR_INVALID_ARG
    assert call_decode(lib, shape(batch=-1)) == pb.PA_ERR_INVALID_ARG
    assert call_decode(lib, shape(max_blocks_per_seq=1 << 28, page_size=256)) == pb.PA_ERR_INVALID_ARG
    assert lib.pa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, None, 0.1, FAKE, None, 1, None, 0, None) == pb.PA_ERR_INVALID_ARG


def test_pointer_and_argument_validation(lib):
    s = shape()
    assert call_decode(lib, s, q=None) == pb.PA_ERR_INVALID_ARG
    assert call_decode(lib, s, out=None) == pb.PA_ERR_INVALID_ARG
    assert call_decode(lib, s, k=FAKE + 8) == pb.PA_ERR_INVALID_ARG  # not 16-byte aligned
    assert call_decode(lib, s, scale=float("nan")) == pb.PA_ERR_INVALID_ARG
    assert call_decode(lib, s, scale=float("inf")) == pb.PA_ERR_INVALID_ARG
    assert call_decode(lib, s, splits=-1) == pb.PA_ERR_INVALID_ARG
    # Nothing to do: OK without touching the device.
    assert call_decode(lib, shape(batch=0)) == pb.PA_OK


def test_fp8_and_tidar_validation(lib):
    s = shape()
    assert lib.pa_decode_fp8(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, FAKE, None, 1,
                             None, 0, None) == pb.PA_ERR_INVALID_ARG
    assert lib.pa_decode_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(shape(head_dim=64)), 0.1,
                             FAKE, None, 1, None, 0, None) == pb.PA_ERR_UNSUPPORTED
    assert lib.pa_decode_tidar(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, FAKE, None, 1,
                               None, 0, None) == pb.PA_ERR_INVALID_ARG
    for bs in (0, -3):
        assert lib.pa_decode_tidar_masked(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, bs, FAKE,
                                          None, 1, None, 0, None) == pb.PA_ERR_INVALID_ARG
    assert lib.pa_decode_tidar_masked(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, ctypes.byref(s), 0.1, 2, FAKE,
                                      None, 1, None, 0, None) == pb.PA_ERR_INVALID_ARG
    assert lib.pa_decode_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             ctypes.byref(shape(q_tokens=8, num_q_heads=16, num_kv_heads=2)), 0.1, FAKE, None, 1,
                             None, 0, None) == pb.PA_ERR_UNSUPPORTED  # fp8: at most 32 rows


def test_reduce_validation(lib):
    s = shape()
    assert lib.pa_decode_reduce(None, FAKE, 3, ctypes.byref(s), FAKE, None, None) == pb.PA_ERR_INVALID_ARG
    assert lib.pa_decode_reduce(FAKE, FAKE, 0, ctypes.byref(s), FAKE, None, None) == pb.PA_ERR_INVALID_ARG
    assert lib.pa_decode_reduce(FAKE, FAKE, 3, ctypes.byref(shape(head_dim=6)), FAKE, None,
                                None) == pb.PA_ERR_INVALID_ARG
    assert lib.pa_decode_reduce(FAKE, FAKE, 3, ctypes.byref(shape(batch=0)), FAKE, None, None) == pb.PA_OK


def test_explicit_split_workspace_size(lib):
    s = shape(batch=3, q_tokens=2, num_q_heads=8, head_dim=64)
    assert lib.pa_decode_workspace_size(ctypes.byref(s), 1) == 0
    rows = 3 * 2 * 8 * 5
    expect = (rows * 64 * 4 + 255) // 256 * 256 + (rows * 4 + 255) // 256 * 256
    assert lib.pa_decode_workspace_size(ctypes.byref(s), 5) == expect
    assert lib.pa_decode_workspace_size(ctypes.byref(shape(head_dim=96)), 5) == 0
    assert lib.pa_decode_workspace_size(ctypes.byref(s), -2) == 0


def test_choose_splits_rejects_bad_shapes(lib):
    assert lib.pa_decode_choose_splits(ctypes.byref(shape(head_dim=96)), 0) == -1
    assert lib.pa_decode_choose_splits(ctypes.byref(shape(head_dim=64)), 1) == -1  # fp8 needs D >= 128
    assert lib.pa_decode_choose_splits(ctypes.byref(shape(q_tokens=0)), 0) == -1


def test_kernel_choice_per_path(lib):
    """Host-only kernel choice: by default the paired-role kernel for fp8
    caches and the warp-level kernel otherwise; with a path forced, the
    shapes that kernel covers run it and the others keep the warp-level
    kernel; invalid paths are rejected."""
    bf16, fp8, f16, draft = 0, 1, 2, 3
    qrow_shapes = [  # (shape, format): 64 query rows per unit, D = 128, 16-bit
        (shape(q_tokens=8, num_q_heads=32, num_kv_heads=8, num_pages=400, max_blocks_per_seq=100), draft),
        (shape(q_tokens=16, num_q_heads=32, num_kv_heads=8, num_pages=400, max_blocks_per_seq=100), draft),
        (shape(q_tokens=1, num_q_heads=64, num_kv_heads=2), bf16),
        (shape(q_tokens=1, num_q_heads=64, num_kv_heads=1), f16),
    ]
    other = [
        (shape(), bf16),                                              # G * T = 4
        (shape(q_tokens=1, num_q_heads=64, num_kv_heads=2), fp8),     # fp8
        (shape(q_tokens=1, num_q_heads=64, num_kv_heads=2, head_dim=64), bf16),   # D = 64
        (shape(q_tokens=3, num_q_heads=16, num_kv_heads=1), draft),   # 48 rows per kv head
        (shape(q_tokens=1, num_q_heads=32, num_kv_heads=1), bf16),    # G = 32 with one kv head: no pair
    ]
    try:
        for s, fmt in qrow_shapes + other:  # automatic: fp8 caches on the paired-role kernel
            want = pb.KERNEL_WARP_PAIR if fmt == fp8 else pb.KERNEL_WARP_MMA
            assert lib.pa_decode_kernel_for(ctypes.byref(s), fmt) == want
        pb.set_kernel_path(pb.KERNEL_WARP_MMA)
        for s, fmt in qrow_shapes + other:
            assert lib.pa_decode_kernel_for(ctypes.byref(s), fmt) == pb.KERNEL_WARP_MMA
        pb.set_kernel_path(pb.KERNEL_TCGEN05_QROW)
        for s, fmt in qrow_shapes:
            assert lib.pa_decode_kernel_for(ctypes.byref(s), fmt) == pb.KERNEL_TCGEN05_QROW
        for s, fmt in other:
            assert lib.pa_decode_kernel_for(ctypes.byref(s), fmt) == pb.KERNEL_WARP_MMA
        pb.set_kernel_path(pb.KERNEL_WARP_PAIR)
        pair_shapes = [  # fp8, up to 32 query rows per kv head
            (shape(q_tokens=1, num_q_heads=32, num_kv_heads=2, head_dim=256), fp8),
            (shape(q_tokens=1, num_q_heads=16, num_kv_heads=1, head_dim=128), fp8),
            (shape(), fp8),
        ]
        for s, fmt in pair_shapes:
            assert lib.pa_decode_kernel_for(ctypes.byref(s), fmt) == pb.KERNEL_WARP_PAIR
        # 16-bit: the paired kernel's units of four row tiles at D = 128
        # (33-64 query rows), the warp-level kernel elsewhere.
        pair16 = qrow_shapes + [other[3]]
        for s, fmt in pair16:
            assert lib.pa_decode_kernel_for(ctypes.byref(s), fmt) == pb.KERNEL_WARP_PAIR
        for s, fmt in other[:3] + other[4:]:
            if fmt != fp8:
                assert lib.pa_decode_kernel_for(ctypes.byref(s), fmt) == pb.KERNEL_WARP_MMA
        assert lib.pa_decode_set_kernel_path(5) == pb.PA_ERR_INVALID_ARG
        assert lib.pa_decode_set_combine(2) == pb.PA_ERR_INVALID_ARG
        assert lib.pa_decode_set_combine(-1) == pb.PA_ERR_INVALID_ARG
        assert lib.pa_decode_set_kernel_path(-1) == pb.PA_ERR_INVALID_ARG
    finally:
        pb.set_kernel_path(pb.KERNEL_AUTO)


def test_heads_per_unit(lib):
    """Host-only unit geometry: a unit grows from one kv head while its page
    box (16 rows x heads x row bytes) stays under 16 KB and an instance
    covers its rows: four heads for the D = 128 GQA shape, eight at D = 64
    (16-bit; fp8 has no such instance), and fewer where the group shape or
    the head count stops it."""
    bf16, fp8, f16 = 0, 1, 2
    cases = [
        (shape(num_q_heads=32, num_kv_heads=8), bf16, 4),                    # gqa: 16 x 4 x 256 B
        (shape(num_q_heads=32, num_kv_heads=8, head_dim=64), bf16, 8),       # gqa_d64: 16 x 8 x 128 B
        (shape(num_q_heads=32, num_kv_heads=8, head_dim=64), f16, 8),
        (shape(num_q_heads=64, num_kv_heads=16, head_dim=64), bf16, 8),
        (shape(num_q_heads=16, num_kv_heads=4, head_dim=64), bf16, 4),       # only four kv heads
        (shape(num_q_heads=64, num_kv_heads=8, head_dim=64), bf16, 4),       # G 8: 64 rows at 8 heads
        (shape(num_q_heads=32, num_kv_heads=8, head_dim=256), bf16, 2),      # 16 x 2 x 512 B
        (shape(num_q_heads=32, num_kv_heads=2, head_dim=256), fp8, 2),       # the fp8 workload's units
        (shape(num_q_heads=32, num_kv_heads=8, page_size=64), bf16, 1),      # a 64-row box of one head: 16 KB
        (shape(num_q_heads=32, num_kv_heads=8, head_dim=64, page_size=64), bf16, 2),   # 64 x 2 x 128 B
        (shape(num_q_heads=32, num_kv_heads=8, head_dim=64, page_size=256), bf16, 1),  # 128-row stage
        (shape(q_tokens=4, num_q_heads=8, num_kv_heads=8, head_dim=64), bf16, 8),      # G 1 x T 4
    ]
    draft = 3
    cases += [  # draft blocks: the scratch stage's T (rounded up to 8) rows per head fit one stage tile
        (shape(q_tokens=8, num_q_heads=32, num_kv_heads=8), draft, 2),                   # TiDAR: 2 x 32 rows
        (shape(q_tokens=16, num_q_heads=32, num_kv_heads=8), draft, 1),                  # the long draft
        (shape(q_tokens=4, num_q_heads=16, num_kv_heads=4, head_dim=256), draft, 2),     # 2 x 8 of 32 rows
        (shape(q_tokens=32, num_q_heads=4, num_kv_heads=4, head_dim=256), draft, 1),     # 32 of 32 rows
    ]
    for s, fmt, want in cases:
        assert lib.pa_decode_heads_per_unit(ctypes.byref(s), fmt) == want, (s.num_kv_heads, s.head_dim, fmt)
    assert lib.pa_decode_heads_per_unit(ctypes.byref(shape(head_dim=96)), bf16) == -1
    assert lib.pa_decode_heads_per_unit(ctypes.byref(shape()), 7) == -1


def test_append_validation(lib):
    def call(s, fp8=False, **kw):
        a = dict(kn=FAKE, vn=FAKE, bt=FAKE, cl=FAKE, kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE)
        a.update(kw)
        if fp8:
            return lib.pa_kv_append_fp8(a["kn"], a["vn"], a["bt"], a["cl"], ctypes.byref(s), a["kc"], a["vc"],
                                        a["ks"], a["vs"], None)
        return lib.pa_kv_append(a["kn"], a["vn"], a["bt"], a["cl"], ctypes.byref(s), a["kc"], a["vc"], None)

    assert call(shape(head_dim=96)) == pb.PA_ERR_UNSUPPORTED
    assert call(shape(q_tokens=0)) == pb.PA_ERR_INVALID_ARG
    assert call(shape(), kn=None) == pb.PA_ERR_INVALID_ARG
    assert call(shape(), vc=FAKE + 8) == pb.PA_ERR_INVALID_ARG          # misaligned
    assert call(shape(), fp8=True, ks=None) == pb.PA_ERR_INVALID_ARG
    assert call(shape(batch=0)) == pb.PA_OK                              # nothing to do, no launch
    assert call(shape(batch=0), fp8=True) == pb.PA_OK
    assert lib.pa_kv_append(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, None) == pb.PA_ERR_INVALID_ARG


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(pb, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(pb, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        pb.lib()


C_PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include "pa_decode.h"

/* Stand-ins for device buffers: aligned host memory that no call below
   reaches, since each one fails (or finishes) in its host-side checks. */
static int32_t buf[64] __attribute__((aligned(256)));

typedef void (*any_fn)(void);

int main(void) {
  void* p = buf;
  const int32_t* ip = buf;
  uint8_t* u8 = (uint8_t*)buf;
  float* fp = (float*)buf;
  pa_shape s = {2, 1, 8, 2, 128, 16, 64, 8};
  pa_shape bad = s;
  bad.head_dim = 96;
  /* every entry point the header declares resolves at link time */
  any_fn entries[] = {
      (any_fn)pa_decode_workspace_size, (any_fn)pa_decode_choose_splits, (any_fn)pa_decode,
      (any_fn)pa_decode_fp8, (any_fn)pa_decode_f16, (any_fn)pa_decode_tidar, (any_fn)pa_decode_tidar_masked,
      (any_fn)pa_decode_reduce, (any_fn)pa_kv_append, (any_fn)pa_kv_append_fp8, (any_fn)pa_decode_noalloc,
      (any_fn)pa_status_string, (any_fn)pa_decode_profile_events, (any_fn)pa_decode_device_error,
      (any_fn)pa_decode_heads_per_unit};
  for (unsigned i = 0; i < sizeof entries / sizeof entries[0]; ++i)
    if (!entries[i]) return 10;
  if (!pa_status_string(PA_OK)[0] || !pa_status_string((pa_status)99)[0]) return 1;
  if (pa_decode(p, p, p, ip, ip, &bad, 0.1f, p, NULL, 1, NULL, 0, NULL) != PA_ERR_UNSUPPORTED) return 2;
  if (pa_decode(NULL, p, p, ip, ip, &s, 0.1f, p, NULL, 1, NULL, 0, NULL) != PA_ERR_INVALID_ARG) return 3;
  if (pa_decode_workspace_size(&s, 1) != 0) return 4;
  if (pa_decode_choose_splits(&bad, 0) != -1) return 5;
  if (pa_kv_append(NULL, p, ip, ip, &s, p, p, NULL) != PA_ERR_INVALID_ARG) return 6;
  if (pa_kv_append_fp8(p, p, ip, ip, &bad, u8, u8, fp, fp, NULL) != PA_ERR_UNSUPPORTED) return 7;
  if (pa_decode_tidar_masked(p, p, p, p, p, ip, ip, &s, 0.1f, 0, p, NULL, 1, NULL, 0, NULL) != PA_ERR_INVALID_ARG)
    return 8;
  if (pa_decode_reduce(fp, fp, 0, &s, p, NULL, NULL) != PA_ERR_INVALID_ARG) return 9;
  if (pa_decode_profile_events(NULL, NULL) != PA_OK) return 11;
  printf("c abi ok %u\n", (unsigned)PA_NOALLOC_SCRATCH_BYTES);
  return 0;
}
"""


def test_header_compiles_as_c99_and_links(lib, tmp_path):
    """A plain C program (gcc, -std=c99, no CUDA headers) includes the header,
    links the library and gets its argument checks through the C ABI."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(pb.LIB_PATH)
    include = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    cc = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-o", str(exe), str(src), "-I", include,
                         "-L", libdir, "-lpadecode", "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr[-3000:]
    res = subprocess.run([str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, (res.returncode, res.stdout, res.stderr)
    assert res.stdout.startswith("c abi ok")
