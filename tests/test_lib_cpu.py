"""Host-side checks of the C-ABI library that need no GPU: it builds, loads, and
exports every entry point include/mag.h declares; host-only calls agree with the
pages' closed forms."""
import ctypes
import os
import re

import pytest
import torch

import oracle
import quantized_decode_step_gb300 as mag
from synth.workloads import LLAMA8B, TINY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mag.build()
    return mag.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mag.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mag_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(mag.EXPORTED)


@pytest.mark.parametrize("dt,expect", [(mag.KV_FP16, 131072), (mag.KV_INT8, 66560), (mag.KV_INT4, 40960)])
def test_kv_bytes_per_token(lib, dt, expect):
    cfg = mag.make_config(LLAMA8B, kv_dtype=dt)
    got = mag.kv_bytes_per_token(cfg)
    assert got == expect
    # the values alone follow the closed form of "5. Core modules" 5.4; the rest is per-token metadata
    values = oracle.kv_bytes_per_token(32, 8, 128, {0: 2, 1: 1, 2: 0.5}[dt])
    meta = 2 * 32 * 8 * {0: 0, 1: 2, 2: 16}[dt]
    assert got == values + meta
    assert oracle.kv_block_bytes(8, 128, dt) * 1 == 16 * got // 32  # one block of one layer holds 16 tokens


def test_bad_config_rejected_on_host(lib):
    cfg = mag.make_config(TINY)
    cfg.head_dim = 96
    h = ctypes.c_void_p()
    assert lib.mag_create(ctypes.byref(cfg), None, ctypes.byref(h)) == mag.ERR_INVALID_ARG
    assert not h.value
    cfg = mag.make_config(TINY)
    cfg.n_kv_heads = 3
    assert lib.mag_create(ctypes.byref(cfg), None, ctypes.byref(h)) == mag.ERR_INVALID_ARG
    cfg = mag.make_config(TINY, max_batch=17)
    assert lib.mag_create(ctypes.byref(cfg), None, ctypes.byref(h)) == mag.ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device error path")
def test_create_without_device_reports_cuda_error(lib):
    cfg = mag.make_config(TINY)
    h = ctypes.c_void_p()
    assert lib.mag_create(ctypes.byref(cfg), None, ctypes.byref(h)) == mag.ERR_CUDA
    assert not h.value


def _c_layout(struct, fields):
    """sizeof and offsetof of a struct of include/mag.h, from a host C program built with gcc."""
    import subprocess
    import tempfile
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "mag.h"', 'int main(void) {',
             f'  printf("%zu\\n", sizeof({struct}));']
    lines += [f'  printf("%zu\\n", offsetof({struct}, {f}));' for f in fields]
    lines += ['  return 0;', '}']
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        with open(src, "w") as f:
            f.write("\n".join(lines) + "\n")
        subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()
    return int(out[0]), [int(x) for x in out[1:]]


@pytest.mark.parametrize("struct,cls", [("mag_config", "Config"), ("mag_memory_stats", "MemoryStats"),
                                        ("mag_adapt_config", "AdaptConfig"), ("mag_profile", "Profile"),
                                        ("mag_arena_tensor", "ArenaTensor"), ("mag_step_stats", "StepStats")])
def test_binding_structs_match_the_header(struct, cls):
    """The ctypes mirrors of the header's structs have the C compiler's size and field offsets."""
    c = getattr(mag, cls)
    fields = [f for f, _ in c._fields_]
    size, offs = _c_layout(struct, fields)
    assert ctypes.sizeof(c) == size, (struct, ctypes.sizeof(c), size)
    assert [getattr(c, f).offset for f in fields] == offs, struct


def test_noalloc_documented_limits_follow_the_slab_rule():
    """The K limits the header states for mag_load_weights_f32_noalloc follow from its slab rule: one slab of
    whole 16-row tiles (QKV: one head, d/16 tiles) of 16 * ceil(K/32) * 20 bytes each must fit the scratch."""
    import re
    hdr = open(os.path.join(ROOT, "include", "mag.h")).read()
    doc = hdr[hdr.index("mag_load_weights with MAG_FMT_F32_DENSE"):hdr.index("mag_status mag_load_weights_f32_noalloc")]
    doc = " ".join(doc.replace("*", " ").split())
    scratch_src = open(os.path.join(ROOT, "quantized_decode_step_gb300", "csrc", "noalloc.h")).read()
    m = re.search(r"kNoAllocScratchBytes = (\d+)u << (\d+);", scratch_src)
    scratch = int(m.group(1)) << int(m.group(2))
    assert f"{scratch >> 20} MiB" in doc

    def max_k(tiles_per_slab):
        return 32 * (scratch // (16 * 20 * tiles_per_slab))

    stated = [int(x.replace(",", "")) for x in re.findall(r"(\d{2,3},\d{3})", doc)]
    assert stated == [max_k(1), max_k(128 // 16), max_k(64 // 16)], stated
    # one more group past each limit no longer fits
    for tiles, k in ((1, max_k(1)), (8, max_k(8)), (4, max_k(4))):
        assert 16 * 20 * tiles * (k // 32) <= scratch < 16 * 20 * tiles * (k // 32 + 1)
