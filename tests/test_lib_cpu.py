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
