"""pa_decode_splitkv_noalloc: split-KV decode for callers that may not allocate
device memory (a plugin inside a framework that owns all device memory, a
latency-critical path that cannot afford cudaMalloc's synchronisation, a fixed
memory budget).  It must give what the workspace form gives (pa_decode with a
caller workspace of the same number of segments) and what the CPU oracle gives,
call after call, although its scratch array keeps whatever the previous call left
in it.

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_28_gb300 import _lib
from paged_kv_cache_28_gb300 import workload as wl
from paged_kv_cache_28_gb300.device import DeviceBatch, default_num_segments

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-3, 1e-3      # the bf16 tolerance of the parity tests


def _noalloc(lib, dev, out, num_segments):
    return lib.pa_decode_splitkv_noalloc(
        ctypes.byref(dev.shape), out.data_ptr(), num_segments, dev.q.data_ptr(),
        dev.k_pool.data_ptr(), dev.v_pool.data_ptr(), None, None, dev.block_tables.data_ptr(),
        dev.seq_lens.data_ptr(), ctypes.c_float(dev.batch.sm_scale), dev.err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _close(got, want):
    return np.all(np.abs(got - want) <= ATOL + RTOL * np.abs(want))


def test_noalloc_matches_workspace_form_and_oracle_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    lib = _lib.load()
    rng = np.random.default_rng(5)
    cases = [wl.lognormal_lens(rng, 64, 600, 1, 8192), np.array([3000, 1, 17, 450, 0, 77], np.int32)]
    for i, lens in enumerate(cases):          # two calls in a row, different batches
        batch = wl.build_batch(f"noalloc{i}", lens, Hq=64, Hkv=8, D=128, block_size=16,
                               seed=50 + i)
        dev = DeviceBatch(batch)
        ns = default_num_segments(dev.shape)
        assert _lib.pa_decode_workspace_bytes(dev.shape, ns) <= _lib.PA_NOALLOC_SCRATCH_BYTES
        dev.decode_segments(ns)               # the workspace form, torch-owned workspace
        torch.cuda.synchronize()
        want = dev.out.cpu().numpy()
        got = torch.full_like(dev.out, float("nan"))
        assert _noalloc(lib, dev, got, ns) == _lib.PA_OK
        torch.cuda.synchronize()
        got = got.cpu().numpy()
        assert _close(got, want), f"call {i}: differs from the workspace form"
        ref = oracle.paged_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                  batch.seq_lens, batch.sm_scale, Hkv=batch.Hkv,
                                  block_size=batch.block_size)
        assert _close(got, ref), f"call {i}: differs from the oracle"
        assert dev.read_err() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = _lib.load()
    # 65536 split workers' partials need more than the array holds
    s = _lib.make_shape(256, 64, 8, 128, 16, 60000, 2048)
    assert _lib.pa_decode_workspace_bytes(s, 65536) > _lib.PA_NOALLOC_SCRATCH_BYTES
    st = lib.pa_decode_splitkv_noalloc(ctypes.byref(s), 1 << 20, 65536, 1 << 20, 1 << 20, 1 << 20,
                                       None, None, 1 << 20, 1 << 20, ctypes.c_float(0.1), None,
                                       None)
    assert st == _lib.PA_ERR_INVALID_ARG
    # an empty batch is a no-op whatever the segment count, as for pa_decode
    s0 = _lib.make_shape(0, 64, 8, 128, 16, 60000, 2048)
    assert lib.pa_decode_splitkv_noalloc(ctypes.byref(s0), None, 1 << 20, None, None, None, None,
                                         None, None, None, ctypes.c_float(0.1), None,
                                         None) == _lib.PA_OK
