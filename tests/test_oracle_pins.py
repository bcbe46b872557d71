"""Pins of the CPU oracle against facts fixed outside it (CPU only).

Each test checks the oracle against something it does not compute itself:
values printed in the pages' worked examples (tests/golden/*.json, each with
its source), closed forms, invariants, an independent numpy/scipy restatement
of textbook attention on contiguous K/V, and torch's float8_e4m3fn conversion.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from paged_kv_cache_28_gb300 import workload as wl


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- page examples

def test_gqa_mapping_and_cached_scalars(golden_dir):
    g = _golden(golden_dir, "gqa_mapping.json")
    for name, lay in g["layouts"].items():
        mapping = [oracle.kv_head(h, g["query_heads"], lay["kv_heads"])
                   for h in range(g["query_heads"])]
        assert mapping == lay["mapping"], name
        assert oracle.cached_scalars(1, lay["kv_heads"], g["tokens"], g["head_size"]) == \
            lay["cached_scalars"], name


def test_kv_capacity_figures(golden_dir):
    g = _golden(golden_dir, "kv_capacity.json")
    per_tok16 = oracle.cached_scalars(g["layers"], g["kv_heads"], 1, g["head_dim"]) * \
        g["bytes_per_value_16bit"]
    per_tok8 = oracle.cached_scalars(g["layers"], g["kv_heads"], 1, g["head_dim"]) * \
        g["bytes_per_value_8bit"]
    assert per_tok16 == g["bytes_per_token_16bit"]
    assert g["pool_bytes"] // per_tok16 == g["tokens_in_pool_16bit"]
    assert g["pool_bytes"] // per_tok8 == g["tokens_in_pool_8bit"]
    # one layer of the 70B-class shape: 4,096 bytes per token (the bench's unit)
    assert oracle.cached_scalars(1, 8, 1, 128) * 2 == 4096


def test_quantizer_4bit_example(golden_dir):
    g = _golden(golden_dir, "quant4_absmax.json")
    codes, restored, scale = oracle.quantize_absmax_int(g["values"], g["bits"])
    assert codes.tolist() == g["codes"]
    assert np.round(restored, 3).tolist() == g["restored_3dp"]
    assert scale == pytest.approx(1.0 / 7.0, rel=0, abs=1e-15)


def test_quantizer_ties_to_even_and_zero():
    # x/scale = 2.5 and 3.5 with scale 1 (absmax 7): rint gives 2 and 4
    codes, _, _ = oracle.quantize_absmax_int([2.5, 3.5, -2.5, 7.0], 4)
    assert codes.tolist() == [2, 4, -2, 7]
    codes, restored, scale = oracle.quantize_absmax_int([0.0, 0.0], 4)
    assert codes.tolist() == [0, 0] and scale == 0.0 and restored.tolist() == [0.0, 0.0]


def test_allocator_example(golden_dir):
    g = _golden(golden_dir, "paging_allocation.json")
    alloc = wl.BlockAllocator(g["initial_free"])
    a = alloc.allocate(3)
    b = alloc.allocate(2)
    alloc.release(a)
    free_after = list(alloc.free)
    c = alloc.allocate(2)
    assert (a, b, free_after, c) == (g["request_a"], g["request_b"],
                                     g["free_after_a_finishes"], g["request_c"])


# ---------------------------------------------------------------- E4M3 format

def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_to_double(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])
    assert np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])
    assert mine[0x7E] == 448.0 and mine[0xFE] == -448.0
    assert mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6 and mine[0x38] == 1.0
    finite = mine[:0x7F]
    assert np.all(np.diff(finite) > 0)          # magnitudes increase with the code


def _torch_e4m3_satfinite(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.clip(x, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("scale", [1.0, 1.0 / 448.0, 3.0 / 448.0, 0.0173, 7.25, 1e-3])
def test_e4m3_encode_every_bf16(scale):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = wl.bf16_to_float(bits)
    x = x[np.isfinite(x)]
    with np.errstate(over="ignore"):
        y = (x / np.float32(scale)).astype(np.float32)      # overflow -> inf saturates too
    assert np.array_equal(oracle.e4m3_from_float(y), _torch_e4m3_satfinite(y))


def test_e4m3_encode_ties_and_saturation():
    x = np.array([2.0 ** -10, 1.5 * 2.0 ** -9, 1.0625, 1.1875, 448.0, 464.0, 1e30, -1e30,
                  -1e-9, np.nan], dtype=np.float32)
    got = oracle.e4m3_from_float(x).tolist()
    assert got[:4] == [0x00, 0x02, 0x38, 0x3A]      # ties go to the even code
    assert got[4:8] == [0x7E, 0x7E, 0x7E, 0xFE]     # saturation to +-448
    assert got[8] == 0x80                           # sign kept on underflow
    assert got[9] == 0x7F


# ---------------------------------------------------------------- cache write

def test_reshape_and_cache_bf16_canary():
    rng = np.random.default_rng(5)
    nblocks, bs, Hkv, D, T = 9, 16, 2, 64, 7
    k_pool = np.full((nblocks, bs, Hkv, D), 0xBEEF, np.uint16)
    v_pool = np.full((nblocks, bs, Hkv, D), 0xCAFE, np.uint16)
    k_new = rng.integers(0, 65536, (T, Hkv, D)).astype(np.uint16)
    v_new = rng.integers(0, 65536, (T, Hkv, D)).astype(np.uint16)
    slots = np.array([0, 17, -1, 143, 5, -7, 100], np.int64)
    ek, ev = k_pool.copy(), v_pool.copy()
    for t, s in enumerate(slots):
        if s >= 0:
            ek[s // bs, s % bs] = k_new[t]
            ev[s // bs, s % bs] = v_new[t]
    oracle.reshape_and_cache_bf16(k_new, v_new, k_pool, v_pool, slots, bs)
    assert np.array_equal(k_pool, ek) and np.array_equal(v_pool, ev)


def _fp8_setup(D=8, bs=4, nblocks=3, Hkv=1):
    k_pool = np.zeros((nblocks, bs, Hkv, D), np.uint8)
    v_pool = np.zeros((nblocks, bs, Hkv, D), np.uint8)
    k_scale = np.full((nblocks, Hkv), 123.0, np.float32)
    v_scale = np.full((nblocks, Hkv), 123.0, np.float32)
    return k_pool, v_pool, k_scale, v_scale


def _write(vals, slot, pools):
    kp, vp, ks, vs = pools
    x = wl.bf16_bits(np.asarray(vals, np.float32)).reshape(1, 1, -1)
    oracle.reshape_and_cache_fp8(x, x, kp, vp, ks, vs, np.array([slot], np.int64),
                                 kp.shape[1])


def test_fp8_write_first_token_sets_scale():
    pools = _fp8_setup()
    vals = [1.0, -0.5, 0.25, 3.0, -3.0, 0.0, 0.1, 2.0]
    _write(vals, 4, pools)          # block 1, offset 0: a fresh scale
    kp, vp, ks, vs = pools
    scale = np.float32(3.0) / np.float32(448.0)
    assert ks[1, 0] == scale and vs[1, 0] == scale and ks[0, 0] == 123.0
    xf = wl.bf16_to_float(wl.bf16_bits(np.asarray(vals, np.float32)))
    assert np.array_equal(kp[1, 0, 0], _torch_e4m3_satfinite(xf / scale))
    assert kp[1, 0, 0, 3] == 0x7E and kp[1, 0, 0, 4] == 0xFE       # absmax -> +-448
    assert np.array_equal(kp, vp)


def test_fp8_write_smaller_keeps_scale_larger_requantises():
    pools = _fp8_setup()
    kp, vp, ks, vs = pools
    _write([1.0, 0.5, -0.25, 0.0, 0, 0, 0, 0], 0, pools)
    s0 = np.float32(1.0) / np.float32(448.0)
    row0 = kp[0, 0, 0].copy()
    _write([0.5, 0.125, 0, 0, 0, 0, 0, 0], 1, pools)        # smaller: scale unchanged
    assert ks[0, 0] == s0 and np.array_equal(kp[0, 0, 0], row0)
    assert kp[0, 1, 0, 0] == _torch_e4m3_satfinite(np.array([np.float32(0.5) / s0]))[0]
    _write([2.0, 0, 0, 0, 0, 0, 0, 0], 2, pools)            # larger: rows 0, 1 re-encoded
    s1 = np.float32(2.0) / np.float32(448.0)
    assert ks[0, 0] == s1
    restored0 = (torch.from_numpy(row0).view(torch.float8_e4m3fn).to(torch.float32).numpy()
                 * s0).astype(np.float32)
    assert np.array_equal(kp[0, 0, 0], _torch_e4m3_satfinite(restored0 / s1))
    # the value 1.0 now sits at code 224 (half the range), 2.0 at 448
    assert kp[0, 0, 0, 0] == _torch_e4m3_satfinite(np.array([224.0], np.float32))[0]
    assert kp[0, 2, 0, 0] == 0x7E
    # scale equals absmax over everything written / 448
    assert ks[0, 0] == np.float32(2.0) / np.float32(448.0)


def test_fp8_write_offset0_resets_and_zero_scale():
    pools = _fp8_setup()
    kp, vp, ks, vs = pools
    _write([4.0] * 8, 8, pools)
    _write([0.0] * 8, 8, pools)                 # offset 0 again: fresh, zero scale
    assert ks[2, 0] == 0.0 and np.all(kp[2, 0] == 0)
    _write([1.0] * 8, 9, pools)                 # grows from 0: old codes stay 0
    assert ks[2, 0] == np.float32(1.0) / np.float32(448.0)
    assert np.all(kp[2, 0] == 0) and np.all(kp[2, 1] == 0x7E)
    _write([5.0] * 8, -1, pools)                # padding slot writes nothing
    assert ks[2, 0] == np.float32(1.0) / np.float32(448.0)


def test_fp8_write_error_bound_random():
    rng = np.random.default_rng(11)
    pools = _fp8_setup(D=32, bs=16, nblocks=1)
    kp, vp, ks, vs = pools
    xs = []
    for off in range(16):
        v = rng.standard_normal(32).astype(np.float32) * np.float32(rng.uniform(0.1, 3))
        xs.append(wl.bf16_to_float(wl.bf16_bits(v)))
        _write(v, off, pools)
    xs = np.array(xs)
    assert ks[0, 0] == np.float32(np.abs(xs).max()) / np.float32(448.0)
    restored = oracle.e4m3_to_double(kp[0, :, 0]) * float(ks[0, 0])
    # each requantisation adds at most half an E4M3 step (relative 2^-4) plus the
    # subnormal spacing; 16 writes bound the drift well below 6 steps
    step = np.maximum(np.abs(xs) * 2.0 ** -3, 2.0 ** -9 * float(ks[0, 0]))
    assert np.all(np.abs(restored - xs) <= 6 * step)


# ---------------------------------------------------------------- 4-bit cache write

def _int4_setup(D=8, bs=4, nblocks=3, Hkv=1):
    k_pool = np.zeros((nblocks, bs, Hkv, D // 2), np.uint8)
    v_pool = np.zeros((nblocks, bs, Hkv, D // 2), np.uint8)
    k_scale = np.full((nblocks, Hkv), 123.0, np.float32)
    v_scale = np.full((nblocks, Hkv), 123.0, np.float32)
    return k_pool, v_pool, k_scale, v_scale


def _write4(vals, slot, pools):
    kp, vp, ks, vs = pools
    x = wl.bf16_bits(np.asarray(vals, np.float32)).reshape(1, 1, -1)
    oracle.reshape_and_cache_int4(x, x, kp, vp, ks, vs, np.array([slot], np.int64), kp.shape[1])


def _unpack4(row):
    """Independent unpacking: element 2j in the low nibble of byte j, offset by 8."""
    row = np.asarray(row, np.uint8)
    out = np.empty(row.size * 2, np.int64)
    out[0::2] = (row & 0xF).astype(np.int64) - 8
    out[1::2] = (row >> 4).astype(np.int64) - 8
    return out


def test_int4_writer_reproduces_page_example(golden_dir):
    g = _golden(golden_dir, "quant4_absmax.json")
    pools = _int4_setup(D=6, bs=2, nblocks=1)
    _write4(g["values"], 0, pools)
    kp, vp, ks, vs = pools
    assert _unpack4(kp[0, 0, 0]).tolist() == g["codes"]
    restored = oracle.int4_restore(kp[0, 0, 0], float(ks[0, 0]))
    assert np.round(restored, 3).tolist() == g["restored_3dp"]
    assert ks[0, 0] == np.float32(1.0) / np.float32(7.0)


def test_int4_writer_growth_requantises():
    pools = _int4_setup()
    kp, vp, ks, vs = pools
    _write4([1.0, 0.3, -0.5 / 7, 0, 0, 0, 0, 0], 0, pools)   # codes 7, 2, 0 (-0.499 -> 0)
    assert _unpack4(kp[0, 0, 0])[:3].tolist() == [7, 2, 0]
    _write4([0.5, 0, 0, 0, 0, 0, 0, 0], 1, pools)             # smaller: scale kept
    assert ks[0, 0] == np.float32(1.0) / np.float32(7.0)
    # fp32: 0.5 / fl(1/7) = 3.4999999, just below the tie, so the code is 3
    assert _unpack4(kp[0, 1, 0])[0] == 3
    _write4([2.4 / 7, 0, 0, 0, 0, 0, 0, 0], 3, pools)         # bf16(2.4/7) / fl(1/7) = 2.40 -> 2
    assert _unpack4(kp[0, 3, 0])[0] == 2
    _write4([-3.0, 0, 0, 0, 0, 0, 0, 0], 2, pools)            # larger: rows 0, 1 re-encoded
    assert ks[0, 0] == np.float32(3.0) / np.float32(7.0)
    assert _unpack4(kp[0, 0, 0])[:2].tolist() == [2, 1]       # 1.0 -> 2.33 -> 2; 0.29 -> 0.67 -> 1
    assert _unpack4(kp[0, 1, 0])[0] == 1                      # 0.43 -> 1.0 -> 1
    assert _unpack4(kp[0, 2, 0])[0] == -7
    _write4([0.0] * 8, 4, pools)                              # block 1 offset 0: zero scale
    assert ks[1, 0] == 0.0 and np.all(_unpack4(kp[1, 0, 0]) == 0)


def test_int4_writer_scale_is_block_absmax_random():
    rng = np.random.default_rng(12)
    pools = _int4_setup(D=32, bs=16, nblocks=1)
    kp, vp, ks, vs = pools
    xs = []
    for off in range(16):
        v = rng.standard_normal(32).astype(np.float32) * np.float32(rng.uniform(0.1, 3))
        xs.append(wl.bf16_to_float(wl.bf16_bits(v)))
        _write4(v, off, pools)
    xs = np.array(xs)
    assert ks[0, 0] == np.float32(np.abs(xs).max()) / np.float32(7.0)
    codes = np.array([_unpack4(kp[0, r, 0]) for r in range(16)])
    assert np.all(np.abs(codes) <= 7)
    restored = codes * float(ks[0, 0])
    # each requantisation moves a value by at most half a step of the scale it used
    assert np.all(np.abs(restored - xs) <= 16 * 0.5 * float(ks[0, 0]) + 1e-7)


def test_int4_restore_closed_form():
    row = np.array([0x8F, 0x18, 0x77], np.uint8)          # nibbles (low, high): 15,8 8,1 7,7
    got = oracle.int4_restore(row, 0.5)
    assert got.tolist() == [3.5, 0.0, 0.0, -3.5, -0.5, -0.5]


# ---------------------------------------------------------------- decode attention

def _contiguous_reference(batch, window=0):
    """Independent restatement: gather each sequence's K/V into contiguous
    arrays with numpy fancy indexing and apply scipy's softmax (over the last
    `window` rows when window > 0)."""
    B, Hq, Hkv, D, bs = batch.B, batch.Hq, batch.Hkv, batch.D, batch.block_size
    G = Hq // Hkv
    q = wl.bf16_to_float(batch.q).astype(np.float64)
    if batch.kv_dtype == "fp8_e4m3":
        lut = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(
            torch.float64).numpy()
        kf = lut[batch.k_pool] * batch.k_scale.astype(np.float64)[:, None, :, None]
        vf = lut[batch.v_pool] * batch.v_scale.astype(np.float64)[:, None, :, None]
    elif batch.kv_dtype == "int4":
        def unpack(pool):
            out = np.empty(pool.shape[:-1] + (pool.shape[-1] * 2,), np.float64)
            out[..., 0::2] = (pool & 0xF).astype(np.float64) - 8
            out[..., 1::2] = (pool >> 4).astype(np.float64) - 8
            return out
        kf = unpack(batch.k_pool) * batch.k_scale.astype(np.float64)[:, None, :, None]
        vf = unpack(batch.v_pool) * batch.v_scale.astype(np.float64)[:, None, :, None]
    else:
        kf = wl.bf16_to_float(batch.k_pool).astype(np.float64)
        vf = wl.bf16_to_float(batch.v_pool).astype(np.float64)
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(batch.seq_lens[b])
        if L == 0:
            continue
        t = np.arange(L)
        if window > 0:
            t = t[-window:]
        blocks = batch.block_tables[b, t // bs]
        K = kf[blocks, t % bs]          # [L, Hkv, D]
        V = vf[blocks, t % bs]
        for h in range(Hq):
            s = batch.sm_scale * (K[:, h // G, :] @ q[b, h])
            out[b, h] = softmax(s) @ V[:, h // G, :]
    return out


def _oracle(batch, **kw):
    return oracle.paged_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                               batch.seq_lens, batch.sm_scale, Hkv=batch.Hkv,
                               block_size=batch.block_size, k_scale=batch.k_scale,
                               v_scale=batch.v_scale, **kw)


def test_decode_tiny_config_vs_contiguous_numpy():
    batch = wl.make("tiny")
    assert np.allclose(_oracle(batch), _contiguous_reference(batch), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("Hq,Hkv,D,bs", [(8, 8, 64, 16), (8, 1, 64, 32), (16, 4, 128, 16),
                                         (12, 3, 64, 32)])
def test_decode_random_shapes_vs_contiguous_numpy(Hq, Hkv, D, bs):
    batch = wl.build_batch("t", [0, 1, 15, 16, 17, 40, 97], Hq=Hq, Hkv=Hkv, D=D,
                           block_size=bs, seed=Hq * 7 + bs)
    assert np.allclose(_oracle(batch), _contiguous_reference(batch), rtol=1e-12, atol=1e-13)


def test_decode_fp8_vs_contiguous_numpy():
    batch = wl.build_batch("t", [3, 16, 33, 70], Hq=8, Hkv=2, D=64, block_size=16, seed=3,
                           kv_dtype="fp8_e4m3")
    assert np.allclose(_oracle(batch), _contiguous_reference(batch), rtol=1e-12, atol=1e-13)


def test_window_positions_page_trace(golden_dir):
    g = _golden(golden_dir, "sliding_window.json")
    for token, want in enumerate(g["retained_after_token"]):
        assert oracle.window_positions(token + 1, g["window"]) == want
    assert max(len(oracle.window_positions(n, g["window"])) for n in range(1, 50)) == \
        g["maximum_retained"]
    assert oracle.window_positions(7, 0) == list(range(7))          # no window


@pytest.mark.parametrize("window", [1, 4, 16, 17, 50, 1000])
def test_decode_window_vs_contiguous_numpy(window):
    batch = wl.build_batch("t", [1, 15, 16, 17, 40, 97, 0], Hq=8, Hkv=2, D=64, block_size=16,
                           seed=60 + window)
    got = _oracle(batch, window=window)
    assert np.allclose(got, _contiguous_reference(batch, window), rtol=1e-12, atol=1e-13)
    if window >= batch.seq_lens.max():
        assert np.array_equal(got, _oracle(batch))


def test_decode_window_ignores_blocks_before_it():
    batch = wl.build_batch("t", [100, 70], Hq=8, Hkv=2, D=64, block_size=16, seed=66)
    ref = _oracle(batch, window=20)
    batch.block_tables[0, :4] = 10 ** 6        # blocks wholly before position 80: never read
    batch.block_tables[1, :3] = -5             # before position 50
    assert np.array_equal(_oracle(batch, window=20), ref)


def test_decode_int4_vs_contiguous_numpy():
    batch = wl.build_batch("t", [3, 16, 33, 70, 0], Hq=8, Hkv=2, D=64, block_size=16, seed=5,
                           kv_dtype="int4")
    assert np.allclose(_oracle(batch), _contiguous_reference(batch), rtol=1e-12, atol=1e-13)


def test_decode_rows_subset_matches_full():
    batch = wl.build_batch("t", [5, 30, 64], Hq=8, Hkv=2, D=64, block_size=16, seed=9)
    full = _oracle(batch)
    rows = np.array([[2, 7], [0, 0], [1, 3]])
    part = _oracle(batch, rows=rows)
    for i, (b, h) in enumerate(rows):
        assert np.array_equal(part[i], full[b, h])


def test_decode_length_one_returns_v_exactly():
    batch = wl.build_batch("t", [1, 1], Hq=8, Hkv=2, D=64, block_size=16, seed=4)
    out = _oracle(batch)
    vf = wl.bf16_to_float(batch.v_pool).astype(np.float64)
    for b in range(2):
        blk = batch.block_tables[b, 0]
        for h in range(8):
            assert np.array_equal(out[b, h], vf[blk, 0, h // 4])


def test_decode_zero_query_gives_mean_of_v():
    batch = wl.build_batch("t", [37], Hq=4, Hkv=1, D=64, block_size=16, seed=6)
    batch.q[:] = 0
    out = _oracle(batch)
    vf = wl.bf16_to_float(batch.v_pool).astype(np.float64)
    t = np.arange(37)
    V = vf[batch.block_tables[0, t // 16], t % 16, 0]
    assert np.allclose(out[0], V.mean(axis=0)[None, :], rtol=1e-13, atol=1e-14)


def test_decode_two_tokens_logistic_closed_form():
    batch = wl.build_batch("t", [2], Hq=2, Hkv=1, D=64, block_size=16, seed=8)
    out = _oracle(batch)
    kf = wl.bf16_to_float(batch.k_pool).astype(np.float64)
    vf = wl.bf16_to_float(batch.v_pool).astype(np.float64)
    q = wl.bf16_to_float(batch.q).astype(np.float64)
    blk = batch.block_tables[0, 0]
    for h in range(2):
        s0 = batch.sm_scale * kf[blk, 0, 0] @ q[0, h]
        s1 = batch.sm_scale * kf[blk, 1, 0] @ q[0, h]
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        expect = w0 * vf[blk, 0, 0] + (1.0 - w0) * vf[blk, 1, 0]
        assert np.allclose(out[0, h], expect, rtol=1e-13, atol=1e-14)


def test_decode_needle():
    batch = wl.build_batch("t", [50], Hq=1, Hkv=1, D=64, block_size=16, seed=12)
    q = wl.bf16_to_float(batch.q[0, 0]).astype(np.float32)
    blk, off = batch.block_tables[0, 23 // 16], 23 % 16
    batch.k_pool[blk, off, 0] = wl.bf16_bits(q * np.float32(100.0 / np.linalg.norm(q)) * 8)
    out = _oracle(batch)
    v = wl.bf16_to_float(batch.v_pool[blk, off, 0]).astype(np.float64)
    assert np.allclose(out[0, 0], v, atol=1e-6)


def _permute_blocks(batch, perm):
    """Relabel physical block i as perm[i] (moving its rows): the logical cache is unchanged."""
    k = np.empty_like(batch.k_pool)
    v = np.empty_like(batch.v_pool)
    k[perm] = batch.k_pool
    v[perm] = batch.v_pool
    tables = batch.block_tables.copy()
    used = tables >= 0
    tables[used] = perm[tables[used]]
    return k, v, tables


def test_decode_block_permutation_invariance_bitwise():
    batch = wl.build_batch("t", [3, 40, 77, 16], Hq=8, Hkv=2, D=64, block_size=16, seed=13)
    ref = _oracle(batch)
    perm = np.random.default_rng(1).permutation(batch.nblocks)
    k, v, tables = _permute_blocks(batch, perm)
    out = oracle.paged_decode(batch.q, k, v, tables, batch.seq_lens, batch.sm_scale,
                              Hkv=batch.Hkv, block_size=batch.block_size)
    assert np.array_equal(out, ref)


def test_decode_shared_vs_duplicated_prefix_bitwise():
    groups = ((40, [0, 1, 2]),)                # 2 full shared blocks + a copied 8-row tail
    batch = wl.build_batch("t", [45, 90, 41], Hq=8, Hkv=2, D=64, block_size=16, seed=14,
                           prefix_groups=groups, pool_factor=2.0)
    assert batch.block_tables[0, 0] == batch.block_tables[1, 0] == batch.block_tables[2, 0]
    ref = _oracle(batch)
    # duplicate the shared blocks into free blocks for sequences 1 and 2
    used = set(batch.block_tables[batch.block_tables >= 0].tolist())
    free = [i for i in range(batch.nblocks) if i not in used]
    tables = batch.block_tables.copy()
    k, v = batch.k_pool.copy(), batch.v_pool.copy()
    for b in (1, 2):
        for j in range(2):
            dst = free.pop()
            k[dst], v[dst] = k[tables[b, j]], v[tables[b, j]]
            tables[b, j] = dst
    out = oracle.paged_decode(batch.q, k, v, tables, batch.seq_lens, batch.sm_scale,
                              Hkv=batch.Hkv, block_size=batch.block_size)
    assert np.array_equal(out, ref)


def test_decode_gqa_group_shares_kv():
    # identical queries within a group give identical outputs; across groups they differ
    batch = wl.build_batch("t", [33], Hq=8, Hkv=2, D=64, block_size=16, seed=15)
    batch.q[0, :] = batch.q[0, 0]
    out = _oracle(batch)
    for h in range(4):
        assert np.array_equal(out[0, h], out[0, 0])
        assert np.array_equal(out[0, 4 + h], out[0, 4])
    assert not np.array_equal(out[0, 0], out[0, 4])


# ---------------------------------------------------------------- Quest page selection

def test_quest_page_example(golden_dir):
    g = _golden(golden_dir, "quest_pages.json")
    pages = np.array(g["pages"], dtype=np.float64)
    q = np.array(g["query"])
    scores = []
    for page in pages:
        mn, mx = oracle.page_summary(page)
        assert mn.tolist() == page.min(axis=0).tolist() and mx.tolist() == page.max(axis=0).tolist()
        scores.append(oracle.page_score(q, mn, mx))
    assert scores == g["page_scores"]
    sel = oracle.select_pages(scores, 2)
    assert sel == g["selected_pages"]
    assert len(sel) * pages.shape[1] == g["kv_entries_read"]
    assert pages.shape[0] * pages.shape[1] == g["kv_entries_stored"]


def test_quest_score_bounds_every_key():
    rng = np.random.default_rng(3)
    for _ in range(50):
        keys = rng.standard_normal((16, 8))
        q = rng.standard_normal(8)
        mn, mx = oracle.page_summary(keys)
        s = oracle.page_score(q, mn, mx)
        assert np.all(keys @ q <= s + 1e-12)                   # an upper bound of q . k
        # and tight: the corner of the box it picks reaches it
        corner = np.where(q >= 0, mx, mn)
        assert abs(corner @ q - s) < 1e-12


def test_select_pages_ties_and_short():
    assert oracle.select_pages([1.0, 3.0, 3.0, 2.0], 2) == [1, 2]
    assert oracle.select_pages([5.0, 5.0, 5.0], 2) == [0, 1]      # ties: lower index
    assert oracle.select_pages([0.5, -1.0], 4) == [0, 1]          # fewer pages than k


def _quest_reference(batch, topk):
    """numpy restatement: summaries, group-max scores, top-k, attention on those tokens."""
    B, Hq, Hkv, D, bs = batch.B, batch.Hq, batch.Hkv, batch.D, batch.block_size
    G = Hq // Hkv
    q = wl.bf16_to_float(batch.q).astype(np.float64)
    kf = wl.bf16_to_float(batch.k_pool).astype(np.float64)
    vf = wl.bf16_to_float(batch.v_pool).astype(np.float64)
    out = np.zeros((B, Hq, D))
    sel_all = np.full((B, Hkv, topk), -1)
    for b in range(B):
        L = int(batch.seq_lens[b])
        t = np.arange(L)
        K = kf[batch.block_tables[b, t // bs], t % bs]
        V = vf[batch.block_tables[b, t // bs], t % bs]
        npg = (L + 15) // 16
        for kvh in range(Hkv):
            sc = []
            for j in range(npg):
                kk = K[16 * j:16 * j + 16, kvh]
                qs = q[b, kvh * G:(kvh + 1) * G]
                sc.append(max(np.maximum(qs * kk.min(0), qs * kk.max(0)).sum(1)))
            order = sorted(range(npg), key=lambda j: (-sc[j], j))[:topk]
            sel = sorted(order)
            sel_all[b, kvh, :len(sel)] = sel
            idx = np.concatenate([np.arange(16 * j, min(L, 16 * j + 16)) for j in sel]) \
                if sel else np.zeros(0, int)
            for g in range(G):
                h = kvh * G + g
                if idx.size:
                    out[b, h] = softmax(batch.sm_scale * K[idx, kvh] @ q[b, h]) @ V[idx, kvh]
    return out, sel_all


@pytest.mark.parametrize("topk", [1, 3, 8, 100])
def test_quest_decode_vs_numpy(topk):
    batch = wl.build_batch("t", [1, 15, 16, 17, 70, 200, 0], Hq=8, Hkv=2, D=64, block_size=32,
                           seed=80 + topk)
    out, sel = oracle.quest_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                   batch.seq_lens, batch.sm_scale, Hkv=2, block_size=32, topk=topk)
    ref, ref_sel = _quest_reference(batch, topk)
    assert np.array_equal(sel, ref_sel)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-13)
    if topk >= 200 // 16 + 1:
        assert np.allclose(out, _oracle(batch), rtol=1e-12, atol=1e-13)


def _bf16_neighbours(x):
    """bf16 values (as doubles) near x, found from the bit patterns around float32(x)."""
    b = int(np.float32(x).view(np.uint32)) >> 16
    out = []
    for pat in range(b - 3, b + 4):
        pat &= 0xFFFF
        v = float(np.uint32(pat << 16).view(np.float32))
        if math.isfinite(v):
            out.append(v)
        v = float(np.uint32((pat ^ 0x8000) << 16).view(np.float32))   # across zero
        if math.isfinite(v):
            out.append(v)
    return out + [0.0]


def test_bf16_directed_rounding():
    """round_down(x) is the largest bf16 value <= x and round_up(x) the smallest >= x,
    checked against the bf16 patterns next to x; bf16 values are fixed points."""
    rng = np.random.default_rng(5)
    xs = [1.0 + 2.0 ** -9, -(1.0 + 2.0 ** -9), 3.0, -0.0, 2.0 ** -130 * 1.3, -2.0 ** -128 * 1.7,
          448.0 * 0.37, 1e-3, -7.0 * 0.4321]
    xs += list(rng.standard_normal(300) * np.exp(rng.uniform(-40, 40, 300)))
    for x in xs:
        lo, hi = oracle.bf16_round_down(x), oracle.bf16_round_up(x)
        cand = _bf16_neighbours(x)
        assert lo == max(c for c in cand if c <= x), x
        assert hi == min(c for c in cand if c >= x), x
        assert oracle.bf16_round_down(-x) == -hi and oracle.bf16_round_up(-x) == -lo
    assert oracle.bf16_round_down(1.0 + 2.0 ** -9) == 1.0
    assert oracle.bf16_round_up(1.0 + 2.0 ** -9) == 1.0 + 2.0 ** -7
    for bits in rng.integers(0, 0x7F80, 200):
        v = float(np.uint32(int(bits) << 16).view(np.float32))
        assert oracle.bf16_round_down(v) == v == oracle.bf16_round_up(v)


def test_page_summary_bf16_bounds():
    """Stored summaries bound every key and are the tightest bf16 bounds; on bf16 keys
    they are the exact minimum and maximum."""
    rng = np.random.default_rng(6)
    keys = rng.integers(-7, 8, (16, 64)) * 0.0137           # restored 4-bit-like keys
    mn, mx = oracle.page_summary_bf16(keys)
    assert np.all(mn[None] <= keys) and np.all(mx[None] >= keys)
    emn, emx = keys.min(0), keys.max(0)
    for d in range(64):
        assert max(c for c in _bf16_neighbours(emn[d]) if c <= emn[d]) == mn[d]
        assert min(c for c in _bf16_neighbours(emx[d]) if c >= emx[d]) == mx[d]
    kb = wl.bf16_to_float(wl.bf16_bits(rng.standard_normal((9, 32)))).astype(np.float64)
    mn, mx = oracle.page_summary_bf16(kb)
    assert np.array_equal(mn, kb.min(0)) and np.array_equal(mx, kb.max(0))


def _restored_bf16_batch(batch):
    """The same batch with its quantised pools replaced by bf16 pools of the restored
    values (exact when every scale is a power of two), codes decoded by torch / by hand."""
    import copy
    out = copy.copy(batch)
    pools = []
    for pool, sc in ((batch.k_pool, batch.k_scale), (batch.v_pool, batch.v_scale)):
        if batch.kv_dtype == "fp8_e4m3":
            vals = torch.from_numpy(pool).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        else:
            lo = (pool & 0xF).astype(np.int64) - 8
            hi = (pool >> 4).astype(np.int64) - 8
            vals = np.stack([lo, hi], -1).reshape(pool.shape[:-1] + (pool.shape[-1] * 2,))
        vals = vals * sc.astype(np.float64)[:, None, :, None]
        bits = wl.bf16_bits(vals.astype(np.float32))
        assert np.array_equal(wl.bf16_to_float(bits).astype(np.float64), vals)   # exact
        pools.append(bits)
    out.k_pool, out.v_pool = pools
    out.k_scale = out.v_scale = None
    out.kv_dtype = "bf16"
    return out


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "int4"])
def test_quest_decode_quantised_pools(kv_dtype):
    """Quest over E4M3 / 4-bit pools: with power-of-two scales the restored keys are
    bf16 values, so it must equal Quest over bf16 pools holding them (selection and
    output, exactly); choosing every page must equal the full decode of the pools."""
    batch = wl.build_batch("t", [1, 15, 16, 17, 70, 200, 0], Hq=16, Hkv=2, D=128, block_size=16,
                           seed=83, kv_dtype=kv_dtype)
    rng = np.random.default_rng(7)
    for sc in (batch.k_scale, batch.v_scale):
        sc[...] = 2.0 ** rng.integers(-4, 3, sc.shape)
    plain = _restored_bf16_batch(batch)
    for topk in (1, 4, 100):
        out, sel = oracle.quest_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                       batch.seq_lens, batch.sm_scale, Hkv=2, block_size=16,
                                       topk=topk, k_scale=batch.k_scale, v_scale=batch.v_scale)
        ref, ref_sel = oracle.quest_decode(plain.q, plain.k_pool, plain.v_pool,
                                           plain.block_tables, plain.seq_lens, plain.sm_scale,
                                           Hkv=2, block_size=16, topk=topk)
        assert np.array_equal(sel, ref_sel), topk
        assert np.array_equal(out, ref), topk
    full = oracle.paged_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                               batch.seq_lens, batch.sm_scale, Hkv=2, block_size=16,
                               k_scale=batch.k_scale, v_scale=batch.v_scale)
    assert np.allclose(out, full, rtol=1e-12, atol=1e-13)


def _restored_keys(batch):
    """Restored key pool [nblocks, bs, Hkv, D] in fp64: E4M3 codes decoded by torch,
    4-bit nibbles by hand (element 2j in the low nibble of byte j), times the scale."""
    if batch.kv_dtype == "bf16":
        return wl.bf16_to_float(batch.k_pool).astype(np.float64)
    if batch.kv_dtype == "fp8_e4m3":
        kv = torch.from_numpy(batch.k_pool).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    else:
        lo = (batch.k_pool & 0xF).astype(np.int64) - 8
        hi = (batch.k_pool >> 4).astype(np.int64) - 8
        kv = np.stack([lo, hi], -1).reshape(batch.k_pool.shape[:-1] + (batch.D,))
    return kv.astype(np.float64) * batch.k_scale.astype(np.float64)[:, None, :, None]


@pytest.mark.parametrize("kv_dtype,bs", [("fp8_e4m3", 16), ("int4", 32), ("bf16", 32),
                                         ("fp8_e4m3", 32)])
def test_quest_page_summary_from_pool(kv_dtype, bs):
    """The stored summary of a pool page: min and max of the page's restored keys over
    its first `rows` rows, rounded down / up to bf16 (neighbour search), element-exact;
    on bf16 pools the plain minimum and maximum."""
    batch = wl.build_batch("t", [40, 97], Hq=16, Hkv=2, D=128, block_size=bs, seed=85,
                           kv_dtype=kv_dtype)
    kv = _restored_keys(batch)
    down = np.vectorize(lambda x: max(c for c in _bf16_neighbours(x) if c <= x))
    up = np.vectorize(lambda x: min(c for c in _bf16_neighbours(x) if c >= x))
    rows_all = kv.reshape(-1, 2, 128)                   # pool rows in order
    inexact = 0
    for page, rows, kvh in ((0, 16, 0), (1, 7, 1), (3, 1, 0), (5, 16, 1), (2, 12, 1)):
        mn, mx = oracle.quest_page_summary(batch.k_pool, page, rows, kvh, Hkv=2, D=128,
                                           block_size=bs, k_scale=batch.k_scale)
        kk = rows_all[16 * page:16 * page + rows, kvh]
        assert np.array_equal(mn, down(kk.min(0))) and np.array_equal(mx, up(kk.max(0)))
        inexact += int(np.sum(mn != kk.min(0)) + np.sum(mx != kk.max(0)))
    assert (inexact == 0) == (kv_dtype == "bf16")


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "int4"])
def test_quest_selection_quantised_rounded_summaries(kv_dtype):
    """With arbitrary scales the restored keys are not bf16 values: the selection must be
    the top-k of scores over summaries whose minimum is rounded down and maximum up to
    bf16 (restated here with the neighbour search and numpy)."""
    batch = wl.build_batch("t", [40, 97, 200, 333], Hq=16, Hkv=2, D=128, block_size=32,
                           seed=84, kv_dtype=kv_dtype)
    topk = 5
    _, sel = oracle.quest_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                 batch.seq_lens, batch.sm_scale, Hkv=2, block_size=32,
                                 topk=topk, k_scale=batch.k_scale, v_scale=batch.v_scale)
    kv = _restored_keys(batch)
    q = wl.bf16_to_float(batch.q).astype(np.float64)
    down = np.vectorize(lambda x: max(c for c in _bf16_neighbours(x) if c <= x))
    up = np.vectorize(lambda x: min(c for c in _bf16_neighbours(x) if c >= x))
    inexact = 0
    for b in range(batch.B):
        L = int(batch.seq_lens[b])
        t = np.arange(L)
        K = kv[batch.block_tables[b, t // 32], t % 32]
        for kvh in range(2):
            sc = []
            for j in range((L + 15) // 16):
                kk = K[16 * j:16 * j + 16, kvh]
                mn, mx = down(kk.min(0)), up(kk.max(0))
                inexact += int(np.sum(mn != kk.min(0)) + np.sum(mx != kk.max(0)))
                qs = q[b, kvh * 8:(kvh + 1) * 8]
                sc.append(np.max(np.maximum(qs * mn, qs * mx).sum(1)))
            want = sorted(sorted(range(len(sc)), key=lambda j: (-sc[j], j))[:topk])
            assert list(sel[b, kvh, :len(want)]) == want, (b, kvh)
    assert inexact > 0          # the rounding was exercised


# ---------------------------------------------------------------- split + merge

def test_split_merge_identity_random():
    batch = wl.build_batch("t", [1, 33, 200, 0], Hq=8, Hkv=2, D=64, block_size=16, seed=16)
    full = _oracle(batch)
    rng = np.random.default_rng(2)
    for b in range(batch.B):
        nb = (int(batch.seq_lens[b]) + 15) // 16
        for h in (0, 5):
            for S in (1, 2, 5):
                cuts = np.sort(rng.integers(0, nb + 1, S - 1)) if S > 1 else np.array([], int)
                beg = np.concatenate([[0], cuts, [nb]]).astype(np.int32)
                o, lse = oracle.split_partials(batch.q, batch.k_pool, batch.v_pool,
                                               batch.block_tables, batch.seq_lens,
                                               batch.sm_scale, b, h, beg, Hkv=2, block_size=16)
                merged = oracle.merge_lse(o, lse)
                assert np.allclose(merged, full[b, h], rtol=1e-12, atol=1e-13)
                if S == 1:
                    assert np.array_equal(o[0], full[b, h])


def test_merge_empty_splits_carry_no_weight():
    o = np.array([[1.0, 2.0], [np.nan, np.nan], [3.0, 4.0]])
    lse = np.array([0.0, -np.inf, math.log(3.0)])
    assert np.allclose(oracle.merge_lse(o, lse), [(1 + 9) / 4, (2 + 12) / 4], rtol=1e-15)
    assert np.array_equal(oracle.merge_lse(o[1:2], lse[1:2]), [0.0, 0.0])


def test_token_partials_block_cuts_equal_split_partials():
    """Token pieces at block multiples are the block-aligned split: the same numbers."""
    batch = wl.build_batch("t", [1, 40, 100, 0], Hq=8, Hkv=2, D=64, block_size=32, seed=17)
    rng = np.random.default_rng(3)
    for b in range(batch.B):
        nb = (int(batch.seq_lens[b]) + 31) // 32
        cuts = np.sort(rng.integers(0, nb + 1, 2))
        beg = np.concatenate([[0], cuts, [nb]]).astype(np.int32)
        o1, l1 = oracle.split_partials(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                       batch.seq_lens, batch.sm_scale, b, 3, beg, Hkv=2,
                                       block_size=32)
        o2, l2 = oracle.token_partials(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                       batch.seq_lens, batch.sm_scale, b, 3, beg * 32, Hkv=2,
                                       block_size=32)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_token_partials_merge_identity_and_single_token():
    """Merging pieces cut anywhere (16-token and ragged cuts, empty pieces) gives the
    unsplit attention; a one-token piece has lse = its score and o = its V row."""
    batch = wl.build_batch("t", [1, 33, 200, 0, 97], Hq=8, Hkv=2, D=64, block_size=16, seed=18)
    full = _oracle(batch)
    rng = np.random.default_rng(4)
    kf = wl.bf16_to_float(batch.k_pool).astype(np.float64)
    vf = wl.bf16_to_float(batch.v_pool).astype(np.float64)
    q = wl.bf16_to_float(batch.q).astype(np.float64)
    for b in range(batch.B):
        L = int(batch.seq_lens[b])
        for h in (0, 6):
            for S in (1, 3, 6):
                cuts = np.sort(rng.integers(0, L + 1, S - 1))
                if S == 6 and L > 32:
                    cuts[:2] = (cuts[:2] // 16) * 16            # some 16-token cuts
                beg = np.concatenate([[0], np.sort(cuts), [L]]).astype(np.int32)
                o, lse = oracle.token_partials(batch.q, batch.k_pool, batch.v_pool,
                                               batch.block_tables, batch.seq_lens,
                                               batch.sm_scale, b, h, beg, Hkv=2, block_size=16)
                assert np.allclose(oracle.merge_lse(o, lse), full[b, h], rtol=1e-12, atol=1e-13)
                for i in range(S):
                    if beg[i] == beg[i + 1]:
                        assert lse[i] == -np.inf and not o[i].any()
            if L > 5:
                t = 5
                o, lse = oracle.token_partials(batch.q, batch.k_pool, batch.v_pool,
                                               batch.block_tables, batch.seq_lens,
                                               batch.sm_scale, b, h,
                                               np.array([t, t + 1], np.int32), Hkv=2,
                                               block_size=16)
                blk = batch.block_tables[b, t // 16]
                assert np.array_equal(o[0], vf[blk, t % 16, h // 4])
                assert math.isclose(lse[0], batch.sm_scale * (kf[blk, t % 16, h // 4] @ q[b, h]),
                                    rel_tol=1e-12, abs_tol=1e-12)


def test_paged_decode_pages_all_pages_one_page_and_merge():
    """Every page chosen equals the full decode; one page equals softmax attention over
    that page's rows (numpy on contiguous rows); several pages equal the merge of their
    one-page partials; -1 entries and pages past the end are skipped."""
    batch = wl.build_batch("t", [1, 15, 16, 17, 100, 0], Hq=8, Hkv=2, D=64, block_size=32,
                           seed=19)
    B, Hkv, G = batch.B, 2, 4
    npg = (batch.seq_lens + 15) // 16
    allp = np.full((B, Hkv, 8), -1, np.int32)
    for b in range(B):
        allp[b, :, :npg[b]] = np.arange(npg[b])
    full = _oracle(batch)
    got = oracle.paged_decode_pages(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                    batch.seq_lens, batch.sm_scale, allp, Hkv=Hkv, block_size=32)
    assert np.allclose(got, full, rtol=1e-12, atol=1e-13)
    kf = wl.bf16_to_float(batch.k_pool).astype(np.float64)
    vf = wl.bf16_to_float(batch.v_pool).astype(np.float64)
    q = wl.bf16_to_float(batch.q).astype(np.float64)
    rng = np.random.default_rng(5)
    sel = np.full((B, Hkv, 3), -1, np.int32)
    for b in range(B):
        for kvh in range(Hkv):
            k = min(3, int(npg[b]))
            sel[b, kvh, :k] = np.sort(rng.choice(npg[b], k, replace=False))
    sel[4, 1, 2] = 99                                           # past the end: skipped
    got = oracle.paged_decode_pages(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                    batch.seq_lens, batch.sm_scale, sel, Hkv=Hkv, block_size=32)
    for b in range(B):
        L = int(batch.seq_lens[b])
        for h in range(batch.Hq):
            pages = [int(p) for p in sel[b, h // G] if 0 <= p and 16 * p < L]
            if not pages:
                assert not got[b, h].any()
                continue
            t = np.concatenate([np.arange(16 * p, min(L, 16 * p + 16)) for p in pages])
            K = kf[batch.block_tables[b, t // 32], t % 32, h // G]
            V = vf[batch.block_tables[b, t // 32], t % 32, h // G]
            ref = softmax(batch.sm_scale * (K @ q[b, h])) @ V
            assert np.allclose(got[b, h], ref, rtol=1e-12, atol=1e-13)
            beg = [16 * p for p in pages]
            parts = [oracle.token_partials(batch.q, batch.k_pool, batch.v_pool,
                                           batch.block_tables, batch.seq_lens, batch.sm_scale,
                                           b, h, np.array([s, min(L, s + 16)], np.int32),
                                           Hkv=Hkv, block_size=32) for s in beg]
            o = np.concatenate([p[0] for p in parts])
            lse = np.concatenate([p[1] for p in parts])
            assert np.allclose(oracle.merge_lse(o, lse), got[b, h], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("topk", [1, 4])
def test_paged_decode_pages_on_quest_selection(topk):
    """The pages quest_decode chooses, read by paged_decode_pages, give quest_decode's
    output."""
    batch = wl.build_batch("t", [1, 15, 16, 17, 70, 200, 0], Hq=8, Hkv=2, D=64, block_size=32,
                           seed=90 + topk)
    out, sel = oracle.quest_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                   batch.seq_lens, batch.sm_scale, Hkv=2, block_size=32, topk=topk)
    got = oracle.paged_decode_pages(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                    batch.seq_lens, batch.sm_scale, sel, Hkv=2, block_size=32)
    assert np.allclose(got, out, rtol=1e-12, atol=1e-13)
