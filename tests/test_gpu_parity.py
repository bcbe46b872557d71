"""Parity of the CUDA path (libpa.so through its C ABI) with the CPU oracle.

Every test here needs a GB300.  The bar: bit-exact for the cache write and for
indexing invariants; |gpu - oracle| <= 1e-3 + 1e-3 |oracle| elementwise for
bf16 caches and <= 2e-2 + 2e-2 |oracle| for FP8 caches (the oracle reads the
same codes and scales).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_28_gb300 import _lib
from paged_kv_cache_28_gb300 import workload as wl
from paged_kv_cache_28_gb300.device import DeviceBatch, default_num_segments, default_num_splits

pytestmark = pytest.mark.gpu

TOL_BF16 = (1e-3, 1e-3)   # (atol, rtol)
TOL_FP8 = (2e-2, 2e-2)    # FP8 and 4-bit caches, against an oracle reading the same codes


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    _lib.load()


def _tol(batch):
    return TOL_FP8 if batch.quantized else TOL_BF16


def assert_close(gpu, ref, batch, what=""):
    atol, rtol = _tol(batch)
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance; worst at {i}:"
                             f" gpu={gpu[i]!r} oracle={ref[i]!r}")


def oracle_after_write(batch, rows=None, write=True, window=0):
    """Oracle output after applying this step's cache write to host copies of the pools."""
    kp, vp = batch.k_pool.copy(), batch.v_pool.copy()
    ks = None if batch.k_scale is None else batch.k_scale.copy()
    vs = None if batch.v_scale is None else batch.v_scale.copy()
    if write:
        if batch.kv_dtype == "fp8_e4m3":
            oracle.reshape_and_cache_fp8(batch.k_new, batch.v_new, kp, vp, ks, vs,
                                         batch.slot_mapping, batch.block_size)
        elif batch.kv_dtype == "int4":
            oracle.reshape_and_cache_int4(batch.k_new, batch.v_new, kp, vp, ks, vs,
                                          batch.slot_mapping, batch.block_size)
        else:
            oracle.reshape_and_cache_bf16(batch.k_new, batch.v_new, kp, vp, batch.slot_mapping,
                                          batch.block_size)
    out = oracle.paged_decode(batch.q, kp, vp, batch.block_tables, batch.seq_lens,
                              batch.sm_scale, Hkv=batch.Hkv, block_size=batch.block_size,
                              k_scale=ks, v_scale=vs, rows=rows, window=window)
    return out, (kp, vp, ks, vs)


def run_gpu(dev, mode, num_splits=None, window=0):
    """mode "decode": pa_decode without a workspace; "decode_ws": pa_decode with one (its
    default segments); "split": pa_decode with a workspace of num_splits segments;
    "parts": pa_decode_splitkv with num_splits slots per head, then pa_merge_lse."""
    dev.out.fill_(float("nan"))
    if mode == "decode":
        dev.decode(window=window)
    elif mode == "decode_ws":                    # pa_decode given a workspace: split + merge
        dev.decode(window=window, workspace=True)
    elif mode == "parts":
        dev.decode_splitkv(num_splits, window=window)
    else:
        dev.decode_segments(num_splits, window=window)
    torch.cuda.synchronize()
    return dev.out.cpu().numpy()


MODES = [("decode", None), ("decode_ws", None), ("split", 1), ("split", 3), ("split", 7),
         ("split", 64), ("split", 1000), ("split", "default"), ("parts", 1), ("parts", 2),
         ("parts", 5), ("parts", "default")]


def _mode_count(dev, mode, ns):
    if ns != "default":
        return ns
    return default_num_splits(dev.shape) if mode == "parts" else default_num_segments(dev.shape)


def _modes_run(dev, batch, ref, label):
    for mode, ns in MODES:
        ns = _mode_count(dev, mode, ns)
        out = run_gpu(dev, mode, ns)
        assert_close(out, ref, batch, f"{label} {mode} num_splits={ns}")
    assert dev.read_err() == 0


# ---------------------------------------------------------------- cache write

def test_reshape_and_cache_bf16_bit_exact():
    batch = wl.make("tiny")
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    _, (kp, vp, _, _) = oracle_after_write(batch)
    gk, gv, _, _ = dev.pools_numpy()
    assert np.array_equal(gk, kp) and np.array_equal(gv, vp)
    assert dev.read_err() == 0


def test_reshape_and_cache_bf16_canary_and_padding():
    rng = np.random.default_rng(3)
    T, Hkv, D, bs, nblocks = 37, 4, 128, 32, 11
    k_pool = np.full((nblocks, bs, Hkv, D), 0xBEEF, np.uint16)
    v_pool = np.full((nblocks, bs, Hkv, D), 0xCAFE, np.uint16)
    slots = rng.choice(nblocks * bs, T, replace=False).astype(np.int64)
    slots[::5] = -1
    k_new = rng.integers(0, 65536, (T, Hkv, D)).astype(np.uint16)
    v_new = rng.integers(0, 65536, (T, Hkv, D)).astype(np.uint16)
    dk = torch.from_numpy(k_pool.view(np.int16)).cuda()
    dv = torch.from_numpy(v_pool.view(np.int16)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    shape = _lib.make_shape(T, Hkv, Hkv, D, bs, nblocks, 1)
    _lib.pa_reshape_and_cache(shape, torch.from_numpy(k_new.view(np.int16)).cuda(),
                              torch.from_numpy(v_new.view(np.int16)).cuda(), dk, dv, None, None,
                              torch.from_numpy(slots).cuda(), err)
    oracle.reshape_and_cache_bf16(k_new, v_new, k_pool, v_pool, slots, bs)
    assert np.array_equal(dk.cpu().numpy().view(np.uint16), k_pool)
    assert np.array_equal(dv.cpu().numpy().view(np.uint16), v_pool)
    assert _lib.pa_read_error_flag(err) == 0


def _fp8_write_case(seed, T, Hkv, bs, nblocks, steps, int4=False):
    """Several write calls; each writes one token into each of T distinct blocks at
    increasing offsets, so scales grow and rows get re-encoded."""
    rng = np.random.default_rng(seed)
    D = 128
    if int4:      # any nibbles 1..15 (codes -7..7)
        k_pool = (rng.integers(1, 16, (nblocks, bs, Hkv, D // 2)) |
                  (rng.integers(1, 16, (nblocks, bs, Hkv, D // 2)) << 4)).astype(np.uint8)
    else:
        k_pool = rng.integers(0, 256, (nblocks, bs, Hkv, D)).astype(np.uint8)
        k_pool[k_pool == 0x7F] = 0
        k_pool[k_pool == 0xFF] = 0
    v_pool = k_pool.copy()
    k_scale = rng.uniform(0.001, 0.01, (nblocks, Hkv)).astype(np.float32)
    v_scale = k_scale.copy()
    dk, dv = torch.from_numpy(k_pool).cuda(), torch.from_numpy(v_pool).cuda()
    dks, dvs = torch.from_numpy(k_scale).cuda(), torch.from_numpy(v_scale).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    blocks = rng.choice(nblocks, T, replace=False)
    shape = _lib.make_shape(T, Hkv, Hkv, D, bs, nblocks, 1,
                            _lib.PA_KV_INT4 if int4 else _lib.PA_KV_FP8_E4M3)
    write = oracle.reshape_and_cache_int4 if int4 else oracle.reshape_and_cache_fp8
    for step in range(steps):
        scale = rng.uniform(0.05, 4.0, (T, 1, 1)).astype(np.float32)
        x = rng.standard_normal((T, Hkv, D)).astype(np.float32) * scale
        if step == 1:
            x[0] = 0.0                               # all-zero token
        k_new = wl.bf16_bits(x)
        v_new = wl.bf16_bits(x[::-1].copy())
        slots = (blocks * bs + step).astype(np.int64)
        slots[1] = -1                                # padding row
        _lib.pa_reshape_and_cache(shape, torch.from_numpy(k_new.view(np.int16)).cuda(),
                                  torch.from_numpy(v_new.view(np.int16)).cuda(), dk, dv, dks, dvs,
                                  torch.from_numpy(slots).cuda(), err)
        write(k_new, v_new, k_pool, v_pool, k_scale, v_scale, slots, bs)
    torch.cuda.synchronize()
    assert _lib.pa_read_error_flag(err) == 0
    return (dk.cpu().numpy(), dv.cpu().numpy(), dks.cpu().numpy(), dvs.cpu().numpy()), \
        (k_pool, v_pool, k_scale, v_scale)


@pytest.mark.parametrize("seed,T,Hkv,bs,steps", [(0, 5, 2, 16, 16), (1, 64, 8, 16, 6),
                                                  (2, 9, 1, 32, 32)])
def test_reshape_and_cache_fp8_bit_exact(seed, T, Hkv, bs, steps):
    got, want = _fp8_write_case(seed, T, Hkv, bs, 3 * T + 2, steps)
    for g, w, name in zip(got, want, ("k_pool", "v_pool", "k_scale", "v_scale")):
        assert np.array_equal(g.view(np.uint8) if g.dtype != np.float32 else g.view(np.uint32),
                              w.view(np.uint8) if w.dtype != np.float32 else w.view(np.uint32)), name


@pytest.mark.parametrize("seed,T,Hkv,bs,steps", [(3, 5, 2, 16, 16), (4, 64, 8, 16, 6),
                                                  (5, 9, 1, 32, 32)])
def test_reshape_and_cache_int4_bit_exact(seed, T, Hkv, bs, steps):
    got, want = _fp8_write_case(seed, T, Hkv, bs, 3 * T + 2, steps, int4=True)
    for g, w, name in zip(got, want, ("k_pool", "v_pool", "k_scale", "v_scale")):
        assert np.array_equal(g.view(np.uint8) if g.dtype != np.float32 else g.view(np.uint32),
                              w.view(np.uint8) if w.dtype != np.float32 else w.view(np.uint32)), name


def _quant_pools(rng, nblocks, bs, Hkv, int4):
    D = 128
    if int4:      # any nibbles 1..15 (codes -7..7)
        k_pool = (rng.integers(1, 16, (nblocks, bs, Hkv, D // 2)) |
                  (rng.integers(1, 16, (nblocks, bs, Hkv, D // 2)) << 4)).astype(np.uint8)
    else:
        k_pool = rng.integers(0, 256, (nblocks, bs, Hkv, D)).astype(np.uint8)
        k_pool[k_pool == 0x7F] = 0
        k_pool[k_pool == 0xFF] = 0
    k_scale = rng.uniform(0.001, 0.01, (nblocks, Hkv)).astype(np.float32)
    return k_pool, k_pool.copy(), k_scale, k_scale.copy()


def _quant_write(pools, k_new, v_new, slots, bs, int4):
    """One call on the GPU and the oracle's write on host copies: (gpu, oracle, err)."""
    k_pool, v_pool, k_scale, v_scale = (a.copy() for a in pools)
    T, Hkv, D = k_new.shape
    dk, dv = torch.from_numpy(k_pool).cuda(), torch.from_numpy(v_pool).cuda()
    dks, dvs = torch.from_numpy(k_scale).cuda(), torch.from_numpy(v_scale).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    shape = _lib.make_shape(T, Hkv, Hkv, D, bs, k_pool.shape[0], 1,
                            _lib.PA_KV_INT4 if int4 else _lib.PA_KV_FP8_E4M3)
    _lib.pa_reshape_and_cache(shape, torch.from_numpy(k_new.view(np.int16)).cuda(),
                              torch.from_numpy(v_new.view(np.int16)).cuda(), dk, dv, dks, dvs,
                              torch.from_numpy(slots).cuda(), err)
    write = oracle.reshape_and_cache_int4 if int4 else oracle.reshape_and_cache_fp8
    write(k_new, v_new, k_pool, v_pool, k_scale, v_scale, slots, bs)
    flag = _lib.pa_read_error_flag(err)
    got = (dk.cpu().numpy(), dv.cpu().numpy(), dks.cpu().numpy(), dvs.cpu().numpy())
    return got, (k_pool, v_pool, k_scale, v_scale), flag


def _assert_pools_equal(got, want):
    for g, w, name in zip(got, want, ("k_pool", "v_pool", "k_scale", "v_scale")):
        assert np.array_equal(g.view(np.uint8) if g.dtype != np.float32 else g.view(np.uint32),
                              w.view(np.uint8) if w.dtype != np.float32 else w.view(np.uint32)), name


@pytest.mark.parametrize("int4", [False, True])
@pytest.mark.parametrize("bs", [16, 32])
def test_quantised_prompt_written_in_one_call(bs, int4):
    """A 100-token prompt and a 37-token one written in one call (their tokens share
    blocks, so each block's tokens are applied in token order: scales grow, earlier
    rows are re-encoded), with growing magnitudes, a prompt continuing a half-filled
    block, padding rows and one token of another sequence between them; the tokens are
    shuffled so that a block's tokens are not adjacent in the call.  Codes and scales
    bit for bit against the oracle."""
    rng = np.random.default_rng(400 + bs + int4)
    Hkv, nblocks = 4, 40
    pools = _quant_pools(rng, nblocks, bs, Hkv, int4)
    blocks = rng.permutation(nblocks)
    slots = [int(blocks[p // bs]) * bs + p % bs for p in range(100)]              # positions 0..99
    start = bs // 2                                                                # mid-block start
    slots += [int(blocks[10 + (start + p) // bs]) * bs + (start + p) % bs for p in range(37)]
    slots += [int(blocks[30]) * bs + 3, -1, -1]
    T = len(slots)
    mag = np.concatenate([np.linspace(0.1, 6.0, 100), rng.uniform(0.05, 3.0, T - 100)])
    x = (rng.standard_normal((T, Hkv, 128)) * mag[:, None, None]).astype(np.float32)
    x[5] = 0.0                                                                     # a zero token
    order = rng.permutation(T)
    slots = np.asarray(slots, np.int64)[order]
    k_new, v_new = wl.bf16_bits(x[order]), wl.bf16_bits(x[order][::-1].copy())
    got, want, flag = _quant_write(pools, k_new, v_new, slots, bs, int4)
    _assert_pools_equal(got, want)
    assert flag == 0


@pytest.mark.parametrize("int4", [False, True])
@pytest.mark.parametrize("bs", [16, 32])
def test_quantised_long_prompt_in_order(bs, int4):
    """A 3,000-token prompt written in one call in token order (each block's later tokens
    follow one of their own block, so they leave without scanning the call), after a
    block already half full, with a second sequence's tokens and padding rows between
    some of them.  Codes and scales bit for bit against the oracle."""
    rng = np.random.default_rng(450 + bs + int4)
    Hkv, nblocks = 2, 3200 // bs + 16
    pools = _quant_pools(rng, nblocks, bs, Hkv, int4)
    blocks = rng.permutation(nblocks)
    start = bs // 2
    slots = [int(blocks[(start + p) // bs]) * bs + (start + p) % bs for p in range(3000)]
    other = [int(blocks[-1]) * bs + j for j in range(5)]
    for j, at in enumerate(sorted(rng.choice(3000, 5, replace=False))[::-1]):
        slots.insert(int(at), other[j])
    slots.insert(1234, -1)
    T = len(slots)
    mag = rng.uniform(0.05, 4.0, T)
    x = (rng.standard_normal((T, Hkv, 128)) * mag[:, None, None]).astype(np.float32)
    k_new, v_new = wl.bf16_bits(x), wl.bf16_bits(x[::-1].copy())
    got, want, flag = _quant_write(pools, k_new, v_new, np.asarray(slots, np.int64), bs, int4)
    _assert_pools_equal(got, want)
    assert flag == 0


@pytest.mark.parametrize("int4", [False, True])
def test_quantised_duplicate_slot_applied_in_order_and_flagged(int4):
    """Two tokens of one call with the same slot: both applied, the later one last (the
    oracle's order), and PA_DEVERR_FP8_CONFLICT set; distinct slots of a block are not
    a conflict."""
    rng = np.random.default_rng(420 + int4)
    bs, Hkv, nblocks = 16, 2, 6
    pools = _quant_pools(rng, nblocks, bs, Hkv, int4)
    slots = np.array([16, 17, 16, 40, 18], np.int64)          # 16 twice; 17, 18 share block 1
    x = rng.standard_normal((5, Hkv, 128)).astype(np.float32)
    x[2] *= 5.0
    got, want, flag = _quant_write(pools, wl.bf16_bits(x), wl.bf16_bits(-x), slots, bs, int4)
    _assert_pools_equal(got, want)
    assert flag == _lib.PA_DEVERR_FP8_CONFLICT
    slots = np.array([16, 17, 40, 18], np.int64)
    got, want, flag = _quant_write(pools, wl.bf16_bits(x[:4]), wl.bf16_bits(-x[:4]), slots, bs,
                                   int4)
    _assert_pools_equal(got, want)
    assert flag == 0


# ---------------------------------------------------------------- decode parity

def test_tiny_config_all_modes():
    batch = wl.make("tiny")
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    _modes_run(dev, batch, ref, "tiny")


SHAPES = [
    # Hq, Hkv, D, bs, lens
    (8, 2, 64, 16, [1, 17, 33, 100]),
    (64, 8, 128, 16, [1, 15, 16, 17, 31, 32, 33, 250, 1000, 3]),
    (64, 8, 128, 32, [0, 1, 47, 64, 65, 700]),
    (16, 16, 64, 16, [5, 300, 0, 129]),           # MHA (G = 1)
    (32, 2, 128, 16, [77, 1, 500]),               # G = 16 (two n-tiles)
    (12, 1, 64, 32, [33, 2, 90]),                  # MQA, G = 12
    (24, 4, 128, 16, [129, 4, 1]),                 # G = 6 (padded group)
]


@pytest.mark.parametrize("Hq,Hkv,D,bs,lens", SHAPES)
def test_random_shapes_all_modes(Hq, Hkv, D, bs, lens):
    batch = wl.build_batch("t", lens, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, seed=Hq + bs + D,
                           max_blocks=(max(lens) + bs - 1) // bs + 3)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    _modes_run(dev, batch, ref, f"Hq={Hq} Hkv={Hkv} D={D} bs={bs}")



def _fuzz_case(case):
    """Seeded draw of one configuration: cache type, group size, head dim, block size,
    lengths (zeros, tails and longer sequences), a window or none, and split counts."""
    rng = np.random.default_rng(1000 + case)
    kv = ["bf16", "fp8_e4m3", "int4"][case % 3]
    D = 128 if kv != "bf16" else int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 3, 4, 8]))
    G = int(rng.choice([1, 2, 4, 6, 8, 12, 16]))
    bs = int(rng.choice([16, 32]))
    B = int(rng.integers(1, 11))
    lens = [int(x) for x in rng.choice([0, 1, 15, 16, 17, 33, 64, 129, 300, 777, 1500], B)]
    window = int(rng.integers(1, 600)) if rng.random() < 0.3 else 0
    splits = [int(x) for x in rng.choice([1, 2, 5, 17, 64, 333], 2, replace=False)]
    return kv, D, Hkv, G, bs, lens, window, splits


@pytest.mark.parametrize("case", range(24))
def test_fuzz_configurations(case):
    """24 seeded random configurations, each through the cache write and every decode
    path (pa_decode with and without a workspace, the split decode at two segment counts,
    pa_decode_splitkv + pa_merge_lse at two slot counts), against the oracle."""
    kv, D, Hkv, G, bs, lens, window, splits = _fuzz_case(case)
    batch = wl.build_batch("t", lens, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs, seed=2000 + case,
                           kv_dtype=kv, max_blocks=(max(lens) + bs - 1) // bs + 2)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch, window=window)
    label = f"case {case}: {kv} D={D} Hkv={Hkv} G={G} bs={bs} lens={lens} window={window}"
    modes = ([("decode", None), ("decode_ws", None)] + [("split", n) for n in splits] +
             [("parts", n) for n in splits])
    for mode, ns in modes:
        assert_close(run_gpu(dev, mode, ns, window), ref, batch, f"{label} {mode} {ns}")
    assert dev.read_err() == 0

@pytest.mark.parametrize("kv,D,G", [("bf16", 64, 1), ("fp8_e4m3", 128, 1), ("int4", 128, 8)])
def test_largest_kv_head_count(kv, D, G):
    """Hkv = 2048, the most the decode's tile records can name (the KV head sits in 11
    bits): ragged lengths through the cache write and every decode path.  The 4-bit case
    reads its heads in pairs (G = 8), so its unit view has 1024 KV heads of 16 query rows."""
    lens = [1, 17, 40]
    batch = wl.build_batch("max_hkv", lens, Hq=G * 2048, Hkv=2048, D=D, block_size=16, seed=77,
                           kv_dtype=kv, max_blocks=4)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    for mode, ns in [("decode", None), ("decode_ws", None), ("split", 5), ("split", "default"),
                     ("parts", 3), ("parts", "default")]:
        ns = _mode_count(dev, mode, ns)
        assert_close(run_gpu(dev, mode, ns), ref, batch, f"Hkv=2048 {kv} {mode} {ns}")
    assert dev.read_err() == 0


@pytest.mark.parametrize("kv_dtype,Hq,Hkv,bs", [("bf16", 64, 8, 16), ("bf16", 32, 2, 32),
                                                  ("bf16", 16, 1, 16), ("fp8_e4m3", 64, 8, 16),
                                                  ("int4", 64, 8, 16), ("int4", 16, 2, 32)])
def test_pa_decode_cluster_split_skewed(kv_dtype, Hq, Hkv, bs):
    """pa_decode without a workspace on a small, skewed batch.  With few (sequence, KV
    head) units each is served by a cluster of CTAs: a long sequence's tiles spread over
    all of them and CTA 0 merges their states through distributed shared memory; a short
    one keeps CTA 0 alone and the others leave.  Clusters take the sequences longest
    first.  Windows shorten the long sequences' tile lists."""
    lens = [5000, 1, 17, 300, 0, 1025, 64, 3333]
    batch = wl.build_batch("cl", lens, Hq=Hq, Hkv=Hkv, D=128, block_size=bs, seed=77,
                           kv_dtype=kv_dtype)
    dev = DeviceBatch(batch)
    ref, _ = oracle_after_write(batch, write=False)
    out = run_gpu(dev, "decode")
    assert_close(out, ref, batch, "cluster decode")
    for w in (1, 100, 2000):
        ref_w, _ = oracle_after_write(batch, write=False, window=w)
        assert_close(run_gpu(dev, "decode", window=w), ref_w, batch, f"cluster decode window {w}")
    assert np.array_equal(_bits(run_gpu(dev, "decode")), _bits(out)), "not repeatable"
    assert dev.read_err() == 0


def test_fp8_small_all_modes():
    batch = wl.build_batch("t", [1, 16, 17, 200, 33, 0, 1000], Hq=64, Hkv=8, D=128, block_size=16,
                           seed=21, kv_dtype="fp8_e4m3")
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    _modes_run(dev, batch, ref, "fp8")


def test_int4_small_all_modes():
    batch = wl.build_batch("t", [1, 16, 17, 200, 33, 0, 1000], Hq=64, Hkv=8, D=128, block_size=16,
                           seed=23, kv_dtype="int4")
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    _modes_run(dev, batch, ref, "int4")


def test_int4_g16_bs32_window():
    batch = wl.build_batch("t", [3, 64, 65, 400], Hq=32, Hkv=2, D=128, block_size=32, seed=24,
                           kv_dtype="int4")
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    _modes_run(dev, batch, ref, "int4 G=16 bs=32")
    ref, _ = oracle_after_write(batch, window=50)
    for mode, ns in (("decode", None), ("split", 7)):
        assert_close(run_gpu(dev, mode, ns, window=50), ref, batch, f"int4 window {mode}")


def test_int4_odd_kv_heads():
    """G = 8 with an odd number of KV heads: 4-bit heads are served one at a time."""
    batch = wl.build_batch("t", [1, 16, 17, 200, 0, 500], Hq=24, Hkv=3, D=128, block_size=16,
                           seed=25, kv_dtype="int4")
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    _modes_run(dev, batch, ref, "int4 Hkv=3")


def test_int4_selection_serves_heads_singly():
    """A per-KV-head selection on a shape whose heads are otherwise read in pairs:
    choosing every page must equal the full decode."""
    batch = wl.build_batch("t", [5, 70, 300, 1], Hq=64, Hkv=8, D=128, block_size=16, seed=26,
                           kv_dtype="int4")
    dev = DeviceBatch(batch)
    ref, _ = oracle_after_write(batch, write=False)
    topk = 24
    sel = np.full((batch.B, batch.Hkv, topk), -1, np.int32)
    for b, L in enumerate(batch.seq_lens):
        n = (int(L) + 15) // 16
        sel[b, :, :n] = np.arange(n)
    sel = torch.from_numpy(sel).to(dev.device)
    for mode, ns in (("decode", None), ("split", 1), ("split", 9), ("split", 200)):
        dev.out.fill_(float("nan"))
        (dev.decode(selected_pages=sel) if mode == "decode"
         else dev.decode_segments(ns, selected_pages=sel))
        torch.cuda.synchronize()
        assert_close(dev.out.cpu().numpy(), ref, batch, f"int4 all pages chosen {mode} {ns}")
    assert dev.read_err() == 0


@pytest.mark.parametrize("kv_dtype,Hq,Hkv", [("fp8_e4m3", 64, 8), ("int4", 64, 8),
                                             ("int4", 24, 3)])
def test_quantised_zero_scales(kv_dtype, Hq, Hkv):
    """A (block, head) whose scale is 0 restores to zeros (the writer stores scale 0
    for an all-zero block): its K rows score 0 and its V rows add nothing."""
    batch = wl.build_batch("t", [40, 300, 17, 64], Hq=Hq, Hkv=Hkv, D=128, block_size=16,
                           seed=27, kv_dtype=kv_dtype)
    rng = np.random.default_rng(7)
    for b, L in enumerate(batch.seq_lens):
        for j in range((int(L) + 15) // 16):
            blk = batch.block_tables[b, j]
            for h in range(Hkv):
                r = rng.integers(0, 4)           # 0: V scale 0, 1: K scale 0, 2: both, 3: none
                if r in (0, 2):
                    batch.v_scale[blk, h] = 0.0
                if r in (1, 2):
                    batch.k_scale[blk, h] = 0.0
    dev = DeviceBatch(batch)
    ref, _ = oracle_after_write(batch, write=False)
    for mode, ns in (("decode", None), ("split", 1), ("split", 7), ("split", 100)):
        out = run_gpu(dev, mode, ns)
        assert np.isfinite(out).all(), (mode, ns)
        assert_close(out, ref, batch, f"{kv_dtype} zero scales {mode} {ns}")
    assert dev.read_err() == 0


@pytest.mark.parametrize("kv_dtype,Hq,Hkv", [("fp8_e4m3", 64, 8), ("int4", 64, 8),
                                             ("fp8_e4m3", 32, 2)])
def test_quantised_scale_spread(kv_dtype, Hq, Hkv):
    """Per-block V scales spread over six decades inside one sequence: the decode's
    accumulator changes its V-scale unit along the way, and large V values of
    opposite signs cancel.  The quantised tolerance holds with no allowance (the
    weights reach the PV product as two f16 terms)."""
    batch = wl.build_batch("t", [40, 700, 17, 1500], Hq=Hq, Hkv=Hkv, D=128, block_size=16,
                           seed=28, kv_dtype=kv_dtype)
    rng = np.random.default_rng(8)
    batch.k_scale[:] *= (10.0 ** rng.uniform(-2, 1, batch.k_scale.shape)).astype(np.float32)
    batch.v_scale[:] *= (10.0 ** rng.uniform(-3, 3, batch.v_scale.shape)).astype(np.float32)
    dev = DeviceBatch(batch)
    ref, _ = oracle_after_write(batch, write=False)
    for mode, ns in (("decode", None), ("split", 1), ("split", 5), ("split", 64)):
        out = run_gpu(dev, mode, ns)
        assert np.isfinite(out).all(), (mode, ns)
        assert_close(out, ref, batch, f"{kv_dtype} scale spread {mode} {ns}")
    assert dev.read_err() == 0


def test_fp8_g16_and_bs32():
    batch = wl.build_batch("t", [3, 64, 65, 400], Hq=32, Hkv=2, D=128, block_size=32, seed=22,
                           kv_dtype="fp8_e4m3")
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    _modes_run(dev, batch, ref, "fp8 G=16 bs=32")


# ---------------------------------------------------------------- sliding window

@pytest.mark.parametrize("kv_dtype,bs", [("bf16", 16), ("bf16", 32), ("fp8_e4m3", 16),
                                        ("fp8_e4m3", 32), ("int4", 16), ("int4", 32)])
def test_window_all_modes(kv_dtype, bs):
    lens = [1, 15, 16, 17, 40, 97, 333, 1200, 0, 64]
    batch = wl.build_batch("t", lens, Hq=64, Hkv=8, D=128, block_size=bs, seed=70 + bs,
                           kv_dtype=kv_dtype)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    for window in (1, 4, 16, 17, 100, 5000):
        ref, _ = oracle_after_write(batch, window=window)
        for mode, ns in (("decode", None), ("split", 1), ("split", 9), ("split", 300),
                         ("parts", 1), ("parts", 3)):
            out = run_gpu(dev, mode, ns, window)
            assert_close(out, ref, batch, f"window={window} {mode} {ns}")
    assert dev.read_err() == 0


def test_window_one_returns_last_v_and_skips_old_blocks():
    batch = wl.build_batch("t", [100, 37, 1], Hq=64, Hkv=8, D=128, block_size=16, seed=75)
    vf = wl.bf16_to_float(batch.v_pool)
    # blocks wholly before a 20-token window are never read: sequence 0 (L=100)
    # attends from position 80 (block 5), sequence 1 (L=37) from 17 (block 1)
    batch.block_tables[0, :5] = -1
    batch.block_tables[1, :1] = batch.nblocks + 100
    dev = DeviceBatch(batch)
    for mode, ns in (("decode", None), ("split", 5)):
        out = run_gpu(dev, mode, ns, window=1)
        for b, L in enumerate(batch.seq_lens):
            t = L - 1
            blk = batch.block_tables[b, t // 16]
            for h in range(64):
                assert np.array_equal(_bits(out[b, h]), _bits(vf[blk, t % 16, h // 8])), (mode, b)
        out = run_gpu(dev, mode, ns, window=20)
        ref, _ = oracle_after_write(batch, write=False, window=20)
        assert_close(out, ref, batch, f"window 20 {mode}")
    assert dev.read_err() == 0


# ---------------------------------------------------------------- Quest page selection

def _quest_scores_numpy(batch):
    """Exact page scores [B][Hkv] -> list over pages (group max), from the pool."""
    bs, G = batch.block_size, batch.Hq // batch.Hkv
    q = wl.bf16_to_float(batch.q).astype(np.float64)
    kf = wl.bf16_to_float(batch.k_pool).astype(np.float64)
    out = {}
    for b in range(batch.B):
        L = int(batch.seq_lens[b])
        t = np.arange(L)
        K = kf[batch.block_tables[b, t // bs], t % bs]
        for kvh in range(batch.Hkv):
            sc = []
            for j in range((L + 15) // 16):
                kk = K[16 * j:16 * j + 16, kvh]
                qs = q[b, kvh * G:(kvh + 1) * G]
                sc.append(np.max(np.maximum(qs * kk.min(0), qs * kk.max(0)).sum(1)))
            out[b, kvh] = np.array(sc)
    return out


def _check_selection(batch, gpu_sel, ref_sel, topk):
    """Selections agree wherever the exact k-th / (k+1)-th score gap exceeds fp32
    rounding; elsewhere the GPU's choice must still be a valid top-k."""
    scores = _quest_scores_numpy(batch)
    agree = np.zeros(gpu_sel.shape[:2], bool)
    for (b, kvh), sc in scores.items():
        g, r = gpu_sel[b, kvh], ref_sel[b, kvh]
        n = min(topk, sc.size)
        assert np.all(g[n:] == -1) and np.all(np.diff(g[:n]) > 0)
        if np.array_equal(g, r):
            agree[b, kvh] = True
            continue
        srt = np.sort(sc)[::-1]
        gap = srt[n - 1] - srt[n] if n < sc.size else np.inf
        assert gap <= 1e-4 * max(1.0, abs(srt[n - 1])), (b, kvh, gap)
        assert sc[g[:n]].min() >= srt[n - 1] - 1e-4 * max(1.0, abs(srt[n - 1]))
    return agree


def test_quest_summaries_bit_exact():
    batch = wl.build_batch("t", [1, 15, 16, 17, 100, 333], Hq=16, Hkv=4, D=128, block_size=32,
                           seed=90)
    dev = DeviceBatch(batch)
    dev.quest_build_summaries()
    torch.cuda.synchronize()
    got = dev.key_summaries.view(torch.int16).cpu().numpy().view(np.uint16)
    kf = wl.bf16_to_float(batch.k_pool)
    for b in range(batch.B):
        L = int(batch.seq_lens[b])
        for j in range((L + 15) // 16):
            t = np.arange(16 * j, min(L, 16 * j + 16))
            rows = kf[batch.block_tables[b, t // 32], t % 32]          # [n, Hkv, D]
            page = batch.block_tables[b, 16 * j // 32] * 2 + (16 * j % 32) // 16
            assert np.array_equal(got[page, :, 0], wl.bf16_bits(rows.min(0)))
            assert np.array_equal(got[page, :, 1], wl.bf16_bits(rows.max(0)))
    assert dev.read_err() == 0


def _oracle_page_scores(batch):
    """[B][Hkv] -> (scores over pages, fp32 error bound) from the oracle's page summary
    and page score, group max taken here; the bound is 32 units of fp32 rounding of the
    sum of |terms| (the kernel's sums are about nine additions deep)."""
    bs, G = batch.block_size, batch.Hq // batch.Hkv
    q = wl.bf16_to_float(batch.q).astype(np.float64)
    kf = wl.bf16_to_float(batch.k_pool).astype(np.float64)
    out = {}
    for b in range(batch.B):
        L = int(batch.seq_lens[b])
        t = np.arange(L)
        K = kf[batch.block_tables[b, t // bs], t % bs]
        for kvh in range(batch.Hkv):
            sc, tol = [], []
            for j in range((L + 15) // 16):
                mn, mx = oracle.page_summary(K[16 * j:16 * j + 16, kvh])
                qs = q[b, kvh * G:(kvh + 1) * G]
                sc.append(max(oracle.page_score(qs[g], mn, mx) for g in range(G)))
                mag = np.abs(qs) @ np.maximum(np.abs(mn), np.abs(mx))
                tol.append(32 * 2.0 ** -24 * mag.max())
            out[b, kvh] = (np.array(sc), np.array(tol))
    return out


@pytest.mark.parametrize("bs,Hq,Hkv,D", [(16, 32, 4, 128), (32, 32, 4, 128),
                                         (16, 32, 2, 128), (16, 16, 4, 64), (32, 32, 2, 64)])
def test_quest_page_scores(bs, Hq, Hkv, D):
    """Scores for every page, for G = 4, 8 and 16 (one or two 8-head n-tiles) and D = 64
    and 128."""
    lens = [1, 15, 16, 17, 100, 333, 1000, 2047, 0, 64, 4000]
    batch = wl.build_batch("t", lens, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, seed=97 + bs + Hq + D)
    dev = DeviceBatch(batch)
    dev.quest_build_summaries()
    dev.quest_buffers(8)
    dev.page_scores.fill_(float("nan"))
    dev.quest_select(8)
    torch.cuda.synchronize()
    got = dev.page_scores.cpu().numpy()
    for (b, kvh), (sc, tol) in _oracle_page_scores(batch).items():
        n = sc.size
        assert np.all(np.abs(got[b, kvh, :n] - sc) <= tol), (b, kvh)
        assert np.all(np.isnan(got[b, kvh, n:])), (b, kvh)            # untouched
    assert dev.read_err() == 0


@pytest.mark.parametrize("topk,bs,Hq,Hkv,D", [(1, 16, 64, 8, 128), (4, 16, 64, 8, 128),
                                              (13, 32, 64, 8, 128), (64, 16, 64, 8, 128),
                                              (6, 16, 32, 2, 128), (9, 32, 16, 4, 64)])
def test_quest_select_and_sparse_decode(topk, bs, Hq, Hkv, D):
    lens = [1, 15, 16, 17, 100, 333, 1000, 2047, 0, 64]
    batch = wl.build_batch("t", lens, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, seed=91 + topk)
    dev = DeviceBatch(batch)
    dev.quest_build_summaries()
    sel = dev.quest_select(topk)
    torch.cuda.synchronize()
    gpu_sel = sel.cpu().numpy()
    ref, ref_sel = oracle.quest_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                       batch.seq_lens, batch.sm_scale, Hkv=batch.Hkv,
                                       block_size=bs, topk=topk)
    agree = _check_selection(batch, gpu_sel, ref_sel, topk)
    # every row against the oracle's decode over the GPU's own (checked) selection; rows
    # whose selection is the oracle's also against the oracle's Quest decode
    ref_sel_gpu = oracle.paged_decode_pages(batch.q, batch.k_pool, batch.v_pool,
                                            batch.block_tables, batch.seq_lens, batch.sm_scale,
                                            gpu_sel, Hkv=batch.Hkv, block_size=bs)
    G = batch.Hq // batch.Hkv
    rows = np.array([(b, h) for b in range(batch.B) for h in range(batch.Hq) if agree[b, h // G]])
    for mode, ns in (("decode", None), ("split", 1), ("split", 11), ("split", 500),
                     ("parts", 1), ("parts", 4)):
        dev.out.fill_(float("nan"))
        if mode == "decode":
            dev.decode(selected_pages=sel)
        elif mode == "parts":
            dev.decode_splitkv(ns, selected_pages=sel)
        else:
            dev.decode_segments(ns, selected_pages=sel)
        torch.cuda.synchronize()
        out = dev.out.cpu().numpy()
        assert_close(out, ref_sel_gpu, batch, f"quest topk={topk} {mode} {ns} (every row)")
        assert_close(out[rows[:, 0], rows[:, 1]], ref[rows[:, 0], rows[:, 1]], batch,
                     f"quest topk={topk} {mode} {ns}")
    assert dev.read_err() == 0


@pytest.mark.parametrize("kv_dtype,bs", [("fp8_e4m3", 16), ("fp8_e4m3", 32), ("int4", 16),
                                         ("int4", 32)])
def test_quest_summaries_quantised_bit_exact(kv_dtype, bs):
    """Summaries of E4M3 / 4-bit pools: the oracle's outward-rounded bf16 bounds of the
    restored keys, bit for bit, for every page of every sequence (full and partial pages,
    pages sharing a block)."""
    batch = wl.build_batch("t", [1, 15, 16, 17, 100, 333], Hq=16, Hkv=4, D=128, block_size=bs,
                           seed=92 + bs, kv_dtype=kv_dtype)
    dev = DeviceBatch(batch)
    dev.quest_build_summaries()
    torch.cuda.synchronize()
    got = dev.key_summaries.view(torch.int16).cpu().numpy().view(np.uint16)
    checked = 0
    for b in range(batch.B):
        L = int(batch.seq_lens[b])
        for j in range((L + 15) // 16):
            rows = min(16, L - 16 * j)
            page = batch.block_tables[b, 16 * j // bs] * (bs // 16) + (16 * j % bs) // 16
            for h in range(batch.Hkv):
                mn, mx = oracle.quest_page_summary(batch.k_pool, page, rows, h, Hkv=batch.Hkv,
                                                   D=128, block_size=bs, k_scale=batch.k_scale)
                assert np.array_equal(got[page, h, 0], wl.bf16_bits(mn.astype(np.float32))), \
                    (b, j, h)
                assert np.array_equal(got[page, h, 1], wl.bf16_bits(mx.astype(np.float32))), \
                    (b, j, h)
                checked += 1
    assert checked > 40 and dev.read_err() == 0


def _oracle_quant_page_scores(batch):
    """[B][Hkv] -> exact page scores (group max) over the oracle's stored summaries."""
    bs, G = batch.block_size, batch.Hq // batch.Hkv
    q = wl.bf16_to_float(batch.q).astype(np.float64)
    out = {}
    for b in range(batch.B):
        L = int(batch.seq_lens[b])
        for kvh in range(batch.Hkv):
            sc = []
            for j in range((L + 15) // 16):
                page = batch.block_tables[b, 16 * j // bs] * (bs // 16) + (16 * j % bs) // 16
                mn, mx = oracle.quest_page_summary(batch.k_pool, page, min(16, L - 16 * j), kvh,
                                                   Hkv=batch.Hkv, D=batch.D, block_size=bs,
                                                   k_scale=batch.k_scale)
                qs = q[b, kvh * G:(kvh + 1) * G]
                sc.append(max(oracle.page_score(qs[g], mn, mx) for g in range(G)))
            out[b, kvh] = np.array(sc)
    return out


@pytest.mark.parametrize("kv_dtype,topk,bs", [("fp8_e4m3", 4, 16), ("fp8_e4m3", 13, 32),
                                              ("int4", 4, 16), ("int4", 9, 32)])
def test_quest_quantised_select_and_sparse_decode(kv_dtype, topk, bs):
    """Quest end to end on E4M3 / 4-bit pools: the selection is the oracle's wherever the
    k-th / (k+1)-th score gap exceeds fp32 rounding (else a valid top-k), and every row's
    output matches the oracle's decode over the GPU's selection (quantised tolerance)."""
    lens = [1, 15, 16, 17, 100, 333, 1000, 0, 64]
    batch = wl.build_batch("t", lens, Hq=64, Hkv=8, D=128, block_size=bs, seed=93 + topk,
                           kv_dtype=kv_dtype)
    dev = DeviceBatch(batch)
    dev.quest_build_summaries()
    sel = dev.quest_select(topk)
    torch.cuda.synchronize()
    gpu_sel = sel.cpu().numpy()
    _, ref_sel = oracle.quest_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                     batch.seq_lens, batch.sm_scale, Hkv=batch.Hkv,
                                     block_size=bs, topk=topk, k_scale=batch.k_scale,
                                     v_scale=batch.v_scale)
    same = 0
    for (b, kvh), sc in _oracle_quant_page_scores(batch).items():
        g, r = gpu_sel[b, kvh], ref_sel[b, kvh]
        n = min(topk, sc.size)
        assert np.all(g[n:] == -1) and np.all(np.diff(g[:n]) > 0)
        if np.array_equal(g, r):
            same += 1
            continue
        srt = np.sort(sc)[::-1]
        gap = srt[n - 1] - srt[n] if n < sc.size else np.inf
        assert gap <= 1e-4 * max(1.0, abs(srt[n - 1])), (b, kvh, gap)
        assert sc[g[:n]].min() >= srt[n - 1] - 1e-4 * max(1.0, abs(srt[n - 1]))
    assert same >= 0.9 * batch.B * batch.Hkv
    ref = oracle.paged_decode_pages(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                    batch.seq_lens, batch.sm_scale, gpu_sel, Hkv=batch.Hkv,
                                    block_size=bs, k_scale=batch.k_scale, v_scale=batch.v_scale)
    for mode, ns in (("decode", None), ("split", 1), ("split", 11), ("parts", 4)):
        dev.out.fill_(float("nan"))
        if mode == "decode":
            dev.decode(selected_pages=sel)
        elif mode == "parts":
            dev.decode_splitkv(ns, selected_pages=sel)
        else:
            dev.decode_segments(ns, selected_pages=sel)
        torch.cuda.synchronize()
        assert_close(dev.out.cpu().numpy(), ref, batch, f"{kv_dtype} quest topk={topk} {mode} {ns}")
    assert dev.read_err() == 0


def test_quest_all_pages_equals_full_decode():
    batch = wl.build_batch("t", [5, 70, 300], Hq=64, Hkv=8, D=128, block_size=16, seed=95)
    dev = DeviceBatch(batch)
    dev.quest_build_summaries()
    sel = dev.quest_select(64)                    # more pages than any sequence has
    ref, _ = oracle_after_write(batch, write=False)
    for mode, ns in (("decode", None), ("split", 9)):
        dev.out.fill_(float("nan"))
        (dev.decode(selected_pages=sel) if mode == "decode"
         else dev.decode_segments(ns, selected_pages=sel))
        torch.cuda.synchronize()
        assert_close(dev.out.cpu().numpy(), ref, batch, f"quest all pages {mode}")
    assert dev.read_err() == 0


# ---------------------------------------------------------------- invariants

def _bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def test_length_one_returns_v_bitwise():
    batch = wl.build_batch("t", [1, 1, 1], Hq=64, Hkv=8, D=128, block_size=16, seed=31)
    dev = DeviceBatch(batch)
    vf = wl.bf16_to_float(batch.v_pool)
    for mode, ns in (("decode", None), ("split", 5)):
        out = run_gpu(dev, mode, ns)
        for b in range(3):
            blk = batch.block_tables[b, 0]
            for h in range(64):
                assert np.array_equal(_bits(out[b, h]), _bits(vf[blk, 0, h // 8])), (mode, b, h)


def _permuted(batch, perm):
    k = np.empty_like(batch.k_pool)
    v = np.empty_like(batch.v_pool)
    k[perm] = batch.k_pool
    v[perm] = batch.v_pool
    t = batch.block_tables.copy()
    t[t >= 0] = perm[t[t >= 0]]
    return k, v, t


def test_block_permutation_invariance_bitwise():
    batch = wl.build_batch("t", [3, 400, 77, 1600, 16], Hq=64, Hkv=8, D=128, block_size=16,
                           seed=32)
    dev = DeviceBatch(batch)
    outs = [run_gpu(dev, "decode"), run_gpu(dev, "split", 37)]
    perm = np.random.default_rng(0).permutation(batch.nblocks)
    k, v, t = _permuted(batch, perm)
    batch2 = wl.Batch(**{**batch.__dict__, "k_pool": k, "v_pool": v, "block_tables": t})
    dev2 = DeviceBatch(batch2)
    outs2 = [run_gpu(dev2, "decode"), run_gpu(dev2, "split", 37)]
    for a, b in zip(outs, outs2):
        assert np.array_equal(_bits(a), _bits(b))


def test_shared_vs_duplicated_prefix_bitwise():
    groups = ((900, [0, 1, 2, 3]),)
    batch = wl.build_batch("t", [950, 2000, 901, 1500], Hq=64, Hkv=8, D=128, block_size=16,
                           seed=33, prefix_groups=groups, pool_factor=2.0)
    dev = DeviceBatch(batch)
    outs = [run_gpu(dev, "decode"), run_gpu(dev, "split", 29)]
    used = set(batch.block_tables[batch.block_tables >= 0].tolist())
    free = [i for i in range(batch.nblocks) if i not in used]
    tables = batch.block_tables.copy()
    k, v = batch.k_pool.copy(), batch.v_pool.copy()
    for b in (1, 2, 3):
        for j in range(900 // 16):
            dst = free.pop()
            k[dst], v[dst] = k[tables[b, j]], v[tables[b, j]]
            tables[b, j] = dst
    batch2 = wl.Batch(**{**batch.__dict__, "k_pool": k, "v_pool": v, "block_tables": tables})
    dev2 = DeviceBatch(batch2)
    outs2 = [run_gpu(dev2, "decode"), run_gpu(dev2, "split", 29)]
    for a, b in zip(outs, outs2):
        assert np.array_equal(_bits(a), _bits(b))


def test_shared_prefix_hint_changes_nothing_bitwise():
    groups = ((900, list(range(12))), (3000, [12, 13, 14]))
    lens = [950, 2000, 901, 1500, 3000, 905, 1000, 2500, 4000, 999, 1200, 960, 3100, 5000, 3001]
    batch = wl.build_batch("t", lens, Hq=64, Hkv=8, D=128, block_size=16, seed=40,
                           prefix_groups=groups)
    assert batch.shared_prefix_lens is not None
    dev = DeviceBatch(batch)
    ref, _ = oracle_after_write(batch, write=False)
    outs = []
    for hints in (False, True):
        dev.out.fill_(float("nan"))
        dev.decode_segments(23, hints=hints)
        torch.cuda.synchronize()
        outs.append(dev.out.cpu().numpy())
        assert_close(outs[-1], ref, batch, f"hints={hints}")
    assert np.array_equal(_bits(outs[0]), _bits(outs[1]))
    # any hint values (here: random, including past the end) give the same bits
    dev.shared_prefix_lens = torch.from_numpy(
        np.random.default_rng(1).integers(0, 6000, batch.B).astype(np.int32)).cuda()
    dev.out.fill_(float("nan"))
    dev.decode_segments(23)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(dev.out.cpu().numpy()), _bits(outs[0]))
    # pa_decode_splitkv takes it too: the same bits with and without
    parts = []
    for hints in (False, True):
        dev.out.fill_(float("nan"))
        dev.decode_splitkv(6, hints=hints)
        torch.cuda.synchronize()
        parts.append(dev.out.cpu().numpy())
        assert_close(parts[-1], ref, batch, f"splitkv hints={hints}")
    assert np.array_equal(_bits(parts[0]), _bits(parts[1]))
    # pa_decode without a workspace (one CTA per sequence and KV head) takes the hint too
    pair = []
    for hints in (False, True):
        dev.out.fill_(float("nan"))
        dev.decode(hints=hints)
        torch.cuda.synchronize()
        pair.append(dev.out.cpu().numpy())
        assert_close(pair[-1], ref, batch, f"pa_decode hints={hints}")
    assert np.array_equal(_bits(pair[0]), _bits(pair[1]))
    assert dev.read_err() == 0


def test_zero_query_gives_mean_of_v():
    batch = wl.build_batch("t", [333, 16], Hq=8, Hkv=1, D=128, block_size=16, seed=34)
    batch.q[:] = 0
    dev = DeviceBatch(batch)
    vf = wl.bf16_to_float(batch.v_pool).astype(np.float64)
    for mode, ns in (("decode", None), ("split", 9)):
        out = run_gpu(dev, mode, ns)
        for b, L in enumerate(batch.seq_lens):
            t = np.arange(L)
            mean = vf[batch.block_tables[b, t // 16], t % 16, 0].mean(axis=0)
            assert_close(out[b], np.broadcast_to(mean, out[b].shape), batch, "q=0")


def test_repeatable_bitwise():
    batch = wl.build_batch("t", [1200, 5, 3000], Hq=64, Hkv=8, D=128, block_size=16, seed=35)
    dev = DeviceBatch(batch)
    a = run_gpu(dev, "split", 111)
    b = run_gpu(dev, "split", 111)
    assert np.array_equal(_bits(a), _bits(b))


def test_empty_batch_rows_and_all_empty():
    batch = wl.build_batch("t", [0, 0, 40, 0], Hq=8, Hkv=2, D=64, block_size=16, seed=36)
    dev = DeviceBatch(batch)
    ref, _ = oracle_after_write(batch, write=False)
    for mode, ns in (("decode", None), ("split", 4)):
        out = run_gpu(dev, mode, ns)
        assert np.all(out[[0, 1, 3]] == 0.0)
        assert_close(out, ref, batch, mode)
    empty = wl.build_batch("t", [0, 0], Hq=8, Hkv=2, D=64, block_size=16, seed=37)
    dev = DeviceBatch(empty)
    for mode, ns in (("decode", None), ("split", 4)):
        assert np.all(run_gpu(dev, mode, ns) == 0.0)


# ---------------------------------------------------------------- device error flags

def test_bad_block_id_flagged():
    batch = wl.build_batch("t", [40, 40], Hq=8, Hkv=2, D=64, block_size=16, seed=38)
    batch.block_tables[1, 1] = batch.nblocks + 5
    dev = DeviceBatch(batch)
    for mode, ns in (("decode", None), ("split", 3)):
        dev.err.zero_()
        out = run_gpu(dev, mode, ns)
        assert dev.read_err() & _lib.PA_DEVERR_BLOCK_ID
        ref, _ = oracle_after_write(wl.Batch(**{**batch.__dict__, "seq_lens": batch.seq_lens[:1],
                                                "q": batch.q[:1], "B": 1}), write=False)
        assert_close(out[:1], ref, batch, "untouched sequence")


def test_bad_seq_len_and_slot_flagged():
    batch = wl.build_batch("t", [20, 20], Hq=8, Hkv=2, D=64, block_size=16, seed=39)
    batch.seq_lens[0] = batch.max_blocks * 16 + 1
    dev = DeviceBatch(batch)
    for mode, ns in (("decode", None), ("split", 3)):
        dev.err.zero_()
        run_gpu(dev, mode, ns)
        assert dev.read_err() & _lib.PA_DEVERR_SEQ_LEN
    dev.err.zero_()
    dev.slot_mapping[0] = batch.nblocks * 16 + 3
    dev.reshape_and_cache()
    assert dev.read_err() & _lib.PA_DEVERR_SLOT


# ---------------------------------------------------------------- full-size configs

def _sample_rows(batch, rng, n_random=192):
    lens = batch.seq_lens
    pick = {int(np.argmax(lens)), int(np.argmin(lens))}
    pick.update(int(b) for b in rng.choice(batch.B, min(batch.B, 3), replace=False))
    rows = [(b, h) for b in sorted(pick) for h in range(batch.Hq)]
    rows += [(int(rng.integers(batch.B)), int(rng.integers(batch.Hq))) for _ in range(n_random)]
    return np.array(rows, dtype=np.int32)


# ---------------------------------------------------------------- cascade (shared prefixes)

def _cascade_batch(Hq, Hkv, D, bs, groups, free_lens, seed, plens=None, kv_dtype="bf16"):
    """groups: [(prefix tokens, [suffix lengths])]; members follow each other, then the
    ungrouped sequences.  plens: the cascade lengths (default: prefix cut to tiles)."""
    lens, pgroups, b = [], [], 0
    for plen, suffixes in groups:
        members = list(range(b, b + len(suffixes)))
        lens += [plen + sfx for sfx in suffixes]
        pgroups.append((plen, members))
        b += len(suffixes)
    lens += list(free_lens)
    batch = wl.build_batch("t", lens, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, seed=seed,
                           prefix_groups=pgroups, kv_dtype=kv_dtype)
    offsets, seqs, plen = wl.cascade_groups(batch)
    if plens is not None:
        plen = np.asarray(plens, np.int32)
    return batch, (offsets, seqs, plen)


@pytest.mark.parametrize("Hq,Hkv,D,lens_kind", [(64, 8, 128, "mixed"), (48, 8, 128, "mixed"),
                                                 (64, 8, 64, "mixed"), (64, 64, 128, "short"),
                                                 (32, 4, 128, "wide")])
def test_pa_decode_many_units(Hq, Hkv, D, lens_kind):
    """pa_decode without a workspace on bf16 batches with more (sequence, KV head) units
    than CTAs at once (one CTA per unit, longest sequences first): lengths from 0 up with
    a few long ones; G = 8 and 6 (a padded group); D = 128 and 64; 12,800 short units (200
    sequences); 300 sequences over five orders of magnitude (the bucketed order, several
    sequences per thread in its search).  Against the oracle, with a window and with
    Quest pages too, and repeatable bit for bit."""
    rng = np.random.default_rng(500 + Hq + Hkv + D)
    if lens_kind == "mixed":
        lens = list(rng.integers(0, 600, 110)) + [0, 1, 15, 16, 17] + [4000, 2500]
    elif lens_kind == "wide":
        lens = list((10 ** rng.uniform(0, 3.8, 296)).astype(int)) + [0, 0, 1, 16]
    else:
        lens = list(rng.integers(1, 40, 200))          # 12,800 units
    batch = wl.build_batch("t", lens, Hq=Hq, Hkv=Hkv, D=D, block_size=16, seed=510 + D)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    for window in (0, 100):
        ref, _ = oracle_after_write(batch, window=window)
        out = run_gpu(dev, "decode", window=window)
        assert_close(out, ref, batch, f"many units window={window}")
        assert np.array_equal(_bits(run_gpu(dev, "decode", window=window)), _bits(out))
    assert dev.read_err() == 0
    if D == 128 and lens_kind in ("mixed", "wide"):
        dev.quest_build_summaries()
        sel = dev.quest_select(5)
        torch.cuda.synchronize()
        ref = oracle.paged_decode_pages(batch.q, dev.pools_numpy()[0], dev.pools_numpy()[1],
                                        batch.block_tables, batch.seq_lens, batch.sm_scale,
                                        sel.cpu().numpy(), Hkv=Hkv, block_size=16)
        dev.out.fill_(float("nan"))
        dev.decode(selected_pages=sel)
        torch.cuda.synchronize()
        assert_close(dev.out.cpu().numpy(), ref, batch, "many units quest")
        assert dev.read_err() == 0


@pytest.mark.parametrize("kind", ["prefix", "one_long", "tiny_units", "max_units", "g6_d64",
                                  "mixed_4000", "bs32", "g1", "g2"])
def test_pa_decode_persistent(kind):
    """pa_decode without a workspace on bf16 batches of more units than two per resident
    CTA and at most 4,096, with no window or page selection: persistent CTAs of eight
    warps on a water-filled schedule, each CTA's tiles cut into one contiguous segment per
    warp, units that cross segments joined in shared memory.  A shared 900-token prefix
    with the L2 hints (800 units); one 30,000-token sequence among short ones (its units
    outweigh a CTA's mean share and cross every segment of their CTAs); 2,048 units of 0
    to 40 tokens (empty units, segments of a few tiles); 4,096 single-head sequences (the
    largest list); G = 6 at D = 64; 4,000 units of up to 1,500 tokens; 32-token blocks;
    G = 1 and 2.
    Against the oracle, repeatable bit for bit, and (on the shared prefix) the same bits
    for any hint values."""
    rng = np.random.default_rng({"prefix": 601, "one_long": 602, "tiny_units": 603,
                                 "max_units": 604, "g6_d64": 605, "mixed_4000": 606,
                                 "bs32": 607, "g1": 608, "g2": 609}[kind])
    Hq, Hkv, D, groups, bs = 64, 8, 128, (), 16
    if kind == "prefix":
        lens = [900 + int(x) for x in wl.lognormal_lens(rng, 100, 600, 1, 6000)]
        groups = ((900, list(range(100))),)
    elif kind == "one_long":
        lens = [30000] + list(rng.integers(1, 800, 79))
    elif kind == "tiny_units":
        lens = list(rng.integers(0, 41, 256))
    elif kind == "max_units":
        Hq, Hkv = 8, 1
        lens = list(rng.integers(1, 700, 4096))
    elif kind == "mixed_4000":
        lens = list(rng.integers(0, 1501, 500))
    elif kind == "bs32":                           # 32-token blocks: two tiles per block
        bs = 32
        lens = list(rng.integers(0, 2000, 120)) + [31, 32, 33, 4000]
    elif kind in ("g1", "g2"):                     # one or two query heads per KV head
        Hq = 8 if kind == "g1" else 16
        lens = list(rng.integers(0, 1200, 96)) + [1, 16, 17, 3000]
    else:
        Hq, Hkv, D = 48, 8, 64          # four CTAs per SM otherwise: 1,216 resident
        lens = list(rng.integers(0, 1500, 196)) + [0, 1, 16, 17]
    batch = wl.build_batch("t", lens, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, seed=610,
                           prefix_groups=groups)
    assert 2 * (4 if D == 64 else 2) * 152 < batch.B * Hkv <= 4096
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    dev.out.fill_(float("nan"))
    dev.decode(hints=kind == "prefix")
    torch.cuda.synchronize()
    out = dev.out.cpu().numpy()
    assert_close(out, ref, batch, f"persistent {kind}")
    assert dev.read_err() == 0
    for _ in range(2):
        assert np.array_equal(_bits(run_gpu(dev, "decode")), _bits(out)), f"{kind} not repeatable"
    if kind == "prefix":   # any hint values (random, past the end too) give the same bits
        dev.shared_prefix_lens = torch.from_numpy(
            rng.integers(0, 8000, batch.B).astype(np.int32)).cuda()
        dev.out.fill_(float("nan"))
        dev.decode(hints=True)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(dev.out.cpu().numpy()), _bits(out))
    assert dev.read_err() == 0


# ---------------------------------------------------------------- caller-visible partials

def _splitkv_pieces(batch, S, workers):
    """(b, unit) -> token ranges of its pieces in slot order, as include/pa.h defines the
    cut of pa_decode_splitkv (no window): segments of W tiles over the (b, unit,
    position) tile stream, W = max(ceil(total / workers), ceil((n_max - 1) / (S - 1)));
    with S = 1 every unit is one piece.  A unit is (b, KV head), or (b, KV heads 2u,
    2u + 1) for 4-bit and E4M3 pools read in pairs."""
    paired = (batch.kv_dtype in ("int4", "fp8_e4m3") and batch.D == 128
              and batch.Hkv % 2 == 0 and batch.Hq == 8 * batch.Hkv)
    Hu = batch.Hkv // (2 if paired else 1)
    n = [(int(L) + 15) // 16 for L in batch.seq_lens]
    prefix = np.concatenate([[0], np.cumsum([Hu * x for x in n])]).astype(np.int64)
    total = int(prefix[-1])
    W = max(1, -(-total // workers))
    if S >= 2:
        W = max(W, -(-(max(n) - 1) // (S - 1)))
    pieces = {}
    for b, L in enumerate(int(x) for x in batch.seq_lens):
        for u in range(Hu):
            start, end = int(prefix[b]) + u * n[b], int(prefix[b]) + (u + 1) * n[b]
            if n[b] == 0:
                pieces[b, u] = []
            elif S == 1:
                pieces[b, u] = [(0, L)]
            else:
                pieces[b, u] = [(16 * (max(start, g * W) - start),
                                 min(L, 16 * (min(end, (g + 1) * W) - start)))
                                for g in range(start // W, (end - 1) // W + 1)]
    return pieces, Hu


@pytest.mark.parametrize("kv_dtype,Hq,Hkv,bs,lens,S", [
    ("bf16", 64, 8, 16, [1, 17, 700, 0, 3000, 40], 4),
    ("bf16", 64, 8, 32, [1, 17, 700, 0, 3000, 40], 1),
    ("bf16", 16, 2, 16, [5000, 3, 64], 2),
    ("bf16", 32, 2, 16, [900, 77], 9),                 # G = 16
    ("fp8_e4m3", 64, 8, 16, [1, 250, 2000, 0], 3),
    ("int4", 64, 8, 16, [33, 1200, 1], 5),            # paired 4-bit units
    ("int4", 24, 3, 32, [600, 9], 2),                 # 4-bit heads served singly
])
def test_splitkv_partials_match_oracle_per_slot(kv_dtype, Hq, Hkv, bs, lens, S):
    """pa_decode_splitkv's caller-visible partials: every slot against the oracle's
    partial over that slot's tokens (o within the cache type's tolerance, lse within
    1e-3), empty slots lse = -inf; then pa_merge_lse against the oracle's decode."""
    batch = wl.build_batch("t", lens, Hq=Hq, Hkv=Hkv, D=128, block_size=bs, seed=300 + S,
                           kv_dtype=kv_dtype)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, (kp, vp, ks, vs) = oracle_after_write(batch)
    dev.ensure_parts(S)
    dev.o_part.fill_(float("nan"))
    dev.lse.fill_(float("nan"))
    dev.decode_splitkv(S)
    torch.cuda.synchronize()
    o_part, lse = dev.o_part.cpu().numpy(), dev.lse.cpu().numpy()
    pieces, Hu = _splitkv_pieces(batch, S, default_num_segments(dev.shape))
    G = Hq // Hu
    for (b, u), rng in pieces.items():
        assert len(rng) <= S
        beg = np.array([r[0] for r in rng] + [rng[-1][1]] if rng else [0, 0], np.int32)
        for g in range(G):
            h = u * G + g
            if rng:
                o_ref, l_ref = oracle.token_partials(batch.q, kp, vp, batch.block_tables,
                                                     batch.seq_lens, batch.sm_scale, b, h, beg,
                                                     Hkv=Hkv, block_size=bs, k_scale=ks,
                                                     v_scale=vs)
                assert_close(o_part[b, h, :len(rng)], o_ref, batch, f"o_part b={b} h={h}")
                assert np.all(np.abs(lse[b, h, :len(rng)] - l_ref) <= 1e-3), (b, h)
            assert np.all(lse[b, h, len(rng):] == -np.inf), (b, h)
    assert_close(dev.out.cpu().numpy(), ref, batch, f"merged S={S}")
    assert dev.read_err() == 0


@pytest.mark.parametrize("S,D", [(6, 128), (40, 128), (33, 64)])
def test_merge_lse_of_oracle_partials(S, D):
    """pa_merge_lse fed with partials it did not write: the oracle's partials over random
    token cuts (empty pieces included), in random slots, with NaN in the o rows of empty
    slots (which must not be read); against the oracle's merge of the same fp32 inputs and
    its plain decode.  More than 32 slots take the merge's chunk loop."""
    batch = wl.build_batch("t", [1, 40, 300, 0, 777, 16], Hq=16, Hkv=4, D=D, block_size=16,
                           seed=310 + S)
    B, Hq = batch.B, batch.Hq
    full = oracle.paged_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                               batch.seq_lens, batch.sm_scale, Hkv=4, block_size=16)
    rng = np.random.default_rng(11)
    o_part = np.full((B, Hq, S, D), np.nan, np.float32)
    lse = np.full((B, Hq, S), -np.inf, np.float32)
    for b in range(B):
        L = int(batch.seq_lens[b])
        for h in range(Hq):
            npc = int(rng.integers(1, S + 1))
            cuts = np.sort(rng.integers(0, L + 1, npc - 1))
            beg = np.concatenate([[0], cuts, [L]]).astype(np.int32)
            o, l = oracle.token_partials(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                         batch.seq_lens, batch.sm_scale, b, h, beg, Hkv=4,
                                         block_size=16)
            slots = rng.permutation(S)[:npc]
            for i, sl in enumerate(slots):
                if l[i] != -np.inf:
                    o_part[b, h, sl] = o[i]
                    lse[b, h, sl] = l[i]
    want = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            want[b, h] = oracle.merge_lse(o_part[b, h].astype(np.float64), lse[b, h].astype(np.float64))
    dev = DeviceBatch(batch)
    do, dl = torch.from_numpy(o_part).cuda(), torch.from_numpy(lse).cuda()
    dev.out.fill_(float("nan"))
    _lib.pa_merge_lse(dev.shape, dev.out, do, dl, S)
    torch.cuda.synchronize()
    got = dev.out.cpu().numpy()
    assert np.isfinite(got).all()
    assert_close(got, want, batch, "merge of oracle partials vs oracle merge")
    assert_close(got, full, batch, "merge of oracle partials vs plain decode")
    assert not got[3].any()                      # sequence of length 0: every slot empty


def _run_cascade(dev, num_splits):
    dev.out.fill_(float("nan"))
    dev.decode_segments(num_splits, cascade=True)
    torch.cuda.synchronize()
    return dev.out.cpu().numpy()


CASCADE_CASES = [
    # Hq, Hkv, D, bs, groups [(prefix, suffixes)], ungrouped lengths
    (64, 8, 128, 16, [(900, [1, 5, 17, 300, 2, 64, 40, 1000]), (300, [3, 30])], [7, 500, 1]),
    (64, 8, 128, 16, [(2000, [1, 2, 3])], [100]),                    # four pieces per member
    (16, 4, 64, 32, [(97, [1, 31, 32, 200]), (64, [50])], [1, 70]),  # G = 4, bs = 32
    (32, 2, 128, 16, [(500, [9, 90, 900]), (16, [1, 2])], [33]),     # G = 16 (two n-tiles)
    (8, 8, 128, 16, [(160, [5, 6, 7, 8, 9])], []),                   # G = 1
    # 160 stacked rows (two chunks of 128, the second part padding); two pieces
    (64, 8, 128, 16, [(1100, [1 + i % 7 for i in range(20)])], [3]),
    (32, 8, 128, 32, [(704, list(range(1, 41))), (32, [4, 4])], [9]),  # G = 4, bs = 32
]


@pytest.mark.parametrize("Hq,Hkv,D,bs,groups,free", CASCADE_CASES)
def test_cascade_matches_oracle(Hq, Hkv, D, bs, groups, free):
    """Shared prefixes attended once per group (stacked queries), the rest per
    sequence, joined by the merge: equal to the plain decode of the oracle."""
    batch, cg = _cascade_batch(Hq, Hkv, D, bs, groups, free, seed=Hq + D + bs)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    for side in (True, False):        # the cascade beside the split kernel, or after it
        dev.enable_cascade(cg, side_stream=side)
        for ns in (1, 3, 17, 64, 500, default_num_segments(dev.shape)):
            assert_close(_run_cascade(dev, ns), ref, batch, f"cascade side={side} segments={ns}")
    assert dev.read_err() == 0



QUANT_CASCADE_CASES = [
    (64, 8, 16, [(900, [1, 5, 17, 300, 2, 64, 40, 1000]), (300, [3, 30])], [7, 500, 1]),
    (64, 8, 16, [(2000, [1, 2, 3])], [100]),                          # four pieces per member
    (32, 2, 16, [(500, [9, 90, 900]), (16, [1, 2])], [33]),           # G = 16 (two n-tiles)
    (8, 8, 16, [(160, [5, 6, 7, 8, 9])], []),                         # G = 1
    (32, 8, 32, [(704, list(range(1, 41))), (32, [4, 4])], [9]),      # G = 4, bs = 32
]


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "int4"])
@pytest.mark.parametrize("Hq,Hkv,bs,groups,free", QUANT_CASCADE_CASES)
def test_cascade_quantised_matches_oracle(kv_dtype, Hq, Hkv, bs, groups, free):
    """The cascade over E4M3 and 4-bit pools (codes restored with their block scales,
    this step's quantised cache write applied first): equal to the oracle's plain decode
    at the quantised tolerance, beside or after the split kernel, at several segment
    counts."""
    batch, cg = _cascade_batch(Hq, Hkv, 128, bs, groups, free, seed=300 + Hq + bs,
                               kv_dtype=kv_dtype)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    for side in (True, False):
        dev.enable_cascade(cg, side_stream=side)
        for ns in (1, 17, 500, default_num_segments(dev.shape)):
            assert_close(_run_cascade(dev, ns), ref, batch,
                         f"{kv_dtype} cascade side={side} segments={ns}")
    assert dev.read_err() == 0


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "int4"])
def test_cascade_quantised_scale_spread(kv_dtype):
    """Quantised cascade with K and V block scales spread over 2^-12 .. 2^6 (the
    accumulator is re-expressed when a tile's V-scale ratio leaves [2^-12, 2^7]; large
    restored V values) and a zero V scale on some blocks."""
    batch, cg = _cascade_batch(64, 8, 128, 16, [(1200, [1, 9, 300]), (320, [4, 60])], [77],
                               seed=311, kv_dtype=kv_dtype)
    rng = np.random.default_rng(311)
    batch.k_scale[...] = (2.0 ** rng.uniform(-12, 2, batch.k_scale.shape)).astype(np.float32)
    batch.v_scale[...] = (2.0 ** rng.uniform(-12, 6, batch.v_scale.shape)).astype(np.float32)
    batch.v_scale[rng.random(batch.v_scale.shape) < 0.05] = 0.0
    dev = DeviceBatch(batch)
    ref, _ = oracle_after_write(batch, write=False)
    dev.enable_cascade(cg)
    for ns in (1, 9, default_num_segments(dev.shape)):
        assert_close(_run_cascade(dev, ns), ref, batch, f"{kv_dtype} cascade scale spread {ns}")
    assert dev.read_err() == 0


@pytest.mark.parametrize("kv_dtype", ["bf16", "int4"])
def test_cascade_through_pa_decode(kv_dtype):
    """pa_decode with a workspace runs the split decode with the cascade and the merge in
    one call; without a workspace it ignores the groups and attends over every token (on
    4-bit pools: heads read in pairs without the cascade, one at a time with it)."""
    batch, cg = _cascade_batch(64, 8, 128, 16, [(900, [1, 5, 17, 300]), (300, [3, 30])],
                               [7, 500], seed=152, kv_dtype=kv_dtype)
    dev = DeviceBatch(batch)
    dev.enable_cascade(cg)
    ref, _ = oracle_after_write(batch, write=False)
    for ns in (0, 13):
        dev.ensure_workspace(ns or default_num_segments(dev.shape))
        for ws in (dev.workspace, None):
            dev.out.fill_(float("nan"))
            _lib.pa_decode(dev.shape, dev.out, dev.q, dev.k_pool, dev.v_pool, dev.k_scale,
                           dev.v_scale, dev.block_tables, dev.seq_lens, batch.sm_scale, dev.err,
                           None,
                           workspace=ws, num_segments=ns, shared_prefix_lens=dev.shared_prefix_lens,
                           cascade=dev.cascade)
            torch.cuda.synchronize()
            assert_close(dev.out.cpu().numpy(), ref, batch,
                         f"{kv_dtype} pa_decode cascade workspace={ws is not None} segments={ns}")
    assert dev.read_err() == 0


def test_cascade_prefix_is_whole_sequence():
    """Members whose every token is in the shared prefix (nothing left for the split
    kernel) and groups with a zero-length prefix."""
    batch, cg = _cascade_batch(64, 8, 128, 16, [(320, [0, 0, 16, 1]), (48, [2, 3])], [5],
                               seed=101)
    dev = DeviceBatch(batch)
    ref, _ = oracle_after_write(batch, write=False)
    offsets, seqs, plen = cg
    plen2 = plen.copy()
    plen2[1] = 0                                    # the second group shares nothing
    for groups in ((offsets, seqs, plen), (offsets, seqs, plen2)):
        dev.enable_cascade(groups)
        for ns in (1, 5, 77):
            assert_close(_run_cascade(dev, ns), ref, batch, f"cascade whole prefix {ns}")
    assert dev.read_err() == 0


def test_cascade_bad_groups_set_error_flag():
    """A member shorter than its group's prefix, or a sequence in two groups, is a
    caller error: the device flag reports it, nothing faults."""
    batch, (offsets, seqs, plen) = _cascade_batch(64, 8, 128, 16, [(64, [5, 6])], [9], seed=102)
    dev = DeviceBatch(batch)
    dev.enable_cascade((offsets, seqs, np.array([96], np.int32)))       # 96 > 64 + 5
    _run_cascade(dev, 7)
    assert dev.read_err() & _lib.PA_DEVERR_SEQ_LEN
    dev.err.zero_()
    two = (np.array([0, 2, 3], np.int32), np.array([0, 1, 0], np.int32),
           np.array([64, 64], np.int32))                               # sequence 0 twice
    dev.enable_cascade(two)
    _run_cascade(dev, 7)
    assert dev.read_err() & _lib.PA_DEVERR_SEQ_LEN


def test_largest_split_batch_and_split_count():
    """16,384 sequences (the split kernel's largest batch: its length scan sits in shared
    memory; also pa_decode's largest longest-first batch, 128 sequences per thread in its
    search) of 1..48 tokens, then 65,536 splits (the largest count) on a small batch."""
    rng = np.random.default_rng(120)
    lens = rng.integers(1, 49, 16384)
    batch = wl.build_batch("t", lens, Hq=16, Hkv=2, D=64, block_size=16, seed=120)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    out = run_gpu(dev, "split", default_num_segments(dev.shape))
    assert dev.read_err() == 0
    rows = np.stack([rng.integers(0, batch.B, 512), rng.integers(0, batch.Hq, 512)], 1)
    rows = np.concatenate([rows, [[0, 0], [batch.B - 1, batch.Hq - 1]]]).astype(np.int32)
    ref, _ = oracle_after_write(batch, rows=rows)
    assert_close(out[rows[:, 0], rows[:, 1]], ref, batch, "B = 16384")
    out = run_gpu(dev, "decode")
    assert dev.read_err() == 0
    assert_close(out[rows[:, 0], rows[:, 1]], ref, batch, "B = 16384, pa_decode")
    small = wl.build_batch("t", [1, 700, 33], Hq=64, Hkv=8, D=128, block_size=16, seed=121)
    dev = DeviceBatch(small)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(small)
    assert_close(run_gpu(dev, "split", 65536), ref, small, "65536 splits")
    assert dev.read_err() == 0


def test_cascade_many_small_groups():
    """500 groups of two sequences each (the cascade's group scan spans many groups)."""
    groups = [(16 * (1 + g % 9), [1 + g % 5, 2]) for g in range(500)]
    batch, cg = _cascade_batch(32, 4, 128, 16, groups, [3, 100], seed=122)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    dev.enable_cascade(cg)
    ref, _ = oracle_after_write(batch)
    for ns in (7, default_num_segments(dev.shape)):
        assert_close(_run_cascade(dev, ns), ref, batch, f"500 groups segments={ns}")
    assert dev.read_err() == 0



@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_unattended_rows_hold_nonfinite_values(kv_dtype):
    """Pool rows a decode does not attend -- past a sequence's length in its last block,
    and before a window's start inside the first tile it keeps -- hold NaN and Inf
    (E4M3 NaN codes for FP8).  Every decode path gives the same bits as with clean rows:
    those rows are masked, not multiplied by a zero weight."""
    lens = [5, 17, 31, 100, 333]
    W = 20
    batch = wl.build_batch("t", lens, Hq=32, Hkv=4, D=128, block_size=16, seed=170,
                           kv_dtype=kv_dtype)
    clean = DeviceBatch(batch)
    runs = [(mode, ns, w) for w in (0, W) for mode, ns in (("decode", None), ("decode_ws", None),
                                                            ("split", 1), ("split", 9))]
    want = [run_gpu(clean, m, ns, w).copy() for m, ns, w in runs]
    bad_k, bad_v = (0x7FC0, 0x7F80) if kv_dtype == "bf16" else (0x7F, 0xFF)   # NaN, Inf / NaN
    for b, L in enumerate(lens):                                # past the length
        blk = batch.block_tables[b, (L - 1) // 16]
        batch.k_pool[blk, L % 16 or 16:] = bad_k
        batch.v_pool[blk, L % 16 or 16:] = bad_v
    for w in (0, W):
        if w:                                                   # before the window, same tile
            for b, L in enumerate(lens):
                if L <= w:
                    continue
                for t in range(((L - w) // 16) * 16, L - w):
                    batch.k_pool[batch.block_tables[b, t // 16], t % 16] = bad_k
                    batch.v_pool[batch.block_tables[b, t // 16], t % 16] = bad_v
        poisoned = DeviceBatch(batch)
        for (m, ns, ww), ref in zip(runs, want):
            if ww != w:
                continue
            got = run_gpu(poisoned, m, ns, w)
            assert np.isfinite(got).all(), (m, ns, w)
            assert np.array_equal(_bits(got), _bits(ref)), (m, ns, w)
        assert poisoned.read_err() == 0

# ---------------------------------------------------------------- online-softmax reference

def _staircase_keys(batch, seqs, steps, rng):
    """Keys whose scores (log2 units) step by steps[i] from one 16-token tile to the
    next in sequence seqs[i] (None: a random walk of up to +-6 per tile).  Every query
    head of a KV head's group gets the same query u; a key is f u / (|u|^2 sm_scale
    log2 e) plus noise, so its score is about f.  bf16 pools take the keys as they are;
    FP8 and 4-bit pools get absmax codes and scales per (block, KV head) over the rows
    written here, and their V scales are spread over 2^-5 .. 2^5 per block."""
    G, D, bs = batch.Hq // batch.Hkv, batch.D, batch.block_size
    l2 = batch.sm_scale * np.log2(np.e)
    keys = {}
    for b, step in zip(seqs, steps):
        L = int(batch.seq_lens[b])
        ntile = (L + 15) // 16
        f = (np.arange(ntile) * step if step is not None
             else np.cumsum(rng.uniform(-6, 6, ntile)))
        for h in range(batch.Hkv):
            ub = wl.bf16_bits(rng.standard_normal(D).astype(np.float32))
            batch.q[b, h * G:(h + 1) * G] = ub
            uf = wl.bf16_to_float(ub).astype(np.float64)
            for t in range(L):
                k = f[t // 16] / l2 * uf / uf.dot(uf) + 0.05 * rng.standard_normal(D)
                keys.setdefault((int(batch.block_tables[b, t // bs]), h), {})[t % bs] = k
    for (blk, h), rows in keys.items():
        if batch.kv_dtype == "bf16":
            for r, k in rows.items():
                batch.k_pool[blk, r, h] = wl.bf16_bits(k.astype(np.float32))
            continue
        amax = max(np.abs(k).max() for k in rows.values())
        if batch.kv_dtype == "fp8_e4m3":
            scale = np.float32(amax / 448.0)
            for r, k in rows.items():
                batch.k_pool[blk, r, h] = oracle.e4m3_from_float((k / scale).astype(np.float32))
        else:
            scale = np.float32(amax / 7.0)
            for r, k in rows.items():
                c = np.clip(np.rint(k / scale), -7, 7).astype(np.int16) + 8
                batch.k_pool[blk, r, h] = (c[0::2] | (c[1::2] << 4)).astype(np.uint8)
        batch.k_scale[blk, h] = scale
        batch.v_scale[blk, h] *= np.float32(2.0 ** rng.uniform(-5, 5))


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "int4"])
def test_softmax_reference_staircase_scores(kv_dtype):
    """Scores that climb by 10 per tile (the running maximum moves on every tile), by 3
    per tile (it stays up to 2^8 above an older reference for several tiles), fall by
    2 per tile, or wander: every decode path against the oracle.  Quantised pools add
    V scales over ten octaves, so P times the V-scale ratio must stay inside f16."""
    batch = wl.build_batch("t", [700, 900, 500, 800], Hq=32, Hkv=4, D=128, block_size=16,
                           seed=140, kv_dtype=kv_dtype)
    _staircase_keys(batch, [0, 1, 2, 3], [10.0, 3.0, -2.0, None], np.random.default_rng(140))
    dev = DeviceBatch(batch)
    ref, _ = oracle_after_write(batch, write=False)
    for mode, ns in MODES:
        ns = _mode_count(dev, mode, ns)
        out = run_gpu(dev, mode, ns)
        assert np.isfinite(out).all(), (mode, ns)
        assert_close(out, ref, batch, f"{kv_dtype} staircase {mode} {ns}")
    assert dev.read_err() == 0


def test_cascade_staircase_prefix():
    """The cascade kernel's running maximum per stacked row: a shared prefix whose
    scores climb by 10 per tile (every tile moves it) and one whose scores climb by 3
    (weights up to 2^8 against an older reference), joined with the suffixes."""
    batch, cg = _cascade_batch(32, 4, 128, 16, [(1100, [1, 40, 7]), (640, [3, 300])], [50],
                               seed=141)
    # the prefix blocks are shared: one member per group writes them, the others take
    # its query so the whole group sees the staircase
    _staircase_keys(batch, [2, 4, 5], [10.0, 3.0, None], np.random.default_rng(141))
    batch.q[[0, 1]] = batch.q[2]
    batch.q[3] = batch.q[4]
    dev = DeviceBatch(batch)
    dev.enable_cascade(cg)
    ref, _ = oracle_after_write(batch, write=False)
    for ns in (1, 9, default_num_segments(dev.shape)):
        assert_close(_run_cascade(dev, ns), ref, batch, f"staircase cascade segments={ns}")
    assert dev.read_err() == 0


@pytest.mark.parametrize("mode", ["split", "cascade", "fp8", "decode"])
def test_step_captured_in_cuda_graph(mode):
    """One decode step (cache write, split decode, merge; with the cascade also its plan,
    side-stream fork and join; "decode": pa_decode without a workspace, here a cluster
    launch) captured into a CUDA graph and replayed: the replay gives the oracle's
    result.  The step's launches chain by programmatic dependent launch, which the graph
    keeps."""
    if mode == "fp8":
        batch = wl.build_batch("t", [1, 40, 300, 17], Hq=64, Hkv=8, D=128, block_size=16,
                               seed=111, kv_dtype="fp8_e4m3")
        cg = None
    else:
        batch, cg = _cascade_batch(64, 8, 128, 16, [(400, [3, 50, 7]), (96, [1, 2])], [33, 5],
                                   seed=110)
    dev = DeviceBatch(batch)
    ns = 37
    dev.ensure_workspace(ns)
    if mode == "cascade":
        dev.enable_cascade(cg)

    def step():
        dev.reshape_and_cache()
        if mode == "decode":
            dev.decode()
        else:
            dev.decode_segments(ns, cascade=(mode == "cascade"))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                  # warm-up outside the capture
        for _ in range(3):
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    ref, _ = oracle_after_write(batch)
    for _ in range(2):
        dev.out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert_close(dev.out.cpu().numpy(), ref, batch, f"graph replay {mode}")
    assert dev.read_err() == 0


@pytest.mark.parametrize("name", ["llama70b_layer", "prefix_sharing", "long_context", "fp8_mixed",
                                  "int4_mixed", "code_assistant_turns"])
def test_full_size_config_sampled(name):
    """The bench's launch configurations at full size (pa_decode_splitkv + pa_merge_lse
    at the default slots, the split decode at the default segments) and pa_decode
    without a workspace (the call the FP8 workload names; a cluster of CTAs per unit on
    the 70B and long-context batches, longest sequences first on the prefix batch);
    every head of the longest, shortest and three random sequences plus 192 random
    (b, h) rows are compared with the oracle."""
    batch = wl.make(name)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    out = run_gpu(dev, "parts", default_num_splits(dev.shape))
    assert dev.read_err() == 0
    rows = _sample_rows(batch, np.random.default_rng(7))
    ref, _ = oracle_after_write(batch, rows=rows)
    assert_close(out[rows[:, 0], rows[:, 1]], ref, batch, name + " splitkv + merge")
    out = run_gpu(dev, "split", default_num_segments(dev.shape))
    assert dev.read_err() == 0
    assert_close(out[rows[:, 0], rows[:, 1]], ref, batch, name + " segments")
    out_ws = run_gpu(dev, "decode_ws")            # the one-call form of the same path
    assert dev.read_err() == 0
    assert_close(out_ws[rows[:, 0], rows[:, 1]], ref, batch, name + " pa_decode + workspace")
    out2 = run_gpu(dev, "decode")                 # pa_decode without a workspace, same rows
    assert dev.read_err() == 0
    assert_close(out2[rows[:, 0], rows[:, 1]], ref, batch, name + " decode")
    # its CTAs merge their warps' states through shared memory (and a cluster's CTAs
    # through distributed shared memory): a second call must give the same bits
    # everywhere (a race there shows up as a few stray values)
    assert np.array_equal(_bits(run_gpu(dev, "decode")), _bits(out2)), name + " decode not repeatable"
    if name in ("prefix_sharing", "code_assistant_turns"):   # the cascade (bench.py --cascade)
        out3 = _run_cascade(dev, default_num_segments(dev.shape))
        assert dev.read_err() == 0
        assert_close(out3[rows[:, 0], rows[:, 1]], ref, batch, name + " cascade")



def test_two_streams_decode_concurrently():
    """Two batches, each with its own workspace, cascade groups and cascade side stream,
    decoded over and over on two caller streams at once: neither result may see the
    other's work."""
    b1, cg1 = _cascade_batch(64, 8, 128, 16, [(900, [1, 5, 17, 300]), (300, [3, 30])], [7, 500],
                             seed=150)
    b2, cg2 = _cascade_batch(32, 4, 128, 16, [(1600, [2, 9, 40]), (64, [5])], [1000, 3],
                             seed=151)
    d1, d2 = DeviceBatch(b1), DeviceBatch(b2)
    d1.enable_cascade(cg1)
    d2.enable_cascade(cg2)
    ref1, _ = oracle_after_write(b1, write=False)
    ref2, _ = oracle_after_write(b2, write=False)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ns1, ns2 = default_num_segments(d1.shape), 77
    torch.cuda.synchronize()
    for _ in range(20):
        d1.decode_segments(ns1, stream=s1.cuda_stream, cascade=True)
        d2.decode_segments(ns2, stream=s2.cuda_stream, cascade=True)
    torch.cuda.synchronize()
    assert_close(d1.out.cpu().numpy(), ref1, b1, "stream 1")
    assert_close(d2.out.cpu().numpy(), ref2, b2, "stream 2")
    assert d1.read_err() == 0 and d2.read_err() == 0

# ---------------------------------------------------------------- failure handling

def test_bounded_wait_reports_timeout_and_context_survives(tmp_path):
    """A pipeline wait that nothing completes: the library's bounded mbarrier wait (here
    with a short bound) gives up, the kernel sets PA_DEVERR_TIMEOUT and returns, and
    the same context then runs a decode that matches the oracle.  The kernel is built
    here from tests/csrc/wait_timeout.cu against the library's own wait helper."""
    import ctypes
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    so = str(tmp_path / "libwait_timeout.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared",
                    "-I", os.path.join(root, "include"),
                    "-I", os.path.join(root, "paged_kv_cache_28_gb300", "csrc"),
                    os.path.join(root, "tests", "csrc", "wait_timeout.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.run_wait_nothing_arrives.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    flags = torch.zeros(2, dtype=torch.int32, device="cuda")
    rc = lib.run_wait_nothing_arrives(flags.data_ptr(), flags.data_ptr() + 4)
    assert rc == 0                                   # the kernel returned: no fault, no hang
    err, finished = flags.cpu().tolist()
    assert err & _lib.PA_DEVERR_TIMEOUT and finished == 1
    batch = wl.make("tiny")
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    assert_close(run_gpu(dev, "split", 3), ref, batch, "after a timed-out wait")
    assert dev.read_err() == 0


def test_c_program_drives_the_abi(tmp_path):
    """The C ABI from plain C99 and the CUDA runtime, no Python in the loop
    (tests/c/decode_from_c.c): cache write, then pa_decode_splitkv + pa_merge_lse,
    pa_decode with and without a workspace, and pa_merge_lse of the oracle's partials
    over random token cuts, on a small bf16 batch, against the oracle."""
    import shutil
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(shutil.which("nvcc"))))
    pkg = os.path.join(root, "paged_kv_cache_28_gb300")
    exe = str(tmp_path / "decode_from_c")
    subprocess.run(["gcc", "-std=c99", "-O2", "-I", os.path.join(root, "include"),
                    "-I", os.path.join(cuda, "include"), os.path.join(root, "tests", "c", "decode_from_c.c"),
                    "-L", pkg, "-lpa", "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    "-Wl,-rpath," + pkg, "-o", exe], check=True)
    batch = wl.build_batch("t", [1, 17, 33, 100, 300], Hq=16, Hkv=2, D=128, block_size=16, seed=160)
    ref, (kp, vp, _, _) = oracle_after_write(batch)
    S_ext = 4
    rng = np.random.default_rng(12)
    ext_o = np.full((batch.B, batch.Hq, S_ext, batch.D), np.nan, np.float32)
    ext_l = np.full((batch.B, batch.Hq, S_ext), -np.inf, np.float32)
    for b in range(batch.B):
        L = int(batch.seq_lens[b])
        for h in range(batch.Hq):
            beg = np.concatenate([[0], np.sort(rng.integers(0, L + 1, S_ext - 1)), [L]])
            o, l = oracle.token_partials(batch.q, kp, vp, batch.block_tables, batch.seq_lens,
                                         batch.sm_scale, b, h, beg.astype(np.int32), Hkv=2,
                                         block_size=16)
            keep = l != -np.inf
            ext_o[b, h, keep], ext_l[b, h, keep] = o[keep], l[keep]
    inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([batch.B, batch.Hq, batch.Hkv, batch.D, batch.block_size, batch.nblocks,
                          batch.max_blocks, 7, 29, S_ext], np.int32).tobytes())
        f.write(np.array([batch.sm_scale], np.float32).tobytes())
        for a in (batch.q, batch.k_pool, batch.v_pool, batch.k_new, batch.v_new,
                  batch.block_tables.astype(np.int32), batch.seq_lens.astype(np.int32),
                  batch.slot_mapping.astype(np.int64), ext_o, ext_l):
            f.write(np.ascontiguousarray(a).tobytes())
    subprocess.run([exe, str(inp), str(outp)], check=True)
    raw = np.fromfile(outp, dtype=np.uint8)
    n = batch.B * batch.Hq * batch.D
    outs = raw[:16 * n].view(np.float32).reshape(4, batch.B, batch.Hq, batch.D)
    assert raw[16 * n:].view(np.int32)[0] == 0
    assert_close(outs[0], ref, batch, "from C: pa_decode_splitkv + pa_merge_lse")
    assert_close(outs[1], ref, batch, "from C: pa_decode with a workspace")
    assert_close(outs[2], ref, batch, "from C: pa_decode")
    assert_close(outs[3], ref, batch, "from C: pa_merge_lse of the oracle's partials")
