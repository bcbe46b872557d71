"""Randomised parity sweep (GPU): seeded random decode problems through every decode call.

Each case draws a shape -- D, KV heads, group size G (1..16, including groups that pad an
8-row n-tile), block size, KV dtype -- and lengths that favour tile and block edges
(0, 1, 15, 16, 17, 31, 32, 33 and random ones), writes this step's tokens through the
cache write, then runs pa_decode with and without a workspace and pa_decode_splitkv +
pa_merge_lse at random segment / slot counts, with and without a sliding window, each
against the oracle at its tolerance.  Cases are fixed by their seeds, so a failure
reproduces exactly.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_28_gb300 import workload as wl
from paged_kv_cache_28_gb300.device import DeviceBatch

from paged_kv_cache_28_gb300 import _lib
from test_gpu_parity import assert_close, oracle_after_write, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    _lib.load()

EDGE_LENS = [0, 1, 15, 16, 17, 31, 32, 33, 47, 48, 49]


def _case(seed):
    rng = np.random.default_rng(10_000 + seed)
    kv = ["bf16", "bf16", "fp8_e4m3", "int4"][seed % 4]
    D = 128 if kv != "bf16" else int(rng.choice([64, 128]))
    G = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))
    Hkv = int(rng.choice([1, 2, 3, 4, 8]))
    bs = int(rng.choice([16, 32]))
    B = int(rng.integers(1, 24))
    lens = [int(x) for x in rng.choice(EDGE_LENS, B)]
    lens = [L if rng.random() < 0.5 else int(rng.integers(0, 700)) for L in lens]
    if max(lens) == 0:
        lens[0] = 1
    window = int(rng.choice([0, 0, 1, 16, 17, 100]))
    return dict(kv=kv, D=D, G=G, Hkv=Hkv, bs=bs, lens=lens, window=window,
                rng_seed=20_000 + seed)


@pytest.mark.parametrize("seed", range(40))
def test_random_shapes(seed):
    c = _case(seed)
    batch = wl.build_batch("rand", c["lens"], Hq=c["G"] * c["Hkv"], Hkv=c["Hkv"], D=c["D"],
                           block_size=c["bs"], seed=c["rng_seed"], kv_dtype=c["kv"])
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    label = f"seed {seed} {c}"
    rng = np.random.default_rng(30_000 + seed)
    for window in sorted({0, c["window"]}):
        ref, _ = oracle_after_write(batch, window=window)
        modes = [("decode", None), ("decode_ws", None),
                 ("split", int(rng.integers(1, 200))), ("parts", int(rng.integers(1, 9)))]
        for mode, ns in modes:
            out = run_gpu(dev, mode, ns, window=window)
            assert_close(out, ref, batch, f"{label} window={window} {mode} {ns}")
    assert dev.read_err() == 0
