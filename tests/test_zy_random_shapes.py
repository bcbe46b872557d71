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


def _page_scores(batch):
    """[b, kvh] -> exact group-max score of every page, over the oracle's stored summaries."""
    import oracle
    bs, G = batch.block_size, batch.Hq // batch.Hkv
    q = wl.bf16_to_float(batch.q).astype(np.float64)
    out = {}
    for b in range(batch.B):
        L = int(batch.seq_lens[b])
        for h in range(batch.Hkv):
            sc = []
            for j in range((L + 15) // 16):
                page = batch.block_tables[b, 16 * j // bs] * (bs // 16) + (16 * j % bs) // 16
                mn, mx = oracle.quest_page_summary(batch.k_pool, page, min(16, L - 16 * j), h,
                                                   Hkv=batch.Hkv, D=batch.D, block_size=bs,
                                                   k_scale=batch.k_scale)
                qs = q[b, h * G:(h + 1) * G]
                sc.append(max(oracle.page_score(qs[g], mn, mx) for g in range(G)))
            out[b, h] = np.array(sc)
    return out


@pytest.mark.parametrize("seed", range(16))
def test_random_quest(seed):
    """Quest on random shapes and pool kinds: the GPU's pages are a valid top-k of the
    oracle's exact scores (up to fp32 rounding between near-equal pages), and every row's
    output matches the oracle's decode over those pages, in a random decode call."""
    import oracle
    c = _case(100 + seed)
    batch = wl.build_batch("rand", c["lens"], Hq=c["G"] * c["Hkv"], Hkv=c["Hkv"], D=c["D"],
                           block_size=c["bs"], seed=c["rng_seed"], kv_dtype=c["kv"])
    dev = DeviceBatch(batch)
    rng = np.random.default_rng(40_000 + seed)
    topk = int(rng.integers(1, 12))
    dev.quest_build_summaries()
    sel = dev.quest_select(topk)
    torch.cuda.synchronize()
    gsel = sel.cpu().numpy()
    for (b, h), sc in _page_scores(batch).items():
        g = gsel[b, h]
        n = min(topk, sc.size)
        assert np.all(g[n:] == -1) and np.all(np.diff(g[:n]) > 0), (seed, b, h)
        if n:
            kth = np.sort(sc)[::-1][n - 1]
            assert sc[g[:n]].min() >= kth - 1e-4 * max(1.0, abs(kth)), (seed, b, h)
    ref = oracle.paged_decode_pages(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                                    batch.seq_lens, batch.sm_scale, gsel, Hkv=batch.Hkv,
                                    block_size=batch.block_size, k_scale=batch.k_scale,
                                    v_scale=batch.v_scale)
    call = ["decode", "split", "parts"][seed % 3]
    dev.out.fill_(float("nan"))
    if call == "decode":
        dev.decode(selected_pages=sel)
    elif call == "parts":
        dev.decode_splitkv(int(rng.integers(1, 9)), selected_pages=sel)
    else:
        dev.decode_segments(int(rng.integers(1, 200)), selected_pages=sel)
    torch.cuda.synchronize()
    assert_close(dev.out.cpu().numpy(), ref, batch, f"quest seed {seed} {c} topk={topk} {call}")
    assert dev.read_err() == 0


@pytest.mark.parametrize("seed", range(16))
def test_random_cascade(seed):
    """The cascade on random groups: prefix lengths (multiples of 16), member counts,
    suffixes, free sequences, pool kinds and group sizes; beside or after the split kernel
    at a random segment count; against the oracle's plain decode."""
    from paged_kv_cache_28_gb300.workload import cascade_groups
    rng = np.random.default_rng(50_000 + seed)
    kv = ["bf16", "fp8_e4m3", "int4", "bf16"][seed % 4]
    D = 128 if kv != "bf16" else int(rng.choice([64, 128]))
    G = int(rng.choice([1, 2, 4, 6, 8, 16]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([16, 32]))
    groups, lens, b = [], [], 0
    for _ in range(int(rng.integers(1, 4))):
        plen = 16 * int(rng.integers(1, 40))
        # at least one private token each: this step's new token lands after the prefix
        sfx = [int(x) for x in rng.integers(1, 300, int(rng.integers(1, 7)))]
        groups.append((plen, list(range(b, b + len(sfx)))))
        lens += [plen + s for s in sfx]
        b += len(sfx)
    lens += [int(x) for x in rng.integers(0, 400, int(rng.integers(0, 4)))]
    if max(lens) == 0:
        lens[0] = 1
    batch = wl.build_batch("rand", lens, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs,
                           seed=60_000 + seed, kv_dtype=kv, prefix_groups=groups)
    dev = DeviceBatch(batch)
    dev.reshape_and_cache()
    ref, _ = oracle_after_write(batch)
    dev.enable_cascade(cascade_groups(batch), side_stream=bool(seed % 2))
    ns = int(rng.integers(1, 300))
    dev.out.fill_(float("nan"))
    dev.decode_segments(ns, cascade=True)
    torch.cuda.synchronize()
    label = f"cascade seed {seed} kv={kv} D={D} G={G} Hkv={Hkv} bs={bs} groups={groups} ns={ns}"
    assert_close(dev.out.cpu().numpy(), ref, batch, label)
    assert dev.read_err() == 0
