"""CPU oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.

The oracle is a plain, slow C library (``pa_oracle.c``, fp64 unless a step
fixes its own precision) and this ctypes wrapper around it.  It checks the CUDA
path; it is not part of it.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import it.  It imports
nothing from the ``paged_kv_cache_28_gb300`` package and the package never
imports it.

Functions and what pins each one (tests in ``tests/test_oracle_pins.py``):

=============================  ==============================================
function                       pinned by
=============================  ==============================================
kv_head                        the GQA/MHA/MQA head mappings printed in
                               "KV Cache Engineering for LLM Serving", sec. 1
cached_scalars                 the 768/192/96 scalar counts of the same
                               example; the 320 KB/token figure of
                               "appendonly" (Paging); the 8 GB pool capacities
                               of "KV Cache Engineering", sec. 10
quantize_absmax_int            the 4-bit codes and restored values printed in
                               "KV Cache Engineering", sec. 8
e4m3_to_double                 closed-form values of the OFP8 E4M3 format and
                               torch.float8_e4m3fn (all 256 codes)
e4m3_from_float                torch.float8_e4m3fn rounding on every finite
                               bf16 pattern x several scales; saturation
reshape_and_cache_bf16         canary-filled pools: exactly the addressed
                               rows change, byte for byte
reshape_and_cache_fp8          closed-form scale/requantisation cases built by
                               hand from the reading in pa_oracle.c
reshape_and_cache_int4         the 4-bit codes and restored values printed in
                               "KV Cache Engineering", sec. 8, through the
                               writer; closed-form growth/requantisation cases
int4_restore                   closed form (nibble - 8) * scale
paged_decode                   numpy/scipy softmax attention on contiguous
                               (unpaged) K/V; L=1 -> V; q=0 -> mean(V);
                               L=2 logistic closed form; needle; block
                               permutation and shared-vs-copied prefix
                               invariance; GQA grouping
window_positions               the four-token window trace printed in
                               "KV Cache Engineering", sec. 3
paged_decode(window=W)         numpy/scipy attention over the last W rows of
                               the contiguous K/V; W >= L equals no window
page_summary / page_score /    the Quest example printed in "KV Cache
select_pages                   Engineering", sec. 7 (scores 2.5, 6.0, 4.0,
                               -1.0; pages [1, 2]); brute force over all
                               key choices for the upper-bound property
quest_decode                   textbook attention restricted to the chosen
                               pages' tokens (numpy), topk >= pages equals
                               full decode; selection by brute-force scores;
                               on E4M3 / 4-bit pools with power-of-two scales
                               equal to Quest over bf16 pools of the restored
                               values; with other scales the top-k of numpy
                               scores over outward-rounded summaries
quest_page_summary             numpy min / max of the page's restored keys
                               (torch E4M3 decode, nibbles by hand), rounded
                               outward by a search of the neighbouring bf16
                               bit patterns, element-exact
bf16_round_down / _up          the neighbouring bf16 bit patterns of x (the
                               largest <= x, the smallest >= x); bf16 values
                               are fixed points; round_down(-x) = -round_up(x)
split_partials / merge_lse     merge(split(x)) == unsplit(x) to 1e-12 for
                               random splits; one split is the identity;
                               empty splits carry no weight
token_partials                 block-aligned cuts equal split_partials;
                               merge over random token cuts (16-token and
                               ragged) == unsplit to 1e-12; a one-token
                               piece has lse = score, o = its V row
paged_decode_pages             every page chosen == paged_decode; one page ==
                               numpy softmax over that page's rows; chosen
                               pages == merge of one-page partials; the
                               pages quest_decode chooses give its output
=============================  ==============================================

No function is left unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-std=c99", "-Wall"]


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` into ``liboracle.so`` next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_bf16_to_double.restype = D
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_e4m3_to_double.restype = D
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
            lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_to_double_array.restype = None
            lib.oracle_e4m3_to_double_array.argtypes = [P, ctypes.c_longlong, P]
            lib.oracle_e4m3_from_float_array.restype = None
            lib.oracle_e4m3_from_float_array.argtypes = [P, ctypes.c_longlong, P]
            lib.oracle_kv_head.restype = I
            lib.oracle_kv_head.argtypes = [I, I, I]
            lib.oracle_cached_scalars.restype = ctypes.c_longlong
            lib.oracle_cached_scalars.argtypes = [I, I, ctypes.c_longlong, I]
            lib.oracle_quantize_absmax_int.restype = None
            lib.oracle_quantize_absmax_int.argtypes = [P, I, I, P, P, P]
            lib.oracle_reshape_and_cache_bf16.restype = None
            lib.oracle_reshape_and_cache_bf16.argtypes = [I, I, I, I, P, P, P, P, P]
            lib.oracle_reshape_and_cache_fp8.restype = None
            lib.oracle_reshape_and_cache_fp8.argtypes = [I, I, I, I, P, P, P, P, P, P, P]
            lib.oracle_reshape_and_cache_int4.restype = None
            lib.oracle_reshape_and_cache_int4.argtypes = [I, I, I, I, P, P, P, P, P, P, P]
            lib.oracle_int4_restore.restype = None
            lib.oracle_int4_restore.argtypes = [P, I, ctypes.c_float, P]
            lib.oracle_page_summary.restype = None
            lib.oracle_page_summary.argtypes = [P, I, I, P, P]
            lib.oracle_page_score.restype = D
            lib.oracle_page_score.argtypes = [P, P, P, I]
            lib.oracle_select_pages.restype = I
            lib.oracle_select_pages.argtypes = [P, I, I, P]
            lib.oracle_quest_decode.restype = None
            lib.oracle_quest_decode.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P, D, I,
                                                P, P, I]
            lib.oracle_quest_page_summary.restype = None
            lib.oracle_quest_page_summary.argtypes = [I, I, I, I, P, P, ctypes.c_longlong, I, I,
                                                      P, P]
            lib.oracle_bf16_round_down.restype = D
            lib.oracle_bf16_round_down.argtypes = [D]
            lib.oracle_bf16_round_up.restype = D
            lib.oracle_bf16_round_up.argtypes = [D]
            lib.oracle_paged_decode.restype = None
            lib.oracle_paged_decode.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P, D,
                                                I, I, P, P, P, I]
            lib.oracle_window_positions.restype = I
            lib.oracle_window_positions.argtypes = [I, I, P]
            lib.oracle_split_partials.restype = None
            lib.oracle_split_partials.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, D,
                                                  I, I, I, P, P, P]
            lib.oracle_token_partials.restype = None
            lib.oracle_token_partials.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, D,
                                                  I, I, I, P, P, P]
            lib.oracle_paged_decode_pages.restype = None
            lib.oracle_paged_decode_pages.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P,
                                                      D, I, P, P, I]
            lib.oracle_merge_lse.restype = None
            lib.oracle_merge_lse.argtypes = [I, I, P, P, P]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    """Contiguous array of the given dtype (no copy when already so)."""
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# scalar formats and small definitions
# --------------------------------------------------------------------------

def bf16_to_double(bits) -> np.ndarray:
    lib = _load()
    bits = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.oracle_bf16_to_double(int(b)) for b in bits.ravel()]).reshape(bits.shape)


def e4m3_to_double(codes) -> np.ndarray:
    lib = _load()
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    lib.oracle_e4m3_to_double_array(_ptr(codes), codes.size, _ptr(out))
    return out


def e4m3_from_float(x) -> np.ndarray:
    lib = _load()
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib.oracle_e4m3_from_float_array(_ptr(x), x.size, _ptr(out))
    return out


def kv_head(h: int, Hq: int, Hkv: int) -> int:
    return _load().oracle_kv_head(h, Hq, Hkv)


def cached_scalars(layers: int, Hkv: int, tokens: int, D: int) -> int:
    return _load().oracle_cached_scalars(layers, Hkv, tokens, D)


def quantize_absmax_int(values, bits: int):
    """Returns (codes int, restored float64, scale float64)."""
    lib = _load()
    x = _c(values, np.float64)
    codes = np.zeros(x.shape, dtype=np.int32)
    restored = np.zeros(x.shape, dtype=np.float64)
    scale = np.zeros(1, dtype=np.float64)
    lib.oracle_quantize_absmax_int(_ptr(x), x.size, bits, _ptr(codes), _ptr(restored),
                                   _ptr(scale))
    return codes, restored, float(scale[0])


# --------------------------------------------------------------------------
# cache write
# --------------------------------------------------------------------------

def reshape_and_cache_bf16(k_new, v_new, k_pool, v_pool, slot_mapping, block_size: int):
    """In place on uint16 numpy pools [nblocks, bs, Hkv, D]."""
    lib = _load()
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
    T, Hkv, D = k_new.shape
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    sm = _c(slot_mapping, np.int64)
    lib.oracle_reshape_and_cache_bf16(T, Hkv, D, block_size, _ptr(kn), _ptr(vn),
                                      _ptr(k_pool), _ptr(v_pool), _ptr(sm))


def reshape_and_cache_fp8(k_new, v_new, k_pool, v_pool, k_scale, v_scale, slot_mapping,
                          block_size: int):
    """In place on uint8 pools [nblocks, bs, Hkv, D] and float32 scales [nblocks, Hkv]."""
    lib = _load()
    for a, dt in ((k_pool, np.uint8), (v_pool, np.uint8), (k_scale, np.float32),
                  (v_scale, np.float32)):
        assert a.dtype == dt and a.flags.c_contiguous
    T, Hkv, D = k_new.shape
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    sm = _c(slot_mapping, np.int64)
    lib.oracle_reshape_and_cache_fp8(T, Hkv, D, block_size, _ptr(kn), _ptr(vn), _ptr(k_pool),
                                     _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(sm))


def reshape_and_cache_int4(k_new, v_new, k_pool, v_pool, k_scale, v_scale, slot_mapping,
                           block_size: int):
    """In place on uint8 pools [nblocks, bs, Hkv, D/2] (two offset-binary nibbles per
    byte) and float32 scales [nblocks, Hkv]."""
    lib = _load()
    for a, dt in ((k_pool, np.uint8), (v_pool, np.uint8), (k_scale, np.float32),
                  (v_scale, np.float32)):
        assert a.dtype == dt and a.flags.c_contiguous
    T, Hkv, D = k_new.shape
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    sm = _c(slot_mapping, np.int64)
    lib.oracle_reshape_and_cache_int4(T, Hkv, D, block_size, _ptr(kn), _ptr(vn), _ptr(k_pool),
                                      _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(sm))


def int4_restore(row, scale: float) -> np.ndarray:
    lib = _load()
    r = _c(row, np.uint8)
    out = np.zeros(r.size * 2, dtype=np.float64)
    lib.oracle_int4_restore(_ptr(r), r.size * 2, float(scale), _ptr(out))
    return out


# --------------------------------------------------------------------------
# decode attention
# --------------------------------------------------------------------------

def _kv_kind(pool, D: int) -> int:
    """0: bf16 (uint16) pool, 1: E4M3 (uint8, D per row), 2: 4-bit (uint8, D/2 per row)."""
    if pool.dtype == np.uint16:
        return 0
    return 2 if pool.shape[-1] * 2 == D else 1


def window_positions(length: int, window: int) -> list[int]:
    lib = _load()
    out = np.zeros(max(length, 1), dtype=np.int32)
    n = lib.oracle_window_positions(int(length), int(window), _ptr(out))
    return out[:n].tolist()


def paged_decode(q, k_pool, v_pool, block_tables, seq_lens, sm_scale: float, *, Hkv: int,
                 block_size: int, k_scale=None, v_scale=None, rows=None,
                 nthreads: int | None = None, window: int = 0) -> np.ndarray:
    """Decode attention in fp64.

    q: uint16 [B, Hq, D] (bf16 bits).  Pools: uint16 (bf16) [nblocks, bs, Hkv, D], uint8
    E4M3 codes [nblocks, bs, Hkv, D] or uint8 4-bit nibble pairs [nblocks, bs, Hkv, D/2]
    (the last two need k_scale / v_scale float32 [nblocks, Hkv]).
    rows: optional int array [n, 2] of (b, h); then the result is [n, D], else [B, Hq, D].
    window: > 0 attends over the last `window` positions of each sequence only.
    """
    lib = _load()
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    kind = _kv_kind(k_pool, D)
    fp8 = kind != 0
    kp = np.ascontiguousarray(k_pool)
    vp = np.ascontiguousarray(v_pool)
    ks = _c(k_scale, np.float32) if fp8 else None
    vs = _c(v_scale, np.float32) if fp8 else None
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    nthreads = nthreads or os.cpu_count() or 1
    if rows is None:
        out = np.zeros((B, Hq, D), dtype=np.float64)
        lib.oracle_paged_decode(B, Hq, Hkv, D, block_size, bt.shape[1], kind, _ptr(q),
                                _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl),
                                float(sm_scale), int(window), 0, None, None, _ptr(out), nthreads)
        return out
    rows = np.asarray(rows, dtype=np.int32).reshape(-1, 2)
    rb = np.ascontiguousarray(rows[:, 0])
    rh = np.ascontiguousarray(rows[:, 1])
    out = np.zeros((rows.shape[0], D), dtype=np.float64)
    lib.oracle_paged_decode(B, Hq, Hkv, D, block_size, bt.shape[1], kind, _ptr(q), _ptr(kp),
                            _ptr(vp), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl), float(sm_scale),
                            int(window), rows.shape[0], _ptr(rb), _ptr(rh), _ptr(out), nthreads)
    return out


def page_summary(keys):
    """(min, max) per channel of keys [n, D]."""
    lib = _load()
    k = _c(keys, np.float64)
    n, D = k.shape
    mn, mx = np.zeros(D), np.zeros(D)
    lib.oracle_page_summary(_ptr(k), n, D, _ptr(mn), _ptr(mx))
    return mn, mx


def page_score(q, mn, mx) -> float:
    lib = _load()
    q, mn, mx = _c(q, np.float64), _c(mn, np.float64), _c(mx, np.float64)
    return lib.oracle_page_score(_ptr(q), _ptr(mn), _ptr(mx), q.size)


def select_pages(scores, k: int) -> list[int]:
    lib = _load()
    s = _c(scores, np.float64)
    out = np.zeros(max(1, s.size), dtype=np.int32)
    m = lib.oracle_select_pages(_ptr(s), s.size, int(k), _ptr(out))
    return out[:m].tolist()


def quest_decode(q, k_pool, v_pool, block_tables, seq_lens, sm_scale: float, *, Hkv: int,
                 block_size: int, topk: int, k_scale=None, v_scale=None,
                 nthreads: int | None = None):
    """Query-aware sparse decode over bf16, E4M3 or 4-bit pools (codes with per-(block,
    head) scales); returns (out [B, Hq, D], sel [B, Hkv, topk])."""
    lib = _load()
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    kind = _kv_kind(k_pool, D)
    quant = kind != 0
    kp = np.ascontiguousarray(k_pool)
    vp = np.ascontiguousarray(v_pool)
    ks = _c(k_scale, np.float32) if quant else None
    vs = _c(v_scale, np.float32) if quant else None
    bt, sl = _c(block_tables, np.int32), _c(seq_lens, np.int32)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    sel = np.zeros((B, Hkv, topk), dtype=np.int32)
    lib.oracle_quest_decode(B, Hq, Hkv, D, block_size, bt.shape[1], kind, _ptr(q), _ptr(kp),
                            _ptr(vp), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl), float(sm_scale),
                            int(topk), _ptr(out), _ptr(sel), nthreads or os.cpu_count() or 1)
    return out, sel


def bf16_round_down(x: float) -> float:
    """The largest bf16 value <= x (finite x)."""
    return _load().oracle_bf16_round_down(float(x))


def bf16_round_up(x: float) -> float:
    """The smallest bf16 value >= x (finite x)."""
    return _load().oracle_bf16_round_up(float(x))


def quest_page_summary(k_pool, page: int, rows: int, kvh: int, *, Hkv: int, D: int,
                       block_size: int, k_scale=None):
    """Quest's stored summary of pool page `page` (pool rows 16 page .. 16 page + rows - 1)
    for KV head kvh: (min rounded down, max rounded up) to bf16, from the restored keys."""
    lib = _load()
    kind = _kv_kind(k_pool, D)
    kp = np.ascontiguousarray(k_pool)
    ks = _c(k_scale, np.float32) if kind != 0 else None
    mn, mx = np.zeros(D), np.zeros(D)
    lib.oracle_quest_page_summary(Hkv, D, block_size, kind, _ptr(kp), _ptr(ks), int(page),
                                  int(rows), int(kvh), _ptr(mn), _ptr(mx))
    return mn, mx


def page_summary_bf16(keys):
    """Quest's stored summary of keys [n, D]: (min rounded down, max rounded up) to bf16."""
    mn, mx = page_summary(keys)
    return (np.array([bf16_round_down(v) for v in mn]),
            np.array([bf16_round_up(v) for v in mx]))


def split_partials(q, k_pool, v_pool, block_tables, seq_lens, sm_scale: float, b: int, h: int,
                   blk_begin, *, Hkv: int, block_size: int, k_scale=None, v_scale=None):
    """Partials (o [S, D], lse [S]) of (b, h) for splits [blk_begin[i], blk_begin[i+1])."""
    lib = _load()
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    kind = _kv_kind(k_pool, D)
    fp8 = kind != 0
    kp = np.ascontiguousarray(k_pool)
    vp = np.ascontiguousarray(v_pool)
    ks = _c(k_scale, np.float32) if fp8 else None
    vs = _c(v_scale, np.float32) if fp8 else None
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    beg = _c(blk_begin, np.int32)
    S = beg.size - 1
    o = np.zeros((S, D), dtype=np.float64)
    lse = np.zeros(S, dtype=np.float64)
    lib.oracle_split_partials(Hq, Hkv, D, block_size, bt.shape[1], kind, _ptr(q), _ptr(kp),
                              _ptr(vp), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl), float(sm_scale),
                              b, h, S, _ptr(beg), _ptr(o), _ptr(lse))
    return o, lse


def token_partials(q, k_pool, v_pool, block_tables, seq_lens, sm_scale: float, b: int, h: int,
                   tok_begin, *, Hkv: int, block_size: int, k_scale=None, v_scale=None):
    """Partials (o [S, D], lse [S]) of (b, h) for token pieces [tok_begin[i], tok_begin[i+1])."""
    lib = _load()
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    kind = _kv_kind(k_pool, D)
    fp8 = kind != 0
    kp = np.ascontiguousarray(k_pool)
    vp = np.ascontiguousarray(v_pool)
    ks = _c(k_scale, np.float32) if fp8 else None
    vs = _c(v_scale, np.float32) if fp8 else None
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    beg = _c(tok_begin, np.int32)
    S = beg.size - 1
    o = np.zeros((S, D), dtype=np.float64)
    lse = np.zeros(S, dtype=np.float64)
    lib.oracle_token_partials(Hq, Hkv, D, block_size, bt.shape[1], kind, _ptr(q), _ptr(kp),
                              _ptr(vp), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl), float(sm_scale),
                              b, h, S, _ptr(beg), _ptr(o), _ptr(lse))
    return o, lse


def paged_decode_pages(q, k_pool, v_pool, block_tables, seq_lens, sm_scale: float,
                       selected_pages, *, Hkv: int, block_size: int, k_scale=None, v_scale=None,
                       nthreads: int | None = None) -> np.ndarray:
    """Decode over chosen 16-token pages: selected_pages int32 [B, Hkv, topk] (-1 = none);
    returns out [B, Hq, D] in fp64."""
    lib = _load()
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    kind = _kv_kind(k_pool, D)
    fp8 = kind != 0
    kp = np.ascontiguousarray(k_pool)
    vp = np.ascontiguousarray(v_pool)
    ks = _c(k_scale, np.float32) if fp8 else None
    vs = _c(v_scale, np.float32) if fp8 else None
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    sel = _c(selected_pages, np.int32)
    topk = sel.shape[-1]
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lib.oracle_paged_decode_pages(B, Hq, Hkv, D, block_size, bt.shape[1], kind, _ptr(q), _ptr(kp),
                                  _ptr(vp), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl),
                                  float(sm_scale), int(topk), _ptr(sel), _ptr(out),
                                  nthreads or os.cpu_count() or 1)
    return out


def merge_lse(o_parts, lse) -> np.ndarray:
    lib = _load()
    o = _c(o_parts, np.float64)
    ls = _c(lse, np.float64)
    S, D = o.shape
    out = np.zeros(D, dtype=np.float64)
    lib.oracle_merge_lse(S, D, _ptr(o), _ptr(ls), _ptr(out))
    return out
