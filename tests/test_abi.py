"""The C ABI without a GPU: libpa.so loads, exports every entry point that
include/pa.h declares, and rejects bad arguments on the host before any CUDA
call."""
import os
import re

import pytest

from paged_kv_cache_28_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_28_gb300 import build
    build.build()
    return _lib.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    declared = header_functions()
    assert declared == sorted(_lib.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(5):
        assert _lib.status_string(s).startswith("PA_")


def shape(**kw):
    base = dict(B=4, Hq=8, Hkv=2, D=64, block_size=16, nblocks=64, max_blocks=8,
                kv_dtype=_lib.PA_KV_BF16)
    base.update(kw)
    return _lib.make_shape(**base)


FAKE = 1 << 20      # a 16-byte aligned non-null address: never dereferenced on these paths


def _decode(lib, s, **ptr):
    p = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, ks=None, vs=None, bt=FAKE, sl=FAKE)
    p.update(ptr)
    return lib.pa_decode(s, p["out"], p["q"], p["k"], p["v"], p["ks"], p["vs"], p["bt"], p["sl"],
                         p.get("opts"), 0.125, None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), _lib.PA_ERR_INVALID_ARG),        # Hq % Hkv != 0
    (dict(Hq=64, Hkv=2), _lib.PA_ERR_UNSUPPORTED),        # G = 32 > 16
    (dict(D=96), _lib.PA_ERR_UNSUPPORTED),
    (dict(block_size=8), _lib.PA_ERR_UNSUPPORTED),
    (dict(kv_dtype=_lib.PA_KV_FP8_E4M3), _lib.PA_ERR_UNSUPPORTED),   # FP8 needs D = 128
    (dict(kv_dtype=_lib.PA_KV_INT4), _lib.PA_ERR_UNSUPPORTED),       # so does 4-bit
    (dict(kv_dtype=7), _lib.PA_ERR_INVALID_ARG),
    (dict(nblocks=0), _lib.PA_ERR_INVALID_ARG),
    (dict(B=-1), _lib.PA_ERR_INVALID_ARG),
    (dict(nblocks=1 << 27, block_size=32), _lib.PA_ERR_INVALID_ARG),   # rows overflow int32
    (dict(Hq=4096, Hkv=4096, nblocks=4), _lib.PA_ERR_UNSUPPORTED),     # KV heads > 2048
])
def test_decode_rejects_bad_shapes(lib, kw, status):
    import ctypes
    assert _decode(lib, ctypes.byref(shape(**kw))) == status


def test_decode_rejects_scale_indices_past_int32(lib):
    # FP8 pool of 2^20 blocks x 2048 KV heads: every other bound holds, but the
    # [nblocks, Hkv] scale arrays have 2^31 entries
    import ctypes
    s = shape(kv_dtype=_lib.PA_KV_FP8_E4M3, D=128, Hq=2048, Hkv=2048, nblocks=1 << 20)
    assert _decode(lib, ctypes.byref(s), ks=FAKE, vs=FAKE) == _lib.PA_ERR_INVALID_ARG


def test_decode_rejects_bad_pointers(lib):
    import ctypes
    s = ctypes.byref(shape())
    assert _decode(lib, s, q=None) == _lib.PA_ERR_INVALID_ARG
    assert _decode(lib, s, k=FAKE + 4) == _lib.PA_ERR_INVALID_ARG     # misaligned
    fp8 = ctypes.byref(shape(D=128, kv_dtype=_lib.PA_KV_FP8_E4M3))
    assert _decode(lib, fp8) == _lib.PA_ERR_INVALID_ARG                # scales missing
    assert lib.pa_decode(None, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, None, 0.1, None,
                         None) == _lib.PA_ERR_INVALID_ARG
    bad = _lib.pa_decode_opts(-1, 0, None, None)
    assert _decode(lib, s, opts=ctypes.byref(bad)) == _lib.PA_ERR_INVALID_ARG   # window < 0
    bad = _lib.pa_decode_opts(0, 4, None, None)
    assert _decode(lib, s, opts=ctypes.byref(bad)) == _lib.PA_ERR_INVALID_ARG   # topk, no pages
    bad = _lib.pa_decode_opts(0, 0, None, FAKE)
    assert _decode(lib, s, opts=ctypes.byref(bad)) == _lib.PA_ERR_INVALID_ARG   # pages, topk 0
    bad = _lib.pa_decode_opts(16, 4, None, FAKE)
    assert _decode(lib, s, opts=ctypes.byref(bad)) == _lib.PA_ERR_INVALID_ARG   # window + topk


def test_empty_batch_is_a_no_op(lib):
    import ctypes
    assert _decode(lib, ctypes.byref(shape(B=0)), q=None) == _lib.PA_OK


def test_decode_workspace_bytes(lib):
    s = shape(B=64, Hq=64, Hkv=8, D=128, max_blocks=2048, nblocks=30000)
    nbytes = _lib.pa_decode_workspace_bytes(s, 1216)
    G = 8
    expect_min = (68 * 4) + 1216 * 2 * G * 4 + 1216 * 2 * G * 128 * 4
    assert expect_min <= nbytes <= expect_min + 3 * 256
    assert _lib.pa_decode_workspace_bytes(s, 0) == 0
    assert _lib.pa_decode_workspace_bytes(s, 70000) == 0
    # 4-bit pools read two KV heads at a time: partials of 16 query heads per piece
    s4 = shape(B=64, Hq=64, Hkv=8, D=128, max_blocks=2048, nblocks=30000,
               kv_dtype=_lib.PA_KV_INT4)
    n4 = _lib.pa_decode_workspace_bytes(s4, 1216)
    expect4 = (68 * 4) + 1216 * 2 * 16 * 4 + 1216 * 2 * 16 * 128 * 4
    assert expect4 <= n4 <= expect4 + 3 * 256


def test_splitkv_partials_host_checks(lib):
    import ctypes
    s = shape(B=64, Hq=64, Hkv=8, D=128, max_blocks=2048, nblocks=30000)
    assert _lib.pa_splitkv_workspace_bytes(s, 16) == 64 * 64 * 16 * 129 * 4   # o_part + lse
    assert _lib.pa_splitkv_workspace_bytes(s, 0) == 0
    assert _lib.pa_splitkv_workspace_bytes(s, 70000) == 0

    def call(sh, o=FAKE, lse=FAKE, S=16, opts=None):
        return lib.pa_decode_splitkv(ctypes.byref(sh), o, lse, S, FAKE, FAKE, FAKE, None, None,
                                     FAKE, FAKE, opts, 0.1, None, None)

    assert call(s, lse=None) == _lib.PA_ERR_INVALID_ARG          # no lse array
    assert call(s, lse=FAKE + 4) == _lib.PA_ERR_INVALID_ARG      # misaligned
    assert call(s, o=None) == _lib.PA_ERR_INVALID_ARG
    assert call(s, S=0) == _lib.PA_ERR_INVALID_ARG
    assert call(s, S=70000) == _lib.PA_ERR_INVALID_ARG
    assert call(shape(B=0), o=None, lse=None) == _lib.PA_OK      # nothing to do
    assert call(_lib.make_shape(16385, 8, 8, 128, 16, 30000, 4)) == _lib.PA_ERR_UNSUPPORTED
    cascade = _lib.pa_decode_opts(0, 0, None, None, 1, FAKE, FAKE, FAKE, FAKE)
    assert call(s, opts=ctypes.byref(cascade)) == _lib.PA_ERR_UNSUPPORTED   # no cascade here
    window = _lib.pa_decode_opts(-1, 0, None, None)
    assert call(s, opts=ctypes.byref(window)) == _lib.PA_ERR_INVALID_ARG

    def merge(sh, out=FAKE, o=FAKE, lse=FAKE, S=16):
        return lib.pa_merge_lse(ctypes.byref(sh), out, o, lse, S, None)

    assert merge(s, S=0) == _lib.PA_ERR_INVALID_ARG
    assert merge(s, o=None) == _lib.PA_ERR_INVALID_ARG
    assert merge(s, lse=FAKE + 8) == _lib.PA_ERR_INVALID_ARG
    assert merge(shape(Hq=6, Hkv=4)) == _lib.PA_ERR_INVALID_ARG
    assert merge(shape(B=0), out=None, o=None, lse=None) == _lib.PA_OK


def test_default_num_segments_is_resident_warps(lib):
    s = shape(B=64, Hq=64, Hkv=8, D=128, max_blocks=2048, nblocks=30000)
    n = _lib.pa_default_num_segments(s, 152)
    assert n % 152 == 0 and 152 * 4 <= n <= 152 * 16
    assert _lib.pa_default_num_segments(s, 0) == 1


def test_default_num_splits_fills_64_mib_of_partials(lib):
    # one slot of o_part is B * Hq * D * 4 bytes: the most slots in 64 MiB, 2..64, and at
    # most the 16-token tiles of a full block table
    def ns(**kw):
        return _lib.pa_default_num_splits(shape(**kw), 152)
    assert ns(B=64, Hq=64, Hkv=8, D=128, max_blocks=2048, nblocks=30000) == 32     # 2 MiB/slot
    assert ns(B=8, Hq=64, Hkv=8, D=128, max_blocks=4096, nblocks=30000, block_size=32) == 64
    assert ns(B=512, Hq=64, Hkv=8, D=128, max_blocks=256, nblocks=30000) == 4      # 16 MiB/slot
    assert ns(B=4096, Hq=64, Hkv=8, D=128, max_blocks=256, nblocks=30000) == 2
    assert ns(B=4, max_blocks=1) == 1                                              # one tile
    assert _lib.pa_default_num_splits(shape(), 0) == 1


def test_reshape_rejects_bad_args(lib):
    import ctypes
    s = ctypes.byref(shape(B=4))
    assert lib.pa_reshape_and_cache(s, FAKE, None, FAKE, FAKE, None, None, FAKE, None,
                                    None) == _lib.PA_ERR_INVALID_ARG
    fp8 = ctypes.byref(shape(D=128, kv_dtype=_lib.PA_KV_FP8_E4M3))
    assert lib.pa_reshape_and_cache(fp8, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None,
                                    None) == _lib.PA_ERR_INVALID_ARG


def test_decode_workspace_host_checks(lib):
    import ctypes
    s = shape(B=8, Hq=64, Hkv=8, D=128, max_blocks=64, nblocks=512)
    need = _lib.pa_decode_workspace_bytes(s, 16)

    def call(ws, nbytes, ns):
        o = _lib.pa_decode_opts(0, 0, None, None, 0, None, None, None, None, ws, nbytes, ns)
        return lib.pa_decode(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE,
                             ctypes.byref(o), 0.1, None, None)

    assert call(FAKE, need - 1, 16) == _lib.PA_ERR_INVALID_ARG         # too small
    assert call(FAKE + 16, need, 16) == _lib.PA_ERR_INVALID_ARG        # not 256-aligned
    assert call(FAKE, need, 70000) == _lib.PA_ERR_INVALID_ARG          # too many segments
    big = _lib.make_shape(16385, 8, 8, 128, 16, 30000, 4)
    o = _lib.pa_decode_opts(0, 0, None, None, 0, None, None, None, None, FAKE,
                            _lib.pa_decode_workspace_bytes(big, 16), 16)
    assert lib.pa_decode(ctypes.byref(big), FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE,
                         ctypes.byref(o), 0.1, None, None) == _lib.PA_ERR_UNSUPPORTED   # B > 16384


def test_cascade_host_checks(lib):
    import ctypes
    s = shape(B=8, Hq=64, Hkv=8, D=128, max_blocks=64, nblocks=512)
    ws = _lib.pa_decode_workspace_bytes(s, 16)
    cb = _lib.pa_cascade_workspace_bytes(s)
    assert cb >= 8 * 64 * 4 * 129 * 4 and _lib.pa_cascade_workspace_bytes(shape(Hq=7)) == 0

    def call(sh, opts):
        return lib.pa_decode(ctypes.byref(sh), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                             ctypes.byref(opts), 0.1, None, None)

    def opts(n=1, offs=FAKE, seqs=FAKE, plen=FAKE, cws=FAKE, window=0, stream=None, events=(None, None)):
        return _lib.pa_decode_opts(window, 0, None, None, n, offs, seqs, plen, cws, FAKE, ws, 16,
                                   stream, (ctypes.c_void_p * 2)(*events))

    assert call(s, opts(n=-1)) == _lib.PA_ERR_INVALID_ARG
    assert call(s, opts(seqs=None)) == _lib.PA_ERR_INVALID_ARG          # no member list
    assert call(s, opts(cws=None)) == _lib.PA_ERR_INVALID_ARG           # no workspace
    assert call(s, opts(cws=FAKE + 16)) == _lib.PA_ERR_INVALID_ARG      # not 256-aligned
    assert call(s, opts(offs=FAKE + 2)) == _lib.PA_ERR_INVALID_ARG      # misaligned int32
    assert call(s, opts(window=64)) == _lib.PA_ERR_INVALID_ARG          # not with a window
    assert call(s, opts(stream=FAKE)) == _lib.PA_ERR_INVALID_ARG        # side stream, no events
    assert call(s, opts(stream=FAKE, events=(FAKE, None))) == _lib.PA_ERR_INVALID_ARG


def test_quest_host_checks(lib):
    import ctypes
    s = ctypes.byref(shape())
    fp8 = ctypes.byref(shape(D=128, kv_dtype=_lib.PA_KV_FP8_E4M3))
    assert lib.pa_quest_summarize(fp8, FAKE, None, FAKE, FAKE, None, None) == \
        _lib.PA_ERR_INVALID_ARG                                          # no k_scale
    assert lib.pa_quest_summarize(s, FAKE, None, None, FAKE, None, None) == \
        _lib.PA_ERR_INVALID_ARG                                          # no summaries
    assert lib.pa_quest_select(s, FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, None, None) == \
        _lib.PA_ERR_INVALID_ARG                                          # topk < 1
    assert lib.pa_quest_select(s, FAKE, FAKE, FAKE, FAKE, 4, None, FAKE, None, None) == \
        _lib.PA_ERR_INVALID_ARG                                          # no page_scores
