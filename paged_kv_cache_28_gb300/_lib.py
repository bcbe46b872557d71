"""ctypes binding of libpa.so (include/pa.h): argument marshalling only.

Every function here has the name of the C entry point it calls and passes torch
tensors through as raw device pointers; all computation happens in the CUDA
kernels.  Loading fails loudly when libpa.so is missing or no CUDA device is
present: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_DEVICE = range(5)
PA_KV_BF16, PA_KV_FP8_E4M3, PA_KV_INT4 = 0, 1, 2
PA_DEVERR_BLOCK_ID, PA_DEVERR_SEQ_LEN, PA_DEVERR_SLOT = 1, 2, 4
PA_DEVERR_FP8_CONFLICT, PA_DEVERR_TIMEOUT = 8, 16

EXPORTED = ("pa_reshape_and_cache", "pa_decode", "pa_splitkv_workspace_bytes",
            "pa_default_num_splits", "pa_decode_splitkv", "pa_merge_lse", "pa_status_string",
            "pa_read_error_flag", "pa_decode_splitkv_noalloc", "pa_quest_summarize",
            "pa_quest_select", "pa_cascade_workspace_bytes", "pa_decode_workspace_bytes",
            "pa_default_num_segments")
PA_NOALLOC_SCRATCH_BYTES = 64 << 20


class pa_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("D", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("nblocks", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32)]


class pa_decode_opts(ctypes.Structure):
    _fields_ = [("window", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("shared_prefix_lens", ctypes.c_void_p), ("selected_pages", ctypes.c_void_p),
                ("num_prefix_groups", ctypes.c_int32), ("group_offsets", ctypes.c_void_p),
                ("group_seqs", ctypes.c_void_p), ("group_prefix_len", ctypes.c_void_p),
                ("cascade_workspace", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("num_segments", ctypes.c_int32),
                ("cascade_stream", ctypes.c_void_p), ("cascade_events", ctypes.c_void_p * 2)]


def _opts(window: int = 0, shared_prefix_lens=None, selected_pages=None, cascade=None,
          workspace=None, num_segments: int = 0):
    """A pa_decode_opts by reference, or None when every setting is the default.
    selected_pages: [B, Hkv, topk] int32 tensor (topk taken from its last dim).
    cascade: (group_offsets, group_seqs, group_prefix_len, cascade_workspace) tensors,
    optionally followed by (side stream, fork event, join event) for a cascade that runs
    beside the split kernel (torch.cuda.Stream / torch.cuda.Event or raw handles).
    workspace: pa_decode's split workspace (uint8 tensor), num_segments (0: default)."""
    if (not window and shared_prefix_lens is None and selected_pages is None and cascade is None
            and workspace is None):
        return None
    topk = 0 if selected_pages is None else int(selected_pages.shape[-1])
    groups = (0, None, None, None, None)
    side = (None, (ctypes.c_void_p * 2)())
    if cascade is not None:
        offsets, seqs, plen, ws = cascade[:4]
        groups = (int(offsets.numel()) - 1, _ptr(offsets), _ptr(seqs), _ptr(plen), _ptr(ws))
        if len(cascade) > 4 and cascade[4] is not None:
            stream, fork, join = cascade[4:7]
            side = (_stream(stream), (ctypes.c_void_p * 2)(_event(fork), _event(join)))
    ws = (None, 0) if workspace is None else (_ptr(workspace),
                                              workspace.numel() * workspace.element_size())
    return ctypes.byref(pa_decode_opts(int(window), topk, _ptr(shared_prefix_lens),
                                       _ptr(selected_pages), *groups, *ws, int(num_segments),
                                       *side))


class PAError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{fn} -> {status_string(status)}{(': ' + detail) if detail else ''}")


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpa.so (no CUDA call is made by loading)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with "
                              "`python -m paged_kv_cache_28_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(path)
        P, I32, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        S = ctypes.POINTER(pa_shape)
        sig = {
            "pa_reshape_and_cache": (I32, [S, P, P, P, P, P, P, P, P, P]),
            "pa_decode": (I32, [S, P, P, P, P, P, P, P, P, P, F, P, P]),
            "pa_splitkv_workspace_bytes": (ctypes.c_size_t, [S, I32]),
            "pa_default_num_splits": (I32, [S, I32]),
            "pa_decode_workspace_bytes": (ctypes.c_size_t, [S, I32]),
            "pa_default_num_segments": (I32, [S, I32]),
            "pa_decode_splitkv": (I32, [S, P, P, I32, P, P, P, P, P, P, P, P, F, P, P]),
            "pa_merge_lse": (I32, [S, P, P, P, I32, P]),
            "pa_status_string": (ctypes.c_char_p, [I32]),
            "pa_read_error_flag": (I32, [P, ctypes.POINTER(I32), P]),
            "pa_decode_splitkv_noalloc": (I32, [S, P, I32, P, P, P, P, P, P, P, F, P, P]),
            "pa_quest_summarize": (I32, [S, P, P, P, P, P, P]),
            "pa_quest_select": (I32, [S, P, P, P, P, I32, P, P, P, P]),
            "pa_cascade_workspace_bytes": (ctypes.c_size_t, [S]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().pa_status_string(status).decode()


# ----------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------

def _ptr(t):
    """Device pointer of a CUDA tensor (None -> NULL).  Plain ints pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libpa takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libpa takes contiguous tensors only")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _event(event):
    """cudaEvent_t of a torch.cuda.Event (created on first use) or a raw handle."""
    if event is None or isinstance(event, int):
        return event
    if event.cuda_event == 0:          # torch creates the event lazily: record it once
        import torch
        event.record(torch.cuda.current_stream())
    return event.cuda_event


def make_shape(B, Hq, Hkv, D, block_size, nblocks, max_blocks, kv_dtype=PA_KV_BF16) -> pa_shape:
    return pa_shape(int(B), int(Hq), int(Hkv), int(D), int(block_size), int(nblocks),
                    int(max_blocks), int(kv_dtype))


def _check(name: str, status: int):
    if status != PA_OK:
        raise PAError(name, status)


# ----------------------------------------------------------------------------
# entry points
# ----------------------------------------------------------------------------

def pa_reshape_and_cache(shape: pa_shape, k_new, v_new, k_pool, v_pool, k_scale, v_scale,
                         slot_mapping, err_flag=None, stream=None) -> None:
    lib = load()
    _check("pa_reshape_and_cache", lib.pa_reshape_and_cache(
        ctypes.byref(shape), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
        _ptr(k_scale), _ptr(v_scale), _ptr(slot_mapping), _ptr(err_flag), _stream(stream)))


def pa_decode(shape: pa_shape, out, q, k_pool, v_pool, k_scale, v_scale, block_tables,
              seq_lens, sm_scale: float, err_flag=None, stream=None, window: int = 0,
              selected_pages=None, workspace=None, num_segments: int = 0,
              shared_prefix_lens=None, cascade=None) -> None:
    """workspace (uint8 device tensor): run the split decode and the merge in this call
    (cascade, see _opts, needs one)."""
    lib = load()
    _check("pa_decode", lib.pa_decode(
        ctypes.byref(shape), _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_tables), _ptr(seq_lens),
        _opts(window, shared_prefix_lens, selected_pages, cascade, workspace, num_segments),
        float(sm_scale), _ptr(err_flag), _stream(stream)))


def pa_decode_workspace_bytes(shape: pa_shape, num_segments: int) -> int:
    return int(load().pa_decode_workspace_bytes(ctypes.byref(shape), int(num_segments)))


def pa_default_num_segments(shape: pa_shape, sm_count: int) -> int:
    return int(load().pa_default_num_segments(ctypes.byref(shape), int(sm_count)))


def pa_splitkv_workspace_bytes(shape: pa_shape, num_splits: int) -> int:
    return int(load().pa_splitkv_workspace_bytes(ctypes.byref(shape), int(num_splits)))


def pa_cascade_workspace_bytes(shape: pa_shape) -> int:
    return int(load().pa_cascade_workspace_bytes(ctypes.byref(shape)))


def pa_default_num_splits(shape: pa_shape, sm_count: int) -> int:
    return int(load().pa_default_num_splits(ctypes.byref(shape), int(sm_count)))


def pa_decode_splitkv(shape: pa_shape, o_part, lse, num_splits: int, q, k_pool, v_pool,
                      k_scale, v_scale, block_tables, seq_lens, sm_scale: float, err_flag=None,
                      stream=None, window: int = 0, selected_pages=None,
                      shared_prefix_lens=None) -> None:
    """Partials o_part [B, Hq, S, D] and lse [B, Hq, S] (fp32 device tensors), S = num_splits."""
    lib = load()
    _check("pa_decode_splitkv", lib.pa_decode_splitkv(
        ctypes.byref(shape), _ptr(o_part), _ptr(lse), int(num_splits), _ptr(q), _ptr(k_pool),
        _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(seq_lens),
        _opts(window, shared_prefix_lens, selected_pages), float(sm_scale), _ptr(err_flag),
        _stream(stream)))


def pa_merge_lse(shape: pa_shape, out, o_part, lse, num_splits: int, stream=None) -> None:
    lib = load()
    _check("pa_merge_lse", lib.pa_merge_lse(ctypes.byref(shape), _ptr(out), _ptr(o_part),
                                            _ptr(lse), int(num_splits), _stream(stream)))


def pa_read_error_flag(err_flag, stream=None) -> int:
    """Synchronise the stream and return the device error bits (0 = none)."""
    lib = load()
    v = ctypes.c_int32(0)
    st = lib.pa_read_error_flag(_ptr(err_flag), ctypes.byref(v), _stream(stream))
    if st not in (PA_OK, PA_ERR_DEVICE):
        raise PAError("pa_read_error_flag", st)
    return int(v.value)


def pa_decode_splitkv_noalloc(shape: pa_shape, out, num_segments: int, q, k_pool, v_pool,
                              k_scale, v_scale, block_tables, seq_lens, sm_scale: float,
                              err_flag=None, stream=None) -> None:
    """Split-KV decode + merge with the library's own fixed scratch array, for
    callers that may not allocate device memory (see include/pa.h)."""
    lib = load()
    _check("pa_decode_splitkv_noalloc", lib.pa_decode_splitkv_noalloc(
        ctypes.byref(shape), _ptr(out), int(num_segments), _ptr(q), _ptr(k_pool), _ptr(v_pool),
        _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), _ptr(seq_lens), float(sm_scale),
        _ptr(err_flag), _stream(stream)))


def pa_quest_summarize(shape: pa_shape, k_pool, k_scale, key_summaries, slot_mapping,
                       err_flag=None, stream=None) -> None:
    lib = load()
    _check("pa_quest_summarize", lib.pa_quest_summarize(
        ctypes.byref(shape), _ptr(k_pool), _ptr(k_scale), _ptr(key_summaries),
        _ptr(slot_mapping), _ptr(err_flag), _stream(stream)))


def pa_quest_select(shape: pa_shape, q, key_summaries, block_tables, seq_lens, topk: int,
                    page_scores, selected_pages, err_flag=None, stream=None) -> None:
    lib = load()
    _check("pa_quest_select", lib.pa_quest_select(
        ctypes.byref(shape), _ptr(q), _ptr(key_summaries), _ptr(block_tables), _ptr(seq_lens),
        int(topk), _ptr(page_scores), _ptr(selected_pages), _ptr(err_flag), _stream(stream)))
