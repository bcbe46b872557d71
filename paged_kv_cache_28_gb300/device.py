"""Device-side buffers for a decode batch and the calls that run on them.

DeviceBatch uploads a workload.Batch (numpy) to the GPU as torch tensors in the
layouts of include/pa.h and calls the C ABI through the binding.  It only moves
data and passes pointers; every step of the hot path runs in libpa.so.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib
from .workload import Batch, cascade_groups


def to_device_bf16(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(
        torch.bfloat16)


class DeviceBatch:
    def __init__(self, batch: Batch, device="cuda", pools=None):
        """pools: optional (k_pool, v_pool, k_scale, v_scale) device tensors to use
        instead of uploading batch.k_pool / batch.v_pool (for large generated pools)."""
        self.batch = batch
        self.device = torch.device(device)
        fp8 = batch.quantized            # code pools (E4M3 or 4-bit) with scales
        self.fp8 = fp8
        kind = {"bf16": _lib.PA_KV_BF16, "fp8_e4m3": _lib.PA_KV_FP8_E4M3,
                "int4": _lib.PA_KV_INT4}[batch.kv_dtype]
        self.shape = _lib.make_shape(batch.B, batch.Hq, batch.Hkv, batch.D, batch.block_size,
                                     batch.nblocks, batch.max_blocks, kind)
        self.q = to_device_bf16(batch.q, self.device)
        self.k_new = to_device_bf16(batch.k_new, self.device)
        self.v_new = to_device_bf16(batch.v_new, self.device)
        self.block_tables = torch.from_numpy(batch.block_tables).to(self.device)
        self.seq_lens = torch.from_numpy(batch.seq_lens).to(self.device)
        self.slot_mapping = torch.from_numpy(batch.slot_mapping).to(self.device)
        self.shared_prefix_lens = (None if batch.shared_prefix_lens is None else
                                   torch.from_numpy(batch.shared_prefix_lens).to(self.device))
        if pools is not None:
            self.k_pool, self.v_pool, self.k_scale, self.v_scale = pools
        elif fp8:
            self.k_pool = torch.from_numpy(batch.k_pool).to(self.device)
            self.v_pool = torch.from_numpy(batch.v_pool).to(self.device)
            self.k_scale = torch.from_numpy(batch.k_scale).to(self.device)
            self.v_scale = torch.from_numpy(batch.v_scale).to(self.device)
        else:
            self.k_pool = to_device_bf16(batch.k_pool, self.device)
            self.v_pool = to_device_bf16(batch.v_pool, self.device)
            self.k_scale = self.v_scale = None
        self.out = torch.zeros((batch.B, batch.Hq, batch.D), dtype=torch.float32,
                               device=self.device)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.workspace = None
        self.num_segments = None
        self.cascade = None
        self.o_part = self.lse = None

    # -- calls -----------------------------------------------------------------

    def reshape_and_cache(self, stream=None):
        _lib.pa_reshape_and_cache(self.shape, self.k_new, self.v_new, self.k_pool, self.v_pool,
                                  self.k_scale, self.v_scale, self.slot_mapping, self.err,
                                  stream)

    def decode(self, stream=None, window: int = 0, selected_pages=None,
               workspace: bool = False, hints: bool = False, num_segments: int | None = None,
               cascade: bool = False):
        """pa_decode; workspace: hand it a split workspace (num_segments, default: the
        resident split workers), so that it runs the split decode and the merge itself;
        hints: pass the batch's shared-prefix lengths (if any); cascade: attend over the
        prefix groups (enable_cascade) once per group (needs the workspace)."""
        ws = None
        if workspace or cascade:
            ns = default_num_segments(self.shape, self.device) if num_segments is None else num_segments
            if self.workspace is None or self.num_segments != ns:
                self.ensure_workspace(ns)
            ws = self.workspace
        if cascade and self.cascade is None:
            self.enable_cascade()
        _lib.pa_decode(self.shape, self.out, self.q, self.k_pool, self.v_pool, self.k_scale,
                       self.v_scale, self.block_tables, self.seq_lens, self.batch.sm_scale,
                       self.err, stream, window, selected_pages, ws,
                       self.num_segments if ws is not None else 0,
                       shared_prefix_lens=self.shared_prefix_lens if hints else None,
                       cascade=self.cascade if cascade else None)

    def ensure_workspace(self, num_segments: int):
        nbytes = _lib.pa_decode_workspace_bytes(self.shape, num_segments)
        if nbytes == 0:
            raise ValueError("invalid shape or num_segments for the split decode")
        if self.workspace is None or self.workspace.numel() < nbytes:
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self.num_segments = num_segments

    def enable_cascade(self, groups=None, side_stream: bool = True):
        """Prefix-aware decode: groups = (group_offsets, group_seqs, group_prefix_len) int32
        arrays, by default the batch's own prefix groups; side_stream: run the cascade
        kernel beside the split kernel on a stream of its own (else after it)."""
        offsets, seqs, plen = cascade_groups(self.batch) if groups is None else groups
        ws = torch.empty(_lib.pa_cascade_workspace_bytes(self.shape), dtype=torch.uint8,
                         device=self.device)
        self.cascade = tuple(torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(
            self.device) for a in (offsets, seqs, plen)) + (ws,)
        if side_stream:
            events = []
            for _ in range(2):           # created now (recorded once), reused by every call
                e = torch.cuda.Event()
                e.record(torch.cuda.current_stream(self.device))
                events.append(e)
            self.cascade = self.cascade + (torch.cuda.Stream(self.device), *events)

    def decode_segments(self, num_segments: int | None = None, stream=None, hints: bool = True,
                        window: int = 0, selected_pages=None, cascade: bool = False):
        """pa_decode with a workspace of num_segments (the load-balanced split decode and
        its merge); hints: pass the batch's shared-prefix lengths (if any); cascade: attend
        over the prefix groups (enable_cascade) once per group."""
        self.decode(stream, window, selected_pages, workspace=True, hints=hints,
                    num_segments=num_segments, cascade=cascade)

    def ensure_parts(self, num_splits: int):
        """Caller-visible partials o_part [B, Hq, S, D] and lse [B, Hq, S]."""
        b = self.batch
        if getattr(self, "o_part", None) is None or self.o_part.shape[2] != num_splits:
            self.o_part = torch.empty((b.B, b.Hq, num_splits, b.D), dtype=torch.float32,
                                      device=self.device)
            self.lse = torch.empty((b.B, b.Hq, num_splits), dtype=torch.float32,
                                   device=self.device)

    def decode_splitkv(self, num_splits: int | None = None, stream=None, merge: bool = True,
                       window: int = 0, selected_pages=None, hints: bool = False):
        """pa_decode_splitkv into o_part / lse (num_splits slots per query head, default
        pa_default_num_splits), then pa_merge_lse into out; hints: pass the batch's
        shared-prefix lengths (if any)."""
        if num_splits is None:
            num_splits = default_num_splits(self.shape, self.device)
        self.ensure_parts(num_splits)
        _lib.pa_decode_splitkv(self.shape, self.o_part, self.lse, num_splits, self.q,
                               self.k_pool, self.v_pool, self.k_scale, self.v_scale,
                               self.block_tables, self.seq_lens, self.batch.sm_scale, self.err,
                               stream, window, selected_pages,
                               self.shared_prefix_lens if hints else None)
        if merge:
            _lib.pa_merge_lse(self.shape, self.out, self.o_part, self.lse, num_splits, stream)

    # -- Quest page selection ------------------------------------------------------

    def quest_summary_slots(self) -> torch.Tensor:
        """Slots of every page's last valid token: summarising them builds all pages."""
        b = self.batch
        slots = []
        for s in range(b.B):
            L = int(b.seq_lens[s])
            for j in range((L + 15) // 16):
                t = min(L, 16 * (j + 1)) - 1
                slots.append(int(b.block_tables[s, t // b.block_size]) * b.block_size +
                             t % b.block_size)
        return torch.tensor(slots if slots else [-1], dtype=torch.int64, device=self.device)

    def quest_build_summaries(self, stream=None):
        b = self.batch
        npages = b.nblocks * b.block_size // 16
        self.key_summaries = torch.zeros((npages, b.Hkv, 2, b.D), dtype=torch.bfloat16,
                                         device=self.device)
        slots = self.quest_summary_slots()
        shape = _lib.make_shape(slots.numel(), b.Hq, b.Hkv, b.D, b.block_size, b.nblocks,
                                b.max_blocks, self.shape.kv_dtype)
        _lib.pa_quest_summarize(shape, self.k_pool, self.k_scale, self.key_summaries, slots,
                                self.err, stream)

    def quest_buffers(self, topk: int):
        """page_scores [B, Hkv, pages per block-table row] and selected_pages [B, Hkv, topk]."""
        b = self.batch
        max_pages = (b.max_blocks * b.block_size + 15) // 16
        self.page_scores = torch.zeros((b.B, b.Hkv, max_pages), dtype=torch.float32,
                                       device=self.device)
        self.selected_pages = torch.empty((b.B, b.Hkv, topk), dtype=torch.int32,
                                          device=self.device)

    def quest_select(self, topk: int, stream=None) -> torch.Tensor:
        if getattr(self, "selected_pages", None) is None or self.selected_pages.shape[2] != topk:
            self.quest_buffers(topk)
        _lib.pa_quest_select(self.shape, self.q, self.key_summaries, self.block_tables,
                             self.seq_lens, topk, self.page_scores, self.selected_pages,
                             self.err, stream)
        return self.selected_pages

    def read_err(self, stream=None) -> int:
        return _lib.pa_read_error_flag(self.err, stream)

    # -- host copies for checking ------------------------------------------------

    def pools_numpy(self):
        if self.fp8:
            return (self.k_pool.cpu().numpy(), self.v_pool.cpu().numpy(),
                    self.k_scale.cpu().numpy(), self.v_scale.cpu().numpy())
        return (self.k_pool.view(torch.int16).cpu().numpy().view(np.uint16),
                self.v_pool.view(torch.int16).cpu().numpy().view(np.uint16), None, None)


def _sm_count(device=None) -> int:
    return torch.cuda.get_device_properties(device or 0).multi_processor_count


def default_num_segments(shape, device=None) -> int:
    """Segments of pa_decode's split decode: the resident split workers."""
    return _lib.pa_default_num_segments(shape, _sm_count(device))


def default_num_splits(shape, device=None) -> int:
    """Partial slots per query head of pa_decode_splitkv."""
    return _lib.pa_default_num_splits(shape, _sm_count(device))
