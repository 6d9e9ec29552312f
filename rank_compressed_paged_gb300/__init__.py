"""Rank-compressed paged attention on GB300 (sm_103a).

A thin Python layer over the C ABI of ``librcp.so`` (``include/rcp.h``): it passes torch
device pointers and the current CUDA stream through ctypes and does nothing else; every
step of the path runs in the library's CUDA kernels.

    cache = PagedCoeffCache(num_heads=32, head_dim=128, rank_k=64, rank_v=1024,
                            num_blocks=..., U_k=U, W_v=W)       # U, W: fp16 CUDA tensors
    cache.append_kv(k, v, slot_mapping)                          # project + scatter
    out = cache.decode_attn(q, block_table, seq_lens)            # [B][H][d] fp16
    out = cache.prefill_attn(q, cu_chunk_lens, block_table, seq_lens)
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import RcpError  # noqa: F401

BLOCK_SIZE = 16
RECONSTRUCT_MIN_CHUNK = 16   # mean chunk rows from which prefill_attn(variant="auto") rebuilds V


def _ptr(t) -> int:
    return t.data_ptr()


def _stream(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


class PagedCoeffCache:
    """Paged low-rank coefficient cache on one GPU.

    Owns (as torch tensors) the K pages [num_blocks][H][16][r_k], V pages
    [num_blocks][16][R], the factors, a device error word and a reusable workspace; the
    library handle borrows their pointers.  page_format "fp16" stores fp16 coefficients,
    "fp8_e4m3" stores E4M3 codes (uint8 tensors; prefill on them takes the reconstructing
    variant, which first widens the pages it reads to fp16 in the workspace).
    """

    def __init__(self, num_heads: int, head_dim: int, rank_k: int, rank_v: int,
                 num_blocks: int, U_k, W_v, k_pages=None, v_pages=None, device=None,
                 page_format: str = "fp16"):
        import torch
        lib = _lib.load()
        dev = U_k.device if device is None else torch.device(device)
        fmt = {"fp16": _lib.RCP_PAGES_FP16, "fp8_e4m3": _lib.RCP_PAGES_FP8_E4M3}[page_format]
        page_dtype = torch.float16 if fmt == _lib.RCP_PAGES_FP16 else torch.uint8
        self.page_format = page_format
        self.shape = dict(num_heads=num_heads, head_dim=head_dim, rank_k=rank_k, rank_v=rank_v)
        self.num_blocks = int(num_blocks)
        self.U_k = U_k.contiguous()
        self.W_v = W_v.contiguous()
        if k_pages is None:
            k_pages = torch.zeros((num_blocks, num_heads, BLOCK_SIZE, rank_k),
                                  dtype=page_dtype, device=dev)
        if v_pages is None:
            v_pages = torch.zeros((num_blocks, BLOCK_SIZE, rank_v), dtype=page_dtype,
                                  device=dev)
        for pg in (k_pages, v_pages):
            if pg.element_size() != (2 if fmt == _lib.RCP_PAGES_FP16 else 1):
                raise ValueError(f"{page_format} pages need {page_dtype} elements, got {pg.dtype}")
        self.k_pages = k_pages
        self.v_pages = v_pages
        self.dev_error = torch.zeros(1, dtype=torch.int32, device=dev)
        self._ws = None
        self._cfg = _lib.CacheConfig(num_heads, head_dim, rank_k, rank_v, BLOCK_SIZE,
                                     self.num_blocks, fmt)
        h = ctypes.c_void_p()
        _lib.check("rcp_create_cache", lib.rcp_create_cache(
            ctypes.byref(self._cfg), _ptr(self.k_pages), _ptr(self.v_pages), _ptr(self.U_k),
            _ptr(self.W_v), _ptr(self.dev_error), ctypes.byref(h)))
        self._h = h
        self._lib = lib

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._lib.rcp_destroy_cache(h)
            self._h = None

    # ------------------------------------------------------------------ block pool
    def alloc_blocks(self, n: int):
        ids = (ctypes.c_int32 * max(n, 1))()
        _lib.check("rcp_alloc_blocks", self._lib.rcp_alloc_blocks(self._h, n, ids))
        return [ids[i] for i in range(n)]

    def free_blocks(self, ids) -> None:
        arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _lib.check("rcp_free_blocks", self._lib.rcp_free_blocks(self._h, len(ids), arr))

    def num_free_blocks(self) -> int:
        n = ctypes.c_int64()
        _lib.check("rcp_num_free_blocks", self._lib.rcp_num_free_blocks(self._h, ctypes.byref(n)))
        return n.value

    # ------------------------------------------------------------------ workspace
    def workspace_bytes(self, rows: int) -> int:
        n = ctypes.c_size_t()
        _lib.check("rcp_workspace_size",
                   self._lib.rcp_workspace_size(self._h, rows, ctypes.byref(n)))
        return n.value

    def workspace(self, rows: int, need: int | None = None):
        import torch
        need = self.workspace_bytes(rows) if need is None else need
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.k_pages.device)
        return self._ws

    def reconstruct_workspace_bytes(self, rows: int, batch: int, max_blocks_per_seq: int) -> int:
        n = ctypes.c_size_t()
        _lib.check("rcp_prefill_reconstruct_workspace_size",
                   self._lib.rcp_prefill_reconstruct_workspace_size(
                       self._h, rows, batch, max_blocks_per_seq, ctypes.byref(n)))
        return n.value

    def prefill_crossover_rows(self) -> int:
        n = ctypes.c_int32()
        _lib.check("rcp_prefill_crossover_rows",
                   self._lib.rcp_prefill_crossover_rows(self._h, ctypes.byref(n)))
        return n.value

    def read_device_error(self) -> int:
        return int(self.dev_error.item())

    def clear_device_error(self) -> None:
        self.dev_error.zero_()

    def set_profile_events(self, start=None, stop=None) -> None:
        """Record torch.cuda.Event pair around the split-K attention kernel (None: off)."""
        def handle(ev):
            if ev is None:
                return None
            if not ev.cuda_event:
                ev.record()            # torch creates the CUDA event lazily
            return ev.cuda_event
        _lib.check("rcp_set_profile_events",
                   self._lib.rcp_set_profile_events(self._h, handle(start), handle(stop)))

    # ------------------------------------------------------------------ hot path
    def append_kv(self, k, v, slot_mapping, stream=None) -> None:
        """k, v: [T][H][d] fp16; slot_mapping: [T] int64 (all on the cache's device)."""
        T = int(slot_mapping.shape[0])
        _lib.check("rcp_append_kv", self._lib.rcp_append_kv(
            self._h, _ptr(k), _ptr(v), _ptr(slot_mapping), T, _stream(stream)))

    def decode_attn(self, q, block_table, seq_lens, out=None, workspace=None, stream=None):
        """q: [B][H][d] fp16; block_table: [B][max_blocks] int32; seq_lens: [B] int32."""
        import torch
        B = int(q.shape[0])
        if out is None:
            out = torch.empty_like(q)
        ws = self.workspace(B) if workspace is None else workspace
        _lib.check("rcp_decode_attn", self._lib.rcp_decode_attn(
            self._h, _ptr(q), _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens), B,
            _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))
        return out

    def decode_attn_sparse(self, q, block_table, seq_lens, skip_threshold: float,
                           page_kept=None, out=None, workspace=None, stream=None):
        """Block-sparse decode: as decode_attn, but a page is left out (its values unread,
        its tokens out of the softmax) when every head's largest weight in it is below
        ``skip_threshold`` times that head's running maximum weight.  ``page_kept``: None
        or a [B][max_blocks] uint8 tensor that receives 1 / 0 per page read / left out."""
        import torch
        B = int(q.shape[0])
        if out is None:
            out = torch.empty_like(q)
        if page_kept is not None and (page_kept.dtype != torch.uint8 or
                                      tuple(page_kept.shape) != tuple(block_table.shape)):
            raise ValueError("page_kept must be uint8 shaped like block_table")
        ws = self.workspace(B) if workspace is None else workspace
        _lib.check("rcp_decode_attn_sparse", self._lib.rcp_decode_attn_sparse(
            self._h, _ptr(q), _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens), B,
            float(skip_threshold), _ptr(page_kept) if page_kept is not None else None,
            _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))
        return out

    def decode_step(self, k, v, slot_mapping, q, block_table, seq_lens, out=None, workspace=None,
                    stream=None):
        """append_kv(k, v, slot_mapping) then decode_attn(q, ...), queued as one step."""
        import torch
        B = int(q.shape[0])
        if out is None:
            out = torch.empty_like(q)
        ws = self.workspace(B) if workspace is None else workspace
        _lib.check("rcp_decode_step", self._lib.rcp_decode_step(
            self._h, _ptr(k), _ptr(v), _ptr(slot_mapping), int(slot_mapping.shape[0]), _ptr(q),
            _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens), B, _ptr(out), _ptr(ws),
            ws.numel() * ws.element_size(), _stream(stream)))
        return out

    def prefill_attn(self, q, cu_chunk_lens, block_table, seq_lens, out=None, workspace=None,
                     stream=None, variant: str = "auto"):
        """q: [sum chunk][H][d] fp16; cu_chunk_lens: [B+1] int32; seq_lens include the chunk.

        variant: "rank" (joint-coefficient contraction per head), "reconstruct" (dense values
        C_v W_v rebuilt once per key), or "auto": reconstruct when chunks average at least
        RECONSTRUCT_MIN_CHUNK rows.  The multiply-add count favours reconstruction above
        prefill_crossover_rows() (147 for R = 1024, d = 128); measured on GB300 it is the
        faster variant from 16-row chunks on (priors 4096 to 32768), because a chunk shorter
        than one 128-row tile costs the rank-space kernel a whole tile per R slice."""
        import torch
        rows = int(q.shape[0])
        B = int(seq_lens.shape[0])
        mb = int(block_table.shape[1])
        if variant == "auto":
            variant = "reconstruct" if (self.page_format == "fp8_e4m3" or
                                        (B > 0 and rows >= B * RECONSTRUCT_MIN_CHUNK)) else "rank"
        if variant not in ("rank", "reconstruct"):
            raise ValueError(f"unknown prefill variant {variant!r}")
        if out is None:
            out = torch.empty_like(q)
        if variant == "rank":
            ws = self.workspace(rows) if workspace is None else workspace
            fn, name = self._lib.rcp_prefill_attn, "rcp_prefill_attn"
        else:
            ws = self.workspace(rows, self.reconstruct_workspace_bytes(rows, B, mb)) \
                if workspace is None else workspace
            fn, name = self._lib.rcp_prefill_attn_reconstruct, "rcp_prefill_attn_reconstruct"
        _lib.check(name, fn(
            self._h, _ptr(q), _ptr(cu_chunk_lens), rows, _ptr(block_table), mb, _ptr(seq_lens), B,
            _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))
        return out
