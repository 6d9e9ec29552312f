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


def _need(name: str, x, dtype, shape=None, device=None) -> None:
    """Check one tensor argument before its pointer crosses the C ABI, which cannot see
    dtypes, strides or devices: raise ValueError unless ``x`` is a contiguous tensor of
    ``dtype`` on ``device`` whose shape matches ``shape`` (None entries match any size)."""
    import torch
    if not isinstance(x, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor, got {type(x).__name__}")
    if x.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {x.dtype}")
    if shape is not None:
        if x.dim() != len(shape) or any(e is not None and x.shape[i] != e
                                        for i, e in enumerate(shape)):
            want = "[" + ", ".join("*" if e is None else str(e) for e in shape) + "]"
            raise ValueError(f"{name} must have shape {want}, got {list(x.shape)}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and x.device != device:
        raise ValueError(f"{name} must be on {device}, got {x.device}")


def _validate_append(device, H: int, d: int, k, v, slot_mapping) -> int:
    """k, v: [T][H][d] fp16; slot_mapping: [T] int64.  Returns T."""
    import torch
    _need("slot_mapping", slot_mapping, torch.int64, (None,), device)
    T = int(slot_mapping.shape[0])
    _need("k", k, torch.float16, (T, H, d), device)
    _need("v", v, torch.float16, (T, H, d), device)
    return T


def _validate_decode(device, H: int, d: int, q, block_table, seq_lens, out) -> int:
    """q, out: [B][H][d] fp16; block_table: [>= B][max_blocks] int32; seq_lens: [B] int32.
    Returns B."""
    import torch
    _need("q", q, torch.float16, (None, H, d), device)
    B = int(q.shape[0])
    _need("seq_lens", seq_lens, torch.int32, (B,), device)
    _need("block_table", block_table, torch.int32, (None, None), device)
    if block_table.shape[0] < B or block_table.shape[1] < 1:
        raise ValueError(f"block_table needs at least {B} rows and one column, "
                         f"got {list(block_table.shape)}")
    _need("out", out, torch.float16, (B, H, d), device)
    return B


def _validate_prefill(device, H: int, d: int, q, cu_chunk_lens, block_table, seq_lens,
                      out) -> tuple[int, int]:
    """q, out: [rows][H][d] fp16; seq_lens: [B] int32; cu_chunk_lens: [B+1] int32;
    block_table: [>= B][max_blocks] int32.  Returns (rows, B)."""
    import torch
    _need("q", q, torch.float16, (None, H, d), device)
    rows = int(q.shape[0])
    _need("seq_lens", seq_lens, torch.int32, (None,), device)
    B = int(seq_lens.shape[0])
    _need("cu_chunk_lens", cu_chunk_lens, torch.int32, (B + 1,), device)
    _need("block_table", block_table, torch.int32, (None, None), device)
    if block_table.shape[0] < B or block_table.shape[1] < 1:
        raise ValueError(f"block_table needs at least {B} rows and one column, "
                         f"got {list(block_table.shape)}")
    _need("out", out, torch.float16, (rows, H, d), device)
    return rows, B


def _validate_workspace(device, ws) -> None:
    import torch
    _need("workspace", ws, torch.uint8, (None,), device)


def _stream(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def int4_page_bytes(num_heads: int, rank_k: int, rank_v: int):
    """Bytes of one 4-bit K page and one V page: the codes (two per byte), then the fp16
    scales (one per key row of a head, one per 64 value coefficients of a token)."""
    k = num_heads * BLOCK_SIZE * rank_k // 2 + num_heads * BLOCK_SIZE * 2
    v = BLOCK_SIZE * rank_v // 2 + BLOCK_SIZE * (rank_v // 64) * 2
    return k, v


class PagedCoeffCache:
    """Paged low-rank coefficient cache on one GPU.

    Owns (as torch tensors) the K pages [num_blocks][H][16][r_k], V pages
    [num_blocks][16][R], the factors, a device error word and a reusable workspace; the
    library handle borrows their pointers.  page_format "fp16" stores fp16 coefficients,
    "fp8_e4m3" stores E4M3 codes (uint8 tensors), "int4" stores 4-bit codes with fp16
    scales as raw bytes (K pages [num_blocks][int4_page_bytes()[0]], V pages
    [num_blocks][int4_page_bytes()[1]], uint8).  A prefill on quantized pages first widens
    the pages it reads to fp16 in the workspace (the "auto" variant reconstructs); they have
    no block-sparse decode.
    """

    def __init__(self, num_heads: int, head_dim: int, rank_k: int, rank_v: int,
                 num_blocks: int, U_k, W_v, k_pages=None, v_pages=None, device=None,
                 page_format: str = "fp16"):
        import torch
        lib = _lib.load()
        dev = U_k.device if device is None else torch.device(device)
        if dev.type != "cuda":
            raise ValueError(f"the cache lives on a CUDA device, got {dev}")
        if dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        formats = {"fp16": _lib.RCP_PAGES_FP16, "fp8_e4m3": _lib.RCP_PAGES_FP8_E4M3,
                   "int4": _lib.RCP_PAGES_INT4}
        if page_format not in formats:
            raise ValueError(f"unknown page_format {page_format!r}")
        fmt = formats[page_format]
        page_dtype = torch.float16 if fmt == _lib.RCP_PAGES_FP16 else torch.uint8
        self.page_format = page_format
        self.shape = dict(num_heads=num_heads, head_dim=head_dim, rank_k=rank_k, rank_v=rank_v)
        self.num_blocks = int(num_blocks)
        self.device = dev
        _need("U_k", U_k, torch.float16, (num_heads, rank_k, head_dim), dev)
        _need("W_v", W_v, torch.float16, (rank_v, num_heads * head_dim), dev)
        self.U_k = U_k
        self.W_v = W_v
        if fmt == _lib.RCP_PAGES_INT4:
            kb, vb = int4_page_bytes(num_heads, rank_k, rank_v)
            k_shape, v_shape = (num_blocks, kb), (num_blocks, vb)
        else:
            k_shape = (num_blocks, num_heads, BLOCK_SIZE, rank_k)
            v_shape = (num_blocks, BLOCK_SIZE, rank_v)
        if k_pages is None:
            k_pages = torch.zeros(k_shape, dtype=page_dtype, device=dev)
        if v_pages is None:
            v_pages = torch.zeros(v_shape, dtype=page_dtype, device=dev)
        _need("k_pages", k_pages, page_dtype, k_shape, dev)
        _need("v_pages", v_pages, page_dtype, v_shape, dev)
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
        H, d = self.shape["num_heads"], self.shape["head_dim"]
        T = _validate_append(self.device, H, d, k, v, slot_mapping)
        _lib.check("rcp_append_kv", self._lib.rcp_append_kv(
            self._h, _ptr(k), _ptr(v), _ptr(slot_mapping), T, _stream(stream)))

    def decode_attn(self, q, block_table, seq_lens, out=None, workspace=None, stream=None):
        """q: [B][H][d] fp16; block_table: [B][max_blocks] int32; seq_lens: [B] int32."""
        import torch
        if out is None:
            out = torch.empty_like(q)
        H, d = self.shape["num_heads"], self.shape["head_dim"]
        B = _validate_decode(self.device, H, d, q, block_table, seq_lens, out)
        ws = self.workspace(B) if workspace is None else workspace
        _validate_workspace(self.device, ws)
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
        if out is None:
            out = torch.empty_like(q)
        H, d = self.shape["num_heads"], self.shape["head_dim"]
        B = _validate_decode(self.device, H, d, q, block_table, seq_lens, out)
        if page_kept is not None:
            _need("page_kept", page_kept, torch.uint8, tuple(block_table.shape), self.device)
        ws = self.workspace(B) if workspace is None else workspace
        _validate_workspace(self.device, ws)
        _lib.check("rcp_decode_attn_sparse", self._lib.rcp_decode_attn_sparse(
            self._h, _ptr(q), _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens), B,
            float(skip_threshold), _ptr(page_kept) if page_kept is not None else None,
            _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))
        return out

    def decode_step(self, k, v, slot_mapping, q, block_table, seq_lens, out=None, workspace=None,
                    stream=None):
        """append_kv(k, v, slot_mapping) then decode_attn(q, ...), queued as one step."""
        import torch
        if out is None:
            out = torch.empty_like(q)
        H, d = self.shape["num_heads"], self.shape["head_dim"]
        _validate_append(self.device, H, d, k, v, slot_mapping)
        B = _validate_decode(self.device, H, d, q, block_table, seq_lens, out)
        ws = self.workspace(B) if workspace is None else workspace
        _validate_workspace(self.device, ws)
        _lib.check("rcp_decode_step", self._lib.rcp_decode_step(
            self._h, _ptr(k), _ptr(v), _ptr(slot_mapping), int(slot_mapping.shape[0]), _ptr(q),
            _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens), B, _ptr(out), _ptr(ws),
            ws.numel() * ws.element_size(), _stream(stream)))
        return out

    def _prefill_variant(self, variant: str, rows: int, B: int) -> str:
        if variant == "auto":
            variant = "reconstruct" if (self.page_format != "fp16" or
                                        (B > 0 and rows >= B * RECONSTRUCT_MIN_CHUNK)) else "rank"
        if variant not in ("rank", "reconstruct"):
            raise ValueError(f"unknown prefill variant {variant!r}")
        return variant

    def _prefill_workspace(self, variant: str, rows: int, B: int, mb: int):
        # quantized pages are widened into the workspace first (both variants)
        if variant == "rank" and self.page_format == "fp16":
            return self.workspace(rows, self.workspace_bytes(rows))
        return self.workspace(rows, self.reconstruct_workspace_bytes(rows, B, mb))

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
        if out is None:
            out = torch.empty_like(q)
        H, d = self.shape["num_heads"], self.shape["head_dim"]
        rows, B = _validate_prefill(self.device, H, d, q, cu_chunk_lens, block_table, seq_lens,
                                    out)
        mb = int(block_table.shape[1])
        variant = self._prefill_variant(variant, rows, B)
        ws = self._prefill_workspace(variant, rows, B, mb) if workspace is None else workspace
        if variant == "rank":
            fn, name = self._lib.rcp_prefill_attn, "rcp_prefill_attn"
        else:
            fn, name = self._lib.rcp_prefill_attn_reconstruct, "rcp_prefill_attn_reconstruct"
        _validate_workspace(self.device, ws)
        _lib.check(name, fn(
            self._h, _ptr(q), _ptr(cu_chunk_lens), rows, _ptr(block_table), mb, _ptr(seq_lens), B,
            _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))
        return out

    def prefill_step(self, k, v, slot_mapping, q, cu_chunk_lens, block_table, seq_lens,
                     out=None, workspace=None, stream=None, variant: str = "auto"):
        """append_kv(k, v, slot_mapping) then prefill_attn(q, cu_chunk_lens, ...), queued as
        one step (the chunk's query projection shares the append's launch).  Arguments and
        variant choice as the two calls."""
        import torch
        if out is None:
            out = torch.empty_like(q)
        H, d = self.shape["num_heads"], self.shape["head_dim"]
        T = _validate_append(self.device, H, d, k, v, slot_mapping)
        rows, B = _validate_prefill(self.device, H, d, q, cu_chunk_lens, block_table, seq_lens,
                                    out)
        mb = int(block_table.shape[1])
        variant = self._prefill_variant(variant, rows, B)
        ws = self._prefill_workspace(variant, rows, B, mb) if workspace is None else workspace
        _validate_workspace(self.device, ws)
        _lib.check("rcp_prefill_step", self._lib.rcp_prefill_step(
            self._h, _ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(q), _ptr(cu_chunk_lens), rows,
            _ptr(block_table), mb, _ptr(seq_lens), B, 1 if variant == "reconstruct" else 0,
            _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))
        return out
