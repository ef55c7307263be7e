"""GB300 (sm_103a) NVFP4 lightning indexer -- Python binding.

A thin ctypes layer over ``libnvfp4_indexer.so`` (C ABI declared in
``include/nvfp4_indexer.h``).  It only marshals arguments: checks dtypes,
shapes, devices and contiguity of torch tensors, passes raw device pointers
and the current CUDA stream, and turns non-zero status codes into
``IndexerError``.  Every step of the indexer runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback.  If the library has not been
built, importing the functions below raises.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

__all__ = ["Plan", "insert", "insert_norm_rope", "decode_noalloc", "sparse_attend", "IndexerError", "load_library", "library_path", "declared_symbols",
           "STATUS_BAD_PAGE", "STATUS_BAD_TABLE", "STATUS_TIMEOUT", "STATUS_BAD_SLOT", "STATUS_BAD_POSITION",
           "TOPK", "PAGE"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_LIB_PATH = os.path.join(_HERE, "libnvfp4_indexer.so")
_HEADER = os.path.join(_ROOT, "include", "nvfp4_indexer.h")

PAGE = 128
TOPK = 16
STATUS_BAD_PAGE, STATUS_BAD_TABLE, STATUS_TIMEOUT, STATUS_BAD_SLOT, STATUS_BAD_POSITION = 1, 2, 4, 8, 16
IDX_OK, IDX_EINVAL, IDX_EUNSUPPORTED, IDX_ECUDA, IDX_ENOSPACE, IDX_EDEVICE = 0, -1, -2, -3, -4, -5
IDX_PAGES_NVFP4, IDX_PAGES_MXFP4 = 0, 1

_lib = None


class IndexerError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def declared_symbols() -> list:
    """Function names declared in include/nvfp4_indexer.h."""
    text = open(_HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)


def load_library():
    """Load the built library (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.indexer_plan.argtypes = [ctypes.POINTER(P), I, I, I, I, I, I]
    lib.indexer_plan_destroy.argtypes = [P]
    lib.indexer_decode.argtypes = [P, P, P, I, P, I, P, I, I, P, P, I, P]
    lib.indexer_prefill.argtypes = [P, P, P, I, I, I, P, I, P, I, P, P, P, I, P]
    lib.nvfp4_insert.argtypes = [P, P, I, P, I, P, P]
    lib.indexer_decode_mxfp4.argtypes = lib.indexer_decode.argtypes
    lib.indexer_prefill_mxfp4.argtypes = lib.indexer_prefill.argtypes
    lib.mxfp4_insert.argtypes = lib.nvfp4_insert.argtypes
    lib.nvfp4_insert_norm_rope.argtypes = [P, P, P, I, P, ctypes.c_float, P, I, I, I, P, I, P, P]
    lib.indexer_decode_partial.argtypes = [P, I, P, P, I, P, I, P, P, P, I, I, P, P]
    lib.indexer_merge_candidates.argtypes = [P, I, I, I, I, P, P, P, P]
    lib.indexer_get_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
    lib.indexer_plan_set_wait_limit.argtypes = [P, ctypes.c_uint64]
    lib.indexer_last_error.restype = ctypes.c_char_p
    lib.indexer_version.restype = ctypes.c_char_p
    for name in ("indexer_plan", "indexer_plan_destroy", "indexer_decode", "indexer_prefill",
                 "nvfp4_insert", "indexer_get_status", "indexer_decode_mxfp4", "indexer_prefill_mxfp4",
                 "mxfp4_insert", "indexer_decode_partial", "indexer_merge_candidates", "nvfp4_insert_norm_rope",
                 "indexer_plan_set_wait_limit"):
        getattr(lib, name).restype = I
    _lib = lib
    return lib


def _check(rc: int):
    if rc != IDX_OK:
        raise IndexerError(rc, load_library().indexer_last_error().decode())


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t, dtype, name, ndim=None):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got {tuple(t.shape)}")
    return t.data_ptr()


class Plan:
    """Owns the indexer's device scratch for calls up to the given sizes
    (``indexer_plan``).  ``num_heads`` in {1, 2, 4, 8}; ``max_query_len`` 1..8."""

    def __init__(self, num_heads: int, max_reqs: int, max_query_len: int, max_pages_per_req: int,
                 max_prefill_tokens: int = 0, max_prefill_reqs: int = 0):
        lib = load_library()
        h = ctypes.c_void_p()
        _check(lib.indexer_plan(ctypes.byref(h), num_heads, max_reqs, max_query_len,
                                max_pages_per_req, max_prefill_tokens, max_prefill_reqs))
        self._h = h
        self.num_heads = num_heads
        self.max_pages_per_req = max_pages_per_req

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            load_library().indexer_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def decode(self, q, kv_pages, page_table, seq_lens, query_len: int, out=None, scores_dbg=None,
               stream=None):
        """Top-k pages of a uniform decode batch over NVFP4 pages [num_blocks, 128, 72];
        returns ``out`` int32 [rows, H, 16]."""
        return self._decode("indexer_decode", 3, q, kv_pages, page_table, seq_lens, query_len, out,
                            scores_dbg, stream)

    def decode_mxfp4(self, q, pages, page_table, seq_lens, query_len: int, out=None, scores_dbg=None,
                     stream=None):
        """``decode`` over MXFP4 pages [num_blocks, 8704] (``indexer_decode_mxfp4``)."""
        return self._decode("indexer_decode_mxfp4", 2, q, pages, page_table, seq_lens, query_len, out,
                            scores_dbg, stream)

    def prefill(self, q, cu_seqlens_q, kv_pages, page_table, seq_lens, max_seqlen_q: int, out=None,
                scores_dbg=None, stream=None):
        """Top-k pages of ragged prefill rows over NVFP4 pages [num_blocks, 128, 72];
        returns ``out`` int32 [total_q, H, 16]."""
        return self._prefill("indexer_prefill", 3, q, cu_seqlens_q, kv_pages, page_table, seq_lens,
                             max_seqlen_q, out, scores_dbg, stream)

    def prefill_mxfp4(self, q, cu_seqlens_q, pages, page_table, seq_lens, max_seqlen_q: int, out=None,
                      scores_dbg=None, stream=None):
        """``prefill`` over MXFP4 pages [num_blocks, 8704] (``indexer_prefill_mxfp4``)."""
        return self._prefill("indexer_prefill_mxfp4", 2, q, cu_seqlens_q, pages, page_table, seq_lens,
                             max_seqlen_q, out, scores_dbg, stream)

    def decode_partial(self, q, pages, page_table, seq_lens, page_lo, page_hi, query_len: int,
                       page_format: str = "nvfp4", cand_out=None, stream=None):
        """One context-parallel rank's share of a decode batch
        (``indexer_decode_partial``): scores request r's history pages in
        [page_lo[r], page_hi[r]) only and returns the rows' candidates, float32
        [rows, H, 15, 2] of (score, page id bits)."""
        import torch
        H = self.num_heads
        num_reqs = int(seq_lens.shape[0])
        if q.dim() != 3 or q.shape[0] != num_reqs * query_len or q.shape[1] != H or q.shape[2] != 128:
            raise ValueError(f"q: expected [{num_reqs * query_len}, {H}, 128], got {tuple(q.shape)}")
        fmt = {"nvfp4": (IDX_PAGES_NVFP4, 3), "mxfp4": (IDX_PAGES_MXFP4, 2)}[page_format]
        if cand_out is None:
            cand_out = torch.empty((q.shape[0], H, 15, 2), dtype=torch.float32, device=q.device)
        _check(load_library().indexer_decode_partial(
            self._h, fmt[0], _ptr(q, torch.uint8, "q"), _ptr(pages, torch.uint8, "pages", fmt[1]),
            int(pages.shape[0]), _ptr(page_table, torch.int32, "page_table", 2), int(page_table.shape[1]),
            _ptr(seq_lens, torch.int32, "seq_lens", 1), _ptr(page_lo, torch.int32, "page_lo", 1),
            _ptr(page_hi, torch.int32, "page_hi", 1), num_reqs, int(query_len),
            _ptr(cand_out, torch.float32, "cand_out", 4), _stream_ptr(stream)))
        return cand_out

    def _decode(self, fn, pages_ndim, q, kv_pages, page_table, seq_lens, query_len, out, scores_dbg,
                stream):
        import torch
        H = self.num_heads
        if q.dim() != 3 or q.shape[1] != H or q.shape[2] != 128:
            raise ValueError(f"q: expected [rows, {H}, 128], got {tuple(q.shape)}")
        num_reqs = int(seq_lens.shape[0])
        if q.shape[0] != num_reqs * query_len:
            raise ValueError("q rows != num_reqs * query_len")
        if out is None:
            out = torch.empty((q.shape[0], H, TOPK), dtype=torch.int32, device=q.device)
        dbg_stride = 0
        if scores_dbg is not None:
            dbg_stride = int(scores_dbg.shape[-1])
        _check(getattr(load_library(), fn)(
            self._h, _ptr(q, torch.uint8, "q"), _ptr(kv_pages, torch.uint8, "kv_pages", pages_ndim),
            int(kv_pages.shape[0]), _ptr(page_table, torch.int32, "page_table", 2), int(page_table.shape[1]),
            _ptr(seq_lens, torch.int32, "seq_lens", 1), num_reqs, int(query_len),
            _ptr(out, torch.int32, "out"), _ptr(scores_dbg, torch.float32, "scores_dbg"), dbg_stride,
            _stream_ptr(stream)))
        return out

    def _prefill(self, fn, pages_ndim, q, cu_seqlens_q, kv_pages, page_table, seq_lens, max_seqlen_q,
                 out, scores_dbg, stream):
        import torch
        H = self.num_heads
        if q.dim() != 3 or q.shape[1] != H or q.shape[2] != 128:
            raise ValueError(f"q: expected [total_q, {H}, 128], got {tuple(q.shape)}")
        num_reqs = int(seq_lens.shape[0])
        if cu_seqlens_q.shape[0] != num_reqs + 1:
            raise ValueError("cu_seqlens_q must have num_reqs + 1 entries")
        total_q = int(q.shape[0])
        if out is None:
            out = torch.empty((total_q, H, TOPK), dtype=torch.int32, device=q.device)
        dbg_stride = int(scores_dbg.shape[-1]) if scores_dbg is not None else 0
        _check(getattr(load_library(), fn)(
            self._h, _ptr(q, torch.uint8, "q"), _ptr(cu_seqlens_q, torch.int32, "cu_seqlens_q", 1),
            num_reqs, total_q, int(max_seqlen_q), _ptr(kv_pages, torch.uint8, "kv_pages", pages_ndim),
            int(kv_pages.shape[0]), _ptr(page_table, torch.int32, "page_table", 2), int(page_table.shape[1]),
            _ptr(seq_lens, torch.int32, "seq_lens", 1), _ptr(out, torch.int32, "out"),
            _ptr(scores_dbg, torch.float32, "scores_dbg"), dbg_stride, _stream_ptr(stream)))
        return out

    def set_wait_limit(self, wait_ns: int = 0):
        """Wall-time limit (ns) of every bounded wait inside the decode and
        prefill kernels of later calls (``indexer_plan_set_wait_limit``);
        0 restores the default of 2 s."""
        _check(load_library().indexer_plan_set_wait_limit(self._h, int(wait_ns)))

    def status(self, stream=None) -> int:
        """Synchronise, read and clear the device status word (IDX_STATUS_* bits)."""
        bits = ctypes.c_int32(0)
        rc = load_library().indexer_get_status(self._h, _stream_ptr(stream), ctypes.byref(bits))
        if rc not in (IDX_OK, IDX_EDEVICE):
            _check(rc)
        return int(bits.value)


def insert(k_bf16, slot_mapping, kv_pages, status=None, stream=None):
    """Quantise bf16 keys [n, 128] to NVFP4 and write them at ``slot_mapping``
    (``nvfp4_insert``; pages [num_blocks, 128, 72])."""
    return _insert("nvfp4_insert", 3, k_bf16, slot_mapping, kv_pages, status, stream)


def mxfp4_insert(k_bf16, slot_mapping, pages, status=None, stream=None):
    """Quantise bf16 keys [n, 128] to MXFP4 and write them at ``slot_mapping``
    (``mxfp4_insert``; pages [num_blocks, 8704])."""
    return _insert("mxfp4_insert", 2, k_bf16, slot_mapping, pages, status, stream)


def insert_norm_rope(k_bf16, positions, slot_mapping, norm_weight, eps, cos_sin_cache, rotary_dim: int,
                     is_neox: bool, kv_pages, status=None, stream=None):
    """qk-norm (RMSNorm with ``norm_weight`` bf16 [128] and ``eps``), RoPE
    from ``cos_sin_cache`` float32 [max_pos, rotary_dim] at ``positions``
    int64 [n], bf16 rounding, then the NVFP4 insert of keys [n, 128] into
    ``kv_pages`` [num_blocks, 128, 72] (``nvfp4_insert_norm_rope``)."""
    import torch
    if k_bf16.dim() != 2 or k_bf16.shape[1] != 128:
        raise ValueError("k_bf16: expected [n, 128]")
    kb = k_bf16.view(torch.int16) if k_bf16.dtype == torch.bfloat16 else k_bf16
    wb = norm_weight.view(torch.int16) if norm_weight.dtype == torch.bfloat16 else norm_weight
    n = int(kb.shape[0])
    if slot_mapping.shape[0] != n or (positions is not None and positions.shape[0] != n):
        raise ValueError("slot_mapping and positions must have one entry per key")
    if wb.numel() != 128:
        raise ValueError("norm_weight: expected 128 elements")
    max_pos = 0
    if cos_sin_cache is not None:
        if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != rotary_dim:
            raise ValueError(f"cos_sin_cache: expected [max_pos, {rotary_dim}]")
        max_pos = int(cos_sin_cache.shape[0])
    _check(load_library().nvfp4_insert_norm_rope(
        _ptr(kb, torch.int16, "k_bf16"), _ptr(positions, torch.int64, "positions", 1),
        _ptr(slot_mapping, torch.int64, "slot_mapping", 1), n, _ptr(wb, torch.int16, "norm_weight"),
        float(eps), _ptr(cos_sin_cache, torch.float32, "cos_sin_cache"), max_pos, int(rotary_dim),
        1 if is_neox else 0, _ptr(kv_pages, torch.uint8, "kv_pages", 3), int(kv_pages.shape[0]),
        _ptr(status, torch.int32, "status"), _stream_ptr(stream)))
    return kv_pages


def _insert(fn, pages_ndim, k_bf16, slot_mapping, kv_pages, status, stream):
    import torch
    if k_bf16.dim() != 2 or k_bf16.shape[1] != 128:
        raise ValueError("k_bf16: expected [n, 128]")
    kb = k_bf16.view(torch.int16) if k_bf16.dtype == torch.bfloat16 else k_bf16
    n = int(kb.shape[0])
    if slot_mapping.shape[0] != n:
        raise ValueError("slot_mapping must have one entry per key")
    _check(getattr(load_library(), fn)(
        _ptr(kb, torch.int16, "k_bf16"), _ptr(slot_mapping, torch.int64, "slot_mapping", 1), n,
        _ptr(kv_pages, torch.uint8, "kv_pages", pages_ndim), int(kv_pages.shape[0]),
        _ptr(status, torch.int32, "status"), _stream_ptr(stream)))
    return kv_pages


def merge_candidates(cand_all, seq_lens, query_len: int, num_heads: int, out=None, status=None, stream=None):
    """``indexer_merge_candidates``: final rows [rows, H, 16] from the
    candidates of ``world`` ranks, ``cand_all`` float32 [world, rows, H, 15, 2]."""
    import torch
    if cand_all.dim() != 5 or cand_all.shape[2] != num_heads or cand_all.shape[3] != 15:
        raise ValueError(f"cand_all: expected [world, rows, {num_heads}, 15, 2], got {tuple(cand_all.shape)}")
    num_reqs = int(seq_lens.shape[0])
    if cand_all.shape[1] != num_reqs * query_len:
        raise ValueError("cand_all rows != num_reqs * query_len")
    if out is None:
        out = torch.empty((cand_all.shape[1], num_heads, TOPK), dtype=torch.int32, device=cand_all.device)
    _check(load_library().indexer_merge_candidates(
        _ptr(cand_all, torch.float32, "cand_all", 5), int(cand_all.shape[0]), num_reqs, int(query_len),
        int(num_heads), _ptr(seq_lens, torch.int32, "seq_lens", 1), _ptr(out, torch.int32, "out"),
        _ptr(status, torch.int32, "status"), _stream_ptr(stream)))
    return out


def gather_candidates(cand, group=None):
    """All-gather every rank's candidates into one rank-major tensor
    [world, rows, H, 15, 2] (torch.distributed; the one exchange of decode
    context parallelism).  Without an initialised process group: one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return cand.unsqueeze(0)
    world = dist.get_world_size(group)
    parts = [torch.empty_like(cand) for _ in range(world)]
    dist.all_gather(parts, cand.contiguous(), group=group)
    return torch.stack(parts)


def decode_cp(plan, q, pages, page_table, seq_lens, page_lo, page_hi, query_len: int, page_format="nvfp4",
              group=None, out=None, stream=None):
    """Decode context parallelism: this rank's share (``decode_partial``), one
    all-gather of the candidates over ``group``, then the merge; returns the
    final rows on every rank."""
    cand = plan.decode_partial(q, pages, page_table, seq_lens, page_lo, page_hi, query_len,
                               page_format=page_format, stream=stream)
    return merge_candidates(gather_candidates(cand, group), seq_lens, query_len, plan.num_heads, out=out,
                            stream=stream)


def sparse_attend(q, k_cache, v_cache, page_table, row_req, row_pos, topk_ids, scale: float, out=None,
                  status=None, stream=None):
    """``indexer_sparse_attend``: block-sparse attention of bf16 queries
    [rows, H * G, 128] over the pages in ``topk_ids`` [rows, H, 16] of a bf16
    main cache [num_blocks, 128, H, 128] (K and V); returns fp32
    [rows, H * G, 128]."""
    import torch
    lib = load_library()
    fn = lib.indexer_sparse_attend
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, P, P, I, P, I, I, P, P, P, I, I, I, ctypes.c_float, P, P, P]
    fn.restype = I
    if k_cache.dim() != 4 or k_cache.shape[1] != PAGE or k_cache.shape[3] != 128 or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache / v_cache: expected the same shape [num_blocks, 128, H, 128]")
    H = int(k_cache.shape[2])
    rows = int(topk_ids.shape[0])
    if topk_ids.dim() != 3 or topk_ids.shape[1] != H or topk_ids.shape[2] != TOPK:
        raise ValueError(f"topk_ids: expected [rows, {H}, 16], got {tuple(topk_ids.shape)}")
    if q.dim() != 3 or q.shape[0] != rows or q.shape[1] % H or q.shape[2] != 128:
        raise ValueError(f"q: expected [{rows}, {H} * G, 128], got {tuple(q.shape)}")
    if row_req.shape[0] != rows or row_pos.shape[0] != rows:
        raise ValueError("row_req / row_pos must have one entry per row")
    qb = q.view(torch.int16) if q.dtype == torch.bfloat16 else q
    kb = k_cache.view(torch.int16) if k_cache.dtype == torch.bfloat16 else k_cache
    vb = v_cache.view(torch.int16) if v_cache.dtype == torch.bfloat16 else v_cache
    if out is None:
        out = torch.empty(tuple(q.shape), dtype=torch.float32, device=q.device)
    _check(fn(_ptr(qb, torch.int16, "q"), _ptr(kb, torch.int16, "k_cache"), _ptr(vb, torch.int16, "v_cache"),
              int(k_cache.shape[0]), _ptr(page_table, torch.int32, "page_table", 2), int(page_table.shape[1]),
              int(page_table.shape[0]), _ptr(row_req, torch.int32, "row_req", 1),
              _ptr(row_pos, torch.int32, "row_pos", 1), _ptr(topk_ids, torch.int32, "topk_ids", 3), rows, H,
              int(q.shape[1]) // H, float(scale), _ptr(out, torch.float32, "out", 3),
              _ptr(status, torch.int32, "status"), _stream_ptr(stream)))
    return out


def decode_noalloc(q, kv_pages, page_table, seq_lens, query_len: int, num_heads: int, out=None,
                   status=None, stream=None):
    """``indexer_decode_noalloc``: the decode indexer for callers that cannot
    allocate device memory (no plan; scratch in a fixed array inside the
    library).  Calls that overlap on the GPU share that array and race."""
    import torch
    lib = load_library()
    fn = lib.indexer_decode_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, P, I, P, I, P, I, I, I, P, P, P]
    fn.restype = I
    num_reqs = int(seq_lens.shape[0])
    if q.dim() != 3 or q.shape[0] != num_reqs * query_len or q.shape[1] != num_heads or q.shape[2] != 128:
        raise ValueError(f"q: expected [{num_reqs * query_len}, {num_heads}, 128], got {tuple(q.shape)}")
    if out is None:
        out = torch.empty((q.shape[0], num_heads, TOPK), dtype=torch.int32, device=q.device)
    _check(fn(_ptr(q, torch.uint8, "q"), _ptr(kv_pages, torch.uint8, "kv_pages", 3), int(kv_pages.shape[0]),
              _ptr(page_table, torch.int32, "page_table", 2), int(page_table.shape[1]),
              _ptr(seq_lens, torch.int32, "seq_lens", 1), num_reqs, int(query_len), int(num_heads),
              _ptr(out, torch.int32, "out"), _ptr(status, torch.int32, "status"), _stream_ptr(stream)))
    return out
