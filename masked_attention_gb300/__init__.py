"""Masked fused attention for one GB300 GPU (sm_103a).

A thin ctypes binding of ``libmattn.so`` (C ABI in ``include/mattn.h``). The
functions here only marshal arguments: every step of the computation runs in
the library's CUDA kernels. There is no CPU fallback: if the library has not
been built (``python -m masked_attention_gb300._build``), loading it raises.

Tensors are passed as torch CUDA tensors (or raw device addresses as ints);
PyTorch provides device memory and streams only.

With the environment variable ``MATTN_DEBUG=1`` set before the first call,
the debug build ``libmattn_debug.so`` is loaded instead (device-side bounds
checks, ``include/mattn_debug.h``; build it with
``python -m masked_attention_gb300._build --debug``); ``debug_record`` and
``debug_selftest`` read and test its checks.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

__all__ = [
    "MASK_CAUSAL", "MASK_WINDOW", "MASK_DOCUMENT", "MASK_PREFIX", "SCORE_ALIBI",
    "SCORE_SOFTCAP", "BF16", "F32", "AttnError", "BlockMask", "attn_fwd", "attn_bwd",
    "attn_decode", "attn_decode_workspace_bytes",
    "build_block_mask", "attn_block_mask_bytes", "attn_bwd_workspace_bytes", "attn_bwd_noalloc",
    "attn_check_status", "attn_status_str", "attn_last_cuda_error", "attn_combine", "lib",
    "LIB_PATH", "LIB_DEBUG_PATH", "debug_record", "debug_selftest",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmattn.so")
LIB_DEBUG_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmattn_debug.so")

# Mirrors of the constants in include/mattn.h (a test checks they agree).
ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_MISALIGNED = 0, 1, 2, 3
ATTN_ERR_WORKSPACE_TOO_SMALL, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = 4, 5, 6
MASK_CAUSAL, MASK_WINDOW, MASK_DOCUMENT, MASK_PREFIX = 1 << 0, 1 << 1, 1 << 2, 1 << 3
SCORE_ALIBI, SCORE_SOFTCAP, SCORE_RELBIAS = 1 << 8, 1 << 9, 1 << 10
BF16, F32 = 0, 1
TILE = 128
FAULT_NO_LOADS = 1


class attn_block_mask(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Sq", ctypes.c_int), ("Skv", ctypes.c_int),
                ("nq", ctypes.c_int), ("nkv", ctypes.c_int), ("variant", ctypes.c_uint),
                ("window", ctypes.c_int), ("doc_id", ctypes.c_void_p),
                ("prefix_len", ctypes.c_void_p), ("full_cnt", ctypes.c_void_p),
                ("part_cnt", ctypes.c_void_p), ("full_idx", ctypes.c_void_p),
                ("part_idx", ctypes.c_void_p), ("order", ctypes.c_void_p),
                ("t_full_cnt", ctypes.c_void_p), ("t_part_cnt", ctypes.c_void_p),
                ("t_full_idx", ctypes.c_void_p), ("t_part_idx", ctypes.c_void_p),
                ("t_order", ctypes.c_void_p), ("q_offset", ctypes.c_int),
                ("kv_offset", ctypes.c_int), ("doc_len", ctypes.c_int)]


class attn_params(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("scale", ctypes.c_float), ("window", ctypes.c_int),
                ("softcap", ctypes.c_float), ("alibi_slopes", ctypes.c_void_p),
                ("doc_id", ctypes.c_void_p), ("prefix_len", ctypes.c_void_p),
                ("block_mask", ctypes.POINTER(attn_block_mask)), ("status", ctypes.c_void_p),
                ("timeout_ns", ctypes.c_ulonglong), ("rel_bias", ctypes.c_void_p),
                ("fault_inject", ctypes.c_uint), ("page_table", ctypes.c_void_p),
                ("page_size", ctypes.c_int), ("pages_per_seq", ctypes.c_int),
                ("num_pages", ctypes.c_int), ("q_offset", ctypes.c_int),
                ("kv_offset", ctypes.c_int), ("doc_len", ctypes.c_int)]


class attn_debug_info(ctypes.Structure):
    _fields_ = [("count", ctypes.c_ulonglong), ("site", ctypes.c_int), ("pad", ctypes.c_int),
                ("index", ctypes.c_longlong), ("bound", ctypes.c_longlong)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        debug = os.environ.get("MATTN_DEBUG", "0") not in ("", "0")
        path = LIB_DEBUG_PATH if debug else LIB_PATH
        if not os.path.exists(path):
            flag = " --debug" if debug else ""
            raise RuntimeError(f"{path} is missing: build it with "
                               f"`python -m masked_attention_gb300._build{flag}` (no CPU fallback)")
        L = ctypes.CDLL(path)
        vp, i, u, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
        P = ctypes.POINTER(attn_params)
        BM = ctypes.POINTER(attn_block_mask)
        L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, u, P, vp]
        L.attn_fwd.restype = i
        L.attn_block_mask_bytes.argtypes = [i, i, i, i]
        L.attn_block_mask_bytes.restype = sz
        L.build_block_mask.argtypes = [u, P, i, i, i, vp, sz, i, BM, vp]
        L.build_block_mask.restype = i
        L.attn_bwd_workspace_bytes.argtypes = [i, i, i]
        L.attn_bwd_workspace_bytes.restype = sz
        L.attn_bwd_workspace_bytes_f16.argtypes = [i, i, i, i, i, i]
        L.attn_bwd_workspace_bytes_f16.restype = sz
        L.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, u, P,
                               vp]
        L.attn_bwd.restype = i
        L.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, u,
                                       P, vp]
        L.attn_bwd_noalloc.restype = i
        L.attn_doc_ids_from_seqlens.argtypes = [vp, i, i, vp, vp]
        L.attn_doc_ids_from_seqlens.restype = i
        L.attn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, u, P, vp, sz, vp]
        L.attn_decode.restype = i
        L.attn_decode_workspace_bytes.argtypes = [i, i, i, i, i, i]
        L.attn_decode_workspace_bytes.restype = sz
        L.attn_combine.argtypes = [vp, vp, i, ctypes.c_longlong, i, i, vp, vp, vp]
        L.attn_combine.restype = i
        L.attn_check_status.argtypes = [vp, vp]
        L.attn_check_status.restype = i
        L.attn_status_str.argtypes = [i]
        L.attn_status_str.restype = ctypes.c_char_p
        L.attn_last_cuda_error.argtypes = []
        L.attn_last_cuda_error.restype = ctypes.c_char_p
        if debug:
            L.attn_debug_record.argtypes = [ctypes.POINTER(attn_debug_info), i]
            L.attn_debug_record.restype = i
            L.attn_debug_site_name.argtypes = [i]
            L.attn_debug_site_name.restype = ctypes.c_char_p
            L.attn_debug_selftest.argtypes = [vp]
            L.attn_debug_selftest.restype = i
        _lib = L
    return _lib


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {attn_status_str(status)} (status {status})"
        if status == ATTN_ERR_CUDA:
            msg += f": {attn_last_cuda_error()}"
        super().__init__(msg)


def _debug_lib():
    L = lib()
    if not hasattr(L, "attn_debug_record"):
        raise RuntimeError("the release library is loaded: set MATTN_DEBUG=1 before the first "
                           "call to load libmattn_debug.so")
    return L


def debug_record(clear: bool = False) -> dict:
    """Debug build: the failed bounds checks of every kernel so far (count,
    and site name, index and bound of the first); ``clear`` resets them."""
    L = _debug_lib()
    info = attn_debug_info()
    _check(L.attn_debug_record(ctypes.byref(info), 1 if clear else 0), "attn_debug_record")
    return {"count": int(info.count), "site": L.attn_debug_site_name(info.site).decode(),
            "index": int(info.index), "bound": int(info.bound)}


def debug_selftest(stream=None) -> None:
    """Debug build: checks that an index planted past a buffer's end is
    refused and recorded (attn_debug_selftest); raises if not."""
    _check(_debug_lib().attn_debug_selftest(_stream(stream)), "attn_debug_selftest")


def attn_last_cuda_error() -> str:
    """Name of the CUDA error behind this thread's most recent ATTN_ERR_CUDA."""
    return lib().attn_last_cuda_error().decode()


def attn_status_str(status: int) -> str:
    return lib().attn_status_str(int(status)).decode()


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != ATTN_OK:
        raise AttnError(status, where)


class BlockMask:
    """A block mask built on the device. Holds the device buffer (a torch
    uint8 tensor) and the host struct that describes it."""

    def __init__(self, buf, struct: attn_block_mask, keep_alive: tuple):
        self.buf = buf
        self.struct = struct
        self._keep = keep_alive

    @property
    def nq(self) -> int:
        return self.struct.nq

    @property
    def nkv(self) -> int:
        return self.struct.nkv

    def to_host(self) -> dict:
        """Copies the lists to the host (for tests and inspection)."""
        import torch
        s = self.struct
        base = self.buf.data_ptr()

        def view(addr, n):
            off = addr - base
            return self.buf[off:off + 4 * n].view(torch.int32).cpu().numpy()

        B, nq, nkv = s.B, s.nq, s.nkv
        out = dict(full_cnt=view(s.full_cnt, B * nq).reshape(B, nq),
                   part_cnt=view(s.part_cnt, B * nq).reshape(B, nq),
                   full_idx=view(s.full_idx, B * nq * nkv).reshape(B, nq, nkv),
                   part_idx=view(s.part_idx, B * nq * nkv).reshape(B, nq, nkv),
                   order=view(s.order, B * nq))
        if s.t_full_cnt:
            out.update(t_full_cnt=view(s.t_full_cnt, B * nkv).reshape(B, nkv),
                       t_part_cnt=view(s.t_part_cnt, B * nkv).reshape(B, nkv),
                       t_full_idx=view(s.t_full_idx, B * nkv * nq).reshape(B, nkv, nq),
                       t_part_idx=view(s.t_part_idx, B * nkv * nq).reshape(B, nkv, nq),
                       t_order=view(s.t_order, B * nkv))
        return out


def _params(dtype: int, scale: float, window: int, softcap: float, alibi_slopes, doc_id,
            prefix_len, block_mask: Optional[BlockMask], status, timeout_ns: int,
            fault_inject: int = 0, rel_bias=None, q_offset: int = 0,
            kv_offset: int = 0) -> attn_params:
    p = attn_params()
    p.dtype = dtype
    p.scale = scale
    p.window = window
    p.softcap = softcap
    p.alibi_slopes = _ptr(alibi_slopes)
    p.doc_id = _ptr(doc_id)
    p.prefix_len = _ptr(prefix_len)
    p.block_mask = ctypes.pointer(block_mask.struct) if block_mask is not None else None
    p.status = _ptr(status)
    p.timeout_ns = timeout_ns
    p.fault_inject = fault_inject
    p.rel_bias = _ptr(rel_bias)
    p.q_offset = q_offset
    p.kv_offset = kv_offset
    # the row length of the document ids, from the tensor ([B, L] or [L])
    p.doc_len = int(doc_id.shape[-1]) if doc_id is not None and hasattr(doc_id, "shape") else 0
    return p


def attn_block_mask_bytes(B: int, Sq: int, Skv: int, transposed: bool = False) -> int:
    return int(lib().attn_block_mask_bytes(B, Sq, Skv, int(transposed)))


def attn_bwd_workspace_bytes(B: int, Hq: int, Sq: int) -> int:
    return int(lib().attn_bwd_workspace_bytes(B, Hq, Sq))


def attn_bwd_workspace_bytes_f16(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int) -> int:
    """Workspace bytes for attn_bwd's fp16 path (fp16 copies of q, k, v, dO)."""
    return int(lib().attn_bwd_workspace_bytes_f16(B, Hq, Hkv, Sq, Skv, D))


def build_block_mask(variant: int, B: int, Sq: int, Skv: int, *, window: int = 0, doc_id=None,
                     prefix_len=None, transposed: bool = False, device="cuda",
                     buf=None, q_offset: int = 0, kv_offset: int = 0,
                     stream=None) -> BlockMask:
    """Builds the block mask on the device (``buf``: optional caller buffer,
    a uint8 CUDA tensor of at least ``attn_block_mask_bytes`` bytes).
    ``q_offset``/``kv_offset``: absolute positions of query row 0 and key 0
    (one shard of a longer sequence)."""
    import torch
    nbytes = attn_block_mask_bytes(B, Sq, Skv, transposed)
    if buf is None:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    p = _params(BF16, 0.0, window, 0.0, None, doc_id, prefix_len, None, None, 0,
                q_offset=q_offset, kv_offset=kv_offset)
    out = attn_block_mask()
    st = lib().build_block_mask(variant, ctypes.byref(p), B, Sq, Skv, _ptr(buf),
                                buf.numel() if hasattr(buf, "numel") else nbytes,
                                int(transposed), ctypes.byref(out), _stream(stream))
    _check(st, "build_block_mask")
    return BlockMask(buf, out, (doc_id, prefix_len))


def attn_fwd(q, k, v, o, lse, variant: int = 0, *, B=None, Hq=None, Hkv=None, Sq=None,
             Skv=None, D=None, dtype: Optional[int] = None, scale: float = 0.0, window: int = 0,
             softcap: float = 0.0, alibi_slopes=None, doc_id=None, prefix_len=None,
             block_mask: Optional[BlockMask] = None, status=None, timeout_ns: int = 0,
             fault_inject: int = 0, rel_bias=None, page_table=None, page_size: int = 0,
             q_offset: int = 0, kv_offset: int = 0, stream=None) -> None:
    """O and LSE of masked attention; writes ``o`` and ``lse`` in place.

    Paged K/V cache: ``k``/``v`` are page pools [num_pages, Hkv, page_size, D]
    and ``page_table`` [B, pages_per_seq] int32 maps logical to physical pages;
    pass ``Skv`` (the shapes cannot tell it).

    One shard of a longer sequence: ``q_offset``/``kv_offset`` are the
    absolute positions of query row 0 and key 0 (mask terms, ALiBi and
    document ids use absolute positions); merge the results over key shards
    with ``attn_combine``.

    ``q`` [B,Hq,Sq,D], ``k``/``v`` [B,Hkv,Skv,D], ``o`` like ``q``, ``lse`` fp32
    [B,Hq,Sq]. Shapes come from the tensors unless given explicitly (needed
    when raw addresses are passed)."""
    if B is None:
        B, Hq, Sq, D = q.shape
        Hkv = k.shape[1]
        if Skv is None:
            Skv = k.shape[2]
    if dtype is None:
        import torch
        dtype = F32 if q.dtype == torch.float32 else BF16
    p = _params(dtype, scale, window, softcap, alibi_slopes, doc_id, prefix_len, block_mask,
                status, timeout_ns, fault_inject, rel_bias, q_offset, kv_offset)
    if page_table is not None:
        p.page_table = _ptr(page_table)
        p.page_size = page_size
        p.pages_per_seq = page_table.shape[1]
        p.num_pages = k.shape[0]
    st = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv, D,
                        variant, ctypes.byref(p), _stream(stream))
    _check(st, "attn_fwd")


def attn_decode_workspace_bytes(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int) -> int:
    return int(lib().attn_decode_workspace_bytes(B, Hq, Hkv, Sq, Skv, D))


def attn_decode(q, k, v, o, lse, variant: int = 0, *, workspace=None, Skv=None,
                scale: float = 0.0, window: int = 0, softcap: float = 0.0, alibi_slopes=None,
                doc_id=None, prefix_len=None, status=None, timeout_ns: int = 0, rel_bias=None,
                page_table=None, page_size: int = 0, q_offset: int = 0, kv_offset: int = 0,
                stream=None) -> None:
    """Decode: few query rows (q [B,Hq,Sq,D], (Hq/Hkv) * Sq <= 16) against a
    long key/value cache, contiguous [B,Hkv,Skv,D] or paged (``page_table``
    [B, pages_per_seq] into pools [num_pages, Hkv, page_size, D]; pass
    ``Skv``). ``workspace``: optional CUDA tensor for the split partial
    results (``attn_decode_workspace_bytes``). Writes ``o`` and ``lse``."""
    B, Hq, Sq, D = q.shape
    Hkv = k.shape[1]
    if Skv is None:
        Skv = k.shape[2]
    p = _params(BF16, scale, window, softcap, alibi_slopes, doc_id, prefix_len, None, status,
                timeout_ns, 0, rel_bias, q_offset, kv_offset)
    if page_table is not None:
        p.page_table = _ptr(page_table)
        p.page_size = page_size
        p.pages_per_seq = page_table.shape[1]
        p.num_pages = k.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv,
                           D, variant, ctypes.byref(p), _ptr(workspace), ws_bytes,
                           _stream(stream))
    _check(st, "attn_decode")


def attn_combine(o_parts, lse_parts, o, lse, stream=None) -> None:
    """Merges results over disjoint key sets (e.g. key/value shards):
    ``o_parts`` [n, ...rows..., D] (bf16 or fp32 CUDA tensor), ``lse_parts``
    fp32 [n, ...rows...]; writes ``o`` [...rows..., D] and ``lse``
    [...rows...] in place: LSE = ln sum_k exp(LSE_k), O = sum_k
    exp(LSE_k - LSE) O_k."""
    import torch
    for name, x in (("o_parts", o_parts), ("lse_parts", lse_parts), ("o", o), ("lse", lse)):
        if not x.is_contiguous():
            raise ValueError(f"attn_combine: {name} must be contiguous")
    n, D = o_parts.shape[0], o_parts.shape[-1]
    rows = lse_parts[0].numel()
    if o.numel() != rows * D or lse.numel() != rows or o_parts.numel() != n * rows * D:
        raise ValueError("attn_combine: shapes of the parts and the outputs disagree")
    dtype = F32 if o_parts.dtype == torch.float32 else BF16
    st = lib().attn_combine(_ptr(o_parts), _ptr(lse_parts), n, rows, D, dtype, _ptr(o),
                            _ptr(lse), _stream(stream))
    _check(st, "attn_combine")


def doc_ids_from_seqlens(cu_seqlens, total: Optional[int] = None, doc_id=None,
                         stream=None):
    """Jagged batches: per-position sequence index of ``total`` packed
    positions from the cumulative lengths ``cu_seqlens`` (int32 CUDA tensor,
    n + 1 entries starting at 0). Use the result as ``doc_id`` ([1, total])
    with ``MASK_DOCUMENT`` and B = 1 to attend within each sequence only."""
    import torch
    n = cu_seqlens.numel() - 1
    if total is None:
        total = int(cu_seqlens[-1].item())
    if doc_id is None:
        doc_id = torch.empty(1, total, dtype=torch.int32, device=cu_seqlens.device)
    st = lib().attn_doc_ids_from_seqlens(_ptr(cu_seqlens), n, total, _ptr(doc_id),
                                         _stream(stream))
    _check(st, "attn_doc_ids_from_seqlens")
    return doc_id


def attn_bwd(q, k, v, o, lse, do, dq, dk, dv, workspace, variant: int = 0, *,
             scale: float = 0.0, window: int = 0, softcap: float = 0.0, alibi_slopes=None,
             doc_id=None, prefix_len=None, block_mask: Optional[BlockMask] = None, status=None,
             timeout_ns: int = 0, fault_inject: int = 0, q_offset: int = 0, kv_offset: int = 0,
             rel_bias=None, stream=None) -> None:
    """dQ, dK, dV of ``sum(dO * O)``; writes ``dq``, ``dk``, ``dv`` in place.
    ``workspace``: a CUDA tensor of at least ``attn_bwd_workspace_bytes`` bytes.
    ``q_offset``/``kv_offset``: absolute positions of query row 0 and key 0
    (one shard of a longer sequence; the block mask must be built for them).
    ``rel_bias``: the forward's relative-position bias table (no gradient)."""
    import torch
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    dtype = F32 if q.dtype == torch.float32 else BF16
    p = _params(dtype, scale, window, softcap, alibi_slopes, doc_id, prefix_len, block_mask,
                status, timeout_ns, fault_inject, rel_bias=rel_bias, q_offset=q_offset,
                kv_offset=kv_offset)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                        _ptr(dk), _ptr(dv), _ptr(workspace), ws_bytes, B, Hq, Hkv, Sq, Skv, D,
                        variant, ctypes.byref(p), _stream(stream))
    _check(st, "attn_bwd")


def attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, variant: int = 0, *,
                     scale: float = 0.0, window: int = 0, softcap: float = 0.0,
                     alibi_slopes=None, doc_id=None, prefix_len=None,
                     block_mask: Optional[BlockMask] = None, status=None, timeout_ns: int = 0,
                     q_offset: int = 0, kv_offset: int = 0, rel_bias=None,
                     stream=None) -> None:
    """attn_bwd without a workspace argument, for callers that cannot allocate
    device memory: the library's own fixed array holds the row terms (at most
    B*Hq*Sq = 2,097,152; see include/mattn.h). Writes dq, dk, dv in place."""
    import torch
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    dtype = F32 if q.dtype == torch.float32 else BF16
    p = _params(dtype, scale, window, softcap, alibi_slopes, doc_id, prefix_len, block_mask,
                status, timeout_ns, rel_bias=rel_bias, q_offset=q_offset,
                kv_offset=kv_offset)
    st = lib().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Skv, D, variant,
                                ctypes.byref(p), _stream(stream))
    _check(st, "attn_bwd_noalloc")


def attn_check_status(status=None, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status word."""
    return int(lib().attn_check_status(_ptr(status), _stream(stream)))


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)
