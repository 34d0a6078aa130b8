"""Python binding of libfa.so: argument marshalling only. Every step of the computation runs in the
library's CUDA kernels; PyTorch provides device memory and the current stream.

Names follow the C ABI (include/fa.h): create_block_mask, flex_forward, flex_decode, ...
The library must have been built (``__graft_entry__.build()`` or ``python -m
block_sparse_masked_create_gb300.build``); a missing library is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

from . import build as _build

MAX_OPS = 16
MAX_TERMS = 8

OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_CHECK, ERR_BUFFER = range(8)
_OPS = {"true": 0, "causal": 1, "window": 2, "prefix": 3, "doc": 4, "and": 5, "or": 6}


class FaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class MaskRule(ctypes.Structure):
    _fields_ = [("n_ops", ctypes.c_int32), ("op", ctypes.c_int32 * MAX_OPS), ("arg", ctypes.c_int64 * MAX_OPS),
                ("doc_ids", ctypes.c_void_p), ("doc_batch", ctypes.c_int32), ("doc_len", ctypes.c_int32),
                ("q_offset", ctypes.c_void_p), ("batch_dependent", ctypes.c_int32),
                ("head_dependent", ctypes.c_int32)]


class ScoreRule(ctypes.Structure):
    _fields_ = [("alibi_slopes", ctypes.c_void_p), ("rel_bias", ctypes.c_void_p), ("softcap", ctypes.c_float)]


class BlockMaskC(ctypes.Structure):
    _fields_ = [("Bm", ctypes.c_int32), ("Hm", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("kv_len", ctypes.c_int32), ("bq", ctypes.c_int32), ("bk", ctypes.c_int32),
                ("nq", ctypes.c_int32), ("nk", ctypes.c_int32),
                ("kv_num", ctypes.c_void_p), ("kv_idx", ctypes.c_void_p), ("full_kv_num", ctypes.c_void_p),
                ("full_kv_idx", ctypes.c_void_p), ("q_num", ctypes.c_void_p), ("q_idx", ctypes.c_void_p),
                ("full_q_num", ctypes.c_void_p), ("full_q_idx", ctypes.c_void_p),
                ("block_class", ctypes.c_void_p), ("doc_run", ctypes.c_void_p), ("doc_sorted", ctypes.c_void_p),
                ("row_order", ctypes.c_void_p), ("rule", MaskRule)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libfa.so (raises if it has not been built: there is no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libfa.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    P = ctypes.POINTER
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [ctypes.c_int]
    lib.fa_version.restype = ctypes.c_char_p
    lib.fa_block_mask_bytes.restype = sz
    lib.fa_block_mask_bytes.argtypes = [P(MaskRule), i32, i32, i32, i32, i32, i32]
    lib.fa_create_block_mask.restype = ctypes.c_int
    lib.fa_create_block_mask.argtypes = [P(MaskRule), i32, i32, i32, i32, i32, i32, vp, sz, P(BlockMaskC), vp]
    fwd_args = [vp, vp, vp, P(BlockMaskC), P(ScoreRule), f32, vp, i32, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.fa_flex_forward.restype = ctypes.c_int
    lib.fa_flex_forward.argtypes = fwd_args
    lib.fa_flex_forward_mma.restype = ctypes.c_int
    lib.fa_flex_forward_mma.argtypes = fwd_args
    lib.fa_block_mask_select_bytes.restype = sz
    lib.fa_block_mask_select_bytes.argtypes = [P(BlockMaskC), i32]
    lib.fa_block_mask_select_rows.restype = ctypes.c_int
    lib.fa_block_mask_select_rows.argtypes = [P(BlockMaskC), vp, i32, vp, sz, P(BlockMaskC), vp, vp]
    lib.fa_forward_split_workspace_bytes.restype = sz
    lib.fa_forward_split_workspace_bytes.argtypes = [P(BlockMaskC), i32, i32, i32, i32]
    lib.fa_flex_forward_split.restype = ctypes.c_int
    lib.fa_flex_forward_split.argtypes = [vp, vp, vp, P(BlockMaskC), P(ScoreRule), f32, vp, i32, vp, i32, i32, i32, i32,
                                          i32, i32, i32, vp, sz, vp, vp]
    lib.fa_forward_host_workspace_bytes.restype = sz
    lib.fa_forward_host_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.fa_flex_forward_host.restype = ctypes.c_int
    lib.fa_flex_forward_host.argtypes = [vp, vp, vp, P(BlockMaskC), P(ScoreRule), f32, vp, i32, vp, i32, i32, i32, i32,
                                         i32, i32, vp, sz, vp, vp]
    lib.fa_flex_forward_paged.restype = ctypes.c_int
    lib.fa_flex_forward_paged.argtypes = [vp, vp, vp, vp, i32, i32, i32, P(BlockMaskC), P(ScoreRule), f32, vp, i32, vp,
                                          i32, i32, i32, i32, i32, i32, vp, vp]
    lib.fa_flex_backward.restype = ctypes.c_int
    lib.fa_flex_backward.argtypes = [vp, vp, vp, vp, i32, vp, vp, P(BlockMaskC), P(ScoreRule), f32, vp, vp, vp, vp,
                                     i32, i32, i32, i32, i32, i32, vp, vp]
    lib.fa_decode_workspace_bytes.restype = sz
    lib.fa_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.fa_flex_decode.restype = ctypes.c_int
    lib.fa_flex_decode.argtypes = [vp, vp, vp, vp, i32, P(BlockMaskC), P(ScoreRule), f32, vp, i32, vp, i32, i32, i32, i32,
                                   i32, i32, vp, sz, vp, vp, vp]
    lib.fa_flex_decode_noalloc.restype = ctypes.c_int
    lib.fa_flex_decode_noalloc.argtypes = [vp, vp, vp, vp, i32, P(BlockMaskC), P(ScoreRule), f32, vp, i32, vp, i32,
                                           i32, i32, i32, i32, i32, vp, vp, vp]
    lib.fa_decode_noalloc_scratch_bytes.restype = sz
    lib.fa_decode_noalloc_scratch_bytes.argtypes = []
    lib.fa_block_mask_stats.restype = ctypes.c_int
    lib.fa_block_mask_stats.argtypes = [P(BlockMaskC), vp, vp]
    lib.fa_check_status.restype = ctypes.c_int
    lib.fa_check_status.argtypes = [vp, vp]
    lib.fa_set_wait_timeout_ns.restype = None
    lib.fa_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.fa_get_wait_timeout_ns.restype = ctypes.c_uint64
    lib.fa_get_wait_timeout_ns.argtypes = []
    lib.fa_debug_wait_timeout.restype = ctypes.c_int
    lib.fa_debug_wait_timeout.argtypes = [vp, ctypes.c_uint64, vp]
    lib.fa_debug_softcap.restype = ctypes.c_int
    lib.fa_debug_softcap.argtypes = [vp, vp, i32, ctypes.c_float, vp]
    lib.fa_debug_tc5_gemm.restype = ctypes.c_int
    lib.fa_debug_tc5_gemm.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
    _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load().fa_status_string(code).decode()
    except Exception:  # library not loadable
        return f"status {code}"


def _check(code: int, what: str):
    if code != OK:
        raise FaError(code, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


# ----------------------------------------------------------------------------------------------
# rules
# ----------------------------------------------------------------------------------------------
def make_mask_rule(spec: Sequence[tuple], doc_ids: Optional[torch.Tensor] = None,
                   q_offset: Optional[torch.Tensor] = None, batch_dependent: Optional[bool] = None,
                   head_dependent: bool = False) -> MaskRule:
    """Rule spec (postfix tuples, see workloads.py) -> fa_mask_rule. doc_ids int32 [doc_batch, doc_len] and
    q_offset int32 [B] must be device tensors and stay alive while the rule is used."""
    if not 1 <= len(spec) <= MAX_OPS:
        raise ValueError("rule must have 1..16 ops")
    r = MaskRule()
    r.n_ops = len(spec)
    for i, op in enumerate(spec):
        r.op[i] = _OPS[op[0]]
        r.arg[i] = int(op[1]) if len(op) > 1 else 0
    if doc_ids is not None:
        if doc_ids.dtype != torch.int32 or doc_ids.dim() != 2 or not doc_ids.is_contiguous():
            raise ValueError("doc_ids must be contiguous int32 [doc_batch, doc_len]")
        r.doc_ids = doc_ids.data_ptr()
        r.doc_batch, r.doc_len = doc_ids.shape
    if q_offset is not None:
        if q_offset.dtype != torch.int32 or not q_offset.is_contiguous():
            raise ValueError("q_offset must be contiguous int32 [B]")
        r.q_offset = q_offset.data_ptr()
    if batch_dependent is None:
        batch_dependent = q_offset is not None or (doc_ids is not None and doc_ids.shape[0] > 1)
    r.batch_dependent = int(bool(batch_dependent))
    r.head_dependent = int(bool(head_dependent))
    r._tensors = (doc_ids, q_offset)  # the raw pointers above stay valid while the rule lives
    return r


def make_score_rule(alibi_slopes: Optional[torch.Tensor] = None, rel_bias: Optional[torch.Tensor] = None,
                    softcap: float = 0.0) -> ScoreRule:
    s = ScoreRule()
    for t in (alibi_slopes, rel_bias):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError("score tables must be contiguous fp32 device tensors")
    s.alibi_slopes = None if alibi_slopes is None else alibi_slopes.data_ptr()
    s.rel_bias = None if rel_bias is None else rel_bias.data_ptr()
    s.softcap = float(softcap or 0.0)
    s._tensors = (alibi_slopes, rel_bias)  # the raw pointers above stay valid while the rule lives
    return s


# ----------------------------------------------------------------------------------------------
# BlockMask
# ----------------------------------------------------------------------------------------------
@dataclass
class BlockMask:
    c: BlockMaskC
    buf: torch.Tensor
    keep: list = field(default_factory=list)   # tensors the rule points into

    @property
    def shape(self):
        return (self.c.Bm, self.c.Hm, self.c.nq, self.c.nk)

    def _view(self, addr: int, n: int, dtype) -> torch.Tensor:
        off = addr - self.buf.data_ptr()
        nbytes = n * (4 if dtype == torch.int32 else 1)
        return self.buf[off:off + nbytes].view(dtype)

    def tables(self) -> dict:
        """Device views of the tables: kv_num [Bm,Hm,nq], kv_idx [Bm,Hm,nq,nk], ..., block_class."""
        Bm, Hm, nq, nk = self.shape
        c = self.c
        out = {}
        for name, n, shp in (("kv_num", Bm * Hm * nq, (Bm, Hm, nq)), ("full_kv_num", Bm * Hm * nq, (Bm, Hm, nq)),
                             ("q_num", Bm * Hm * nk, (Bm, Hm, nk)), ("full_q_num", Bm * Hm * nk, (Bm, Hm, nk)),
                             ("kv_idx", Bm * Hm * nq * nk, (Bm, Hm, nq, nk)),
                             ("full_kv_idx", Bm * Hm * nq * nk, (Bm, Hm, nq, nk)),
                             ("q_idx", Bm * Hm * nk * nq, (Bm, Hm, nk, nq)),
                             ("full_q_idx", Bm * Hm * nk * nq, (Bm, Hm, nk, nq))):
            out[name] = self._view(getattr(c, name), n, torch.int32).view(shp)
        out["block_class"] = self._view(c.block_class, Bm * Hm * nq * nk, torch.uint8).view(Bm, Hm, nq, nk)
        if c.row_order:
            out["row_order"] = self._view(c.row_order, Bm * Hm * nq, torch.int32).view(Bm, Hm, nq)
        return out


def block_mask_bytes(rule: MaskRule, B: int, H: int, Q_LEN: int, KV_LEN: int, Bq: int, Bk: int) -> int:
    return int(load().fa_block_mask_bytes(ctypes.byref(rule), B, H, Q_LEN, KV_LEN, Bq, Bk))


def create_block_mask(rule: MaskRule, B: int, H: int, Q_LEN: int, KV_LEN: int, Bq: int = 128, Bk: int = 128,
                      device="cuda", keep: Optional[list] = None, buf: Optional[torch.Tensor] = None) -> BlockMask:
    """fa_create_block_mask: classify every block, compact the lists, build the transpose (on `device`)."""
    lib = load()
    n = block_mask_bytes(rule, B, H, Q_LEN, KV_LEN, Bq, Bk)
    if n == 0:
        raise FaError(ERR_SHAPE, "fa_block_mask_bytes")
    if buf is None or buf.numel() < n:
        buf = torch.empty(n, dtype=torch.uint8, device=device)
    c = BlockMaskC()
    _check(lib.fa_create_block_mask(ctypes.byref(rule), B, H, Q_LEN, KV_LEN, Bq, Bk, _ptr(buf), buf.numel(),
                                    ctypes.byref(c), _stream(buf.device)), "fa_create_block_mask")
    return BlockMask(c, buf, list(keep or []))


def recreate_block_mask(bm: BlockMask, rule: MaskRule, B: int, H: int, Q_LEN: int, KV_LEN: int, Bq: int,
                        Bk: int) -> None:
    """Rebuild into an existing BlockMask's buffer (same sizes; no allocation)."""
    _check(load().fa_create_block_mask(ctypes.byref(rule), B, H, Q_LEN, KV_LEN, Bq, Bk, _ptr(bm.buf), bm.buf.numel(),
                                       ctypes.byref(bm.c), _stream(bm.buf.device)), "fa_create_block_mask")


def select_rows(src: BlockMask, q_pos: torch.Tensor, out: Optional[BlockMask] = None,
                status: Optional[torch.Tensor] = None) -> BlockMask:
    """fa_block_mask_select_rows: from a table prebuilt for the longest context (global positions), the row
    block holding each request's query position q_pos[b] (device int32 [Bz]), as a one-row-per-request
    mask (Bm = Bz, q_len = 1, Bq = 1) whose rule sees q_pos as the query offset. Reuses `out`'s buffer."""
    if q_pos.dtype != torch.int32 or not q_pos.is_contiguous() or q_pos.dim() != 1:
        raise ValueError("q_pos must be contiguous int32 [Bz]")
    lib = load()
    Bz = q_pos.shape[0]
    n = int(lib.fa_block_mask_select_bytes(ctypes.byref(src.c), Bz))
    if n == 0:
        raise FaError(ERR_SHAPE, "fa_block_mask_select_bytes")
    if out is None or out.buf.numel() < n:
        out = BlockMask(BlockMaskC(), torch.empty(n, dtype=torch.uint8, device=src.buf.device), [])
    out.keep = list(src.keep) + [src, q_pos]
    _check(lib.fa_block_mask_select_rows(ctypes.byref(src.c), _ptr(q_pos), Bz, _ptr(out.buf), out.buf.numel(),
                                         ctypes.byref(out.c), _ptr(status), _stream(out.buf.device)),
           "fa_block_mask_select_rows")
    return out


def block_mask_stats(bm: BlockMask, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """int64[6] on the device: full, partial, empty, max row length, sum of row lengths, rows."""
    if out is None:
        out = torch.empty(6, dtype=torch.int64, device=bm.buf.device)
    _check(load().fa_block_mask_stats(ctypes.byref(bm.c), _ptr(out), _stream(out.device)), "fa_block_mask_stats")
    return out


# ----------------------------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------------------------
def _out_code(out: torch.Tensor) -> int:
    if out.dtype == torch.bfloat16:
        return 0
    if out.dtype == torch.float32:
        return 1
    raise ValueError("out must be bf16 or fp32")


def flex_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block_mask: BlockMask,
                 score: Optional[ScoreRule] = None, scale: Optional[float] = None,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 status: Optional[torch.Tensor] = None, counters: Optional[torch.Tensor] = None,
                 force_mma: bool = False, out_dtype=torch.bfloat16):
    """fa_flex_forward: q [B,Hq,Q_LEN,d], k/v [B,Hkv,KV_LEN,d] bf16 contiguous on the GPU.
    Returns (out [B,Hq,Q_LEN,d] in bf16 or fp32 (the dtype of `out`, else out_dtype), lse fp32 [B,Hq,Q_LEN])."""
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    B, Hq, Q_LEN, d = q.shape
    Hkv, KV_LEN = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Q_LEN), dtype=torch.float32, device=q.device)
    fn = load().fa_flex_forward_mma if force_mma else load().fa_flex_forward
    _check(fn(_ptr(q), _ptr(k), _ptr(v), ctypes.byref(block_mask.c), ctypes.byref(score) if score else None,
              float(scale) if scale else 0.0, _ptr(out), _out_code(out), _ptr(lse), B, Hq, Hkv, Q_LEN, KV_LEN, d,
              _ptr(status), _ptr(counters), _stream(q.device)), "fa_flex_forward")
    return out, lse


def forward_split_workspace_bytes(block_mask: BlockMask, B: int, Hq: int, d: int, chunk_blocks: int) -> int:
    return int(load().fa_forward_split_workspace_bytes(ctypes.byref(block_mask.c), B, Hq, d, chunk_blocks))


def flex_forward_split(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block_mask: BlockMask,
                       score: Optional[ScoreRule] = None, scale: Optional[float] = None, chunk_blocks: int = 16,
                       out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                       out_dtype=torch.bfloat16):
    """fa_flex_forward_split: the forward with each query block row cut into chunks of at most chunk_blocks
    key blocks, run as separate tiles and merged. Same inputs and outputs as flex_forward."""
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    B, Hq, Q_LEN, d = q.shape
    Hkv, KV_LEN = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Q_LEN), dtype=torch.float32, device=q.device)
    n = forward_split_workspace_bytes(block_mask, B, Hq, d, chunk_blocks)
    if n == 0:
        raise FaError(ERR_SHAPE, "fa_forward_split_workspace_bytes")
    if workspace is None or workspace.numel() < n:
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    _check(load().fa_flex_forward_split(_ptr(q), _ptr(k), _ptr(v), ctypes.byref(block_mask.c),
                                        ctypes.byref(score) if score else None, float(scale) if scale else 0.0,
                                        _ptr(out), _out_code(out), _ptr(lse), B, Hq, Hkv, Q_LEN, KV_LEN, d,
                                        chunk_blocks, _ptr(workspace), workspace.numel(), _ptr(status),
                                        _stream(q.device)), "fa_flex_forward_split")
    return out, lse


def forward_host_workspace_bytes(B: int, Hq: int, Hkv: int, Q_LEN: int, KV_LEN: int, d: int,
                                 out_dtype=torch.bfloat16) -> int:
    return int(load().fa_forward_host_workspace_bytes(B, Hq, Hkv, Q_LEN, KV_LEN, d,
                                                      1 if out_dtype == torch.float32 else 0))


def flex_forward_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block_mask: BlockMask,
                      score: Optional[ScoreRule] = None, scale: Optional[float] = None,
                      out: torch.Tensor = None, lse: torch.Tensor = None, workspace: torch.Tensor = None,
                      status: Optional[torch.Tensor] = None, device=None):
    """fa_flex_forward_host: q/k/v (bf16), out (bf16 or fp32) and lse (fp32) are host tensors (pin them for
    full copy speed); the chunks stream through `workspace` on `device`. Returns (out, lse) once the
    current stream of `device` has been synchronised by the caller."""
    for t in (q, k, v, out, lse):
        if t is None or t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v, out, lse must be contiguous host tensors")
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("q, k, v must be bf16")
    B, Hq, Q_LEN, d = q.shape
    Hkv, KV_LEN = k.shape[1], k.shape[2]
    dev = torch.device(device) if device is not None else block_mask.buf.device
    if workspace is None:
        workspace = torch.empty(forward_host_workspace_bytes(B, Hq, Hkv, Q_LEN, KV_LEN, d, out.dtype),
                                dtype=torch.uint8, device=dev)
    _check(load().fa_flex_forward_host(_ptr(q), _ptr(k), _ptr(v), ctypes.byref(block_mask.c),
                                       ctypes.byref(score) if score else None, float(scale) if scale else 0.0,
                                       _ptr(out), _out_code(out), _ptr(lse), B, Hq, Hkv, Q_LEN, KV_LEN, d,
                                       _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev)),
           "fa_flex_forward_host")
    return out, lse


def flex_forward_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, page_table: torch.Tensor,
                       block_mask: BlockMask, KV_LEN: int, score: Optional[ScoreRule] = None,
                       scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                       lse: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                       out_dtype=torch.bfloat16):
    """fa_flex_forward_paged: q [B,Hq,Q_LEN,d]; k/v pages [P,Hkv,page,d] bf16 with page == the mask's Bk;
    page_table int32 [B,max_pages] (logical key block -> physical page)."""
    for t in (q, k_pages, v_pages):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q, k_pages, v_pages must be contiguous bf16 CUDA tensors")
    if page_table.dtype != torch.int32 or not page_table.is_contiguous() or page_table.dim() != 2:
        raise ValueError("page_table must be contiguous int32 [B, max_pages]")
    B, Hq, Q_LEN, d = q.shape
    P, Hkv, page, _ = k_pages.shape
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Q_LEN), dtype=torch.float32, device=q.device)
    _check(load().fa_flex_forward_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), P, page,
                                        page_table.shape[1], ctypes.byref(block_mask.c),
                                        ctypes.byref(score) if score else None, float(scale) if scale else 0.0,
                                        _ptr(out), _out_code(out), _ptr(lse), B, Hq, Hkv, Q_LEN, KV_LEN, d,
                                        _ptr(status), _stream(q.device)), "fa_flex_forward_paged")
    return out, lse


def flex_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
                  dout: torch.Tensor, block_mask: BlockMask, score: Optional[ScoreRule] = None,
                  scale: Optional[float] = None, dq: Optional[torch.Tensor] = None,
                  dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
                  delta: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None):
    """fa_flex_backward: gradients (dq, dk, dv) in fp32 of fa_flex_forward's out for the upstream gradient
    dout (bf16, layout of q); out and lse are that forward's outputs."""
    for t in (q, k, v, dout):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q, k, v, dout must be contiguous bf16 CUDA tensors")
    B, Hq, Q_LEN, d = q.shape
    Hkv, KV_LEN = k.shape[1], k.shape[2]
    dev = q.device
    dq = torch.empty(q.shape, dtype=torch.float32, device=dev) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.float32, device=dev) if dk is None else dk
    dv = torch.empty(v.shape, dtype=torch.float32, device=dev) if dv is None else dv
    delta = torch.empty((B, Hq, Q_LEN), dtype=torch.float32, device=dev) if delta is None else delta
    _check(load().fa_flex_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _out_code(out), _ptr(dout), _ptr(lse),
                                   ctypes.byref(block_mask.c), ctypes.byref(score) if score else None,
                                   float(scale) if scale else 0.0, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(delta),
                                   B, Hq, Hkv, Q_LEN, KV_LEN, d, _ptr(status), _stream(dev)), "fa_flex_backward")
    return dq, dk, dv


def decode_workspace_bytes(Bz: int, Hq: int, d: int, max_pages: int, page: int) -> int:
    return int(load().fa_decode_workspace_bytes(Bz, Hq, d, max_pages, page))


def flex_decode(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, page_table: torch.Tensor,
                block_mask: BlockMask, score: Optional[ScoreRule] = None, scale: Optional[float] = None,
                out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                counters: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16):
    """fa_flex_decode: q [Bz,Hq,d], k/v pages [P,Hkv,page,d] bf16, page_table int32 [Bz,max_pages]."""
    Bz, Hq, d = q.shape
    P, Hkv, page, _ = k_pages.shape
    max_pages = page_table.shape[1]
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((Bz, Hq), dtype=torch.float32, device=q.device)
    need = decode_workspace_bytes(Bz, Hq, d, max_pages, page)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(load().fa_flex_decode(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), P,
                                 ctypes.byref(block_mask.c), ctypes.byref(score) if score else None,
                                 float(scale) if scale else 0.0, _ptr(out), _out_code(out), _ptr(lse), Bz, Hq, Hkv,
                                 d, page, max_pages, _ptr(workspace), workspace.numel(), _ptr(status),
                                 _ptr(counters), _stream(q.device)), "fa_flex_decode")
    return out, lse


def decode_noalloc_scratch_bytes() -> int:
    return int(load().fa_decode_noalloc_scratch_bytes())


def flex_decode_noalloc(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, page_table: torch.Tensor,
                        block_mask: BlockMask, score: Optional[ScoreRule] = None, scale: Optional[float] = None,
                        out: torch.Tensor = None, lse: torch.Tensor = None, status: Optional[torch.Tensor] = None,
                        counters: Optional[torch.Tensor] = None) -> int:
    """fa_flex_decode_noalloc: the paged decode with its split workspace in the library's fixed device
    array, for callers that cannot allocate. `out` and `lse` must be provided (nothing is allocated here).
    Returns the fa_status code (FA_ERR_BUFFER_TOO_SMALL when the problem exceeds the fixed array)."""
    if out is None or lse is None:
        raise ValueError("out and lse must be provided")
    Bz, Hq, d = q.shape
    P, Hkv, page, _ = k_pages.shape
    return int(load().fa_flex_decode_noalloc(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), P, ctypes.byref(block_mask.c),
        ctypes.byref(score) if score else None, float(scale) if scale else 0.0, _ptr(out), _out_code(out), _ptr(lse),
        Bz, Hq, Hkv, d, page, page_table.shape[1], _ptr(status), _ptr(counters), _stream(q.device)))


def check_status(status: torch.Tensor) -> int:
    return int(load().fa_check_status(_ptr(status), _stream(status.device)))


def set_wait_timeout_ns(ns: int) -> None:
    load().fa_set_wait_timeout_ns(int(ns))


def get_wait_timeout_ns() -> int:
    return int(load().fa_get_wait_timeout_ns())


def debug_wait_timeout(status: torch.Tensor, timeout_ns: int) -> int:
    return int(load().fa_debug_wait_timeout(_ptr(status), int(timeout_ns), _stream(status.device)))


def debug_softcap(x: torch.Tensor, c: float) -> torch.Tensor:
    """c * tanh(x / c) as the kernels compute it, for a contiguous fp32 CUDA tensor."""
    y = torch.empty_like(x)
    _check(load().fa_debug_softcap(_ptr(x), _ptr(y), x.numel(), float(c), _stream(x.device)), "fa_debug_softcap")
    return y


def debug_tc5_gemm(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, K: int, b_mn_major: bool, use_tma: bool,
                   status: Optional[torch.Tensor] = None) -> int:
    return int(load().fa_debug_tc5_gemm(_ptr(A), _ptr(B), _ptr(C), K, int(b_mn_major), int(use_tma), _ptr(status),
                                        _stream(A.device)))
