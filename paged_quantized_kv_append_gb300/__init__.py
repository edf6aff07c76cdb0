"""Paged quantized-KV append and paged decode / verify attention on GB300.

A thin ctypes binding of libpqkv.so (include/pqkv.h): it checks tensor
dtypes and shapes, passes device pointers and the current CUDA stream, and
raises on a non-zero return code.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback path.

    kv_append_quant(k, v, slot_mapping, kv_dtype, k_scale, v_scale, pages)
    paged_attention(q, pages, block_table, seq_lens, q_len, kv_dtype,
                    k_scale, v_scale, out)

Pool layout: ``pages`` is [num_pages, num_kv_heads, 2, 16, 128] -- for each
page and kv-head a 16-token K tile followed by a V tile -- of uint8 codes
(E4M3 / INT8) or float16 values.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

FP16 = 0
FP8_E4M3 = 1
INT8 = 2
INT8_ROW = 3          # int8 with a scale per (token, kv-head) row, computed at append time
KV_DTYPES = {"fp16": FP16, "fp8_e4m3": FP8_E4M3, "int8": INT8, "int8_row": INT8_ROW}
_SCALED = (FP8_E4M3, INT8)   # formats that take k_scale / v_scale arguments

HEAD_DIM = 128
PAGE_SIZE = 16

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpqkv.so")

_status_names = {1: "slot beyond the pool", 2: "seq_len out of range", 4: "bad scale",
                 8: "pipeline wait timed out", 16: "block-table page id out of range"}


class PqkvError(RuntimeError):
    pass


_lib = None
_lib_lock = threading.Lock()


def load_library(path: str | None = None):
    """Load libpqkv.so (built in-tree by ``python -m paged_quantized_kv_append_gb300.build``)."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise PqkvError("libpqkv.so is not built (expected at %s); run "
                            "`python -m paged_quantized_kv_append_gb300.build`" % path)
        lib = ctypes.CDLL(path)
        c_i32, c_i64, c_vp, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
        lib.pqkv_kv_append_quant.restype = ctypes.c_int
        lib.pqkv_kv_append_quant.argtypes = [c_vp, c_i64, c_vp, c_i64, c_vp, c_i32, c_i32, c_i32,
                                             c_i32, c_vp, c_vp, c_i32, c_vp, c_i64, c_i32, c_vp,
                                             c_vp]
        lib.pqkv_paged_attention_workspace_size.restype = c_sz
        lib.pqkv_paged_attention_workspace_size.argtypes = [c_i32] * 6
        lib.pqkv_paged_attention.restype = ctypes.c_int
        lib.pqkv_paged_attention.argtypes = [c_vp, c_vp, c_vp, c_i64, c_vp, c_i32, c_vp, c_i32,
                                             c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp,
                                             c_i32, c_i32, c_i32, c_vp, c_sz, c_vp, c_vp]
        lib.pqkv_paged_attention_window.restype = ctypes.c_int
        lib.pqkv_paged_attention_window.argtypes = [c_vp, c_vp, c_vp, c_i64, c_vp, c_i32, c_vp,
                                                    c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                                                    c_i32, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32,
                                                    c_vp, c_sz, c_vp, c_vp]
        lib.pqkv_paged_attention_noalloc.restype = ctypes.c_int
        lib.pqkv_paged_attention_noalloc.argtypes = [c_vp, c_vp, c_vp, c_i64, c_vp, c_i32, c_vp,
                                                     c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                                                     c_i32, c_vp, c_vp, c_i32, c_i32, c_i32, c_vp,
                                                     c_vp]
        lib.pqkv_paged_attention_partial.restype = ctypes.c_int
        lib.pqkv_paged_attention_partial.argtypes = [c_vp, c_vp, c_i64, c_vp, c_i32, c_vp, c_vp,
                                                     c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                                                     c_i32, c_vp, c_vp, c_i32, c_i32, c_i32, c_vp,
                                                     c_vp, c_vp, c_sz, c_vp, c_vp]
        lib.pqkv_lse_merge.restype = ctypes.c_int
        lib.pqkv_lse_merge.argtypes = [c_vp, c_vp, c_i32, c_i64, c_i32, c_vp, c_vp, c_vp]
        lib.pqkv_status_string.restype = ctypes.c_char_p
        lib.pqkv_status_string.argtypes = [ctypes.c_int]
        lib.pqkv_version.restype = ctypes.c_char_p
        lib.pqkv_version.argtypes = []
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = load_library().pqkv_status_string(rc).decode()
        if rc in (-1, -2, -3):
            raise ValueError("%s: %s (code %d)" % (what, msg, rc))
        raise PqkvError("%s: %s (code %d)" % (what, msg, rc))


def _stream(t: torch.Tensor, stream):
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _on_device(dev, **tensors):
    """Every tensor the kernels read or write must live on the pool's GPU: a
    host or other-device pointer would be dereferenced on the device."""
    for name, x in tensors.items():
        if x is not None and (not x.is_cuda or x.device != dev):
            raise ValueError("%s must be a CUDA tensor on %s, got %s" % (name, dev, x.device))


def _check_status(status, dev):
    if status is not None:
        _on_device(dev, status=status)
        if status.dtype != torch.int32 or status.numel() < 1:
            raise ValueError("status must be an int32 CUDA tensor of at least one element")


def _dtype_id(kv_dtype) -> int:
    if isinstance(kv_dtype, str):
        return KV_DTYPES[kv_dtype]
    return int(kv_dtype)


def _row_scale_bytes(num_pages, num_kv_heads):
    return num_pages * num_kv_heads * 2 * PAGE_SIZE * 2          # fp16 scales


def new_pages(num_pages: int, num_kv_heads: int, kv_dtype, device="cuda", fill=None):
    """Allocate a pool [num_pages, num_kv_heads, 2, 16, 128] for ``kv_dtype``.

    An INT8_ROW pool is the code tensor followed, in the same allocation, by
    its row-scale area (zeroed); ``row_scales(pages)`` views that area.
    """
    kd = _dtype_id(kv_dtype)
    dt = torch.float16 if kd == FP16 else torch.uint8
    shape = (num_pages, num_kv_heads, 2, PAGE_SIZE, HEAD_DIM)
    if kd == INT8_ROW:
        codes = num_pages * num_kv_heads * 2 * PAGE_SIZE * HEAD_DIM
        buf = torch.zeros(codes + _row_scale_bytes(num_pages, num_kv_heads), dtype=torch.uint8,
                          device=device)
        if fill is not None:
            buf[:codes].fill_(fill)
        return buf[:codes].view(shape)
    if fill is None:
        return torch.empty(shape, dtype=dt, device=device)
    return torch.full(shape, fill, dtype=dt, device=device)


def row_scales(pages: torch.Tensor) -> torch.Tensor:
    """float16 view [num_pages, Hkv, 2, 2, 8] of an INT8_ROW pool's row scales:
    ``[p, h, kv, r // 8, r % 8]`` is the scale of row r (slot 16 p + r) of K
    (kv 0) or V (kv 1).  The area stores them as [p][h][r % 8][kv][r // 8];
    ``.reshape(n, Hkv, 2, 16)`` gives a row-ordered copy."""
    _check_pages(pages, INT8_ROW)
    n, H = pages.shape[0], pages.shape[1]
    codes = pages.numel()
    whole = torch.empty(0, dtype=torch.uint8, device=pages.device)
    whole.set_(pages.untyped_storage(), pages.storage_offset(),
               (codes + _row_scale_bytes(n, H),))
    return _row_scale_view(whole[codes:], n, H)


def _row_scale_view(area: torch.Tensor, num_pages: int, num_kv_heads: int) -> torch.Tensor:
    """[p, h, kv, r // 8, r % 8] view of a scale area (uint8 bytes) stored as
    fp16 [p][h][i][4] = (K row i, K row i+8, V row i, V row i+8)."""
    return area.view(torch.float16).view(num_pages, num_kv_heads, 8, 2, 2).permute(0, 1, 3, 4, 2)


def _check_pages(pages, kd):
    want = torch.float16 if kd == FP16 else torch.uint8
    if pages.dtype != want or pages.dim() != 5 or pages.shape[2:] != (2, PAGE_SIZE, HEAD_DIM):
        raise ValueError("pages must be %s [num_pages, Hkv, 2, 16, 128], got %s %s"
                         % (want, pages.dtype, tuple(pages.shape)))
    if not pages.is_contiguous() or not pages.is_cuda:
        raise ValueError("pages must be a contiguous CUDA tensor")
    if kd == INT8_ROW:
        room = pages.untyped_storage().nbytes() - pages.storage_offset()
        if room < pages.numel() + _row_scale_bytes(pages.shape[0], pages.shape[1]):
            raise ValueError("an int8_row pool needs its row-scale area after the codes "
                             "(allocate it with new_pages)")


def _check_scale(x, H, name):
    if x.dtype != torch.float32 or not x.is_cuda or x.numel() not in (1, H):
        raise ValueError("%s must be a float32 CUDA tensor of 1 or num_kv_heads elements" % name)
    return 1 if (x.numel() == H and H > 1) else 0


def kv_append_quant(k, v, slot_mapping, kv_dtype, k_scale, v_scale, pages, status=None,
                    stream=None):
    """Quantize k, v ([T, Hkv, 128] fp16, token rows may be strided) into their
    ``slot_mapping`` slots (int64 [T], negative = skip) of ``pages``."""
    kd = _dtype_id(kv_dtype)
    _check_pages(pages, kd)
    H = pages.shape[1]
    for name, x in (("k", k), ("v", v)):
        if x.dtype != torch.float16 or x.dim() != 3 or x.shape[1:] != (H, HEAD_DIM):
            raise ValueError("%s must be fp16 [T, %d, 128], got %s %s" % (name, H, x.dtype, tuple(x.shape)))
        if x.stride(2) != 1 or x.stride(1) != HEAD_DIM or not x.is_cuda:
            raise ValueError("%s: heads and dims must be contiguous on the GPU" % name)
    T = k.shape[0]
    if v.shape[0] != T or slot_mapping.dtype != torch.int64 or slot_mapping.shape != (T,):
        raise ValueError("v / slot_mapping do not match k's token count")
    sph = 0
    if kd in _SCALED:
        sph = _check_scale(k_scale, H, "k_scale")
        if _check_scale(v_scale, H, "v_scale") != sph:
            raise ValueError("k_scale and v_scale must have the same shape")
    dev = pages.device
    _on_device(dev, k=k, v=v, slot_mapping=slot_mapping, k_scale=k_scale if kd in _SCALED else None,
               v_scale=v_scale if kd in _SCALED else None)
    _check_status(status, dev)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.pqkv_kv_append_quant(
            _ptr(k), k.stride(0), _ptr(v), v.stride(0), _ptr(slot_mapping), T, H, HEAD_DIM, kd,
            _ptr(k_scale if kd in _SCALED else None), _ptr(v_scale if kd in _SCALED else None),
            sph, _ptr(pages), pages.shape[0], PAGE_SIZE, _ptr(status), _stream(pages, stream))
    _check(rc, "kv_append_quant")
    return pages


def workspace_size(num_seqs, q_len, num_q_heads, num_kv_heads, num_splits=0) -> int:
    return int(load_library().pqkv_paged_attention_workspace_size(
        num_seqs, q_len, num_q_heads, num_kv_heads, HEAD_DIM, num_splits))


class Workspace:
    """Zero-initialised device scratch for paged_attention, grown on demand.

    The kernels leave the merge counters at its start zeroed again after every
    call, so one workspace serves any number of calls on one stream."""

    def __init__(self, device="cuda"):
        self.device = torch.device(device)
        self.buf = None

    def get(self, nbytes: int):
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws = {}


def _default_workspace(device):
    key = torch.device(device).index
    if key not in _default_ws:
        _default_ws[key] = Workspace(device)
    return _default_ws[key]


def paged_attention(q, pages, block_table, seq_lens, q_len, kv_dtype, k_scale, v_scale, out,
                    num_splits=0, max_seq_len=0, workspace=None, status=None, stream=None,
                    window=0):
    """Decode (q_len 1) or verify (q_len > 1) attention over the paged pool.

    q, out: fp16 [num_seqs * q_len, Hq, 128]; block_table: int32
    [num_seqs, max_pages_per_seq]; seq_lens: int32 [num_seqs] (cached tokens,
    the q_len new ones included).  num_splits 0 balances key pages over the
    GPU; k >= 1 cuts each (sequence, kv-head) into k partitions.  window > 0:
    query position p sees only keys p - window + 1 .. p (sliding window).
    """
    kd = _dtype_id(kv_dtype)
    _check_pages(pages, kd)
    H = pages.shape[1]
    if q.dtype != torch.float16 or q.dim() != 3 or q.shape[2] != HEAD_DIM or not q.is_contiguous():
        raise ValueError("q must be contiguous fp16 [num_seqs*q_len, Hq, 128]")
    if out.shape != q.shape or out.dtype != torch.float16 or not out.is_contiguous():
        raise ValueError("out must be contiguous fp16 shaped like q")
    B = seq_lens.shape[0]
    if seq_lens.dtype != torch.int32 or seq_lens.dim() != 1:
        raise ValueError("seq_lens must be int32 [num_seqs]")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B \
            or not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous int32 [num_seqs, max_pages_per_seq]")
    if q.shape[0] != B * q_len:
        raise ValueError("q has %d rows, expected num_seqs*q_len = %d" % (q.shape[0], B * q_len))
    Hq = q.shape[1]
    sph = 0
    if kd in _SCALED:
        sph = _check_scale(k_scale, H, "k_scale")
        if _check_scale(v_scale, H, "v_scale") != sph:
            raise ValueError("k_scale and v_scale must have the same shape")
    dev = pages.device
    _on_device(dev, q=q, out=out, block_table=block_table, seq_lens=seq_lens,
               k_scale=k_scale if kd in _SCALED else None,
               v_scale=v_scale if kd in _SCALED else None)
    _check_status(status, dev)
    need = workspace_size(B, q_len, Hq, H, num_splits)
    if workspace is None:
        workspace = _default_workspace(dev)
    ws = workspace.get(need) if isinstance(workspace, Workspace) else workspace
    _on_device(dev, workspace=ws)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    lib = load_library()
    if window < 0:
        raise ValueError("window must be >= 0")
    with torch.cuda.device(dev):
        if window > 0:
            rc = lib.pqkv_paged_attention_window(
                _ptr(q), _ptr(out), _ptr(pages), pages.shape[0], _ptr(block_table),
                block_table.shape[1], _ptr(seq_lens), B, q_len, Hq, H, HEAD_DIM, PAGE_SIZE, kd,
                _ptr(k_scale if kd in _SCALED else None), _ptr(v_scale if kd in _SCALED else None),
                sph, num_splits, max_seq_len, window, _ptr(ws), ws_bytes, _ptr(status),
                _stream(q, stream))
        else:
            rc = lib.pqkv_paged_attention(
                _ptr(q), _ptr(out), _ptr(pages), pages.shape[0], _ptr(block_table),
                block_table.shape[1], _ptr(seq_lens), B, q_len, Hq, H, HEAD_DIM, PAGE_SIZE, kd,
                _ptr(k_scale if kd in _SCALED else None), _ptr(v_scale if kd in _SCALED else None),
                sph, num_splits, max_seq_len, _ptr(ws), ws_bytes, _ptr(status), _stream(q, stream))
    _check(rc, "paged_attention")
    return out


def paged_attention_partial(q, pages, block_table, seq_lens, q_pos, q_len, kv_dtype, k_scale,
                            v_scale, out_o, out_lse, num_splits=0, max_seq_len=0, workspace=None,
                            status=None, stream=None):
    """One rank's share of a decode-context-parallel split: attention over the
    keys held here (``seq_lens`` of them per sequence, possibly 0), query i of
    sequence s seeing local keys j <= q_pos[s] + i.  Writes O / l into
    ``out_o`` (fp32, shaped like q) and the natural-log LSE into ``out_lse``
    (fp32 [num_seqs * q_len, Hq]); merge the ranks' results with lse_merge."""
    kd = _dtype_id(kv_dtype)
    _check_pages(pages, kd)
    H = pages.shape[1]
    if q.dtype != torch.float16 or q.dim() != 3 or q.shape[2] != HEAD_DIM or not q.is_contiguous():
        raise ValueError("q must be contiguous fp16 [num_seqs*q_len, Hq, 128]")
    if out_o.shape != q.shape or out_o.dtype != torch.float32 or not out_o.is_contiguous():
        raise ValueError("out_o must be contiguous fp32 shaped like q")
    if out_lse.shape != q.shape[:2] or out_lse.dtype != torch.float32 or not out_lse.is_contiguous():
        raise ValueError("out_lse must be contiguous fp32 [num_seqs*q_len, Hq]")
    B = seq_lens.shape[0]
    for name, x in (("seq_lens", seq_lens), ("q_pos", q_pos)):
        if x.dtype != torch.int32 or x.shape != (B,):
            raise ValueError("%s must be int32 [num_seqs]" % name)
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B \
            or not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous int32 [num_seqs, max_pages_per_seq]")
    if q.shape[0] != B * q_len:
        raise ValueError("q has %d rows, expected num_seqs*q_len = %d" % (q.shape[0], B * q_len))
    Hq = q.shape[1]
    sph = 0
    if kd in _SCALED:
        sph = _check_scale(k_scale, H, "k_scale")
        if _check_scale(v_scale, H, "v_scale") != sph:
            raise ValueError("k_scale and v_scale must have the same shape")
    dev = pages.device
    _on_device(dev, q=q, out_o=out_o, out_lse=out_lse, block_table=block_table,
               seq_lens=seq_lens, q_pos=q_pos, k_scale=k_scale if kd in _SCALED else None,
               v_scale=v_scale if kd in _SCALED else None)
    _check_status(status, dev)
    need = workspace_size(B, q_len, Hq, H, num_splits)
    if workspace is None:
        workspace = _default_workspace(dev)
    ws = workspace.get(need) if isinstance(workspace, Workspace) else workspace
    _on_device(dev, workspace=ws)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.pqkv_paged_attention_partial(
            _ptr(q), _ptr(pages), pages.shape[0], _ptr(block_table), block_table.shape[1],
            _ptr(seq_lens), _ptr(q_pos), B, q_len, Hq, H, HEAD_DIM, PAGE_SIZE, kd,
            _ptr(k_scale if kd in _SCALED else None), _ptr(v_scale if kd in _SCALED else None),
            sph, num_splits, max_seq_len, _ptr(out_o), _ptr(out_lse), _ptr(ws), ws_bytes,
            _ptr(status), _stream(q, stream))
    _check(rc, "paged_attention_partial")
    return out_o, out_lse


def lse_merge(parts_o, parts_lse, out, out_lse=None, stream=None):
    """Combine partial results: parts_o fp32 [P, rows..., 128], parts_lse fp32
    [P, rows...] -> out fp16 [rows..., 128] (and the merged LSE if given)."""
    P = parts_o.shape[0]
    rows = parts_lse[0].numel()
    if parts_o.dtype != torch.float32 or not parts_o.is_contiguous() or \
            parts_o.numel() != P * rows * HEAD_DIM:
        raise ValueError("parts_o must be contiguous fp32 [P, rows..., 128]")
    if parts_lse.dtype != torch.float32 or not parts_lse.is_contiguous() or parts_lse.shape[0] != P:
        raise ValueError("parts_lse must be contiguous fp32 [P, rows...]")
    if out.dtype != torch.float16 or not out.is_contiguous() or out.numel() != rows * HEAD_DIM:
        raise ValueError("out must be contiguous fp16 with rows * 128 elements")
    if out_lse is not None and (out_lse.dtype != torch.float32 or out_lse.numel() != rows):
        raise ValueError("out_lse must be fp32 with one value per row")
    dev = out.device
    _on_device(dev, parts_o=parts_o, parts_lse=parts_lse, out=out, out_lse=out_lse)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.pqkv_lse_merge(_ptr(parts_o), _ptr(parts_lse), P, rows, HEAD_DIM, _ptr(out),
                                _ptr(out_lse), _stream(out, stream))
    _check(rc, "lse_merge")
    return out


NOALLOC_SCRATCH_BYTES = 16 << 20


def paged_attention_noalloc(q, pages, block_table, seq_lens, q_len, kv_dtype, k_scale, v_scale,
                            out, num_splits=0, max_seq_len=0, status=None, stream=None):
    """paged_attention for callers that cannot allocate device memory: the
    library uses its own fixed 16 MiB scratch area instead of a workspace.

    The first call on a device must come before any stream capture; calls on
    one device share the scratch area and must not overlap on the GPU.
    Raises ValueError when the launch this call makes needs more scratch than
    the area holds (include/pqkv.h states the sizes).
    """
    kd = _dtype_id(kv_dtype)
    _check_pages(pages, kd)
    H = pages.shape[1]
    if q.dtype != torch.float16 or q.dim() != 3 or q.shape[2] != HEAD_DIM or not q.is_contiguous():
        raise ValueError("q must be contiguous fp16 [num_seqs*q_len, Hq, 128]")
    if out.shape != q.shape or out.dtype != torch.float16 or not out.is_contiguous():
        raise ValueError("out must be contiguous fp16 shaped like q")
    B = seq_lens.shape[0]
    if seq_lens.dtype != torch.int32 or seq_lens.dim() != 1:
        raise ValueError("seq_lens must be int32 [num_seqs]")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B \
            or not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous int32 [num_seqs, max_pages_per_seq]")
    if q.shape[0] != B * q_len:
        raise ValueError("q has %d rows, expected num_seqs*q_len = %d" % (q.shape[0], B * q_len))
    sph = 0
    if kd in _SCALED:
        sph = _check_scale(k_scale, H, "k_scale")
        if _check_scale(v_scale, H, "v_scale") != sph:
            raise ValueError("k_scale and v_scale must have the same shape")
    dev = pages.device
    _on_device(dev, q=q, out=out, block_table=block_table, seq_lens=seq_lens,
               k_scale=k_scale if kd in _SCALED else None,
               v_scale=v_scale if kd in _SCALED else None)
    _check_status(status, dev)
    lib = load_library()
    with torch.cuda.device(dev):
        rc = lib.pqkv_paged_attention_noalloc(
            _ptr(q), _ptr(out), _ptr(pages), pages.shape[0], _ptr(block_table),
            block_table.shape[1], _ptr(seq_lens), B, q_len, q.shape[1], H, HEAD_DIM, PAGE_SIZE,
            kd, _ptr(k_scale if kd in _SCALED else None),
            _ptr(v_scale if kd in _SCALED else None), sph, num_splits, max_seq_len, _ptr(status),
            _stream(q, stream))
    _check(rc, "paged_attention_noalloc")
    return out


def status_bits(status: torch.Tensor):
    """Names of the device status bits set in an int32 status tensor (syncs)."""
    v = int(status.item())
    return [name for bit, name in _status_names.items() if v & bit]


def version() -> str:
    return load_library().pqkv_version().decode()
