"""Python binding of libmla_paged.so: paged Multi-head Latent Attention on GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels, called through its C ABI (include/mla_paged.h).  There is no CPU path: if the
library is missing or the tensors are not on a CUDA device, the calls raise.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import _build

HEAD_DIM_CKV = 512
HEAD_DIM_KPE = 64
MLA_VALIDATE = 1

_STATUS = {0: "MLA_OK", -1: "MLA_ERR_NULL", -2: "MLA_ERR_DIMS", -3: "MLA_ERR_ALIGN",
           -4: "MLA_ERR_WORKSPACE", -5: "MLA_ERR_LAUNCH", -6: "MLA_ERR_BAD_INDEX",
           -7: "MLA_ERR_TIMEOUT", -8: "MLA_ERR_CUDA", -9: "MLA_ERR_UNSUPPORTED", -10: "MLA_ERR_INTERNAL"}


class MlaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {string_of(status)} ({status})")


class MlaDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_qo_heads", ctypes.c_int32),
                ("head_dim_ckv", ctypes.c_int32), ("head_dim_kpe", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("total_q", ctypes.c_int32), ("num_kv_indices", ctypes.c_int32),
                ("num_workers", ctypes.c_int32)]


_lib = None

# (name, restype, argtypes) of every symbol declared in include/mla_paged.h
_P = ctypes.c_void_p
_SIGNATURES = [
    ("mla_paged_decode", ctypes.c_int,
     [_P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, ctypes.POINTER(MlaDims), _P, ctypes.c_size_t,
      ctypes.c_int, _P]),
    ("mla_paged_prefill", ctypes.c_int,
     [_P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, ctypes.POINTER(MlaDims), _P, ctypes.c_size_t,
      ctypes.c_int, _P]),
    ("mla_paged_decode_mtp", ctypes.c_int,
     [_P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, ctypes.POINTER(MlaDims), ctypes.c_int, _P,
      ctypes.c_size_t, ctypes.c_int, _P]),
    ("mla_paged_decode_sparse", ctypes.c_int,
     [_P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_float, _P, _P, ctypes.POINTER(MlaDims), _P, ctypes.c_size_t,
      ctypes.c_int, _P]),
    ("mla_paged_decode_fp8", ctypes.c_int,
     [_P, _P, _P, _P, _P, ctypes.c_float, _P, _P, ctypes.POINTER(MlaDims), _P, ctypes.c_size_t, ctypes.c_int, _P]),
    ("mla_paged_decode_sparse_fp8", ctypes.c_int,
     [_P, _P, _P, _P, ctypes.c_int, ctypes.c_float, _P, _P, ctypes.POINTER(MlaDims), _P, ctypes.c_size_t,
      ctypes.c_int, _P]),
    ("mla_block_table_to_csr", ctypes.c_int,
     [_P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_longlong, _P]),
    ("mla_workspace_bytes_block_table", ctypes.c_size_t, [ctypes.POINTER(MlaDims), ctypes.c_int]),
    ("mla_paged_decode_block_table", ctypes.c_int,
     [_P, _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_float, _P, _P, ctypes.POINTER(MlaDims), _P, ctypes.c_size_t,
      ctypes.c_int, _P]),
    ("mla_paged_decode_noalloc", ctypes.c_int,
     [_P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, ctypes.POINTER(MlaDims), ctypes.c_int, _P]),
    ("mla_workspace_bytes", ctypes.c_size_t, [ctypes.POINTER(MlaDims), ctypes.c_int]),
    ("mla_workspace_bytes_mtp", ctypes.c_size_t, [ctypes.POINTER(MlaDims), ctypes.c_int]),
    ("mla_default_num_workers", ctypes.c_int, []),
    ("mla_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("mla_read_device_status", ctypes.c_int, [_P, _P]),
    ("mla_noalloc_read_status", ctypes.c_int, [_P]),
    ("mla_debug_inject_timeout", ctypes.c_int, [ctypes.c_int, ctypes.c_ulonglong]),
    ("mla_profile_enable", ctypes.c_int, [ctypes.c_int]),
    ("mla_profile_read", ctypes.c_int, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_int)]),
]


def library_path() -> str:
    return _build.LIB


def lib():
    """Load the library (it must have been built: ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (python -m paged_head_latent_gb300._build)")
        l = ctypes.CDLL(path)
        for name, res, args in _SIGNATURES:
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def string_of(status: int) -> str:
    try:
        return lib().mla_status_string(status).decode()
    except Exception:
        return _STATUS.get(status, "unknown")


def make_dims(batch, num_qo_heads, num_pages, page_size, num_kv_indices, total_q=0, num_workers=0):
    return MlaDims(batch, num_qo_heads, HEAD_DIM_CKV, HEAD_DIM_KPE, num_pages, page_size, total_q,
                   num_kv_indices, num_workers)


def workspace_bytes(dims: MlaDims, is_prefill: bool) -> int:
    return int(lib().mla_workspace_bytes(ctypes.byref(dims), 1 if is_prefill else 0))


def workspace_bytes_mtp(dims: MlaDims, q_len: int) -> int:
    return int(lib().mla_workspace_bytes_mtp(ctypes.byref(dims), int(q_len)))


def workload_dims(w, num_workers=0) -> MlaDims:
    """The dims of a call on a ``workloads.Workload`` (decode, prefill or mtp)."""
    return make_dims(w.batch, w.num_qo_heads, w.num_pages, w.page_size, w.num_kv_indices,
                     total_q=w.rows if w.kind == "prefill" else 0, num_workers=num_workers)


def workload_workspace_bytes(w, num_workers=0) -> int:
    """Workspace bytes a call on ``w`` needs."""
    dims = workload_dims(w, num_workers)
    if w.kind == "mtp":
        return workspace_bytes_mtp(dims, w.mtp_q_len)
    return workspace_bytes(dims, w.kind == "prefill")


def default_num_workers() -> int:
    n = lib().mla_default_num_workers()
    if n < 0:
        raise MlaError(n, "mla_default_num_workers")
    return n


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_cuda(name, t, dtype):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _cache_geometry(ckv_cache, kpe_cache):
    if ckv_cache.dim() != 3 or ckv_cache.shape[-1] != HEAD_DIM_CKV:
        raise ValueError("ckv_cache must be [num_pages, page_size, 512]")
    if kpe_cache.shape != (ckv_cache.shape[0], ckv_cache.shape[1], HEAD_DIM_KPE):
        raise ValueError("kpe_cache must be [num_pages, page_size, 64] matching ckv_cache")
    return ckv_cache.shape[0], ckv_cache.shape[1]


def _call(prefill, q_nope, q_pe, ckv_cache, kpe_cache, qo_indptr, kv_indptr, kv_indices, sm_scale,
          out, lse, workspace, flags, num_workers, stream):
    for n, t in (("q_nope", q_nope), ("q_pe", q_pe), ("ckv_cache", ckv_cache), ("kpe_cache", kpe_cache)):
        _check_cuda(n, t, torch.bfloat16)
    for n, t in (("kv_indptr", kv_indptr), ("kv_indices", kv_indices)) + (
            (("qo_indptr", qo_indptr),) if prefill else ()):
        _check_cuda(n, t, torch.int32)
    rows, heads = q_nope.shape[0], q_nope.shape[1]
    if q_nope.shape != (rows, heads, HEAD_DIM_CKV) or q_pe.shape != (rows, heads, HEAD_DIM_KPE):
        raise ValueError("q_nope must be [rows, H, 512] and q_pe [rows, H, 64]")
    num_pages, page_size = _cache_geometry(ckv_cache, kpe_cache)
    batch = kv_indptr.numel() - 1
    if prefill and qo_indptr.numel() != batch + 1:
        raise ValueError("qo_indptr and kv_indptr must both have batch + 1 entries")
    if not prefill and rows != batch:
        raise ValueError("decode: q_nope.shape[0] must equal len(kv_indptr) - 1")
    dims = make_dims(batch, heads, num_pages, page_size, kv_indices.numel(),
                     total_q=rows if prefill else 0, num_workers=num_workers)
    dev = q_nope.device
    if out is None:
        out = torch.empty(rows, heads, HEAD_DIM_CKV, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(rows, heads, dtype=torch.float32, device=dev)
    _check_cuda("out", out, torch.bfloat16)
    _check_cuda("lse", lse, torch.float32)
    if out.shape != (rows, heads, HEAD_DIM_CKV) or lse.shape != (rows, heads):
        raise ValueError("out must be [rows, H, 512] and lse [rows, H]")
    need = workspace_bytes(dims, prefill)
    if need == 0:
        raise MlaError(-2, "mla_workspace_bytes")
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    with torch.cuda.device(dev):
        if prefill:
            st = lib().mla_paged_prefill(_ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(kpe_cache),
                                         _ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices),
                                         float(sm_scale), _ptr(out), _ptr(lse), ctypes.byref(dims),
                                         _ptr(workspace), workspace.numel(), int(flags), sp)
        else:
            st = lib().mla_paged_decode(_ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(kpe_cache),
                                        _ptr(kv_indptr), _ptr(kv_indices), float(sm_scale), _ptr(out),
                                        _ptr(lse), ctypes.byref(dims), _ptr(workspace), workspace.numel(),
                                        int(flags), sp)
    if st != 0:
        raise MlaError(st, "mla_paged_prefill" if prefill else "mla_paged_decode")
    return out, lse


def mla_paged_decode(q_nope, q_pe, ckv_cache, kpe_cache, kv_indptr, kv_indices, sm_scale,
                     out=None, lse=None, workspace=None, flags=0, num_workers=0,
                     stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Paged MLA decode (flashinfer-bench "MLA Paged", section "decode").  Returns (out, lse)."""
    return _call(False, q_nope, q_pe, ckv_cache, kpe_cache, None, kv_indptr, kv_indices, sm_scale,
                 out, lse, workspace, flags, num_workers, stream)


def mla_paged_prefill(q_nope, q_pe, ckv_cache, kpe_cache, qo_indptr, kv_indptr, kv_indices, sm_scale,
                      out=None, lse=None, workspace=None, flags=0, num_workers=0,
                      stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Paged MLA causal prefill, bottom-right aligned ("MLA Paged", section "prefill")."""
    return _call(True, q_nope, q_pe, ckv_cache, kpe_cache, qo_indptr, kv_indptr, kv_indices, sm_scale,
                 out, lse, workspace, flags, num_workers, stream)


def mla_paged_decode_mtp(q_nope, q_pe, ckv_cache, kpe_cache, kv_indptr, kv_indices, sm_scale,
                         out=None, lse=None, workspace=None, flags=0, num_workers=0,
                         stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Packed multi-token decode: q_nope [batch, q_len, H, 512], q_pe [batch, q_len, H, 64];
    token i of a request sees its first kv_len - q_len + i + 1 keys.  Returns (out
    [batch, q_len, H, 512], lse [batch, q_len, H]).  q_len * H must be <= 128."""
    for n, t in (("q_nope", q_nope), ("q_pe", q_pe), ("ckv_cache", ckv_cache), ("kpe_cache", kpe_cache)):
        _check_cuda(n, t, torch.bfloat16)
    for n, t in (("kv_indptr", kv_indptr), ("kv_indices", kv_indices)):
        _check_cuda(n, t, torch.int32)
    if q_nope.dim() != 4 or q_nope.shape[-1] != HEAD_DIM_CKV:
        raise ValueError("q_nope must be [batch, q_len, H, 512]")
    batch, q_len, heads = q_nope.shape[0], q_nope.shape[1], q_nope.shape[2]
    if q_pe.shape != (batch, q_len, heads, HEAD_DIM_KPE):
        raise ValueError("q_pe must be [batch, q_len, H, 64]")
    if kv_indptr.numel() - 1 != batch:
        raise ValueError("kv_indptr must have batch + 1 entries")
    num_pages, page_size = _cache_geometry(ckv_cache, kpe_cache)
    dims = make_dims(batch, heads, num_pages, page_size, kv_indices.numel(), num_workers=num_workers)
    dev = q_nope.device
    if out is None:
        out = torch.empty(batch, q_len, heads, HEAD_DIM_CKV, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(batch, q_len, heads, dtype=torch.float32, device=dev)
    _check_cuda("out", out, torch.bfloat16)
    _check_cuda("lse", lse, torch.float32)
    if out.shape != (batch, q_len, heads, HEAD_DIM_CKV) or lse.shape != (batch, q_len, heads):
        raise ValueError("out must be [batch, q_len, H, 512] and lse [batch, q_len, H]")
    need = workspace_bytes_mtp(dims, q_len)
    if need == 0:
        raise MlaError(-2, "mla_workspace_bytes_mtp")
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = lib().mla_paged_decode_mtp(_ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(kpe_cache),
                                        _ptr(kv_indptr), _ptr(kv_indices), float(sm_scale), _ptr(out),
                                        _ptr(lse), ctypes.byref(dims), int(q_len), _ptr(workspace),
                                        workspace.numel(), int(flags), ctypes.c_void_p(stream.cuda_stream))
    if st != 0:
        raise MlaError(st, "mla_paged_decode_mtp")
    return out, lse


def mla_paged_decode_sparse(q_nope, q_pe, ckv_cache, kpe_cache, indices, sm_scale, out=None, lse=None,
                            workspace=None, flags=0, num_workers=0,
                            stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Sparse (top-k) decode: row r of q attends to the token slots indices[r, :]
    (entries outside the cache are padding).  q_nope [rows, H, 512], q_pe [rows, H, 64],
    indices [rows, topk] int32.  Returns (out [rows, H, 512], lse [rows, H])."""
    for n, t in (("q_nope", q_nope), ("q_pe", q_pe), ("ckv_cache", ckv_cache), ("kpe_cache", kpe_cache)):
        _check_cuda(n, t, torch.bfloat16)
    _check_cuda("indices", indices, torch.int32)
    rows, heads = q_nope.shape[0], q_nope.shape[1]
    if q_nope.shape != (rows, heads, HEAD_DIM_CKV) or q_pe.shape != (rows, heads, HEAD_DIM_KPE):
        raise ValueError("q_nope must be [rows, H, 512] and q_pe [rows, H, 64]")
    if indices.dim() != 2 or indices.shape[0] != rows:
        raise ValueError("indices must be [rows, topk]")
    topk = indices.shape[1]
    num_pages, page_size = _cache_geometry(ckv_cache, kpe_cache)
    dims = make_dims(rows, heads, num_pages, page_size, rows * topk, num_workers=num_workers)
    dev = q_nope.device
    if out is None:
        out = torch.empty(rows, heads, HEAD_DIM_CKV, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(rows, heads, dtype=torch.float32, device=dev)
    _check_cuda("out", out, torch.bfloat16)
    _check_cuda("lse", lse, torch.float32)
    if out.shape != (rows, heads, HEAD_DIM_CKV) or lse.shape != (rows, heads):
        raise ValueError("out must be [rows, H, 512] and lse [rows, H]")
    need = workspace_bytes(dims, False)
    if need == 0:
        raise MlaError(-2, "mla_workspace_bytes")
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = lib().mla_paged_decode_sparse(_ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(kpe_cache),
                                           _ptr(indices), int(topk), float(sm_scale), _ptr(out), _ptr(lse),
                                           ctypes.byref(dims), _ptr(workspace), workspace.numel(), int(flags),
                                           ctypes.c_void_p(stream.cuda_stream))
    if st != 0:
        raise MlaError(st, "mla_paged_decode_sparse")
    return out, lse


FP8_TOKEN_BYTES = 656


def _fp8_call(name, q_nope, q_pe, kv_fp8, kv_indptr, kv_indices, topk, sm_scale, out, lse, workspace, flags,
              num_workers, stream):
    for n, t in (("q_nope", q_nope), ("q_pe", q_pe)):
        _check_cuda(n, t, torch.bfloat16)
    _check_cuda("kv_fp8", kv_fp8, torch.uint8)
    _check_cuda("kv_indices", kv_indices, torch.int32)
    if kv_fp8.dim() != 3 or kv_fp8.shape[2] != FP8_TOKEN_BYTES:
        raise ValueError("kv_fp8 must be [num_pages, page_size, 656] uint8")
    rows, heads = q_nope.shape[0], q_nope.shape[1]
    if q_nope.shape != (rows, heads, HEAD_DIM_CKV) or q_pe.shape != (rows, heads, HEAD_DIM_KPE):
        raise ValueError("q_nope must be [rows, H, 512] and q_pe [rows, H, 64]")
    num_pages, page_size = kv_fp8.shape[0], kv_fp8.shape[1]
    if topk:
        if kv_indices.shape != (rows, topk):
            raise ValueError("indices must be [rows, topk]")
        n_idx = rows * topk
    else:
        _check_cuda("kv_indptr", kv_indptr, torch.int32)
        if kv_indptr.numel() != rows + 1:
            raise ValueError("decode: q_nope.shape[0] must equal len(kv_indptr) - 1")
        n_idx = kv_indices.numel()
    dims = make_dims(rows, heads, num_pages, page_size, n_idx, num_workers=num_workers)
    dev = q_nope.device
    if out is None:
        out = torch.empty(rows, heads, HEAD_DIM_CKV, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(rows, heads, dtype=torch.float32, device=dev)
    _check_cuda("out", out, torch.bfloat16)
    _check_cuda("lse", lse, torch.float32)
    if out.shape != (rows, heads, HEAD_DIM_CKV) or lse.shape != (rows, heads):
        raise ValueError("out must be [rows, H, 512] and lse [rows, H]")
    need = workspace_bytes(dims, False)
    if need == 0:
        raise MlaError(-2, "mla_workspace_bytes")
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    with torch.cuda.device(dev):
        if topk:
            st = lib().mla_paged_decode_sparse_fp8(_ptr(q_nope), _ptr(q_pe), _ptr(kv_fp8), _ptr(kv_indices),
                                                   int(topk), float(sm_scale), _ptr(out), _ptr(lse),
                                                   ctypes.byref(dims), _ptr(workspace), workspace.numel(),
                                                   int(flags), sp)
        else:
            st = lib().mla_paged_decode_fp8(_ptr(q_nope), _ptr(q_pe), _ptr(kv_fp8), _ptr(kv_indptr),
                                            _ptr(kv_indices), float(sm_scale), _ptr(out), _ptr(lse),
                                            ctypes.byref(dims), _ptr(workspace), workspace.numel(), int(flags), sp)
    if st != 0:
        raise MlaError(st, name)
    return out, lse


def mla_paged_decode_fp8(q_nope, q_pe, kv_fp8, kv_indptr, kv_indices, sm_scale, out=None, lse=None,
                         workspace=None, flags=0, num_workers=0, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Paged MLA decode over an FP8 cache kv_fp8 [num_pages, page_size, 656] uint8 (512
    E4M3 latent values, 4 float32 scales, 64 bf16 rope values per token)."""
    return _fp8_call("mla_paged_decode_fp8", q_nope, q_pe, kv_fp8, kv_indptr, kv_indices, 0, sm_scale, out, lse,
                     workspace, flags, num_workers, stream)


def mla_paged_decode_sparse_fp8(q_nope, q_pe, kv_fp8, indices, sm_scale, out=None, lse=None, workspace=None,
                                flags=0, num_workers=0, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Sparse (top-k) decode over an FP8 cache: indices [rows, topk] int32 token slots."""
    return _fp8_call("mla_paged_decode_sparse_fp8", q_nope, q_pe, kv_fp8, None, indices, indices.shape[1],
                     sm_scale, out, lse, workspace, flags, num_workers, stream)


def block_table_to_csr(block_table, seq_lens, page_size, capacity=None, stream=None):
    """Token-slot CSR (kv_indptr [batch + 1], kv_indices [capacity]) of a block table
    [batch, max_blocks] and seq_lens [batch] (int32, on the GPU): request b's keys are the
    first seq_lens[b] slots of its pages in table order.  capacity defaults to
    batch * max_blocks * page_size; entries past the total are left unset."""
    _check_cuda("block_table", block_table, torch.int32)
    _check_cuda("seq_lens", seq_lens, torch.int32)
    if block_table.dim() != 2 or seq_lens.shape != (block_table.shape[0],):
        raise ValueError("block_table must be [batch, max_blocks] and seq_lens [batch]")
    batch, max_blocks = block_table.shape
    if capacity is None:
        capacity = batch * max_blocks * page_size
    dev = block_table.device
    kv_indptr = torch.empty(batch + 1, dtype=torch.int32, device=dev)
    kv_indices = torch.empty(max(int(capacity), 1), dtype=torch.int32, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = lib().mla_block_table_to_csr(_ptr(block_table), _ptr(seq_lens), int(batch), int(max_blocks),
                                          int(page_size), _ptr(kv_indptr), _ptr(kv_indices), int(capacity),
                                          ctypes.c_void_p(stream.cuda_stream))
    if st != 0:
        raise MlaError(st, "mla_block_table_to_csr")
    return kv_indptr, kv_indices[:int(capacity)]


def mla_paged_decode_block_table(q_nope, q_pe, ckv_cache, kpe_cache, block_table, seq_lens, sm_scale, out=None,
                                 lse=None, workspace=None, num_workers=0,
                                 stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Paged MLA decode from a block table [batch, max_blocks] and seq_lens [batch]
    (int32): the conversion to the token-slot CSR and the decode in one call.
    Returns (out [batch, H, 512], lse [batch, H])."""
    for n, t in (("q_nope", q_nope), ("q_pe", q_pe), ("ckv_cache", ckv_cache), ("kpe_cache", kpe_cache)):
        _check_cuda(n, t, torch.bfloat16)
    _check_cuda("block_table", block_table, torch.int32)
    _check_cuda("seq_lens", seq_lens, torch.int32)
    batch, heads = q_nope.shape[0], q_nope.shape[1]
    if q_nope.shape != (batch, heads, HEAD_DIM_CKV) or q_pe.shape != (batch, heads, HEAD_DIM_KPE):
        raise ValueError("q_nope must be [batch, H, 512] and q_pe [batch, H, 64]")
    if block_table.dim() != 2 or block_table.shape[0] != batch or seq_lens.shape != (batch,):
        raise ValueError("block_table must be [batch, max_blocks] and seq_lens [batch]")
    max_blocks = block_table.shape[1]
    num_pages, page_size = _cache_geometry(ckv_cache, kpe_cache)
    dims = make_dims(batch, heads, num_pages, page_size, 0, num_workers=num_workers)
    dev = q_nope.device
    if out is None:
        out = torch.empty(batch, heads, HEAD_DIM_CKV, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(batch, heads, dtype=torch.float32, device=dev)
    _check_cuda("out", out, torch.bfloat16)
    _check_cuda("lse", lse, torch.float32)
    if out.shape != (batch, heads, HEAD_DIM_CKV) or lse.shape != (batch, heads):
        raise ValueError("out must be [batch, H, 512] and lse [batch, H]")
    need = lib().mla_workspace_bytes_block_table(ctypes.byref(dims), int(max_blocks))
    if need == 0:
        raise MlaError(-2, "mla_workspace_bytes_block_table")
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = lib().mla_paged_decode_block_table(_ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(kpe_cache),
                                                _ptr(block_table), _ptr(seq_lens), int(max_blocks),
                                                float(sm_scale), _ptr(out), _ptr(lse), ctypes.byref(dims),
                                                _ptr(workspace), workspace.numel(), 0,
                                                ctypes.c_void_p(stream.cuda_stream))
    if st != 0:
        raise MlaError(st, "mla_paged_decode_block_table")
    return out, lse


def mla_paged_decode_noalloc(q_nope, q_pe, ckv_cache, kpe_cache, kv_indptr, kv_indices, sm_scale,
                             out, lse, num_workers=0, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Paged MLA decode without a workspace argument, for callers that cannot allocate
    device memory: the library's own static 32 MiB device scratch holds the split-KV
    partials.  ``out`` and ``lse`` must be given (nothing is allocated here either).
    Calls that overlap on the GPU race on the shared scratch."""
    for n, t in (("q_nope", q_nope), ("q_pe", q_pe), ("ckv_cache", ckv_cache), ("kpe_cache", kpe_cache),
                 ("out", out)):
        _check_cuda(n, t, torch.bfloat16)
    for n, t in (("kv_indptr", kv_indptr), ("kv_indices", kv_indices)):
        _check_cuda(n, t, torch.int32)
    _check_cuda("lse", lse, torch.float32)
    rows, heads = q_nope.shape[0], q_nope.shape[1]
    num_pages, page_size = _cache_geometry(ckv_cache, kpe_cache)
    if kv_indptr.numel() - 1 != rows or out.shape != (rows, heads, HEAD_DIM_CKV) or lse.shape != (rows, heads):
        raise ValueError("shape mismatch between q_nope, kv_indptr, out and lse")
    dims = make_dims(rows, heads, num_pages, page_size, kv_indices.numel(), num_workers=num_workers)
    if stream is None:
        stream = torch.cuda.current_stream(q_nope.device)
    with torch.cuda.device(q_nope.device):
        st = lib().mla_paged_decode_noalloc(_ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(kpe_cache),
                                            _ptr(kv_indptr), _ptr(kv_indices), float(sm_scale), _ptr(out),
                                            _ptr(lse), ctypes.byref(dims), 0, ctypes.c_void_p(stream.cuda_stream))
    if st != 0:
        raise MlaError(st, "mla_paged_decode_noalloc")
    return out, lse


def noalloc_read_status(device=None, stream=None) -> int:
    """Synchronise, read and clear the status word of the most recent
    ``mla_paged_decode_noalloc`` call on ``device``."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        return int(lib().mla_noalloc_read_status(ctypes.c_void_p(stream.cuda_stream)))


def read_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise, read and clear the device status word in ``workspace``."""
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    return int(lib().mla_read_device_status(_ptr(workspace), ctypes.c_void_p(stream.cuda_stream)))


def profile_enable(on: bool = True) -> None:
    lib().mla_profile_enable(1 if on else 0)


def profile_read():
    """(main-kernel ms, combine ms, timed calls) since the last read."""
    a, b, n = ctypes.c_double(), ctypes.c_double(), ctypes.c_int()
    st = lib().mla_profile_read(ctypes.byref(a), ctypes.byref(b), ctypes.byref(n))
    if st != 0:
        raise MlaError(st, "mla_profile_read")
    return a.value, b.value, n.value


def bind_workload(w, out, lse, workspace, stream, flags=0, num_workers=0):
    """Check and marshal the arguments of one decode or prefill call on a
    ``workloads.Workload`` once, and return a function of no arguments that makes exactly
    that C-ABI call again (for loops that repeat a call, such as a benchmark's timed
    region, where the per-call argument checks would otherwise cost host time)."""
    prefill = w.kind == "prefill"
    run_workload(w, out=out, lse=lse, workspace=workspace, flags=flags, num_workers=num_workers,
                 stream=stream)  # validates everything once
    dims = workload_dims(w, num_workers)
    sp = ctypes.c_void_p(stream.cuda_stream)
    name = {"decode": "mla_paged_decode", "prefill": "mla_paged_prefill", "mtp": "mla_paged_decode_mtp",
            "sparse": "mla_paged_decode_sparse", "decode_fp8": "mla_paged_decode_fp8",
            "sparse_fp8": "mla_paged_decode_sparse_fp8"}[w.kind]
    if w.kind == "decode_fp8":
        fn = lib().mla_paged_decode_fp8
        args = (_ptr(w.q_nope), _ptr(w.q_pe), _ptr(w.kv_fp8), _ptr(w.kv_indptr), _ptr(w.kv_indices),
                float(w.sm_scale), _ptr(out), _ptr(lse), ctypes.byref(dims), _ptr(workspace), workspace.numel(),
                int(flags), sp)
    elif w.kind == "sparse_fp8":
        fn = lib().mla_paged_decode_sparse_fp8
        args = (_ptr(w.q_nope), _ptr(w.q_pe), _ptr(w.kv_fp8), _ptr(w.indices), int(w.topk), float(w.sm_scale),
                _ptr(out), _ptr(lse), ctypes.byref(dims), _ptr(workspace), workspace.numel(), int(flags), sp)
    elif w.kind == "sparse":
        fn = lib().mla_paged_decode_sparse
        args = (_ptr(w.q_nope), _ptr(w.q_pe), _ptr(w.ckv_cache), _ptr(w.kpe_cache), _ptr(w.indices),
                int(w.topk), float(w.sm_scale), _ptr(out), _ptr(lse), ctypes.byref(dims), _ptr(workspace),
                workspace.numel(), int(flags), sp)
    elif w.kind == "mtp":
        fn = lib().mla_paged_decode_mtp
        args = (_ptr(w.q_nope), _ptr(w.q_pe), _ptr(w.ckv_cache), _ptr(w.kpe_cache), _ptr(w.kv_indptr),
                _ptr(w.kv_indices), float(w.sm_scale), _ptr(out), _ptr(lse), ctypes.byref(dims),
                int(w.mtp_q_len), _ptr(workspace), workspace.numel(), int(flags), sp)
    elif prefill:
        fn = lib().mla_paged_prefill
        args = (_ptr(w.q_nope), _ptr(w.q_pe), _ptr(w.ckv_cache), _ptr(w.kpe_cache), _ptr(w.qo_indptr),
                _ptr(w.kv_indptr), _ptr(w.kv_indices), float(w.sm_scale), _ptr(out), _ptr(lse),
                ctypes.byref(dims), _ptr(workspace), workspace.numel(), int(flags), sp)
    else:
        fn = lib().mla_paged_decode
        args = (_ptr(w.q_nope), _ptr(w.q_pe), _ptr(w.ckv_cache), _ptr(w.kpe_cache), _ptr(w.kv_indptr),
                _ptr(w.kv_indices), float(w.sm_scale), _ptr(out), _ptr(lse), ctypes.byref(dims),
                _ptr(workspace), workspace.numel(), int(flags), sp)
    keep = (w, out, lse, workspace, stream, dims)  # keep the tensors and dims alive

    def call():
        st = fn(*args)
        if st != 0:
            raise MlaError(st, name)
        return keep[1], keep[2]

    return call


def run_workload(w, out=None, lse=None, workspace=None, flags=0, num_workers=0, stream=None):
    """Call decode, prefill, packed multi-token or sparse decode on a ``workloads.Workload`` whose
    tensors are on the GPU.  Returns (out, lse) shaped [rows, H, 512] and [rows, H]."""
    if w.kind == "mtp":
        b, q, h = w.batch, w.mtp_q_len, w.num_qo_heads
        o4 = None if out is None else out.view(b, q, h, HEAD_DIM_CKV)
        l3 = None if lse is None else lse.view(b, q, h)
        o4, l3 = mla_paged_decode_mtp(w.q_nope.view(b, q, h, HEAD_DIM_CKV), w.q_pe.view(b, q, h, HEAD_DIM_KPE),
                                      w.ckv_cache, w.kpe_cache, w.kv_indptr, w.kv_indices, w.sm_scale,
                                      o4, l3, workspace, flags, num_workers, stream)
        return o4.view(b * q, h, HEAD_DIM_CKV), l3.view(b * q, h)
    if w.kind == "decode_fp8":
        return mla_paged_decode_fp8(w.q_nope, w.q_pe, w.kv_fp8, w.kv_indptr, w.kv_indices, w.sm_scale,
                                    out, lse, workspace, flags, num_workers, stream)
    if w.kind == "sparse_fp8":
        return mla_paged_decode_sparse_fp8(w.q_nope, w.q_pe, w.kv_fp8, w.indices, w.sm_scale,
                                           out, lse, workspace, flags, num_workers, stream)
    if w.kind == "sparse":
        return mla_paged_decode_sparse(w.q_nope, w.q_pe, w.ckv_cache, w.kpe_cache, w.indices, w.sm_scale,
                                       out, lse, workspace, flags, num_workers, stream)
    if w.kind == "decode":
        return mla_paged_decode(w.q_nope, w.q_pe, w.ckv_cache, w.kpe_cache, w.kv_indptr, w.kv_indices,
                                w.sm_scale, out, lse, workspace, flags, num_workers, stream)
    return mla_paged_prefill(w.q_nope, w.q_pe, w.ckv_cache, w.kpe_cache, w.qo_indptr, w.kv_indptr,
                             w.kv_indices, w.sm_scale, out, lse, workspace, flags, num_workers, stream)
