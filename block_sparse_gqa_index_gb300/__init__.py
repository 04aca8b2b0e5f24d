"""MiniMax Sparse Attention (MSA) forward path on GB300 (sm_103a).

Thin Python binding of libmsa.so (C ABI in include/msa.h). Every function here
only checks and marshals its torch arguments (device pointers, sizes, the
current CUDA stream) and calls the library entry point of the same name; all
computation happens in the library's CUDA kernels. There is no other backend:
importing this package fails if libmsa.so has not been built.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmsa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
        "(or python block_sparse_gqa_index_gb300/build.py); there is no fallback path")

_lib = ctypes.CDLL(LIB_PATH)

MSA_OK, MSA_ERR_INVALID_ARG, MSA_ERR_UNSUPPORTED, MSA_ERR_WORKSPACE, MSA_ERR_CUDA, \
    MSA_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
MSA_KV_BF16, MSA_KV_E4M3 = 0, 1

_P, _I, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


def _sig(name, argtypes, restype=ctypes.c_int):
    fn = getattr(_lib, name)
    fn.argtypes = argtypes
    fn.restype = restype
    return fn


_status_string = _sig("msa_status_string", [_I], ctypes.c_char_p)
_version = _sig("msa_version", [])
_ws_index = _sig("msa_index_select_workspace_bytes", [_I64, _I, _I, _I, _I], _SZ)
_index_select = _sig("msa_index_select", [_P, _P, _I64, _I, _I, _I, _I, _P, _P, _P, _SZ, _P])
_topk = _sig("msa_topk_blocks", [_P, _I64, _I, _I64, _I, _I, _I64, _P, _P, _P])
_ws_attn = _sig("msa_sparse_attn_workspace_bytes", [_I64, _I64, _I, _I, _I, _I, _I], _SZ)
_sparse_attn = _sig("msa_sparse_attn", [_P, _P, _P, _P, _I64, _I, _I, _I, _I, _I, _F, _P, _P,
                                        _P, _SZ, _P])
_ws_index_dec = _sig("msa_index_select_decode_workspace_bytes", [_I, _I, _I], _SZ)
_index_dec = _sig("msa_index_select_decode", [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P,
                                              _P, _SZ, _P])
_ws_dec = _sig("msa_decode_workspace_bytes", [_I, _I, _I, _I], _SZ)
_decode = _sig("msa_decode", [_P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                              _P, _P, _P, _SZ, _P])
_decode_fp4 = _sig("msa_decode_nvfp4", [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                         _I, _F, _P, _P, _P, _SZ, _P])
_get_error = _sig("msa_get_error", [_P])
_set_wait = _sig("msa_set_wait_limit", [_I64], _I64)
_launch_count = _sig("msa_launch_count", [], _I64)
_index_dec_noalloc = _sig("msa_index_select_decode_noalloc", [_P, _P, _P, _P, _I, _I, _I, _I, _I,
                                                              _I, _P, _P])
_noalloc_max = _sig("msa_index_select_decode_noalloc_max_scores", [], _I64)
_index_project = _sig("msa_index_project", [_P, _P, _P, _I64, _I, _I, _I, _P, _P, _P])
_index_fp8 = _sig("msa_index_select_fp8", [_P, _P, _I64, _I, _I, _I, _I, _P, _P, _F, _P])
_ws_index_fp4 = _sig("msa_index_select_nvfp4_workspace_bytes", [_I64, _I, _I], _SZ)
_index_fp4 = _sig("msa_index_select_nvfp4", [_P, _P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P,
                                             _SZ, _P])
_index_varlen = _sig("msa_index_select_varlen", [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P])
_ws_attn_varlen = _sig("msa_sparse_attn_varlen_workspace_bytes", [_P, _I, _I, _I, _I, _I, _I],
                       _SZ)
_attn_varlen = _sig("msa_sparse_attn_varlen", [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F,
                                               _P, _P, _P, _SZ, _P])
_index_dec_fp4 = _sig("msa_index_select_decode_nvfp4", [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                                         _I, _P, _P, _F, _P, _SZ, _P])
_ws_kl = _sig("msa_kl_teacher_workspace_bytes", [_I64, _I64, _I, _I, _I, _I, _I], _SZ)
_kl = _sig("msa_kl_teacher", [_P, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                              _SZ, _P])
_index_dec_fp8 = _sig("msa_index_select_decode_fp8", [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                                      _P, _P, _F, _P, _SZ, _P])
_index_paged = _sig("msa_index_select_paged", [_P, _P, _I64, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                               _P, _P])
_ws_attn_paged = _sig("msa_sparse_attn_paged_workspace_bytes", [_P, _P, _I, _I, _I, _I, _I, _I,
                                                                _I], _SZ)
_attn_paged = _sig("msa_sparse_attn_paged", [_P, _P, _P, _I64, _P, _I, _P, _P, _P, _I, _I, _I, _I,
                                             _I, _I, _F, _P, _P, _P, _SZ, _P])

EXPORTS = ["msa_status_string", "msa_version", "msa_index_select_workspace_bytes",
           "msa_index_select", "msa_topk_blocks", "msa_sparse_attn_workspace_bytes",
           "msa_sparse_attn", "msa_index_select_decode_workspace_bytes",
           "msa_index_select_decode", "msa_decode_workspace_bytes", "msa_decode",
           "msa_get_error", "msa_set_wait_limit", "msa_launch_count",
           "msa_index_select_decode_noalloc", "msa_index_select_decode_noalloc_max_scores",
           "msa_index_select_fp8", "msa_index_select_varlen",
           "msa_sparse_attn_varlen_workspace_bytes",
           "msa_sparse_attn_varlen", "msa_index_select_paged",
           "msa_sparse_attn_paged_workspace_bytes", "msa_sparse_attn_paged",
           "msa_index_select_decode_fp8", "msa_kl_teacher_workspace_bytes",
           "msa_kl_teacher", "msa_index_select_decode_nvfp4", "msa_index_project",
           "msa_decode_nvfp4", "msa_index_select_nvfp4_workspace_bytes",
           "msa_index_select_nvfp4"]


class MSAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_status_string(status).decode()} ({status})")


def _check(rc: int, where: str):
    if rc != MSA_OK:
        raise MSAError(rc, where)


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _req(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def version() -> int:
    return _version()


def msa_status_string(status: int) -> str:
    return _status_string(status).decode()


# ------------------------------------------------------------------ prefill
def msa_index_select(q_idx: torch.Tensor, k_idx: torch.Tensor, Bk: int = 128, k: int = 16,
                     block_ids: Optional[torch.Tensor] = None,
                     block_scores: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Index branch of prefill. q_idx [N, n_groups, d_idx] bf16, k_idx [N, d_idx]
    bf16 -> block_ids [N, n_groups, k] int32 (and block_scores [N, n_groups,
    ceil(N/Bk)] fp32 filled on the visible part when given)."""
    N, n_g, d_idx = q_idx.shape
    _req(q_idx, "q_idx", torch.bfloat16)
    _req(k_idx, "k_idx", torch.bfloat16, (N, d_idx))
    if block_ids is None:
        block_ids = torch.empty((N, n_g, k), dtype=torch.int32, device=q_idx.device)
    _req(block_ids, "block_ids", torch.int32, (N, n_g, k))
    if block_scores is not None:
        _req(block_scores, "block_scores", torch.float32, (N, n_g, (N + Bk - 1) // Bk))
    _check(_index_select(q_idx.data_ptr(), k_idx.data_ptr(), N, n_g, d_idx, Bk, k,
                         block_ids.data_ptr(), _ptr(block_scores), None, 0, _stream(q_idx)),
           "msa_index_select")
    return block_ids


def msa_index_project(x: torch.Tensor, w_qidx: torch.Tensor, w_kidx: torch.Tensor,
                      q_idx: Optional[torch.Tensor] = None,
                      k_idx: Optional[torch.Tensor] = None):
    """Index-branch projections: x [N, d_model] bf16, w_qidx [n_groups * d_idx,
    d_model] bf16, w_kidx [d_idx, d_model] bf16 -> (q_idx [N, n_groups, d_idx],
    k_idx [N, d_idx]) bf16."""
    N, d_model = x.shape
    d_idx = w_kidx.shape[0]
    n_g = w_qidx.shape[0] // d_idx
    _req(x, "x", torch.bfloat16)
    _req(w_qidx, "w_qidx", torch.bfloat16, (n_g * d_idx, d_model))
    _req(w_kidx, "w_kidx", torch.bfloat16, (d_idx, d_model))
    if q_idx is None:
        q_idx = torch.empty((N, n_g, d_idx), dtype=torch.bfloat16, device=x.device)
    if k_idx is None:
        k_idx = torch.empty((N, d_idx), dtype=torch.bfloat16, device=x.device)
    _req(q_idx, "q_idx", torch.bfloat16, (N, n_g, d_idx))
    _req(k_idx, "k_idx", torch.bfloat16, (N, d_idx))
    _check(_index_project(x.data_ptr(), w_qidx.data_ptr(), w_kidx.data_ptr(), N, d_model, n_g,
                          d_idx, q_idx.data_ptr(), k_idx.data_ptr(), _stream(x)),
           "msa_index_project")
    return q_idx, k_idx


def msa_index_select_fp8(q_idx: torch.Tensor, k_idx: torch.Tensor, Bk: int = 128, k: int = 16,
                         block_ids: Optional[torch.Tensor] = None,
                         block_scores: Optional[torch.Tensor] = None,
                         score_scale: float = 1.0) -> torch.Tensor:
    """Index branch on FP8-E4M3 codes: q_idx [N, n_groups, 128] and k_idx [N, 128]
    torch.float8_e4m3fn (or uint8 holding the codes) -> block_ids [N, n_groups, k];
    block_scores, when given, receive the pooled scores times score_scale."""
    N, n_g, d_idx = q_idx.shape
    for t, name in ((q_idx, "q_idx"), (k_idx, "k_idx")):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise TypeError(f"{name} must hold E4M3 codes (float8_e4m3fn or uint8)")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if tuple(k_idx.shape) != (N, d_idx):
        raise ValueError("k_idx must be [N, d_idx]")
    if block_ids is None:
        block_ids = torch.empty((N, n_g, k), dtype=torch.int32, device=q_idx.device)
    _req(block_ids, "block_ids", torch.int32, (N, n_g, k))
    if block_scores is not None:
        _req(block_scores, "block_scores", torch.float32, (N, n_g, (N + Bk - 1) // Bk))
    _check(_index_fp8(q_idx.data_ptr(), k_idx.data_ptr(), N, n_g, d_idx, Bk, k,
                      block_ids.data_ptr(), _ptr(block_scores), score_scale, _stream(q_idx)),
           "msa_index_select_fp8")
    return block_ids


def msa_index_select_nvfp4_workspace_bytes(N: int, n_groups: int, d_idx: int) -> int:
    return _ws_index_fp4(N, n_groups, d_idx)


def msa_index_select_nvfp4(q_codes: torch.Tensor, q_scales: torch.Tensor,
                           k_codes: torch.Tensor, k_scales: torch.Tensor, Bk: int = 128,
                           k: int = 16, block_ids: Optional[torch.Tensor] = None,
                           block_scores: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Index branch on NVFP4 operands: q_codes [N, n_groups, d_idx / 2] and
    k_codes [N, d_idx / 2] uint8 (two E2M1 codes per byte, even dimension low),
    q_scales [N, n_groups, d_idx / 16] and k_scales [N, d_idx / 16] E4M3 scales
    (float8_e4m3fn or uint8) -> block_ids [N, n_groups, k]."""
    N, n_g, half = q_codes.shape
    d_idx = 2 * half
    for t, name, shape in ((q_codes, "q_codes", (N, n_g, half)),
                           (q_scales, "q_scales", (N, n_g, d_idx // 16)),
                           (k_codes, "k_codes", (N, half)),
                           (k_scales, "k_scales", (N, d_idx // 16))):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise TypeError(f"{name} must be uint8 (or float8_e4m3fn for the scales)")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {list(shape)}")
    if block_ids is None:
        block_ids = torch.empty((N, n_g, k), dtype=torch.int32, device=q_codes.device)
    _req(block_ids, "block_ids", torch.int32, (N, n_g, k))
    if block_scores is not None:
        _req(block_scores, "block_scores", torch.float32, (N, n_g, (N + Bk - 1) // Bk))
    need = _ws_index_fp4(N, n_g, d_idx)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_codes.device)
    _check(_index_fp4(q_codes.data_ptr(), q_scales.data_ptr(), k_codes.data_ptr(),
                      k_scales.data_ptr(), N, n_g, d_idx, Bk, k, block_ids.data_ptr(),
                      _ptr(block_scores), workspace.data_ptr(),
                      workspace.numel() * workspace.element_size(), _stream(q_codes)),
           "msa_index_select_nvfp4")
    return block_ids


def msa_topk_blocks(block_scores: torch.Tensor, Bk: int = 128, k: int = 16, q_offset: int = 0,
                    seq_lens: Optional[torch.Tensor] = None,
                    block_ids: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Exp-free top-k over block scores [N, n_groups, nb] fp32 -> [N, n_groups, k]."""
    N, n_g, nb = block_scores.shape
    _req(block_scores, "block_scores", torch.float32)
    if seq_lens is not None:
        _req(seq_lens, "seq_lens", torch.int32, (N,))
    if block_ids is None:
        block_ids = torch.empty((N, n_g, k), dtype=torch.int32, device=block_scores.device)
    _req(block_ids, "block_ids", torch.int32, (N, n_g, k))
    _check(_topk(block_scores.data_ptr(), N, n_g, nb, Bk, k, q_offset, _ptr(seq_lens),
                 block_ids.data_ptr(), _stream(block_scores)), "msa_topk_blocks")
    return block_ids


def msa_sparse_attn_workspace_bytes(chunk_rows: int, N: int, H_q: int, H_kv: int, d: int,
                                    Bk: int = 128, k: int = 16) -> int:
    return _ws_attn(chunk_rows, N, H_q, H_kv, d, Bk, k)


def msa_sparse_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block_ids: torch.Tensor,
                    Bk: int = 128, scale: Optional[float] = None,
                    workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None, want_lse: bool = True):
    """Main branch of prefill. q [N, H_q, d], k/v [N, H_kv, d] bf16, block_ids
    [N, H_kv, topk] int32 -> (out [N, H_q, d] bf16, lse [N, H_q] fp32)."""
    N, H_q, d = q.shape
    H_kv = k.shape[1]
    topk = block_ids.shape[-1]
    _req(q, "q", torch.bfloat16)
    _req(k, "k", torch.bfloat16, (N, H_kv, d))
    _req(v, "v", torch.bfloat16, (N, H_kv, d))
    _req(block_ids, "block_ids", torch.int32, (N, H_kv, topk))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = torch.empty(msa_sparse_attn_workspace_bytes(N, N, H_q, H_kv, d, Bk, topk),
                                dtype=torch.uint8, device=q.device)
    _req(workspace, "workspace", torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    _req(out, "out", torch.bfloat16, (N, H_q, d))
    if lse is None and want_lse:
        lse = torch.empty((N, H_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _req(lse, "lse", torch.float32, (N, H_q))
    _check(_sparse_attn(q.data_ptr(), k.data_ptr(), v.data_ptr(), block_ids.data_ptr(), N, H_q,
                        H_kv, d, Bk, topk, scale, out.data_ptr(), _ptr(lse),
                        workspace.data_ptr(), workspace.numel(), _stream(q)), "msa_sparse_attn")
    return out, lse


# ------------------------------------------------------------ varlen prefill
def _cu_array(cu_seqlens):
    """Host int64 copy of the cumulative sequence offsets [B + 1]."""
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int64, device="cpu").contiguous()
    if cu.dim() != 1 or cu.numel() < 1:
        raise ValueError("cu_seqlens must be a 1-D sequence of B + 1 offsets")
    return cu


def msa_index_select_varlen(q_idx: torch.Tensor, k_idx: torch.Tensor, cu_seqlens,
                            Bk: int = 128, k: int = 16,
                            block_ids: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Index branch over B sequences packed back to back: sequence b holds rows
    cu_seqlens[b] .. cu_seqlens[b + 1] - 1 of q_idx [T, n_groups, d_idx] and
    k_idx [T, d_idx]; -> block_ids [T, n_groups, k], counted from each
    sequence's first token."""
    cu = _cu_array(cu_seqlens)
    T, n_g, d_idx = q_idx.shape
    _req(q_idx, "q_idx", torch.bfloat16)
    _req(k_idx, "k_idx", torch.bfloat16, (T, d_idx))
    if int(cu[-1]) != T:
        raise ValueError("cu_seqlens[-1] must equal the number of rows")
    if block_ids is None:
        block_ids = torch.empty((T, n_g, k), dtype=torch.int32, device=q_idx.device)
    _req(block_ids, "block_ids", torch.int32, (T, n_g, k))
    _check(_index_varlen(q_idx.data_ptr(), k_idx.data_ptr(), cu.data_ptr(), cu.numel() - 1, n_g,
                         d_idx, Bk, k, block_ids.data_ptr(), _stream(q_idx)),
           "msa_index_select_varlen")
    return block_ids


def msa_sparse_attn_varlen_workspace_bytes(cu_seqlens, H_q: int, H_kv: int, d: int,
                                           Bk: int = 128, k: int = 16) -> int:
    cu = _cu_array(cu_seqlens)
    return _ws_attn_varlen(cu.data_ptr(), cu.numel() - 1, H_q, H_kv, d, Bk, k)


def msa_sparse_attn_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                           block_ids: torch.Tensor, cu_seqlens, Bk: int = 128,
                           scale: Optional[float] = None,
                           workspace: Optional[torch.Tensor] = None,
                           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                           want_lse: bool = True):
    """Main branch over B packed sequences (rows as in msa_index_select_varlen):
    q [T, H_q, d], k / v [T, H_kv, d] bf16, block_ids [T, H_kv, topk] ->
    out [T, H_q, d] bf16, lse [T, H_q] fp32."""
    cu = _cu_array(cu_seqlens)
    T, H_q, d = q.shape
    H_kv = k.shape[1]
    topk = block_ids.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _req(q, "q", torch.bfloat16)
    _req(k, "k", torch.bfloat16, (T, H_kv, d))
    _req(v, "v", torch.bfloat16, (T, H_kv, d))
    _req(block_ids, "block_ids", torch.int32, (T, H_kv, topk))
    if int(cu[-1]) != T:
        raise ValueError("cu_seqlens[-1] must equal the number of rows")
    if workspace is None:
        workspace = torch.empty(max(1, _ws_attn_varlen(cu.data_ptr(), cu.numel() - 1, H_q, H_kv,
                                                       d, Bk, topk)),
                                dtype=torch.uint8, device=q.device)
    _req(workspace, "workspace", torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    _req(out, "out", torch.bfloat16, (T, H_q, d))
    if lse is None and want_lse:
        lse = torch.empty((T, H_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _req(lse, "lse", torch.float32, (T, H_q))
    _check(_attn_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), block_ids.data_ptr(),
                        cu.data_ptr(), cu.numel() - 1, H_q, H_kv, d, Bk, topk, scale,
                        out.data_ptr(), _ptr(lse), workspace.data_ptr(), workspace.numel(),
                        _stream(q)), "msa_sparse_attn_varlen")
    return out, lse


def msa_kl_teacher(q: torch.Tensor, k: torch.Tensor, q_idx: torch.Tensor, k_idx: torch.Tensor,
                   block_ids: torch.Tensor, lse: torch.Tensor, Bk: int = 128,
                   scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """KL alignment signal of the index branch: q [N, H_q, d], k [N, H_kv, d],
    q_idx [N, H_kv, d_idx], k_idx [N, d_idx] bf16, block_ids [N, H_kv, topk],
    lse [N, H_q] fp32 (the main branch's, on the same ids) -> kl [N, H_kv] fp32,
    KL(group-averaged main-branch distribution || index softmax) over each
    row's selected tokens."""
    N, H_q, d = q.shape
    H_kv = k.shape[1]
    d_idx = q_idx.shape[2]
    topk = block_ids.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _req(q, "q", torch.bfloat16)
    _req(k, "k", torch.bfloat16, (N, H_kv, d))
    _req(q_idx, "q_idx", torch.bfloat16, (N, H_kv, d_idx))
    _req(k_idx, "k_idx", torch.bfloat16, (N, d_idx))
    _req(block_ids, "block_ids", torch.int32, (N, H_kv, topk))
    _req(lse, "lse", torch.float32, (N, H_q))
    if workspace is None:
        workspace = torch.empty(max(1, _ws_kl(N, N, H_q, H_kv, d, Bk, topk)), dtype=torch.uint8,
                                device=q.device)
    _req(workspace, "workspace", torch.uint8)
    if out is None:
        out = torch.empty((N, H_kv), dtype=torch.float32, device=q.device)
    _req(out, "out", torch.float32, (N, H_kv))
    _check(_kl(q.data_ptr(), k.data_ptr(), q_idx.data_ptr(), k_idx.data_ptr(),
               block_ids.data_ptr(), lse.data_ptr(), N, H_q, H_kv, d, d_idx, Bk, topk, scale,
               out.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(q)),
           "msa_kl_teacher")
    return out


# ------------------------------------------------------------ paged prefill
def _paged_args(page_table: torch.Tensor, cu_q, kv_lens):
    cu = _cu_array(cu_q)
    kv = torch.as_tensor(kv_lens, dtype=torch.int64, device="cpu").contiguous().reshape(-1)
    B = cu.numel() - 1
    if kv.numel() != B:
        raise ValueError("kv_lens must hold one length per sequence")
    _req(page_table, "page_table", torch.int32)
    if page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError("page_table must be [B, max_pages]")
    return cu, kv, B, page_table.shape[1]


def msa_index_select_paged(q_idx: torch.Tensor, k_idx_pages: torch.Tensor,
                           page_table: torch.Tensor, cu_q, kv_lens, Bk: int = 128, k: int = 16,
                           block_ids: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Index branch of a chunked prefill over a paged k_idx cache: sequence b
    holds kv_lens[b] tokens, its last cu_q[b + 1] - cu_q[b] are its queries
    (rows of q_idx [T, n_groups, d_idx]); k_idx_pages [P, Bk, d_idx], page_table
    [B, max_pages] int32 -> block_ids [T, n_groups, k]."""
    cu, kv, B, max_pages = _paged_args(page_table, cu_q, kv_lens)
    T, n_g, d_idx = q_idx.shape
    _req(q_idx, "q_idx", torch.bfloat16)
    _req(k_idx_pages, "k_idx_pages", torch.bfloat16)
    if k_idx_pages.dim() != 3 or k_idx_pages.shape[1] != Bk or k_idx_pages.shape[2] != d_idx:
        raise ValueError("k_idx_pages must be [P, Bk, d_idx]")
    if int(cu[-1]) != T:
        raise ValueError("cu_q[-1] must equal the number of query rows")
    if block_ids is None:
        block_ids = torch.empty((T, n_g, k), dtype=torch.int32, device=q_idx.device)
    _req(block_ids, "block_ids", torch.int32, (T, n_g, k))
    _check(_index_paged(q_idx.data_ptr(), k_idx_pages.data_ptr(), k_idx_pages.shape[0],
                        page_table.data_ptr(), max_pages, cu.data_ptr(), kv.data_ptr(), B, n_g,
                        d_idx, Bk, k, block_ids.data_ptr(), _stream(q_idx)),
           "msa_index_select_paged")
    return block_ids


def msa_sparse_attn_paged_workspace_bytes(cu_q, kv_lens, max_pages: int, H_q: int, H_kv: int,
                                          d: int, Bk: int = 128, k: int = 16) -> int:
    cu = _cu_array(cu_q)
    kv = torch.as_tensor(kv_lens, dtype=torch.int64, device="cpu").contiguous().reshape(-1)
    return _ws_attn_paged(cu.data_ptr(), kv.data_ptr(), cu.numel() - 1, max_pages, H_q, H_kv, d,
                          Bk, k)


def msa_sparse_attn_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
                          page_table: torch.Tensor, block_ids: torch.Tensor, cu_q, kv_lens,
                          Bk: int = 128, scale: Optional[float] = None,
                          workspace: Optional[torch.Tensor] = None,
                          out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                          want_lse: bool = True):
    """Main branch of a chunked prefill over paged K / V ([P, H_kv, Bk, d]
    bf16, the decode layout): q [T, H_q, d], block_ids [T, H_kv, topk] ->
    out [T, H_q, d] bf16, lse [T, H_q] fp32."""
    cu, kv, B, max_pages = _paged_args(page_table, cu_q, kv_lens)
    T, H_q, d = q.shape
    P, H_kv = k_pages.shape[0], k_pages.shape[1]
    topk = block_ids.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _req(q, "q", torch.bfloat16)
    _req(k_pages, "k_pages", torch.bfloat16, (P, H_kv, Bk, d))
    _req(v_pages, "v_pages", torch.bfloat16, (P, H_kv, Bk, d))
    _req(block_ids, "block_ids", torch.int32, (T, H_kv, topk))
    if int(cu[-1]) != T:
        raise ValueError("cu_q[-1] must equal the number of query rows")
    if workspace is None:
        workspace = torch.empty(max(1, _ws_attn_paged(cu.data_ptr(), kv.data_ptr(), B, max_pages,
                                                      H_q, H_kv, d, Bk, topk)),
                                dtype=torch.uint8, device=q.device)
    _req(workspace, "workspace", torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    _req(out, "out", torch.bfloat16, (T, H_q, d))
    if lse is None and want_lse:
        lse = torch.empty((T, H_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _req(lse, "lse", torch.float32, (T, H_q))
    _check(_attn_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), P,
                       page_table.data_ptr(), max_pages, block_ids.data_ptr(), cu.data_ptr(),
                       kv.data_ptr(), B, H_q, H_kv, d, Bk, topk, scale, out.data_ptr(), _ptr(lse),
                       workspace.data_ptr(), workspace.numel(), _stream(q)),
           "msa_sparse_attn_paged")
    return out, lse


# ------------------------------------------------------------------- decode
def msa_index_select_decode(q_idx: torch.Tensor, k_idx_pages: torch.Tensor,
                            page_table: torch.Tensor, seq_lens: torch.Tensor, Bk: int = 128,
                            k: int = 16, block_ids: Optional[torch.Tensor] = None,
                            block_scores: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Index branch of decode. q_idx [B, n_groups, d_idx], k_idx_pages [P, Bk,
    d_idx] bf16, page_table [B, max_pages] int32, seq_lens [B] int32 ->
    block_ids [B, n_groups, k] int32."""
    B, n_g, d_idx = q_idx.shape
    max_pages = page_table.shape[1]
    _req(q_idx, "q_idx", torch.bfloat16)
    _req(k_idx_pages, "k_idx_pages", torch.bfloat16)
    if k_idx_pages.shape[1:] != (Bk, d_idx):
        raise ValueError("k_idx_pages must be [P, Bk, d_idx]")
    _req(page_table, "page_table", torch.int32, (B, max_pages))
    _req(seq_lens, "seq_lens", torch.int32, (B,))
    if block_ids is None:
        block_ids = torch.empty((B, n_g, k), dtype=torch.int32, device=q_idx.device)
    _req(block_ids, "block_ids", torch.int32, (B, n_g, k))
    if block_scores is not None:
        _req(block_scores, "block_scores", torch.float32, (B, n_g, max_pages))
    elif workspace is None:
        workspace = torch.empty(_ws_index_dec(B, max_pages, n_g), dtype=torch.uint8,
                                device=q_idx.device)
    ws_ptr, ws_n = (None, 0) if workspace is None else (_req(workspace, "workspace", torch.uint8),
                                                         workspace.numel())
    _check(_index_dec(q_idx.data_ptr(), k_idx_pages.data_ptr(), page_table.data_ptr(),
                      seq_lens.data_ptr(), B, max_pages, n_g, d_idx, Bk, k, block_ids.data_ptr(),
                      _ptr(block_scores), ws_ptr, ws_n, _stream(q_idx)),
           "msa_index_select_decode")
    return block_ids


def msa_index_select_decode_fp8(q_idx: torch.Tensor, k_idx_pages: torch.Tensor,
                                page_table: torch.Tensor, seq_lens: torch.Tensor, Bk: int = 128,
                                k: int = 16, block_ids: Optional[torch.Tensor] = None,
                                block_scores: Optional[torch.Tensor] = None,
                                score_scale: float = 1.0,
                                workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Index branch of decode over an E4M3 k_idx cache: q_idx [B, n_groups, d_idx]
    and k_idx_pages [P, Bk, d_idx] torch.float8_e4m3fn (or uint8 holding the
    codes), page_table [B, max_pages] int32, seq_lens [B] int32 -> block_ids
    [B, n_groups, k]; block_scores, when given, receive the pooled scores times
    score_scale."""
    B, n_g, d_idx = q_idx.shape
    max_pages = page_table.shape[1]
    for t, name in ((q_idx, "q_idx"), (k_idx_pages, "k_idx_pages")):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise TypeError(f"{name} must hold E4M3 codes (float8_e4m3fn or uint8)")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k_idx_pages.dim() != 3 or tuple(k_idx_pages.shape[1:]) != (Bk, d_idx):
        raise ValueError("k_idx_pages must be [P, Bk, d_idx]")
    _req(page_table, "page_table", torch.int32, (B, max_pages))
    _req(seq_lens, "seq_lens", torch.int32, (B,))
    if block_ids is None:
        block_ids = torch.empty((B, n_g, k), dtype=torch.int32, device=q_idx.device)
    _req(block_ids, "block_ids", torch.int32, (B, n_g, k))
    if block_scores is not None:
        _req(block_scores, "block_scores", torch.float32, (B, n_g, max_pages))
    elif workspace is None:
        workspace = torch.empty(_ws_index_dec(B, max_pages, n_g), dtype=torch.uint8,
                                device=q_idx.device)
    ws_ptr, ws_n = (None, 0) if workspace is None else (_req(workspace, "workspace", torch.uint8),
                                                         workspace.numel())
    _check(_index_dec_fp8(q_idx.data_ptr(), k_idx_pages.data_ptr(), page_table.data_ptr(),
                          seq_lens.data_ptr(), B, max_pages, n_g, d_idx, Bk, k,
                          block_ids.data_ptr(), _ptr(block_scores), score_scale, ws_ptr, ws_n,
                          _stream(q_idx)),
           "msa_index_select_decode_fp8")
    return block_ids


def msa_index_select_decode_nvfp4(q_idx: torch.Tensor, k_idx_codes: torch.Tensor,
                                  k_idx_scales: torch.Tensor, page_table: torch.Tensor,
                                  seq_lens: torch.Tensor, Bk: int = 128, k: int = 16,
                                  block_ids: Optional[torch.Tensor] = None,
                                  block_scores: Optional[torch.Tensor] = None,
                                  score_scale: float = 1.0,
                                  workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Index branch of decode over an NVFP4 k_idx cache: q_idx [B, n_groups, d_idx]
    bf16, k_idx_codes [P, Bk, d_idx / 2] uint8 (two E2M1 codes per byte, even
    dimension in the low nibble), k_idx_scales [P, Bk, d_idx / 16] uint8 (E4M3,
    one per 16 dimensions), page_table [B, max_pages] int32, seq_lens [B] int32
    -> block_ids [B, n_groups, k]."""
    B, n_g, d_idx = q_idx.shape
    max_pages = page_table.shape[1]
    _req(q_idx, "q_idx", torch.bfloat16)
    P = k_idx_codes.shape[0]
    _req(k_idx_codes, "k_idx_codes", torch.uint8, (P, Bk, d_idx // 2))
    _req(k_idx_scales, "k_idx_scales", torch.uint8, (P, Bk, d_idx // 16))
    _req(page_table, "page_table", torch.int32, (B, max_pages))
    _req(seq_lens, "seq_lens", torch.int32, (B,))
    if block_ids is None:
        block_ids = torch.empty((B, n_g, k), dtype=torch.int32, device=q_idx.device)
    _req(block_ids, "block_ids", torch.int32, (B, n_g, k))
    if block_scores is not None:
        _req(block_scores, "block_scores", torch.float32, (B, n_g, max_pages))
    elif workspace is None:
        workspace = torch.empty(_ws_index_dec(B, max_pages, n_g), dtype=torch.uint8,
                                device=q_idx.device)
    ws_ptr, ws_n = (None, 0) if workspace is None else (_req(workspace, "workspace", torch.uint8),
                                                         workspace.numel())
    _check(_index_dec_fp4(q_idx.data_ptr(), k_idx_codes.data_ptr(), k_idx_scales.data_ptr(),
                          page_table.data_ptr(), seq_lens.data_ptr(), B, max_pages, n_g, d_idx,
                          Bk, k, block_ids.data_ptr(), _ptr(block_scores), score_scale, ws_ptr,
                          ws_n, _stream(q_idx)),
           "msa_index_select_decode_nvfp4")
    return block_ids


def msa_index_select_decode_noalloc(q_idx: torch.Tensor, k_idx_pages: torch.Tensor,
                                    page_table: torch.Tensor, seq_lens: torch.Tensor,
                                    Bk: int = 128, k: int = 16,
                                    block_ids: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Decode index branch that allocates nothing on the device: the block
    scores go to the library's fixed scratch array (see include/msa.h). Pass
    `block_ids` to avoid the one torch allocation made here otherwise."""
    B, n_g, d_idx = q_idx.shape
    max_pages = page_table.shape[1]
    _req(q_idx, "q_idx", torch.bfloat16)
    _req(k_idx_pages, "k_idx_pages", torch.bfloat16)
    if k_idx_pages.shape[1:] != (Bk, d_idx):
        raise ValueError("k_idx_pages must be [P, Bk, d_idx]")
    _req(page_table, "page_table", torch.int32, (B, max_pages))
    _req(seq_lens, "seq_lens", torch.int32, (B,))
    if block_ids is None:
        block_ids = torch.empty((B, n_g, k), dtype=torch.int32, device=q_idx.device)
    _req(block_ids, "block_ids", torch.int32, (B, n_g, k))
    _check(_index_dec_noalloc(q_idx.data_ptr(), k_idx_pages.data_ptr(), page_table.data_ptr(),
                              seq_lens.data_ptr(), B, max_pages, n_g, d_idx, Bk, k,
                              block_ids.data_ptr(), _stream(q_idx)),
           "msa_index_select_decode_noalloc")
    return block_ids


def msa_index_select_decode_noalloc_max_scores() -> int:
    return _noalloc_max()


def msa_index_select_decode_workspace_bytes(B: int, max_pages: int, n_groups: int) -> int:
    return _ws_index_dec(B, max_pages, n_groups)


def msa_decode_workspace_bytes(B: int, H_q: int, d: int, k: int = 16) -> int:
    return _ws_dec(B, H_q, d, k)


def msa_decode(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
               page_table: torch.Tensor, seq_lens: torch.Tensor, block_ids: torch.Tensor,
               Bk: int = 128, scale: Optional[float] = None,
               k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
               lse: Optional[torch.Tensor] = None, want_lse: bool = True):
    """Main branch of decode. q [B, H_q, d] bf16; k_pages/v_pages [P, H_kv, Bk, d]
    (head-major pages) bf16, or uint8 E4M3 codes with k_scale/v_scale [H_kv] fp32."""
    B, H_q, d = q.shape
    P, H_kv, _, _ = k_pages.shape
    max_pages = page_table.shape[1]
    topk = block_ids.shape[-1]
    fp8 = k_pages.dtype == torch.uint8
    kv_dtype = MSA_KV_E4M3 if fp8 else MSA_KV_BF16
    _req(q, "q", torch.bfloat16)
    _req(k_pages, "k_pages", torch.uint8 if fp8 else torch.bfloat16, (P, H_kv, Bk, d))
    _req(v_pages, "v_pages", torch.uint8 if fp8 else torch.bfloat16, (P, H_kv, Bk, d))
    _req(page_table, "page_table", torch.int32, (B, max_pages))
    _req(seq_lens, "seq_lens", torch.int32, (B,))
    _req(block_ids, "block_ids", torch.int32, (B, H_kv, topk))
    if fp8:
        _req(k_scale, "k_scale", torch.float32, (H_kv,))
        _req(v_scale, "v_scale", torch.float32, (H_kv,))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = torch.empty(_ws_dec(B, H_q, d, topk), dtype=torch.uint8, device=q.device)
    _req(workspace, "workspace", torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    _req(out, "out", torch.bfloat16, (B, H_q, d))
    if lse is None and want_lse:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _req(lse, "lse", torch.float32, (B, H_q))
    _check(_decode(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), kv_dtype,
                   _ptr(k_scale), _ptr(v_scale), page_table.data_ptr(), seq_lens.data_ptr(),
                   block_ids.data_ptr(), B, max_pages, H_q, H_kv, d, Bk, topk, scale,
                   out.data_ptr(), _ptr(lse), workspace.data_ptr(), workspace.numel(),
                   _stream(q)), "msa_decode")
    return out, lse


def msa_decode_nvfp4(q: torch.Tensor, k_codes: torch.Tensor, k_scales: torch.Tensor,
                     v_codes: torch.Tensor, v_scales: torch.Tensor, page_table: torch.Tensor,
                     seq_lens: torch.Tensor, block_ids: torch.Tensor, Bk: int = 128,
                     scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None,
                     out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                     want_lse: bool = True):
    """Main branch of decode over an NVFP4 KV cache. q [B, H_q, d] bf16;
    k_codes/v_codes [P, H_kv, Bk, d / 2] uint8 (two E2M1 codes per byte, even
    dimension low); k_scales/v_scales [P, H_kv, Bk, d / 16] uint8 (E4M3)."""
    B, H_q, d = q.shape
    P, H_kv = k_codes.shape[0], k_codes.shape[1]
    max_pages = page_table.shape[1]
    topk = block_ids.shape[-1]
    _req(q, "q", torch.bfloat16)
    for t, n in ((k_codes, "k_codes"), (v_codes, "v_codes")):
        _req(t, n, torch.uint8, (P, H_kv, Bk, d // 2))
    for t, n in ((k_scales, "k_scales"), (v_scales, "v_scales")):
        _req(t, n, torch.uint8, (P, H_kv, Bk, d // 16))
    _req(page_table, "page_table", torch.int32, (B, max_pages))
    _req(seq_lens, "seq_lens", torch.int32, (B,))
    _req(block_ids, "block_ids", torch.int32, (B, H_kv, topk))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = torch.empty(_ws_dec(B, H_q, d, topk), dtype=torch.uint8, device=q.device)
    _req(workspace, "workspace", torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    _req(out, "out", torch.bfloat16, (B, H_q, d))
    if lse is None and want_lse:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _req(lse, "lse", torch.float32, (B, H_q))
    _check(_decode_fp4(q.data_ptr(), k_codes.data_ptr(), k_scales.data_ptr(), v_codes.data_ptr(),
                       v_scales.data_ptr(), page_table.data_ptr(), seq_lens.data_ptr(),
                       block_ids.data_ptr(), B, max_pages, H_q, H_kv, d, Bk, topk, scale,
                       out.data_ptr(), _ptr(lse), workspace.data_ptr(), workspace.numel(),
                       _stream(q)), "msa_decode_nvfp4")
    return out, lse


# -------------------------------------------------------------- diagnostics
def msa_get_error(stream=None) -> int:
    """Synchronise and return (and clear) the device error word."""
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    return _get_error(stream)


def msa_set_wait_limit(polls: int) -> int:
    return _set_wait(polls)


def msa_launch_count() -> int:
    """Kernel launches (and device memsets) enqueued by libmsa so far."""
    return _launch_count()
