"""CPU oracle of the MSA forward path (test infrastructure only).

Thin ctypes marshalling over liboracle.so (msa_oracle.cpp), which holds every
step of the method in plain fp64 loops. Only the tests, the smoke check and
the benchmark's CPU-baseline leg use it; the GPU path never does.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None

P = ctypes.c_void_p
I64, I32, D = ctypes.c_int64, ctypes.c_int, ctypes.c_double


def lib():
    global _lib
    if _lib is None:
        from . import build as _b
        _lib = ctypes.CDLL(_b.build())
        L = _lib
        L.oracle_num_threads.restype = I32
        L.oracle_hardware_concurrency.restype = ctypes.c_uint
        L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f64.restype = D
        L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_f64.restype = D
        L.oracle_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_to_f64.restype = D
        L.oracle_index_select.argtypes = [P, P, I64, P, I32, I32, I32, I32, I64, P, P]
        L.oracle_topk_blocks.argtypes = [P, P, I64, I32, I64, I32, I32, P]
        L.oracle_sparse_attn.argtypes = [P, P, I64, P, P, P, I32, I32, I32, I32, I32, D, P, P]
        L.oracle_dense_gqa.argtypes = [P, P, I64, P, P, I32, I32, I32, D, P, P]
        L.oracle_kl_teacher.argtypes = [P, P, P, I64, P, P, P, I32, I32, I32, I32, I32, I32, D,
                                        P, P]
        L.oracle_index_project.argtypes = [P, P, P, I64, I32, I32, I32, P, P]
        L.oracle_index_brute.argtypes = [P, P, I64, P, I32, I32, I32, I32, P]
        L.oracle_decode_index_select.argtypes = [P, P, P, P, I32, I32, I32, I32, I32, I32, I64,
                                                 P, P]
        L.oracle_decode_attn.argtypes = [P, P, P, I32, P, P, P, P, P, I32, I32, I32, I32, I32,
                                         I32, I32, D, P, P]
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def _ok(rc):
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")


def threads() -> int:
    return lib().oracle_num_threads()


def bf16_to_f64(bits: int) -> float:
    return lib().oracle_bf16_to_f64(bits)


def e4m3_to_f64(bits: int) -> float:
    return lib().oracle_e4m3_to_f64(bits)


def e2m1_to_f64(code: int) -> float:
    """OCP FP4 E2M1 code (low 4 bits) -> value."""
    return lib().oracle_e2m1_to_f64(code & 0xF)


def index_select(q_idx_rows, rows, k_idx, Bk, k, nb_out=0, want_scores=False):
    """q_idx_rows [n, n_g, d_idx] bf16 bits; rows [n] positions; k_idx [>=max+1, d_idx].
    Returns ids [n, n_g, k] (and fp64 scores [n, n_g, nb_out] when asked)."""
    q, qp = _c(q_idx_rows, np.uint16)
    r, rp = _c(rows, np.int64)
    kk, kp = _c(k_idx, np.uint16)
    n, n_g, d_idx = q.shape
    ids = np.empty((n, n_g, k), dtype=np.int32)
    sc = np.empty((n, n_g, nb_out), dtype=np.float64) if want_scores else None
    _ok(lib().oracle_index_select(qp, rp, n, kp, n_g, d_idx, Bk, k, nb_out,
                                  sc.ctypes.data if want_scores else None, ids.ctypes.data))
    return (ids, sc) if want_scores else ids


def topk_blocks(S_rows, rows, Bk, k):
    """S_rows [n, n_g, nb] fp32 block scores of rows at positions rows[n]."""
    S, sp = _c(S_rows, np.float32)
    r, rp = _c(rows, np.int64)
    n, n_g, nb = S.shape
    ids = np.full((n, n_g, k), -2, dtype=np.int32)
    _ok(lib().oracle_topk_blocks(sp, rp, n, n_g, nb, Bk, k, ids.ctypes.data))
    return ids


def kl_teacher(q_rows, qi_rows, rows, K, k_idx, ids, Bk, scale):
    """KL(teacher || index distribution) per (row, group) over the selected
    tokens: q_rows [n, H_q, d], qi_rows [n, n_g, d_idx], K [N, H_kv, d], k_idx
    [N, d_idx] bf16 bits, ids [n, n_g, k]. Returns (kl, mag) fp64 [n, n_g], mag
    the summed size of the terms (sum p_main (|log p_main| + |log p_idx|))."""
    q, qp = _c(q_rows, np.uint16)
    qi, qip = _c(qi_rows, np.uint16)
    r, rp = _c(rows, np.int64)
    K = np.ascontiguousarray(K, dtype=np.uint16)
    kk = np.ascontiguousarray(k_idx, dtype=np.uint16)
    ii, ip = _c(ids, np.int32)
    n, H_q, d = q.shape
    H_kv = K.shape[-2]
    d_idx = qi.shape[-1]
    k = ii.shape[-1]
    kl = np.empty((n, H_kv), dtype=np.float64)
    mag = np.empty((n, H_kv), dtype=np.float64)
    _ok(lib().oracle_kl_teacher(qp, qip, rp, n, K.ctypes.data, kk.ctypes.data, ip, H_q, H_kv, d,
                                d_idx, Bk, k, float(scale), kl.ctypes.data, mag.ctypes.data))
    return kl, mag


def sparse_attn(q_rows, rows, K, V, ids, Bk, scale):
    """q_rows [n, H_q, d]; K, V [N, H_kv, d] bf16 bits; ids [n, n_g, k]."""
    q, qp = _c(q_rows, np.uint16)
    r, rp = _c(rows, np.int64)
    K = np.ascontiguousarray(K, dtype=np.uint16)
    V = np.ascontiguousarray(V, dtype=np.uint16)
    ii, ip = _c(ids, np.int32)
    n, H_q, d = q.shape
    H_kv = K.shape[-2]
    k = ii.shape[-1]
    o = np.empty((n, H_q, d), dtype=np.float64)
    lse = np.empty((n, H_q), dtype=np.float64)
    _ok(lib().oracle_sparse_attn(qp, rp, n, K.ctypes.data, V.ctypes.data, ip, H_q, H_kv, d,
                                 Bk, k, scale, o.ctypes.data, lse.ctypes.data))
    return o, lse


def index_project(x, w_qidx, w_kidx):
    """x [n, d_model], w_qidx [n_g * d_idx, d_model], w_kidx [d_idx, d_model] bf16
    bits -> (q_idx [n, n_g, d_idx], k_idx [n, d_idx]) fp64."""
    xx, xp = _c(x, np.uint16)
    wq, wqp = _c(w_qidx, np.uint16)
    wk, wkp = _c(w_kidx, np.uint16)
    n, d_model = xx.shape
    d_idx = wk.shape[0]
    n_g = wq.shape[0] // d_idx
    assert wq.shape == (n_g * d_idx, d_model) and wk.shape == (d_idx, d_model)
    q = np.empty((n, n_g, d_idx), dtype=np.float64)
    k = np.empty((n, d_idx), dtype=np.float64)
    _ok(lib().oracle_index_project(xp, wqp, wkp, n, d_model, n_g, d_idx, q.ctypes.data,
                                   k.ctypes.data))
    return q, k


def dense_gqa(q_rows, rows, K, V, scale):
    q, qp = _c(q_rows, np.uint16)
    r, rp = _c(rows, np.int64)
    K = np.ascontiguousarray(K, dtype=np.uint16)
    V = np.ascontiguousarray(V, dtype=np.uint16)
    n, H_q, d = q.shape
    H_kv = K.shape[-2]
    o = np.empty((n, H_q, d), dtype=np.float64)
    lse = np.empty((n, H_q), dtype=np.float64)
    _ok(lib().oracle_dense_gqa(qp, rp, n, K.ctypes.data, V.ctypes.data, H_q, H_kv, d, scale,
                               o.ctypes.data, lse.ctypes.data))
    return o, lse


def index_brute(q_idx_rows, rows, k_idx, Bk, k):
    q, qp = _c(q_idx_rows, np.uint16)
    r, rp = _c(rows, np.int64)
    kk, kp = _c(k_idx, np.uint16)
    n, n_g, d_idx = q.shape
    ids = np.empty((n, n_g, k), dtype=np.int32)
    _ok(lib().oracle_index_brute(qp, rp, n, kp, n_g, d_idx, Bk, k, ids.ctypes.data))
    return ids


def decode_index_select(q_idx, k_idx_pages, page_table, seq_lens, Bk, k, nb_out=0,
                        want_scores=False):
    """q_idx [B, n_g, d_idx]; k_idx_pages [P, Bk, d_idx]; page_table [B, max_pages]."""
    q, qp = _c(q_idx, np.uint16)
    kk = np.ascontiguousarray(k_idx_pages, dtype=np.uint16)
    pt, ptp = _c(page_table, np.int32)
    sl, slp = _c(seq_lens, np.int32)
    B, n_g, d_idx = q.shape
    ids = np.empty((B, n_g, k), dtype=np.int32)
    sc = np.empty((B, n_g, nb_out), dtype=np.float64) if want_scores else None
    _ok(lib().oracle_decode_index_select(qp, kk.ctypes.data, ptp, slp, B, pt.shape[1], n_g,
                                         d_idx, Bk, k, nb_out,
                                         sc.ctypes.data if want_scores else None,
                                         ids.ctypes.data))
    return (ids, sc) if want_scores else ids


def decode_attn(q, k_pages, v_pages, page_table, seq_lens, ids, Bk, scale, fp8=False,
                k_scale=None, v_scale=None):
    """q [B, H_q, d]; k_pages, v_pages [P, H_kv, Bk, d] (bf16 bits, or E4M3 bits
    with per-kv-head fp32 scales when fp8)."""
    qq, qp = _c(q, np.uint16)
    kdt = np.uint8 if fp8 else np.uint16
    kp = np.ascontiguousarray(k_pages, dtype=kdt)
    vp = np.ascontiguousarray(v_pages, dtype=kdt)
    pt, ptp = _c(page_table, np.int32)
    sl, slp = _c(seq_lens, np.int32)
    ii, ip = _c(ids, np.int32)
    B, H_q, d = qq.shape
    H_kv = kp.shape[1]
    ks = np.ascontiguousarray(k_scale if k_scale is not None else np.ones(H_kv), np.float32)
    vs = np.ascontiguousarray(v_scale if v_scale is not None else np.ones(H_kv), np.float32)
    o = np.empty((B, H_q, d), dtype=np.float64)
    lse = np.empty((B, H_q), dtype=np.float64)
    _ok(lib().oracle_decode_attn(qp, kp.ctypes.data, vp.ctypes.data, int(fp8), ks.ctypes.data,
                                 vs.ctypes.data, ptp, slp, ip, B, pt.shape[1], H_q, H_kv, d, Bk,
                                 ii.shape[-1], scale, o.ctypes.data, lse.ctypes.data))
    return o, lse
