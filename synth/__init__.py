"""Seeded synthetic workloads for the MSA forward path.

Shared input generation for the CPU oracle side (host fill) and the GPU side
(device fill). Holds no step of the method: only the value distributions and
structure (planted blocks, page tables) of the workloads, keyed by seed.
Both fills come from one C recipe (``synth_recipe.h``) and are bit-identical.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))

T_Q, T_K, T_V, T_QIDX, T_KIDX, T_DIR, T_PLANT, T_PERM = 1, 2, 3, 4, 5, 6, 7, 8
KIND_GAUSS, KIND_INT = 0, 1
MASK64 = (1 << 64) - 1


def mix64(x: int) -> int:
    """splitmix64 finaliser (same constants as synth.h)."""
    x = (x + 0x9E3779B97F4A7C15) & MASK64
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & MASK64
    return x ^ (x >> 31)


def key(seed: int, tensor: int) -> int:
    return mix64(mix64(seed) ^ ((tensor * 0xD1B54A32D192ED03) & MASK64))


def draw(k: int, idx: int, j: int) -> int:
    return mix64((k + idx * 8 + j) & MASK64)


class SynthSpec(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("kind", ctypes.c_int32),
        ("B", ctypes.c_int32),
        ("L", ctypes.c_int64),
        ("H_q", ctypes.c_int32),
        ("H_kv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("n_g", ctypes.c_int32),
        ("d_idx", ctypes.c_int32),
        ("Bk", ctypes.c_int32),
        ("nb", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("q_off", ctypes.c_double),
        ("plant_amp", ctypes.c_double),
        ("fp8_mult", ctypes.c_double),
        ("planted", ctypes.c_void_p),
    ]


# FP8 E4M3 KV: codes are e4m3(z * 448/6) (|z| <= 6 for Irwin-Hall(12) - 6), and
# the per-(K/V, kv head) dequantisation scales below vary by head so that the
# head indexing of the scales is exercised.
FP8_MULT = 448.0 / 6.0


def fp8_scales(H_kv: int):
    base = 6.0 / 448.0
    k_scale = np.array([base * (1.0 + 0.125 * h) for h in range(H_kv)], dtype=np.float32)
    v_scale = np.array([base * (1.0 + 0.0625 * h) for h in range(H_kv)], dtype=np.float32)
    return k_scale, v_scale


@dataclasses.dataclass
class Workload:
    """One synthetic MSA workload (prefill: B = 1, L = N; decode: B sequences
    whose new token sits at position L - 1)."""

    name: str
    seed: int
    kind: int
    B: int
    L: int
    H_q: int
    H_kv: int
    d: int
    d_idx: int
    Bk: int = 128
    k: int = 16
    q_off: float = 0.0
    plant_amp: float = 0.0
    planted: Optional[np.ndarray] = None  # uint8 [B * nb]
    decode: bool = False

    @property
    def n_g(self) -> int:
        return self.H_kv

    @property
    def N(self) -> int:
        return self.L

    @property
    def nb(self) -> int:
        return (self.L + self.Bk - 1) // self.Bk

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def spec(self, planted_ptr: Optional[int] = None) -> SynthSpec:
        s = SynthSpec()
        s.seed = self.seed
        s.kind = self.kind
        s.B = self.B
        s.L = self.L
        s.H_q, s.H_kv, s.d = self.H_q, self.H_kv, self.d
        s.n_g, s.d_idx = self.n_g, self.d_idx
        s.Bk, s.nb = self.Bk, self.nb
        s.q_off, s.plant_amp, s.fp8_mult = self.q_off, self.plant_amp, FP8_MULT
        s.planted = planted_ptr
        return s


def _plant_fraction(seed: int, B: int, nb: int, per10000: int) -> np.ndarray:
    k = key(seed, T_PLANT)
    out = np.zeros(B * nb, dtype=np.uint8)
    for i in range(B * nb):
        if draw(k, i, 1) % 10000 < per10000:
            out[i] = 1
    return out


def _plant_count(seed: int, B: int, nb: int, count: int, lo: int, hi: int) -> np.ndarray:
    """`count` distinct planted blocks per sequence, drawn in [lo, hi)."""
    k = key(seed, T_PLANT)
    out = np.zeros(B * nb, dtype=np.uint8)
    for s in range(B):
        chosen = []
        j = 0
        while len(chosen) < min(count, hi - lo):
            b = lo + draw(k, s * 4096 + j, 2) % (hi - lo)
            j += 1
            if b not in chosen:
                chosen.append(b)
        for b in chosen:
            out[s * nb + b] = 1
    return out


def make(name: str, **over) -> Workload:
    """The five named workloads, plus overrides for smaller test shapes.

    tiny   : N=4096, H_q=4, H_kv=1, d=d_idx=64, integer index inputs, 4 planted
             far blocks (k_idx = 3 s) among blocks 0..15, seed 0
    32k    : N=32768, H_q=32, H_kv=8, d=d_idx=128, Gaussian, 5% of blocks
             planted with k_idx += 2 s, q_idx += s / sqrt(d_idx), seed 1
    128k   : N=131072, same heads, Gaussian, 4 planted far blocks (k_idx += 3 s)
             among the first quarter of blocks, q_idx += s / sqrt(d_idx), seed 2
    decode : 64 sequences of 131072 cached tokens + 1 new token (L=131073),
             same heads, 4 planted far blocks per sequence (k_idx += 3 s), seed 3
    1m     : N=1048576, same heads, Gaussian, 1% of blocks planted (k_idx += 2 s),
             seed 4
    """
    base = dict(
        tiny=dict(seed=0, kind=KIND_INT, B=1, L=4096, H_q=4, H_kv=1, d=64, d_idx=64,
                  plant_amp=3.0),
        **{"32k": dict(seed=1, kind=KIND_GAUSS, B=1, L=32768, H_q=32, H_kv=8, d=128,
                       d_idx=128, plant_amp=2.0)},
        **{"128k": dict(seed=2, kind=KIND_GAUSS, B=1, L=131072, H_q=32, H_kv=8, d=128,
                        d_idx=128, plant_amp=3.0)},
        decode=dict(seed=3, kind=KIND_GAUSS, B=64, L=131073, H_q=32, H_kv=8, d=128,
                    d_idx=128, plant_amp=3.0, decode=True),
        **{"1m": dict(seed=4, kind=KIND_GAUSS, B=1, L=1048576, H_q=32, H_kv=8, d=128,
                      d_idx=128, plant_amp=2.0)},
    )[name]
    base.update(over)
    planted = base.pop("planted", None)
    w = Workload(name=name, **base)
    if w.kind == KIND_GAUSS:
        w.q_off = 1.0 / math.sqrt(w.d_idx)
    if planted is None:
        nb = w.nb
        if name == "tiny":
            planted = _plant_count(w.seed, w.B, nb, 4, 0, min(16, nb))
        elif name == "32k":
            planted = _plant_fraction(w.seed, w.B, nb, 500)
        elif name == "128k":
            planted = _plant_count(w.seed, w.B, nb, 4, 0, max(1, nb // 4))
        elif name == "decode":
            planted = _plant_count(w.seed, w.B, nb, 4, 0, max(1, nb - 1))
        else:
            planted = _plant_fraction(w.seed, w.B, nb, 100)
    w.planted = np.ascontiguousarray(planted, dtype=np.uint8)
    return w


def page_table(w: Workload, permute: bool = True) -> np.ndarray:
    """[B, nb] int32 page table over B * nb physical pages; a seeded
    permutation when `permute`, else the identity (page = s * nb + b)."""
    P = w.B * w.nb
    ident = np.arange(P, dtype=np.int64)
    if permute:
        k = key(w.seed, T_PERM)
        rnd = np.array([draw(k, i, 3) for i in range(P)], dtype=np.uint64)
        ident = np.argsort(rnd, kind="stable")
    return ident.astype(np.int32).reshape(w.B, w.nb)


# ---------------------------------------------------------------- host fill
_host = None


def _host_lib():
    global _host
    if _host is None:
        path = os.path.join(HERE, "libsynth_host.so")
        if not os.path.exists(path):
            from . import build as _b
            _b.build_host()
        lib = ctypes.CDLL(path)
        lib.synth_host_fill_bf16.argtypes = [ctypes.POINTER(SynthSpec), ctypes.c_int,
                                             ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p]
        lib.synth_host_fill_e4m3.argtypes = lib.synth_host_fill_bf16.argtypes
        lib.synth_host_bf16_rne.argtypes = [ctypes.c_double]
        lib.synth_host_bf16_rne.restype = ctypes.c_uint16
        lib.synth_host_e4m3_rne.argtypes = [ctypes.c_double]
        lib.synth_host_e4m3_rne.restype = ctypes.c_uint8
        lib.synth_host_gauss.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_uint64]
        lib.synth_host_gauss.restype = ctypes.c_double
        lib.synth_host_draw.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_uint64,
                                        ctypes.c_uint32]
        lib.synth_host_draw.restype = ctypes.c_uint64
        lib.synth_host_spec_size.restype = ctypes.c_size_t
        assert lib.synth_host_spec_size() == ctypes.sizeof(SynthSpec)
        _host = lib
    return _host


def _dims(w: Workload, tensor: int):
    """(H, D) of a tensor in the logical [B, L, H, D] layout."""
    return {T_Q: (w.H_q, w.d), T_K: (w.H_kv, w.d), T_V: (w.H_kv, w.d),
            T_QIDX: (w.n_g, w.d_idx), T_KIDX: (1, w.d_idx)}[tensor]


def host_fill(w: Workload, tensor: int, out: np.ndarray, idx0: int, count: int,
              fp8: bool = False, dst0: Optional[int] = None) -> None:
    """Write elements [idx0, idx0 + count) into out.flat[dst0 : dst0 + count]
    (dst0 defaults to idx0)."""
    lib = _host_lib()
    sp = w.spec(w.planted.ctypes.data)
    itemsize = 1 if fp8 else 2
    dst0 = idx0 if dst0 is None else dst0
    assert out.dtype.itemsize == itemsize and out.flags["C_CONTIGUOUS"]
    assert dst0 + count <= out.size
    ptr = out.ctypes.data + dst0 * itemsize
    if fp8:
        lib.synth_host_fill_e4m3(ctypes.byref(sp), tensor, idx0, count, ptr)
    else:
        lib.synth_host_fill_bf16(ctypes.byref(sp), tensor, idx0, count, ptr)


def host_tensor(w: Workload, tensor: int, fp8: bool = False) -> np.ndarray:
    """Whole tensor in logical layout [B, L, H, D] (bf16 bits or E4M3 bits)."""
    H, D = _dims(w, tensor)
    out = np.empty((w.B, w.L, H, D), dtype=np.uint8 if fp8 else np.uint16)
    host_fill(w, tensor, out, 0, out.size, fp8)
    return out


def host_rows(w: Workload, tensor: int, seq: int, rows) -> np.ndarray:
    """Rows t of sequence `seq`: [len(rows), H, D] bf16 bits."""
    H, D = _dims(w, tensor)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((len(rows), H, D), dtype=np.uint16)
    per = H * D
    tmp = np.empty(per, dtype=np.uint16)
    lib = _host_lib()
    sp = w.spec(w.planted.ctypes.data)
    for i, t in enumerate(rows):
        idx0 = (seq * w.L + int(t)) * per
        lib.synth_host_fill_bf16(ctypes.byref(sp), tensor, idx0, per, tmp.ctypes.data)
        out[i] = tmp.reshape(H, D)
    return out


def host_sparse_blocks(w: Workload, tensor: int, blocks_per_seq, fp8: bool = False) -> np.ndarray:
    """Full-size logical tensor [B, L, H, D] that holds real values only in the
    listed blocks of each sequence (zeros elsewhere; the zero pages are never
    touched, so the host memory used is about the filled part)."""
    H, D = _dims(w, tensor)
    out = np.zeros((w.B, w.L, H, D), dtype=np.uint8 if fp8 else np.uint16)
    per = H * D
    for s, blocks in enumerate(blocks_per_seq):
        for b in sorted(set(int(x) for x in blocks if x >= 0)):
            t0 = b * w.Bk
            t1 = min(w.L, t0 + w.Bk)
            host_fill(w, tensor, out, (s * w.L + t0) * per, (t1 - t0) * per, fp8)
    return out


def host_paged(w: Workload, tensor: int, blocks_per_seq=None, fp8: bool = False) -> np.ndarray:
    """Identity-paged cache [B * nb, H, Bk, D] (page = s * nb + b, head-major
    pages). Holds every block when blocks_per_seq is None, else only the listed
    blocks of each sequence (zeros elsewhere; untouched zero pages cost no host
    memory)."""
    H, D = _dims(w, tensor)
    dt = np.uint8 if fp8 else np.uint16
    out = np.zeros((w.B * w.nb, H, w.Bk, D), dtype=dt)
    per = H * D
    tmp = np.empty(w.Bk * per, dtype=dt)
    for s in range(w.B):
        blocks = range(w.nb) if blocks_per_seq is None else \
            sorted(set(int(x) for x in blocks_per_seq[s] if x >= 0))
        for b in blocks:
            t0, t1 = b * w.Bk, min(w.L, (b + 1) * w.Bk)
            n = (t1 - t0) * per
            host_fill(w, tensor, tmp, (s * w.L + t0) * per, n, fp8, dst0=0)
            out[s * w.nb + b, :, :t1 - t0] = tmp[:n].reshape(t1 - t0, H, D).transpose(1, 0, 2)
    return out


# -------------------------------------------------------------- device fill
_dev = None


def _dev_lib():
    global _dev
    if _dev is None:
        path = os.path.join(HERE, "libsynth_dev.so")
        if not os.path.exists(path):
            raise RuntimeError("libsynth_dev.so is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        lib.synth_dev_fill_bf16.argtypes = [ctypes.POINTER(SynthSpec), ctypes.c_int,
                                            ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p,
                                            ctypes.c_void_p]
        lib.synth_dev_fill_paged.argtypes = [ctypes.POINTER(SynthSpec), ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                             ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_dev_spec_size.restype = ctypes.c_size_t
        assert lib.synth_dev_spec_size() == ctypes.sizeof(SynthSpec)
        _dev = lib
    return _dev


def device_tensor(w: Workload, tensor: int, device="cuda"):
    """Whole tensor [B*L, H, D] (prefill: [N, H, D]) as a torch bf16 tensor."""
    import torch
    H, D = _dims(w, tensor)
    out = torch.empty((w.B * w.L, H, D), dtype=torch.bfloat16, device=device)
    planted = torch.from_numpy(w.planted).to(device)
    sp = w.spec(planted.data_ptr())
    stream = torch.cuda.current_stream(out.device).cuda_stream
    rc = _dev_lib().synth_dev_fill_bf16(ctypes.byref(sp), tensor, 0, out.numel(),
                                        out.data_ptr(), stream)
    if rc != 0:
        raise RuntimeError("synth device fill failed")
    torch.cuda.current_stream(out.device).synchronize()
    return out


def device_rows(w: Workload, tensor: int, seq_rows, device="cuda"):
    """Rows (s, t) of a tensor: [len(seq_rows), H, D] torch bf16 on the device."""
    import torch
    H, D = _dims(w, tensor)
    out = torch.empty((len(seq_rows), H, D), dtype=torch.bfloat16, device=device)
    planted = torch.from_numpy(w.planted).to(device)
    sp = w.spec(planted.data_ptr())
    stream = torch.cuda.current_stream(out.device).cuda_stream
    per = H * D
    for i, (s, t) in enumerate(seq_rows):
        rc = _dev_lib().synth_dev_fill_bf16(ctypes.byref(sp), tensor, (s * w.L + t) * per, per,
                                            out[i].data_ptr(), stream)
        if rc != 0:
            raise RuntimeError("synth device fill failed")
    torch.cuda.current_stream(out.device).synchronize()
    return out


def device_paged(w: Workload, tensor: int, table, fp8: bool = False, device="cuda"):
    """Paged cache [B*nb pages, H, Bk, D] (head-major pages) placed by `table`
    ([B, nb] int32 torch tensor on the device); bf16, or E4M3 bits as
    torch.uint8 when fp8."""
    import torch
    H, D = _dims(w, tensor)
    P = w.B * w.nb
    dtype = torch.uint8 if fp8 else torch.bfloat16
    out = torch.zeros((P, H, w.Bk, D), dtype=dtype, device=device)
    planted = torch.from_numpy(w.planted).to(device)
    sp = w.spec(planted.data_ptr())
    stream = torch.cuda.current_stream(out.device).cuda_stream
    rc = _dev_lib().synth_dev_fill_paged(ctypes.byref(sp), tensor, H, D, int(fp8),
                                         table.data_ptr(), table.shape[1], out.data_ptr(), stream)
    if rc != 0:
        raise RuntimeError("synth paged fill failed")
    torch.cuda.current_stream(out.device).synchronize()
    return out
