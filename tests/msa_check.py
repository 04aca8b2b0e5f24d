"""Comparison rules shared by the GPU parity tests (pure numpy; no method arithmetic).

Block selection: bit-exact where the index scores are exact in fp32 (integer
inputs). On real-valued inputs the GPU's fp32 scores may order near-ties
differently from the oracle's fp64 ones, so the GPU set may differ from the
oracle set only by swaps whose oracle block-score gap is <= rel * max(|S_x|,
|S_y|) (rel = 1e-3). Every GPU row must also be structurally valid: ascending,
no duplicates, -1 padding last, local block present, nothing after it, exactly
min(k, loc + 1) blocks.
"""
import numpy as np


def check_structure(ids, positions, Bk):
    """ids [n, n_g, k]; positions [n] (query position of each row)."""
    ids = np.asarray(ids)
    n, n_g, k = ids.shape
    for i in range(n):
        loc = int(positions[i]) // Bk
        want = min(k, loc + 1)
        for g in range(n_g):
            r = ids[i, g]
            valid = r[:want]
            assert np.all(r[want:] == -1), (i, g, r)
            assert np.all(valid >= 0), (i, g, r)
            assert np.all(np.diff(valid) > 0), (i, g, r)
            assert valid[-1] == loc, (i, g, r, loc)


def compare_selection(gpu_ids, ref_ids, ref_scores, positions, Bk, rel=1e-3):
    """Returns the number of (row, group) pairs that differ by allowed swaps."""
    gpu_ids = np.asarray(gpu_ids)
    ref_ids = np.asarray(ref_ids)
    check_structure(gpu_ids, positions, Bk)
    n, n_g, k = gpu_ids.shape
    swaps = 0
    for i in range(n):
        for g in range(n_g):
            a = set(int(x) for x in ref_ids[i, g] if x >= 0)
            b = set(int(x) for x in gpu_ids[i, g] if x >= 0)
            if a == b:
                continue
            x_only = sorted(b - a, key=lambda x: -ref_scores[i, g, x])
            y_only = sorted(a - b, key=lambda y: -ref_scores[i, g, y])
            assert len(x_only) == len(y_only), (i, g, a, b)
            for x, y in zip(x_only, y_only):
                sx, sy = ref_scores[i, g, x], ref_scores[i, g, y]
                assert abs(sx - sy) <= rel * max(abs(sx), abs(sy)), \
                    f"row {i} group {g}: block {x} (S={sx}) taken instead of {y} (S={sy})"
            swaps += 1
    return swaps


def bf16_to_np(t):
    """torch bf16 tensor -> float64 numpy."""
    return t.float().cpu().numpy().astype(np.float64)


def check_close(name, got, want, atol, rtol=0.0):
    """|got - want| <= atol + rtol * |want| everywhere; returns the largest |got - want|."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    excess = err - (atol + rtol * np.abs(want))
    worst = np.unravel_index(np.argmax(excess), err.shape) if err.size else ()
    assert err.size == 0 or excess.max() <= 0.0, \
        f"{name}: |err| {err[worst]:.3e} > {atol} + {rtol} |want| at {worst} " \
        f"(got {got[worst]}, want {want[worst]})"
    return float(err.max()) if err.size else 0.0
