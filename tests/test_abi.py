"""CPU tests of the C ABI: the library loads, exports every declared entry
point, and rejects bad arguments with status codes before launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_gqa_index_gb300 as m
    return m


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_\w+)\s*\(", src)))


def test_header_symbols_exported(msa):
    names = declared()
    assert len(names) >= 12
    lib = ctypes.CDLL(msa.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
        assert n in msa.EXPORTS, n


def test_status_strings(msa):
    for code, name in [(0, "MSA_OK"), (-1, "MSA_ERR_INVALID_ARG"), (-2, "MSA_ERR_UNSUPPORTED"),
                       (-3, "MSA_ERR_WORKSPACE"), (-4, "MSA_ERR_CUDA"), (-5, "MSA_ERR_TIMEOUT")]:
        assert msa.msa_status_string(code) == name
    assert msa.version() == 0x000100


FAKE = 0x10000  # aligned, never dereferenced: every call below fails its checks first


def test_index_select_rejects(msa):
    f = msa._index_select
    assert f(None, FAKE, 10, 1, 64, 128, 16, FAKE, None, None, 0, None) == -1  # null q_idx
    assert f(FAKE, FAKE, -1, 1, 64, 128, 16, FAKE, None, None, 0, None) == -1  # N < 0
    assert f(FAKE + 4, FAKE, 10, 1, 64, 128, 16, FAKE, None, None, 0, None) == -1  # misaligned
    assert f(FAKE, FAKE, 10, 1, 64, 64, 16, FAKE, None, None, 0, None) == -2  # Bk != 128
    assert f(FAKE, FAKE, 10, 1, 64, 128, 17, FAKE, None, None, 0, None) == -2  # k > 16
    assert f(FAKE, FAKE, 10, 1, 96, 128, 16, FAKE, None, None, 0, None) == -2  # d_idx
    assert f(FAKE, FAKE, 0, 1, 64, 128, 16, FAKE, None, None, 0, None) == 0   # empty: no-op


def test_topk_rejects(msa):
    f = msa._topk
    assert f(FAKE, 300, 2, 2, 128, 16, 0, None, FAKE, None) == -1   # row 299 needs block 2
    assert f(FAKE, 10, 2, 4, 128, 0, 0, None, FAKE, None) == -1     # k < 1
    assert f(FAKE, 10, 2, 4, 128, 20, 0, None, FAKE, None) == -2    # k > 16
    assert f(None, 10, 2, 4, 128, 16, 0, None, FAKE, None) == -1


def test_sparse_attn_rejects_and_workspace(msa):
    f = msa._sparse_attn
    args = lambda **kw: [kw.get(n, d) for n, d in [  # noqa: E731
        ("q", FAKE), ("k", FAKE), ("v", FAKE), ("ids", FAKE), ("N", 1000), ("H_q", 8),
        ("H_kv", 2), ("d", 128), ("Bk", 128), ("topk", 16), ("scale", 0.1), ("out", FAKE),
        ("lse", None), ("ws", FAKE), ("wsb", 0), ("st", None)]]
    assert f(*args(H_q=6, H_kv=4)) == -1          # H_q % H_kv
    assert f(*args(d=96)) == -2
    assert f(*args(H_q=12, H_kv=4)) == -2         # G = 3 does not divide 128
    assert f(*args(out=None)) == -1
    assert f(*args(wsb=100)) == -3                # too small for a single row
    w1 = msa.msa_sparse_attn_workspace_bytes(1, 1000, 8, 2, 128)
    wN = msa.msa_sparse_attn_workspace_bytes(1000, 1000, 8, 2, 128)
    assert 0 < w1 < wN
    assert msa.msa_sparse_attn_workspace_bytes(5000, 1000, 8, 2, 128) == wN
    # partials dominate: chunk * H_q * k * (d * 2 + 4) bytes
    assert wN >= 1000 * 8 * 16 * (128 * 2 + 4)


def test_decode_rejects(msa):
    f = msa._decode
    base = [FAKE, FAKE, FAKE, 0, None, None, FAKE, FAKE, FAKE, 4, 10, 32, 8, 128, 128, 16, 0.1,
            FAKE, None, FAKE, 1 << 30, None]
    a = list(base); a[3] = 7
    assert f(*a) == -1                             # bad kv dtype
    a = list(base); a[3] = 1
    assert f(*a) == -1                             # E4M3 without scales
    a = list(base); a[19] = None
    assert f(*a) == -3                             # no workspace
    a = list(base); a[11], a[12] = 32, 2
    assert f(*a) == -2                             # G = 16 > 8
    g = msa._index_dec
    assert g(FAKE, FAKE, FAKE, FAKE, 4, 10, 9, 128, 128, 16, FAKE, None, FAKE, 1 << 20, None) == -2
    assert g(FAKE, FAKE, FAKE, FAKE, 4, 10, 8, 128, 128, 16, FAKE, None, None, 0, None) == -3
    # rows of 1025 scores padded to 1028 (16-byte aligned rows)
    assert msa.msa_index_select_decode_workspace_bytes(64, 1025, 8) == 64 * 1028 * 8 * 4


def test_decode_index_fp8_rejects(msa):
    g = msa._index_dec_fp8
    # q_idx, k_idx_pages, page_table, seq_lens, B, max_pages, n_g, d_idx, Bk, k, ids, scores,
    # score_scale, ws, ws_bytes, stream
    assert g(FAKE, FAKE, FAKE, FAKE, 4, 10, 9, 128, 128, 16, FAKE, None, 1.0, FAKE, 1 << 20,
             None) == -2                                             # 9 groups
    assert g(FAKE, FAKE, FAKE, FAKE, 4, 10, 8, 96, 128, 16, FAKE, None, 1.0, FAKE, 1 << 20,
             None) == -2                                             # d_idx
    assert g(FAKE, FAKE, FAKE, FAKE, 4, 10, 8, 128, 128, 16, FAKE, None, 1.0, None, 0,
             None) == -3                                             # no scores, no workspace
    assert g(None, FAKE, FAKE, FAKE, 4, 10, 8, 128, 128, 16, FAKE, None, 1.0, FAKE, 1 << 20,
             None) == -1
    assert g(FAKE, FAKE, FAKE, FAKE, 0, 10, 8, 128, 128, 16, FAKE, None, 1.0, None, 0,
             None) == 0                                              # empty batch


def test_decode_index_nvfp4_rejects(msa):
    g = msa._index_dec_fp4
    # q_idx, codes, scales, page_table, seq_lens, B, max_pages, n_g, d_idx, Bk, k, ids, scores,
    # score_scale, ws, ws_bytes, stream
    assert g(FAKE, FAKE, None, FAKE, FAKE, 4, 10, 8, 128, 128, 16, FAKE, None, 1.0, FAKE, 1 << 20,
             None) == -1                                             # no scales
    assert g(FAKE, FAKE, FAKE + 8, FAKE, FAKE, 4, 10, 8, 128, 128, 16, FAKE, None, 1.0, FAKE,
             1 << 20, None) == -1                                    # misaligned scales
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, 9, 128, 128, 16, FAKE, None, 1.0, FAKE, 1 << 20,
             None) == -2                                             # 9 groups
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, 8, 96, 128, 16, FAKE, None, 1.0, FAKE, 1 << 20,
             None) == -2                                             # d_idx
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, 8, 128, 128, 16, FAKE, None, 1.0, None, 0,
             None) == -3                                             # no workspace


def test_decode_nvfp4_rejects(msa):
    f = msa._decode_fp4
    # q, k_codes, k_scales, v_codes, v_scales, page_table, seq_lens, ids, B, max_pages, H_q,
    # H_kv, d, Bk, k, scale, out, lse, ws, ws_bytes, stream
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, 32, 8, 128, 128, 16, 0.1,
            FAKE, None, FAKE, 1 << 30, None]
    a = list(base); a[4] = None
    assert f(*a) == -1                             # no V scales
    a = list(base); a[2] = FAKE + 8
    assert f(*a) == -1                             # misaligned K scales
    a = list(base); a[10], a[11] = 32, 2
    assert f(*a) == -2                             # G = 16 > 8
    a = list(base); a[12] = 96
    assert f(*a) == -2                             # d not 64 or 128
    a = list(base); a[13] = 64
    assert f(*a) == -2                             # Bk != 128
    a = list(base); a[18] = None
    assert f(*a) == -3                             # no workspace
    a = list(base); a[8] = 0
    assert f(*a) == 0                              # no sequences: nothing to do


def test_index_nvfp4_rejects(msa):
    f = msa._index_fp4
    ws = msa.msa_index_select_nvfp4_workspace_bytes(4096, 8, 128)
    # the decoded q_idx and k_idx rows (bf16), each area rounded up to 256 bytes
    assert ws == 4096 * 8 * 128 * 2 + 4096 * 128 * 2
    assert msa.msa_index_select_nvfp4_workspace_bytes(3, 1, 64) == 512 + 512
    # q_codes, q_scales, k_codes, k_scales, N, n_g, d_idx, Bk, k, ids, scores, ws, ws_bytes,
    # stream
    base = [FAKE, FAKE, FAKE, FAKE, 4096, 8, 128, 128, 16, FAKE, None, FAKE, ws, None]
    a = list(base); a[3] = None
    assert f(*a) == -1                             # no k_idx scales
    a = list(base); a[2] = FAKE + 8
    assert f(*a) == -1                             # misaligned k_idx codes
    a = list(base); a[11] = None
    assert f(*a) == -1                             # no workspace
    a = list(base); a[6] = 96
    assert f(*a) == -2                             # d_idx not 64 or 128
    a = list(base); a[7] = 64
    assert f(*a) == -2                             # Bk != 128
    a = list(base); a[8] = 17
    assert f(*a) == -2                             # k > 16
    a = list(base); a[12] = ws - 1
    assert f(*a) == -3                             # workspace one byte short
    a = list(base); a[4] = 0
    assert f(*a) == 0                              # no queries: nothing to do


def test_wait_limit_roundtrip(msa):
    old = msa.msa_set_wait_limit(123)
    assert msa.msa_set_wait_limit(old) == 123


def _shared_pass_bytes(chunk, nb, H_kv=8, k=16, G=4, d=128):
    """Workspace the single-sequence main branch adds for its shared-block pass:
    a row mask, 16 shared ids per (query tile, group) and qt records per (query
    tile, group) after the block-outer partials, each area rounded up to 256 B."""
    a256 = lambda x: (x + 255) // 256 * 256
    qt, rec = 128 // G, G * d * 2 + G * 4
    n_qt = -(-chunk // qt)
    tiles = (chunk * H_kv * k + qt - 1) // qt + H_kv * nb
    return a256(chunk * H_kv * 4) + a256(n_qt * H_kv * 16 * 4) + \
        a256((tiles * qt + n_qt * H_kv * qt) * rec) - a256(tiles * qt * rec)


def test_varlen_rejects(msa):
    """Varlen prefill validates the cumulative offsets, the sizes and (for the
    main branch) the per-sequence alignment on the host, before anything is
    launched."""
    import ctypes as C

    def cu(*xs):
        a = (C.c_int64 * len(xs))(*xs)
        return C.cast(a, C.c_void_p), a

    fi, fa = msa._index_varlen, msa._attn_varlen
    p, keep = cu(1, 5)  # first offset must be 0
    assert fi(FAKE, FAKE, p, 1, 8, 128, 128, 16, FAKE, None) == -1
    p, keep = cu(0, 7, 5)  # offsets must not decrease
    assert fi(FAKE, FAKE, p, 2, 8, 128, 128, 16, FAKE, None) == -1
    assert fi(FAKE, FAKE, None, 1, 8, 128, 128, 16, FAKE, None) == -1  # no offsets
    p, keep = cu(0)
    assert fi(FAKE, FAKE, p, 0, 8, 128, 128, 16, FAKE, None) == 0  # no sequences
    p, keep = cu(0, 0, 0)
    assert fi(FAKE, FAKE, p, 2, 8, 128, 128, 16, FAKE, None) == 0  # only empty sequences
    p, keep = cu(0, 100)
    assert fi(FAKE, FAKE, p, 1, 8, 128, 64, 16, FAKE, None) == -2   # Bk != 128
    assert fi(FAKE, FAKE, p, 1, 8, 96, 128, 16, FAKE, None) == -2   # d_idx not 64 or 128
    assert fi(FAKE, FAKE, p, 1, 8, 128, 128, 17, FAKE, None) == -2  # k above the largest top-k
    p, keep = cu(0, 1 << 28)
    assert fi(FAKE, FAKE, p, 1, 8, 128, 128, 16, FAKE, None) == -2  # 2^31 (t, g) rows
    p, keep = cu(0, 100)
    assert fi(None, FAKE, p, 1, 8, 128, 128, 16, FAKE, None) == -1  # null q_idx
    # main branch: same offset rules, then the single-sequence shape rules
    args = (FAKE, FAKE, FAKE, FAKE)
    p, keep = cu(3, 10)
    assert fa(*args, p, 1, 32, 8, 128, 128, 16, 0.1, FAKE, None, FAKE, 1 << 20, None) == -1
    p, keep = cu(0, 10)
    assert fa(*args, p, 1, 12, 4, 128, 128, 16, 0.1, FAKE, None, FAKE, 1 << 20, None) == -2  # G=3
    assert fa(*args, p, 1, 32, 8, 96, 128, 16, 0.1, FAKE, None, FAKE, 1 << 20, None) == -2
    assert fa(*args, p, 1, 32, 8, 128, 64, 16, 0.1, FAKE, None, FAKE, 1 << 20, None) == -2
    assert fa(*args, p, 1, 32, 8, 128, 128, 16, 0.1, FAKE, None, FAKE, 1000, None) == -3
    # workspace query: 0 for bad offsets; one pass = 8 bytes per query and per
    # block of the sequences with queries, plus the bucketing of all rows over
    # those blocks (here 3 + 6 blocks, like one sequence of 9 blocks)
    p, keep = cu(0, 7, 5)
    assert msa._ws_attn_varlen(p, 2, 32, 8, 128, 128, 16) == 0
    p, keep = cu(0, 300, 300, 1000)
    # the single-sequence call also holds the shared-block pass; packed sequences do not
    assert msa._ws_attn_varlen(p, 3, 32, 8, 128, 128, 16) == \
        8192 + 256 + msa.msa_sparse_attn_workspace_bytes(1000, 9 * 128, 32, 8, 128) - \
        _shared_pass_bytes(1000, 9)


def test_paged_rejects(msa):
    """Paged prefill checks the query offsets, the cached lengths against the
    page table's width and the shapes on the host."""
    import ctypes as C

    def arr(*xs):
        a = (C.c_int64 * len(xs))(*xs)
        return C.cast(a, C.c_void_p), a

    fi, fa, fw = msa._index_paged, msa._attn_paged, msa._ws_attn_paged
    cu, k1 = arr(0, 100, 150)
    kv, k2 = arr(1000, 50)
    # index: q_idx, k_idx_pages, P, page_table, max_pages, cu_q, kv_lens, B, n_g, d_idx, Bk, k
    bad, k3 = arr(1000, 40)   # 50 queries but 40 keys
    assert fi(FAKE, FAKE, 64, FAKE, 8, cu, bad, 2, 8, 128, 128, 16, FAKE, None) == -1
    big, k4 = arr(1025, 50)   # 1025 keys do not fit 8 pages of 128
    assert fi(FAKE, FAKE, 64, FAKE, 8, cu, big, 2, 8, 128, 128, 16, FAKE, None) == -1
    assert fi(FAKE, FAKE, 64, None, 8, cu, kv, 2, 8, 128, 128, 16, FAKE, None) == -1
    assert fi(FAKE, FAKE, 64, FAKE, 8, cu, kv, 2, 8, 128, 64, 16, FAKE, None) == -2
    assert fi(FAKE, FAKE, 0, FAKE, 8, cu, kv, 2, 8, 128, 128, 16, FAKE, None) == -1
    empty, k5 = arr(0, 0, 0)
    assert fi(FAKE, FAKE, 64, FAKE, 8, empty, kv, 2, 8, 128, 128, 16, FAKE, None) == 0
    # main branch: q, k_pages, v_pages, P, page_table, max_pages, ids, cu_q, kv_lens, B, H_q,
    # H_kv, d, Bk, topk, scale, out, lse, ws, ws_bytes, stream
    base = [FAKE, FAKE, FAKE, 64, FAKE, 8, FAKE, cu, kv, 2, 32, 8, 128, 128, 16, 0.1, FAKE, None,
            FAKE, 1 << 20, None]
    a = list(base); a[8] = bad
    assert fa(*a) == -1
    a = list(base); a[4] = None
    assert fa(*a) == -1
    a = list(base); a[10] = 24
    assert fa(*a) == -2                            # G = 3
    a = list(base); a[19] = 64
    assert fa(*a) == -3
    assert fw(cu, bad, 2, 8, 32, 8, 128, 128, 16) == 0
    # one pass: 150 queries and 8 + 1 blocks of the two sequences, with the
    # per-tile query bases of paged K / V
    assert fw(cu, kv, 2, 8, 32, 8, 128, 128, 16) > \
        msa.msa_sparse_attn_workspace_bytes(150, 9 * 128, 32, 8, 128) - _shared_pass_bytes(150, 9)


def test_index_fp8_rejects(msa):
    f = msa._index_fp8
    assert f(None, FAKE, 10, 1, 128, 128, 16, FAKE, None, 1.0, None) == -1   # null q_idx
    assert f(FAKE + 8, FAKE, 10, 1, 128, 128, 16, FAKE, None, 1.0, None) == -1  # misaligned
    assert f(FAKE, FAKE, 10, 1, 64, 128, 16, FAKE, None, 1.0, None) == -2    # d_idx != 128
    assert f(FAKE, FAKE, 10, 1, 128, 64, 16, FAKE, None, 1.0, None) == -2    # Bk != 128
    assert f(FAKE, FAKE, 0, 1, 128, 128, 16, FAKE, None, 1.0, None) == 0     # empty: no-op


def test_kl_teacher_rejects(msa):
    f = msa._kl
    # q, k, q_idx, k_idx, block_ids, lse, N, H_q, H_kv, d, d_idx, Bk, topk, scale, kl, ws, bytes
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 10, 32, 8, 128, 128, 128, 16, 0.1, FAKE, FAKE,
            1 << 40, None]
    a = list(base); a[0] = None
    assert f(*a) == -1                             # null q
    a = list(base); a[5] = FAKE + 4
    assert f(*a) == -1                             # misaligned lse
    a = list(base); a[7] = 12
    assert f(*a) == -1                             # H_q not a multiple of H_kv
    a = list(base); a[8] = 2
    assert f(*a) == -2                             # G = 16 > 8
    a = list(base); a[11] = 64
    assert f(*a) == -2                             # Bk != 128
    a = list(base); a[9] = 96
    assert f(*a) == -2                             # d
    a = list(base); a[12] = 17
    assert f(*a) == -2                             # top-k > 16
    a = list(base); a[6] = 1 << 27
    assert f(*a) == -2                             # N too large
    a = list(base); a[16] = 16
    assert f(*a) == -3                             # workspace holds no chunk of rows
    a = list(base); a[15] = None
    assert f(*a) == -1                             # no workspace
    a = list(base); a[6] = 0
    assert f(*a) == 0                              # empty: no-op
    a = list(base); a[6] = -1
    assert f(*a) == -1                             # N < 0


def test_index_project_rejects(msa):
    f = msa._index_project
    # x, w_qidx, w_kidx, N, d_model, n_groups, d_idx, q_idx, k_idx, stream
    base = [FAKE, FAKE, FAKE, 10, 4096, 8, 128, FAKE, FAKE, None]
    a = list(base); a[1] = None
    assert f(*a) == -1                             # null w_qidx
    a = list(base); a[8] = FAKE + 2
    assert f(*a) == -1                             # misaligned k_idx
    a = list(base); a[4] = 4100
    assert f(*a) == -2                             # d_model not a multiple of 8
    a = list(base); a[6] = 96
    assert f(*a) == -2                             # d_idx
    a = list(base); a[3] = 1 << 31
    assert f(*a) == -2                             # N too large
    a = list(base); a[3] = -1
    assert f(*a) == -1                             # N < 0
    a = list(base); a[3] = 0
    assert f(*a) == 0                              # empty: no-op


def test_decode_index_noalloc_rejects(msa):
    f = msa._index_dec_noalloc
    cap = msa._noalloc_max()
    assert cap == 1 << 20
    # q_idx, k_idx_pages, page_table, seq_lens, B, max_pages, n_groups, d_idx, Bk, k, ids, stream
    base = [FAKE, FAKE, FAKE, FAKE, 4, 10, 8, 128, 128, 16, FAKE, None]
    a = list(base); a[2] = None
    assert f(*a) == -1                             # null page table
    a = list(base); a[0] = FAKE + 8
    assert f(*a) == -1                             # misaligned q_idx
    a = list(base); a[8] = 64
    assert f(*a) == -2                             # Bk != 128
    a = list(base); a[9] = 17
    assert f(*a) == -2                             # k > 16
    a = list(base); a[6] = 9
    assert f(*a) == -2                             # more than 8 groups
    a = list(base); a[7] = 96
    assert f(*a) == -2                             # d_idx
    a = list(base); a[4], a[5] = 128, cap // (128 * 8) + 1
    assert f(*a) == -3                             # scores beyond the fixed array
    a = list(base); a[4] = 0
    assert f(*a) == 0                              # empty: no-op
    a = list(base); a[4] = -1
    assert f(*a) == -1                             # B < 0
