"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test fixes part of the oracle against something it does not compute
itself: a library routine (torch SDPA, numpy matmul, torch dtype casts), a
closed form, a hand-worked fixture, an independently coded brute force, or an
invariant the pages state (softmax keeps order; the local block is always
kept; one block set per GQA group).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(x):
    """float array -> bf16 bits via torch (round to nearest even)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()


def rand_bf16(rng, shape, scale=1.0):
    return bf16_bits(rng.standard_normal(shape) * scale)


def rand_int_bf16(rng, shape, lo=-4, hi=4):
    return bf16_bits(rng.integers(lo, hi + 1, size=shape).astype(np.float32))


# ----------------------------------------------------------------- decoders

def test_bf16_decoder_exhaustive_vs_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    lib = oracle.lib()
    mine = np.array([lib.oracle_bf16_to_f64(int(c)) for c in codes])
    fin = np.isfinite(ref)
    assert np.array_equal(mine[fin], ref[fin])
    assert np.array_equal(np.isnan(mine), np.isnan(ref))


def test_e4m3_decoder_exhaustive_vs_torch_and_ocp():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    mine = np.array([oracle.e4m3_to_f64(int(c)) for c in codes])
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(mine[fin], ref[fin])
    # OCP E4M3 landmarks: max finite 448, min subnormal 2^-9, min normal 2^-6, NaN at 0x7F/0xFF
    assert oracle.e4m3_to_f64(0x7E) == 448.0
    assert oracle.e4m3_to_f64(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_f64(0x08) == 2.0 ** -6
    assert math.isnan(oracle.e4m3_to_f64(0x7F)) and math.isnan(oracle.e4m3_to_f64(0xFF))
    assert oracle.e4m3_to_f64(0xB8) == -1.0


# ------------------------------------------------------------- index branch

def test_golden_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "index_hand_example.json")))
    sh = g["shape"]
    kidx = bf16_bits(np.array(g["k_idx"], dtype=np.float32))
    qidx = bf16_bits(np.array(g["q_idx"], dtype=np.float32))
    rows = np.arange(sh["N"])
    ids, sc = oracle.index_select(qidx, rows, kidx, sh["Bk"], sh["k"], nb_out=4, want_scores=True)
    for t, exp in g["expected_ids"].items():
        assert ids[int(t)].tolist() == exp, t
    assert sc[7].tolist() == g["expected_block_max_row7"]
    assert np.isneginf(sc[0, :, 1:]).all()  # invisible blocks


def _golden_scores(rows):
    """JSON numbers, with "-0" for a negative zero, as fp32."""
    return np.array([[[(-0.0 if v == "-0" else float(v)) for v in g] for g in r] for r in rows],
                    dtype=np.float32)


def test_golden_topk_hand_example():
    """The standalone top-k step on hand-worked block scores: q_offset > 0, two
    groups, ties among candidates, -0 against +0, a local block with the
    highest score (forced, never ranked), blocks after the query holding the
    largest values (never read), and rows whose local block is the last one."""
    g = json.load(open(os.path.join(GOLDEN, "topk_hand_example.json")))
    sh = g["shape"]
    S = _golden_scores(g["block_scores"])
    assert S.shape == (sh["N"], sh["n_g"], sh["nb"])
    assert np.signbit(S[0, 1, 1]) and not np.signbit(S[0, 1, 2])  # the -0 / +0 pair
    rows = sh["q_offset"] + np.arange(sh["N"])
    ids = oracle.topk_blocks(S, rows, sh["Bk"], sh["k"])
    assert ids.tolist() == g["expected_ids"]


def test_golden_attn_hand_example():
    """Main-branch attention on hand-worked values: scores that are whole
    multiples of ln 2 make every softmax weight a power of two, so o and
    exp(lse) are exact fractions. Pins the causal cut inside the local block
    (rows 2 and 4), the use of only the selected blocks (row 5 skips the block
    with the largest scores), the scale, the natural-log LSE and two query heads
    sharing one group."""
    from fractions import Fraction
    g = json.load(open(os.path.join(GOLDEN, "attn_hand_example.json")))
    sh = g["shape"]
    tok = g["tokens"]
    to_bits = lambda a: (np.asarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    K = to_bits(tok["K"]).reshape(sh["N"], sh["H_kv"], sh["d"])
    V = to_bits(tok["V"]).reshape(sh["N"], sh["H_kv"], sh["d"])
    q = to_bits(np.broadcast_to(np.asarray(g["q_heads"], dtype=np.float32),
                                (sh["N"], sh["H_q"], sh["d"])))
    # K rows follow the stated scores kappa (head 0 scores kappa, head 1 1 - kappa)
    Kf = np.asarray(tok["K"], dtype=np.float64)
    assert np.array_equal(Kf @ np.asarray(g["q_heads"][0]), tok["kappa"])
    ids = np.asarray(g["ids"], dtype=np.int32)
    o, lse = oracle.sparse_attn(q, np.arange(sh["N"]), K, V, ids, sh["Bk"], math.log(2.0))
    want_o = np.vectorize(lambda x: float(Fraction(x)))(np.asarray(g["expected_o"]))
    want_lse = np.vectorize(lambda x: math.log(Fraction(x)))(np.asarray(g["expected_exp_lse"]))
    assert np.allclose(o, want_o, rtol=1e-12, atol=1e-12), (o, want_o)
    assert np.allclose(lse, want_lse, rtol=0, atol=1e-12), (lse, want_lse)


@pytest.mark.parametrize("Bk,N,q_offset,n_g,k", [
    (8, 40, 0, 2, 3), (8, 57, 96, 3, 4), (16, 64, 300, 2, 16), (4, 33, 21, 4, 5),
    (128, 200, 2000, 2, 16), (2, 30, 7, 1, 2)])
def test_topk_blocks_equals_index_select_on_integer_inputs(Bk, N, q_offset, n_g, k):
    """The top-k step alone, given the block scores index_select pools, picks
    what index_select picks (itself pinned to the brute force above). Integer
    inputs make every score an integer below 2^24, so the fp32 block scores are
    exact, and many scores tie. Rows sit at q_offset + i with n_g groups each."""
    rng = np.random.default_rng(7 * N + Bk + q_offset)
    d_idx = 8
    L = q_offset + N
    qidx = rand_int_bf16(rng, (N, n_g, d_idx), -2, 2)
    kidx = rand_int_bf16(rng, (L, d_idx), -2, 2)
    rows = q_offset + np.arange(N)
    nb = (L + Bk - 1) // Bk
    ids, sc = oracle.index_select(qidx, rows, kidx, Bk, k, nb_out=nb, want_scores=True)
    vis = np.isfinite(sc)
    assert np.array_equal(sc[vis], sc[vis].astype(np.float32).astype(np.float64))
    got = oracle.topk_blocks(sc.astype(np.float32), rows, Bk, k)
    assert np.array_equal(got, ids)
    # scores past each row's local block do not matter
    noisy = sc.astype(np.float32)
    noisy[~vis] = 1e30
    assert np.array_equal(oracle.topk_blocks(noisy, rows, Bk, k), ids)


def test_topk_blocks_skips_rows_past_the_score_rows():
    """A row whose local block lies beyond the given nb blocks is left untouched."""
    S = np.zeros((3, 2, 4), dtype=np.float32)
    ids = oracle.topk_blocks(S, np.array([0, 511, 512]), 128, 2)
    assert ids[0].tolist() == [[0, -1], [0, -1]]
    assert ids[1].tolist() == [[0, 3], [0, 3]]
    assert (ids[2] == -2).all()  # the wrapper's fill value: not written


@pytest.mark.parametrize("Bk,N,n_g,k", [
    (1, 23, 1, 1), (1, 40, 2, 3), (2, 33, 1, 2), (2, 64, 4, 3), (4, 61, 2, 16),
    (8, 64, 4, 3), (4, 64, 1, 2), (8, 57, 2, 1), (2, 50, 4, 16)])
def test_index_matches_brute_force(Bk, N, n_g, k):
    rng = np.random.default_rng(1000 * Bk + N + 7 * k)
    d_idx = 8
    # integer inputs make many exact ties, so the tie-break is exercised
    qidx = rand_int_bf16(rng, (N, n_g, d_idx), -2, 2)
    kidx = rand_int_bf16(rng, (N, d_idx), -2, 2)
    rows = np.arange(N)
    a = oracle.index_select(qidx, rows, kidx, Bk, k)
    b = oracle.index_brute(qidx, rows, kidx, Bk, k)
    assert np.array_equal(a, b)


def test_token_level_special_case_by_numpy():
    """Bk = 1: the method reduces to token-level top-k with a forced diagonal,
    i.e. t itself plus the k-1 best earlier tokens (numpy matmul + lexsort)."""
    rng = np.random.default_rng(5)
    N, n_g, d_idx, k = 48, 2, 16, 5
    qidx = rand_bf16(rng, (N, n_g, d_idx))
    kidx = rand_bf16(rng, (N, d_idx))
    ids = oracle.index_select(qidx, np.arange(N), kidx, 1, k)
    s = np.einsum("tgc,jc->tgj", bits_to_f64(qidx), bits_to_f64(kidx))
    for t in range(N):
        for g in range(n_g):
            earlier = np.arange(t)
            order = earlier[np.lexsort((earlier, -s[t, g, :t]))] if t else earlier
            want = sorted(list(order[:k - 1]) + [t])
            want = want + [-1] * (k - len(want))
            assert ids[t, g].tolist() == want


def test_block_scores_match_numpy_pool():
    """a1-a2: block scores equal a numpy causal matmul followed by a reshape max."""
    rng = np.random.default_rng(9)
    N, n_g, d_idx, Bk = 96, 3, 32, 16
    qidx = rand_bf16(rng, (N, n_g, d_idx))
    kidx = rand_bf16(rng, (N, d_idx))
    nb = N // Bk
    _, sc = oracle.index_select(qidx, np.arange(N), kidx, Bk, 4, nb_out=nb, want_scores=True)
    s = np.einsum("tgc,jc->tgj", bits_to_f64(qidx), bits_to_f64(kidx))
    mask = np.arange(N)[None, None, :] > np.arange(N)[:, None, None]
    s = np.where(mask, -np.inf, s)
    pooled = s.reshape(N, n_g, nb, Bk).max(axis=-1)
    assert np.allclose(sc, pooled, rtol=1e-13, atol=1e-12, equal_nan=False)


def test_exp_free_equals_probability_ranking():
    """Kernel co-design: ranking raw block scores picks the same blocks as
    ranking their softmax probabilities (done here in log space, exactly)."""
    rng = np.random.default_rng(11)
    N, n_g, d_idx, Bk, k = 256, 2, 32, 8, 6
    qidx = rand_bf16(rng, (N, n_g, d_idx), 2.0)
    kidx = rand_bf16(rng, (N, d_idx), 2.0)
    nb = N // Bk
    ids, sc = oracle.index_select(qidx, np.arange(N), kidx, Bk, k, nb_out=nb, want_scores=True)
    for t in range(0, N, 5):
        loc = t // Bk
        for g in range(n_g):
            S = sc[t, g, :loc + 1]
            lp = S - (S.max() + np.log(np.exp(S - S.max()).sum()))  # log-softmax
            cand = np.arange(loc)
            order = cand[np.lexsort((cand, -lp[:loc]))]
            want = sorted(list(order[:k - 1]) + [loc])
            want += [-1] * (k - len(want))
            assert ids[t, g].tolist() == want


def test_ties_go_to_lower_block_id():
    N, n_g, d_idx, Bk, k = 40 * 8, 2, 16, 8, 5
    rng = np.random.default_rng(3)
    qidx = rand_int_bf16(rng, (N, n_g, d_idx))
    kidx = np.zeros((N, d_idx), dtype=np.uint16)  # every score is 0
    ids = oracle.index_select(qidx, np.arange(N), kidx, Bk, k)
    for t in range(N):
        loc = t // Bk
        want = sorted(list(range(min(k - 1, loc))) + [loc])
        want += [-1] * (k - len(want))
        assert ids[t, 0].tolist() == want and ids[t, 1].tolist() == want
    # duplicated blocks: copy block 2 into blocks 5 and 7 -> on a tie the lower id wins
    kidx = rand_int_bf16(rng, (N, d_idx))
    for b in (5, 7):
        kidx[b * Bk:(b + 1) * Bk] = kidx[2 * Bk:3 * Bk]
    ids, sc = oracle.index_select(qidx, np.arange(N), kidx, Bk, 2, nb_out=40, want_scores=True)
    for t in range(8 * Bk, N):
        for g in range(n_g):
            assert sc[t, g, 2] == sc[t, g, 5] == sc[t, g, 7]
            assert ids[t, g, 0] not in (5, 7)


def test_structural_invariants_tiny_workload():
    w = synth.make("tiny", L=1024)
    qidx = synth.host_tensor(w, synth.T_QIDX)[0]
    kidx = synth.host_tensor(w, synth.T_KIDX)[0, :, 0]
    rows = np.arange(w.N)
    ids = oracle.index_select(qidx, rows, kidx, w.Bk, w.k)
    for t in range(w.N):
        loc = t // w.Bk
        for g in range(w.n_g):
            r = ids[t, g]
            valid = r[r >= 0]
            assert loc in valid
            assert valid.max() == loc
            assert len(set(valid.tolist())) == len(valid)
            assert len(valid) == min(w.k, loc + 1)
            assert np.all(np.diff(valid) > 0) and np.all(r[len(valid):] == -1)


# ------------------------------------------------------------ main branch

def sdpa_ref(q, K, V, scale):
    """torch SDPA (fp64, causal) + torch.logsumexp for the LSE."""
    qt = torch.from_numpy(bits_to_f64(q)).permute(1, 0, 2)[None]   # [1, H_q, N, d]
    H_q, H_kv = q.shape[1], K.shape[1]
    G = H_q // H_kv
    kt = torch.from_numpy(bits_to_f64(K)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    vt = torch.from_numpy(bits_to_f64(V)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    s = (qt @ kt.transpose(-1, -2)) * scale
    N = q.shape[0]
    s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), -math.inf)
    lse = torch.logsumexp(s, dim=-1)
    return o[0].permute(1, 0, 2).numpy(), lse[0].permute(1, 0).numpy()


@pytest.mark.parametrize("N", [1, 5, 127, 128, 129, 700])
def test_dense_limit_equals_sdpa(N):
    """When k covers every visible block, the main branch is dense causal GQA."""
    rng = np.random.default_rng(N)
    H_q, H_kv, d, Bk, k = 4, 2, 32, 128, 16
    q = rand_bf16(rng, (N, H_q, d))
    K = rand_bf16(rng, (N, H_kv, d))
    V = rand_bf16(rng, (N, H_kv, d))
    qidx = rand_bf16(rng, (N, H_kv, 16))
    kidx = rand_bf16(rng, (N, 16))
    rows = np.arange(N)
    ids = oracle.index_select(qidx, rows, kidx, Bk, k)
    o, lse = oracle.sparse_attn(q, rows, K, V, ids, Bk, 1 / math.sqrt(d))
    ro, rl = sdpa_ref(q, K, V, 1 / math.sqrt(d))
    assert np.allclose(o, ro, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, rl, rtol=1e-12, atol=1e-12)
    od, ld = oracle.dense_gqa(q, rows, K, V, 1 / math.sqrt(d))
    assert np.allclose(od, ro, rtol=1e-12, atol=1e-12) and np.allclose(ld, rl, rtol=1e-12, atol=1e-12)


def test_dense_limit_tiny_workload_k32():
    """The tiny workload (32 blocks) with k = 32: selection = all visible blocks."""
    w = synth.make("tiny", L=4096)
    rows = np.array([0, 1, 127, 128, 1000, 2047, 2048, 4095])
    qidx = synth.host_rows(w, synth.T_QIDX, 0, rows)
    kidx = synth.host_tensor(w, synth.T_KIDX)[0, :, 0]
    ids = oracle.index_select(qidx, rows, kidx, w.Bk, 32)
    q = synth.host_tensor(w, synth.T_Q)[0]
    K = synth.host_tensor(w, synth.T_K)[0]
    V = synth.host_tensor(w, synth.T_V)[0]
    o, lse = oracle.sparse_attn(q[rows], rows, K, V, ids, w.Bk, w.scale)
    od, ld = oracle.dense_gqa(q[rows], rows, K, V, w.scale)
    assert np.allclose(o, od, rtol=1e-12, atol=1e-12) and np.allclose(lse, ld, rtol=1e-12)
    # and the dense routine agrees with SDPA on the first 129 rows
    ro, rl = sdpa_ref(q[:129], K[:129], V[:129], w.scale)
    od2, ld2 = oracle.dense_gqa(q[:129], np.arange(129), K[:129], V[:129], w.scale)
    assert np.allclose(od2, ro, rtol=1e-12, atol=1e-12) and np.allclose(ld2, rl, rtol=1e-12)


def _random_ids(rng, rows, n_g, Bk, k):
    out = np.full((len(rows), n_g, k), -1, dtype=np.int32)
    for i, t in enumerate(rows):
        loc = t // Bk
        for g in range(n_g):
            far = rng.choice(loc, size=min(k - 1, loc), replace=False) if loc else []
            sel = sorted(list(far) + [loc])
            out[i, g, :len(sel)] = sel
    return out


def _key_set(t, ids, Bk):
    J = set()
    for b in ids:
        if b >= 0:
            J.update(j for j in range(b * Bk, (b + 1) * Bk) if j <= t)
    return sorted(J)


def test_closed_forms():
    rng = np.random.default_rng(21)
    N, H_q, H_kv, d, Bk, k = 300, 4, 2, 16, 16, 4
    scale = 0.25
    rows = np.array([0, 1, 15, 16, 17, 100, 255, 299])
    q = rand_bf16(rng, (N, H_q, d))
    K = rand_bf16(rng, (N, H_kv, d))
    ids = _random_ids(rng, rows, H_kv, Bk, k)
    # (i) constant V -> o equals that constant, whatever the selection
    c = rand_bf16(rng, (H_kv, d))
    V = np.broadcast_to(c, (N, H_kv, d)).copy()
    o, _ = oracle.sparse_attn(q[rows], rows, K, V, ids, Bk, scale)
    for h in range(H_q):
        assert np.allclose(o[:, h], bits_to_f64(c[h // 2])[None], rtol=0, atol=1e-14)
    # (ii) t = 0 -> o = v_0, lse = scale * q.k_0
    V = rand_bf16(rng, (N, H_kv, d))
    o, lse = oracle.sparse_attn(q[:1], np.array([0]), K, V, ids[:1], Bk, scale)
    for h in range(H_q):
        assert np.array_equal(o[0, h], bits_to_f64(V[0, h // 2]))
        want = scale * float(np.dot(bits_to_f64(q[0, h]), bits_to_f64(K[0, h // 2])))
        assert abs(lse[0, h] - want) < 1e-12
    # (iii) all keys equal -> o = mean of V over J, lse = scale q.k + ln |J|,
    #       and |J| = n_sel(t) = t+1 if t/Bk < k else (k-1) Bk + t mod Bk + 1
    Keq = np.broadcast_to(K[3], (N, H_kv, d)).copy()
    full_ids = np.full((len(rows), H_kv, k), -1, dtype=np.int32)
    for i, t in enumerate(rows):
        loc = t // Bk
        sel = sorted(list(range(max(0, loc - (k - 1)), loc)) + [loc])
        full_ids[i, :, :len(sel)] = sel
    o, lse = oracle.sparse_attn(q[rows], rows, Keq, V, full_ids, Bk, scale)
    for i, t in enumerate(rows):
        nsel = t + 1 if t // Bk + 1 <= k else (k - 1) * Bk + t % Bk + 1
        J = _key_set(t, full_ids[i, 0], Bk)
        assert len(J) == nsel
        for h in range(H_q):
            g = h // 2
            mean = bits_to_f64(V[J, g]).mean(axis=0)
            assert np.allclose(o[i, h], mean, rtol=1e-12, atol=1e-13)
            qk = scale * float(np.dot(bits_to_f64(q[t, h]), bits_to_f64(Keq[0, g])))
            assert abs(lse[i, h] - (qk + math.log(nsel))) < 1e-11
    # (iv) permuting tokens inside a non-local selected block changes nothing
    o1, l1 = oracle.sparse_attn(q[rows], rows, K, V, ids, Bk, scale)
    K2, V2 = K.copy(), V.copy()
    b = 2  # a block that rows >= 48 may select as non-local
    perm = rng.permutation(Bk)
    K2[b * Bk:(b + 1) * Bk] = K[b * Bk:(b + 1) * Bk][perm]
    V2[b * Bk:(b + 1) * Bk] = V[b * Bk:(b + 1) * Bk][perm]
    o2, l2 = oracle.sparse_attn(q[rows], rows, K2, V2, ids, Bk, scale)
    far = rows >= (b + 1) * Bk
    assert np.allclose(o1[far], o2[far], rtol=1e-12, atol=1e-13)
    assert np.allclose(l1[far], l2[far], rtol=1e-12, atol=1e-13)


def test_group_sharing_and_head_to_group_map():
    """Each head h uses the block set and K/V of its group h // G."""
    rng = np.random.default_rng(31)
    N, H_q, H_kv, d, Bk, k = 200, 6, 3, 8, 8, 3
    rows = np.array([7, 64, 150, 199])
    q = rand_bf16(rng, (N, H_q, d))
    K = rand_bf16(rng, (N, H_kv, d))
    V = rand_bf16(rng, (N, H_kv, d))
    ids = _random_ids(rng, rows, H_kv, Bk, k)
    o, lse = oracle.sparse_attn(q[rows], rows, K, V, ids, Bk, 0.3)
    for h in range(H_q):
        g = h // 2
        oh, lh = oracle.sparse_attn(q[rows][:, h:h + 1], rows, K[:, g:g + 1], V[:, g:g + 1],
                                    ids[:, g:g + 1], Bk, 0.3)
        assert np.array_equal(oh[:, 0], o[:, h]) and np.array_equal(lh[:, 0], lse[:, h])


# ----------------------------------------------------------------- decode

def test_decode_equals_prefill_row():
    """Decoding token t against a (permuted) paged cache of tokens 0..t gives
    prefill row t: same block ids, same output."""
    w = synth.make("decode", B=3, L=1000, H_q=4, H_kv=2, d=32, d_idx=32, Bk=64, k=4)
    pt = synth.page_table(w, permute=True)
    seq_lens = np.array([1000, 1000, 1000], dtype=np.int32)
    kidx = synth.host_tensor(w, synth.T_KIDX)  # [B, L, 1, d_idx]
    K = synth.host_tensor(w, synth.T_K)
    V = synth.host_tensor(w, synth.T_V)
    qidx_all = synth.host_tensor(w, synth.T_QIDX)
    q_all = synth.host_tensor(w, synth.T_Q)

    def paged(x):  # [B, L, H, D] -> head-major pages [P, H, Bk, D] through the page table
        B, L, H, D = x.shape
        P = pt.size
        out = np.zeros((P, H, w.Bk, D), dtype=x.dtype)
        for s in range(B):
            for b in range(w.nb):
                t0, t1 = b * w.Bk, min(L, (b + 1) * w.Bk)
                out[pt[s, b], :, :t1 - t0] = x[s, t0:t1].transpose(1, 0, 2)
        return out

    t = w.L - 1
    ids_d = oracle.decode_index_select(qidx_all[:, t], paged(kidx)[:, 0], pt, seq_lens,
                                       w.Bk, w.k)
    o_d, l_d = oracle.decode_attn(q_all[:, t], paged(K), paged(V), pt, seq_lens, ids_d, w.Bk,
                                  w.scale)
    for s in range(w.B):
        ids_p = oracle.index_select(qidx_all[s, t:t + 1], np.array([t]), kidx[s, :, 0], w.Bk, w.k)
        assert np.array_equal(ids_p[0], ids_d[s])
        o_p, l_p = oracle.sparse_attn(q_all[s, t:t + 1], np.array([t]), K[s], V[s], ids_p,
                                      w.Bk, w.scale)
        assert np.allclose(o_p[0], o_d[s], rtol=1e-13, atol=1e-14)
        assert np.allclose(l_p[0], l_d[s], rtol=1e-13, atol=1e-13)


def test_decode_fp8_path_equals_bf16_on_exact_values():
    """One page, scale 1, values exact in both E4M3 and bf16: both KV paths agree."""
    rng = np.random.default_rng(41)
    Bk, H_kv, H_q, d = 128, 2, 4, 16
    vals = rng.integers(-16, 17, size=(1, H_kv, Bk, d)).astype(np.float32) / 4.0
    kb = bf16_bits(vals)
    k8 = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    vv = rng.integers(-16, 17, size=(1, H_kv, Bk, d)).astype(np.float32) / 8.0
    vb = bf16_bits(vv)
    v8 = torch.from_numpy(vv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    q = rand_bf16(rng, (1, H_q, d))
    pt = np.zeros((1, 1), dtype=np.int32)
    sl = np.array([100], dtype=np.int32)
    ids = np.array([[[0, -1], [0, -1]]], dtype=np.int32)
    o1, l1 = oracle.decode_attn(q, kb, vb, pt, sl, ids, Bk, 0.25)
    o2, l2 = oracle.decode_attn(q, k8, v8, pt, sl, ids, Bk, 0.25, fp8=True,
                                k_scale=np.ones(H_kv), v_scale=np.ones(H_kv))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # scales multiply the dequantised values: V scaled by 2 doubles o exactly
    o3, l3 = oracle.decode_attn(q, k8, v8, pt, sl, ids, Bk, 0.25, fp8=True,
                                k_scale=np.ones(H_kv), v_scale=np.full(H_kv, 2.0))
    assert np.array_equal(o3, 2 * o1) and np.array_equal(l3, l1)


# ----------------------------------------------------- KL alignment signal
def _sig(x):
    return 1.0 / (1.0 + math.exp(-x))


def test_kl_two_tokens_bernoulli_closed_form():
    """t = 1 sees tokens {0, 1}: the teacher and the student are Bernoulli
    distributions, so the KL is the textbook two-point form. Two heads with
    different attention check the group average; the two directions of KL
    differ here, so a swapped KL fails."""
    q = bf16_bits([[[2, 0], [0, 1]]])             # [1 row, H_q = 2, d = 2]
    K = bf16_bits([[[1, 0]], [[0, 1]]])           # [2 tokens, H_kv = 1, d = 2]
    qi = bf16_bits([[[1, 3]]])                    # [1 row, n_g = 1, d_idx = 2]
    ki = bf16_bits([[1, 1], [0, 2]])              # [2 tokens, d_idx = 2]
    ids = np.array([[[0, -1]]], dtype=np.int32)
    kl, mag = oracle.kl_teacher(q, qi, np.array([1]), K, ki, ids, 128, 1.0)
    a = (_sig(2.0) + _sig(-1.0)) / 2.0            # teacher mass on token 0
    b = _sig(4.0 - 6.0)                           # student mass on token 0
    want = a * math.log(a / b) + (1 - a) * math.log((1 - a) / (1 - b))
    assert abs(kl[0, 0] - want) < 1e-12
    assert abs(want - (b * math.log(b / a) + (1 - b) * math.log((1 - b) / (1 - a)))) > 1e-3
    assert mag[0, 0] >= kl[0, 0]


def test_kl_zero_when_index_scores_equal_scaled_attention_logits():
    """G = 1 with q_idx = scale * q and k_idx = k: the student equals the
    teacher on every row and every selection, so the KL is 0. Fails if the
    teacher drops the scale or the student scales its raw scores."""
    rng = np.random.default_rng(3)
    N, d, Bk, k = 300, 64, 16, 4
    qf = rng.integers(-4, 5, size=(N, 1, d)).astype(np.float32)
    kf = rng.integers(-4, 5, size=(N, 1, d)).astype(np.float32)
    q, K = bf16_bits(qf), bf16_bits(kf)
    qi, ki = bf16_bits(qf / 8.0), bf16_bits(kf[:, 0])
    rows = np.arange(N)
    ids = oracle.index_select(qi, rows, ki, Bk, k)
    kl, _ = oracle.kl_teacher(q, qi, rows, K, ki, ids, Bk, 1.0 / 8.0)
    assert np.abs(kl).max() < 1e-9


def test_kl_nonnegative_and_group_of_equal_heads():
    """Gibbs' inequality on Gaussian inputs, and a group of G equal heads
    gives the KL of one head (the group average of equal distributions)."""
    rng = np.random.default_rng(4)
    N, d, Bk, k = 200, 32, 8, 5
    q1 = rand_bf16(rng, (N, 2, d))
    K = rand_bf16(rng, (N, 2, d))
    qi = rand_bf16(rng, (N, 2, d))
    ki = rand_bf16(rng, (N, d))
    rows = np.arange(N)
    ids = oracle.index_select(qi, rows, ki, Bk, k)
    kl1, _ = oracle.kl_teacher(q1, qi, rows, K, ki, ids, Bk, 0.2)
    assert kl1.min() > -1e-12
    assert kl1.max() > 1e-3
    q3 = np.repeat(q1, 3, axis=1)                 # heads 0,0,0 | 1,1,1: G = 3
    kl3, _ = oracle.kl_teacher(q3, qi, rows, K, ki, ids, Bk, 0.2)
    assert np.allclose(kl3, kl1, rtol=1e-12, atol=1e-12)


def test_kl_matches_brute_force_on_tiny_inputs():
    """An independently written per-token loop on tiny shapes with a real
    selection (k below the visible blocks): every selected block's tokens up
    to t, each head's softmax, the group mean, the index softmax."""
    rng = np.random.default_rng(5)
    N, H_q, H_kv, d, Bk, k = 40, 4, 2, 8, 4, 3
    q = rand_bf16(rng, (N, H_q, d))
    K = rand_bf16(rng, (N, H_kv, d))
    qi = rand_bf16(rng, (N, H_kv, d))
    ki = rand_bf16(rng, (N, d))
    rows = np.arange(N)
    ids = oracle.index_select(qi, rows, ki, Bk, k)
    kl, _ = oracle.kl_teacher(q, qi, rows, K, ki, ids, Bk, 0.3)
    qf, Kf, qif, kif = bits_to_f64(q), bits_to_f64(K), bits_to_f64(qi), bits_to_f64(ki)
    G = H_q // H_kv
    for t in range(N):
        for g in range(H_kv):
            toks = [j for j in range(t + 1) if j // Bk in set(int(b) for b in ids[t, g] if b >= 0)]
            teacher = [0.0] * len(toks)
            for h in range(g * G, (g + 1) * G):
                logits = [0.3 * sum(qf[t, h, c] * Kf[j, g, c] for c in range(d)) for j in toks]
                top = max(logits)
                z = sum(math.exp(x - top) for x in logits)
                for u, x in enumerate(logits):
                    teacher[u] += math.exp(x - top) / z / G
            sc = [sum(qif[t, g, c] * kif[j, c] for c in range(d)) for j in toks]
            top = max(sc)
            z = sum(math.exp(x - top) for x in sc)
            student = [math.exp(x - top) / z for x in sc]
            want = sum(p * math.log(p / s) for p, s in zip(teacher, student) if p > 0)
            assert abs(kl[t, g] - want) < 1e-10 * max(1.0, abs(want)), (t, g)


def test_e2m1_decoder_exhaustive_vs_ocp():
    """All 16 FP4 E2M1 codes against the OCP table: sign bit 3, exponent bits
    2..1 with bias 1, one mantissa bit, exponent 0 subnormal (m * 0.5)."""
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        want = table[c & 7] * (-1.0 if c & 8 else 1.0)
        got = oracle.e2m1_to_f64(c)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), c


# --------------------------------------------------- index-branch projections
def test_projection_one_hot_rows_pick_weight_columns():
    """x = e_m (one-hot) gives q_idx[g, c] = w_qidx[g * d_idx + c, m] and
    k_idx[c] = w_kidx[c, m]: pins the [out, in] weight layout, the group-major
    split of the query outputs and the two outputs' ranges."""
    rng = np.random.default_rng(61)
    d_model, n_g, d_idx = 24, 3, 8
    wq = rand_bf16(rng, (n_g * d_idx, d_model))
    wk = rand_bf16(rng, (d_idx, d_model))
    x = bf16_bits(np.eye(d_model, dtype=np.float32))
    q, k = oracle.index_project(x, wq, wk)
    wqf, wkf = bits_to_f64(wq), bits_to_f64(wk)
    for m in range(d_model):
        for g in range(n_g):
            assert np.array_equal(q[m, g], wqf[g * d_idx:(g + 1) * d_idx, m])
        assert np.array_equal(k[m], wkf[:, m])


def test_projection_integer_inputs_equal_integer_matmul():
    """Integer-valued x and weights: the fp64 sums are exact integers, equal to
    numpy's int64 matrix product (an independent routine)."""
    rng = np.random.default_rng(62)
    n, d_model, n_g, d_idx = 37, 96, 4, 16
    xi = rng.integers(-8, 9, (n, d_model))
    wqi = rng.integers(-8, 9, (n_g * d_idx, d_model))
    wki = rng.integers(-8, 9, (d_idx, d_model))
    q, k = oracle.index_project(bf16_bits(xi.astype(np.float32)), bf16_bits(wqi.astype(np.float32)),
                                bf16_bits(wki.astype(np.float32)))
    assert np.array_equal(q.reshape(n, -1), (xi @ wqi.T).astype(np.float64))
    assert np.array_equal(k, (xi @ wki.T).astype(np.float64))


def test_projection_is_linear():
    """project(x1 + 2 x2) = project(x1) + 2 project(x2) for values exact in bf16."""
    rng = np.random.default_rng(63)
    n, d_model, n_g, d_idx = 9, 40, 2, 8
    x1 = rng.integers(-4, 5, (n, d_model)).astype(np.float32) / 4
    x2 = rng.integers(-4, 5, (n, d_model)).astype(np.float32) / 4
    wq = rand_bf16(rng, (n_g * d_idx, d_model))
    wk = rand_bf16(rng, (d_idx, d_model))
    qa, ka = oracle.index_project(bf16_bits(x1 + 2 * x2), wq, wk)
    q1, k1 = oracle.index_project(bf16_bits(x1), wq, wk)
    q2, k2 = oracle.index_project(bf16_bits(x2), wq, wk)
    assert np.allclose(qa, q1 + 2 * q2, rtol=1e-12, atol=1e-12)
    assert np.allclose(ka, k1 + 2 * k2, rtol=1e-12, atol=1e-12)
