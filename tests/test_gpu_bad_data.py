"""Device-side invalid data: block ids and sequence lengths that the host cannot
check (they live in device memory) are skipped by the kernels and reported
through the device error word, which msa_get_error returns as
MSA_ERR_INVALID_ARG.

Every invalid value used here addresses memory inside its own tensor (a block
id between the row's local block and the last block of the sequence, a
sequence length one page past its page-table row), so a kernel that failed to
check would compute something wrong, never read out of bounds. Each test
checks the error code, that the rows without invalid data keep the results of
a clean call (bit for bit, or to rounding where they share a query tile with a
planted row in the prefill main branch), how the row with invalid data is
treated, and that the next clean call gives the clean bits again.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.msa_check import bf16_to_np, check_close

pytestmark = pytest.mark.gpu

MSA_ERR_INVALID_ARG = -1


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_gqa_index_gb300 as m
    torch.cuda.set_device(0)
    return m


def test_sparse_attn_skips_causally_invalid_ids(msa):
    """A block id after the row's local block (still below nb) is skipped: the
    row attends over its other blocks (the oracle on the ids with that slot
    emptied), the other rows keep their results, and the error word says so."""
    w = synth.make("tiny", L=1000, H_q=8, H_kv=2, d=64, d_idx=64)
    qidx = synth.device_tensor(w, synth.T_QIDX)
    kidx = synth.device_tensor(w, synth.T_KIDX)[:, 0].contiguous()
    q = synth.device_tensor(w, synth.T_Q)
    kk = synth.device_tensor(w, synth.T_K)
    v = synth.device_tensor(w, synth.T_V)
    ids = msa.msa_index_select(qidx, kidx, w.Bk, w.k)
    out0, lse0 = msa.msa_sparse_attn(q, kk, v, ids, w.Bk, w.scale)
    assert msa.msa_get_error() == 0
    bad = ids.clone()
    # (row, group, slot, id): a padded slot and a real slot, ids in (t / Bk, nb)
    plant = [(300, 0, 5, 6), (300, 1, 3, 7), (640, 1, 0, 7), (129, 0, 2, 2)]
    for t, g, s, b in plant:
        assert t // w.Bk < b < w.nb
        bad[t, g, s] = b
    out1, lse1 = msa.msa_sparse_attn(q, kk, v, bad, w.Bk, w.scale)
    assert msa.msa_get_error() == MSA_ERR_INVALID_ARG
    assert msa.msa_get_error() == 0  # read and cleared
    rows_bad = sorted({t for t, _, _, _ in plant})
    # rows in other query tiles (128 / G queries) keep their bits; rows that
    # share a tile with a planted row agree to rounding: the tile's blocks
    # selected by at least half of its queries are combined in one pass, and a
    # planted id can move a block across that line
    qt = 128 // (w.H_q // w.H_kv)
    tiles_bad = {t // qt for t in rows_bad}
    keep = np.array([t for t in range(w.N) if t // qt not in tiles_bad])
    near = np.array([t for t in range(w.N) if t // qt in tiles_bad and t not in rows_bad])
    kt = torch.from_numpy(keep).cuda()
    assert torch.equal(out1[kt], out0[kt]) and torch.equal(lse1[kt], lse0[kt])
    nt = torch.from_numpy(near).cuda()
    check_close("o near", bf16_to_np(out1[nt]), bf16_to_np(out0[nt]), 1e-2)
    check_close("lse near", lse1[nt].cpu().numpy(), lse0[nt].cpu().numpy(), 1e-4)
    # the planted rows: attention over their remaining valid blocks
    emptied = bad.cpu().numpy()
    for t, g, s, b in plant:
        emptied[t, g, s] = -1
    rows = np.array(rows_bad)
    o_ref, l_ref = oracle.sparse_attn(synth.host_tensor(w, synth.T_Q)[0][rows], rows,
                                      synth.host_tensor(w, synth.T_K)[0],
                                      synth.host_tensor(w, synth.T_V)[0], emptied[rows], w.Bk,
                                      w.scale)
    rt = torch.from_numpy(rows).cuda()
    check_close("o", bf16_to_np(out1[rt]), o_ref, 1e-2)
    check_close("lse", lse1[rt].cpu().numpy(), l_ref, 1e-3)
    out2, lse2 = msa.msa_sparse_attn(q, kk, v, ids, w.Bk, w.scale)
    assert msa.msa_get_error() == 0
    assert torch.equal(out2, out0) and torch.equal(lse2, lse0)


def _decode_inputs(w, fp8):
    dev = torch.device("cuda")
    pt = torch.from_numpy(synth.page_table(w)).to(dev)
    last = [(s, w.L - 1) for s in range(w.B)]
    q = synth.device_rows(w, synth.T_Q, last)
    qidx = synth.device_rows(w, synth.T_QIDX, last)
    kidx = synth.device_paged(w, synth.T_KIDX, pt)[:, 0].contiguous()
    kp = synth.device_paged(w, synth.T_K, pt, fp8=fp8)
    vp = synth.device_paged(w, synth.T_V, pt, fp8=fp8)
    ks, vs = synth.fp8_scales(w.H_kv)
    kw = dict(k_scale=torch.from_numpy(ks).to(dev), v_scale=torch.from_numpy(vs).to(dev)) \
        if fp8 else {}
    return pt, q, qidx, kidx, kp, vp, kw


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_skips_causally_invalid_ids(msa, fp8):
    """Decode attention with a block id past the sequence's last block (inside
    the page table): the slot is skipped, the other (sequence, group) rows keep
    their bits, and the error word reports it."""
    w = synth.make("decode", B=4, L=128 * 6 + 9, H_q=8, H_kv=2, d=128, d_idx=128,
                   kind=synth.KIND_INT, k=4)
    dev = torch.device("cuda")
    pt, q, qidx, kidx, kp, vp, kw = _decode_inputs(w, fp8)
    lens = torch.tensor([w.L, w.L, 300, w.L], dtype=torch.int32, device=dev)
    ids = msa.msa_index_select_decode(qidx, kidx, pt, lens, w.Bk, w.k)
    out0, lse0 = msa.msa_decode(q, kp, vp, pt, lens, ids, w.Bk, w.scale, **kw)
    assert msa.msa_get_error() == 0
    bad = ids.clone()
    assert bad[2, 1, 3].item() == -1  # sequence 2 sees 3 blocks: its 4th slot is padding
    bad[2, 1, 3] = 5                  # a block past its last one, inside its table row
    out1, lse1 = msa.msa_decode(q, kp, vp, pt, lens, bad, w.Bk, w.scale, **kw)
    assert msa.msa_get_error() == MSA_ERR_INVALID_ARG
    # heads of the planted (sequence, group) keep their other blocks: same bits,
    # since the skipped slot was padding; every other head is untouched too
    assert torch.equal(out1, out0) and torch.equal(lse1, lse0)
    out2, lse2 = msa.msa_decode(q, kp, vp, pt, lens, ids, w.Bk, w.scale, **kw)
    assert msa.msa_get_error() == 0
    assert torch.equal(out2, out0) and torch.equal(lse2, lse0)


def test_decode_index_rejects_length_past_page_table(msa):
    """A sequence length one page past its page-table row: that sequence gets
    only -1 padding, the others keep their ids, and the error word reports it.
    The same length in the decode attention leaves that sequence's heads at a
    zero output with LSE -inf and the other sequences untouched."""
    w = synth.make("decode", B=3, L=128 * 5, H_q=8, H_kv=2, d=64, d_idx=64,
                   kind=synth.KIND_INT, k=4)
    dev = torch.device("cuda")
    pt, q, qidx, kidx, kp, vp, kw = _decode_inputs(w, False)
    max_pages = pt.shape[1]
    lens = torch.full((w.B,), w.L, dtype=torch.int32, device=dev)
    ids0 = msa.msa_index_select_decode(qidx, kidx, pt, lens, w.Bk, w.k)
    out0, lse0 = msa.msa_decode(q, kp, vp, pt, lens, ids0, w.Bk, w.scale)
    assert msa.msa_get_error() == 0
    bad = lens.clone()
    bad[1] = max_pages * w.Bk + 1
    ids1 = msa.msa_index_select_decode(qidx, kidx, pt, bad, w.Bk, w.k)
    assert msa.msa_get_error() == MSA_ERR_INVALID_ARG
    assert (ids1[1] == -1).all()
    assert torch.equal(ids1[0], ids0[0]) and torch.equal(ids1[2], ids0[2])
    out1, lse1 = msa.msa_decode(q, kp, vp, pt, bad, ids0, w.Bk, w.scale)
    assert msa.msa_get_error() == MSA_ERR_INVALID_ARG
    assert torch.equal(out1[0], out0[0]) and torch.equal(out1[2], out0[2])
    assert torch.equal(lse1[0], lse0[0]) and torch.equal(lse1[2], lse0[2])
    assert (out1[1].float() == 0).all() and torch.isneginf(lse1[1]).all()
    ids2 = msa.msa_index_select_decode(qidx, kidx, pt, lens, w.Bk, w.k)
    assert msa.msa_get_error() == 0
    assert torch.equal(ids2, ids0)


def test_topk_rejects_rows_past_the_scores(msa):
    """seq_lens mode with one row whose position lies past the nb given blocks:
    that row gets -1 padding, the others are exact, the error word reports it."""
    rng = np.random.default_rng(5)
    B, n_g, nb = 6, 4, 40
    S = rng.standard_normal((B, n_g, nb)).astype(np.float32)
    lens = np.array([1, 129, nb * 128, 3000, 5000, 777], dtype=np.int32)
    lens_bad = lens.copy()
    lens_bad[2] = nb * 128 + 1
    St = torch.from_numpy(S).cuda()
    good = msa.msa_topk_blocks(St, 128, 16, seq_lens=torch.from_numpy(lens).cuda())
    assert msa.msa_get_error() == 0
    got = msa.msa_topk_blocks(St, 128, 16, seq_lens=torch.from_numpy(lens_bad).cuda())
    assert msa.msa_get_error() == MSA_ERR_INVALID_ARG
    got, good = got.cpu().numpy(), good.cpu().numpy()
    assert (got[2] == -1).all()
    rest = [0, 1, 3, 4, 5]
    want = oracle.topk_blocks(S[rest], lens[rest].astype(np.int64) - 1, 128, 16)
    assert np.array_equal(got[rest], want) and np.array_equal(good[rest], want)
