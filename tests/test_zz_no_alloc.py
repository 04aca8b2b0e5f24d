"""The allocation-free decode index entry point.

Some callers cannot allocate device memory while they run (engines that
reserve all device memory at start-up, code where an allocation could stall
other work on the device). msa_index_select_decode_noalloc serves them by
keeping its block-score scratch in a fixed array inside the library. These
tests call it through the C ABI and check that it returns exactly what the
workspace-based msa_index_select_decode returns, on two different calls in a
row (the shared array keeps the previous call's contents, which must not
leak into the next result). This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_gqa_index_gb300 as m
    torch.cuda.set_device(0)
    return m


def _decode_inputs(w, lens):
    dev = torch.device("cuda")
    pt = torch.from_numpy(synth.page_table(w)).to(dev)
    kidx_p = synth.device_paged(w, synth.T_KIDX, pt)[:, 0].contiguous()
    qidx = synth.device_rows(w, synth.T_QIDX, [(s, int(lens[s]) - 1) for s in range(w.B)])
    return qidx, kidx_p, pt, torch.from_numpy(np.asarray(lens, dtype=np.int32)).to(dev)


def test_noalloc_matches_workspace_path_two_calls(msa):
    # first call: Gaussian inputs, full-length sequences
    wa = synth.make("decode", B=6, L=128 * 40 + 1, H_q=32, H_kv=8, d=128, d_idx=128)
    # second call: integer inputs (many ties), fewer groups, ragged lengths, d_idx 64
    wb = synth.make("decode", B=3, L=1000, H_q=8, H_kv=2, d=64, d_idx=64, k=5,
                    kind=synth.KIND_INT)
    cases = [(wa, [wa.L] * wa.B), (wb, [1, 300, 1000])]
    for w, lens in cases:
        qidx, kidx_p, pt, sl = _decode_inputs(w, lens)
        want = msa.msa_index_select_decode(qidx, kidx_p, pt, sl, w.Bk, w.k)
        got = torch.full_like(want, -7)
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        msa.msa_index_select_decode_noalloc(qidx, kidx_p, pt, sl, w.Bk, w.k, block_ids=got)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == before
        assert torch.equal(got, want)
        assert msa.msa_get_error() == 0


def test_noalloc_rejects_requests_beyond_the_array(msa):
    cap = msa.msa_index_select_decode_noalloc_max_scores()
    assert cap == 1 << 20
    dev = torch.device("cuda")
    B, n_g, max_pages = 64, 8, cap // (64 * 8) + 1  # one page more than fits
    qidx = torch.zeros((B, n_g, 128), dtype=torch.bfloat16, device=dev)
    kidx = torch.zeros((1, 128, 128), dtype=torch.bfloat16, device=dev)
    pt = torch.zeros((B, max_pages), dtype=torch.int32, device=dev)
    sl = torch.ones((B,), dtype=torch.int32, device=dev)
    with pytest.raises(msa.MSAError) as e:
        msa.msa_index_select_decode_noalloc(qidx, kidx, pt, sl)
    assert e.value.status == msa.MSA_ERR_WORKSPACE
