"""Failure detection without a GPU fault.

Every mbarrier wait in the tensor-core kernels (index branch, main-branch tiles)
is a bounded poll loop. With the poll limit set to 0 a wait gives up at its first
unsatisfied poll: the kernel raises its abort flag, lets the copies and MMAs it
has issued complete, frees its tensor memory and returns, and the device error
word reports MSA_ERR_TIMEOUT. These tests force that path through the C ABI,
read the status with msa_get_error, and check that the context stays usable: the
next call with the normal limit returns exactly what a call made before the
timeout returned. Nothing here faults, traps or hangs the GPU.
"""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

MSA_ERR_TIMEOUT = -5


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_gqa_index_gb300 as m
    torch.cuda.set_device(0)
    return m


@pytest.fixture(scope="module")
def prefill():
    # 32K-workload shapes cut to 8269 tokens: 259 row tiles of up to 65 key
    # blocks, so every CTA of the index kernel has more blocks than ring stages
    w = synth.make("32k", L=8192 + 77)
    return dict(w=w, qidx=synth.device_tensor(w, synth.T_QIDX),
                kidx=synth.device_tensor(w, synth.T_KIDX)[:, 0].contiguous(),
                q=synth.device_tensor(w, synth.T_Q), k=synth.device_tensor(w, synth.T_K),
                v=synth.device_tensor(w, synth.T_V))


def _timed_out(msa, call):
    """Runs call() with the poll limit at 0 and returns the device status."""
    assert msa.msa_get_error() == 0
    old = msa.msa_set_wait_limit(0)
    try:
        call()
        rc = msa.msa_get_error()
    finally:
        msa.msa_set_wait_limit(old)
    return rc


def test_index_branch_timeout_is_reported_and_context_survives(msa, prefill):
    p, w = prefill, prefill["w"]
    ref = msa.msa_index_select(p["qidx"], p["kidx"], w.Bk, w.k)
    rc = _timed_out(msa, lambda: msa.msa_index_select(p["qidx"], p["kidx"], w.Bk, w.k))
    assert rc == MSA_ERR_TIMEOUT
    again = msa.msa_index_select(p["qidx"], p["kidx"], w.Bk, w.k)
    assert msa.msa_get_error() == 0
    assert torch.equal(again, ref)


def test_main_branch_timeout_is_reported_and_context_survives(msa, prefill):
    p, w = prefill, prefill["w"]
    ids = msa.msa_index_select(p["qidx"], p["kidx"], w.Bk, w.k)
    o_ref, l_ref = msa.msa_sparse_attn(p["q"], p["k"], p["v"], ids, w.Bk, w.scale)
    rc = _timed_out(msa, lambda: msa.msa_sparse_attn(p["q"], p["k"], p["v"], ids, w.Bk,
                                                     w.scale))
    assert rc == MSA_ERR_TIMEOUT
    o, l = msa.msa_sparse_attn(p["q"], p["k"], p["v"], ids, w.Bk, w.scale)
    assert msa.msa_get_error() == 0
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)
