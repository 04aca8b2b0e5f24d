"""GPU parity of the index-branch projections (msa_index_project) against the
oracle's fp64 linear maps.

Integer-valued inputs make every fp32 partial sum exact, so the GPU's bf16
outputs must equal the oracle's values rounded once to bf16, bit for bit
(ragged row counts, a K depth that is not a multiple of the 64-wide K step,
output widths that end inside a 256-column tile). Gaussian inputs at a
model-sized depth are checked to one bf16 rounding plus fp32 accumulation.
The projected q_idx / k_idx then go through the GPU index branch and must give
the oracle's block ids.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_gqa_index_gb300 as m
    torch.cuda.set_device(0)
    return m


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _to_bf16_bits(a):
    """fp64 -> bf16 bits, one round to nearest even."""
    return _bits(torch.from_numpy(np.asarray(a, dtype=np.float64)).to(torch.bfloat16))


@pytest.mark.parametrize("N,d_model,n_g,d_idx", [
    (1, 64, 8, 128), (127, 136, 3, 64), (129, 512, 8, 128), (1000, 256, 1, 64),
    (300, 1024, 2, 128)])
def test_projection_exact_on_integer_inputs(msa, N, d_model, n_g, d_idx):
    g = torch.Generator().manual_seed(N + d_model)
    x = torch.randint(-4, 5, (N, d_model), generator=g).to(torch.bfloat16)
    wq = torch.randint(-4, 5, (n_g * d_idx, d_model), generator=g).to(torch.bfloat16)
    wk = torch.randint(-4, 5, (d_idx, d_model), generator=g).to(torch.bfloat16)
    q, k = msa.msa_index_project(x.cuda(), wq.cuda(), wk.cuda())
    torch.cuda.synchronize()
    qo, ko = oracle.index_project(_bits(x), _bits(wq), _bits(wk))
    assert np.array_equal(_bits(q), _to_bf16_bits(qo))
    assert np.array_equal(_bits(k), _to_bf16_bits(ko))
    assert msa.msa_get_error() == 0


def test_projection_gauss_model_width(msa):
    """x ~ N(0, 1), weights ~ N(0, 1 / d_model) at d_model = 4096 (H_q * d of the
    128K workload's heads): each output within one bf16 rounding plus the fp32
    accumulation error of the oracle's fp64 value."""
    N, d_model, n_g, d_idx = 2048 + 77, 4096, 8, 128
    g = torch.Generator().manual_seed(5)
    x = torch.randn((N, d_model), generator=g).to(torch.bfloat16)
    wq = (torch.randn((n_g * d_idx, d_model), generator=g) / d_model ** 0.5).to(torch.bfloat16)
    wk = (torch.randn((d_idx, d_model), generator=g) / d_model ** 0.5).to(torch.bfloat16)
    q, k = msa.msa_index_project(x.cuda(), wq.cuda(), wk.cuda())
    torch.cuda.synchronize()
    qo, ko = oracle.index_project(_bits(x), _bits(wq), _bits(wk))
    for got, want in ((q.float().cpu().numpy().astype(np.float64), qo),
                      (k.float().cpu().numpy().astype(np.float64), ko)):
        err = np.abs(got - want)
        bound = 2.0 ** -8 * np.abs(want) + 1e-4
        assert (err <= bound).all(), float((err - bound).max())


def test_projection_full_128k_sampled(msa):
    """The benchmarked configuration (131072 rows, d_model = 4096, eight groups of
    d_idx = 128), Gaussian as above, in one launch: sampled rows (the first and
    last, every tile's first row, random rows) against the oracle, within one
    bf16 rounding plus the fp32 accumulation error."""
    N, d_model, n_g, d_idx = 131072, 4096, 8, 128
    g = torch.Generator(device="cuda").manual_seed(6)
    x = torch.randn((N, d_model), generator=g, device="cuda").to(torch.bfloat16)
    wq = (torch.randn((n_g * d_idx, d_model), generator=g, device="cuda") /
          d_model ** 0.5).to(torch.bfloat16)
    wk = (torch.randn((d_idx, d_model), generator=g, device="cuda") /
          d_model ** 0.5).to(torch.bfloat16)
    q, k = msa.msa_index_project(x, wq, wk)
    torch.cuda.synchronize()
    assert msa.msa_get_error() == 0
    rng = np.random.default_rng(6)
    rows = np.unique(np.concatenate([[0, N - 1], np.arange(0, N, 128),
                                     rng.integers(0, N, 256)]))
    rt = torch.from_numpy(rows).cuda()
    qo, ko = oracle.index_project(_bits(x[rt]), _bits(wq), _bits(wk))
    for got, want in ((q[rt].float().cpu().numpy().astype(np.float64), qo),
                      (k[rt].float().cpu().numpy().astype(np.float64), ko)):
        err = np.abs(got - want)
        bound = 2.0 ** -8 * np.abs(want) + 1e-4
        assert (err <= bound).all(), float((err - bound).max())


def test_projection_feeds_index_branch(msa):
    """x -> projections -> index branch on the GPU selects the oracle's blocks for
    the oracle's projections of the same x (integer data: exact scores)."""
    N, d_model, n_g, d_idx = 3000, 128, 4, 64
    g = torch.Generator().manual_seed(9)
    x = torch.randint(-2, 3, (N, d_model), generator=g).to(torch.bfloat16)
    wq = torch.randint(-1, 2, (n_g * d_idx, d_model), generator=g).to(torch.bfloat16)
    wk = torch.randint(-1, 2, (d_idx, d_model), generator=g).to(torch.bfloat16)
    q, k = msa.msa_index_project(x.cuda(), wq.cuda(), wk.cuda())
    ids = msa.msa_index_select(q, k, 128, 16)
    torch.cuda.synchronize()
    qo, ko = oracle.index_project(_bits(x), _bits(wq), _bits(wk))
    assert np.abs(qo).max() < 256 and np.abs(ko).max() < 256  # exact in bf16
    want = oracle.index_select(_to_bf16_bits(qo), np.arange(N), _to_bf16_bits(ko), 128, 16)
    assert np.array_equal(ids.cpu().numpy(), want)
