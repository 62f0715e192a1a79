"""mla_top_k_renorm_prob against the oracle: the kept set exactly (it is decided by order
alone), the renormalised values within float32 summation error."""
import numpy as np
import pytest
import torch

import mla_latent_kv_attention_gb300 as mla
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _check(probs, ks):
    out = mla.mla_top_k_renorm_prob(probs.to(DEV), ks if isinstance(ks, int) else
                                    torch.tensor(ks, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()
    ref = oracle.top_k_renorm_prob(probs.double().numpy(), ks)
    assert np.array_equal(got > 0, ref > 0)  # the kept set (zeros stay zero either way)
    assert np.allclose(got, ref, rtol=2e-6, atol=1e-12)


@pytest.mark.parametrize("V", [1, 1000, 16385, 129280, 131073, 163840, 262147])
def test_random_rows(V):
    g = torch.Generator().manual_seed(V)
    B = 8
    probs = torch.softmax(torch.randn(B, V, generator=g) * 4, dim=1)
    _check(probs, [1, 2, 20, 50, 1000 % V + 1, V - 1, V, 0])


def test_scalar_k_and_ties():
    g = torch.Generator().manual_seed(3)
    probs = torch.softmax(torch.randn(4, 4096, generator=g), dim=1)
    probs[:, 100:400] = probs[:, 100:101]  # a long run of equal values
    probs[1, 500:1500] = 0.0               # and zeros
    probs = probs / probs.sum(1, keepdim=True)
    for k in (1, 50, 250, 3000):
        _check(probs, k)


def test_selection_paths():
    """Each way the pivot is found, on rows built to take it: few entries in the bin of the
    k-th largest (ranked directly), a few hundred to thousands (rank 0's radix passes), a bin
    fuller than rank 0 holds (the later passes over the whole cluster), and the bin kept
    whole. The k-th largest and the kept set are exact in every case."""
    g = torch.Generator().manual_seed(11)
    V = 129280
    tail = torch.softmax(torch.randn(2, V, generator=g) * 3, dim=1)   # sparse top: small bins
    median = torch.softmax(torch.randn(2, V, generator=g), dim=1)     # dense middle
    # one bin for nearly everything: 1/V times 1 + tiny noise, a few large entries on top
    flat = torch.full((2, V), 1.0 / V) * (1 + 1e-4 * torch.rand(2, V, generator=g))
    flat[:, :7] = 0.01
    flat = flat / flat.sum(1, keepdim=True)
    probs = torch.cat([tail, median, flat])
    # tail rows: k = 5 (a handful of candidates), V/2 (about 1,500: rank 0's radix passes);
    # median rows: around 4,000 to 4,500 in the bin; flat rows: V/2 (about 129,000: the
    # later cluster passes), 7 (the seven large entries: their bin kept whole)
    _check(probs, [5, V // 2, V // 3, V // 2, V // 2, 7])


def test_misaligned_rows_and_outputs():
    """Rows that start off the 16-byte grid (odd V), and an output whose alignment differs
    from the input's (a view one element in): the vector loads and stores keep to the row."""
    g = torch.Generator().manual_seed(12)
    B, V = 5, 40001
    probs = torch.softmax(torch.randn(B, V, generator=g) * 3, dim=1).to(DEV)
    ks = torch.tensor([1, 17, 333, V // 2, V - 1], dtype=torch.int32, device=DEV)
    big = torch.full((B * V + 1,), -7.0, device=DEV)
    out = big[1:].view(B, V)
    mla.mla_top_k_renorm_prob(probs, ks, out=out)
    torch.cuda.synchronize()
    assert float(big[0]) == -7.0  # nothing written before the output
    ref = oracle.top_k_renorm_prob(probs.cpu().double().numpy(), ks.cpu().tolist())
    got = out.cpu().double().numpy()
    assert np.array_equal(got > 0, ref > 0)
    assert np.allclose(got, ref, rtol=2e-6, atol=1e-12)
