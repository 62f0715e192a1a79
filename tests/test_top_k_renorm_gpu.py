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
