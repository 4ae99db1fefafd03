"""Sampling distributions and uniforms on the GPU against the float64 oracle
and the input generator.

The GPU holds a row's sampling distribution as fixed-point masses computed
from fp32 logits (temperature, nucleus); the oracle computes it in float64
from the same fp32 logits.  Probabilities are compared within the fp32
bound; where the nucleus cut lies within rounding of a tie, the GPU's
nucleus must be one of the correct ones.  The device Philox4x32-10 must give
the input generator's uniforms bit for bit.
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

# Relative difference of a probability between the fp32 / fixed-point path
# and float64 on the same fp32 logits: expf (2 ulp) plus the argument's
# three roundings (l - m, 1/T, the product: 1.8e-7 x |arg|, |arg| <= 31
# where a mass survives the 2^-44 grid) is at most 5.8e-6 per mass, so at
# most 1.2e-5 for a mass over the row's total.
PROB_RTOL = 2e-5
PROB_ATOL = 1e-12
# Nucleus cuts closer than this to a tie may go either way.
MARGIN = 5e-5


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__ as g
    g.build()
    import block_diffusion_speculative_layer_gb300 as m
    return m


def logit_rows(rows, V, scale, seed):
    """fp32 logits with planted ties (also at the maximum) and signed zeros."""
    g = np.random.default_rng(seed)
    x = (g.standard_normal((rows, V)) * scale).astype(np.float32)
    if V >= 8:
        for r in range(rows):
            idx = g.choice(V, size=6, replace=False)
            x[r, idx[1:3]] = x[r, idx[0]]
            x[r, idx[3]] = x[r].max()
            x[r, idx[4]] = 0.0
            x[r, idx[5]] = -0.0
    return x


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ----------------------------------------------------------------- generator
@pytest.mark.parametrize("seed,stream,offset,n", [(0, 0, 0, 1000), (7, 3, 5, 37), (2 ** 40 + 3, 11, 2 ** 33 - 2, 300)])
def test_device_uniforms_equal_the_generator(dfl, seed, stream, offset, n):
    got = dfl.philox_uniforms(seed, stream, offset, n).cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(got, syn.philox_uniforms(seed, stream, offset, n))


# ----------------------------------------------------------------- distributions
PROB_CASES = [(V, T, p) for V in (1, 7, 1000, 4097) for T in (0.0, 0.5, 1.0, 1.7) for p in (1.0, 0.9, 0.5, 0.05)]
PROB_CASES += [(151936, 1.0, 1.0), (151936, 0.7, 0.9), (151936, 0.0, 1.0), (151936, 1.0, 0.5)]


@pytest.mark.parametrize("V,T,top_p", PROB_CASES)
def test_sampling_probs_parity(dfl, V, T, top_p):
    rows = 6
    x = logit_rows(rows, V, 3.0 if V >= 1000 else 1.5, seed=V + int(100 * T) + int(1000 * top_p))
    got = dfl.sampling_probs(cuda(x), T, top_p).cpu().numpy().astype(np.float64)
    x64 = x.astype(np.float64)
    ref = O.sampling_probs(x64, T, top_p)
    for r in range(rows):
        if O.nucleus_margin(x64[r:r + 1], T, top_p) >= MARGIN:
            np.testing.assert_allclose(got[r], ref[r], rtol=PROB_RTOL, atol=PROB_ATOL)
            continue
        # The cut is within rounding of a tie, so more than one nucleus is
        # right: the GPU's must be a prefix of the descending order whose mass
        # crosses top_p within MARGIN, renormalised.
        order = np.lexsort((np.arange(V), -x64[r]))
        full = O.sampling_probs(x64[r:r + 1], T, 1.0)[0]
        csum = np.cumsum(full[order])
        kept = got[r][order] > 0
        m = int(kept.sum())
        assert m >= 1 and kept[:m].all()
        assert csum[m - 1] >= top_p - MARGIN and (m == 1 or csum[m - 2] < top_p + MARGIN)
        alt = np.zeros(V)
        alt[order[:m]] = full[order[:m]]
        np.testing.assert_allclose(got[r], alt / alt.sum(), rtol=PROB_RTOL, atol=PROB_ATOL)
