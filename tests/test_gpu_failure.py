"""Failure detection without a GPU fault.

Every wait in the engine's kernels is bounded (about two seconds of the
device timer).  df_debug_wait_probe launches one kernel whose bounded wait
on a barrier that nothing completes runs out: the kernel records the
timeout in the handle's error word and returns, so the CUDA context stays
usable.  The call must return DF_ETIMEOUT, the handle must stay failed, and
a new handle in the same process must decode correctly.
"""
import time

import numpy as np
import pytest

import synthetic as syn
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__ as g
    g.build()
    import block_diffusion_speculative_layer_gb300 as m
    return m


def test_bounded_wait_reports_a_timeout(dfl):
    shape = syn.TINY
    w = syn.make_weights(shape)
    p = syn.make_prompt(shape, 24, stream=80)
    ref = O.greedy_generate(O.Model(O.Weights(w), shape), p, 16)
    eng = dfl.Engine(shape, w, max_batch=1, max_ctx=128)
    try:
        out, _ = eng.generate([p], 16)
        np.testing.assert_array_equal(out[0], ref)
        t0 = time.time()
        with pytest.raises(dfl.DfError) as e:
            eng.wait_probe()
        waited = time.time() - t0
        assert e.value.status == dfl.DF_ETIMEOUT
        assert 0.5 < waited < 60.0
        # the handle stays failed
        with pytest.raises(dfl.DfError) as e2:
            eng.generate([p], 4)
        assert e2.value.status == dfl.DF_ECUDA
    finally:
        eng.close()
    # the context is intact: a new handle decodes correctly
    with dfl.Engine(shape, w, max_batch=1, max_ctx=128) as eng2:
        out, _ = eng2.generate([p], 16)
    np.testing.assert_array_equal(out[0], ref)
    assert torch.cuda.is_available() and torch.zeros(4, device="cuda").sum().item() == 0.0
