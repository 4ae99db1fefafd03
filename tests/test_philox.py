"""The counter-based generator of the synthetic inputs: Philox4x32-10 against
the known-answer vectors published with it, and the uniforms built on it;
the library's own Philox (its device generator's source, run on the host)
against the same vectors."""
import os

import numpy as np

import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "philox4x32_10_kat.txt")


def kat_vectors():
    """(counter, key, output) triples of the published known-answer tests."""
    out = []
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            w = [int(x, 16) for x in line.split()]
            out.append((w[0:4], w[4:6], w[6:10]))
    return out


KAT = kat_vectors()


def test_philox_known_answers():
    for ctr, key, want in KAT:
        assert syn.philox4x32(ctr, key) == want


def test_uniforms_layout_and_range():
    u = syn.philox_uniforms(7, 3, 0, 4000)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))          # 24 random bits, exact in float32
    assert abs(u.mean() - 0.5) < 0.02 and abs(u.var() - 1 / 12) < 0.01
    # offsets address the same sequence
    np.testing.assert_array_equal(syn.philox_uniforms(7, 3, 10, 20), u[10:30])
    # word layout: uniform 4b + w is word w of block b
    w = syn.philox4x32([2, 0, 3, 0], [7, 0])
    np.testing.assert_array_equal(u[8:12], [(x >> 8) / 2 ** 24 for x in w])
    # streams and seeds differ
    assert not np.array_equal(syn.philox_uniforms(7, 4, 0, 16), u[:16])
    assert not np.array_equal(syn.philox_uniforms(8, 3, 0, 16), u[:16])


def test_library_philox_known_answers():
    # the CUDA library implements the generator separately from the inputs
    # module; its block function runs on the host through the C ABI
    import __graft_entry__ as g
    g.build()
    import block_diffusion_speculative_layer_gb300 as dfl
    assert len(KAT) == 3
    for ctr, key, want in KAT:
        assert dfl.philox4x32_10(ctr, key) == want
    rng = np.random.default_rng(0)
    for _ in range(50):
        ctr = [int(x) for x in rng.integers(0, 2 ** 32, 4)]
        key = [int(x) for x in rng.integers(0, 2 ** 32, 2)]
        assert dfl.philox4x32_10(ctr, key) == syn.philox4x32(ctr, key)
