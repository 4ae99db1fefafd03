"""The counter-based generator of the synthetic inputs: Philox4x32-10 against
the known-answer vectors published with it, and the uniforms built on it."""
import numpy as np

import synthetic as syn

# (counter, key) -> output, the published known-answer tests of philox4x32 with 10 rounds
KAT = [
    ([0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
    ([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
    ([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
     [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
]


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
