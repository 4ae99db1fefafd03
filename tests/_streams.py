"""Sampled token streams of the engine against the oracle's sampled loop.

The oracle draws from the same Philox4x32-10 uniforms as the GPU (stream i of
the call's seed for sequence i, in the loop's order), on float64 logits of
its own model; the GPU's logits are fp32.  A decision (a nucleus cut, a draw,
a test) closer to a tie than the two logit sets differ may go either way, so
streams are compared only for seeds whose every decision is farther than
STREAM_MARGIN from a tie (the oracle reports each decision's distance).
"""
import numpy as np

import synthetic as syn
from oracle import dflash_oracle as O

STREAM_MARGIN = 2e-4   # fp32 logits of the tiny model differ from float64 by about 1e-6 relative


class Uniforms:
    """The oracle's uniform source: Philox stream `stream` of `seed`, in order."""

    def __init__(self, seed, stream):
        self.seed, self.stream, self.off = seed, stream, 0

    def __call__(self, n):
        u = syn.philox_uniforms(self.seed, self.stream, self.off, n)
        self.off += n
        return u


def stream_case(eng, model, prompt, n_new, T, top_p, seed, block=None):
    """(oracle result, GPU stream, GPU per-cycle k histogram, smallest
    decision margin) for one sequence (Philox stream 0)."""
    margins = []
    m = model if block is None else O.Model(model.W, model.cfg.replace(block_size=block))
    ref = O.spec_generate_sampled(m, prompt, n_new, T, top_p, Uniforms(seed, 0), margins)
    got, _ = eng.generate_sampled([prompt], n_new, temperature=T, top_p=top_p, seed=seed)
    return ref, got[0], eng.accept_hist_per_seq(1)[0], min(margins)


def assert_stream_matches(eng, model, prompt, n_new, T, top_p, seeds, block=None, need=2):
    """Over `seeds`, every seed whose decisions are all clear of ties gives
    the oracle's stream and per-cycle accepted counts; at least `need` do."""
    compared, seen = 0, []
    for seed in seeds:
        ref, got, hist, margin = stream_case(eng, model, prompt, n_new, T, top_p, seed, block)
        seen.append((seed, margin))
        if margin < STREAM_MARGIN:
            continue
        np.testing.assert_array_equal(got, ref.tokens, err_msg=f"seed {seed}")
        np.testing.assert_array_equal(hist, np.bincount(ref.accepted, minlength=33)[:33], err_msg=f"seed {seed}")
        compared += 1
        if compared >= need + 1:
            break
    assert compared >= need, f"too few seeds clear of ties: {seen}"
