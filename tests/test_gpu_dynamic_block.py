"""Block size per group of cycles on the GPU (df_set_block_range).

Source: [ABS] "DFlash：基于块扩散的闪存推测解码方法", 实践 2 and its 注意事项
(a large block rolls back more in long generations; the block size may follow
how predictable the text is).  Whatever the block sizes, every cycle emits
the target's own next tokens, so the output stays the greedy stream.

* A fixed block b < B: the tiny fp32 model's streams equal the oracle's
  greedy decoding, and each sequence's accepted counts equal the oracle's
  loop run with block size b; a batch of ragged prompts exercises the
  per-sequence strides of b-slot blocks.
* The adaptive range: lossless (tiny fp32 against the oracle, a small bf16
  model against the GPU's greedy decode); the block histogram shows the
  first group at b_max and later groups at the rule's size.
* Whole blocks accepted at b < B: a model whose target and drafter both
  always pick one token (a common direction added to every embedding row
  and to that token's LM-head row) keeps b - 1 drafts every cycle.
* Sampling at b = 4 equals the oracle's sampled loop with block size 4.
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import dflash_oracle as O

from _streams import assert_stream_matches

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SHAPE = syn.TINY


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__ as g
    g.build()
    import block_diffusion_speculative_layer_gb300 as m
    return m


@pytest.fixture(scope="module")
def tiny(dfl):
    w = syn.make_weights(SHAPE)
    eng = dfl.Engine(SHAPE, w, max_batch=3, max_ctx=256)
    yield eng, O.Model(O.Weights(w), SHAPE)
    eng.close()


def prompts3():
    return [syn.make_prompt(SHAPE, L, stream=s) for s, L in [(60, 33), (61, 12), (62, 50)]]


@pytest.mark.parametrize("b", [2, 4])
def test_fixed_block_equals_the_oracle(tiny, b):
    eng, model = tiny
    ps = prompts3()
    n_new = 41
    eng.set_block_range(b, b)
    try:
        out, stats = eng.generate(ps, n_new)
        hist = eng.accept_hist_per_seq(len(ps))
    finally:
        eng.set_block_range(SHAPE.block_size, SHAPE.block_size)
    assert stats["block_hist"][b] == stats["cycles"]
    mb = O.Model(model.W, SHAPE.replace(block_size=b))
    for i, p in enumerate(ps):
        np.testing.assert_array_equal(out[i], O.greedy_generate(model, p, n_new))
        ref = O.spec_generate(mb, p, n_new)
        np.testing.assert_array_equal(out[i], ref.tokens)
        np.testing.assert_array_equal(hist[i], np.bincount(ref.accepted, minlength=33)[:33])


def test_adaptive_range_is_lossless_tiny(tiny):
    eng, model = tiny
    ps = prompts3()[:2]
    eng.set_block_range(2, 8)
    try:
        out, stats = eng.generate(ps, 64)
    finally:
        eng.set_block_range(SHAPE.block_size, SHAPE.block_size)
    for i, p in enumerate(ps):
        np.testing.assert_array_equal(out[i], O.greedy_generate(model, p, 64))
    bh = stats["block_hist"]
    assert bh[8] >= 1                      # the first group runs at b_max
    assert sum(bh) == stats["cycles"]
    # random weights keep about one token per cycle: the rule then asks for b = 2
    assert bh[2] >= 1


def test_adaptive_range_is_lossless_bf16(dfl):
    shape = syn.ModelShape("small-bf16-blk", n_layers=8, d_model=512, n_q_heads=4, n_kv_heads=2, head_dim=128,
                           d_ffn=1024, vocab=2048, draft_layers=1, block_size=16, dtype="bf16")
    with dfl.Engine(shape, syn.make_weights(shape), max_batch=3, max_ctx=512) as eng:
        ps = [syn.make_prompt(shape, L, stream=s) for s, L in [(1, 70), (2, 9), (3, 130)]]
        greedy = eng.greedy_reference(ps, 48)
        for lo, hi in [(4, 4), (2, 16), (8, 8)]:
            eng.set_block_range(lo, hi)
            out, stats = eng.generate(ps, 48)
            np.testing.assert_array_equal(out, greedy, err_msg=f"range {lo}..{hi}")
            assert sum(stats["block_hist"]) == stats["cycles"]


def one_token_weights(shape, token, alpha=32.0, beta=1.0, seed=5):
    """Weights whose target and drafter always pick `token`: every embedding
    row gets alpha * u and LM-head row `token` gets beta * u, for one unit
    vector u, so the final normalised rows point along u."""
    w = syn.make_weights(shape)
    u = np.random.default_rng(seed).standard_normal(shape.d_model)
    u /= np.linalg.norm(u)
    w["embed"] = (w["embed"] + alpha * u[None, :]).astype(np.float32)
    lm = w["lm_head"].copy()
    lm[token] += (beta * u).astype(np.float32)
    w["lm_head"] = lm
    return w


@pytest.mark.parametrize("lo,hi", [(4, 4), (2, 8), (3, 3)])
def test_whole_blocks_accepted_at_smaller_blocks(dfl, lo, hi):
    tok = 5
    w = one_token_weights(SHAPE, tok)
    model = O.Model(O.Weights(w), SHAPE)
    ps = prompts3()
    n_new = 45
    with dfl.Engine(SHAPE, w, max_batch=3, max_ctx=256) as eng:
        eng.set_block_range(lo, hi)
        out, stats = eng.generate(ps, n_new)
        hist = eng.accept_hist_per_seq(len(ps))
    for i, p in enumerate(ps):
        ref = O.greedy_generate(model, p, n_new)
        assert (ref == tok).all()
        np.testing.assert_array_equal(out[i], ref)
    # every cycle keeps all b - 1 drafts; with b_min < b_max the block stays at b_max
    assert stats["block_hist"][hi] == stats["cycles"]
    assert (hist[:, hi - 1] >= 1).all() and hist[:, :hi - 1].sum() == 0
    assert stats["accepted_drafts"] == (hi - 1) * stats["cycles"]


def test_sampled_fixed_block_equals_the_oracle(tiny):
    eng, model = tiny
    prompt = syn.make_prompt(SHAPE, 40, stream=63)
    eng.set_block_range(4, 4)
    try:
        assert_stream_matches(eng, model, prompt, 24, 0.05, 1.0, range(1, 17), block=4)
    finally:
        eng.set_block_range(SHAPE.block_size, SHAPE.block_size)
