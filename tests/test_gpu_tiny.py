"""Tiny fp32 decoder through the C ABI against the float64 oracle.

The GPU computes in plain fp32 (no TF32), the oracle in float64; the token
streams must match exactly.  Drafts must match wherever the oracle's top-2
margin is clear of fp32 rounding.
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import dflash_oracle as O

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
def weights():
    return syn.make_weights(SHAPE)


@pytest.fixture(scope="module")
def model(weights):
    return O.Model(O.Weights(weights), SHAPE)


@pytest.fixture(scope="module")
def engine(dfl, weights):
    eng = dfl.Engine(SHAPE, weights, max_batch=4, max_ctx=256)
    yield eng
    eng.close()


@pytest.fixture(scope="module")
def prompt():
    return syn.make_prompt(SHAPE, 64)


@pytest.fixture(scope="module")
def oracle_greedy(model, prompt):
    return O.greedy_generate(model, prompt, 128)


def test_speculative_stream_equals_oracle(engine, oracle_greedy, prompt):
    out, stats = engine.generate([prompt], 128)
    np.testing.assert_array_equal(out[0], oracle_greedy)
    assert stats["cycles"] >= 1
    assert stats["emitted_tokens"] == 128


def test_gpu_greedy_equals_oracle(engine, oracle_greedy, prompt):
    np.testing.assert_array_equal(engine.greedy_reference([prompt], 128)[0], oracle_greedy)


def test_cycle_by_cycle_against_oracle(engine, model, prompt):
    # Step the cycle through the ABI and compare drafts, k and bonus per cycle.
    ref = O.spec_generate(model, prompt, 64)
    b0 = engine.prefill(0, prompt)
    assert b0 == ref.tokens[0]
    try:
        for c in ref.cycles:
            assert engine.seq_info(0) == (c.position, c.bonus)
            drafts = engine.draft_block([0])[0]
            dp = O.draft_blocks(model.W, SHAPE, _oracle_ctx(model, prompt, ref, c.position), [(c.bonus, c.position)])
            srt = np.sort(dp.logits[1:], axis=1)
            clear = (srt[:, -1] - srt[:, -2]) > 1e-4
            np.testing.assert_array_equal(drafts[clear], c.drafts[clear])
            acc, n = engine.verify_accept([0], c.drafts)   # verify the oracle's drafts: same k
            assert n[0] == c.k + 1
            np.testing.assert_array_equal(acc[0, : c.k], c.drafts[: c.k])
            assert acc[0, c.k] == c.greedy[c.k]
    finally:
        engine.reset_seq(0)


_ctx_cache = {}


def _oracle_ctx(model, prompt, ref, position):
    """Oracle context cache for the verified stream up to `position`."""
    toks = np.concatenate([prompt, ref.tokens])[:position]
    key = position
    if key not in _ctx_cache:
        tp = O.teacher_forced(model, toks)
        cc = O.ContextCache(SHAPE.draft_layers, SHAPE.n_kv_heads, SHAPE.head_dim)
        O.inject_kv(model.W, SHAPE, cc, O.fuse_features(model.W, SHAPE, tp.taps))
        _ctx_cache[key] = cc
    return _ctx_cache[key]


def test_forced_correct_drafts_accept_all(engine, oracle_greedy, prompt):
    B = SHAPE.block_size
    engine.prefill(1, prompt)
    try:
        i = 0
        for _ in range(6):
            drafts = oracle_greedy[i + 1:i + B]
            acc, n = engine.verify_accept([1], drafts)
            assert n[0] == B
            np.testing.assert_array_equal(acc[0], oracle_greedy[i + 1:i + B + 1])
            i += B
    finally:
        engine.reset_seq(1)


@pytest.mark.parametrize("j", [1, 3, 7])
def test_forced_mismatch_at_j(engine, oracle_greedy, prompt, j):
    B = SHAPE.block_size
    engine.prefill(2, prompt)
    try:
        i = 0
        for _ in range(4):
            drafts = oracle_greedy[i + 1:i + B].copy()
            drafts[j - 1] = (drafts[j - 1] + 1) % (SHAPE.vocab - 1)
            acc, n = engine.verify_accept([2], drafts)
            assert n[0] == j
            np.testing.assert_array_equal(acc[0, :j], oracle_greedy[i + 1:i + j + 1])
            i += j
    finally:
        engine.reset_seq(2)


def test_batch_of_sequences_equals_oracle(engine, model):
    prompts = [syn.make_prompt(SHAPE, L, stream=s) for s, L in [(1, 20), (2, 33), (3, 47)]]
    out, _ = engine.generate(prompts, 40)
    for p, o in zip(prompts, out):
        np.testing.assert_array_equal(o, O.greedy_generate(model, p, 40))


def test_no_flow_between_blocks_of_a_batch(dfl, engine):
    # Two sequences drafted in one pass: changing the second one's prompt
    # leaves the first one's drafts and drafter states bit-identical.
    pa = syn.make_prompt(SHAPE, 30, stream=10)
    pb = syn.make_prompt(SHAPE, 30, stream=11)
    pc = syn.make_prompt(SHAPE, 30, stream=12)
    engine.debug(True)
    try:
        res = []
        for other in (pb, pc):
            engine.prefill(0, pa)
            engine.prefill(1, other)
            d = engine.draft_block([0, 1])
            h = engine.debug_read(dfl.DF_DBG_DRAFT_HIDDEN)
            res.append((d, h))
            engine.reset_seq(0)
            engine.reset_seq(1)
        B = SHAPE.block_size
        np.testing.assert_array_equal(res[0][0][0], res[1][0][0])
        np.testing.assert_array_equal(res[0][1][:B], res[1][1][:B])
        assert np.abs(res[0][1][B:] - res[1][1][B:]).max() > 0
    finally:
        engine.debug(False)


def test_shared_embedding_and_lm_head(dfl, engine):
    assert engine.weight_ptr(0) == engine.weight_ptr(1)
    assert engine.weight_ptr(2) == engine.weight_ptr(3)
    assert engine.weight_ptr(0) != engine.weight_ptr(2)


def test_errors_are_reported(dfl, engine, prompt):
    with pytest.raises(dfl.DfError) as e:
        engine.draft_block([3])            # slot never prefilled
    assert e.value.status == dfl.DF_ESTATE
    with pytest.raises(dfl.DfError) as e:
        engine.prefill(0, np.array([SHAPE.vocab + 5], np.int32))
    assert e.value.status == dfl.DF_EINVAL
    with pytest.raises(dfl.DfError):
        engine.prefill(0, np.zeros(300, np.int32))   # longer than max_ctx
    # the handle still works afterwards
    out, _ = engine.generate([prompt[:10]], 5)
    assert out.shape == (1, 5)
