"""Pins of the oracle's sampling verification (no GPU).

What fixes the rule independently of the oracle's own code:
* temperature and nucleus filtering: scipy's softmax, hand-worked nucleus
  examples, and the greedy limit at temperature 0;
* the inverse-CDF draw: its interval boundaries;
* the rejection test: it reduces to the greedy prefix rule for one-hot
  distributions, keeps every draft when drafter and target agree, and (the
  property the pages state) leaves the target's distribution unchanged.  The
  last one is checked by simulation on a toy target whose next-token
  distribution depends on the prefix: the frequencies of the first and of
  the first two emitted tokens must match autoregressive sampling from the
  target within sampling error;
* the whole loop at temperature 0 equals greedy speculative decoding.
"""
import numpy as np
import pytest
from scipy.special import softmax

import synthetic as syn
from oracle import dflash_oracle as O


def test_temperature_is_a_scaled_softmax():
    rng = np.random.default_rng(1)
    logits = rng.normal(size=(3, 11))
    for t in (0.5, 0.7, 1.0, 1.6):
        np.testing.assert_allclose(O.sampling_probs(logits, t), softmax(logits / t, axis=1), rtol=1e-12)


def test_nucleus_keeps_the_fewest_tokens_reaching_top_p():
    p = np.array([[0.5, 0.3, 0.15, 0.05]])
    np.testing.assert_allclose(O.sampling_probs(np.log(p), 1.0, 0.7), [[0.625, 0.375, 0.0, 0.0]])
    np.testing.assert_allclose(O.sampling_probs(np.log(p), 1.0, 0.5), [[1.0, 0.0, 0.0, 0.0]])
    np.testing.assert_allclose(O.sampling_probs(np.log(p), 1.0, 0.96), [[0.5, 0.3, 0.15, 0.05]], rtol=1e-12)
    # unsorted input and a tie: the lower index of the tied pair enters first
    q = np.array([[0.1, 0.35, 0.2, 0.35]])
    np.testing.assert_allclose(O.sampling_probs(np.log(q), 1.0, 0.3), [[0.0, 1.0, 0.0, 0.0]])
    np.testing.assert_allclose(O.sampling_probs(np.log(q), 1.0, 0.4), [[0.0, 0.5, 0.0, 0.5]])
    np.testing.assert_allclose(O.sampling_probs(np.log(q), 1.0, 0.75), [[0.0, 0.35, 0.2, 0.35]] / np.float64(0.9))


def test_temperature_zero_is_the_argmax():
    logits = np.array([[0.1, 2.0, 2.0, -1.0], [3.0, 0.0, 1.0, 2.9]])
    np.testing.assert_array_equal(O.sampling_probs(logits, 0.0), [[0, 1, 0, 0], [1, 0, 0, 0]])


def test_draw_follows_the_cumulative_mass():
    assert [O.draw([0.2, 0.3, 0.5], u) for u in (0.0, 0.19, 0.2, 0.49, 0.5, 0.999)] == [0, 0, 1, 1, 2, 2]
    assert [O.draw([2.0, 0.0, 6.0], u) for u in (0.0, 0.24, 0.25, 0.9)] == [0, 0, 2, 2]   # unnormalised


def test_one_hot_distributions_give_the_greedy_rule():
    rng = np.random.default_rng(2)
    V, B = 5, 6
    for _ in range(300):
        drafts = rng.integers(0, V, B - 1)
        greedy = rng.integers(0, V, B)
        # make long matching prefixes likely
        m = rng.integers(0, B)
        greedy[: min(m, B - 1)] = drafts[: min(m, B - 1)]
        q = np.eye(V)[drafts]
        p = np.eye(V)[greedy]
        u_acc = rng.random(B - 1)
        got = O.accept_sampled(drafts, q, p, u_acc, float(rng.random()))
        assert got == O.accept_prefix(drafts, greedy)


def test_agreeing_drafter_keeps_every_draft():
    rng = np.random.default_rng(3)
    V, B = 7, 5
    for _ in range(200):
        rows = rng.dirichlet(np.ones(V), size=B)
        drafts = [O.draw(rows[i], rng.random()) for i in range(B - 1)]
        k, _ = O.accept_sampled(drafts, rows[: B - 1], rows, rng.random(B - 1), float(rng.random()))
        assert k == B - 1


class ToyTarget:
    """A next-token distribution for every prefix, drawn once per prefix."""

    def __init__(self, V, seed):
        self.V, self.rng, self.rows = V, np.random.default_rng(seed), {}

    def __call__(self, prefix):
        key = tuple(int(t) for t in prefix)
        if key not in self.rows:
            self.rows[key] = self.rng.dirichlet(np.full(self.V, 0.7))
        return self.rows[key]


def simulate(accept, target, q, n, seed):
    """n cycles from the empty prefix: drafts from q, the rejection test,
    the emitted tokens of each cycle."""
    rng = np.random.default_rng(seed)
    B = len(q) + 1
    out = []
    for _ in range(n):
        u = rng.random(2 * (B - 1) + 1)
        drafts = [O.draw(q[i], u[i]) for i in range(B - 1)]
        p_rows = np.stack([target(drafts[:i]) for i in range(B)])
        k, tok = accept(drafts, q, p_rows, u[B - 1: 2 * (B - 1)], float(u[-1]))
        out.append(drafts[:k] + [tok])
    return out


def check_keeps_target_distribution(accept, n=120_000, seed=11):
    V = 4
    target = ToyTarget(V, seed=5)
    # a drafter that disagrees with the target on purpose
    q = np.array([[0.55, 0.05, 0.1, 0.3], [0.1, 0.6, 0.25, 0.05]])
    cyc = simulate(accept, target, q, n, seed)
    p0 = target([])
    # first token of the generation
    first = np.bincount([c[0] for c in cyc], minlength=V) / n
    tol = 5 * np.sqrt(p0 * (1 - p0) / n) + 1e-4
    assert np.all(np.abs(first - p0) <= tol), (first, p0)
    # first two tokens: from this cycle, or (one token emitted) from the next
    # cycle, whose first token follows the target at prefix (t1,)
    joint = np.zeros((V, V))
    for c in cyc:
        if len(c) >= 2:
            joint[c[0], c[1]] += 1.0
        else:
            joint[c[0]] += target([c[0]])
    joint /= n
    exact = np.array([[p0[a] * target([a])[b] for b in range(V)] for a in range(V)])
    tol2 = 5 * np.sqrt(exact * (1 - exact) / n) + 1e-4
    assert np.all(np.abs(joint - exact) <= tol2), (joint, exact)


def test_rejection_test_keeps_the_target_distribution():
    check_keeps_target_distribution(O.accept_sampled)


def test_sampling_loop_at_temperature_zero_is_greedy_speculation():
    shape = syn.TINY.replace(n_layers=8, d_model=64, n_q_heads=2, n_kv_heads=2, head_dim=32, d_ffn=128,
                             vocab=64, block_size=4)
    w = syn.make_weights(shape, gain_std=0.2)
    m = O.Model(O.Weights(w), shape)
    prompt = syn.make_prompt(shape, 12, stream=3)
    rng = np.random.default_rng(4)
    got = O.spec_generate_sampled(m, prompt, 20, 0.0, 1.0, lambda n: rng.random(n))
    ref = O.spec_generate(m, prompt, 20)
    np.testing.assert_array_equal(got.tokens, ref.tokens)
    np.testing.assert_array_equal(got.tokens, O.greedy_generate(m, prompt, 20))
    assert got.accepted == ref.accepted


def test_draw_margin_is_the_distance_to_the_deciding_interval():
    assert O.draw_margin([0.2, 0.3, 0.5], 0.25) == pytest.approx(0.05)
    assert O.draw_margin([0.2, 0.3, 0.5], 0.1) == pytest.approx(0.1)
    assert O.draw_margin([0.2, 0.3, 0.5], 0.0) == 0.0          # on the lower end
    assert O.draw_margin([0.2, 0.3, 0.5], 0.5) == 0.0          # on a boundary
    assert O.draw_margin([2.0, 6.0], 0.5) == pytest.approx(0.25)   # unnormalised: fraction of the total


def test_margins_bound_the_effect_of_perturbed_masses():
    # a draw or a test whose margin exceeds the perturbation keeps its result
    rng = np.random.default_rng(8)
    kept = 0
    for _ in range(400):
        V, B = 6, 4
        q = rng.dirichlet(np.ones(V), size=B - 1)
        p = rng.dirichlet(np.ones(V), size=B)
        drafts = [O.draw(q[i], rng.random()) for i in range(B - 1)]
        ua, uf = rng.random(B - 1), float(rng.random())
        m = O.accept_margin(drafts, q, p, ua, uf)
        eps = 1e-3
        if m <= 20 * eps:
            continue
        kept += 1
        q2 = q * (1 + eps * rng.uniform(-1, 1, q.shape))
        p2 = p * (1 + eps * rng.uniform(-1, 1, p.shape))
        q2 /= q2.sum(axis=1, keepdims=True)
        p2 /= p2.sum(axis=1, keepdims=True)
        assert O.accept_sampled(drafts, q2, p2, ua, uf) == O.accept_sampled(drafts, q, p, ua, uf)
        u = float(rng.random())
        if O.draw_margin(p[0], u) > 20 * eps:
            assert O.draw(p2[0], u) == O.draw(p[0], u)
    assert kept > 200


def test_accept_margin_examples():
    q = np.array([[0.5, 0.5]])
    p = np.array([[0.25, 0.75], [1.0, 0.0]])
    # kept (0.4 < p/q = 0.5, margin 0.1), then the final draw from [1, 0] at 0.1 (margin 0.1)
    assert O.accept_sampled([0], q, p, [0.4], 0.1) == (1, 0)
    assert O.accept_margin([0], q, p, [0.4], 0.1) == pytest.approx(0.1)
    # rejected (0.55 > 0.5, margin 0.05); residual [0, 0.25] drawn at 0.1 (margin 0.1)
    assert O.accept_sampled([0], q, p, [0.55], 0.1) == (0, 1)
    assert O.accept_margin([0], q, p, [0.55], 0.1) == pytest.approx(0.05)


def test_nucleus_margin_examples():
    lg = np.log([[0.5, 0.3, 0.15, 0.05]])
    assert O.nucleus_margin(lg, 1.0, 0.7) == pytest.approx(0.1)     # cut after 0.8; 0.5 is 0.2 below
    assert O.nucleus_margin(lg, 1.0, 0.79) == pytest.approx(0.01)
    assert O.nucleus_margin(lg, 1.0, 1.0) == np.inf
    assert O.nucleus_margin(lg, 0.0, 0.5) == np.inf
