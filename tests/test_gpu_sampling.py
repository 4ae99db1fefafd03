"""Speculative sampling on the GPU against the float64 oracle.

Sources: [ABS] "DFlash：基于块扩散的闪存推测解码方法", 实践 4 (temperature and
top-p sampling with drafter and target aligned) and 核心思想 step 3 with its
Q&A (verification keeps the target's output distribution).

* Draws and the rejection test, one operation at a time, on the same fp32
  logits and uniforms as the oracle; where a decision lies within rounding
  of a tie (closer than MARGIN) the GPU's result must be one of the correct
  ones instead.
* The property the pages state, measured on the GPU: over many blocks the
  first emitted token follows the target's distribution, whatever the
  drafter's (Monte Carlo, five standard errors).
* Temperature 0 is greedy decoding: df_generate_sampled(T = 0) equals
  df_generate and the GPU's greedy decode.
* The tiny fp32 model's sampled stream equals the oracle's
  ``spec_generate_sampled`` with the same Philox uniforms, for seeds whose
  every decision is farther than STREAM_MARGIN from a tie (the fp32 logits
  differ from float64 by about 1e-6 relative).
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import dflash_oracle as O

from _streams import Uniforms, assert_stream_matches

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

MARGIN = 5e-5          # decisions closer than this to a tie may go either way (single ops)


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__ as g
    g.build()
    import block_diffusion_speculative_layer_gb300 as m
    return m


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def logits(rows, V, scale, seed):
    g = np.random.default_rng(seed)
    return (g.standard_normal((rows, V)) * scale).astype(np.float32)


# ----------------------------------------------------------------- draws
# Logit scales keep most decisions clear of ties: a flat row over 151936
# tokens puts every nucleus cut within 1e-5 of top_p.
@pytest.mark.parametrize("V,T,top_p,scale", [(7, 1.0, 1.0, 2.0), (1000, 0.7, 0.9, 2.0), (4097, 1.3, 0.5, 2.0),
                                             (151936, 1.0, 0.95, 8.0), (151936, 0.6, 1.0, 2.0), (1000, 0.0, 1.0, 2.0)])
def test_draws_equal_the_oracle(dfl, V, T, top_p, scale):
    rows = 64
    x = logits(rows, V, scale, seed=V + 17)
    u = syn.philox_uniforms(5, V, 0, rows)
    got = dfl.sample_draw(cuda(x), T, top_p, cuda(u.astype(np.float32))).cpu().numpy()
    x64 = x.astype(np.float64)
    checked = 0
    for r in range(rows):
        probs = O.sampling_probs(x64[r:r + 1], T, top_p)[0]
        if O.nucleus_margin(x64[r:r + 1], T, top_p) >= MARGIN and O.draw_margin(probs, u[r]) >= MARGIN:
            assert got[r] == O.draw(probs, u[r]), f"row {r}"
            checked += 1
        else:
            full = O.sampling_probs(x64[r:r + 1], T, 1.0)[0]
            assert full[got[r]] > 0      # a token the distribution can give
    assert checked >= rows // 2


# ----------------------------------------------------------------- the rejection test
@pytest.mark.parametrize("B,V,T,top_p,relation,scale", [(4, 50, 1.0, 1.0, "independent", 2.0),
                                                        (8, 1000, 0.8, 0.9, "close", 4.0),
                                                        (16, 300, 1.0, 1.0, "equal", 2.0),
                                                        (2, 5, 1.2, 1.0, "independent", 2.0),
                                                        (16, 151936, 1.0, 0.9, "close", 8.0)])
def test_accept_sampled_equals_the_oracle(dfl, B, V, T, top_p, relation, scale):
    nseq = 24 if V < 100000 else 6
    rng = np.random.default_rng(B * 1000 + V)
    p = (rng.standard_normal((nseq, B, V)) * scale).astype(np.float32)
    if relation == "independent":
        q = (rng.standard_normal((nseq, B - 1, V)) * scale).astype(np.float32)
    elif relation == "equal":
        q = p[:, :B - 1].copy()
    else:
        q = (p[:, :B - 1] + rng.standard_normal((nseq, B - 1, V)) * 0.15 * scale).astype(np.float32)
    ud = syn.philox_uniforms(9, B, 0, nseq * (B - 1)).reshape(nseq, B - 1)
    ut = syn.philox_uniforms(9, B + 100, 0, nseq * B).reshape(nseq, B)
    q64, p64 = q.astype(np.float64), p.astype(np.float64)
    drafts = np.zeros((nseq, B - 1), np.int32)
    for b in range(nseq):
        qr = O.sampling_probs(q64[b], T, top_p)
        drafts[b] = [O.draw(qr[i], ud[b, i]) for i in range(B - 1)]
    k, tok = dfl.accept_sampled(cuda(drafts), cuda(q), cuda(p), T, top_p, cuda(ut.astype(np.float32)))
    k, tok = k.cpu().numpy(), tok.cpu().numpy()
    checked = 0
    for b in range(nseq):
        qr = O.sampling_probs(q64[b], T, top_p)
        pr = O.sampling_probs(p64[b], T, top_p)
        margin = min(O.nucleus_margin(q64[b], T, top_p), O.nucleus_margin(p64[b], T, top_p),
                     O.accept_margin(drafts[b], qr, pr, ut[b, :B - 1], ut[b, B - 1]))
        kk, tt = O.accept_sampled(drafts[b], qr, pr, ut[b, :B - 1], ut[b, B - 1])
        if margin >= MARGIN:
            assert (k[b], tok[b]) == (kk, tt), f"block {b}"
            checked += 1
        else:
            assert 0 <= k[b] <= B - 1 and 0 <= tok[b] < V
    assert checked >= nseq // 2
    if relation == "equal":
        assert (k == B - 1).all()       # a drafter equal to the target keeps every draft


def test_rejection_keeps_the_target_distribution(dfl):
    """Many independent blocks of two slots with fixed drafter and target
    distributions: the first emitted token (the kept draft, or the
    replacement) must follow the target's distribution p_0, and after a kept
    draft the next token must follow p_1."""
    V, n = 6, 1 << 18
    ql = np.array([2.0, 0.5, 0.0, -1.0, 1.0, 0.3], np.float32)
    pl0 = np.array([0.0, 1.5, 0.2, 0.9, -0.5, 0.7], np.float32)
    pl1 = np.array([1.0, -1.0, 0.0, 0.5, 0.2, -0.3], np.float32)
    T = 1.0
    q = cuda(np.broadcast_to(ql, (n, 1, V)))
    p = cuda(np.broadcast_to(np.stack([pl0, pl1]), (n, 2, V)))
    ud = dfl.philox_uniforms(3, 0, 0, n)
    ut = dfl.philox_uniforms(3, 1, 0, 2 * n).reshape(n, 2)
    drafts = dfl.sample_draw(q.reshape(n, V), T, 1.0, ud).reshape(n, 1)
    k, tok = dfl.accept_sampled(drafts, q, p, T, 1.0, ut)
    k, tok, d = k.cpu().numpy(), tok.cpu().numpy(), drafts.cpu().numpy()[:, 0]
    first = np.where(k == 1, d, tok)
    p0 = O.sampling_probs(pl0.astype(np.float64)[None], T)[0]
    freq = np.bincount(first, minlength=V) / n
    se = np.sqrt(p0 * (1 - p0) / n)
    assert (np.abs(freq - p0) <= 5 * se).all(), (freq, p0)
    second = tok[k == 1]
    p1 = O.sampling_probs(pl1.astype(np.float64)[None], T)[0]
    f1 = np.bincount(second, minlength=V) / len(second)
    se1 = np.sqrt(p1 * (1 - p1) / len(second))
    assert (np.abs(f1 - p1) <= 5 * se1).all(), (f1, p1)


# ----------------------------------------------------------------- the engine's sampled cycle
@pytest.fixture(scope="module")
def tiny(dfl):
    w = syn.make_weights(syn.TINY)
    eng = dfl.Engine(syn.TINY, w, max_batch=3, max_ctx=256)
    yield eng, O.Model(O.Weights(w), syn.TINY)
    eng.close()


def test_temperature_zero_is_greedy_tiny(tiny):
    eng, _ = tiny
    prompts = [syn.make_prompt(syn.TINY, L, stream=s) for s, L in [(30, 40), (31, 17)]]
    samp, _ = eng.generate_sampled(prompts, 48, temperature=0.0, top_p=1.0, seed=1)
    greedy, _ = eng.generate(prompts, 48)
    np.testing.assert_array_equal(samp, greedy)
    np.testing.assert_array_equal(greedy, eng.greedy_reference(prompts, 48))


def test_temperature_zero_is_greedy_bf16(dfl):
    shape = syn.ModelShape("small-bf16-samp", n_layers=8, d_model=512, n_q_heads=4, n_kv_heads=2, head_dim=128,
                           d_ffn=1024, vocab=2048, draft_layers=1, block_size=8, dtype="bf16")
    with dfl.Engine(shape, syn.make_weights(shape), max_batch=2, max_ctx=256) as eng:
        prompts = [syn.make_prompt(shape, L, stream=s) for s, L in [(1, 33), (2, 60)]]
        samp, _ = eng.generate_sampled(prompts, 40, temperature=0.0, top_p=0.9, seed=4)
        np.testing.assert_array_equal(samp, eng.greedy_reference(prompts, 40))


# (temperature, top_p, new tokens) whose streams mostly stay clear of ties
@pytest.mark.parametrize("T,top_p,n_new", [(0.03, 1.0, 24), (0.05, 0.8, 16), (0.05, 1.0, 24)])
def test_sampled_stream_equals_the_oracle_tiny(tiny, T, top_p, n_new):
    eng, model = tiny
    prompt = syn.make_prompt(syn.TINY, 48, stream=40)
    assert_stream_matches(eng, model, prompt, n_new, T, top_p, range(1, 17))


def test_sampled_is_deterministic_and_batch_invariant(tiny):
    eng, _ = tiny
    prompts = [syn.make_prompt(syn.TINY, L, stream=s) for s, L in [(50, 20), (51, 45), (52, 9)]]
    a, _ = eng.generate_sampled(prompts, 40, temperature=0.8, top_p=0.9, seed=77)
    b, _ = eng.generate_sampled(prompts, 40, temperature=0.8, top_p=0.9, seed=77)
    np.testing.assert_array_equal(a, b)
    # sequence i draws from Philox stream i: alone in its batch (as stream 0) only the first matches
    alone, _ = eng.generate_sampled(prompts[:1], 40, temperature=0.8, top_p=0.9, seed=77)
    np.testing.assert_array_equal(alone[0], a[0])
