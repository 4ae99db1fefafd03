"""Pins of the CPU oracle against things other than itself.

Library routines (torch CPU attention, RMSNorm, SiLU), closed forms, golden
values the pages fix, invariants the method guarantees and brute force on
tiny inputs.  No GPU.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synthetic as syn
from oracle import dflash_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny(**kw):
    return syn.TINY.replace(**kw)


def model(shape, seed=0, gain_std=0.0):
    return O.Model(O.Weights(syn.make_weights(shape, seed=seed, gain_std=gain_std)), shape)


# ---------------------------------------------------------------- feature layers

def test_feature_layers_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "feature_layers.txt")) if l.strip() and l[0] != "#"]
    assert rows
    for r in rows:
        L, want = int(r[0]), [int(x) for x in r[1:]]
        assert O.feature_layers(L) == want


@pytest.mark.parametrize("L", range(8, 130))
def test_feature_layers_uniform(L):
    s = O.feature_layers(L)
    assert s[0] == 2 and s[-1] == L - 2
    assert all(b > a for a, b in zip(s, s[1:]))
    exact = [2 + i * (L - 4) / 4 for i in range(5)]
    assert all(abs(a - b) <= 0.5 for a, b in zip(s, exact))


def test_feature_layers_rejects_shallow():
    with pytest.raises(ValueError):
        O.feature_layers(7)


# ---------------------------------------------------------------- building blocks

def test_rms_norm_matches_torch():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 96))
    g = 1 + 0.1 * rng.standard_normal(96)
    ref = F.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(x, g, 1e-6), ref, rtol=1e-12, atol=1e-12)


def test_silu_matches_torch():
    x = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(O.silu(x), F.silu(torch.from_numpy(x)).numpy(), rtol=1e-12, atol=1e-15)


def test_rope_is_complex_rotation():
    # Independent formulation: pair (x_j, x_{j+hd/2}) as a complex number times e^{i pos w_j}.
    rng = np.random.default_rng(4)
    hd, theta = 64, 1e6
    x = rng.standard_normal((5, 3, hd))
    pos = np.array([0, 1, 7, 300, 40000])
    z = x[..., : hd // 2] + 1j * x[..., hd // 2:]
    w = np.array([theta ** (-(2 * j) / hd) for j in range(hd // 2)])
    zr = z * np.exp(1j * pos[:, None, None] * w[None, None, :])
    want = np.concatenate([zr.real, zr.imag], axis=-1)
    np.testing.assert_allclose(O.rope(x, pos, theta), want, rtol=1e-10, atol=1e-10)


def test_rope_relative_position():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    dots = []
    for m, n in [(10, 3), (107, 100), (1007, 1000)]:
        dots.append(float(np.sum(O.rope(q, np.array([m]), 1e6) * O.rope(k, np.array([n]), 1e6))))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)
    np.testing.assert_allclose(O.rope(q, np.array([0]), 1e6), q)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (32, 8)])
def test_attention_matches_torch_sdpa(hq, hkv):
    rng = np.random.default_rng(6)
    n, T, hd = 6, 11, 32
    q = rng.standard_normal((n, hq, hd))
    k = rng.standard_normal((T, hkv, hd))
    v = rng.standard_normal((T, hkv, hd))
    pos = np.arange(T - n, T)
    visible = np.arange(T)[None, :] <= pos[:, None]
    got = O.attention(q, k, v, visible)
    tq = torch.from_numpy(q).permute(1, 0, 2)                      # [H, n, hd]
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(visible)).permute(1, 0, 2)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_argmax_lowest_index_on_ties():
    x = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0]])
    assert O.argmax_lowest(x).tolist() == [1, 0]


# ---------------------------------------------------------------- target decoder

def test_target_single_token_closed_form():
    # One token, one layer: softmax over a single key is 1, so the attention
    # output is v itself; the whole pass has a closed form.
    s = tiny(n_layers=8)
    m = model(s, seed=11, gain_std=0.1)
    W = m.W
    cache = O.KVCache(s.n_layers, s.n_kv_heads, s.head_dim)
    tok = 17
    tp = O.target_forward(W, s, [tok], cache)
    h = W["embed"][[tok]]
    eps = s.rms_eps
    for l in range(s.n_layers):
        x = h / np.sqrt(np.mean(h * h) + eps) * W[f"t{l}.attn_norm"]
        v = x @ W[f"t{l}.wv"].T                                # [1, kv_dim]; heads equal groups here
        h = h + v @ W[f"t{l}.wo"].T
        y = h / np.sqrt(np.mean(h * h) + eps) * W[f"t{l}.mlp_norm"]
        g, u = y @ W[f"t{l}.w_gate"].T, y @ W[f"t{l}.w_up"].T
        h = h + (g / (1 + np.exp(-g)) * u) @ W[f"t{l}.w_down"].T
    hf = h / np.sqrt(np.mean(h * h) + eps) * W["final_norm"]
    np.testing.assert_allclose(tp.logits, hf @ W["lm_head"].T, rtol=1e-10, atol=1e-12)


def test_target_incremental_equals_full():
    s = tiny()
    m = model(s, seed=12)
    toks = syn.make_prompt(s, 20, seed=5)
    full = O.target_forward(m.W, s, toks, O.KVCache(s.n_layers, s.n_kv_heads, s.head_dim))
    cache = O.KVCache(s.n_layers, s.n_kv_heads, s.head_dim)
    parts = [O.target_forward(m.W, s, toks[:13], cache), O.target_forward(m.W, s, toks[13:17], cache)]
    parts += [O.target_forward(m.W, s, [t], cache) for t in toks[17:]]
    inc = np.concatenate([p.logits for p in parts])
    np.testing.assert_allclose(inc, full.logits, rtol=1e-9, atol=1e-11)
    taps = np.concatenate([p.taps for p in parts])
    np.testing.assert_allclose(taps, full.taps, rtol=1e-9, atol=1e-11)


def test_target_causal():
    s = tiny()
    m = model(s, seed=13)
    toks = syn.make_prompt(s, 12, seed=6)
    a = O.teacher_forced(m, toks)
    t2 = toks.copy()
    t2[8] = (t2[8] + 1) % (s.vocab - 1)
    b = O.teacher_forced(m, t2)
    np.testing.assert_array_equal(a.logits[:8], b.logits[:8])
    assert np.abs(a.logits[8:] - b.logits[8:]).max() > 0


def test_target_relative_positions():
    # RoPE makes attention depend on position differences only: shifting
    # every position of a causal segment by the same amount leaves a decoder
    # layer's output unchanged (up to rounding).
    s = tiny()
    m = model(s, seed=21)
    rng = np.random.default_rng(22)
    h = rng.standard_normal((9, s.d_model))

    def run(offset):
        pos = np.arange(offset, offset + 9)

        def kv_source(k, v):
            return k, v, np.arange(9)[None, :] <= np.arange(9)[:, None]

        return O.decoder_layer(m.W, "t0", s, h, pos, kv_source)

    np.testing.assert_allclose(run(0), run(1000), rtol=1e-8, atol=1e-9)
    # ...and the order of earlier tokens matters (a model without RoPE on
    # both q and k would be blind to it in a way this catches above).
    def run_keys(offset_q, offset_k):
        pos_q = np.arange(offset_q, offset_q + 9)
        pos_k = np.arange(offset_k, offset_k + 9)
        x = O.rms_norm(h, m.W["t0.attn_norm"], s.rms_eps)
        q = O.rope((x @ m.W["t0.wq"].T).reshape(9, s.n_q_heads, s.head_dim), pos_q, s.rope_theta)
        k = O.rope((x @ m.W["t0.wk"].T).reshape(9, s.n_kv_heads, s.head_dim), pos_k, s.rope_theta)
        return np.einsum("qhd,khd->hqk", q, k)

    np.testing.assert_allclose(run_keys(0, 0), run_keys(500, 500), rtol=1e-8, atol=1e-9)
    assert np.abs(run_keys(0, 0) - run_keys(0, 3)).max() > 1e-3


def test_taps_are_layer_outputs():
    s = tiny()
    m = model(s, seed=14)
    tp = O.teacher_forced(m, syn.make_prompt(s, 5, seed=7))
    for i, l in enumerate(O.feature_layers(s.n_layers)):
        np.testing.assert_array_equal(tp.taps[:, i], tp.hidden[l])


def _truncated(m, keep):
    """The same model with only its first `keep` target layers."""
    raw = {k: v for k, v in m.W.raw.items() if not (k[0] == "t" and int(k[1:k.index(".")]) >= keep)}
    return O.Model(O.Weights(raw), m.cfg.replace(n_layers=keep))


def _silenced(m, keep):
    """The same model with target layers keep.. made the identity (their
    attention output and down projections zeroed)."""
    raw = dict(m.W.raw)
    for l in range(keep, m.cfg.n_layers):
        for name in (f"t{l}.wo", f"t{l}.w_down"):
            raw[name] = np.zeros_like(raw[name])
    return O.Model(O.Weights(raw), m.cfg)


def test_tap_is_the_output_of_its_layer():
    # Tap i of an L-layer model is the output of (1-based) layer s_i: the
    # pre-norm final residual of the same model cut after s_i layers, either
    # truncated (s_i >= 8, the oracle's smallest model) or with the layers
    # after s_i made the identity.  Independent of the tap loop's indexing.
    s = tiny(n_layers=20)
    m = model(s, seed=23)
    toks = syn.make_prompt(s, 6, seed=8)
    full = O.teacher_forced(m, toks)
    feats = O.feature_layers(s.n_layers)
    assert feats == [2, 6, 10, 14, 18]
    for i, layer in enumerate(feats):
        cut = O.teacher_forced(_silenced(m, layer), toks).hidden[-1]
        np.testing.assert_allclose(full.taps[:, i], cut, rtol=0, atol=1e-12)
        if layer >= 8:
            trunc = O.teacher_forced(_truncated(m, layer), toks).hidden[-1]
            np.testing.assert_allclose(full.taps[:, i], trunc, rtol=0, atol=1e-12)
        # not the input of that layer, nor the output of the next one
        assert np.abs(full.taps[:, i] - O.teacher_forced(_silenced(m, layer - 1), toks).hidden[-1]).max() > 1e-6
        assert np.abs(full.taps[:, i] - O.teacher_forced(_silenced(m, layer + 1), toks).hidden[-1]).max() > 1e-6


# ---------------------------------------------------------------- fusion, injection, drafter

def test_fused_context_has_unit_rms():
    s = tiny()
    m = model(s, seed=15)
    taps = np.random.default_rng(8).standard_normal((9, 5, s.d_model))
    ctx = O.fuse_features(m.W, s, taps)
    rms = np.sqrt(np.mean(ctx * ctx, axis=1))
    # gain 1: RMSNorm makes each row's RMS sqrt(ms / (ms + eps)), i.e. 1 up to eps.
    np.testing.assert_allclose(rms, 1.0, atol=1e-5)


def test_fusion_concat_order_shallow_to_deep():
    # With W_fc = [I 0 0 0 0] only the shallowest tap survives, etc.
    s = tiny()
    d = s.d_model
    rng = np.random.default_rng(9)
    taps = rng.standard_normal((3, 5, d))
    for j in range(5):
        fc = np.zeros((d, 5 * d))
        fc[:, j * d:(j + 1) * d] = np.eye(d)
        W = O.Weights({"fc": fc.astype(np.float32), "fc_norm": np.ones(d, np.float32)})
        ctx = O.fuse_features(W, s, taps)
        np.testing.assert_allclose(ctx, O.rms_norm(taps[:, j], np.ones(d), s.rms_eps), rtol=1e-12)


def test_injected_keys_match_block_keys_for_same_input():
    # Injection uses the drafter layer's own W_k/W_v and RoPE at the context
    # row's absolute position: injecting a context row equal to a block
    # token's normalised layer input, at that token's position, gives the key
    # and value the drafter layer itself makes for the token in a block pass
    # (read from the layer's keys/values, not restated).
    s = tiny(draft_layers=2)
    m = model(s, seed=16, gain_std=0.1)
    W = m.W
    B = s.block_size
    anchor = 7
    toks = np.asarray([3] + [s.mask_token_id] * (B - 1))
    pos = np.arange(anchor, anchor + B)
    h = W["embed"][toks]
    for l in range(s.draft_layers):
        seen = {}

        def kv(k_new, v_new):
            seen["k"], seen["v"] = k_new, v_new
            return k_new, v_new, np.ones((B, B), bool)

        h_next = O.decoder_layer(W, f"d{l}", s, h, pos, kv)
        x = O.rms_norm(h, W[f"d{l}.attn_norm"], s.rms_eps)
        cc = O.ContextCache(s.draft_layers, s.n_kv_heads, s.head_dim)
        O.inject_kv(W, s, cc, np.random.default_rng(10).standard_normal((anchor, s.d_model)))
        O.inject_kv(W, s, cc, x)
        np.testing.assert_allclose(cc.k[l][anchor:], seen["k"], rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(cc.v[l][anchor:], seen["v"], rtol=1e-10, atol=1e-13)
        h = h_next


def _ctx_cache(m, n, seed):
    s = m.cfg
    cc = O.ContextCache(s.draft_layers, s.n_kv_heads, s.head_dim)
    taps = np.random.default_rng(seed).standard_normal((n, 5, s.d_model))
    O.inject_kv(m.W, s, cc, O.fuse_features(m.W, s, taps))
    return cc


def test_no_information_flow_between_blocks():
    s = tiny(draft_layers=2)
    m = model(s, seed=17)
    cc = _ctx_cache(m, 40, 11)
    joint = O.draft_blocks(m.W, s, cc, [(5, 20), (9, 30)])
    alone = O.draft_blocks(m.W, s, cc, [(5, 20)])
    B = s.block_size
    np.testing.assert_allclose(joint.hidden[:B], alone.hidden, rtol=1e-12, atol=1e-14)
    # perturb the later block's anchor: the earlier block is bit-unchanged
    pert = O.draft_blocks(m.W, s, cc, [(5, 20), (10, 30)])
    np.testing.assert_array_equal(pert.hidden[:B], joint.hidden[:B])
    assert np.abs(pert.hidden[B:] - joint.hidden[B:]).max() > 0


def test_bidirectional_inside_block():
    # A later slot influences an earlier one: change the last slot's input by
    # moving the block to a different anchor token only at slot 0 vs keep it
    # and change the context past the anchor (never visible).
    s = tiny(draft_layers=1)
    m = model(s, seed=18)
    cc = _ctx_cache(m, 30, 12)
    a = O.draft_blocks(m.W, s, cc, [(5, 20)])
    # Slot 0 changes -> every slot changes (slot 0 is visible to all).
    b = O.draft_blocks(m.W, s, cc, [(6, 20)])
    assert np.all(np.abs(a.hidden - b.hidden).max(axis=1) > 0)
    # Context entries at or after the anchor position are invisible.
    cc2 = _ctx_cache(m, 30, 12)
    cc2.k[0][20:] += 1.0
    cc2.v[0][20:] -= 1.0
    c = O.draft_blocks(m.W, s, cc2, [(5, 20)])
    np.testing.assert_array_equal(a.hidden, c.hidden)


def test_bidirectional_later_slot_reaches_earlier_slot():
    # Build the drafter input by hand with a different token in the last slot:
    # slot 1's output must change (a causal mask would leave it unchanged).
    s = tiny(draft_layers=1)
    m = model(s, seed=19)
    cc = _ctx_cache(m, 10, 13)
    B = s.block_size
    orig_mask = s.mask_token_id
    base = O.draft_blocks(m.W, s, cc, [(5, 10)])
    W2 = dict(m.W.raw)
    emb = W2["embed"].copy()
    # give the mask id a new embedding only for the comparison run: every
    # masked slot changes, slot 0 does not; slot 0's output must change
    # through attention to the later slots.
    emb[orig_mask] = emb[orig_mask] + 0.5
    W2["embed"] = emb
    alt = O.draft_blocks(O.Weights(W2), s, cc, [(5, 10)])
    assert np.abs(alt.hidden[0] - base.hidden[0]).max() > 1e-6
    assert alt.hidden.shape[0] == B


# ---------------------------------------------------------------- acceptance

def brute_force_k(drafts, greedy):
    best = 0
    for j in range(len(drafts) + 1):
        if all(drafts[i] == greedy[i] for i in range(j)):
            best = j
    return best


def test_accept_brute_force():
    rng = np.random.default_rng(20)
    for _ in range(3000):
        B = int(rng.integers(2, 17))
        g = rng.integers(0, 3, size=B)
        d = rng.integers(0, 3, size=B - 1)
        k, bonus = O.accept_prefix(d, g)
        assert k == brute_force_k(d, g)
        assert bonus == g[k]


# ---------------------------------------------------------------- losslessness

@pytest.mark.parametrize("B,seed", [(2, 0), (4, 1), (8, 0), (8, 2)])
def test_spec_equals_greedy(B, seed):
    s = tiny(block_size=B)
    m = model(s, seed=seed)
    prompt = syn.make_prompt(s, 24, seed=seed + 1)
    g = O.greedy_generate(m, prompt, 40)
    r = O.spec_generate(m, prompt, 40)
    np.testing.assert_array_equal(r.tokens, g)
    assert sum(c.k + 1 for c in r.cycles) + 1 >= 40


def test_forced_correct_drafts_accept_everything():
    s = tiny(block_size=8)
    m = model(s, seed=3)
    prompt = syn.make_prompt(s, 16, seed=4)
    g = O.greedy_generate(m, prompt, 60)
    P = len(prompt)

    def hook(bonus, pos, drafts):
        i = pos - P            # index of the bonus in the output stream
        return g[i + 1:i + s.block_size]

    r = O.spec_generate(m, prompt, 50, draft_hook=hook)
    np.testing.assert_array_equal(r.tokens, g[:50])
    assert all(c.k == s.block_size - 1 for c in r.cycles)


@pytest.mark.parametrize("j", range(1, 8))
def test_forced_mismatch_at_j(j):
    s = tiny(block_size=8)
    m = model(s, seed=5)
    prompt = syn.make_prompt(s, 16, seed=6)
    g = O.greedy_generate(m, prompt, 80)
    P = len(prompt)

    def hook(bonus, pos, drafts):
        i = pos - P
        d = g[i + 1:i + s.block_size].copy()
        d[j - 1] = (d[j - 1] + 1) % (s.vocab - 1)
        return d

    r = O.spec_generate(m, prompt, 60, draft_hook=hook)
    np.testing.assert_array_equal(r.tokens, g[:60])
    for c in r.cycles:
        assert c.k == j - 1
        assert c.greedy[c.k] == g[c.position - P + c.k + 1]


def test_all_wrong_drafts_is_plain_ar():
    s = tiny(block_size=4)
    m = model(s, seed=6)
    prompt = syn.make_prompt(s, 10, seed=7)
    g = O.greedy_generate(m, prompt, 30)
    P = len(prompt)

    def hook(bonus, pos, drafts):
        i = pos - P
        return (g[i + 1:i + 4] + 1) % (s.vocab - 1)

    r = O.spec_generate(m, prompt, 30, draft_hook=hook)
    np.testing.assert_array_equal(r.tokens, g)
    assert all(c.k == 0 for c in r.cycles)
    assert len(r.cycles) == 29


def test_context_cache_tracks_verified_positions():
    s = tiny(block_size=4)
    m = model(s, seed=7)
    prompt = syn.make_prompt(s, 12, seed=8)
    r = O.spec_generate(m, prompt, 25)
    pos = len(prompt)
    for c in r.cycles:
        assert c.position == pos
        pos += c.k + 1
