"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin fails.

Each case patches one function of the oracle with a wrong variant and runs
the pin that must catch it.  A pin that still passes means the oracle could
carry that mistake unseen.
"""
import math

import numpy as np
import pytest

from oracle import dflash_oracle as O
from tests import test_oracle_pins as P
from tests import test_oracle_sampling as S


def _wrong_rope(x, positions, theta):
    hd = x.shape[-1]
    half = hd // 2
    inv = theta ** (-np.arange(half) * 2.0 / hd)
    ang = np.asarray(positions, float)[:, None] * inv[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], axis=-1)     # rotates the wrong way


def _wrong_gqa(q, k, v, visible):
    n, hq, hd = q.shape
    hkv = k.shape[1]
    out = np.zeros_like(q)
    for j in range(hq):
        kh = j % hkv                                                          # interleaved instead of grouped
        s = (q[:, j] @ k[:, kh].T) / math.sqrt(hd)
        s = np.where(visible, s, -np.inf)
        p = np.exp(s - s.max(1, keepdims=True))
        out[:, j] = (p / p.sum(1, keepdims=True)) @ v[:, kh]
    return out


def _wrong_accept(drafts, greedy):
    k = 0
    while k < len(drafts) and int(drafts[k]) == int(greedy[k + 1 if k + 1 < len(greedy) else k]):
        k += 1                                                                 # compares d_i with g_i
    return k, int(greedy[k])


def _wrong_layers(L):
    return [1 + int(math.floor(i * (L - 4) / 4.0 + 0.5)) for i in range(5)]   # 0-based slip


_orig_fuse = O.fuse_features


def _wrong_fuse(W, cfg, taps):
    return _orig_fuse(W, cfg, taps[:, ::-1])                                  # deep to shallow


_orig_draft = O.draft_blocks


def _causal_draft(W, cfg, ctx_cache, anchors):
    # same as the drafter but with a causal mask inside the block
    orig_attention = O.attention

    def causal_attention(q, k, v, visible):
        T = k.shape[0]
        n = q.shape[0]
        C = T - n
        tri = np.arange(n)[None, :] <= np.arange(n)[:, None]
        vis = visible.copy()
        vis[:, C:] &= tri
        return orig_attention(q, k, v, vis)

    O.attention = causal_attention
    try:
        return _orig_draft(W, cfg, ctx_cache, anchors)
    finally:
        O.attention = orig_attention


_orig_rms = O.rms_norm


def _rms_no_eps(x, g, eps):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + 1e-2) * g   # wrong epsilon


def _rms_no_gain(x, g, eps):
    return _orig_rms(x, np.ones_like(g), eps)


_orig_decoder_layer = O.decoder_layer


def _layer_without_q_rope(W, prefix, cfg, h, positions, kv_source):
    orig = O.rope

    calls = {"n": 0}

    def rope_k_only(x, pos, theta):
        calls["n"] += 1
        return x if calls["n"] == 1 else orig(x, pos, theta)                  # skip RoPE on q

    O.rope = rope_k_only
    try:
        return _orig_decoder_layer(W, prefix, cfg, h, positions, kv_source)
    finally:
        O.rope = orig


def _accept_residual_from_p(drafts, q_rows, p_rows, u_accept, u_final):
    k = 0
    while k < len(drafts):
        d = int(drafts[k])
        if q_rows[k][d] > 0 and u_accept[k] < p_rows[k][d] / q_rows[k][d]:
            k += 1
            continue
        return k, O.draw(p_rows[k], u_final)                                   # resamples from p, not max(0, p - q)
    return k, O.draw(p_rows[k], u_final)


def _accept_inverted_ratio(drafts, q_rows, p_rows, u_accept, u_final):
    k = 0
    while k < len(drafts):
        d = int(drafts[k])
        if p_rows[k][d] > 0 and u_accept[k] < q_rows[k][d] / p_rows[k][d]:   # q / p instead of p / q
            k += 1
            continue
        return k, O.draw(np.maximum(p_rows[k] - q_rows[k], 0.0), u_final)
    return k, O.draw(p_rows[k], u_final)


def _accept_wrong_row(drafts, q_rows, p_rows, u_accept, u_final):
    k = 0
    while k < len(drafts):
        d = int(drafts[k])
        pk = p_rows[k + 1][d]                                                  # the row after the draft
        if q_rows[k][d] > 0 and u_accept[k] < pk / q_rows[k][d]:
            k += 1
            continue
        return k, O.draw(np.maximum(p_rows[k + 1] - q_rows[k], 0.0), u_final)
    return k, O.draw(p_rows[k], u_final)


_orig_inject = O.inject_kv


def _inject_without_rope(W, cfg, ctx_cache, ctx):
    orig = O.rope
    O.rope = lambda x, positions, theta: x                                   # keys injected unrotated
    try:
        return _orig_inject(W, cfg, ctx_cache, ctx)
    finally:
        O.rope = orig


def _inject_positions_from_zero(W, cfg, ctx_cache, ctx):
    # keys of appended rows rotated as if they started at position 0
    n = ctx.shape[0]
    tmp = O.ContextCache(cfg.draft_layers, cfg.n_kv_heads, cfg.head_dim)
    _orig_inject(W, cfg, tmp, ctx)
    for l in range(cfg.draft_layers):
        ctx_cache.k[l] = np.concatenate([ctx_cache.k[l], tmp.k[l][:n]], axis=0)
        ctx_cache.v[l] = np.concatenate([ctx_cache.v[l], tmp.v[l][:n]], axis=0)


def _inject_value_from_key_matrix(W, cfg, ctx_cache, ctx):
    class Swap:
        def __getitem__(self, name):
            return W[name.replace(".wv", ".wk")] if name.endswith(".wv") else W[name]
    return _orig_inject(Swap(), cfg, ctx_cache, ctx)


_orig_target = O.target_forward


def _tap_layer_input(W, cfg, tokens, cache):
    # taps the residual entering layer s instead of the output of layer s
    tp = _orig_target(W, cfg, tokens, cache)
    for i, l in enumerate(O.feature_layers(cfg.n_layers)):
        tp.taps[:, i] = tp.hidden[l - 1]
    return tp


def _tap_next_layer(W, cfg, tokens, cache):
    tp = _orig_target(W, cfg, tokens, cache)
    for i, l in enumerate(O.feature_layers(cfg.n_layers)):
        tp.taps[:, i] = tp.hidden[l + 1]
    return tp


def _sampled_pin():
    S.check_keeps_target_distribution(O.accept_sampled, n=40_000)


MUTATIONS = [
    ("rope", _wrong_rope, [P.test_rope_is_complex_rotation]),
    ("attention", _wrong_gqa, [lambda: P.test_attention_matches_torch_sdpa(8, 2)]),
    ("accept_prefix", _wrong_accept, [P.test_accept_brute_force]),
    ("feature_layers", _wrong_layers, [P.test_feature_layers_golden]),
    ("fuse_features", _wrong_fuse, [P.test_fusion_concat_order_shallow_to_deep]),
    ("draft_blocks", _causal_draft, [P.test_bidirectional_later_slot_reaches_earlier_slot]),
    ("rms_norm", _rms_no_eps, [P.test_rms_norm_matches_torch]),
    ("rms_norm", _rms_no_gain, [P.test_rms_norm_matches_torch]),
    ("decoder_layer", _layer_without_q_rope, [lambda: P.test_target_relative_positions()]),
    ("inject_kv", _inject_without_rope, [P.test_injected_keys_match_block_keys_for_same_input]),
    ("inject_kv", _inject_positions_from_zero, [P.test_injected_keys_match_block_keys_for_same_input]),
    ("inject_kv", _inject_value_from_key_matrix, [P.test_injected_keys_match_block_keys_for_same_input]),
    ("target_forward", _tap_layer_input, [P.test_tap_is_the_output_of_its_layer]),
    ("target_forward", _tap_next_layer, [P.test_tap_is_the_output_of_its_layer]),
    ("accept_sampled", _accept_residual_from_p, [_sampled_pin]),
    ("accept_sampled", _accept_inverted_ratio, [_sampled_pin]),
    ("accept_sampled", _accept_wrong_row, [_sampled_pin]),
]


@pytest.mark.parametrize("name,bad,pins", MUTATIONS, ids=[f"{m[0]}-{m[1].__name__}" for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, bad, pins):
    monkeypatch.setattr(O, name, bad)
    caught = False
    for pin in pins:
        try:
            pin()
        except AssertionError:
            caught = True
    assert caught, f"no pin caught the planted mistake in {name}"
