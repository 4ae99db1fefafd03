"""CPU oracle of the DFlash draft-and-verify cycle.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
link this module: only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` use it.  It shares no code with the CUDA
path; the two meet only in the seeded input generators of ``synthetic``.

Everything is plain numpy in float64, step by step in the order the pages
describe the method.  Sources (web pages, cited by title and section):

* [ARCH] "DFlash 的架构密码——扩散模型如何「寄生」在自回归模型上"
  (zhichai.net), sections 第一层 Feature Fusion, 第二层 KV Injection,
  第三层 Block Diffusion, 训练策略 (Random Sampling of Masked Blocks;
  Shared Embedding & LM Head) and 技术细节补充 (提取层数, 投影层,
  稀疏注意力训练).
* [ABS] "DFlash：基于块扩散的闪存推测解码方法" (ai-stack.site), 摘要
  (single forward pass, features of the target as the condition, lossless),
  实践 2 (block verification, keep up to the last correct token),
  实践 3 (the drafter never writes the target's KV cache).
* [PRESS] the DFlash press repost on zaocj.com (藍戒AI知行): one forward pass
  with bidirectional attention fills the 8-16 slots after the verified token;
  lossless speed-up on Qwen3-8B.

The target is the plain pre-norm decoder the shapes name (RMSNorm, RoPE,
grouped-query attention, SwiGLU).  Where the pages are silent the readings
are:

* feature layers: 1-based layer outputs s_i = 2 + round_half_up(i (L-4) / 4);
* the fused context is RMSNorm(concat(h_s1..h_s5) @ W_fc^T), shallow to deep,
  no bias, eps 1e-6;
* injected K/V use each drafter layer's own W_k/W_v; K gets RoPE at the
  context token's absolute position;
* context features exist for every verified position (the prompt, then each
  cycle's bonus token and accepted drafts); the newest bonus token is block
  slot 0, not context;
* mask slots hold the reserved id vocab-1; slot i (1..B-1) proposes the
  token at slot i; slot 0's own output is unused;
* argmax compares the logits as computed and keeps the lowest index on ties;
* verification keeps the longest prefix of drafts that equal the target's
  greedy tokens, then the target's token after it (the bonus);
* sampling (temperature T > 0, nucleus top_p): the pages state that a draft
  is accepted or rejected by the target's distribution, that a rejected
  position is sampled again, and that the output keeps the target's
  distribution; with drafter and target at the same T and top_p.  The
  plainest rule with that property is the standard speculative-sampling
  test: keep d_i with probability min(1, p(d_i) / q(d_i)), replace the first
  rejected draft by a draw from max(0, p - q) normalised, and draw the token
  after a fully kept block from p.  The uniforms every draw uses are inputs.

Parity is pinned by tests against library routines (torch CPU attention and
RMSNorm), closed forms (feature layers, unit-RMS context rows, RoPE as a
complex rotation) and invariants (speculative output equals greedy decoding,
brute-force longest prefix, no flow between blocks).  The drafter's hidden
states and drafts for random weights have no worked example on the pages:
their parity is unpinned beyond those invariants.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np


# ----------------------------------------------------------------------------
# Building blocks
# ----------------------------------------------------------------------------

def feature_layers(n_layers: int) -> List[int]:
    """Five target layers sampled uniformly from layer 2 to the third-from-last.

    [ARCH] 技术细节补充, 提取层数.  Layers are numbered from 1; the value is the
    output of that layer (the residual stream after it).  The ends are 2 and
    L-2; the three inner points are rounded half up.
    """
    if n_layers < 8:
        raise ValueError("need at least 8 target layers for 5 distinct feature layers")
    lo, hi = 2, n_layers - 2
    return [lo + int(math.floor(i * (hi - lo) / 4.0 + 0.5)) for i in range(5)]


def rms_norm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gain over the last axis ([ARCH] 投影层: RMSNorm)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gain


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotary position embedding, rotate-half form.

    x: [n, heads, hd]; positions: [n].  Dimension pairs are (j, j + hd/2),
    rotated by the angle pos * theta^(-2j/hd).
    """
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / hd)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, visible: np.ndarray) -> np.ndarray:
    """Softmax attention with grouped KV heads.

    q: [n, Hq, hd]; k, v: [T, Hkv, hd]; visible: bool [n, T].  Query head j
    reads KV head j // (Hq / Hkv).  Scale 1/sqrt(hd).  Returns [n, Hq, hd].
    """
    n, hq, hd = q.shape
    hkv = k.shape[1]
    group = hq // hkv
    out = np.zeros_like(q)
    scale = 1.0 / math.sqrt(hd)
    for j in range(hq):
        kh = j // group
        s = (q[:, j, :] @ k[:, kh, :].T) * scale          # [n, T]
        s = np.where(visible, s, -np.inf)
        m = np.max(s, axis=1, keepdims=True)
        p = np.exp(s - m)
        p = p / np.sum(p, axis=1, keepdims=True)
        out[:, j, :] = p @ v[:, kh, :]
    return out


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Row-wise argmax; the lowest index wins a tie (np.argmax keeps the first)."""
    return np.argmax(logits, axis=-1).astype(np.int64)


# ----------------------------------------------------------------------------
# Weights
# ----------------------------------------------------------------------------

class Weights:
    """float64 view of the synthetic weights (bf16 patterns widened exactly)."""

    def __init__(self, raw: Dict[str, np.ndarray], cache: bool = True):
        self.raw = raw
        self.cache = cache
        self._f64: Dict[str, np.ndarray] = {}

    def __getitem__(self, name: str) -> np.ndarray:
        if name in self._f64:
            return self._f64[name]
        a = self.raw[name]
        if a.dtype == np.uint16:
            a = (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
        a = a.astype(np.float64)
        if self.cache:
            self._f64[name] = a
        return a


# ----------------------------------------------------------------------------
# Shapes (duck-typed: any object with these attributes works)
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Shape:
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ffn: int
    vocab: int
    draft_layers: int
    block_size: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def mask_token_id(self) -> int:
        return self.vocab - 1


# ----------------------------------------------------------------------------
# One decoder layer (shared shape by the target and the drafter)
# ----------------------------------------------------------------------------

def _proj(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    return x @ w.T


def decoder_layer(W: Weights, prefix: str, cfg, h: np.ndarray, positions: np.ndarray,
                  kv_source: Callable[[np.ndarray, np.ndarray], Tuple[np.ndarray, np.ndarray, np.ndarray]]
                  ) -> np.ndarray:
    """Pre-norm layer: h += Wo Attn(RMSNorm(h)); h += W_down(SiLU(W_gate y) * W_up y).

    ``kv_source(k_new, v_new)`` receives the layer's own keys/values (RoPE
    already applied to keys) and returns (keys, values, visible) to attend
    over; that is where the target (causal cache) and the drafter (context
    cache + bidirectional block) differ.
    """
    n = h.shape[0]
    hd = cfg.head_dim
    x = rms_norm(h, W[f"{prefix}.attn_norm"], cfg.rms_eps)
    q = _proj(x, W[f"{prefix}.wq"]).reshape(n, cfg.n_q_heads, hd)
    k = _proj(x, W[f"{prefix}.wk"]).reshape(n, cfg.n_kv_heads, hd)
    v = _proj(x, W[f"{prefix}.wv"]).reshape(n, cfg.n_kv_heads, hd)
    q = rope(q, positions, cfg.rope_theta)
    k = rope(k, positions, cfg.rope_theta)
    keys, values, visible = kv_source(k, v)
    a = attention(q, keys, values, visible).reshape(n, cfg.n_q_heads * hd)
    h = h + _proj(a, W[f"{prefix}.wo"])
    y = rms_norm(h, W[f"{prefix}.mlp_norm"], cfg.rms_eps)
    g = _proj(y, W[f"{prefix}.w_gate"])
    u = _proj(y, W[f"{prefix}.w_up"])
    h = h + _proj(silu(g) * u, W[f"{prefix}.w_down"])
    return h


# ----------------------------------------------------------------------------
# Target decoder with a growing KV cache
# ----------------------------------------------------------------------------

class KVCache:
    """Per-layer keys/values [T, Hkv, hd] in position order; rollback truncates."""

    def __init__(self, n_layers: int, n_kv_heads: int, head_dim: int):
        self.k = [np.zeros((0, n_kv_heads, head_dim)) for _ in range(n_layers)]
        self.v = [np.zeros((0, n_kv_heads, head_dim)) for _ in range(n_layers)]

    @property
    def length(self) -> int:
        return self.k[0].shape[0]

    def truncate(self, length: int) -> None:
        self.k = [a[:length] for a in self.k]
        self.v = [a[:length] for a in self.v]


@dataclasses.dataclass
class TargetPass:
    taps: np.ndarray      # [n, 5, d]: outputs of the feature layers, shallow to deep
    logits: np.ndarray    # [n, V]
    hidden: List[np.ndarray]  # residual stream entering each layer, plus the last output


def target_forward(W: Weights, cfg, tokens: Sequence[int], cache: KVCache) -> TargetPass:
    """Run the target over ``tokens`` placed right after the cached positions.

    Token i sits at position cache.length + i and sees every cached position
    and the new tokens up to itself (causal).  Its keys/values are appended.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    n = len(tokens)
    p0 = cache.length
    positions = np.arange(p0, p0 + n)
    feats = feature_layers(cfg.n_layers)
    h = W["embed"][tokens]
    taps = np.zeros((n, 5, cfg.d_model))
    hidden = []
    for l in range(cfg.n_layers):
        # h is the output of layer l (1-based numbering); tap it if selected.
        if l in feats:
            taps[:, feats.index(l), :] = h
        hidden.append(h)

        def kv_source(k_new, v_new, l=l):
            cache.k[l] = np.concatenate([cache.k[l], k_new], axis=0)
            cache.v[l] = np.concatenate([cache.v[l], v_new], axis=0)
            T = cache.k[l].shape[0]
            visible = np.arange(T)[None, :] <= positions[:, None]
            return cache.k[l], cache.v[l], visible

        h = decoder_layer(W, f"t{l}", cfg, h, positions, kv_source)
    hidden.append(h)
    hf = rms_norm(h, W["final_norm"], cfg.rms_eps)
    logits = hf @ W["lm_head"].T
    return TargetPass(taps=taps, logits=logits, hidden=hidden)


# ----------------------------------------------------------------------------
# Drafter: feature fusion, KV injection, one bidirectional block pass
# ----------------------------------------------------------------------------

def fuse_features(W: Weights, cfg, taps: np.ndarray) -> np.ndarray:
    """[ARCH] 第一层 / 投影层: concat the 5 tapped states, light FC, RMSNorm.

    taps: [n, 5, d] -> ctx [n, d].
    """
    n = taps.shape[0]
    cat = taps.reshape(n, 5 * cfg.d_model)
    return rms_norm(cat @ W["fc"].T, W["fc_norm"], cfg.rms_eps)


class ContextCache:
    """Drafter-side keys/values built from injected context features ([ARCH] 第二层)."""

    def __init__(self, draft_layers: int, n_kv_heads: int, head_dim: int):
        self.k = [np.zeros((0, n_kv_heads, head_dim)) for _ in range(draft_layers)]
        self.v = [np.zeros((0, n_kv_heads, head_dim)) for _ in range(draft_layers)]

    @property
    def length(self) -> int:
        return self.k[0].shape[0]


def inject_kv(W: Weights, cfg, ctx_cache: ContextCache, ctx: np.ndarray) -> None:
    """Project context features through every drafter layer's W_k / W_v.

    [ARCH] 第二层 KV Injection: the feature goes into the K and V projections
    of every layer, not only the input.  Rows are appended at positions
    ctx_cache.length, ctx_cache.length + 1, ...
    """
    n = ctx.shape[0]
    positions = np.arange(ctx_cache.length, ctx_cache.length + n)
    hd = cfg.head_dim
    for l in range(cfg.draft_layers):
        k = (ctx @ W[f"d{l}.wk"].T).reshape(n, cfg.n_kv_heads, hd)
        v = (ctx @ W[f"d{l}.wv"].T).reshape(n, cfg.n_kv_heads, hd)
        k = rope(k, positions, cfg.rope_theta)
        ctx_cache.k[l] = np.concatenate([ctx_cache.k[l], k], axis=0)
        ctx_cache.v[l] = np.concatenate([ctx_cache.v[l], v], axis=0)


@dataclasses.dataclass
class DraftPass:
    drafts: np.ndarray   # [blocks, B-1] proposed tokens for slots 1..B-1
    logits: np.ndarray   # [blocks * B, V]
    hidden: np.ndarray   # [blocks * B, d] drafter output before the final norm


def draft_blocks(W: Weights, cfg, ctx_cache: ContextCache, anchors: Sequence[Tuple[int, int]]) -> DraftPass:
    """One drafter forward pass over one or more blocks.

    anchors: (anchor_token, anchor_position) per block.  Block j holds
    [anchor, MASK x (B-1)] at positions a_j .. a_j + B - 1.  A block sees the
    context entries before its anchor position and every slot of its own block
    (bidirectional), and nothing of any other block ([ARCH] 稀疏注意力训练:
    bidirectional inside a block, no information flow between blocks;
    [PRESS]: single forward pass fills the 8-16 slots).
    """
    B = cfg.block_size
    nb = len(anchors)
    tokens = []
    positions = []
    for tok, pos in anchors:
        tokens += [tok] + [cfg.mask_token_id] * (B - 1)
        positions += list(range(pos, pos + B))
    tokens = np.asarray(tokens, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    blk = np.repeat(np.arange(nb), B)
    h = W["embed"][tokens]
    C = ctx_cache.length
    for l in range(cfg.draft_layers):
        def kv_source(k_new, v_new, l=l):
            keys = np.concatenate([ctx_cache.k[l], k_new], axis=0)
            values = np.concatenate([ctx_cache.v[l], v_new], axis=0)
            ctx_pos = np.arange(C)
            anchor_pos = np.asarray([a[1] for a in anchors])[blk]            # [nB]
            vis_ctx = ctx_pos[None, :] < anchor_pos[:, None]
            vis_blk = blk[:, None] == blk[None, :]
            return keys, values, np.concatenate([vis_ctx, vis_blk], axis=1)

        h = decoder_layer(W, f"d{l}", cfg, h, positions, kv_source)
    hf = rms_norm(h, W["d_final_norm"], cfg.rms_eps)
    logits = hf @ W["lm_head"].T                      # shared LM head ([ARCH] 训练策略 3)
    ids = argmax_lowest(logits).reshape(nb, B)
    return DraftPass(drafts=ids[:, 1:], logits=logits, hidden=h)


# ----------------------------------------------------------------------------
# Verification and the loops
# ----------------------------------------------------------------------------

def accept_prefix(drafts: Sequence[int], greedy: Sequence[int]) -> Tuple[int, int]:
    """Longest accepted prefix and the bonus token.

    drafts = d_1..d_{B-1}; greedy = g_0..g_{B-1}, where g_i is the target's
    argmax at block slot i (its guess for slot i+1).  d_i is accepted while
    d_i == g_{i-1} for every i up to it.  Returns (k, g_k): k accepted drafts,
    then the target's own token after them ([ABS] 实践 2: keep up to the last
    correct token; [ARCH] the next block starts at the bonus token).
    """
    k = 0
    while k < len(drafts) and int(drafts[k]) == int(greedy[k]):
        k += 1
    return k, int(greedy[k])


@dataclasses.dataclass
class Model:
    W: Weights
    cfg: object


def greedy_generate(m: Model, prompt: Sequence[int], n_new: int) -> np.ndarray:
    """Token-by-token greedy decoding of the target (the lossless reference)."""
    cfg = m.cfg
    cache = KVCache(cfg.n_layers, cfg.n_kv_heads, cfg.head_dim)
    out: List[int] = []
    tp = target_forward(m.W, cfg, prompt, cache)
    tok = int(argmax_lowest(tp.logits[-1:])[0])
    out.append(tok)
    while len(out) < n_new:
        tp = target_forward(m.W, cfg, [tok], cache)
        tok = int(argmax_lowest(tp.logits)[0])
        out.append(tok)
    return np.asarray(out[:n_new], dtype=np.int64)


@dataclasses.dataclass
class Cycle:
    position: int          # position of the bonus token (block slot 0)
    bonus: int
    drafts: np.ndarray     # d_1..d_{B-1}
    greedy: np.ndarray     # g_0..g_{B-1}
    k: int                 # accepted drafts
    taps: np.ndarray       # [B, 5, d] from the verify pass
    logits: np.ndarray     # [B, V] from the verify pass


@dataclasses.dataclass
class SpecResult:
    tokens: np.ndarray
    cycles: List[Cycle]

    @property
    def accepted(self) -> List[int]:
        return [c.k for c in self.cycles]

    @property
    def mean_accept_len(self) -> float:
        return float(np.mean([c.k + 1 for c in self.cycles])) if self.cycles else 0.0


DraftHook = Callable[[int, int, np.ndarray], Optional[Sequence[int]]]


def spec_generate(m: Model, prompt: Sequence[int], n_new: int,
                  draft_hook: Optional[DraftHook] = None) -> SpecResult:
    """DFlash speculative decoding, one sequence, greedy.

    Prefill: run the target over the prompt, take its argmax at the last
    position as the first bonus token, fuse the prompt's tapped features and
    inject them into the drafter's context cache.  Then repeat:
      draft  - one drafter pass over [bonus, MASK x (B-1)];
      verify - one target pass over [bonus, d_1..d_{B-1}];
      accept - longest greedy-matching prefix k, bonus' = g_k; roll the target
               cache back to bonus position + k + 1;
      inject - fuse the taps of the k+1 verified rows into the context cache.
    ``draft_hook(bonus, position, drafts)`` may replace the drafts (tests).
    Output is truncated to exactly n_new tokens.
    """
    cfg = m.cfg
    W = m.W
    B = cfg.block_size
    cache = KVCache(cfg.n_layers, cfg.n_kv_heads, cfg.head_dim)
    ctxc = ContextCache(cfg.draft_layers, cfg.n_kv_heads, cfg.head_dim)
    tp = target_forward(W, cfg, prompt, cache)
    bonus = int(argmax_lowest(tp.logits[-1:])[0])
    inject_kv(W, cfg, ctxc, fuse_features(W, cfg, tp.taps))
    pos = len(prompt)
    out = [bonus]
    cycles: List[Cycle] = []
    while len(out) < n_new:
        assert cache.length == pos and ctxc.length == pos
        dp = draft_blocks(W, cfg, ctxc, [(bonus, pos)])
        drafts = dp.drafts[0]
        if draft_hook is not None:
            repl = draft_hook(bonus, pos, drafts)
            if repl is not None:
                drafts = np.asarray(repl, dtype=np.int64)
        vp = target_forward(W, cfg, [bonus] + [int(t) for t in drafts], cache)
        g = argmax_lowest(vp.logits)
        k, new_bonus = accept_prefix(drafts, g)
        cycles.append(Cycle(pos, bonus, np.asarray(drafts), g, k, vp.taps, vp.logits))
        cache.truncate(pos + k + 1)
        inject_kv(W, cfg, ctxc, fuse_features(W, cfg, vp.taps[: k + 1]))
        out += [int(t) for t in drafts[:k]] + [new_bonus]
        bonus = new_bonus
        pos += k + 1
    return SpecResult(tokens=np.asarray(out[:n_new], dtype=np.int64), cycles=cycles)


# ----------------------------------------------------------------------------
# Sampling: the lossless rejection test ([ABS] 实践 4 on temperature and top-p,
# 核心思想 step 3 and the Q&A on losslessness)
# ----------------------------------------------------------------------------

def sampling_probs(logits: np.ndarray, temperature: float, top_p: float = 1.0) -> np.ndarray:
    """Rows of next-token probabilities for sampling.

    softmax(logits / T), then restricted to the nucleus (the fewest most
    probable tokens whose mass reaches top_p, ties by lower index) and
    renormalised.  T == 0 means greedy: one-hot at the argmax (lowest index
    on ties)."""
    logits = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    n, V = logits.shape
    if temperature == 0.0:
        out = np.zeros((n, V))
        out[np.arange(n), argmax_lowest(logits)] = 1.0
        return out
    z = logits / float(temperature)
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z)
    probs = e / e.sum(axis=1, keepdims=True)
    if top_p >= 1.0:
        return probs
    out = np.zeros_like(probs)
    for r in range(n):
        order = np.lexsort((np.arange(V), -probs[r]))      # descending mass, lower index first on ties
        csum = np.cumsum(probs[r, order])
        keep = order[: int(np.searchsorted(csum, top_p)) + 1]
        out[r, keep] = probs[r, keep]
        out[r] /= out[r].sum()
    return out


def draw(probs: np.ndarray, u: float) -> int:
    """Inverse-CDF draw from one row of (possibly unnormalised) mass with a
    uniform u in [0, 1): the lowest index whose cumulative mass exceeds
    u x total."""
    c = np.cumsum(np.asarray(probs, dtype=np.float64))
    return int(min(np.searchsorted(c, u * c[-1], side="right"), len(c) - 1))


def accept_sampled(drafts: Sequence[int], q_rows: np.ndarray, p_rows: np.ndarray,
                   u_accept: Sequence[float], u_final: float) -> Tuple[int, int]:
    """Speculative sampling over one block.

    drafts = d_1..d_{B-1}, d_i drawn from q_rows[i-1] (the drafter's
    distribution at slot i); p_rows[i] is the target's distribution for the
    token after slot i (row i of the verify pass), i = 0..B-1.  d_i is kept
    while u_accept[i-1] < p_{i-1}(d_i) / q_{i-1}(d_i); at the first rejection
    the token is drawn from max(0, p - q) (normalised) with u_final, and if
    every draft is kept the token after the block is drawn from p_{B-1} with
    u_final.  Returns (k, token): k kept drafts, then that token."""
    k = 0
    while k < len(drafts):
        d = int(drafts[k])
        pk, qk = p_rows[k][d], q_rows[k][d]
        if qk > 0.0 and u_accept[k] < pk / qk:
            k += 1
            continue
        residual = np.maximum(p_rows[k] - q_rows[k], 0.0)
        if residual.sum() <= 0.0:          # p == q: nothing to correct
            residual = p_rows[k]
        return k, draw(residual, u_final)
    return k, draw(p_rows[k], u_final)


def draw_margin(probs: np.ndarray, u: float) -> float:
    """How far u x total lies from the ends of the interval that decides
    draw(probs, u), as a fraction of the total mass (0 on a boundary).  A
    draw from masses that differ by less than this picks the same index."""
    c = np.cumsum(np.asarray(probs, dtype=np.float64))
    total = c[-1]
    j = draw(probs, u)
    lo = c[j - 1] if j > 0 else 0.0
    t = u * total
    return float(min(t - lo, c[j] - t) / total)


def nucleus_margin(logits: np.ndarray, temperature: float, top_p: float) -> float:
    """Smallest distance, over the rows, between top_p and the cumulative
    masses on either side of the row's nucleus cut (inf without a cut)."""
    if temperature == 0.0 or top_p >= 1.0:
        return math.inf
    probs = sampling_probs(logits, temperature, 1.0)
    out = math.inf
    for r in range(probs.shape[0]):
        order = np.lexsort((np.arange(probs.shape[1]), -probs[r]))
        csum = np.cumsum(probs[r, order])
        j = min(int(np.searchsorted(csum, top_p)), len(csum) - 1)
        out = min(out, abs(csum[j] - top_p))
        if j > 0:
            out = min(out, abs(top_p - csum[j - 1]))
    return float(out)


def accept_margin(drafts: Sequence[int], q_rows: np.ndarray, p_rows: np.ndarray,
                  u_accept: Sequence[float], u_final: float) -> float:
    """Smallest distance from a tie of the decisions accept_sampled takes on
    these inputs: |u_i - p/q| of each test it makes, then its final draw's
    draw_margin."""
    m = math.inf
    k = 0
    while k < len(drafts):
        d = int(drafts[k])
        pk, qk = p_rows[k][d], q_rows[k][d]
        if qk > 0.0:
            m = min(m, abs(u_accept[k] - pk / qk))
            if u_accept[k] < pk / qk:
                k += 1
                continue
        residual = np.maximum(p_rows[k] - q_rows[k], 0.0)
        if residual.sum() <= 0.0:
            residual = p_rows[k]
        return min(m, draw_margin(residual, u_final))
    return min(m, draw_margin(p_rows[k], u_final))


Uniforms = Callable[[int], np.ndarray]


def sample_generate(m: Model, prompt: Sequence[int], n_new: int, temperature: float, top_p: float,
                    uniforms: Uniforms) -> np.ndarray:
    """Token-by-token sampling from the target (the distribution speculative
    sampling must keep); uniforms(n) gives the next n uniforms."""
    cfg = m.cfg
    cache = KVCache(cfg.n_layers, cfg.n_kv_heads, cfg.head_dim)
    out: List[int] = []
    tp = target_forward(m.W, cfg, prompt, cache)
    while True:
        tok = draw(sampling_probs(tp.logits[-1:], temperature, top_p)[0], float(uniforms(1)[0]))
        out.append(tok)
        if len(out) >= n_new:
            return np.asarray(out, dtype=np.int64)
        tp = target_forward(m.W, cfg, [tok], cache)


def spec_generate_sampled(m: Model, prompt: Sequence[int], n_new: int, temperature: float, top_p: float,
                          uniforms: Uniforms, margins: Optional[List[float]] = None) -> SpecResult:
    """DFlash speculative decoding with sampling, one sequence.

    The cycle of ``spec_generate``, with each slot's draft drawn from the
    drafter's distribution at that slot (same temperature and top_p as the
    target) and ``accept_sampled`` in place of the greedy prefix test.  The
    bonus token after the prompt is drawn from the target's distribution.
    Uniforms per cycle: B-1 for the drafts, B-1 for the tests, 1 for the
    final draw.  At temperature 0 this is exactly ``spec_generate``.
    margins (optional) receives, in order, each decision's distance from a
    tie (nucleus cuts, draws, tests), for comparisons with other arithmetic."""
    cfg = m.cfg
    W = m.W
    B = cfg.block_size
    cache = KVCache(cfg.n_layers, cfg.n_kv_heads, cfg.head_dim)
    ctxc = ContextCache(cfg.draft_layers, cfg.n_kv_heads, cfg.head_dim)
    tp = target_forward(W, cfg, prompt, cache)
    p0 = sampling_probs(tp.logits[-1:], temperature, top_p)[0]
    u0 = float(uniforms(1)[0])
    bonus = draw(p0, u0)
    if margins is not None:
        margins += [nucleus_margin(tp.logits[-1:], temperature, top_p), draw_margin(p0, u0)]
    inject_kv(W, cfg, ctxc, fuse_features(W, cfg, tp.taps))
    pos = len(prompt)
    out = [bonus]
    cycles: List[Cycle] = []
    while len(out) < n_new:
        dp = draft_blocks(W, cfg, ctxc, [(bonus, pos)])
        q_rows = sampling_probs(dp.logits[1:B], temperature, top_p)     # slots 1..B-1
        u = uniforms(2 * (B - 1) + 1)
        drafts = np.asarray([draw(q_rows[i], float(u[i])) for i in range(B - 1)], dtype=np.int64)
        vp = target_forward(W, cfg, [bonus] + [int(t) for t in drafts], cache)
        p_rows = sampling_probs(vp.logits, temperature, top_p)
        k, new_bonus = accept_sampled(drafts, q_rows, p_rows, u[B - 1: 2 * (B - 1)], float(u[-1]))
        if margins is not None:
            margins.append(nucleus_margin(dp.logits[1:B], temperature, top_p))
            margins += [draw_margin(q_rows[i], float(u[i])) for i in range(B - 1)]
            margins.append(nucleus_margin(vp.logits, temperature, top_p))
            margins.append(accept_margin(drafts, q_rows, p_rows, u[B - 1: 2 * (B - 1)], float(u[-1])))
        cycles.append(Cycle(pos, bonus, drafts, argmax_lowest(vp.logits), k, vp.taps, vp.logits))
        cache.truncate(pos + k + 1)
        inject_kv(W, cfg, ctxc, fuse_features(W, cfg, vp.taps[: k + 1]))
        out += [int(t) for t in drafts[:k]] + [new_bonus]
        bonus = new_bonus
        pos += k + 1
    return SpecResult(tokens=np.asarray(out[:n_new], dtype=np.int64), cycles=cycles)


def teacher_forced(m: Model, tokens: Sequence[int]) -> TargetPass:
    """Target pass over a whole token stream (prompt + generated), for comparisons."""
    cfg = m.cfg
    cache = KVCache(cfg.n_layers, cfg.n_kv_heads, cfg.head_dim)
    return target_forward(m.W, cfg, tokens, cache)
