"""Seeded synthetic inputs for the DFlash draft-and-verify cycle.

This module is the one thing the CUDA path and the CPU oracle share: it
draws random-init weights, prompt token ids and microbenchmark hidden
states from fixed seeds, and it describes the model shapes.  It holds none
of the method's arithmetic (no norms, projections, attention, layer
selection or acceptance rule).

Conventions
-----------
* Every matrix is stored like a linear layer's weight, ``[out_features,
  in_features]`` row-major, so a projection reads ``y = x @ W.T``.
* Matrices are drawn N(0, 0.02); RMSNorm gains are 1 (or, for tests that
  must catch a gain that is ignored, 1 + N(0, gain_std)).
* A matrix is drawn in blocks of ``BLOCK`` consecutive elements (row-major
  order); block ``b`` of weight number ``i`` comes from
  ``PCG64(SeedSequence([seed, i, b]))``.  The values therefore do not depend
  on how many threads draw them.
* ``bf16`` shapes keep each draw rounded to bfloat16 (round to nearest,
  ties to even) and return the 16-bit patterns as ``uint16``; ``fp32``
  shapes return ``float32``.
* Prompt ids are uniform over ``[0, vocab - 2]``: id ``vocab - 1`` is kept
  for the drafter's mask slot.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Iterator, List, Sequence, Tuple

import numpy as np

BLOCK = 1 << 22
WEIGHT_STD = 0.02


@dataclasses.dataclass(frozen=True)
class ModelShape:
    """Sizes of the target decoder and of the block drafter."""

    name: str
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ffn: int
    vocab: int
    draft_layers: int
    block_size: int
    dtype: str  # "fp32" or "bf16"
    rms_eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def mask_token_id(self) -> int:
        return self.vocab - 1

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def replace(self, **kw) -> "ModelShape":
        return dataclasses.replace(self, **kw)


# The tiny fp32 decoder: 8 layers, d=256, 4 heads of 64, SwiGLU 1024, vocab 1024;
# one drafter layer of the same width; block of 8.
TINY = ModelShape("tiny-fp32", n_layers=8, d_model=256, n_q_heads=4, n_kv_heads=4,
                  head_dim=64, d_ffn=1024, vocab=1024, draft_layers=1,
                  block_size=8, dtype="fp32")

# Qwen3-8B-shaped target (36 layers, d=4096, GQA 32/8 x 128, SwiGLU 12288,
# vocab 151936) with a 5-layer drafter of the same width; block of 16.
QWEN3_8B = ModelShape("qwen3-8b-shape", n_layers=36, d_model=4096, n_q_heads=32,
                      n_kv_heads=8, head_dim=128, d_ffn=12288, vocab=151936,
                      draft_layers=5, block_size=16, dtype="bf16")

# 27B-class target (64 layers, d=5120, GQA 40/8 x 128, SwiGLU 17408) with a
# 5-layer drafter of the same width.
DENSE_27B = ModelShape("27b-class", n_layers=64, d_model=5120, n_q_heads=40,
                       n_kv_heads=8, head_dim=128, d_ffn=17408, vocab=151936,
                       draft_layers=5, block_size=16, dtype="bf16")

PROMPT_SEED = 1
HIDDEN_SEED = 2
WEIGHT_SEED = 0

LAYER_MATS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")


def weight_specs(s: ModelShape) -> List[Tuple[str, Tuple[int, ...]]]:
    """Canonical (name, shape) list.  Its order is the order the C ABI takes."""
    d, F, V = s.d_model, s.d_ffn, s.vocab

    def layer(prefix: str) -> List[Tuple[str, Tuple[int, ...]]]:
        return [
            (f"{prefix}.attn_norm", (d,)),
            (f"{prefix}.wq", (s.q_dim, d)),
            (f"{prefix}.wk", (s.kv_dim, d)),
            (f"{prefix}.wv", (s.kv_dim, d)),
            (f"{prefix}.wo", (d, s.q_dim)),
            (f"{prefix}.mlp_norm", (d,)),
            (f"{prefix}.w_gate", (F, d)),
            (f"{prefix}.w_up", (F, d)),
            (f"{prefix}.w_down", (d, F)),
        ]

    specs: List[Tuple[str, Tuple[int, ...]]] = [("embed", (V, d))]
    for l in range(s.n_layers):
        specs += layer(f"t{l}")
    specs += [("final_norm", (d,)), ("lm_head", (V, d))]
    specs += [("fc", (d, 5 * d)), ("fc_norm", (d,))]
    for l in range(s.draft_layers):
        specs += layer(f"d{l}")
    specs += [("d_final_norm", (d,))]
    return specs


def _is_norm(name: str) -> bool:
    return name.endswith("norm")


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _draw_block(seed: int, index: int, block: int, n: int, std: float, mean: float) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, index, block])))
    out = g.standard_normal(n, dtype=np.float32)
    out *= np.float32(std)
    if mean:
        out += np.float32(mean)
    return out


def draw_weight(s: ModelShape, index: int, name: str, shape: Tuple[int, ...], seed: int = WEIGHT_SEED,
                gain_std: float = 0.0, pool: ThreadPoolExecutor | None = None) -> np.ndarray:
    """Draw weight number ``index`` of ``weight_specs(s)``."""
    n = int(np.prod(shape))
    if _is_norm(name):
        if gain_std == 0.0:
            flat = np.ones(n, dtype=np.float32)
        else:
            flat = _draw_block(seed, index, 0, n, gain_std, 1.0)
    else:
        nblk = (n + BLOCK - 1) // BLOCK
        sizes = [min(BLOCK, n - b * BLOCK) for b in range(nblk)]
        if pool is not None and nblk > 1:
            parts = list(pool.map(lambda b: _draw_block(seed, index, b, sizes[b], WEIGHT_STD, 0.0), range(nblk)))
        else:
            parts = [_draw_block(seed, index, b, sizes[b], WEIGHT_STD, 0.0) for b in range(nblk)]
        flat = np.concatenate(parts) if nblk > 1 else parts[0]
    flat = flat.reshape(shape)
    if s.dtype == "bf16":
        return f32_to_bf16_bits(flat)
    return flat


def iter_weights(s: ModelShape, seed: int = WEIGHT_SEED, gain_std: float = 0.0,
                 threads: int | None = None) -> Iterator[Tuple[str, np.ndarray]]:
    """Yield (name, array) in canonical order, one matrix at a time."""
    threads = threads or min(16, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as pool:
        for i, (name, shape) in enumerate(weight_specs(s)):
            yield name, draw_weight(s, i, name, shape, seed, gain_std, pool)


def iter_weights_device(s: ModelShape, seed: int = WEIGHT_SEED):
    """Yield (name, tensor) in canonical order, drawn on the current CUDA
    device: N(0, 0.02) matrices and unit norm gains, all in the model dtype.  A
    different stream from iter_weights (torch's device generator, seeded per
    matrix); for throughput runs of large shapes, where drawing on the host
    would take minutes.  Imports torch on first use."""
    import torch

    dt = torch.bfloat16 if s.dtype == "bf16" else torch.float32
    for i, (name, shape) in enumerate(weight_specs(s)):
        if _is_norm(name):
            yield name, torch.ones(shape, dtype=dt, device="cuda")
            continue
        g = torch.Generator(device="cuda").manual_seed(seed * 1_000_003 + i)
        w = torch.empty(shape, dtype=torch.float32, device="cuda")
        w.normal_(0.0, 0.02, generator=g)
        yield name, w.to(dt)
        del w


def make_weights(s: ModelShape, seed: int = WEIGHT_SEED, gain_std: float = 0.0) -> Dict[str, np.ndarray]:
    return dict(iter_weights(s, seed, gain_std))


def as_float(arr: np.ndarray) -> np.ndarray:
    """float32 view of a weight as drawn (bf16 bit patterns are widened exactly)."""
    if arr.dtype == np.uint16:
        return bf16_bits_to_f32(arr)
    return arr


def make_prompt(s: ModelShape, length: int, seed: int = PROMPT_SEED, stream: int = 0) -> np.ndarray:
    """Prompt ids, uniform over [0, vocab - 2]."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))
    return g.integers(0, s.vocab - 1, size=length, dtype=np.int64).astype(np.int32)


def make_prompt_lengths(n: int, lo: int, hi: int, seed: int = PROMPT_SEED) -> np.ndarray:
    """Prompt lengths uniform over [lo, hi] (serving-shaped batches)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1 << 20])))
    return g.integers(lo, hi + 1, size=n, dtype=np.int64).astype(np.int32)


def make_hidden(rows: int, cols: int, seed: int = HIDDEN_SEED, stream: int = 0) -> np.ndarray:
    """N(0, 1) float32 rows (stand-ins for tapped hidden states)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))
    return g.standard_normal((rows, cols), dtype=np.float32)


def make_normal(shape: Tuple[int, ...], std: float, seed: int, stream: int = 0,
                threads: int | None = None) -> np.ndarray:
    """N(0, std) float32 array drawn in BLOCK-sized pieces, block b from
    PCG64(SeedSequence([seed, stream, b])); the result does not depend on threads."""
    n = int(np.prod(shape))
    nblk = (n + BLOCK - 1) // BLOCK
    sizes = [min(BLOCK, n - b * BLOCK) for b in range(nblk)]

    def one(b):
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, b])))
        out = g.standard_normal(sizes[b], dtype=np.float32)
        out *= np.float32(std)
        return out

    threads = threads or min(16, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as pool:
        parts = list(pool.map(one, range(nblk)))
    return np.concatenate(parts).reshape(shape) if nblk > 1 else parts[0].reshape(shape)


# ----------------------------------------------------------------------------
# Counter-based uniforms: Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
# "Parallel random numbers: as easy as 1, 2, 3", SC'11), for draws that the
# CPU and the GPU must reproduce bit for bit.  A kernel that draws implements
# the same generator from the same definition.
# ----------------------------------------------------------------------------

_PHILOX_M = (0xD2511F53, 0xCD9E8D57)
_PHILOX_W = (0x9E3779B9, 0xBB67AE85)
_U32 = 0xFFFFFFFF


def philox4x32(ctr: Sequence[int], key: Sequence[int], rounds: int = 10) -> List[int]:
    """Philox4x32 block function: 4 x 32-bit counter, 2 x 32-bit key -> 4 x 32-bit."""
    c = [int(x) & _U32 for x in ctr]
    k = [int(x) & _U32 for x in key]
    for _ in range(rounds):
        p0 = _PHILOX_M[0] * c[0]
        p1 = _PHILOX_M[1] * c[2]
        c = [((p1 >> 32) ^ c[1] ^ k[0]) & _U32, p1 & _U32, ((p0 >> 32) ^ c[3] ^ k[1]) & _U32, p0 & _U32]
        k = [(k[0] + _PHILOX_W[0]) & _U32, (k[1] + _PHILOX_W[1]) & _U32]
    return c


def philox_uniforms(seed: int, stream: int, offset: int, n: int) -> np.ndarray:
    """Uniforms number offset .. offset + n - 1 of (seed, stream), in [0, 1)
    with 24 random bits each (exact in float32).  Uniform j is word j % 4 of
    philox4x32(counter = (b, b >> 32, stream, 0), key = (seed, seed >> 32)),
    b = j // 4, mapped as u = (word >> 8) * 2^-24."""
    out = np.empty(n, dtype=np.float64)
    for i in range(n):
        j = offset + i
        blk = j // 4
        w = philox4x32([blk & _U32, (blk >> 32) & _U32, stream & _U32, 0], [seed & _U32, (seed >> 32) & _U32])[j % 4]
        out[i] = (w >> 8) * (1.0 / 16777216.0)
    return out
