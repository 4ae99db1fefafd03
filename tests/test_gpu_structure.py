"""The cycle's structure on the GPU.

Sources: [ARCH] "DFlash 的架构密码", 第三层 Block Diffusion (the drafter fills
the whole block in one forward pass) and 技术细节补充, 稀疏注意力训练
(bidirectional attention inside a block, no information flow between
blocks); [PRESS] (one forward pass with bidirectional attention fills the
8-16 slots after the verified token).

* One drafter pass per cycle: over a generation, the engine's launch record
  (df_profile_read) holds exactly one drafter pass (Ld layers of four GEMMs,
  one LM head) and one verify pass (L layers, one LM head) per cycle, plus
  the prefill: the drafter never runs once per slot.
* Bidirectional inside a block: the same drafter, context and bonus token
  drafted with blocks of 8 and of 4 slots.  A causal drafter would give the
  first four slots the same hidden states in both; on the GPU they differ
  (later slots reach earlier ones), and each block size matches the oracle.
* No flow between blocks is checked in tests/test_gpu_tiny.py (two
  sequences drafted in one pass).
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__ as g
    g.build()
    import block_diffusion_speculative_layer_gb300 as m
    return m


SMALL_BF16 = syn.ModelShape("small-bf16-struct", n_layers=8, d_model=512, n_q_heads=4, n_kv_heads=2, head_dim=128,
                            d_ffn=1024, vocab=2048, draft_layers=2, block_size=16, dtype="bf16")


@pytest.mark.parametrize("shape", [syn.TINY, SMALL_BF16], ids=["tiny-fp32", "small-bf16"])
def test_one_drafter_pass_per_cycle(dfl, shape):
    per_gemm = 1 if shape.dtype == "bf16" else 2     # the fp32 GEMM is a product kernel and an epilogue kernel
    with dfl.Engine(shape, syn.make_weights(shape), max_batch=1, max_ctx=256) as eng:
        p = syn.make_prompt(shape, 40, stream=70)
        eng.profile(True)
        out, stats = eng.generate([p], 30)
        prof = eng.profile_read()
        eng.profile(False)
    C = stats["cycles"]
    L, Ld = shape.n_layers, shape.draft_layers
    assert C >= 2
    calls = {k: v["launches"] // per_gemm for k, v in prof.items() if k in ("gemm", "lm_head", "fuse", "inject")}
    # prefill: L target layers, one LM head row, fusion + injection of the prompt;
    # each cycle: Ld drafter layers + L target layers, two LM heads, one fusion + injection
    assert calls["gemm"] == 4 * L * (1 + C) + 4 * Ld * C
    assert calls["lm_head"] == 1 + 2 * C
    assert calls["fuse"] == 1 + C and calls["inject"] == 1 + C


def test_later_slots_reach_earlier_slots(dfl):
    shape8 = syn.TINY
    shape4 = syn.TINY.replace(block_size=4)
    w = syn.make_weights(shape8)
    model = O.Model(O.Weights(w), shape8)
    p = syn.make_prompt(shape8, 30, stream=71)
    hidden = {}
    for shape in (shape8, shape4):
        with dfl.Engine(shape, w, max_batch=1, max_ctx=128) as eng:
            eng.debug(True)
            bonus = eng.prefill(0, p)
            eng.draft_block([0])
            hidden[shape.block_size] = eng.debug_read(dfl.DF_DBG_DRAFT_HIDDEN)
            ctx = eng.debug_read(dfl.DF_DBG_CTX)
    assert hidden[8].shape == (8, shape8.d_model) and hidden[4].shape == (4, shape8.d_model)
    # each block size against the oracle's drafter on the same context
    cc = O.ContextCache(1, shape8.n_kv_heads, shape8.head_dim)
    tp = O.teacher_forced(model, p)
    O.inject_kv(model.W, shape8, cc, O.fuse_features(model.W, shape8, tp.taps))
    for b, shape in ((8, shape8), (4, shape4)):
        ref = O.draft_blocks(model.W, shape, cc, [(bonus, len(p))]).hidden
        np.testing.assert_allclose(hidden[b], ref, rtol=0, atol=1e-4 * np.abs(ref).max())
    # slots 0..3 see slots 4..7 in the block of 8: their states differ from the block of 4
    diff = np.abs(hidden[8][:4] - hidden[4]).max(axis=1)
    assert (diff > 1e-3 * np.abs(hidden[4]).max()).all(), diff


def test_in_situ_timing_partitions_the_cycles(dfl):
    """df_profile_enable mode 2: the captured cycles stamp every GEMM and
    attention launch; the per-class times add up to (at most) the cycles'
    device time, the launch counts are one drafter and one verify pass per
    cycle, and the decoded stream is unchanged."""
    shape = SMALL_BF16
    with dfl.Engine(shape, syn.make_weights(shape), max_batch=1, max_ctx=512) as eng:
        p = syn.make_prompt(shape, 64, stream=72)
        ref = eng.greedy_reference([p], 60)
        eng.generate([p], 20)                   # first cycles (eager) and graph capture
        eng.profile(True, in_situ=True)
        out, stats = eng.generate([p], 60)
        prof = eng.profile_read()
        eng.profile(False)
    np.testing.assert_array_equal(out, ref)
    C = stats["cycles"]
    L, Ld = shape.n_layers, shape.draft_layers
    assert prof["gemm"]["launches"] == 4 * (L + Ld) * C
    assert prof["lm_head"]["launches"] == 2 * C
    assert prof["fuse"]["launches"] == C and prof["inject"]["launches"] == C
    assert prof["attention"]["launches"] == (L + Ld) * C
    total_us = sum(v["us"] for v in prof.values())
    cycle_us = stats["draft_us"] + stats["verify_us"]
    assert all(v["us"] >= 0 for v in prof.values())
    # the stamps cut the cycles' timeline: their sum cannot exceed it by more than rounding
    assert 0.5 * cycle_us < total_us < 1.05 * cycle_us + 50.0, (total_us, cycle_us)
