"""The pipelined tcgen05 attention (df_config.attn_kernel = DF_ATTN_PIPE).

Source: [ARCH] "DFlash 的架构密码", 第三层 Block Diffusion and 稀疏注意力训练
(the drafter's block attends over the injected context and, bidirectionally,
its own block; the target's verify pass is causal).

The same bars as the default kernel: per-layer teacher-forced parity with the
float64 oracle within 2e-2 (tests/_teacher.py), speculative output equal to
the GPU's own greedy decode (lossless), no flow between the sequences of a
batch.  Query-head groups of 4 (the Qwen3-8B grouping), 5 (the 27B class:
the fifth head of a group sits in the second half of a tensor-memory lane
quadrant) and 8, single sequences, ragged batches with long prompts and a
long context whose chunks run through every pipeline stage several times.
"""
import numpy as np
import pytest

import synthetic as syn
from oracle import dflash_oracle as O

import _teacher as T

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


G4 = syn.ModelShape("pipe-g4", n_layers=8, d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128,
                    d_ffn=2048, vocab=4096, draft_layers=2, block_size=16, dtype="bf16")
G5 = syn.ModelShape("pipe-g5", n_layers=8, d_model=1280, n_q_heads=10, n_kv_heads=2, head_dim=128,
                    d_ffn=2048, vocab=4096, draft_layers=1, block_size=16, dtype="bf16")
G8 = syn.ModelShape("pipe-g8", n_layers=8, d_model=2048, n_q_heads=16, n_kv_heads=2, head_dim=128,
                    d_ffn=2048, vocab=4096, draft_layers=1, block_size=8, dtype="bf16")


def engine(dfl, shape, w, max_batch, max_ctx):
    return dfl.Engine(shape, w, max_batch=max_batch, max_ctx=max_ctx, attn_kernel=dfl.DF_ATTN_PIPE)


@pytest.mark.parametrize("shape,prompt_len", [(G4, 48), (G5, 40), (G8, 40), (G4, 500)],
                         ids=["g4", "g5", "g8", "g4-500"])
def test_layer_parity(dfl, shape, prompt_len):
    w = syn.make_weights(shape, gain_std=0.1)
    model = O.Model(O.Weights(w), shape)
    with engine(dfl, shape, w, 1, 1024) as eng:
        prompt = syn.make_prompt(shape, prompt_len, stream=90)
        g = eng.greedy_reference([prompt], 2 * shape.block_size + 1)[0]
        rep = T.Report(T.TOL)
        T.forced_cycles(dfl, eng, model.W, shape, prompt, g, 2, rep)
    print(f"\n[{shape.name} pipelined attention] worst {rep.worst():.3e}")
    rep.check()


@pytest.mark.parametrize("shape", [G4, G5, G8], ids=["g4", "g5", "g8"])
def test_lossless_ragged_batch(dfl, shape):
    w = syn.make_weights(shape)
    with engine(dfl, shape, w, 4, 2048 + 128) as eng:
        lens = [17, 700, 5, 2048 - 64]
        prompts = [syn.make_prompt(shape, L, stream=91 + i) for i, L in enumerate(lens)]
        spec, _ = eng.generate(prompts, 40)
        greedy = eng.greedy_reference(prompts, 40)
        np.testing.assert_array_equal(spec, greedy)
        alone, _ = eng.generate(prompts[1:2], 40)      # a sequence alone == in the batch
        np.testing.assert_array_equal(alone[0], spec[1])


def test_long_context_lossless(dfl):
    # 9000 positions: 141 chunks of 64 keys, 8 to 9 per CTA of a 16-CTA
    # cluster, so each of the four stages is refilled
    shape = G4
    w = syn.make_weights(shape, gain_std=0.1)
    with engine(dfl, shape, w, 1, 9216) as eng:
        p = syn.make_prompt(shape, 9000, stream=95)
        spec, _ = eng.generate([p], 24)
        np.testing.assert_array_equal(spec, eng.greedy_reference([p], 24))


def test_long_context_parity(dfl):
    # 3300 positions (52 chunks): the first cycle after the prompt against the
    # oracle run on its own; the small model's accumulated error stays within 2e-2
    shape = G4
    w = syn.make_weights(shape, gain_std=0.1)
    p = syn.make_prompt(shape, 3300, stream=8)
    B = shape.block_size
    with engine(dfl, shape, w, 1, 3456) as eng:
        g = eng.greedy_reference([p], B + 1)[0]
        eng.debug(True)
        try:
            eng.prefill(0, p)
            eng.verify_accept([0], g[1:B])
            logits = eng.debug_read(dfl.DF_DBG_LOGITS)
            hidden = eng.debug_read(dfl.DF_DBG_HIDDEN)
        finally:
            eng.reset_seq(0)
            eng.debug(False)
    model = O.Model(O.Weights(w), shape)
    cache = O.KVCache(shape.n_layers, shape.n_kv_heads, shape.head_dim)
    O.target_forward(model.W, shape, p, cache)
    ver = O.target_forward(model.W, shape, g[:B], cache)
    assert T.rel_err(hidden, ver.hidden[-1]) <= T.TOL
    assert T.rel_err(logits, ver.logits) <= T.TOL


def test_no_flow_between_sequences(dfl):
    shape = G4
    w = syn.make_weights(shape)
    pa, pb, pc = (syn.make_prompt(shape, 300, stream=s) for s in (96, 97, 98))
    with engine(dfl, shape, w, 2, 1024) as eng:
        eng.debug(True)
        res = []
        for other in (pb, pc):
            eng.prefill(0, pa)
            eng.prefill(1, other)
            d = eng.draft_block([0, 1])
            res.append((d, eng.debug_read(dfl.DF_DBG_DRAFT_HIDDEN)))
            eng.reset_seq(0)
            eng.reset_seq(1)
        eng.debug(False)
    B = shape.block_size
    np.testing.assert_array_equal(res[0][0][0], res[1][0][0])
    np.testing.assert_array_equal(res[0][1][:B], res[1][1][:B])
    assert np.abs(res[0][1][B:] - res[1][1][B:]).max() > 0


@pytest.mark.parametrize("page_tokens", [8, 32, 64])
@pytest.mark.parametrize("kernel", ["pipe", "mma"])
def test_lossless_other_page_sizes(dfl, page_tokens, kernel):
    # KV pages of 8, 32 or 64 tokens (one TMA box per page half): a ragged batch
    # decodes the GPU's own greedy stream, and a sequence alone equals itself in the batch
    shape = G4
    w = syn.make_weights(shape)
    k = dfl.DF_ATTN_PIPE if kernel == "pipe" else dfl.DF_ATTN_MMA
    with dfl.Engine(shape, w, max_batch=4, max_ctx=1024 + 128, page_tokens=page_tokens, attn_kernel=k) as eng:
        lens = [33, 700, 5, 1000]
        prompts = [syn.make_prompt(shape, L, stream=120 + i) for i, L in enumerate(lens)]
        spec, _ = eng.generate(prompts, 32)
        np.testing.assert_array_equal(spec, eng.greedy_reference(prompts, 32))
        alone, _ = eng.generate(prompts[3:4], 32)
        np.testing.assert_array_equal(alone[0], spec[3])


def test_page_size_does_not_change_the_stream(dfl):
    # the attention's arithmetic depends on chunk positions, not on the page size
    shape = G4
    w = syn.make_weights(shape)
    p = syn.make_prompt(shape, 300, stream=130)
    outs = []
    for pt in (16, 64):
        with dfl.Engine(shape, w, max_batch=1, max_ctx=512, page_tokens=pt, attn_kernel=dfl.DF_ATTN_PIPE) as eng:
            outs.append(eng.generate([p], 24)[0])
    np.testing.assert_array_equal(outs[0], outs[1])
