"""The benchmark's own depths on the GPU: the 36-layer Qwen3-8B-shaped model
(d 4096, GQA 32/8 x 128, SwiGLU 12288, vocab 151936, 5-layer drafter, block
16) and the 64-layer 27B-class model (d 5120, GQA 40/8, SwiGLU 17408).

Weights are drawn on the GPU (``synthetic.iter_weights_device``: N(0, 0.02),
unit gains); the oracle reads host copies of the matrices it needs.

* Lossless: the speculative stream equals the GPU's token-by-token greedy
  decode, bit for bit, for 128 new tokens (two ragged prompts in one batch
  for the 27B-class model).
* Parity at 2e-2 under per-layer teacher forcing (tests/_teacher.py) on the
  first, a middle and the last target layer, the first and last drafter
  layer, the fusion and both LM heads, over two fully accepted cycles; every
  tap is checked exactly against the residual rows of its layer.
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


def device_weights(shape, host_names):
    """(device weights in canonical order, host uint16/float32 copies of host_names)."""
    dev, host = [], {}
    for name, t in syn.iter_weights_device(shape):
        dev.append((name, t))
        if name in host_names:
            a = t.contiguous().cpu()
            host[name] = a.view(torch.int16).numpy().view(np.uint16) if shape.dtype == "bf16" else a.numpy()
    return dev, host


def host_names(shape, target_layers, drafter_layers):
    names = {"final_norm", "lm_head", "fc", "fc_norm", "d_final_norm"}
    for l in target_layers:
        names |= {f"t{l}.{m}" for m in syn.LAYER_MATS}
    for l in range(shape.draft_layers):   # injection uses every drafter layer's W_k / W_v
        names |= {f"d{l}.wk", f"d{l}.wv"}
    for l in drafter_layers:
        names |= {f"d{l}.{m}" for m in syn.LAYER_MATS}
    return names


def run_depth(dfl, shape, prompts, n_new, target_layers, drafter_layers, parity_prompt):
    names = host_names(shape, target_layers, drafter_layers)
    dev, host = device_weights(shape, names)
    max_ctx = ((max(len(p) for p in prompts + [parity_prompt]) + n_new + 4 * shape.block_size + 63) // 64) * 64
    eng = dfl.Engine(shape, dev, max_batch=len(prompts), max_ctx=max_ctx)
    del dev
    torch.cuda.empty_cache()
    try:
        spec, stats = eng.generate(prompts, n_new)
        greedy = eng.greedy_reference(prompts, n_new)
        np.testing.assert_array_equal(spec, greedy)
        assert stats["emitted_tokens"] == n_new * len(prompts)

        B = shape.block_size
        g = eng.greedy_reference([parity_prompt], 2 * B + 1)[0]
        rep = T.Report(T.TOL)
        W = O.Weights(host, cache=False)
        T.forced_cycles(dfl, eng, W, shape, parity_prompt, g, 2, rep, target_layers=target_layers,
                        drafter_layers=drafter_layers)
        print(f"\n[{shape.name}] per-layer teacher forcing, worst {rep.worst():.3e}\n" + rep.text())
        rep.check()
    finally:
        eng.close()


def test_qwen3_8b_full_depth(dfl):
    s = syn.QWEN3_8B
    prompts = [syn.make_prompt(s, 512, stream=0)]
    run_depth(dfl, s, prompts, 128, [0, s.n_layers // 2, s.n_layers - 1], [0, s.draft_layers - 1],
              syn.make_prompt(s, 64, stream=21))


def test_27b_class_full_depth(dfl):
    s = syn.DENSE_27B
    prompts = [syn.make_prompt(s, 200, stream=0), syn.make_prompt(s, 77, stream=1)]
    run_depth(dfl, s, prompts, 128, [0, s.n_layers // 2, s.n_layers - 1], [0, s.draft_layers - 1],
              syn.make_prompt(s, 64, stream=22))
