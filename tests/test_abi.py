"""The C ABI library: builds, loads, exports every declared symbol, and its
host-only calls agree with the pages' closed forms.  No GPU is touched."""
import ctypes
import os
import re

import numpy as np
import pytest

import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__ as g
    g.build()
    import block_diffusion_speculative_layer_gb300 as dfl
    return dfl.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(df_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_cycle_calls():
    syms = declared_symbols()
    for s in ["df_init", "df_prefill", "df_draft_block", "df_verify_accept", "df_generate", "df_greedy_reference",
              "df_reset_seq", "df_destroy", "df_last_error", "df_default_feat_layers"]:
        assert s in syms


def test_library_exports_every_declared_symbol(L):
    missing = [s for s in declared_symbols() if not hasattr(L, s)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    import block_diffusion_speculative_layer_gb300 as dfl
    assert sorted(dfl.EXPORTED) == declared_symbols()


def test_feature_layers_from_library(L):
    import block_diffusion_speculative_layer_gb300 as dfl
    golden = os.path.join(ROOT, "tests", "golden", "feature_layers.txt")
    for line in open(golden):
        if line.strip() and not line.startswith("#"):
            v = [int(x) for x in line.split()]
            assert dfl.default_feat_layers(v[0]) == v[1:]
    out = (ctypes.c_int32 * 5)()
    assert L.df_default_feat_layers(7, out) == dfl.DF_EINVAL


@pytest.mark.parametrize("shape", [syn.TINY, syn.QWEN3_8B, syn.DENSE_27B])
def test_weight_list_matches_generator(L, shape):
    import block_diffusion_speculative_layer_gb300 as dfl
    cfg = dfl.make_config(shape, 1, 1024)
    assert dfl.weight_info(cfg) == syn.weight_specs(shape)


def test_init_rejects_bad_config_without_gpu(L):
    import block_diffusion_speculative_layer_gb300 as dfl
    cfg = dfl.make_config(syn.TINY, 1, 256)
    cfg.head_dim = 96
    h = ctypes.c_void_p()
    ptrs = (ctypes.c_void_p * 1)()
    assert L.df_init(ctypes.byref(cfg), ptrs, 1, None, ctypes.byref(h)) == dfl.DF_EINVAL
    assert not h.value
    cfg = dfl.make_config(syn.TINY, 1, 256)
    cfg.block_size = 1
    assert L.df_init(ctypes.byref(cfg), ptrs, 1, None, ctypes.byref(h)) == dfl.DF_EINVAL


def test_null_handle_calls_fail_cleanly(L):
    import block_diffusion_speculative_layer_gb300 as dfl
    assert L.df_prefill(None, 0, None, 0, None) == dfl.DF_EINVAL
    assert L.df_last_error(None) == b"null handle"
    L.df_destroy(None)


def test_parameter_counts_match_pages_sizing():
    # The 27B-class drafter (5 layers of width 5120, no own embedding/LM head)
    # has about 1.78B parameters: the "about 2B drafter" sizing of the pages.
    s = syn.DENSE_27B
    n = sum(int(np.prod(shp)) for name, shp in syn.weight_specs(s) if name.startswith("d") or name.startswith("fc"))
    assert 1.7e9 < n < 2.0e9


def test_sampling_calls_reject_bad_arguments_without_gpu(L):
    # every check below returns before anything is launched
    import block_diffusion_speculative_layer_gb300 as dfl
    n = None
    assert L.df_op_sampling_probs(n, 1, 10, -1.0, 1.0, n, n, n) == dfl.DF_EINVAL           # negative temperature
    assert L.df_op_sampling_probs(n, 1, 10, 1e-4, 1.0, n, n, n) == dfl.DF_EINVAL           # below 1e-3
    assert L.df_op_sampling_probs(n, 1, 10, float("nan"), 1.0, n, n, n) == dfl.DF_EINVAL
    assert L.df_op_sampling_probs(n, 1, 10, 1.0, 1.5, n, n, n) == dfl.DF_EINVAL            # top_p above 1
    assert L.df_op_sampling_probs(n, 1, 10, 1.0, -0.1, n, n, n) == dfl.DF_EINVAL
    assert L.df_op_sampling_probs(n, 1, (1 << 19) + 1, 1.0, 1.0, n, n, n) == dfl.DF_EINVAL  # vocabulary too large
    assert L.df_op_sampling_probs(n, 1, 10, 1.0, 0.9, n, n, n) == dfl.DF_EINVAL            # missing buffers
    assert L.df_op_sampling_probs(n, 0, 10, 1.0, 0.9, n, n, n) == dfl.DF_OK                # no rows: nothing to do
    assert L.df_op_sample_draw(n, 1, 10, 0.0, 1.0, n, n, n, n) == dfl.DF_EINVAL
    assert L.df_op_accept_sampled(n, n, n, 1, 1, 10, 1.0, 1.0, n, n, n, n, n) == dfl.DF_EINVAL   # B < 2
    assert L.df_op_accept_sampled(n, n, n, 1, 33, 10, 1.0, 1.0, n, n, n, n, n) == dfl.DF_EINVAL  # B > 32
    assert L.df_op_accept_sampled(n, n, n, 0, 4, 10, 1.0, 1.0, n, n, n, n, n) == dfl.DF_OK
    assert L.df_op_philox_uniforms(0, 0, 0, -1, n, n) == dfl.DF_EINVAL
    assert L.df_op_philox_uniforms(0, 0, 0, 0, n, n) == dfl.DF_OK
    assert L.df_generate_sampled(n, n, n, 1, 1, 1.0, 1.0, 0, n, n) == dfl.DF_EINVAL        # null handle


def test_block_size_rule():
    # the smallest power of two >= 2 x tokens per cycle, clamped to [b_min, b_max]
    import block_diffusion_speculative_layer_gb300 as dfl
    f = dfl.block_size_for
    assert [f(t, 2, 16) for t in (0.0, 1.0, 1.2, 2.0, 2.5, 4.0, 5.0, 8.0, 30.0)] == [2, 2, 4, 4, 8, 8, 16, 16, 16]
    assert f(1.0, 4, 16) == 4 and f(7.0, 2, 12) == 12 and f(3.0, 6, 6) == 6
    for b in (2, 4, 8):
        assert f(float(b), 2, 16) == min(2 * b, 16)     # a group that keeps every draft doubles the block
    prev = 0
    for t in np.linspace(0.0, 20.0, 401):
        b = f(float(t), 2, 16)
        assert b >= prev and (b >= 2 * t or b == 16) and b in (2, 4, 8, 16)
        prev = b
    for bad in [(1.0, 1, 8), (1.0, 8, 4), (1.0, 2, 33), (-1.0, 2, 8)]:
        with pytest.raises(dfl.DfError):
            f(*bad)


def test_block_range_needs_a_handle(L):
    import block_diffusion_speculative_layer_gb300 as dfl
    assert L.df_set_block_range(None, 2, 8) == dfl.DF_EINVAL
    out = (ctypes.c_int64 * 33)()
    assert L.df_generate_accept_hist(None, 0, out) == dfl.DF_EINVAL
    assert L.df_debug_wait_probe(None) == dfl.DF_EINVAL


def test_attention_op_rejects_bad_arguments(L):
    # every case is refused before any CUDA call (fake device addresses are never touched)
    import block_diffusion_speculative_layer_gb300 as dfl
    P = ctypes.c_void_p
    fake = P(0x1000)
    base = dict(q=fake, out=fake, cache=fake, n_pages=4, pt=fake, pt_stride=8, pos=fake, seq=fake, blk=fake,
                rows_cap=16, nseq=1, rows=16, hq=32, hkv=8, causal=0, max_len=100, kernel=dfl.DF_ATTN_MMA, cla=0,
                err=fake)

    def call(**kw):
        a = dict(base, **kw)
        return L.df_op_attention_bf16(a["q"], a["out"], a["cache"], a["n_pages"], a["pt"], a["pt_stride"], a["pos"],
                                      a["seq"], a["blk"], a["rows_cap"], a["nseq"], a["rows"], a["hq"], a["hkv"],
                                      a["causal"], a["max_len"], a["kernel"], a["cla"], a["err"], None)

    assert call(q=None) == dfl.DF_EINVAL
    assert call(kernel=0) == dfl.DF_EINVAL            # AUTO is an engine setting, not a kernel
    assert call(kernel=3) == dfl.DF_EINVAL
    assert call(hq=36) == dfl.DF_EINVAL               # not a multiple of the KV heads
    assert call(hq=72) == dfl.DF_EINVAL               # more than 8 query heads per KV head
    assert call(causal=2) == dfl.DF_EINVAL
    assert call(max_len=8 * 16 + 1) == dfl.DF_EINVAL  # more positions than the page table holds
    assert call(blk=None) == dfl.DF_EINVAL            # the block form needs the block rows
    assert call(rows=65) == dfl.DF_EINVAL             # a block holds at most 64 rows
    assert call(rows_cap=8) == dfl.DF_EINVAL          # fewer block rows than query rows
    assert call(cla=3) == dfl.DF_EINVAL               # clusters of 2, 4, 8 or 16 CTAs
