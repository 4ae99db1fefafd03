"""Kernel microbenchmarks through the C ABI (device time from CUDA events).

  python -m block_diffusion_speculative_layer_gb300.microbench gemm --M 16 --N 24576 --K 4096 --iters 20
  python -m block_diffusion_speculative_layer_gb300.microbench lmhead --M 16 --N 151936 --K 4096
  python -m block_diffusion_speculative_layer_gb300.microbench drafter [--blocks 8,16] [--ctx 1024,4096,16384,32768]
                                                                       [--batch 1,4,16,32]
  python -m block_diffusion_speculative_layer_gb300.microbench ar_proxy
  python -m block_diffusion_speculative_layer_gb300.microbench serving [--new 1024]
  python -m block_diffusion_speculative_layer_gb300.microbench dense27b [--new 1024]
  python -m block_diffusion_speculative_layer_gb300.microbench profile_cycle [--ctx 1024] [--batch 1] [--vocab 4096]
  python -m block_diffusion_speculative_layer_gb300.microbench offpath [--model fp32|bf16]
  python -m block_diffusion_speculative_layer_gb300.microbench attention [--ctx ...] [--batch ...] [--attn mma|pipe|auto]
                                                                         [--causal] [--iters 5] [--pages shuffled|runs]

Inputs are seeded synthetic bf16 (N(0,1) activations, N(0,0.02) weights)
drawn on the GPU by torch.  For small shapes several weight copies are used
in turn so that launches never hit in L2.  The GEMM loop runs inside the
library (df_op_bench_gemm_bf16): no host work between launches.
"""
import argparse
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def drafter(a):
    """Drafter step alone on the Qwen3-8B width: fusion, injection, block attention, LM-head argmax."""
    import numpy as np
    import torch

    import block_diffusion_speculative_layer_gb300 as dfl
    import synthetic as syn

    blocks = [int(x) for x in a.blocks.split(",")]
    ctxs = [int(x) for x in a.ctx.split(",")]
    batches = [int(x) for x in a.batch.split(",")]
    for B in blocks:
        # the target is not used by the drafter step: its minimum depth keeps memory low
        shape = syn.QWEN3_8B.replace(name=f"drafter-step-B{B}", n_layers=8, block_size=B)
        if a.reduced:
            # Qwen3-8B width and heads, one drafter layer, a 4096-token vocabulary:
            # the same kernels on a few GB of device memory (profiling captures)
            shape = shape.replace(draft_layers=1, vocab=4096)
        d, kvd = shape.d_model, shape.kv_dim
        taps = syn.make_hidden(512, 5 * d).reshape(512, 5, d)   # N(0, 1) feature rows
        # one engine per batch size, configured for that batch (the attention kernel and its
        # cluster size are chosen per engine from max_batch and max_ctx)
        for nb in batches:
            eng = dfl.Engine(shape, syn.iter_weights_device(shape), max_batch=nb, max_ctx=max(ctxs) + 2 * B,
                             attn_kernel=_attn(a), page_tokens=a.page_tokens)
            torch.cuda.empty_cache()
            for C in ctxs:
                r = eng.bench_drafter_step(nb, C, taps, iters=a.iters)
                M = nb * B
                byts = {
                    "fuse": 2 * d * 5 * d + M * 5 * d * 2 + M * d * 2,
                    "inject": 2 * shape.draft_layers * 2 * kvd * d + M * d * 2 + M * shape.draft_layers * 2 * kvd * 2,
                    "block_attention": shape.draft_layers * (nb * (C + B) * 2 * kvd * 2 + 2 * M * shape.q_dim * 2),
                    "lm_head": 2 * shape.vocab * d + M * d * 2 + M * 8,
                }
                us = {"fuse": r["fuse_us"], "inject": r["inject_us"], "block_attention": r["block_attention_us"],
                      "lm_head": r["lm_head_us"]}
                print(json.dumps({"op": "drafter_step", "block": B, "ctx": C, "batch": nb, "attn": a.attn,
                                  "page_tokens": a.page_tokens,
                                  "us": {k: round(v, 2) for k, v in us.items()},
                                  "drafter_pass_us": round(r["drafter_pass_us"], 2),
                                  "total_us": round(sum(us.values()), 2),
                                  "GB/s": {k: round(byts[k] / (us[k] * 1e-6) / 1e9, 1) for k in us if us[k] > 0}}),
                      flush=True)
            eng.close()


def ar_proxy(a):
    """Draft latency of one 5-layer, 16-slot drafter pass against an
    autoregressive 1-layer drafter making 8 drafts in 8 sequential passes
    (each pass: one layer over a 2-row block and the LM head), both at the
    Qwen3-8B width, batch 1, 1024 context positions."""
    import block_diffusion_speculative_layer_gb300 as dfl
    import synthetic as syn

    C = 1024
    taps = syn.make_hidden(512, 5 * 4096).reshape(512, 5, 4096)
    res = {}
    for name, layers, B in (("dflash_5layer_block16", 5, 16), ("ar_1layer_step", 1, 2)):
        shape = syn.QWEN3_8B.replace(name=name, n_layers=8, draft_layers=layers, block_size=B)
        eng = dfl.Engine(shape, syn.iter_weights(shape), max_batch=1, max_ctx=C + 2 * B)
        res[name] = eng.bench_drafter_step(1, C, taps, iters=10)["drafter_pass_us"]
        eng.close()
    ar8 = 8 * res["ar_1layer_step"]
    print(json.dumps({"op": "draft_latency_proxy", "ctx": C,
                      "dflash_5layer_16slots_us": round(res["dflash_5layer_block16"], 2),
                      "ar_1layer_8steps_us": round(ar8, 2),
                      "ratio_ar_over_dflash": round(ar8 / res["dflash_5layer_block16"], 3),
                      "note": "random weights: latency only; one drafter pass includes its LM head"}))


def _generation(shape, prompts, n_new, max_ctx, label, config, block_range=None, sampling=None, attn=0,
                profile=False, page_tokens=16):
    """One timed df_generate over a batch (device weights drawn on the GPU),
    after one untimed warm-up generation of 16 tokens.  block_range: (b_min,
    b_max) for df_set_block_range, or None for the configured block size.
    sampling: (temperature, top_p, seed) for df_generate_sampled, or None."""
    import numpy as np
    import torch

    import block_diffusion_speculative_layer_gb300 as dfl
    import synthetic as syn

    t0 = time.time()
    eng = dfl.Engine(shape, syn.iter_weights_device(shape), max_batch=len(prompts), max_ctx=max_ctx,
                     attn_kernel=attn, page_tokens=page_tokens)
    torch.cuda.empty_cache()
    setup_s = time.time() - t0
    if block_range:
        eng.set_block_range(*block_range)

    def run(n):
        if sampling:
            return eng.generate_sampled(prompts, n, temperature=sampling[0], top_p=sampling[1], seed=sampling[2])
        return eng.generate(prompts, n)

    run(16)
    torch.cuda.synchronize()
    eng.reset_stats()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(eng.stream)
    out, st = run(n_new)
    e1.record(eng.stream)
    torch.cuda.synchronize()
    secs = e0.elapsed_time(e1) / 1000.0
    s2 = eng.stats()
    hist = [int(x) for x in s2["accept_hist"]]
    per_seq = eng.accept_hist_per_seq(len(prompts))
    insitu = None
    if profile:
        # one more generation with in-situ stamps: device time per kernel class inside the cycles
        eng.profile(True, in_situ=True)
        run(n_new)
        pr = eng.profile_read()
        eng.profile(False)
        insitu = {k: {"launches": v["launches"], "ms": round(v["us"] / 1000.0, 3),
                      "GB/s": round(v["bytes"] / (v["us"] * 1e-6) / 1e9, 1) if v["us"] > 0 and v["bytes"] > 0 else None,
                      "TFLOP/s": round(v["flops"] / (v["us"] * 1e-6) / 1e12, 1) if v["us"] > 0 and v["flops"] > 0 else None}
                  for k, v in pr.items() if v["launches"]}
    eng.close()
    tokens = len(prompts) * n_new
    print(json.dumps({"op": label, "config": config, "attn_kernel": attn, "page_tokens": page_tokens, "sequences": len(prompts),
                      "new_tokens_each": n_new,
                      "tokens_per_s": tokens / secs, "wall_s": secs, "cycles": s2["cycles"],
                      # the engine counts one cycle per sequence per draft + verify pass
                      "mean_accept_len": s2["emitted_tokens"] / max(1, s2["cycles"]),
                      "accept_hist_k": {str(k): v for k, v in enumerate(hist) if v},
                      "accept_hist_k_per_sequence": [{str(k): int(v) for k, v in enumerate(h) if v} for h in per_seq],
                      "block_range": list(block_range) if block_range else None,
                      "sampling": {"temperature": sampling[0], "top_p": sampling[1], "seed": sampling[2]}
                      if sampling else None,
                      "block_hist": {str(b): v for b, v in enumerate(s2["block_hist"]) if v},
                      # device time is summed once per cycle of the batch, cycles once per sequence
                      "draft_us_per_cycle": s2["draft_us"] * len(prompts) / max(1, s2["cycles"]),
                      "verify_us_per_cycle": s2["verify_us"] * len(prompts) / max(1, s2["cycles"]),
                      "prefill_us": s2["prefill_us"], "kernel_launches": s2["kernel_launches"],
                      "setup_s": setup_s, "in_situ": insitu,
                      "data": "synthetic, weights drawn on the GPU (seeded), random prompt ids"}),
          flush=True)


def serving(a):
    """Serving-shaped batch on the Qwen3-8B shape: 16 sequences, prompt lengths
    uniform over 128..2048, 16-token pages, block 16, greedy."""
    import synthetic as syn

    shape = syn.QWEN3_8B
    lens = syn.make_prompt_lengths(16, 128, 2048)
    prompts = [syn.make_prompt(shape, int(L), stream=200 + i) for i, L in enumerate(lens)]
    max_ctx = ((int(max(lens)) + a.new + 16 + 2 * shape.block_size + 63) // 64) * 64
    _generation(shape, prompts, a.new, max_ctx, "serving_batch16",
                "qwen3-8b-shape bf16, 16 sequences, prompts U[128,2048], block 16, %d new each" % a.new,
                _block_range(a), attn=_attn(a), profile=a.profile, page_tokens=a.page_tokens)


def sampled(a):
    """Speculative sampling on the Qwen3-8B shape at batch 1: prompt 512,
    block 16, temperature and top_p from --sampling (default 0.8, 0.95)."""
    import synthetic as syn

    shape = syn.QWEN3_8B
    T, top_p = (float(x) for x in a.sampling.split(","))
    prompts = [syn.make_prompt(shape, 512)]
    _generation(shape, prompts, a.new, 512 + a.new + 64, "sampled_bs1",
                "qwen3-8b-shape bf16, batch 1, prompt 512, block 16, %d new, temperature %g, top_p %g"
                % (a.new, T, top_p), _block_range(a), (T, top_p, 1), attn=_attn(a), profile=a.profile)


def dense27b(a):
    """27B-class target (64 layers, d 5120, 40/8 heads, FFN 17408, vocabulary
    151936) with a 5-layer drafter, batch 4, 8192-token prompts, block 16."""
    import synthetic as syn

    shape = syn.DENSE_27B
    prompts = [syn.make_prompt(shape, 8192, stream=300 + i) for i in range(4)]
    max_ctx = ((8192 + a.new + 16 + 2 * shape.block_size + 63) // 64) * 64
    _generation(shape, prompts, a.new, max_ctx, "dense27b_batch4",
                "27b-class bf16, batch 4, prompt 8192, block 16, %d new each" % a.new, _block_range(a),
                attn=_attn(a), profile=a.profile, page_tokens=a.page_tokens)


def profile_cycle(a):
    """Every kernel of one decode cycle, for profilers: the Qwen3-8B width and
    heads with 8 target layers, 1 drafter layer and a vocabulary of --vocab
    (weights drawn on the GPU), batch --batch with prompts of --ctx tokens, a
    few cycles run one call at a time (df_draft_block, df_verify_accept),
    cycle 2 inside the NVTX range "cycle".  Then the sampling operations on
    fp32 logits of 16 rows x 151936 inside the NVTX range "sampling"."""
    import numpy as np
    import torch

    import block_diffusion_speculative_layer_gb300 as dfl
    import synthetic as syn

    shape = syn.QWEN3_8B.replace(name="profile-cycle", n_layers=8, draft_layers=1, vocab=a.vocab)
    nb, C = a.batch, a.ctx
    eng = dfl.Engine(shape, syn.iter_weights_device(shape), max_batch=nb, max_ctx=C + 8 * shape.block_size,
                     attn_kernel=_attn(a))
    torch.cuda.empty_cache()
    seqs = list(range(nb))
    for i in seqs:
        eng.prefill(i, syn.make_prompt(shape, C, stream=400 + i))
    for c in range(4):
        if c == 2:
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_push("cycle")
        eng.draft_block(seqs)
        eng.verify_accept(seqs)
        if c == 2:
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_pop()
    eng.close()
    V, rows = 151936, 16
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn(rows, V, device="cuda", generator=g) * 4.0
    p = torch.randn(1, rows + 1, V, device="cuda", generator=g) * 4.0
    u = dfl.philox_uniforms(1, 0, 0, rows)
    for it in range(3):
        if it == 2:
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_push("sampling")
        dfl.sampling_probs(q, 0.8, 0.95)
        d = dfl.sample_draw(q, 0.8, 0.95, u)
        dfl.accept_sampled(d.reshape(1, rows), q.reshape(1, rows, V), p, 0.8, 0.95,
                           dfl.philox_uniforms(2, 0, 0, rows + 1).reshape(1, rows + 1))
        if it == 2:
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    print(json.dumps({"op": "profile_cycle", "batch": nb, "ctx": C, "vocab": a.vocab, "ok": True}))


def attention(a):
    """One attention launch alone (df_op_attention_bf16) on the Qwen3-8B heads
    (32 query / 8 KV x 128): the drafter's block attention over a context of
    C positions plus its 16-row block (or, with --causal, the target's causal
    attention of 16 verify rows), for each context and batch, on the
    mma.sync and/or pipelined kernel.  Keys and values are random bf16 in a
    paged cache whose pages are a random permutation of the pool (--pages
    shuffled) or each sequence's run of consecutive ids, as the engine's
    allocator hands them out (--pages runs); L2 is flushed (a 256 MB write) before
    every timed launch, and each launch is timed alone with CUDA events
    (after a device-side sleep that covers the host's preparation of the
    launch, so the events bracket the kernel only)."""
    import numpy as np
    import torch

    import block_diffusion_speculative_layer_gb300 as dfl

    Hq, Hkv, R, PT = 32, 8, 16, 16
    kernels = {"mma": [dfl.DF_ATTN_MMA], "pipe": [dfl.DF_ATTN_PIPE], "auto": [dfl.DF_ATTN_MMA, dfl.DF_ATTN_PIPE]}[a.attn]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(2)
    peak = _hbm_peak()
    for C in [int(x) for x in a.ctx.split(",")]:
        for nb in [int(x) for x in a.batch.split(",")]:
            need = C + (R if a.causal else 0)
            ppseq = (need + PT - 1) // PT
            n_pages = nb * ppseq
            cache = torch.randn((n_pages, 2, Hkv, PT, 128), device="cuda", generator=g).to(torch.bfloat16)
            perm = (torch.randperm(n_pages, device="cuda", generator=g).to(torch.int32) if a.pages == "shuffled"
                    else torch.arange(n_pages, device="cuda", dtype=torch.int32))
            table = perm.reshape(nb, ppseq).contiguous()
            q = torch.randn((nb * R, Hq * 128), device="cuda", generator=g).to(torch.bfloat16)
            blk = torch.randn((2, Hkv, nb * R, 128), device="cuda", generator=g).to(torch.bfloat16)
            pos = torch.tensor(np.concatenate([np.arange(C, C + R)] * nb), dtype=torch.int32, device="cuda")
            seq = torch.tensor(np.repeat(np.arange(nb), R), dtype=torch.int32, device="cuda")
            out = torch.empty_like(q)
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            torch.cuda.empty_cache()  # the fp32 draws' memory goes back before anything is timed or profiled
            visible = C + R
            byts = nb * visible * Hkv * 128 * 2 * 2 + 2 * nb * R * Hq * 128 * 2
            for k in kernels:
                def launch(check=False):
                    dfl.attention_bf16(q, cache, table, pos, seq, nb, R, Hkv, a.causal, need,
                                       blk=None if a.causal else blk, kernel=k, out=out, err=err,
                                       cluster_ctas=a.cla if k == dfl.DF_ATTN_PIPE else 0, check_rows=check)
                for w in range(a.warmup):
                    launch(check=w == 0)
                ts = []
                for _ in range(a.iters):
                    flush.zero_()
                    # the GPU sleeps while the host prepares the launch (tensor map, arguments; nothing
                    # that waits for the stream), so the events bracket the kernel alone
                    torch.cuda._sleep(1_000_000)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    launch()
                    e1.record()
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1000.0)
                us = float(np.median(ts))
                assert int(err.item()) == 0, f"attention error word {int(err.item())}"
                print(json.dumps({"op": "attention", "kernel": "pipe" if k == dfl.DF_ATTN_PIPE else "mma",
                                  "cluster_ctas": a.cla if k == dfl.DF_ATTN_PIPE else 16,
                                  "causal": bool(a.causal), "ctx": C, "batch": nb, "rows_per_seq": R, "pages": a.pages,
                                  "us": round(us, 2), "algorithmic_bytes": byts,
                                  "GB/s": round(byts / (us * 1e-6) / 1e9, 1),
                                  "frac_of_measured_hbm": round(byts / (us * 1e-6) / 1e9 / peak, 3)}), flush=True)
            del cache, perm, table, q, blk, out
            torch.cuda.empty_cache()


def offpath(a):
    """Small generations that launch the kernels the bs1 bf16 decode path does
    not (for ncu captures): the tiny fp32 model (greedy generation, greedy
    reference, sampled generation), or a small bf16 model (8 layers, d 512,
    4 / 2 heads x 128, a 300-token prompt, 16 new tokens) whose attention
    kernel follows DF_ATTN_SPLIT / DF_ATTN_TC in the environment."""
    import torch

    import block_diffusion_speculative_layer_gb300 as dfl
    import synthetic as syn

    if a.model == "fp32":
        shape = syn.TINY
        w = syn.make_weights(shape)
        prompt = syn.make_prompt(shape, 16)
        with dfl.Engine(shape, w, max_batch=1, max_ctx=128) as eng:
            _, st = eng.generate([prompt], 16)
            eng.greedy_reference([prompt], 8)
            eng.generate_sampled([prompt], 16, temperature=0.8, top_p=0.95, seed=3)
    else:
        shape = syn.ModelShape("offpath-bf16", n_layers=8, d_model=512, n_q_heads=4, n_kv_heads=2, head_dim=128,
                               d_ffn=1024, vocab=2048, draft_layers=1, block_size=8, dtype="bf16")
        w = syn.make_weights(shape)
        prompt = syn.make_prompt(shape, 300)
        with dfl.Engine(shape, w, max_batch=1, max_ctx=512) as eng:
            _, st = eng.generate([prompt], 16)
    torch.cuda.synchronize()
    print(json.dumps({"op": "offpath", "model": a.model, "cycles": st["cycles"], "ok": True}))


def _hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)["hbm_gbs"]
    return 6800.0


def _attn(a):
    """df_config.attn_kernel from --attn (auto, mma or pipe)."""
    return {"auto": 0, "mma": 1, "pipe": 2}[a.attn]


def _block_range(a):
    if not a.block_range:
        return None
    lo, hi = (int(x) for x in a.block_range.split(","))
    return lo, hi


def main():
    import torch

    import block_diffusion_speculative_layer_gb300 as dfl
    from block_diffusion_speculative_layer_gb300 import build

    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["gemm", "lmhead", "drafter", "ar_proxy", "serving", "dense27b", "sampled",
                                   "profile_cycle", "attention", "offpath"])
    ap.add_argument("--model", default="fp32", choices=["fp32", "bf16"], help="offpath: which small model")
    ap.add_argument("--causal", action="store_true", help="attention: the target's causal verify rows")
    ap.add_argument("--cla", type=int, default=4, help="attention: CTAs per cluster of the pipelined kernel")
    ap.add_argument("--pages", default="shuffled", choices=["shuffled", "runs"],
                    help="attention: page ids a random permutation of the pool, or consecutive per sequence")
    ap.add_argument("--profile", action="store_true",
                    help="serving/dense27b/sampled: also report in-situ device time per kernel class")
    ap.add_argument("--vocab", type=int, default=4096, help="profile_cycle: vocabulary")
    ap.add_argument("--attn", default="auto", choices=["auto", "mma", "pipe"],
                    help="attention kernel of the engine (df_config.attn_kernel)")
    ap.add_argument("--sampling", default="0.8,0.95", help="sampled: temperature,top_p")
    ap.add_argument("--new", type=int, default=1024, help="serving/dense27b: new tokens per sequence")
    ap.add_argument("--blocks", default="8,16")
    ap.add_argument("--block-range", default="", help="serving/dense27b: b_min,b_max for df_set_block_range")
    ap.add_argument("--ctx", default="1024,4096,16384,32768")
    ap.add_argument("--batch", default="1,4,16,32")
    ap.add_argument("--reduced", action="store_true", help="drafter: 1 drafter layer, vocab 4096")
    ap.add_argument("--page-tokens", type=int, default=16, help="drafter/serving/dense27b: tokens per KV page")
    ap.add_argument("--M", type=int, default=16)
    ap.add_argument("--N", type=int, default=24576)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--token-tile", type=int, default=0)
    a = ap.parse_args()
    build.build()
    if a.op == "serving":
        serving(a)
        return
    if a.op == "dense27b":
        dense27b(a)
        return
    if a.op == "sampled":
        sampled(a)
        return
    if a.op == "attention":
        attention(a)
        return
    if a.op == "offpath":
        offpath(a)
        return
    if a.op == "profile_cycle":
        a.ctx = int(a.ctx.split(",")[0])
        a.batch = int(a.batch.split(",")[0])
        profile_cycle(a)
        return
    if a.op == "ar_proxy":
        ar_proxy(a)
        return
    if a.op == "drafter":
        a.iters = min(a.iters, 5) if a.iters != 20 else 5
        drafter(a)
        return
    g = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn(a.M, a.K, device="cuda", generator=g).to(torch.bfloat16)
    nw = max(1, min(4, int(512e6 // (a.N * a.K * 2)) + 1))
    ws = [(torch.randn(a.N, a.K, device="cuda", generator=g) * 0.02).to(torch.bfloat16) for _ in range(nw)]

    if a.op == "gemm":
        for i in range(a.warmup):
            dfl.bench_gemm_bf16(x, ws[i % nw], iters=1, splits=a.splits, token_tile=a.token_tile)
        us = sum(dfl.bench_gemm_bf16(x, ws[i % nw], iters=a.iters, splits=a.splits, token_tile=a.token_tile)
                 for i in range(nw)) / nw
        out_b = 4 * a.M * a.N
    else:
        for i in range(a.warmup):
            dfl.lmhead_argmax_bf16(x, ws[i % nw])
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(a.iters):
            dfl.lmhead_argmax_bf16(x, ws[i % nw])
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1000.0 / a.iters
        out_b = 8 * a.M
    algo = 2 * a.N * a.K + 2 * a.M * a.K + out_b
    print(json.dumps({"op": a.op, "M": a.M, "N": a.N, "K": a.K, "splits": a.splits, "token_tile": a.token_tile,
                      "us_per_launch": us, "algorithmic_bytes": algo, "GB/s": algo / (us * 1e-6) / 1e9}))


if __name__ == "__main__":
    main()
