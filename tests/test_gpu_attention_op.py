"""One attention launch through df_op_attention_bf16 against the oracle.

Source: [ARCH] "DFlash 的架构密码", 第三层 Block Diffusion and 稀疏注意力训练:
the target's verify rows attend causally over the cache; the drafter's block
rows attend over the injected context before their anchor and, in both
directions, over their own block; nothing crosses sequences.

Random bf16 queries, keys and values in a paged cache with shuffled pages
(and, in one test, pages in runs of consecutive ids, as the engine's
allocator hands them out), ragged context lengths; the reference is the oracle's attention (float64) on
the same bf16 values, gathered and masked by the rule above.  Both kernels
(mma.sync cluster and pipelined tcgen05), query-head groups of 4, 5 and 8.
A row computed alone must equal the same row computed inside its block, bit
for bit (what keeps verification and greedy decoding identical).  The
pipelined kernel runs in clusters of 2, 4 and 16 CTAs (the chunk split, and
so the rounding, follows the cluster size).
"""
import math

import numpy as np
import pytest

from oracle import dflash_oracle as O

import _teacher as T

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

PT, HD = 16, 128


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__ as g
    g.build()
    import block_diffusion_speculative_layer_gb300 as m
    return m


def bf(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).cuda()


def make_case(seed, lens, R, Hq, Hkv, causal, layout="shuffled"):
    """Cache holding each sequence's positions 0..len-1 (plus its block rows for
    the causal case), queries of R rows per sequence.  Pages: "shuffled" (a
    random permutation of the pool), or "runs" (each sequence takes
    consecutive page ids, the last sequence ending at the pool's last page,
    and about a quarter of its 4-page chunks are shuffled inside)."""
    g = np.random.default_rng(seed)
    nseq = len(lens)
    need = [L + (R if causal else 0) for L in lens]
    pt_stride = max((n + PT - 1) // PT for n in need) + 1
    n_pages = sum((n + PT - 1) // PT for n in need) + 3
    perm = g.permutation(n_pages) if layout == "shuffled" else np.arange(3, n_pages)
    table = np.full((nseq, pt_stride), -1, np.int32)
    cache = g.standard_normal((n_pages, 2, Hkv, PT, HD)).astype(np.float32)
    k_seq, v_seq = [], []
    used = 0
    for i, n in enumerate(need):
        npg = (n + PT - 1) // PT
        ids = perm[used:used + npg].copy()
        if layout == "runs":
            for c0 in range(0, npg - 3, 4):
                if g.random() < 0.25:
                    g.shuffle(ids[c0:c0 + 4])
        table[i, :npg] = ids
        used += npg
        ks = cache[table[i, :npg], 0].transpose(0, 2, 1, 3).reshape(npg * PT, Hkv, HD)[:n]
        vs = cache[table[i, :npg], 1].transpose(0, 2, 1, 3).reshape(npg * PT, Hkv, HD)[:n]
        k_seq.append(ks)
        v_seq.append(vs)
    q = g.standard_normal((nseq * R, Hq * HD)).astype(np.float32)
    blk = g.standard_normal((2, Hkv, nseq * R, HD)).astype(np.float32)
    pos = np.concatenate([np.arange(L, L + R) for L in lens]).astype(np.int32)
    seq = np.repeat(np.arange(nseq), R).astype(np.int32)
    return dict(q=q, cache=cache, table=table, k=k_seq, v=v_seq, blk=blk, pos=pos, seq=seq, pt_stride=pt_stride)


def rb(x):
    """Round float32 to bf16 values (the kernels' inputs), as float64."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def reference(c, lens, R, Hq, Hkv, causal):
    out = []
    for i, L in enumerate(lens):
        qi = rb(c["q"][i * R:(i + 1) * R]).reshape(R, Hq, HD)
        if causal:
            keys, vals = rb(c["k"][i]), rb(c["v"][i])
            vis = np.arange(L + R)[None, :] <= np.arange(L, L + R)[:, None]
        else:
            kb = rb(c["blk"][0][:, i * R:(i + 1) * R].transpose(1, 0, 2))
            vb = rb(c["blk"][1][:, i * R:(i + 1) * R].transpose(1, 0, 2))
            keys = np.concatenate([rb(c["k"][i]), kb])
            vals = np.concatenate([rb(c["v"][i]), vb])
            vis = np.ones((R, L + R), bool)
        out.append(O.attention(qi, keys, vals, vis).reshape(R, Hq * HD))
    return np.concatenate(out)


KERNELS = {"mma": (1, 0), "pipe2": (2, 2), "pipe4": (2, 4), "pipe16": (2, 16)}  # (df kernel, CTAs per cluster)


def run(dfl, c, lens, R, Hkv, causal, kernel):
    k, cla = KERNELS[kernel]
    max_len = max(L + (R if causal else 0) for L in lens)
    out, err = dfl.attention_bf16(bf(c["q"]), bf(c["cache"]), torch.from_numpy(c["table"]).cuda(),
                                  torch.from_numpy(c["pos"]).cuda(), torch.from_numpy(c["seq"]).cuda(), len(lens), R,
                                  Hkv, causal, max_len, blk=None if causal else bf(c["blk"]), kernel=k,
                                  cluster_ctas=cla)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.float().cpu().numpy()


CASES = [(4, 8, [1000, 37, 2048 + 5], 16), (5, 8, [300, 1500], 16), (8, 2, [700, 64], 8), (4, 8, [32768 - 16], 16)]


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "block"])
@pytest.mark.parametrize("G,Hkv,lens,R", CASES, ids=["g4-ragged", "g5", "g8", "g4-32k"])
def test_attention_against_the_oracle(dfl, kernel, causal, G, Hkv, lens, R):
    Hq = G * Hkv
    c = make_case(7 + G + len(lens), lens, R, Hq, Hkv, causal)
    got = run(dfl, c, lens, R, Hkv, causal, kernel)
    ref = reference(c, lens, R, Hq, Hkv, causal)
    assert T.rel_err(got, ref) <= 2e-2
    # each row against its own reference (rows differ in length and scale)
    for r in range(0, got.shape[0], max(1, got.shape[0] // 7)):
        assert T.rel_err(got[r], ref[r]) <= 2e-2, r


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_a_row_alone_equals_the_row_in_its_block(dfl, kernel):
    # causal rows: row j of a 16-row verify block and the same position decoded
    # alone (a 1-row block) give bitwise the same output
    k = kernel
    G, Hkv, R = 4, 8, 16
    lens = [900, 333]
    c = make_case(3, lens, R, G * Hkv, Hkv, True)
    full = run(dfl, c, lens, R, Hkv, True, k)
    for j in (0, 5, 15):
        c1 = dict(c)
        c1["q"] = np.concatenate([c["q"][i * R + j:i * R + j + 1] for i in range(len(lens))])
        c1["pos"] = np.asarray([L + j for L in lens], np.int32)
        c1["seq"] = np.arange(len(lens), dtype=np.int32)
        one = run(dfl, c1, lens, 1, Hkv, True, k)
        for i in range(len(lens)):
            np.testing.assert_array_equal(one[i], full[i * R + j])


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "block"])
def test_pages_in_runs(dfl, kernel, causal):
    # pages in runs of consecutive ids (the engine's allocation): the result
    # matches the oracle and equals, bit for bit, the same cache contents
    # placed by a random permutation of the pool
    G, Hkv, R = 4, 8, 16
    lens = [1000, 37, 2048 + 5, 700]
    c = make_case(11, lens, R, G * Hkv, Hkv, causal, layout="runs")
    full_chunks = sum(1 for i, L in enumerate(lens) for c0 in range(0, (L + PT - 1) // PT - 3, 4)
                      if np.all(np.diff(c["table"][i, c0:c0 + 4]) == 1))
    assert full_chunks >= 20  # most chunks are runs
    got = run(dfl, c, lens, R, Hkv, causal, kernel)
    ref = reference(c, lens, R, G * Hkv, Hkv, causal)
    assert T.rel_err(got, ref) <= 2e-2
    for r in range(0, got.shape[0], 9):
        assert T.rel_err(got[r], ref[r]) <= 2e-2, r
    perm = np.random.default_rng(5).permutation(c["cache"].shape[0])
    moved = dict(c)
    moved["cache"] = np.empty_like(c["cache"])
    moved["cache"][perm] = c["cache"]  # page p's contents now sit in page perm[p]
    moved["table"] = np.where(c["table"] >= 0, perm[np.maximum(c["table"], 0)], -1).astype(np.int32)
    np.testing.assert_array_equal(run(dfl, moved, lens, R, Hkv, causal, kernel), got)
