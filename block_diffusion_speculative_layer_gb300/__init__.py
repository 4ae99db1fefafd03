"""Python binding of the GB300 DFlash draft-and-verify engine (libdflash.so).

Argument marshalling only: every step of the cycle runs in the library's
CUDA kernels.  PyTorch provides device memory and the stream.  There is no
CPU path; if the library has not been built, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Iterable, List, Optional, Sequence, Tuple, Union

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libdflash.so")

DF_OK, DF_EINVAL, DF_ENOMEM, DF_ECUDA, DF_ETIMEOUT, DF_ESTATE = range(6)
DF_FP32, DF_BF16 = 0, 1
DF_DBG_TAPS, DF_DBG_LOGITS, DF_DBG_DRAFT_LOGITS, DF_DBG_DRAFT_HIDDEN, DF_DBG_CTX, DF_DBG_HIDDEN = 1, 2, 3, 4, 5, 6
DF_DBG_TARGET_LAYERS, DF_DBG_DRAFT_LAYERS = 7, 8
DF_ATTN_AUTO, DF_ATTN_MMA, DF_ATTN_PIPE = 0, 1, 2
STATUS_NAMES = {0: "DF_OK", 1: "DF_EINVAL", 2: "DF_ENOMEM", 3: "DF_ECUDA", 4: "DF_ETIMEOUT", 5: "DF_ESTATE"}

EXPORTED = [
    "df_default_feat_layers", "df_num_weights", "df_weight_info", "df_init", "df_prefill", "df_draft_block",
    "df_verify_accept", "df_generate", "df_greedy_reference", "df_reset_seq", "df_get_stats", "df_reset_stats",
    "df_seq_info", "df_destroy", "df_last_error", "df_debug_enable", "df_debug_read", "df_debug_weight_ptr",
    "df_op_gemm_bf16", "df_op_lmhead_argmax_bf16", "df_profile_enable", "df_profile_read",
    "df_op_bench_gemm_bf16", "df_op_gemm_bf16_noalloc", "df_bench_drafter_step",
    "df_generate_sampled", "df_philox4x32_10", "df_op_philox_uniforms", "df_op_sampling_probs",
    "df_op_sample_draw", "df_op_accept_sampled", "df_set_block_range", "df_block_size_for",
    "df_generate_accept_hist", "df_debug_wait_probe", "df_op_attention_bf16",
]


class DfError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class DfConfig(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("d_ffn", ctypes.c_int32),
        ("vocab", ctypes.c_int32), ("draft_layers", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("feat_layers", ctypes.c_int32 * 5), ("max_batch", ctypes.c_int32), ("max_ctx", ctypes.c_int32),
        ("page_tokens", ctypes.c_int32), ("dtype", ctypes.c_int32), ("mask_token_id", ctypes.c_int32),
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("attn_kernel", ctypes.c_int32),
    ]


class DfStats(ctypes.Structure):
    _fields_ = [
        ("cycles", ctypes.c_int64), ("accepted_drafts", ctypes.c_int64), ("emitted_tokens", ctypes.c_int64),
        ("accept_hist", ctypes.c_int64 * 65), ("draft_us", ctypes.c_double), ("verify_us", ctypes.c_double),
        ("prefill_us", ctypes.c_double), ("kernel_launches", ctypes.c_int64),
        ("h2d_bytes", ctypes.c_int64), ("d2h_bytes", ctypes.c_int64), ("block_hist", ctypes.c_int64 * 33),
    ]

    def as_dict(self) -> dict:
        return {
            "cycles": self.cycles, "accepted_drafts": self.accepted_drafts, "emitted_tokens": self.emitted_tokens,
            "accept_hist": list(self.accept_hist), "draft_us": self.draft_us, "verify_us": self.verify_us,
            "prefill_us": self.prefill_us, "kernel_launches": self.kernel_launches,
            "h2d_bytes": self.h2d_bytes, "d2h_bytes": self.d2h_bytes, "block_hist": list(self.block_hist),
        }


class DfKernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64), ("total_us", ctypes.c_double),
                ("bytes", ctypes.c_double), ("flops", ctypes.c_double)]


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int32
_IP = ctypes.POINTER(ctypes.c_int32)


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libdflash.so is missing ({LIB_PATH}); build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    L.df_default_feat_layers.argtypes = [_I, _IP]
    L.df_num_weights.argtypes = [ctypes.POINTER(DfConfig)]
    L.df_num_weights.restype = _I
    L.df_weight_info.argtypes = [ctypes.POINTER(DfConfig), _I, ctypes.c_char_p, _IP, ctypes.POINTER(ctypes.c_int64)]
    L.df_init.argtypes = [ctypes.POINTER(DfConfig), ctypes.POINTER(_P), _I, _P, ctypes.POINTER(_P)]
    L.df_prefill.argtypes = [_P, _I, _IP, _I, _IP]
    L.df_draft_block.argtypes = [_P, _IP, _I, _IP]
    L.df_verify_accept.argtypes = [_P, _IP, _I, _IP, _IP, _IP]
    L.df_generate.argtypes = [_P, _IP, _IP, _I, _I, _IP, ctypes.POINTER(DfStats)]
    L.df_greedy_reference.argtypes = [_P, _IP, _IP, _I, _I, _IP]
    L.df_reset_seq.argtypes = [_P, _I]
    L.df_get_stats.argtypes = [_P, ctypes.POINTER(DfStats)]
    L.df_reset_stats.argtypes = [_P]
    L.df_seq_info.argtypes = [_P, _I, _IP, _IP]
    L.df_destroy.argtypes = [_P]
    L.df_destroy.restype = None
    L.df_last_error.argtypes = [_P]
    L.df_last_error.restype = ctypes.c_char_p
    L.df_debug_enable.argtypes = [_P, _I]
    L.df_debug_read.argtypes = [_P, _I, ctypes.POINTER(ctypes.c_float), ctypes.c_int64, _IP]
    L.df_debug_weight_ptr.argtypes = [_P, _I, ctypes.POINTER(ctypes.c_uint64)]
    L.df_op_gemm_bf16.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _P]
    L.df_op_lmhead_argmax_bf16.argtypes = [_P, _P, _P, _I, _I, _I, _P]
    L.df_bench_drafter_step.argtypes = [_P, _I, _I, ctypes.POINTER(ctypes.c_float), _I, _I,
                                         ctypes.POINTER(ctypes.c_double)]
    L.df_op_gemm_bf16_noalloc.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _P]
    L.df_op_bench_gemm_bf16.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, ctypes.POINTER(ctypes.c_float)]
    L.df_profile_enable.argtypes = [_P, _I]
    L.df_profile_read.argtypes = [_P, ctypes.POINTER(DfKernelStat), _I, _IP]
    _F = ctypes.c_float
    L.df_generate_sampled.argtypes = [_P, _IP, _IP, _I, _I, _F, _F, ctypes.c_uint64, _IP, ctypes.POINTER(DfStats)]
    _U32P = ctypes.POINTER(ctypes.c_uint32)
    L.df_philox4x32_10.argtypes = [_U32P, _U32P, _U32P]
    L.df_op_philox_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64, _I, _P, _P]
    L.df_op_sampling_probs.argtypes = [_P, _I, _I, _F, _F, _P, _P, _P]
    L.df_op_sample_draw.argtypes = [_P, _I, _I, _F, _F, _P, _P, _P, _P]
    L.df_op_accept_sampled.argtypes = [_P, _P, _P, _I, _I, _I, _F, _F, _P, _P, _P, _P, _P]
    L.df_set_block_range.argtypes = [_P, _I, _I]
    L.df_generate_accept_hist.argtypes = [_P, _I, ctypes.POINTER(ctypes.c_int64)]
    L.df_debug_wait_probe.argtypes = [_P]
    L.df_op_attention_bf16.argtypes = [_P, _P, _P, _I, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P]
    L.df_block_size_for.argtypes = [ctypes.c_double, _I, _I]
    L.df_block_size_for.restype = _I
    for name in EXPORTED:
        fn = getattr(L, name)
        if fn.restype is ctypes.c_int:  # default restype: the df_status enum
            fn.restype = ctypes.c_int
    _lib = L
    return L


def _ip(a: np.ndarray):
    return a.ctypes.data_as(_IP)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def default_feat_layers(n_layers: int) -> List[int]:
    out = (ctypes.c_int32 * 5)()
    st = lib().df_default_feat_layers(n_layers, out)
    if st != DF_OK:
        raise DfError(st, f"no feature layers for {n_layers} layers")
    return list(out)


def make_config(shape, max_batch: int, max_ctx: int, page_tokens: int = 16,
                feat_layers: Optional[Sequence[int]] = None, attn_kernel: int = DF_ATTN_AUTO) -> DfConfig:
    c = DfConfig()
    c.n_layers, c.d_model, c.n_q_heads = shape.n_layers, shape.d_model, shape.n_q_heads
    c.n_kv_heads, c.head_dim, c.d_ffn, c.vocab = shape.n_kv_heads, shape.head_dim, shape.d_ffn, shape.vocab
    c.draft_layers, c.block_size = shape.draft_layers, shape.block_size
    fl = list(feat_layers) if feat_layers is not None else default_feat_layers(shape.n_layers)
    for i in range(5):
        c.feat_layers[i] = fl[i]
    c.max_batch, c.max_ctx, c.page_tokens = max_batch, max_ctx, page_tokens
    c.dtype = DF_BF16 if shape.dtype == "bf16" else DF_FP32
    c.mask_token_id = shape.vocab - 1
    c.rms_eps, c.rope_theta = shape.rms_eps, shape.rope_theta
    c.attn_kernel = attn_kernel
    return c


def weight_info(cfg: DfConfig) -> List[Tuple[str, Tuple[int, ...]]]:
    L = lib()
    n = L.df_num_weights(ctypes.byref(cfg))
    out = []
    name = ctypes.create_string_buffer(32)
    nd = ctypes.c_int32()
    shp = (ctypes.c_int64 * 2)()
    for i in range(n):
        st = L.df_weight_info(ctypes.byref(cfg), i, name, ctypes.byref(nd), shp)
        if st != DF_OK:
            raise DfError(st, "df_weight_info")
        out.append((name.value.decode(), tuple(shp[: nd.value])))
    return out


def _to_device(arr, torch):
    if isinstance(arr, torch.Tensor):
        return arr.contiguous().cuda()
    a = np.ascontiguousarray(arr)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


class Engine:
    """One DFlash engine (target + drafter) on the current CUDA device."""

    def __init__(self, shape, weights: Union[Dict[str, np.ndarray], Iterable[Tuple[str, np.ndarray]]],
                 max_batch: int = 1, max_ctx: int = 1024, page_tokens: int = 16,
                 feat_layers: Optional[Sequence[int]] = None, stream=None, attn_kernel: int = DF_ATTN_AUTO):
        import torch
        self.L = lib()
        self.shape = shape
        self.cfg = make_config(shape, max_batch, max_ctx, page_tokens, feat_layers, attn_kernel)
        self.B = shape.block_size
        self.V = shape.vocab
        self.d = shape.d_model
        specs = weight_info(self.cfg)
        items = weights.items() if isinstance(weights, dict) else weights
        dev = {}
        for name, arr in items:
            dev[name] = _to_device(arr, torch)
        missing = [n for n, _ in specs if n not in dev]
        if missing:
            raise ValueError(f"missing weights: {missing[:5]}")
        for n, shp in specs:
            if tuple(dev[n].shape) != shp:
                raise ValueError(f"weight {n}: shape {tuple(dev[n].shape)} != {shp}")
        ptrs = (_P * len(specs))(*[dev[n].data_ptr() for n, _ in specs])
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        h = _P()
        torch.cuda.synchronize()
        st = self.L.df_init(ctypes.byref(self.cfg), ptrs, len(specs), _P(self.stream.cuda_stream), ctypes.byref(h))
        del dev
        if st != DF_OK:
            raise DfError(st, "df_init failed (shape, memory or device)")
        self.h = h

    # -------------------------------------------------------------- helpers
    def _check(self, st: int, what: str):
        if st != DF_OK:
            msg = self.L.df_last_error(self.h)
            raise DfError(st, f"{what}: {msg.decode() if msg else ''}")

    def close(self):
        if getattr(self, "h", None):
            self.L.df_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # -------------------------------------------------------------- cycle
    def prefill(self, seq: int, prompt: Sequence[int]) -> int:
        p = _i32(prompt)
        bonus = ctypes.c_int32()
        self._check(self.L.df_prefill(self.h, seq, _ip(p), len(p), ctypes.byref(bonus)), "df_prefill")
        return bonus.value

    def draft_block(self, seqs: Sequence[int]) -> np.ndarray:
        s = _i32(seqs)
        out = np.zeros((len(s), self.B - 1), np.int32)
        self._check(self.L.df_draft_block(self.h, _ip(s), len(s), _ip(out)), "df_draft_block")
        return out

    def verify_accept(self, seqs: Sequence[int], drafts: Optional[np.ndarray] = None):
        s = _i32(seqs)
        acc = np.zeros((len(s), self.B), np.int32)
        n = np.zeros(len(s), np.int32)
        dp = None
        keep = None  # holds the draft buffer alive across the call
        if drafts is not None:
            keep = _i32(drafts).reshape(len(s), self.B - 1)
            dp = _ip(keep)
        self._check(self.L.df_verify_accept(self.h, _ip(s), len(s), dp, _ip(acc), _ip(n)), "df_verify_accept")
        return acc, n

    def generate(self, prompts: Sequence[Sequence[int]], n_new: int):
        lens = _i32([len(p) for p in prompts])
        flat = _i32(np.concatenate([_i32(p) for p in prompts]))
        out = np.zeros((len(prompts), n_new), np.int32)
        stats = DfStats()
        self._check(self.L.df_generate(self.h, _ip(flat), _ip(lens), len(prompts), n_new, _ip(out),
                                       ctypes.byref(stats)), "df_generate")
        return out, stats.as_dict()

    def generate_sampled(self, prompts: Sequence[Sequence[int]], n_new: int, temperature: float = 1.0,
                         top_p: float = 1.0, seed: int = 0):
        """Speculative sampling: drafts drawn from the drafter, the rejection
        test against the target; sequence i uses Philox stream i of `seed`."""
        lens = _i32([len(p) for p in prompts])
        flat = _i32(np.concatenate([_i32(p) for p in prompts]))
        out = np.zeros((len(prompts), n_new), np.int32)
        stats = DfStats()
        self._check(self.L.df_generate_sampled(self.h, _ip(flat), _ip(lens), len(prompts), n_new, float(temperature),
                                               float(top_p), int(seed), _ip(out), ctypes.byref(stats)),
                    "df_generate_sampled")
        return out, stats.as_dict()

    def accept_hist_per_seq(self, nseq: int) -> np.ndarray:
        """[nseq][33]: for each sequence of the last generate call, cycles
        that kept k drafts (k >= 32 at 32), over the cycles that emitted its tokens."""
        out = np.zeros((nseq, 33), np.int64)
        for i in range(nseq):
            self._check(self.L.df_generate_accept_hist(self.h, i, out[i].ctypes.data_as(ctypes.POINTER(ctypes.c_int64))),
                        "df_generate_accept_hist")
        return out

    def set_block_range(self, b_min: int, b_max: int):
        """Block sizes df_generate may use: fixed when equal, else chosen per
        group of cycles from the tokens per cycle seen so far."""
        self._check(self.L.df_set_block_range(self.h, int(b_min), int(b_max)), "df_set_block_range")

    def greedy_reference(self, prompts: Sequence[Sequence[int]], n_new: int) -> np.ndarray:
        lens = _i32([len(p) for p in prompts])
        flat = _i32(np.concatenate([_i32(p) for p in prompts]))
        out = np.zeros((len(prompts), n_new), np.int32)
        self._check(self.L.df_greedy_reference(self.h, _ip(flat), _ip(lens), len(prompts), n_new, _ip(out)),
                    "df_greedy_reference")
        return out

    def reset_seq(self, seq: int):
        self._check(self.L.df_reset_seq(self.h, seq), "df_reset_seq")

    def seq_info(self, seq: int) -> Tuple[int, int]:
        ln, b = ctypes.c_int32(), ctypes.c_int32()
        self._check(self.L.df_seq_info(self.h, seq, ctypes.byref(ln), ctypes.byref(b)), "df_seq_info")
        return ln.value, b.value

    def stats(self) -> dict:
        s = DfStats()
        self._check(self.L.df_get_stats(self.h, ctypes.byref(s)), "df_get_stats")
        return s.as_dict()

    def reset_stats(self):
        self._check(self.L.df_reset_stats(self.h), "df_reset_stats")

    # -------------------------------------------------------------- inspection
    def debug(self, on: bool = True):
        self._check(self.L.df_debug_enable(self.h, 1 if on else 0), "df_debug_enable")

    def debug_read(self, what: int) -> np.ndarray:
        cols = {DF_DBG_TAPS: 5 * self.d, DF_DBG_LOGITS: self.V, DF_DBG_DRAFT_LOGITS: self.V,
                DF_DBG_DRAFT_HIDDEN: self.d, DF_DBG_CTX: self.d, DF_DBG_HIDDEN: self.d,
                DF_DBG_TARGET_LAYERS: self.d, DF_DBG_DRAFT_LAYERS: self.d}[what]
        layers = {DF_DBG_TARGET_LAYERS: self.shape.n_layers + 1, DF_DBG_DRAFT_LAYERS: self.shape.draft_layers + 1}
        cap = max(512, self.cfg.max_batch * self.B) * cols * layers.get(what, 1)
        buf = np.zeros(cap, np.float32)
        rows = ctypes.c_int32()
        self._check(self.L.df_debug_read(self.h, what, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), cap,
                                         ctypes.byref(rows)), "df_debug_read")
        out = buf[: rows.value * cols].reshape(rows.value, cols)
        if what in layers:
            return out.reshape(layers[what], rows.value // layers[what], cols)
        return out

    def profile(self, on: bool = True, in_situ: bool = False):
        """Kernel-class timing: events around every launch (serialised), or
        with in_situ=True device-timer stamps inside the captured cycles."""
        mode = (2 if in_situ else 1) if on else 0
        self._check(self.L.df_profile_enable(self.h, mode), "df_profile_enable")

    def profile_read(self) -> Dict[str, dict]:
        """Per kernel class: launches, device microseconds, algorithmic bytes and flops (then cleared)."""
        arr = (DfKernelStat * 8)()
        n = ctypes.c_int32()
        self._check(self.L.df_profile_read(self.h, arr, 8, ctypes.byref(n)), "df_profile_read")
        return {arr[i].name.decode(): {"launches": arr[i].launches, "us": arr[i].total_us, "bytes": arr[i].bytes,
                                       "flops": arr[i].flops} for i in range(n.value)}

    def bench_drafter_step(self, nseq: int, ctx_len: int, taps: np.ndarray, iters: int = 5) -> Dict[str, float]:
        """Device microseconds per drafter step: fusion, injection, block attention, LM-head argmax."""
        t = np.ascontiguousarray(taps, dtype=np.float32).reshape(-1, 5 * self.d)
        out = (ctypes.c_double * 6)()
        self._check(self.L.df_bench_drafter_step(self.h, nseq, ctx_len,
                                                 t.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), t.shape[0],
                                                 iters, out), "df_bench_drafter_step")
        return {"fuse_us": out[0], "inject_us": out[1], "block_attention_us": out[2], "lm_head_us": out[3],
                "layer_gemms_us": out[4], "drafter_pass_us": out[5]}

    def wait_probe(self):
        """Run the failure-detection check (df_debug_wait_probe): raises
        DfError with DF_ETIMEOUT, and the handle is failed afterwards."""
        self._check(self.L.df_debug_wait_probe(self.h), "df_debug_wait_probe")

    def weight_ptr(self, which: int) -> int:
        a = ctypes.c_uint64()
        self._check(self.L.df_debug_weight_ptr(self.h, which, ctypes.byref(a)), "df_debug_weight_ptr")
        return a.value


# ------------------------------------------------------------------ single ops
def gemm_bf16(x, w, splits: int = 0, token_tile: int = 0, stream=None):
    """y = x @ w.T (bf16 in, fp32 out) on the tcgen05 GEMM.  x: [M, K], w: [N, K] (torch, cuda)."""
    import torch
    assert x.dtype == torch.bfloat16 and w.dtype == torch.bfloat16 and x.is_cuda and w.is_cuda
    M, K = x.shape
    N = w.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = lib().df_op_gemm_bf16(_P(x.data_ptr()), _P(w.data_ptr()), _P(y.data_ptr()), M, N, K, splits, token_tile,
                               _P(s.cuda_stream))
    if st != DF_OK:
        raise DfError(st, "df_op_gemm_bf16")
    return y


def bench_gemm_bf16(x, w, iters: int = 20, splits: int = 0, token_tile: int = 0, stream=None) -> float:
    """Mean device microseconds of the tcgen05 GEMM over `iters` back-to-back launches."""
    import torch
    M, K = x.shape
    N = w.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    us = ctypes.c_float()
    st = lib().df_op_bench_gemm_bf16(_P(x.data_ptr()), _P(w.data_ptr()), _P(y.data_ptr()), M, N, K, splits,
                                     token_tile, iters, _P(s.cuda_stream), ctypes.byref(us))
    if st != DF_OK:
        raise DfError(st, "df_op_bench_gemm_bf16")
    return us.value


def attention_bf16(q, cache, page_table, row_pos, row_seq, nseq: int, rows_per_seq: int, n_kv_heads: int,
                   causal: bool, max_len: int, blk=None, kernel: int = DF_ATTN_PIPE, out=None, err=None,
                   stream=None, cluster_ctas: int = 0, check_rows: bool = True):
    """One attention launch on torch CUDA tensors (df_op_attention_bf16).
    q: [rows, Hq*128] bf16; cache: [n_pages, 2, Hkv, 16, 128] bf16; page_table:
    [slots, pt_stride] int32; row_pos, row_seq: [rows] int32; blk: [2, Hkv,
    rows_cap, 128] bf16 for the drafter's block attention.  Returns (out, err).
    check_rows=False skips the host check that row_seq indexes page_table
    (that check copies row_seq to the host and so waits for the stream)."""
    import torch
    assert q.dtype == torch.bfloat16 and cache.dtype == torch.bfloat16 and q.is_cuda and cache.is_cuda
    rows = q.shape[0]
    Hq = q.shape[1] // 128
    assert rows == nseq * rows_per_seq and row_pos.numel() == rows and row_seq.numel() == rows
    assert page_table.dtype == torch.int32 and row_pos.dtype == torch.int32 and row_seq.dtype == torch.int32
    if check_rows:
        seq_cpu = row_seq.cpu()
        assert int(seq_cpu.min()) >= 0 and int(seq_cpu.max()) < page_table.shape[0], "row_seq must index page_table"
    out = torch.empty_like(q) if out is None else out
    err = _err_word(q.device) if err is None else err
    blk_p = _P(blk.data_ptr()) if blk is not None else None
    rows_cap = blk.shape[2] if blk is not None else 0
    st = lib().df_op_attention_bf16(_P(q.data_ptr()), _P(out.data_ptr()), _P(cache.data_ptr()), cache.shape[0],
                                    _P(page_table.data_ptr()), page_table.shape[1], _P(row_pos.data_ptr()),
                                    _P(row_seq.data_ptr()), blk_p, rows_cap, nseq, rows_per_seq, Hq, n_kv_heads,
                                    1 if causal else 0, max_len, kernel, cluster_ctas, _P(err.data_ptr()),
                                    _stream(stream))
    if st != DF_OK:
        raise DfError(st, "df_op_attention_bf16")
    return out, err


def lmhead_argmax_bf16(x, w, stream=None):
    """ids[m] = argmax_v x[m] . w[v] (fp32 logits, lowest index on ties)."""
    import torch
    M, K = x.shape
    V = w.shape[0]
    ids = torch.empty(M, dtype=torch.int32, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = lib().df_op_lmhead_argmax_bf16(_P(x.data_ptr()), _P(w.data_ptr()), _P(ids.data_ptr()), M, V, K,
                                        _P(s.cuda_stream))
    if st != DF_OK:
        raise DfError(st, "df_op_lmhead_argmax_bf16")
    return ids


# ------------------------------------------------------------------ sampling ops
def philox4x32_10(ctr: Sequence[int], key: Sequence[int]) -> List[int]:
    """The library's Philox4x32-10 block function, evaluated on the host."""
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    o = (ctypes.c_uint32 * 4)()
    st = lib().df_philox4x32_10(c, k, o)
    if st != DF_OK:
        raise DfError(st, "df_philox4x32_10")
    return list(o)


def _stream(stream):
    import torch
    return _P((stream if stream is not None else torch.cuda.current_stream()).cuda_stream)


def _err_word(device):
    import torch
    return torch.zeros(1, dtype=torch.int32, device=device)


def _check_err(err, what: str):
    e = int(err.item())
    if e:
        raise DfError(DF_ECUDA, f"{what}: device error bits {e}")


def philox_uniforms(seed: int, stream_id: int, offset: int, n: int, device="cuda", stream=None):
    """Uniforms offset .. offset + n - 1 of (seed, stream_id), generated on the GPU (float32 tensor)."""
    import torch
    u = torch.empty(max(n, 1), dtype=torch.float32, device=device)
    st = lib().df_op_philox_uniforms(int(seed), int(stream_id), int(offset), n, _P(u.data_ptr()), _stream(stream))
    if st != DF_OK:
        raise DfError(st, "df_op_philox_uniforms")
    return u[:n]


def sampling_probs(logits, temperature: float, top_p: float = 1.0, stream=None):
    """Rows of sampling probabilities of fp32 logits [rows, V] (torch, cuda)."""
    import torch
    assert logits.dtype == torch.float32 and logits.is_cuda and logits.dim() == 2
    x = logits.contiguous()
    rows, V = x.shape
    probs = torch.empty_like(x)
    err = _err_word(x.device)
    st = lib().df_op_sampling_probs(_P(x.data_ptr()), rows, V, float(temperature), float(top_p), _P(probs.data_ptr()),
                                    _P(err.data_ptr()), _stream(stream))
    if st != DF_OK:
        raise DfError(st, "df_op_sampling_probs")
    _check_err(err, "df_op_sampling_probs")
    return probs


def sample_draw(logits, temperature: float, top_p: float, u, stream=None):
    """One inverse-CDF draw per row of fp32 logits [rows, V] with uniforms u [rows]."""
    import torch
    x = logits.contiguous()
    uu = u.to(device=x.device, dtype=torch.float32).contiguous()
    rows, V = x.shape
    assert uu.numel() == rows
    idx = torch.empty(rows, dtype=torch.int32, device=x.device)
    err = _err_word(x.device)
    st = lib().df_op_sample_draw(_P(x.data_ptr()), rows, V, float(temperature), float(top_p), _P(uu.data_ptr()),
                                 _P(idx.data_ptr()), _P(err.data_ptr()), _stream(stream))
    if st != DF_OK:
        raise DfError(st, "df_op_sample_draw")
    _check_err(err, "df_op_sample_draw")
    return idx


def accept_sampled(drafts, q_logits, p_logits, temperature: float, top_p: float, u, stream=None):
    """Speculative-sampling test of nseq blocks: drafts [nseq, B-1], q_logits
    [nseq, B-1, V], p_logits [nseq, B, V], u [nseq, B] -> (k [nseq], token [nseq])."""
    import torch
    p = p_logits.contiguous()
    nseq, B, V = p.shape
    q = q_logits.contiguous()
    d = drafts.to(device=p.device, dtype=torch.int32).contiguous()
    uu = u.to(device=p.device, dtype=torch.float32).contiguous()
    assert q.shape == (nseq, B - 1, V) and d.shape == (nseq, B - 1) and uu.shape == (nseq, B)
    k = torch.empty(nseq, dtype=torch.int32, device=p.device)
    tok = torch.empty(nseq, dtype=torch.int32, device=p.device)
    err = _err_word(p.device)
    st = lib().df_op_accept_sampled(_P(d.data_ptr()), _P(q.data_ptr()), _P(p.data_ptr()), nseq, B, V,
                                    float(temperature), float(top_p), _P(uu.data_ptr()), _P(k.data_ptr()),
                                    _P(tok.data_ptr()), _P(err.data_ptr()), _stream(stream))
    if st != DF_OK:
        raise DfError(st, "df_op_accept_sampled")
    _check_err(err, "df_op_accept_sampled")
    return k, tok


def block_size_for(tokens_per_cycle: float, b_min: int, b_max: int) -> int:
    """The engine's block-size rule (df_block_size_for)."""
    b = lib().df_block_size_for(float(tokens_per_cycle), int(b_min), int(b_max))
    if b < 0:
        raise DfError(DF_EINVAL, "df_block_size_for: bad arguments")
    return b
