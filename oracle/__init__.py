"""fp64 CPU oracle for InfLLM v2 block-sparse attention -- TEST INFRASTRUCTURE.

Only `tests/`, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never imports, links or calls it, and shares no code with it.

The arithmetic lives in `infllmv2_oracle.c` (plain loops, double precision);
this module only marshals numpy arrays into it.  Each function documents the
step of the method it restates; the C file cites the passages.

Parity pins (tests/test_oracle_pins.py) tie every function to something other
than itself: exact rational arithmetic for the bf16 rounding and the kernel
means, brute-force sorting for the top-k, a matrix-form dense softmax for the
attention, and planted-block recovery.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "infllmv2_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liborc_infllmv2.so")
_lock = threading.Lock()
_lib = None

P_FIELDS = ("block_size", "kernel_size", "kernel_stride", "topk", "n_init_blocks",
            "n_local_blocks", "dense_len")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, strict IEEE double: no contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            lib.orc_bf16_round.argtypes = [p, i64, p]
            lib.orc_bf16_round.restype = None
            lib.orc_num_threads.restype = ctypes.c_int
            lib.orc_kernel_pool.argtypes = [p, i64, i64, i64, i64, p, i32, i32, p, p, i64]
            lib.orc_block_scores.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, i32, p, p, i64,
                                             i64, p]
            lib.orc_select.argtypes = [p, p, i64, i64, i64, i32, p, p, i64, i64, i64, p, p, p, p]
            lib.orc_attention.argtypes = [p, p, p, p, p, p, p, p, p, i64, i64, i64, i64, i64, i64,
                                          i64, p, ctypes.c_double, p, i64, p, p]
            lib.orc_attention_f64.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64, i64, i64, p,
                                              ctypes.c_double, p, p]
            lib.orc_attention_bwd.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64, i64, i64, p,
                                              ctypes.c_double, p, p, p, p]
            for f in (lib.orc_kernel_pool, lib.orc_block_scores, lib.orc_select, lib.orc_attention,
                      lib.orc_attention_f64, lib.orc_attention_bwd):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _iparams(params: dict) -> np.ndarray:
    return np.array([int(params[f]) for f in P_FIELDS], dtype=np.int32)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def num_threads() -> int:
    return int(_load().orc_num_threads())


def n_kernels(L: int, c: int, s: int) -> int:
    return 0 if L < c else (L - c) // s + 1


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns, nearest with ties to even."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_bf16_round(_ptr(x), x.size, _ptr(out))
    return out


def kernel_pool(k_cache: np.ndarray, kv_len: np.ndarray, c: int, s: int, M_max: int):
    """Semantic kernels: bf16 mean of K over tokens [j*s, j*s+c) for every complete kernel.

    k_cache: uint16 (bf16 bits) [B, H, L_max, d].  Returns (kern bf16 bits
    [B, H, M_max, d], exact fp64 means); entries past each sequence's last
    complete kernel are zero.
    """
    k_cache = _c(k_cache, np.uint16)
    kv_len = _c(kv_len, np.int32)
    B, H, L_max, d = k_cache.shape
    kern = np.zeros((B, H, M_max, d), dtype=np.uint16)
    exact = np.zeros((B, H, M_max, d), dtype=np.float64)
    _check(_load().orc_kernel_pool(_ptr(k_cache), B, H, L_max, d, _ptr(kv_len), c, s, _ptr(kern),
                                   _ptr(exact), M_max), "kernel_pool")
    return kern, exact


def block_scores(q, kern, kv_len, Hkv, params, t_list=None, tree=False, nblk_max=None):
    """Unscaled block scores S [B, Hkv, n_t, nblk_max] (max over overlapping,
    visible kernels and over the heads of a group); -inf past the query's block."""
    q = _c(q, np.uint16)
    kern = _c(kern, np.uint16)
    kv_len = _c(kv_len, np.int32)
    B, Tq, Hq, d = q.shape
    M_max = kern.shape[2]
    t_list = np.arange(Tq, dtype=np.int32) if t_list is None else _c(t_list, np.int32)
    if nblk_max is None:
        nblk_max = (int(kv_len.max()) - 1) // int(params["block_size"]) + 1
    S = np.empty((B, Hkv, len(t_list), nblk_max), dtype=np.float64)
    _check(_load().orc_block_scores(_ptr(q), _ptr(kern), _ptr(kv_len), B, Tq, Hq, Hkv, d, M_max,
                                    int(tree), _ptr(_iparams(params)), _ptr(t_list), len(t_list),
                                    nblk_max, _ptr(S)), "block_scores")
    return S


def select(S, kv_len, Tq, params, t_list=None, tree=False, S_max=None):
    """Top-k selection with forced init/local blocks and the dense switch.

    Returns (idx int32 [B, Hkv, n_t, S_max] ascending, padded -1; counts;
    kth: score of the last kept candidate; nxt: score of the first left out)."""
    S = _c(S, np.float64)
    kv_len = _c(kv_len, np.int32)
    B, Hkv, n_t, nblk_max = S.shape
    t_list = np.arange(Tq, dtype=np.int32) if t_list is None else _c(t_list, np.int32)
    assert len(t_list) == n_t
    if S_max is None:
        S_max = nblk_max
    idx = np.empty((B, Hkv, n_t, S_max), dtype=np.int32)
    counts = np.empty((B, Hkv, n_t), dtype=np.int32)
    kth = np.empty((B, Hkv, n_t), dtype=np.float64)
    nxt = np.empty((B, Hkv, n_t), dtype=np.float64)
    _check(_load().orc_select(_ptr(S), _ptr(kv_len), B, Hkv, Tq, int(tree), _ptr(_iparams(params)),
                              _ptr(t_list), n_t, nblk_max, S_max, _ptr(idx), _ptr(counts), _ptr(kth),
                              _ptr(nxt)), "select")
    return idx, counts, kth, nxt


def attention(q, k_cache, v_cache, kv_len, idx, counts, params, t_list=None, draft_k=None,
              draft_v=None, tree_mask=None, scale=0.0):
    """Exact softmax attention of the listed queries over their selected blocks.

    idx/counts as returned by `select` for the same t_list (idx None: dense
    causal).  Returns (o float64 [B, n_t, Hq, d], lse float64 [B, Hq, n_t])."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    kv_len = _c(kv_len, np.int32)
    B, Tq, Hq, d = q.shape
    Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
    t_list = np.arange(Tq, dtype=np.int32) if t_list is None else _c(t_list, np.int32)
    n_t = len(t_list)
    idx = _c(idx, np.int32)
    counts = _c(counts, np.int32)
    S_max = 0 if idx is None else idx.shape[-1]
    o = np.empty((B, n_t, Hq, d), dtype=np.float64)
    lse = np.empty((B, Hq, n_t), dtype=np.float64)
    _check(_load().orc_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len),
                                 _ptr(_c(draft_k, np.uint16)), _ptr(_c(draft_v, np.uint16)),
                                 _ptr(_c(tree_mask, np.uint64)), _ptr(idx), _ptr(counts), S_max, B,
                                 Tq, Hq, Hkv, d, L_max, _ptr(_iparams(params)), float(scale),
                                 _ptr(t_list), n_t, _ptr(o), _ptr(lse)), "attention")
    return o, lse


def attention_f64(q, k_cache, v_cache, kv_len, idx, counts, params, scale=0.0):
    """Chunk attention like `attention`, on fp64 inputs (for differentiation).
    Returns (o float64 [B, Tq, Hq, d], lse float64 [B, Hq, Tq])."""
    q = _c(q, np.float64)
    k_cache = _c(k_cache, np.float64)
    v_cache = _c(v_cache, np.float64)
    kv_len = _c(kv_len, np.int32)
    B, Tq, Hq, d = q.shape
    Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
    idx = _c(idx, np.int32)
    counts = _c(counts, np.int32)
    S_max = 0 if idx is None else idx.shape[-1]
    o = np.empty((B, Tq, Hq, d), dtype=np.float64)
    lse = np.empty((B, Hq, Tq), dtype=np.float64)
    _check(_load().orc_attention_f64(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(idx),
                                     _ptr(counts), S_max, B, Tq, Hq, Hkv, d, L_max,
                                     _ptr(_iparams(params)), float(scale), _ptr(o), _ptr(lse)),
           "attention_f64")
    return o, lse


def attention_bwd(q, k_cache, v_cache, kv_len, idx, counts, params, dout, scale=0.0):
    """Gradients of sum(dout * o) of `attention_f64` with the selection fixed.
    Returns (dq [B, Tq, Hq, d], dk [B, Hkv, L_max, d], dv [B, Hkv, L_max, d]), float64."""
    q = _c(q, np.float64)
    k_cache = _c(k_cache, np.float64)
    v_cache = _c(v_cache, np.float64)
    dout = _c(dout, np.float64)
    kv_len = _c(kv_len, np.int32)
    B, Tq, Hq, d = q.shape
    Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
    idx = _c(idx, np.int32)
    counts = _c(counts, np.int32)
    S_max = 0 if idx is None else idx.shape[-1]
    dq = np.empty_like(q)
    dk = np.empty_like(k_cache)
    dv = np.empty_like(v_cache)
    _check(_load().orc_attention_bwd(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(idx),
                                     _ptr(counts), S_max, B, Tq, Hq, Hkv, d, L_max,
                                     _ptr(_iparams(params)), float(scale), _ptr(dout), _ptr(dq),
                                     _ptr(dk), _ptr(dv)), "attention_bwd")
    return dq, dk, dv


def run(inputs: dict, w, t_list=None, kern=None):
    """The whole path for workload `w` on the listed queries: kernels, scores,
    selection, attention.  Returns a dict of every intermediate."""
    tree = w.kind == "tree"
    p = w.params()
    M_max = n_kernels(w.L_max, w.kernel_size, w.kernel_stride)
    if kern is None:
        kern, _ = kernel_pool(inputs["k_cache"], inputs["kv_len"], w.kernel_size, w.kernel_stride,
                              M_max)
    S = block_scores(inputs["q"], kern, inputs["kv_len"], w.Hkv, p, t_list=t_list, tree=tree)
    idx, counts, kth, nxt = select(S, inputs["kv_len"], w.Tq, p, t_list=t_list, tree=tree)
    o, lse = attention(inputs["q"], inputs["k_cache"], inputs["v_cache"], inputs["kv_len"], idx,
                       counts, p, t_list=t_list, draft_k=inputs.get("draft_k"),
                       draft_v=inputs.get("draft_v"), tree_mask=inputs.get("tree_mask"))
    return dict(kern=kern, S=S, idx=idx, counts=counts, kth=kth, nxt=nxt, o=o, lse=lse)
