"""Python binding of libinfllmv2.so (include/infllmv2.h), argument marshalling only.

Every function takes CUDA tensors (PyTorch is used for device memory and
streams), passes their device pointers and sizes to the C ABI entry point of
the same name, and raises `InfLLMv2Error` on a non-zero status.  No step of
the method runs here, and there is no fallback: if the library has not been
built, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libinfllmv2.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "infllmv2.h")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
ERR_DEVICE_TIMEOUT = -5
ERR_DEVICE_INDEX = -6
ERR_NOT_IMPLEMENTED = -7

ENTRY_BLOCK_SELECT = 1
ENTRY_SPARSE_ATTN_FWD = 2
ENTRY_DECODE = 3
ENTRY_SPARSE_ATTN_BWD = 4


class InfLLMv2Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class Params(ctypes.Structure):
    """infllmv2_params: block_size, kernel_size, kernel_stride, topk, n_init_blocks,
    n_local_blocks, dense_len, softmax_scale (0 = 1/sqrt(d))."""
    _fields_ = [("block_size", ctypes.c_int32), ("kernel_size", ctypes.c_int32),
                ("kernel_stride", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("n_init_blocks", ctypes.c_int32), ("n_local_blocks", ctypes.c_int32),
                ("dense_len", ctypes.c_int32), ("softmax_scale", ctypes.c_float)]

    @classmethod
    def make(cls, p) -> "Params":
        if isinstance(p, Params):
            return p
        return cls(int(p["block_size"]), int(p["kernel_size"]), int(p["kernel_stride"]),
                   int(p["topk"]), int(p["n_init_blocks"]), int(p["n_local_blocks"]),
                   int(p["dense_len"]), float(p.get("softmax_scale", 0.0)))


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libinfllmv2.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with block_sparse_long_infllm_gb300.build.build()")
    lib = ctypes.CDLL(path)
    p, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    pp = ctypes.POINTER(Params)
    lib.infllmv2_status_string.argtypes = [i32]
    lib.infllmv2_status_string.restype = ctypes.c_char_p
    lib.infllmv2_version.argtypes = []
    lib.infllmv2_sync_status.argtypes = [p]
    lib.infllmv2_selection_capacity.argtypes = [pp, i32]
    lib.infllmv2_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, pp]
    lib.infllmv2_workspace_size.restype = sz
    lib.infllmv2_kernel_pool.argtypes = [p, p, i32, i32, i32, i32, i32, i32, i32, pp, p]
    lib.infllmv2_append.argtypes = [p, p, p, p, p, p, i32, i32, i32, i32, i32, pp, p]
    lib.infllmv2_kernel_pool_varlen.argtypes = [p, p, p, p, i32, i32, i32, i32, i32, i32, pp, p]
    lib.infllmv2_block_select_varlen.argtypes = [p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32, p, p, i32, p,
                                                 sz, pp, p]
    lib.infllmv2_sparse_attn_fwd_varlen.argtypes = [p, p, p, p, p, i32, p, p, i32, i32, i32, i32, i32, i32, i32, p,
                                                    p, pp, p]
    lib.infllmv2_decode_step.argtypes = [p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, p, p, p, p, i32, p, sz,
                                         pp, p]
    lib.infllmv2_block_select.argtypes = [p, p, p, i32, i32, i32, i32, i32, i32, i32, p, p, i32, p, sz,
                                          pp, p]
    lib.infllmv2_sparse_attn_fwd.argtypes = [p, p, p, p, p, i32, p, i32, i32, i32, i32, i32, i32, p, p,
                                             p, sz, pp, p]
    lib.infllmv2_sparse_attn_bwd.argtypes = [p, p, p, p, p, p, p, p, i32, p, i32, i32, i32, i32, i32, i32, p, p,
                                             p, p, sz, pp, p]
    lib.infllmv2_decode.argtypes = [p, p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, p, p, p,
                                    p, i32, p, sz, pp, p]
    lib.infllmv2_decode_noalloc.argtypes = [p, p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, p, p,
                                            p, p, i32, pp, p]
    lib.infllmv2_decode_noalloc.restype = ctypes.c_int
    lib.infllmv2_decode_host.argtypes = [p, p, p, p, p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, p, sz, pp, p]
    lib.infllmv2_decode_host.restype = ctypes.c_int
    lib.infllmv2_host_memory_direct.argtypes = [p]
    lib.infllmv2_host_memory_direct.restype = ctypes.c_int
    lib.infllmv2_profile_enable.argtypes = [i32]
    lib.infllmv2_profile_read.argtypes = [p, i32, p]
    lib.infllmv2_profile_stage_name.argtypes = [i32]
    lib.infllmv2_profile_stage_name.restype = ctypes.c_char_p
    for name in ("infllmv2_version", "infllmv2_sync_status", "infllmv2_selection_capacity",
                 "infllmv2_profile_enable", "infllmv2_profile_read",
                 "infllmv2_kernel_pool", "infllmv2_append", "infllmv2_block_select", "infllmv2_sparse_attn_fwd",
                 "infllmv2_decode", "infllmv2_decode_step", "infllmv2_kernel_pool_varlen",
                 "infllmv2_block_select_varlen", "infllmv2_sparse_attn_fwd_varlen"):
        getattr(lib, name).restype = ctypes.c_int
    if path == LIB_PATH:
        _lib = lib
    return lib


def declared_functions() -> list[str]:
    """Names of the functions include/infllmv2.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(infllmv2_[a-z_0-9]+)\s*\(", text)))


def status_string(status: int) -> str:
    return load().infllmv2_status_string(int(status)).decode()


def version() -> int:
    return int(load().infllmv2_version())


def _check(rc: int, what: str):
    if rc != OK:
        raise InfLLMv2Error(rc, what)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _host_ptr(t):
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("tensor must live in host memory")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def sync_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load().infllmv2_sync_status(_stream(stream)))


def profile_enable(on: bool = True):
    """Record a CUDA event around every kernel the entry points launch."""
    _check(load().infllmv2_profile_enable(1 if on else 0), "infllmv2_profile_enable")


def profile_read(max_stages: int = 8) -> list[tuple[str, float]]:
    """(stage name, milliseconds) for each kernel of the most recent call (waits for it)."""
    lib = load()
    ms = (ctypes.c_float * max_stages)()
    n = ctypes.c_int(0)
    _check(lib.infllmv2_profile_read(ms, max_stages, ctypes.byref(n)), "infllmv2_profile_read")
    return [(lib.infllmv2_profile_stage_name(i).decode(), float(ms[i])) for i in range(min(n.value, max_stages))]


def selection_capacity(params, L_max: int) -> int:
    return int(load().infllmv2_selection_capacity(ctypes.byref(Params.make(params)), int(L_max)))


def workspace_size(entry: int, B: int, Tq: int, Hq: int, Hkv: int, d: int, L_max: int, params) -> int:
    return int(load().infllmv2_workspace_size(int(entry), B, Tq, Hq, Hkv, d, L_max,
                                              ctypes.byref(Params.make(params))))


def kernel_pool(k_cache, kernel_cache, tok_begin: int, tok_end: int, params, stream=None):
    """Pool the kernels that become complete with tokens [tok_begin, tok_end)."""
    B, Hkv, L_max, d = k_cache.shape
    M_max = kernel_cache.shape[2]
    _check(load().infllmv2_kernel_pool(_ptr(k_cache), _ptr(kernel_cache), B, Hkv, L_max, M_max, d,
                                       int(tok_begin), int(tok_end), ctypes.byref(Params.make(params)),
                                       _stream(stream)), "infllmv2_kernel_pool")


def block_select(q, kernel_cache, kv_len, idx, counts, workspace, params, L_max: int, stream=None):
    """Top-k block selection for a causal chunk (the last Tq tokens of each sequence)."""
    B, Tq, Hq, d = q.shape
    Hkv, M_max = kernel_cache.shape[1], kernel_cache.shape[2]
    _check(load().infllmv2_block_select(_ptr(q), _ptr(kernel_cache), _ptr(kv_len), B, Tq, Hq, Hkv, d,
                                        int(L_max), M_max, _ptr(idx), _ptr(counts), idx.shape[-1],
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        ctypes.byref(Params.make(params)), _stream(stream)),
           "infllmv2_block_select")


def append(k_new, v_new, k_cache, v_cache, kernel_cache, kv_len, params, stream=None):
    """Write each row's new token (position kv_len - 1) into the caches and pool the kernel it completes."""
    B, Hkv, L_max, d = k_cache.shape
    M_max = 0 if kernel_cache is None else kernel_cache.shape[2]
    _check(load().infllmv2_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(kernel_cache),
                                  _ptr(kv_len), B, Hkv, d, L_max, M_max, ctypes.byref(Params.make(params)),
                                  _stream(stream)), "infllmv2_append")


def decode_step(q, k_new, v_new, k_cache, v_cache, kernel_cache, kv_len, o, workspace, params, lse=None,
                idx_out=None, counts_out=None, stream=None):
    """Append each row's new token (and the kernel it completes), then decode q over the caches."""
    B, _, Hq, d = q.shape
    Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
    M_max = kernel_cache.shape[2]
    S_max = 0 if idx_out is None else idx_out.shape[-1]
    _check(load().infllmv2_decode_step(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(kernel_cache), _ptr(kv_len), B, Hq, Hkv, d, L_max, M_max, _ptr(o),
                                       _ptr(lse), _ptr(idx_out), _ptr(counts_out), S_max, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       ctypes.byref(Params.make(params)), _stream(stream)), "infllmv2_decode_step")


def kernel_pool_varlen(k_cache, kernel_cache, kv_len, cu_q, Tq_max: int, params, stream=None):
    """Pool the kernels completed by each sequence's packed chunk (its last cu_q[b+1]-cu_q[b] tokens)."""
    B, Hkv, L_max, d = k_cache.shape
    _check(load().infllmv2_kernel_pool_varlen(_ptr(k_cache), _ptr(kernel_cache), _ptr(kv_len), _ptr(cu_q), B, Hkv,
                                              L_max, kernel_cache.shape[2], d, int(Tq_max),
                                              ctypes.byref(Params.make(params)), _stream(stream)),
           "infllmv2_kernel_pool_varlen")


def block_select_varlen(q, kernel_cache, kv_len, cu_q, Tq_max: int, idx, counts, workspace, params, L_max: int,
                        stream=None):
    """Selection for packed chunks: q [total_q, Hq, d]; idx [Hkv, total_q, S_max], counts [Hkv, total_q]."""
    total_q, Hq, d = q.shape
    B = cu_q.shape[0] - 1
    Hkv, M_max = kernel_cache.shape[1], kernel_cache.shape[2]
    _check(load().infllmv2_block_select_varlen(_ptr(q), _ptr(kernel_cache), _ptr(kv_len), _ptr(cu_q), B, int(Tq_max),
                                               total_q, Hq, Hkv, d, L_max, M_max, _ptr(idx), _ptr(counts),
                                               idx.shape[-1], _ptr(workspace),
                                               workspace.numel() * workspace.element_size(),
                                               ctypes.byref(Params.make(params)), _stream(stream)),
           "infllmv2_block_select_varlen")


def sparse_attn_fwd_varlen(q, k_cache, v_cache, idx, counts, kv_len, cu_q, Tq_max: int, o, params, lse=None,
                           stream=None):
    """Attention for packed chunks: q, o [total_q, Hq, d]; lse [Hq, total_q]; idx None = dense causal."""
    total_q, Hq, d = q.shape
    B = cu_q.shape[0] - 1
    Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
    _check(load().infllmv2_sparse_attn_fwd_varlen(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(idx), _ptr(counts),
                                                  0 if idx is None else idx.shape[-1], _ptr(kv_len), _ptr(cu_q), B,
                                                  int(Tq_max), total_q, Hq, Hkv, d, L_max, _ptr(o), _ptr(lse),
                                                  ctypes.byref(Params.make(params)), _stream(stream)),
           "infllmv2_sparse_attn_fwd_varlen")


def sparse_attn_fwd(q, k_cache, v_cache, idx, counts, kv_len, o, params, lse=None, workspace=None,
                    stream=None):
    """Block-sparse causal attention of a chunk over its selected blocks (idx None: dense)."""
    B, Tq, Hq, d = q.shape
    Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().infllmv2_sparse_attn_fwd(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(idx), _ptr(counts),
                                           0 if idx is None else idx.shape[-1], _ptr(kv_len), B, Tq, Hq,
                                           Hkv, d, L_max, _ptr(o), _ptr(lse), _ptr(workspace), ws_bytes,
                                           ctypes.byref(Params.make(params)), _stream(stream)),
           "infllmv2_sparse_attn_fwd")


def sparse_attn_bwd(q, k_cache, v_cache, o, lse, dout, idx, counts, kv_len, dq, dk, dv, workspace, params,
                    stream=None):
    """Gradients (fp32 dq, dk, dv) of the chunk attention with the selection held fixed."""
    B, Tq, Hq, d = q.shape
    Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().infllmv2_sparse_attn_bwd(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), _ptr(dout),
                                           _ptr(idx), _ptr(counts), 0 if idx is None else idx.shape[-1],
                                           _ptr(kv_len), B, Tq, Hq, Hkv, d, L_max, _ptr(dq), _ptr(dk), _ptr(dv),
                                           _ptr(workspace), ws_bytes, ctypes.byref(Params.make(params)),
                                           _stream(stream)), "infllmv2_sparse_attn_bwd")


def decode(q, k_cache, v_cache, kernel_cache, kv_len, o, workspace, params, lse=None, draft_k=None,
           draft_v=None, tree_mask=None, idx_out=None, counts_out=None, stream=None):
    """Selection + split-KV attention + merge for one decode token or a draft tree."""
    B, n_draft, Hq, d = q.shape
    Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
    M_max = kernel_cache.shape[2]
    S_max = 0 if idx_out is None else idx_out.shape[-1]
    _check(load().infllmv2_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kernel_cache), _ptr(kv_len),
                                  _ptr(draft_k), _ptr(draft_v), _ptr(tree_mask), B, n_draft, Hq, Hkv, d,
                                  L_max, M_max, _ptr(o), _ptr(lse), _ptr(idx_out), _ptr(counts_out), S_max,
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  ctypes.byref(Params.make(params)), _stream(stream)), "infllmv2_decode")


def _check_host_step_buffers(q_host, kv_len_host, o_host, q_dev, kv_len_dev, o_dev, lse_host, lse_dev, Hkv):
    """The host-buffer decode copies B*Hq*d bf16 values of q and o, B int32 lengths and B*Hq fp32
    lse values between the paired tensors: check their types and sizes once, so a wrong tensor
    raises here instead of overrunning memory in the C call."""
    import torch
    B, Hq, d = q_host.shape[0], q_host.shape[-2], q_host.shape[-1]
    n = B * Hq * d
    for name, t in (("q_host", q_host), ("q_dev", q_dev), ("o_host", o_host), ("o_dev", o_dev)):
        if t.dtype != torch.bfloat16 or t.numel() != n:
            raise ValueError(f"{name} must be bf16 with {n} elements (B * Hq * d)")
    for name, t in (("kv_len_host", kv_len_host), ("kv_len_dev", kv_len_dev)):
        if t.dtype != torch.int32 or t.numel() != B:
            raise ValueError(f"{name} must be int32 with {B} elements (B)")
    if (lse_host is None) != (lse_dev is None):
        raise ValueError("lse_host and lse_dev must be given together")
    for name, t in (("lse_host", lse_host), ("lse_dev", lse_dev)):
        if t is not None and (t.dtype != torch.float32 or t.numel() != B * Hq):
            raise ValueError(f"{name} must be fp32 with {B * Hq} elements (B * Hq)")
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of the caches' KV heads")


def decode_host(q_host, kv_len_host, o_host, q_dev, kv_len_dev, o_dev, k_cache, v_cache, kernel_cache,
                workspace, params, lse_host=None, lse_dev=None, stream=None):
    """One single-token decode step with q, kv_len and o in host memory (pinned for asynchronous
    copies): copy in, decode on the device staging tensors, copy out, wait.  The host output is
    complete on return; device errors raise."""
    B, Hq, d = q_host.shape[0], q_host.shape[-2], q_host.shape[-1]
    Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
    M_max = kernel_cache.shape[2]
    _check_host_step_buffers(q_host, kv_len_host, o_host, q_dev, kv_len_dev, o_dev, lse_host, lse_dev, Hkv)
    _check(load().infllmv2_decode_host(_host_ptr(q_host), _host_ptr(kv_len_host), _host_ptr(o_host),
                                       _host_ptr(lse_host), _ptr(q_dev), _ptr(kv_len_dev), _ptr(o_dev),
                                       _ptr(lse_dev), _ptr(k_cache), _ptr(v_cache), _ptr(kernel_cache), B, Hq, Hkv,
                                       d, L_max, M_max, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       ctypes.byref(Params.make(params)), _stream(stream)), "infllmv2_decode_host")


def host_memory_direct() -> bool:
    """Whether decode_host's zero-copy way also takes pageable host buffers on the current device
    (the device reads host memory through the host's page tables)."""
    v = ctypes.c_int(0)
    _check(load().infllmv2_host_memory_direct(ctypes.byref(v)), "infllmv2_host_memory_direct")
    return v.value != 0


class DecodeHostStep:
    """decode_host with its buffers bound once: a serving loop with static buffers (its query,
    length and output tensors refilled in place each step) pays only the C call per step.  The
    tensors must stay alive and in place while the object is used."""

    def __init__(self, q_host, kv_len_host, o_host, q_dev, kv_len_dev, o_dev, k_cache, v_cache, kernel_cache,
                 workspace, params, lse_host=None, lse_dev=None, stream=None):
        B, Hq, d = q_host.shape[0], q_host.shape[-2], q_host.shape[-1]
        Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
        _check_host_step_buffers(q_host, kv_len_host, o_host, q_dev, kv_len_dev, o_dev, lse_host, lse_dev, Hkv)
        self._fn = load().infllmv2_decode_host
        self._params = Params.make(params)
        self._args = (_host_ptr(q_host), _host_ptr(kv_len_host), _host_ptr(o_host), _host_ptr(lse_host), _ptr(q_dev),
                      _ptr(kv_len_dev), _ptr(o_dev), _ptr(lse_dev), _ptr(k_cache), _ptr(v_cache), _ptr(kernel_cache),
                      B, Hq, Hkv, d, L_max, kernel_cache.shape[2], _ptr(workspace),
                      workspace.numel() * workspace.element_size(), ctypes.byref(self._params), _stream(stream))
        self._keep = (q_host, kv_len_host, o_host, lse_host, q_dev, kv_len_dev, o_dev, lse_dev, k_cache, v_cache,
                      kernel_cache, workspace)

    def __call__(self):
        rc = self._fn(*self._args)
        if rc != OK:
            raise InfLLMv2Error(rc, "infllmv2_decode_host")


NOALLOC_SCRATCH_BYTES = 16 << 20  # INFLLMV2_NOALLOC_SCRATCH_BYTES


def decode_noalloc(q, k_cache, v_cache, kernel_cache, kv_len, o, params, lse=None, draft_k=None, draft_v=None,
                   tree_mask=None, idx_out=None, counts_out=None, stream=None):
    """infllmv2_decode without a workspace argument: for callers that cannot allocate
    device memory; the library's fixed scratch array is used instead (see the header)."""
    B, n_draft, Hq, d = q.shape
    Hkv, L_max = k_cache.shape[1], k_cache.shape[2]
    M_max = kernel_cache.shape[2]
    S_max = 0 if idx_out is None else idx_out.shape[-1]
    _check(load().infllmv2_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kernel_cache),
                                          _ptr(kv_len), _ptr(draft_k), _ptr(draft_v), _ptr(tree_mask), B,
                                          n_draft, Hq, Hkv, d, L_max, M_max, _ptr(o), _ptr(lse),
                                          _ptr(idx_out), _ptr(counts_out), S_max,
                                          ctypes.byref(Params.make(params)), _stream(stream)),
           "infllmv2_decode_noalloc")
