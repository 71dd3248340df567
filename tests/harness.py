"""Shared test helpers: upload seeded inputs, run the CUDA path through the C ABI,
run the fp64 oracle on the same inputs, and compare.

The comparison rules:
  * semantic kernels: bit-exact;
  * selections: identical sets, except that a block may be swapped only when its
    oracle score lies within 1e-3 (relative) of the oracle's k-th kept score
    -- a near-tie that fp32 and fp64 may order differently;
  * attention output: max |gpu - oracle| <= 1e-2 and mean <= 1e-3, where the
    oracle attends over the GPU's own selection (so a tolerated near-tie swap
    cannot leak into the attention check).
"""
from __future__ import annotations

import numpy as np

import oracle
from block_sparse_long_infllm_gb300 import synth

MAX_ABS_TOL = 1e-2
MEAN_ABS_TOL = 1e-3
NEAR_TIE_REL = 1e-3


def torch_mod():
    import torch
    return torch


def to_dev(a: np.ndarray, dtype=None):
    torch = torch_mod()
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    if a.dtype == np.uint64:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int64)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_to_np_bits(t) -> np.ndarray:
    torch = torch_mod()
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(t) -> np.ndarray:
    return synth.bf16_bits_to_f32(bf16_to_np_bits(t)).astype(np.float64)


def lib():
    from block_sparse_long_infllm_gb300 import infllmv2
    return infllmv2


def n_kernels(w) -> int:
    return oracle.n_kernels(w.L_max, w.kernel_size, w.kernel_stride)


def run_gpu(w, inp: dict, pool_split: int | None = None, params: dict | None = None) -> dict:
    """Run the whole CUDA path for workload w.  Returns device tensors."""
    torch = torch_mod()
    L = lib()
    p = params or w.params()
    q = to_dev(inp["q"])
    k = to_dev(inp["k_cache"])
    v = to_dev(inp["v_cache"])
    kv_len = to_dev(inp["kv_len"])
    M_max = max(n_kernels(w), 1)
    kern = torch.zeros((w.B, w.Hkv, M_max, w.d), dtype=torch.bfloat16, device="cuda")
    S_cap = L.selection_capacity(p, w.L_max)
    out = dict(q=q, k=k, v=v, kv_len=kv_len, kern=kern, S_cap=S_cap)
    if w.kind == "prefill":
        split = w.q_pos0 if pool_split is None else pool_split
        L.kernel_pool(k, kern, 0, split, p)
        L.kernel_pool(k, kern, split, w.L, p)
        idx = torch.empty((w.B, w.Hkv, w.Tq, S_cap), dtype=torch.int32, device="cuda")
        counts = torch.empty((w.B, w.Hkv, w.Tq), dtype=torch.int32, device="cuda")
        ws = torch.empty(L.workspace_size(L.ENTRY_BLOCK_SELECT, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, p),
                         dtype=torch.uint8, device="cuda")
        L.block_select(q, kern, kv_len, idx, counts, ws, p, w.L_max)
        out["ws"] = ws  # starts with the block scores
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device="cuda")
        L.sparse_attn_fwd(q, k, v, idx, counts, kv_len, o, p, lse=lse)
    else:
        L.kernel_pool(k, kern, 0, w.L, p)
        n = w.Tq
        idx = torch.empty((w.B, w.Hkv, n, S_cap), dtype=torch.int32, device="cuda")
        counts = torch.empty((w.B, w.Hkv, n), dtype=torch.int32, device="cuda")
        ws = torch.empty(L.workspace_size(L.ENTRY_DECODE, w.B, n, w.Hq, w.Hkv, w.d, w.L_max, p),
                         dtype=torch.uint8, device="cuda")
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, n), dtype=torch.float32, device="cuda")
        tree = w.kind == "tree"
        L.decode(q, k, v, kern, kv_len, o, ws, p, lse=lse,
                 draft_k=to_dev(inp["draft_k"]) if tree else None,
                 draft_v=to_dev(inp["draft_v"]) if tree else None,
                 tree_mask=to_dev(inp["tree_mask"]) if tree else None,
                 idx_out=idx, counts_out=counts)
    torch.cuda.synchronize()
    st = L.sync_status()
    assert st == 0, f"device error status {st}: {L.status_string(st)}"
    out.update(idx=idx, counts=counts, o=o, lse=lse)
    return out


def compare_selection(gidx, gcnt, oidx, ocnt, S, kth):
    """Returns (rows, exact, tie_explained, unexplained) over all selection rows."""
    rows = exact = ties = bad = 0
    B, H, T = ocnt.shape
    for b in range(B):
        for g in range(H):
            for t in range(T):
                rows += 1
                gs = set(gidx[b, g, t, :gcnt[b, g, t]].tolist())
                os_ = set(oidx[b, g, t, :ocnt[b, g, t]].tolist())
                if gs == os_:
                    exact += 1
                    continue
                thr = kth[b, g, t]
                diff = gs ^ os_
                if len(gs) == len(os_) and np.isfinite(thr) and all(
                        abs(S[b, g, t, blk] - thr) <= NEAR_TIE_REL * abs(thr) for blk in diff):
                    ties += 1
                else:
                    bad += 1
    return rows, exact, ties, bad


def near_tie_rows(kth, nxt) -> int:
    gap = np.abs(kth - nxt) / np.abs(kth)
    return int(np.sum(np.isfinite(gap) & (gap < NEAR_TIE_REL)))


def check_output(o_gpu: np.ndarray, o_ref: np.ndarray, what: str = "o"):
    err = np.abs(o_gpu - o_ref)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    assert err.max() <= MAX_ABS_TOL, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= MEAN_ABS_TOL, f"{what}: mean abs err {err.mean():.3e}"
    return float(err.max()), float(err.mean())
