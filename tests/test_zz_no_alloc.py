"""The allocation-free decode entry point (infllmv2_decode_noalloc), through the C ABI, against
the regular entry point (infllmv2_decode with a caller workspace) and against the oracle.

infllmv2_decode_noalloc exists for callers that cannot allocate device memory (their memory is
reserved up front by their own pool, or they are plugins that only receive input and output
pointers, or they may not allocate after start-up); it takes its scratch from one fixed array
inside the library instead of a caller workspace.

The scratch is used by the tree-verification path (block scores, the drafts' selections and the
split-KV partials live there), so the main case is a 16-draft tree over a 64K cache: a first call
on other inputs leaves its scores and partials in the array, then two calls in a row on the real
inputs must each give the regular entry point's selection exactly and its output within the
parity tolerance, and agree with the oracle (selection up to near-ties, output within
max-abs 1e-2 / mean-abs 1e-3).  A stale score or partial left by an earlier call would show.
The single-token decode at 128K (which runs one kernel that keeps everything on chip and reads
no scratch) is checked the same way, and problems needing more scratch than the array holds
must be refused before any work is queued.

This file is collected last, so a run that stops at the first failure has already run every
other test; it needs no state from them.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from block_sparse_long_infllm_gb300 import infllmv2, synth

from harness import bf16_to_f64, check_output, compare_selection, n_kernels, to_dev


def test_scratch_size_matches_header():
    """The binding's copy of the scratch size is the header's (no GPU needed)."""
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                             "infllmv2.h")).read()
    m = re.search(r"#define\s+INFLLMV2_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m is not None
    assert int(m.group(1)) << int(m.group(2)) == infllmv2.NOALLOC_SCRATCH_BYTES


def _noalloc_call(w, q, k, v, kern, kv, o, lse, idx, cnt, p, dk=None, dv=None, mask=None):
    """infllmv2_decode_noalloc straight through the C ABI symbol."""
    import torch
    vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return infllmv2.load().infllmv2_decode_noalloc(
        vp(q), vp(k), vp(v), vp(kern), vp(kv), vp(dk), vp(dv), vp(mask),
        w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, kern.shape[2], vp(o), vp(lse), vp(idx), vp(cnt), idx.shape[-1],
        ctypes.byref(infllmv2.Params.make(p)), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _device_inputs(w, inp):
    import torch
    p = w.params()
    t = dict(q=to_dev(inp["q"]), k=to_dev(inp["k_cache"]), v=to_dev(inp["v_cache"]), kv=to_dev(inp["kv_len"]))
    t["kern"] = torch.zeros((w.B, w.Hkv, n_kernels(w), w.d), dtype=torch.bfloat16, device="cuda")
    infllmv2.kernel_pool(t["k"], t["kern"], 0, w.L, p)
    tree = w.kind == "tree"
    t["dk"] = to_dev(inp["draft_k"]) if tree else None
    t["dv"] = to_dev(inp["draft_v"]) if tree else None
    t["mask"] = to_dev(inp["tree_mask"]) if tree else None
    return t


def _outputs(w, S_cap, fill=True):
    import torch
    o = torch.full((w.B, w.Tq, w.Hq, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.Hq, w.Tq), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.full((w.B, w.Hkv, w.Tq, S_cap), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((w.B, w.Hkv, w.Tq), -7, dtype=torch.int32, device="cuda")
    return o, lse, idx, cnt


def _check_two_calls(w, inp, prime_inp):
    import torch
    p = w.params()
    tree = w.kind == "tree"
    S_cap = infllmv2.selection_capacity(p, w.L_max)
    need = infllmv2.workspace_size(infllmv2.ENTRY_DECODE, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, p)
    assert 0 < need <= infllmv2.NOALLOC_SCRATCH_BYTES
    t = _device_inputs(w, inp)

    # the regular entry point with a caller workspace
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o_ref, lse_ref, idx_ref, cnt_ref = _outputs(w, S_cap)
    infllmv2.decode(t["q"], t["k"], t["v"], t["kern"], t["kv"], o_ref, ws, p, lse=lse_ref, draft_k=t["dk"],
                    draft_v=t["dv"], tree_mask=t["mask"], idx_out=idx_ref, counts_out=cnt_ref)
    assert infllmv2.sync_status() == 0

    # the oracle on the same inputs
    kern_ref, _ = oracle.kernel_pool(inp["k_cache"], inp["kv_len"], w.kernel_size, w.kernel_stride, n_kernels(w))
    S = oracle.block_scores(inp["q"], kern_ref, inp["kv_len"], w.Hkv, p, tree=tree)
    oidx, ocnt, kth, _ = oracle.select(S, inp["kv_len"], w.Tq, p, tree=tree, S_max=S_cap)

    # a first call on other inputs leaves its own scores, selections and partials in the scratch
    pt = _device_inputs(w, prime_inp)
    po, plse, pidx, pcnt = _outputs(w, S_cap)
    rc = _noalloc_call(w, pt["q"], pt["k"], pt["v"], pt["kern"], pt["kv"], po, plse, pidx, pcnt, p,
                       pt["dk"], pt["dv"], pt["mask"])
    assert rc == 0, infllmv2.status_string(rc)
    assert infllmv2.sync_status() == 0

    for call in range(2):
        o, lse, idx, cnt = _outputs(w, S_cap)
        rc = _noalloc_call(w, t["q"], t["k"], t["v"], t["kern"], t["kv"], o, lse, idx, cnt, p, t["dk"], t["dv"],
                           t["mask"])
        assert rc == 0, infllmv2.status_string(rc)
        assert infllmv2.sync_status() == 0
        what = f"noalloc call {call}"
        # against the regular entry point: the same selection, the output within tolerance
        assert torch.equal(cnt, cnt_ref) and torch.equal(idx, idx_ref), what
        check_output(bf16_to_f64(o), bf16_to_f64(o_ref), what=what)
        assert np.max(np.abs(lse.cpu().numpy() - lse_ref.cpu().numpy())) < 2e-3, what
        # against the oracle
        gidx, gcnt = idx.cpu().numpy(), cnt.cpu().numpy()
        rows, exact, ties, bad = compare_selection(gidx, gcnt, oidx, ocnt, S, kth)
        assert bad == 0, f"{what}: {bad} of {rows} selections differ outside near-ties"
        o_or, lse_or = oracle.attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["kv_len"], gidx, gcnt, p,
                                        draft_k=inp.get("draft_k"), draft_v=inp.get("draft_v"),
                                        tree_mask=inp.get("tree_mask"))
        check_output(bf16_to_f64(o), o_or, what=what + " vs oracle")
        assert np.max(np.abs(lse.cpu().numpy() - lse_or)) < 2e-3, what


@pytest.mark.gpu
def test_noalloc_tree_verification_uses_its_scratch_on_two_calls(cuda_lib):
    w = synth.WORKLOADS["tree_verify_64k"]
    _check_two_calls(w, synth.make_inputs(w), synth.make_inputs(w.scaled(seed=w.seed + 500)))


@pytest.mark.gpu
def test_noalloc_single_token_decode_on_two_calls(cuda_lib):
    w = synth.WORKLOADS["decode_128k_b4"]
    _check_two_calls(w, synth.make_inputs(w), synth.make_inputs(w.scaled(seed=w.seed + 500)))


@pytest.mark.gpu
def test_noalloc_decode_refuses_problems_beyond_its_scratch(cuda_lib):
    import torch
    w = synth.WORKLOADS["decode_128k_b4"].scaled(B=64, L=4096, seed=4242)
    p = w.params()
    need = infllmv2.workspace_size(infllmv2.ENTRY_DECODE, w.B, 64, w.Hq, w.Hkv, w.d, w.L_max, p)
    assert need > infllmv2.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((w.B, 64, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((w.B, w.Hkv, w.L_max, w.d), dtype=torch.bfloat16, device="cuda")
    kern = torch.zeros((w.B, w.Hkv, n_kernels(w), w.d), dtype=torch.bfloat16, device="cuda")
    kv = torch.full((w.B,), w.L, dtype=torch.int32, device="cuda")
    dk = torch.zeros((w.B, w.Hkv, 64, w.d), dtype=torch.bfloat16, device="cuda")
    mask = torch.ones((w.B, 64), dtype=torch.int64, device="cuda")
    o = torch.empty_like(q)
    with pytest.raises(infllmv2.InfLLMv2Error) as e:
        infllmv2.decode_noalloc(q, kc, kc, kern, kv, o, p, draft_k=dk, draft_v=dk, tree_mask=mask)
    assert e.value.status == infllmv2.ERR_WORKSPACE
    assert infllmv2.sync_status() == 0
