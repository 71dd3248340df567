"""The allocation-free decode entry point (infllmv2_decode_noalloc) against the
regular one (infllmv2_decode), through the C ABI.

infllmv2_decode_noalloc exists for callers that cannot allocate device memory
(their memory is reserved up front by their own pool, or they are plugins that
only receive input and output pointers, or they may not allocate after
start-up); it uses a fixed scratch array inside the library instead of a
caller workspace.  Two calls in a row must both reproduce the regular entry
point's output (within the tolerance the parity tests use) and selection: the
second call reuses the scratch the first one left behind.  Problems needing
more scratch than the array holds must be refused before any work is queued.

This file is collected last, so a run that stops at the first failure has
already run every other test; it needs no state from them.
"""
import ctypes

import numpy as np
import pytest

from block_sparse_long_infllm_gb300 import infllmv2, synth

from harness import bf16_to_f64, check_output, n_kernels, to_dev

pytestmark = pytest.mark.gpu


def _setup(w, inp):
    import torch
    p = w.params()
    q, k, v = (to_dev(inp[x]) for x in ("q", "k_cache", "v_cache"))
    kv = to_dev(inp["kv_len"])
    kern = torch.zeros((w.B, w.Hkv, n_kernels(w), w.d), dtype=torch.bfloat16, device="cuda")
    infllmv2.kernel_pool(k, kern, 0, w.L, p)
    S_cap = infllmv2.selection_capacity(p, w.L_max)
    return p, q, k, v, kv, kern, S_cap


def test_noalloc_decode_matches_decode_on_two_calls(cuda_lib):
    import torch
    w = synth.WORKLOADS["decode_128k_b4"]
    inp = synth.make_inputs(w)
    p, q, k, v, kv, kern, S_cap = _setup(w, inp)
    need = infllmv2.workspace_size(infllmv2.ENTRY_DECODE, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, p)
    assert 0 < need <= infllmv2.NOALLOC_SCRATCH_BYTES

    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o_ref = torch.empty_like(q)
    lse_ref = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device="cuda")
    idx_ref = torch.empty((w.B, w.Hkv, w.Tq, S_cap), dtype=torch.int32, device="cuda")
    cnt_ref = torch.empty((w.B, w.Hkv, w.Tq), dtype=torch.int32, device="cuda")
    infllmv2.decode(q, k, v, kern, kv, o_ref, ws, p, lse=lse_ref, idx_out=idx_ref, counts_out=cnt_ref)
    assert infllmv2.sync_status() == 0
    ref = bf16_to_f64(o_ref)

    for call in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        idx = torch.full_like(idx_ref, -7)
        cnt = torch.full_like(cnt_ref, -7)
        # straight through the C ABI symbol
        rc = infllmv2.load().infllmv2_decode_noalloc(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
            ctypes.c_void_p(kern.data_ptr()), ctypes.c_void_p(kv.data_ptr()), None, None, None,
            w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, kern.shape[2], ctypes.c_void_p(o.data_ptr()),
            ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(cnt.data_ptr()),
            S_cap, ctypes.byref(infllmv2.Params.make(p)),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, infllmv2.status_string(rc)
        assert infllmv2.sync_status() == 0
        check_output(bf16_to_f64(o), ref, what=f"noalloc call {call}")
        assert np.max(np.abs(lse.cpu().numpy() - lse_ref.cpu().numpy())) < 2e-3
        assert torch.equal(cnt, cnt_ref) and torch.equal(idx, idx_ref)


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
