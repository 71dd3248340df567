"""Decode-step append through the C ABI: the new token's K and V land in row kv_len - 1 and the
semantic kernel it completes is pooled, step after step with per-sequence lengths (one sequence
starting empty).  The caches must equal a plain numpy assignment bit for bit, the kernel cache the
oracle's pooling of the final cache bit for bit, and decode after an append the oracle's
selection and attention on the updated cache."""
import numpy as np
import pytest

import oracle
from block_sparse_long_infllm_gb300 import synth

from harness import bf16_to_f64, bf16_to_np_bits, check_output, compare_selection, lib, to_dev, torch_mod

pytestmark = pytest.mark.gpu


def _decode_check(w, p, q_bits, k_np, v_np, kv, k, v, kern, kv_dev):
    torch = torch_mod()
    L = lib()
    q = to_dev(q_bits)
    S_cap = L.selection_capacity(p, w.L_max)
    idx = torch.empty((w.B, w.Hkv, 1, S_cap), dtype=torch.int32, device="cuda")
    cnt = torch.empty((w.B, w.Hkv, 1), dtype=torch.int32, device="cuda")
    ws = torch.empty(L.workspace_size(L.ENTRY_DECODE, w.B, 1, w.Hq, w.Hkv, w.d, w.L_max, p), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device="cuda")
    L.decode(q, k, v, kern, kv_dev, o, ws, p, lse=lse, idx_out=idx, counts_out=cnt)
    torch.cuda.synchronize()
    assert L.sync_status() == 0
    M = oracle.n_kernels(w.L_max, w.kernel_size, w.kernel_stride)
    kern_ref, _ = oracle.kernel_pool(k_np, kv, w.kernel_size, w.kernel_stride, M)
    S = oracle.block_scores(q_bits, kern_ref, kv, w.Hkv, p)
    oidx, ocnt, kth, _ = oracle.select(S, kv, 1, p, S_max=S_cap)
    gidx, gcnt = idx.cpu().numpy(), cnt.cpu().numpy()
    rows, exact, ties, bad = compare_selection(gidx, gcnt, oidx, ocnt, S, kth)
    assert bad == 0, f"{bad} of {rows} selections differ outside near-ties"
    o_ref, _ = oracle.attention(q_bits, k_np, v_np, kv, gidx, gcnt, p)
    check_output(bf16_to_f64(o), o_ref)


@pytest.mark.parametrize("d,bs", [(128, 64), (64, 128)])
def test_append_steps_match_oracle(cuda_lib, d, bs):
    torch = torch_mod()
    L = lib()
    w = synth.WORKLOADS["decode_32k"].scaled(B=2, L=1600, Hq=32, Hkv=2, d=d, block_size=bs, topk=8,
                                              dense_len=0, seed=5100 + d)
    inp = synth.make_inputs(w)
    p = w.params()
    c, s = w.kernel_size, w.kernel_stride
    k_np, v_np = inp["k_cache"].copy(), inp["v_cache"].copy()
    k, v = to_dev(k_np), to_dev(v_np)
    M = oracle.n_kernels(w.L_max, c, s)
    kern = torch.zeros((w.B, w.Hkv, M, w.d), dtype=torch.bfloat16, device="cuda")
    L.kernel_pool(k, kern, 0, w.L_max, p)  # past each length these kernels are stale until appends redo them
    kv = np.array([0, 1251], dtype=np.int32)
    rng = np.random.default_rng(77 + d)
    for step in range(40):
        kn = synth.f32_to_bf16_bits(rng.standard_normal((w.B, w.Hkv, w.d)).astype(np.float32))
        vn = synth.f32_to_bf16_bits(rng.standard_normal((w.B, w.Hkv, w.d)).astype(np.float32))
        kv = kv + 1
        kv_dev = to_dev(kv)
        L.append(to_dev(kn), to_dev(vn), k, v, kern, kv_dev, p)
        for b in range(w.B):
            k_np[b, :, kv[b] - 1] = kn[b]
            v_np[b, :, kv[b] - 1] = vn[b]
        if step in (0, 17, 39):
            q_bits = synth.f32_to_bf16_bits(rng.standard_normal((w.B, 1, w.Hq, w.d)).astype(np.float32))
            _decode_check(w, p, q_bits, k_np, v_np, kv, k, v, kern, kv_dev)
    torch.cuda.synchronize()
    assert L.sync_status() == 0
    assert np.array_equal(bf16_to_np_bits(k), k_np) and np.array_equal(bf16_to_np_bits(v), v_np)
    kern_ref, _ = oracle.kernel_pool(k_np, kv, c, s, M)
    gk = bf16_to_np_bits(kern)
    for b in range(w.B):
        nk = oracle.n_kernels(int(kv[b]), c, s)
        assert np.array_equal(gk[b, :, :nk], kern_ref[b, :, :nk]), f"kernels of sequence {b} differ"


def test_append_length_past_cache_sets_error_and_skips_row(cuda_lib):
    torch = torch_mod()
    L = lib()
    w = synth.WORKLOADS["decode_32k"].scaled(B=2, L=256, Hq=4, Hkv=2, d=128, seed=5200)
    p = w.params()
    k = torch.zeros((w.B, w.Hkv, w.L, w.d), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    kern = torch.zeros((w.B, w.Hkv, oracle.n_kernels(w.L, 32, 16), w.d), dtype=torch.bfloat16, device="cuda")
    kn = torch.ones((w.B, w.Hkv, w.d), dtype=torch.bfloat16, device="cuda")
    kv_dev = to_dev(np.array([w.L + 1, 48], dtype=np.int32))
    L.append(kn, kn, k, v, kern, kv_dev, p)
    torch.cuda.synchronize()
    assert L.sync_status() != 0
    assert float(k[0].abs().sum()) == 0.0            # the bad row wrote nothing
    assert float(k[1, :, 47].float().mean()) == 1.0  # the good row was appended
    assert float(kern[1, :, 1].float().mean()) == 1.0 / 32.0  # kernel 1 = rows 16..47, only row 47 nonzero
    assert L.sync_status() == 0                      # the error word was cleared


@pytest.mark.parametrize("n_local,lists,d,bs", [(2, True, 128, 64), (1, True, 128, 64), (2, False, 128, 64),
                                               (2, True, 64, 128)],
                         ids=["fused", "append_then_decode", "fused_without_block_lists", "fused_d64_block128"])
def test_decode_step_matches_oracle(cuda_lib, n_local, lists, d, bs):
    """infllmv2_decode_step: one call appends and decodes.  With 2 local blocks the single cluster
    kernel does both (the new kernel overlaps only forced blocks); with 1 the append kernel runs
    first.  Caches, kernels and outputs as for append followed by decode.  Without the optional
    block lists: at the checked steps the same step is repeated with them (an append of the same
    row is idempotent) and both outputs must be the same bits."""
    torch = torch_mod()
    L = lib()
    w = synth.WORKLOADS["decode_32k"].scaled(B=2, L=1600, Hq=32, Hkv=2, d=d, block_size=bs, topk=8, n_local=n_local,
                                              dense_len=0, seed=5300 + n_local + (0 if (d, bs) == (128, 64) else d + bs))
    inp = synth.make_inputs(w)
    p = w.params()
    c, s = w.kernel_size, w.kernel_stride
    k_np, v_np = inp["k_cache"].copy(), inp["v_cache"].copy()
    k, v = to_dev(k_np), to_dev(v_np)
    M = oracle.n_kernels(w.L_max, c, s)
    kern = torch.zeros((w.B, w.Hkv, M, w.d), dtype=torch.bfloat16, device="cuda")
    L.kernel_pool(k, kern, 0, w.L_max, p)
    S_cap = L.selection_capacity(p, w.L_max)
    idx = torch.empty((w.B, w.Hkv, 1, S_cap), dtype=torch.int32, device="cuda")
    cnt = torch.empty((w.B, w.Hkv, 1), dtype=torch.int32, device="cuda")
    ws = torch.empty(L.workspace_size(L.ENTRY_DECODE, w.B, 1, w.Hq, w.Hkv, w.d, w.L_max, p), dtype=torch.uint8,
                     device="cuda")
    kv = np.array([0, 1251], dtype=np.int32)
    rng = np.random.default_rng(91 + n_local)
    for step in range(40):
        kn = synth.f32_to_bf16_bits(rng.standard_normal((w.B, w.Hkv, w.d)).astype(np.float32))
        vn = synth.f32_to_bf16_bits(rng.standard_normal((w.B, w.Hkv, w.d)).astype(np.float32))
        q_bits = synth.f32_to_bf16_bits(rng.standard_normal((w.B, 1, w.Hq, w.d)).astype(np.float32))
        kv = kv + 1
        for b in range(w.B):
            k_np[b, :, kv[b] - 1] = kn[b]
            v_np[b, :, kv[b] - 1] = vn[b]
        q = to_dev(q_bits)
        o = torch.empty_like(q)
        L.decode_step(q, to_dev(kn), to_dev(vn), k, v, kern, to_dev(kv), o, ws, p, idx_out=idx if lists else None,
                      counts_out=cnt if lists else None)
        if step in (0, 9, 17, 31, 39):
            if not lists:
                o_lists = torch.empty_like(q)
                L.decode_step(q, to_dev(kn), to_dev(vn), k, v, kern, to_dev(kv), o_lists, ws, p, idx_out=idx,
                              counts_out=cnt)
                torch.cuda.synchronize()
                assert torch.equal(o.view(torch.int16), o_lists.view(torch.int16)), f"step {step}"
            torch.cuda.synchronize()
            assert L.sync_status() == 0
            kern_ref, _ = oracle.kernel_pool(k_np, kv, c, s, M)
            S = oracle.block_scores(q_bits, kern_ref, kv, w.Hkv, p)
            oidx, ocnt, kth, _ = oracle.select(S, kv, 1, p, S_max=S_cap)
            gidx, gcnt = idx.cpu().numpy(), cnt.cpu().numpy()
            rows, exact, ties, bad = compare_selection(gidx, gcnt, oidx, ocnt, S, kth)
            assert bad == 0, f"step {step}: {bad} of {rows} selections differ outside near-ties"
            o_ref, _ = oracle.attention(q_bits, k_np, v_np, kv, gidx, gcnt, p)
            check_output(bf16_to_f64(o), o_ref, f"o at step {step}")
    torch.cuda.synchronize()
    assert L.sync_status() == 0
    assert np.array_equal(bf16_to_np_bits(k), k_np) and np.array_equal(bf16_to_np_bits(v), v_np)
    kern_ref, _ = oracle.kernel_pool(k_np, kv, c, s, M)
    gk = bf16_to_np_bits(kern)
    for b in range(w.B):
        nk = oracle.n_kernels(int(kv[b]), c, s)
        assert np.array_equal(gk[b, :, :nk], kern_ref[b, :, :nk]), f"kernels of sequence {b} differ"
