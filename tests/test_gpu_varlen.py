"""Variable-length batched prefill through the C ABI: sequences with different chunk lengths
(including a one-token and an empty chunk) packed into one launch per step.  Each sequence must
get what the oracle computes for it alone: its chunk's kernels bit for bit, its selections (up to
near-ties), its outputs and lse."""
import numpy as np
import pytest

import oracle
from block_sparse_long_infllm_gb300 import synth

from harness import (bf16_to_f64, bf16_to_np_bits, check_output, compare_selection, lib, to_dev, torch_mod)

pytestmark = pytest.mark.gpu


def _setup(Hq, Hkv, d, bs, lens, kv, L_max, seed, topk=4, n_local=2):
    w = synth.WORKLOADS["chunked_prefill_32k"].scaled(B=len(lens), L=L_max, Tq=max(lens), Hq=Hq, Hkv=Hkv, d=d,
                                                       block_size=bs, topk=topk, n_local=n_local, dense_len=0,
                                                       seed=seed)
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(cu[-1])
    q = synth.f32_to_bf16_bits(rng.standard_normal((total, Hq, d)).astype(np.float32))
    k = synth.f32_to_bf16_bits(rng.standard_normal((len(lens), Hkv, L_max, d)).astype(np.float32))
    v = synth.f32_to_bf16_bits(rng.standard_normal((len(lens), Hkv, L_max, d)).astype(np.float32))
    return w, cu, total, q, k, v, np.array(kv, dtype=np.int32)


CASES = [
    dict(Hq=32, Hkv=2, d=128, bs=128, lens=[203, 64, 1, 0, 130], kv=[2500, 1311, 900, 700, 3000], L_max=3000),
    dict(Hq=8, Hkv=2, d=64, bs=64, lens=[77, 150, 1, 33], kv=[1500, 2000, 64, 700], L_max=2048),
]


@pytest.mark.parametrize("case", CASES, ids=["g16_d128_b128", "g4_d64_b64"])
def test_varlen_prefill_matches_oracle_per_sequence(cuda_lib, case):
    torch = torch_mod()
    L = lib()
    lens = case["lens"]
    w, cu, total, q_np, k_np, v_np, kv = _setup(case["Hq"], case["Hkv"], case["d"], case["bs"], lens, case["kv"],
                                                case["L_max"], seed=6000 + case["d"])
    p = w.params()
    B, Hq, Hkv, d, L_max = len(lens), case["Hq"], case["Hkv"], case["d"], case["L_max"]
    c, s = w.kernel_size, w.kernel_stride
    M = oracle.n_kernels(L_max, c, s)
    q, k, v = to_dev(q_np), to_dev(k_np), to_dev(v_np)
    kv_dev, cu_dev = to_dev(kv), to_dev(cu)
    Tq_max = max(lens)

    # step 1: the chunks' kernels, pooled into an empty kernel cache, against a pool of the whole cache
    kern_full = torch.zeros((B, Hkv, M, d), dtype=torch.bfloat16, device="cuda")
    L.kernel_pool(k, kern_full, 0, L_max, p)
    kern = torch.zeros_like(kern_full)
    L.kernel_pool_varlen(k, kern, kv_dev, cu_dev, Tq_max, p)
    torch.cuda.synchronize()
    assert L.sync_status() == 0
    full, got = bf16_to_np_bits(kern_full), bf16_to_np_bits(kern)
    for b in range(B):
        j_end = oracle.n_kernels(int(kv[b]), c, s)                 # kernels complete after the chunk
        j_beg = oracle.n_kernels(int(kv[b]) - lens[b], c, s)       # ... and before it
        assert np.array_equal(got[b, :, j_beg:j_end], full[b, :, j_beg:j_end]), f"sequence {b}: chunk kernels"
        assert not got[b, :, :j_beg].any() and not got[b, :, j_end:].any(), f"sequence {b}: other kernels touched"
    kern_ref, _ = oracle.kernel_pool(k_np, kv, c, s, M)
    for b in range(B):
        nk = oracle.n_kernels(int(kv[b]), c, s)
        assert np.array_equal(full[b, :, :nk], kern_ref[b, :, :nk])

    # steps 2-3 and 4 on the full kernel cache
    S_cap = L.selection_capacity(p, L_max)
    idx = torch.full((Hkv, total, S_cap), -7, dtype=torch.int32, device="cuda")
    cnt = torch.empty((Hkv, total), dtype=torch.int32, device="cuda")
    ws = torch.empty(L.workspace_size(L.ENTRY_BLOCK_SELECT, 1, total, Hq, Hkv, d, L_max, p), dtype=torch.uint8,
                     device="cuda")
    L.block_select_varlen(q, kern_full, kv_dev, cu_dev, Tq_max, idx, cnt, ws, p, L_max)
    o = torch.empty_like(q)
    lse = torch.empty((Hq, total), dtype=torch.float32, device="cuda")
    L.sparse_attn_fwd_varlen(q, k, v, idx, cnt, kv_dev, cu_dev, Tq_max, o, p, lse=lse)
    o_dense = torch.empty_like(q)
    L.sparse_attn_fwd_varlen(q, k, v, None, None, kv_dev, cu_dev, Tq_max, o_dense, p)
    torch.cuda.synchronize()
    assert L.sync_status() == 0
    gidx_all, gcnt_all = idx.cpu().numpy(), cnt.cpu().numpy()
    o_all, od_all, lse_all = bf16_to_f64(o), bf16_to_f64(o_dense), lse.cpu().numpy()
    for b in range(B):
        n = lens[b]
        if n == 0:
            continue
        r0, r1 = cu[b], cu[b + 1]
        qb = q_np[r0:r1][None]
        kb, vb, kvb = k_np[b:b + 1], v_np[b:b + 1], kv[b:b + 1]
        S = oracle.block_scores(qb, kern_ref[b:b + 1], kvb, Hkv, p)
        oidx, ocnt, kth, _ = oracle.select(S, kvb, n, p, S_max=S_cap)
        gidx = gidx_all[:, r0:r1][None]
        gcnt = gcnt_all[:, r0:r1][None]
        rows, exact, ties, bad = compare_selection(gidx, gcnt, oidx, ocnt, S, kth)
        assert bad == 0, f"sequence {b}: {bad} of {rows} selections differ outside near-ties"
        o_ref, lse_ref = oracle.attention(qb, kb, vb, kvb, gidx, gcnt, p)
        check_output(o_all[r0:r1][None], o_ref, f"o of sequence {b}")
        assert np.max(np.abs(lse_all[:, r0:r1] - lse_ref[0])) < 2e-3
        od_ref, _ = oracle.attention(qb, kb, vb, kvb, None, None, p)
        check_output(od_all[r0:r1][None], od_ref, f"dense o of sequence {b}")
