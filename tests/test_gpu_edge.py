"""GPU edge cases against the oracle: ragged and per-sequence cache lengths,
every supported group size and head dim, both block sizes, the dense switch,
top-k covering every block, dense attention without a selection, wide trees,
queries that are not a multiple of the CTA tile, and device-side error words
(reported, context still usable)."""
import numpy as np
import pytest

import oracle
from block_sparse_long_infllm_gb300 import synth

from harness import (bf16_to_f64, bf16_to_np_bits, check_output, compare_selection, lib, n_kernels,
                     run_gpu, to_dev)

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["decode_32k"]


def _parity(w, inp, params=None):
    p = params or w.params()
    g = run_gpu(w, inp, params=p)
    tree = w.kind == "tree"
    kern_ref, _ = oracle.kernel_pool(inp["k_cache"], inp["kv_len"], w.kernel_size, w.kernel_stride,
                                     max(n_kernels(w), 1))
    kv = inp["kv_len"]
    # kernels past a sequence's own length are not written by the oracle: compare the written ones
    gk = bf16_to_np_bits(g["kern"])
    for b in range(w.B):
        m = oracle.n_kernels(int(kv[b]), w.kernel_size, w.kernel_stride) if w.kind != "prefill" else None
        if m is not None:
            assert np.array_equal(gk[b, :, :m], kern_ref[b, :, :m])
    S = oracle.block_scores(inp["q"], kern_ref, kv, w.Hkv, p, tree=tree,
                            nblk_max=(w.L_max - 1) // w.block_size + 1)
    oidx, ocnt, kth, _ = oracle.select(S, kv, w.Tq, p, tree=tree, S_max=g["S_cap"])
    gidx, gcnt = g["idx"].cpu().numpy(), g["counts"].cpu().numpy()
    rows, exact, ties, bad = compare_selection(gidx, gcnt, oidx, ocnt, S, kth)
    assert bad == 0
    o_ref, lse_ref = oracle.attention(inp["q"], inp["k_cache"], inp["v_cache"], kv, gidx, gcnt, p,
                                      draft_k=inp.get("draft_k"), draft_v=inp.get("draft_v"),
                                      tree_mask=inp.get("tree_mask"))
    check_output(bf16_to_f64(g["o"]), o_ref)
    assert np.max(np.abs(g["lse"].cpu().numpy() - lse_ref)) < 2e-3
    return g, oidx, ocnt


@pytest.mark.parametrize("G,d", [(1, 128), (2, 64), (4, 128), (8, 64), (16, 64)])
def test_decode_group_sizes_and_ragged_lengths(cuda_lib, G, d):
    w = BASE.scaled(B=3, L=4096, Hq=2 * G, Hkv=2, d=d, topk=8, seed=3000 + G + d)
    inp = synth.make_inputs(w)
    inp["kv_len"] = np.array([4096, 4096 - 37, 777], dtype=np.int32)   # ragged last blocks
    w = w.scaled(dense_len=0)
    _parity(w, inp)


@pytest.mark.parametrize("bs", [64, 128])
def test_prefill_block_sizes_ragged_chunk(cuda_lib, bs):
    # 203 queries: not a multiple of the 4-query CTA tile; chunk starts mid-block
    w = synth.WORKLOADS["chunked_prefill_32k"].scaled(L=3000, Tq=203, Hq=8, Hkv=2, block_size=bs,
                                                       topk=3, n_local=2, dense_len=0, seed=3100 + bs)
    inp = synth.make_inputs(w)
    inp["kv_len"] = np.array([3000], dtype=np.int32)
    _parity(w, inp)


def test_prefill_batch_with_different_lengths(cuda_lib):
    w = synth.WORKLOADS["tiny_prefill_2k"].scaled(B=2, L=1500, Tq=100, Hq=4, Hkv=2, d=128, seed=3200)
    inp = synth.make_inputs(w)
    inp["kv_len"] = np.array([1500, 611], dtype=np.int32)
    p = w.params()
    g = run_gpu(w, inp, pool_split=0)
    kern_ref, _ = oracle.kernel_pool(inp["k_cache"], inp["kv_len"], 32, 16, n_kernels(w))
    S = oracle.block_scores(inp["q"], kern_ref, inp["kv_len"], w.Hkv, p)
    oidx, ocnt, kth, _ = oracle.select(S, inp["kv_len"], w.Tq, p, S_max=g["S_cap"])
    gidx, gcnt = g["idx"].cpu().numpy(), g["counts"].cpu().numpy()
    assert compare_selection(gidx, gcnt, oidx, ocnt, S, kth)[3] == 0
    o_ref, _ = oracle.attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["kv_len"], gidx, gcnt, p)
    check_output(bf16_to_f64(g["o"]), o_ref)


def test_dense_switch_and_topk_covering_everything(cuda_lib):
    # kv_len below dense_len: every block; and topk above the block count: also every block
    for kw in (dict(dense_len=5000), dict(dense_len=0, topk=500)):
        w = BASE.scaled(L=4096, seed=3300, **kw)
        inp = synth.make_inputs(w)
        g, oidx, ocnt = _parity(w, inp)
        assert np.all(g["counts"].cpu().numpy() == 64)
        assert np.array_equal(g["idx"].cpu().numpy()[0, 0, 0, :64], np.arange(64))


def test_dense_prefill_without_selection(cuda_lib):
    torch = pytest.importorskip("torch")
    L = lib()
    w = synth.WORKLOADS["tiny_prefill_2k"].scaled(L=700, Tq=130, Hq=4, Hkv=1, d=128, seed=3400)
    inp = synth.make_inputs(w)
    q, k, v, kv = (to_dev(inp[x]) for x in ("q", "k_cache", "v_cache", "kv_len"))
    o = torch.empty_like(q)
    L.sparse_attn_fwd(q, k, v, None, None, kv, o, w.params())
    torch.cuda.synchronize()
    assert L.sync_status() == 0
    o_ref, _ = oracle.attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["kv_len"], None, None, w.params())
    check_output(bf16_to_f64(o), o_ref)


@pytest.mark.parametrize("n_draft", [1, 40, 64])
def test_tree_widths(cuda_lib, n_draft):
    w = synth.WORKLOADS["tree_verify_64k"].scaled(B=2, L=5000, Tq=n_draft, topk=6, seed=3500 + n_draft,
                                                  tree_depth=8)
    inp = synth.make_inputs(w)
    inp["kv_len"] = np.array([5000, 4321], dtype=np.int32)
    _parity(w, inp)


def test_device_index_error_is_reported_and_context_survives(cuda_lib):
    torch = pytest.importorskip("torch")
    L = lib()
    w = BASE.scaled(L=2048, seed=3600)
    inp = synth.make_inputs(w)
    p = w.params()
    q, k, v = (to_dev(inp[x]) for x in ("q", "k_cache", "v_cache"))
    kern = torch.zeros((1, 2, n_kernels(w), 128), dtype=torch.bfloat16, device="cuda")
    L.kernel_pool(k, kern, 0, w.L, p)
    ws = torch.empty(L.workspace_size(L.ENTRY_DECODE, 1, 1, 32, 2, 128, w.L_max, p), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(q)
    bad_len = torch.tensor([w.L_max + 5], dtype=torch.int32, device="cuda")   # past the cache
    L.decode(q, k, v, kern, bad_len, o, ws, p)
    assert L.sync_status() == L.ERR_DEVICE_INDEX
    assert L.sync_status() == 0                                            # cleared once read
    # a selected block past the query's own block
    idx = torch.full((1, 2, 1, L.selection_capacity(p, w.L_max)), -1, dtype=torch.int32, device="cuda")
    idx[..., 0] = 40
    counts = torch.ones((1, 2, 1), dtype=torch.int32, device="cuda")
    kv = torch.tensor([100], dtype=torch.int32, device="cuda")
    L.sparse_attn_fwd(q, k, v, idx, counts, kv, o, p)
    assert L.sync_status() == L.ERR_DEVICE_INDEX
    good = to_dev(inp["kv_len"])
    L.decode(q, k, v, kern, good, o, ws, p)
    assert L.sync_status() == 0


def test_bad_arguments_raise(cuda_lib):
    torch = pytest.importorskip("torch")
    L = lib()
    w = BASE.scaled(L=1024, seed=3700)
    inp = synth.make_inputs(w)
    q, k, v, kv = (to_dev(inp[x]) for x in ("q", "k_cache", "v_cache", "kv_len"))
    kern = torch.zeros((1, 2, n_kernels(w), 128), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(L.InfLLMv2Error) as e:
        L.decode(q, k, v, kern, kv, o, small, w.params())
    assert e.value.status == L.ERR_WORKSPACE
    with pytest.raises(L.InfLLMv2Error) as e:
        L.kernel_pool(k, kern[:, :, :3].contiguous(), 0, w.L, w.params())
    assert e.value.status == L.ERR_INVALID_ARG


@pytest.mark.parametrize("bs,d", [(128, 128), (64, 128), (64, 64), (128, 64)])
def test_prefill_group16_tensor_core_path(cuda_lib, bs, d):
    # 16 heads per KV head take the tcgen05 path; 203 queries leave a ragged last tile of 8,
    # two sequences of different lengths, selection wider than one tile's union
    w = synth.WORKLOADS["chunked_prefill_32k"].scaled(B=2, L=2500, Tq=203, Hq=32, Hkv=2, d=d, block_size=bs,
                                                       topk=4, n_local=2, dense_len=0, seed=3800 + bs + d)
    inp = synth.make_inputs(w)
    inp["kv_len"] = np.array([2500, 1311], dtype=np.int32)
    p = w.params()
    g = run_gpu(w, inp, pool_split=0, params=p)
    kern_ref, _ = oracle.kernel_pool(inp["k_cache"], inp["kv_len"], 32, 16, n_kernels(w))
    S = oracle.block_scores(inp["q"], kern_ref, inp["kv_len"], w.Hkv, p)
    oidx, ocnt, kth, _ = oracle.select(S, inp["kv_len"], w.Tq, p, S_max=g["S_cap"])
    gidx, gcnt = g["idx"].cpu().numpy(), g["counts"].cpu().numpy()
    assert compare_selection(gidx, gcnt, oidx, ocnt, S, kth)[3] == 0
    o_ref, lse_ref = oracle.attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["kv_len"], gidx, gcnt, p)
    check_output(bf16_to_f64(g["o"]), o_ref)
    assert np.max(np.abs(g["lse"].cpu().numpy() - lse_ref)) < 2e-3


def test_prefill_group16_dense_without_selection(cuda_lib):
    torch = pytest.importorskip("torch")
    L = lib()
    w = synth.WORKLOADS["chunked_prefill_32k"].scaled(L=1000, Tq=77, Hq=16, Hkv=1, d=128, block_size=64,
                                                       seed=3900)
    inp = synth.make_inputs(w)
    q, k, v, kv = (to_dev(inp[x]) for x in ("q", "k_cache", "v_cache", "kv_len"))
    o = torch.empty_like(q)
    L.sparse_attn_fwd(q, k, v, None, None, kv, o, w.params())
    torch.cuda.synchronize()
    assert L.sync_status() == 0
    o_ref, _ = oracle.attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["kv_len"], None, None, w.params())
    check_output(bf16_to_f64(o), o_ref)


@pytest.mark.parametrize("bs", [128, 64])
def test_prefill_group16_short_unions(cuda_lib, bs):
    # a chunk that starts an empty cache: tiles see unions of 1, 2, 3 ... blocks, the shortest
    # pipelines of the tensor-core path (fewer blocks than S buffers and K stages)
    w = synth.WORKLOADS["chunked_prefill_32k"].scaled(B=1, L=300, Tq=300, Hq=16, Hkv=1, d=128, block_size=bs,
                                                       topk=2, n_init=1, n_local=1, dense_len=0, seed=3950 + bs)
    inp = synth.make_inputs(w)
    p = w.params()
    g = run_gpu(w, inp, pool_split=0, params=p)
    kern_ref, _ = oracle.kernel_pool(inp["k_cache"], inp["kv_len"], 32, 16, n_kernels(w))
    S = oracle.block_scores(inp["q"], kern_ref, inp["kv_len"], w.Hkv, p)
    oidx, ocnt, kth, _ = oracle.select(S, inp["kv_len"], w.Tq, p, S_max=g["S_cap"])
    gidx, gcnt = g["idx"].cpu().numpy(), g["counts"].cpu().numpy()
    assert compare_selection(gidx, gcnt, oidx, ocnt, S, kth)[3] == 0
    o_ref, lse_ref = oracle.attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["kv_len"], gidx, gcnt, p)
    check_output(bf16_to_f64(g["o"]), o_ref)
    assert np.max(np.abs(g["lse"].cpu().numpy() - lse_ref)) < 2e-3


@pytest.mark.parametrize("bs", [64, 128])
def test_decode_tied_scores_take_lowest_blocks(cuda_lib, bs):
    # every semantic kernel equal (zero): all candidate blocks tie, so the selection is the
    # forced blocks plus the lowest-numbered candidates, exactly
    torch = pytest.importorskip("torch")
    L = lib()
    w = BASE.scaled(B=2, L=20000, block_size=bs, topk=16, dense_len=0, seed=3960 + bs)
    inp = synth.make_inputs(w)
    inp["kv_len"] = np.array([20000, 13001], dtype=np.int32)
    p = w.params()
    q, k, v, kv = (to_dev(inp[x]) for x in ("q", "k_cache", "v_cache", "kv_len"))
    M = max(n_kernels(w), 1)
    kern = torch.zeros((w.B, w.Hkv, M, w.d), dtype=torch.bfloat16, device="cuda")
    S_cap = L.selection_capacity(p, w.L_max)
    idx = torch.empty((w.B, w.Hkv, 1, S_cap), dtype=torch.int32, device="cuda")
    cnt = torch.empty((w.B, w.Hkv, 1), dtype=torch.int32, device="cuda")
    ws = torch.empty(L.workspace_size(L.ENTRY_DECODE, w.B, 1, w.Hq, w.Hkv, w.d, w.L_max, p),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device="cuda")
    L.decode(q, k, v, kern, kv, o, ws, p, lse=lse, idx_out=idx, counts_out=cnt)
    torch.cuda.synchronize()
    assert L.sync_status() == 0
    kern_ref = np.zeros((w.B, w.Hkv, M, w.d), dtype=np.uint16)
    S = oracle.block_scores(inp["q"], kern_ref, inp["kv_len"], w.Hkv, p,
                            nblk_max=(w.L_max - 1) // w.block_size + 1)
    oidx, ocnt, _, _ = oracle.select(S, inp["kv_len"], 1, p, S_max=S_cap)
    gidx, gcnt = idx.cpu().numpy(), cnt.cpu().numpy()
    assert np.array_equal(gcnt, ocnt)
    for b in range(w.B):
        for g in range(w.Hkv):
            n = int(ocnt[b, g, 0])
            assert sorted(gidx[b, g, 0, :n].tolist()) == sorted(oidx[b, g, 0, :n].tolist())
    o_ref, lse_ref = oracle.attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["kv_len"], gidx, gcnt, p)
    check_output(bf16_to_f64(o), o_ref)
    assert np.max(np.abs(lse.cpu().numpy() - lse_ref)) < 2e-3


@pytest.mark.parametrize("decisive", [False, True], ids=["as_written", "decisive"])
def test_decode_output_without_selection_list(cuda_lib, decisive):
    # The single-kernel decode may attend to a candidate-ordered list and skip building the
    # block-ordered selection when the caller does not ask for it: o and lse must be the same
    # bits with and without idx_out, and match the oracle over the oracle's own selection.
    import torch
    w = synth.WORKLOADS["decode_128k_b4"].scaled(B=2, L=65536, seed=3400 + int(decisive))
    inp = synth.make_inputs(w, decisive=decisive)
    g, oidx, ocnt = _parity(w, inp)
    L = lib()
    p = w.params()
    o2 = torch.empty_like(g["o"])
    lse2 = torch.empty_like(g["lse"])
    ws = torch.empty(L.workspace_size(L.ENTRY_DECODE, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, p),
                     dtype=torch.uint8, device="cuda")
    L.decode(g["q"], g["k"], g["v"], g["kern"], g["kv_len"], o2, ws, p, lse=lse2)
    torch.cuda.synchronize()
    assert L.sync_status() == 0
    assert torch.equal(o2.view(torch.int16), g["o"].view(torch.int16))
    assert torch.equal(lse2, g["lse"])
    o_ref, lse_ref = oracle.attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["kv_len"], oidx, ocnt, p)
    check_output(bf16_to_f64(o2), o_ref)


def test_decode_host_buffers_match_device_call(cuda_lib):
    # infllmv2_decode_host: the same step with q, kv_len, o and lse in pinned host memory gives the
    # same bits as the device-buffer call, and matches the oracle
    import torch
    w = synth.WORKLOADS["decode_128k_b4"].scaled(B=2, L=32768, seed=3500)
    inp = synth.make_inputs(w)
    g, oidx, ocnt = _parity(w, inp)
    L = lib()
    p = w.params()
    ws = torch.empty(L.workspace_size(L.ENTRY_DECODE, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, p),
                     dtype=torch.uint8, device="cuda")
    q_host = g["q"].view(w.B, w.Hq, w.d).cpu().pin_memory()
    kv_host = g["kv_len"].cpu().pin_memory()
    o_host = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16).pin_memory()
    lse_host = torch.empty((w.B, w.Hq), dtype=torch.float32).pin_memory()
    q_dev = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    kv_dev = torch.empty_like(g["kv_len"])
    o_dev = torch.empty_like(q_dev)
    lse_dev = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
    L.decode_host(q_host, kv_host, o_host, q_dev, kv_dev, o_dev, g["k"], g["v"], g["kern"], ws, p,
                  lse_host=lse_host, lse_dev=lse_dev)
    assert torch.equal(o_host.view(torch.int16), g["o"].view(w.B, w.Hq, w.d).cpu().view(torch.int16))
    assert torch.equal(lse_host, g["lse"].view(w.B, w.Hq).cpu())
    # the prepared call (buffers bound once) gives the same bits
    o_host.zero_()
    step = L.DecodeHostStep(q_host, kv_host, o_host, q_dev, kv_dev, o_dev, g["k"], g["v"], g["kern"], ws, p,
                            lse_host=lse_host, lse_dev=lse_dev)
    step()
    step()
    assert torch.equal(o_host.view(torch.int16), g["o"].view(w.B, w.Hq, w.d).cpu().view(torch.int16))
    o_ref, _ = oracle.attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["kv_len"], oidx, ocnt, p)
    check_output(bf16_to_f64(o_host.view(w.B, 1, w.Hq, w.d)), o_ref)


@pytest.mark.parametrize("B,Hkv,G,L", [(8, 2, 16, 16384), (12, 4, 4, 8192), (3, 8, 2, 4096)])
def test_decode_many_rows_smaller_clusters(cuda_lib, B, Hkv, G, L):
    # more (sequence, KV head) rows than 12-CTA clusters fit at once: the single-kernel decode
    # takes the largest smaller cluster whose clusters all fit (16 rows: 9 or 10 CTAs on a GB300;
    # 24 and 48 rows: fewer), each CTA then merging more heads and scoring more blocks
    w = BASE.scaled(B=B, L=L, Hq=G * Hkv, Hkv=Hkv, topk=16, dense_len=0, seed=3600 + B + Hkv + G)
    inp = synth.make_inputs(w)
    inp["kv_len"] = np.array([L - 97 * i for i in range(B)], dtype=np.int32)   # per-sequence lengths
    _parity(w, inp)


@pytest.mark.parametrize("B,L", [(1, 262144), (16, 65536)], ids=["256k_rows_over_2048_blocks", "32_rows_at_64k"])
def test_decode_multi_pass_scoring_and_long_rows(cuda_lib, B, L):
    # 256K tokens: 4096 blocks per row, past the fast selection path (the two-bit general search
    # takes over) and several scoring passes per CTA; 32 rows at 64K: clusters of 4 CTAs, each
    # scoring its 256 blocks in two passes
    w = synth.WORKLOADS["decode_128k_b4"].scaled(B=B, L=L, seed=3700 + B)
    inp = synth.make_inputs(w)
    if B > 1:
        inp["kv_len"] = np.array([L - 131 * i for i in range(B)], dtype=np.int32)
    _parity(w, inp)


def test_decode_host_reports_device_errors(cuda_lib):
    # a cache length past the cache, staged from host memory: the host-buffer call returns the
    # device error (and clears the word); the next call with good lengths succeeds
    import torch
    L = lib()
    w = BASE.scaled(L=2048, seed=3800)
    inp = synth.make_inputs(w)
    p = w.params()
    k, v = to_dev(inp["k_cache"]), to_dev(inp["v_cache"])
    kern = torch.zeros((1, 2, n_kernels(w), 128), dtype=torch.bfloat16, device="cuda")
    L.kernel_pool(k, kern, 0, w.L, p)
    ws = torch.empty(L.workspace_size(L.ENTRY_DECODE, 1, 1, 32, 2, 128, w.L_max, p), dtype=torch.uint8,
                     device="cuda")
    q_host = torch.from_numpy(np.ascontiguousarray(inp["q"]).view(np.int16)).view(torch.bfloat16).view(1, 32, 128)
    q_host = q_host.pin_memory()
    o_host = torch.empty((1, 32, 128), dtype=torch.bfloat16).pin_memory()
    q_dev = torch.empty((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    o_dev = torch.empty_like(q_dev)
    kv_dev = torch.empty(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([w.L_max + 5], dtype=torch.int32).pin_memory()
    with pytest.raises(L.InfLLMv2Error) as e:
        L.decode_host(q_host, bad, o_host, q_dev, kv_dev, o_dev, k, v, kern, ws, p)
    assert e.value.status == L.ERR_DEVICE_INDEX
    assert L.sync_status() == 0                                   # cleared by the call
    good = torch.from_numpy(inp["kv_len"]).pin_memory()
    L.decode_host(q_host, good, o_host, q_dev, kv_dev, o_dev, k, v, kern, ws, p)
    assert L.sync_status() == 0


def test_decode_host_pageable_and_page_locked_buffers(cuda_lib):
    # page-locked host buffers take the zero-copy way; pageable ones take it too where the device
    # reads host memory through the host's page tables (Grace), else they are staged through the
    # caller's device buffers; every way gives the same bits as the device-buffer call
    import torch
    w = synth.WORKLOADS["decode_128k_b4"].scaled(B=2, L=16384, seed=3900)
    inp = synth.make_inputs(w)
    g = run_gpu(w, inp)
    L = lib()
    p = w.params()
    ws = torch.empty(L.workspace_size(L.ENTRY_DECODE, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, p),
                     dtype=torch.uint8, device="cuda")
    ref_o = g["o"].view(w.B, w.Hq, w.d).cpu().view(torch.int16)
    ref_lse = g["lse"].view(w.B, w.Hq).cpu()
    direct = L.host_memory_direct()
    for pinned in (False, True):
        q_host = g["q"].view(w.B, w.Hq, w.d).cpu()
        kv_host = g["kv_len"].cpu()
        o_host = torch.zeros((w.B, w.Hq, w.d), dtype=torch.bfloat16)
        lse_host = torch.zeros((w.B, w.Hq), dtype=torch.float32)
        if pinned:
            q_host, kv_host, o_host, lse_host = (t.pin_memory() for t in (q_host, kv_host, o_host, lse_host))
        q_dev = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
        kv_dev = torch.empty_like(g["kv_len"])
        o_dev = torch.full_like(q_dev, float("nan"))
        lse_dev = torch.empty((w.B, w.Hq), dtype=torch.float32, device="cuda")
        L.decode_host(q_host, kv_host, o_host, q_dev, kv_dev, o_dev, g["k"], g["v"], g["kern"], ws, p,
                      lse_host=lse_host, lse_dev=lse_dev)
        assert torch.equal(o_host.view(torch.int16), ref_o), f"pinned={pinned}"
        assert torch.equal(lse_host, ref_lse), f"pinned={pinned}"
        # the staged call used the staging buffers; the zero-copy one left them alone
        assert bool(torch.isnan(o_dev.float()).any()) == (pinned or direct), f"pinned={pinned} direct={direct}"
    assert L.sync_status() == 0


@pytest.mark.parametrize("L", [5000, 40000], ids=["short_rows_bitwise", "long_rows_radix"])
def test_tree_fully_tied_scores_take_the_lowest_blocks(cuda_lib, L):
    # zero semantic kernels: every candidate block of every draft ties, so each draft's selection
    # is its forced blocks plus the lowest-numbered candidates -- through the separate top-k kernel
    # on rows of 79 blocks (bit-by-bit threshold) and of 625 blocks (radix select)
    torch = pytest.importorskip("torch")
    Lb = lib()
    w = synth.WORKLOADS["tree_verify_64k"].scaled(B=1, L=L, Tq=12, topk=16, seed=3980 + L % 97)
    inp = synth.make_inputs(w)
    p = w.params()
    q, k, v, kv = (to_dev(inp[x]) for x in ("q", "k_cache", "v_cache", "kv_len"))
    dk, dv, mask = to_dev(inp["draft_k"]), to_dev(inp["draft_v"]), to_dev(inp["tree_mask"])
    M = max(n_kernels(w), 1)
    kern = torch.zeros((w.B, w.Hkv, M, w.d), dtype=torch.bfloat16, device="cuda")
    S_cap = Lb.selection_capacity(p, w.L_max)
    idx = torch.empty((w.B, w.Hkv, w.Tq, S_cap), dtype=torch.int32, device="cuda")
    cnt = torch.empty((w.B, w.Hkv, w.Tq), dtype=torch.int32, device="cuda")
    ws = torch.empty(Lb.workspace_size(Lb.ENTRY_DECODE, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, p),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    Lb.decode(q, k, v, kern, kv, o, ws, p, draft_k=dk, draft_v=dv, tree_mask=mask, idx_out=idx, counts_out=cnt)
    torch.cuda.synchronize()
    assert Lb.sync_status() == 0
    kern_ref = np.zeros((w.B, w.Hkv, M, w.d), dtype=np.uint16)
    S = oracle.block_scores(inp["q"], kern_ref, inp["kv_len"], w.Hkv, p, tree=True)
    oidx, ocnt, _, _ = oracle.select(S, inp["kv_len"], w.Tq, p, tree=True, S_max=S_cap)
    gidx, gcnt = idx.cpu().numpy(), cnt.cpu().numpy()
    assert np.array_equal(gcnt, ocnt)
    for t in range(w.Tq):
        for g in range(w.Hkv):
            n = int(ocnt[0, g, t])
            assert gidx[0, g, t, :n].tolist() == oidx[0, g, t, :n].tolist()
    o_ref, _ = oracle.attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["kv_len"], gidx, gcnt, p,
                                draft_k=inp["draft_k"], draft_v=inp["draft_v"], tree_mask=inp["tree_mask"])
    check_output(bf16_to_f64(o), o_ref)


@pytest.mark.parametrize("bs,c,s,d", [
    (128, 32, 16, 128),  # 8 kernels per block, one past the group: the shuffle pass (prefill shape)
    (64, 32, 16, 64),    # 4 per block, one past
    (128, 16, 16, 128),  # kernels as wide as the stride: no lane past the group
    (64, 64, 16, 128),   # three past the group (the most the shuffle pass takes)
    (128, 40, 16, 64),   # kernel not a multiple of the stride, two past
    (128, 32, 32, 128),  # 4 per block, kernel = stride
    (128, 32, 24, 128),  # block not a multiple of the stride: the shared-memory pass
    (64, 64, 8, 128),    # seven past the group: the shared-memory pass
    (128, 16, 8, 128),   # 16 per block: the shuffle pass with a fourth exchange step
    (128, 12, 4, 64),    # 32 per block (a whole lane quarter), two past
    (64, 48, 32, 128),   # 2 per block: the shared-memory pass
])
def test_chunk_block_scores_for_kernel_shapes(cuda_lib, bs, c, s, d):
    # the tensor-core scorer's block scores (16 heads per KV head), read from the start of the
    # workspace, against the oracle's for every visible block of every query; two sequences of
    # different lengths and a ragged last tile of 11 queries
    w = synth.WORKLOADS["chunked_prefill_32k"].scaled(B=2, L=3000, Tq=203, Hq=32, Hkv=2, d=d, block_size=bs,
                                                       kernel_size=c, kernel_stride=s, topk=4, n_local=2,
                                                       dense_len=0, seed=4600 + bs + c + s + d)
    inp = synth.make_inputs(w)
    inp["kv_len"] = np.array([3000, 1777], dtype=np.int32)
    p = w.params()
    g = run_gpu(w, inp, pool_split=0, params=p)
    kern_ref, _ = oracle.kernel_pool(inp["k_cache"], inp["kv_len"], c, s, n_kernels(w))
    nblk = (w.L_max - 1) // bs + 1
    S = oracle.block_scores(inp["q"], kern_ref, inp["kv_len"], w.Hkv, p, nblk_max=nblk)
    Sg = g["ws"][: w.B * w.Hkv * w.Tq * nblk * 4].view(dtype=__import__("torch").float32).cpu().numpy()
    Sg = Sg.reshape(w.B, w.Hkv, w.Tq, nblk)
    checked = 0
    for b in range(w.B):
        for t in range(w.Tq):
            bt = (int(inp["kv_len"][b]) - w.Tq + t) // bs
            ref, got = S[b, :, t, :bt + 1], Sg[b, :, t, :bt + 1].astype(np.float64)
            fin = np.isfinite(ref)
            assert np.array_equal(fin, np.isfinite(got)), (b, t)
            assert np.array_equal(ref[~fin], got[~fin]), (b, t)
            assert np.max(np.abs(ref[fin] - got[fin]), initial=0.0) < 1e-3, (b, t)
            checked += int(fin.sum())
    assert checked > 0
    oidx, ocnt, kth, _ = oracle.select(S, inp["kv_len"], w.Tq, p, S_max=g["S_cap"])
    assert compare_selection(g["idx"].cpu().numpy(), g["counts"].cpu().numpy(), oidx, ocnt, S, kth)[3] == 0
