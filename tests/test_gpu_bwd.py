"""GPU backward of the chunk attention (fixed selection) against the oracle's fp64 backward, on
the same bf16 inputs: the library's own forward (selection, o, lse), a seeded dO, then
infllmv2_sparse_attn_bwd vs oracle.attention_bwd over the same selection.

Tolerance, from the arithmetic: P and dS enter the MMAs as bf16 (relative rounding 2^-9) and D
is formed from the bf16 forward output, every sum in fp32; rounding errors of independent terms
add in quadrature, so an output element sits within ~0.5% of the scale of its terms.  Checked:
max |err| <= 1e-2 * max |ref| and mean |err| <= 5e-3 * mean |ref|, per tensor."""
import numpy as np
import pytest

import oracle
from block_sparse_long_infllm_gb300 import synth

from harness import lib, run_gpu, to_dev, torch_mod

pytestmark = pytest.mark.gpu


def _bf16_as_f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _check(name, got, ref):
    err = np.abs(got - ref)
    mx, mean = float(err.max()), float(err.mean())
    scale_max, scale_mean = float(np.abs(ref).max()), float(np.abs(ref).mean())
    assert mx <= 1e-2 * scale_max and mean <= 5e-3 * scale_mean, (name, mx, scale_max, mean, scale_mean)


def _gpu_bwd(w, inp, dense=False):
    """Forward (selection, o, lse) and backward on the GPU; returns (gpu dict, dq, dk, dv, dout bits)."""
    torch = torch_mod()
    L = lib()
    p = w.params()
    g = run_gpu(w, inp, params=p)
    q, k, v, kv = g["q"], g["k"], g["v"], g["kv_len"]
    o, lse = g["o"], g["lse"]
    idx, cnt = (None, None) if dense else (g["idx"], g["counts"])
    if dense:
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device="cuda")
        L.sparse_attn_fwd(q, k, v, None, None, kv, o, p, lse=lse)
    rng = np.random.default_rng(w.seed + 77)
    dout_bits = synth.f32_to_bf16_bits(rng.standard_normal(inp["q"].shape).astype(np.float32))
    dout = to_dev(dout_bits)
    dq = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    dk = torch.empty(k.shape, dtype=torch.float32, device="cuda")
    dv = torch.empty(v.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(L.workspace_size(L.ENTRY_SPARSE_ATTN_BWD, w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max, p),
                     dtype=torch.uint8, device="cuda")
    L.sparse_attn_bwd(q, k, v, o, lse, dout, idx, cnt, kv, dq, dk, dv, ws, p)
    torch.cuda.synchronize()
    assert L.sync_status() == 0
    return g, dq, dk, dv, dout_bits


def _bwd_case(w, inp, dense=False):
    p = w.params()
    g, dq, dk, dv, dout_bits = _gpu_bwd(w, inp, dense)
    gidx = None if dense else g["idx"].cpu().numpy()
    gcnt = None if dense else g["counts"].cpu().numpy()
    rq, rk, rv = oracle.attention_bwd(_bf16_as_f64(inp["q"]), _bf16_as_f64(inp["k_cache"]),
                                      _bf16_as_f64(inp["v_cache"]), inp["kv_len"], gidx, gcnt, p,
                                      _bf16_as_f64(dout_bits))
    _check("dq", dq.cpu().numpy().astype(np.float64), rq)
    _check("dk", dk.cpu().numpy().astype(np.float64), rk)
    _check("dv", dv.cpu().numpy().astype(np.float64), rv)


def test_bwd_tiny_causal_prefill(cuda_lib):
    w = synth.WORKLOADS["tiny_prefill_2k"]
    _bwd_case(w, synth.make_inputs(w))


@pytest.mark.parametrize("bs", [128, 64])
def test_bwd_group16_ragged_chunk(cuda_lib, bs):
    w = synth.WORKLOADS["chunked_prefill_32k"].scaled(B=2, L=1500, Tq=203, Hq=32, Hkv=2, d=128, block_size=bs,
                                                       topk=4, n_local=2, dense_len=0, seed=4100 + bs)
    inp = synth.make_inputs(w)
    inp["kv_len"] = np.array([1500, 911], dtype=np.int32)
    _bwd_case(w, inp)


def test_bwd_dense_causal(cuda_lib):
    w = synth.WORKLOADS["tiny_prefill_2k"].scaled(L=700, Tq=300, seed=4200)
    _bwd_case(w, synth.make_inputs(w), dense=True)


def test_bwd_group16_several_units_per_block(cuda_lib):
    # token lists longer than one 128-token work unit, tiles ending mid-list
    w = synth.WORKLOADS["chunked_prefill_32k"].scaled(B=1, L=2000, Tq=301, Hq=32, Hkv=2, d=128, block_size=128,
                                                       topk=4, n_local=2, dense_len=0, seed=4300)
    _bwd_case(w, synth.make_inputs(w))


def test_bwd_group16_dense(cuda_lib):
    w = synth.WORKLOADS["chunked_prefill_32k"].scaled(B=1, L=700, Tq=300, Hq=16, Hkv=1, d=128, block_size=128,
                                                       dense_len=0, seed=4400)
    _bwd_case(w, synth.make_inputs(w), dense=True)


def test_bwd_full_chunk_32k_sampled(cuda_lib):
    """The 32K-context, 4096-query chunk: dq rows of sampled tokens against the oracle run on those
    tokens alone, and sum_k dV[k] = sum over the group's query rows of dO (softmax rows sum to 1)
    for every (sequence, KV head) at full size."""
    w = synth.WORKLOADS["chunked_prefill_32k"]
    inp = synth.make_inputs(w)
    p = w.params()
    g, dq, dk, dv, dout_bits = _gpu_bwd(w, inp)
    dout = _bf16_as_f64(dout_bits)
    dv_sum = dv.double().sum(dim=2).cpu().numpy()                  # [B, Hkv, d]
    G = w.Hq // w.Hkv
    do_sum = dout.reshape(w.B, w.Tq, w.Hkv, G, w.d).sum(axis=(1, 3))  # [B, Hkv, d]
    do_abs = np.abs(dout).reshape(w.B, w.Tq, w.Hkv, G, w.d).sum(axis=(1, 3))
    assert np.all(np.abs(dv_sum - do_sum) <= 4e-3 * do_abs + 1e-3), float(np.abs(dv_sum - do_sum).max())
    gidx, gcnt = g["idx"].cpu().numpy(), g["counts"].cpu().numpy()
    q64, k64, v64 = _bf16_as_f64(inp["q"]), _bf16_as_f64(inp["k_cache"]), _bf16_as_f64(inp["v_cache"])
    dq_gpu = dq.cpu().numpy().astype(np.float64)
    got, ref = [], []
    for t in np.random.default_rng(5).choice(w.Tq, 6, replace=False).tolist() + [0, w.Tq - 1]:
        pos = w.L - w.Tq + t
        rq, _, _ = oracle.attention_bwd(q64[:, t:t + 1], k64, v64, np.array([pos + 1], dtype=np.int32),
                                        gidx[:, :, t:t + 1], gcnt[:, :, t:t + 1], p, dout[:, t:t + 1])
        got.append(dq_gpu[:, t])
        ref.append(rq[:, 0])
    _check("dq (sampled tokens)", np.stack(got), np.stack(ref))


def test_bwd_group16_many_units_per_cta(cuda_lib):
    """A chunk whose inverse selection holds several times as many work units (a block and up to
    128 of the tokens that chose it) as the GPU has SMs, so every persistent CTA of the tensor-core
    gradient kernel takes several units in turn (TMEM, barrier phases and the dK/dV reductions
    carried from unit to unit).  dq, dk and dv are compared element by element with the oracle;
    the softmax identity sum_k dV = sum dO is checked beside them."""
    torch = torch_mod()
    w = synth.WORKLOADS["chunked_prefill_32k"].scaled(B=4, L=8192, Tq=256, Hq=64, Hkv=4, d=128, block_size=128,
                                                       topk=16, n_local=4, dense_len=0, seed=4500)
    inp = synth.make_inputs(w)
    inp["kv_len"] = np.array([8192, 7000, 8192 - 37, 6500], dtype=np.int32)
    p = w.params()
    g, dq, dk, dv, dout_bits = _gpu_bwd(w, inp)
    gidx, gcnt = g["idx"].cpu().numpy(), g["counts"].cpu().numpy()
    # work units: per (sequence, KV head, block), the tokens that chose it in slices of 128
    units = 0
    for b in range(w.B):
        for gg in range(w.Hkv):
            per_block = np.bincount(np.concatenate([gidx[b, gg, t, :gcnt[b, gg, t]] for t in range(w.Tq)]))
            units += int(np.sum((per_block + 127) // 128))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert units >= 3 * sms, (units, sms)
    dout = _bf16_as_f64(dout_bits)
    rq, rk, rv = oracle.attention_bwd(_bf16_as_f64(inp["q"]), _bf16_as_f64(inp["k_cache"]),
                                      _bf16_as_f64(inp["v_cache"]), inp["kv_len"], gidx, gcnt, p, dout)
    _check("dq", dq.cpu().numpy().astype(np.float64), rq)
    _check("dk", dk.cpu().numpy().astype(np.float64), rk)
    _check("dv", dv.cpu().numpy().astype(np.float64), rv)
    G = w.Hq // w.Hkv
    dv_sum = dv.double().sum(dim=2).cpu().numpy()
    do_sum = dout.reshape(w.B, w.Tq, w.Hkv, G, w.d).sum(axis=(1, 3))
    do_abs = np.abs(dout).reshape(w.B, w.Tq, w.Hkv, G, w.d).sum(axis=(1, 3))
    assert np.all(np.abs(dv_sum - do_sum) <= 4e-3 * do_abs + 1e-3)
