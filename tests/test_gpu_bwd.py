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


def _bwd_case(w, inp, dense=False):
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
