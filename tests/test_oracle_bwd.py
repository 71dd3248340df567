"""Pins of the oracle's attention backward (gradients of sum(dO * O) with the selection held
fixed; "MiniCPM4：如何在手机电脑上高效运行大语言模型", section 1.1: InfLLM v2 is trainable, the
attention runs over the selected blocks only).  Each pin is independent of the backward's own
formulas: central finite differences of the oracle's fp64 forward, conservation identities of
the softmax, and the dense case against the matrix form of attention's gradient."""
import numpy as np
import pytest

import oracle


def _params(bs):
    return dict(block_size=bs, kernel_size=32, kernel_stride=16, topk=1, n_init_blocks=1,
                n_local_blocks=1, dense_len=0)


def _case(seed, B, Tq, L, Hq, Hkv, d, bs, partial_selection=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Tq, Hq, d))
    k = rng.standard_normal((B, Hkv, L, d))
    v = rng.standard_normal((B, Hkv, L, d))
    do = rng.standard_normal((B, Tq, Hq, d))
    kv = np.full(B, L, dtype=np.int32)
    nblk = (L + bs - 1) // bs
    idx = np.full((B, Hkv, Tq, nblk), -1, dtype=np.int32)
    cnt = np.zeros((B, Hkv, Tq), dtype=np.int32)
    for b in range(B):
        for g in range(Hkv):
            for t in range(Tq):
                bt = (L - Tq + t) // bs
                blocks = [x for x in range(bt + 1) if not partial_selection or x == bt or rng.random() < 0.5]
                idx[b, g, t, :len(blocks)] = blocks
                cnt[b, g, t] = len(blocks)
    return q, k, v, do, kv, idx, cnt


def _loss(q, k, v, kv, idx, cnt, p, do):
    o, _ = oracle.attention_f64(q, k, v, kv, idx, cnt, p)
    return float(np.sum(o * do))


@pytest.mark.parametrize("shape", [
    dict(B=1, Tq=24, L=24, Hq=2, Hkv=1, d=4, bs=8),    # causal from an empty cache
    dict(B=2, Tq=7, L=29, Hq=4, Hkv=2, d=3, bs=8),     # ragged chunk after a cached prefix, GQA
    dict(B=1, Tq=1, L=40, Hq=2, Hkv=1, d=4, bs=16),    # a decode row
])
def test_gradients_match_finite_differences(shape):
    q, k, v, do, kv, idx, cnt = _case(7, shape["B"], shape["Tq"], shape["L"], shape["Hq"], shape["Hkv"],
                                      shape["d"], shape["bs"])
    p = _params(shape["bs"])
    dq, dk, dv = oracle.attention_bwd(q, k, v, kv, idx, cnt, p, do)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        flat, nflat = x.reshape(-1), num.reshape(-1)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + eps
            up = _loss(q, k, v, kv, idx, cnt, p, do)
            flat[i] = keep - eps
            dn = _loss(q, k, v, kv, idx, cnt, p, do)
            flat[i] = keep
            nflat[i] = (up - dn) / (2 * eps)
        assert np.max(np.abs(num - g)) < 1e-6 * (1 + np.max(np.abs(g))), name


def test_softmax_conservation():
    # each row's weights sum to one: the dS of a row sums to zero, so dK summed over the keys is
    # zero, and dV summed over the keys is the sum of dO over the group's rows
    q, k, v, do, kv, idx, cnt = _case(11, 2, 9, 33, 4, 2, 5, 8)
    dq, dk, dv = oracle.attention_bwd(q, k, v, kv, idx, cnt, _params(8), do)
    assert np.max(np.abs(dk.sum(axis=2))) < 1e-10
    want = do.reshape(2, 9, 2, 2, 5).sum(axis=(1, 3))
    assert np.max(np.abs(dv.sum(axis=2) - want)) < 1e-10


def test_dense_causal_equals_matrix_form():
    # no selection: dense causal attention, whose gradient in matrix form is
    # dV = P^T dO, dP = dO V^T, dS = P o (dP - rowsum(dO o O)), dQ = s dS K, dK = s dS^T Q
    B, T, H, d = 1, 12, 1, 6
    rng = np.random.default_rng(5)
    q, k, v, do = (rng.standard_normal((B, T, H, d)) for _ in range(4))
    kk, vv = k.transpose(0, 2, 1, 3).copy(), v.transpose(0, 2, 1, 3).copy()
    kv = np.array([T], dtype=np.int32)
    dq, dk, dv = oracle.attention_bwd(q, kk, vv, kv, None, None, _params(4), do)
    s = 1 / np.sqrt(d)
    Q, K, V, dO = q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0]
    Z = s * Q @ K.T + np.triu(np.full((T, T), -np.inf), 1)
    P = np.exp(Z - Z.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    O = P @ V
    dP = dO @ V.T
    dS = P * (dP - (dO * O).sum(axis=1, keepdims=True))
    assert np.allclose(dq[0, :, 0], s * dS @ K, atol=1e-12)
    assert np.allclose(dk[0, 0], s * dS.T @ Q, atol=1e-12)
    assert np.allclose(dv[0, 0], P.T @ dO, atol=1e-12)
