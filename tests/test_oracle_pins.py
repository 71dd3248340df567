"""Pins for the fp64 oracle: each check ties one oracle function to something
other than itself -- exact rational arithmetic, hand-derived cases, brute force
with Python sets and sorting on tiny inputs, the textbook dense softmax in
matrix form, and the invariants the method fixes (forced blocks present,
weights non-negative and summing to one, planted blocks recovered).

Sources: "MiniCPM4: 如何在手机电脑上高效运行大语言模型" (xugj520.cn) section 1.1
"InfLLM v2" (32-token kernels with stride 16, top-K blocks, initial and
sliding-window tokens kept, uint64 tree mask); "MiniCPM40极速狂飙端侧模型的比赛
结束了" (shadowrocket9.top) section "InfLLM v2：重新定义注意力机制" (64-token
blocks, top-64, dense below 8192 tokens).
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
from block_sparse_long_infllm_gb300 import synth

F32_TO_BF16 = synth.f32_to_bf16_bits
BF16_TO_F32 = synth.bf16_bits_to_f32


def bf16_bits_exact(x) -> int:
    """Nearest bf16 (ties to even) of a rational, by exact integer arithmetic."""
    a = Fraction(x)
    if a == 0:
        return 0
    neg = a < 0
    a = abs(a)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e <= a:
        e += 1
    while Fraction(2) ** (e - 1) > a:
        e -= 1
    ulp = Fraction(2) ** (e - 8)            # 8 significant bits: a / ulp in [128, 256)
    r = round(a / ulp)                       # Fraction rounding: half to even
    v = float(r * ulp)
    bits = struct.unpack(">I", struct.pack(">f", v))[0] >> 16
    return bits | (0x8000 if neg else 0)


def params(**kw):
    p = dict(block_size=64, kernel_size=32, kernel_stride=16, topk=4, n_init_blocks=1,
             n_local_blocks=2, dense_len=0, softmax_scale=0.0)
    p.update(kw)
    return p


def rand_bf16(rng, shape, scale=1.0):
    return F32_TO_BF16((rng.standard_normal(shape) * scale).astype(np.float32))


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_round_hand_cases():
    one = 1.0
    cases = {
        one: 0x3F80,
        one + 2.0 ** -8: 0x3F80,            # exact tie, even neighbour is 1.0
        one + 3 * 2.0 ** -8: 0x3F82,        # exact tie, even neighbour is 1 + 2^-6
        one + 2.0 ** -8 + 2.0 ** -30: 0x3F81,  # just above the tie rounds up
        -1.5: 0xBFC0,
        255.5: 0x4380,                      # 8 bits: 255.5 -> 256
        0.0: 0x0000,
    }
    xs = np.array(list(cases), dtype=np.float64)
    got = oracle.bf16_round(xs)
    assert [int(g) for g in got] == list(cases.values())


def test_bf16_round_matches_exact_rationals():
    rng = np.random.default_rng(7)
    xs = np.concatenate([rng.standard_normal(400) * 10.0 ** rng.integers(-6, 6, 400),
                         # values sitting exactly on a rounding midpoint
                         (rng.integers(128, 256, 200) + 0.5) * 2.0 ** rng.integers(-20, 20, 200)])
    got = oracle.bf16_round(xs)
    want = [bf16_bits_exact(x) for x in xs]
    assert [int(g) for g in got] == want
    # float32-representable values also agree with the integer bit trick
    xf = xs.astype(np.float32).astype(np.float64)
    assert np.array_equal(oracle.bf16_round(xf), F32_TO_BF16(xf.astype(np.float32)))


# ---------------------------------------------------------------- step 1: kernels

def test_kernel_count_and_only_complete_kernels_written():
    rng = np.random.default_rng(1)
    k = rand_bf16(rng, (2, 1, 100, 8))
    kv_len = np.array([100, 47], dtype=np.int32)
    kern, _ = oracle.kernel_pool(k, kv_len, 32, 16, 8)
    # kernels ending inside 100 tokens: starts 0,16,...,64 -> 5; inside 47: start 0 only
    assert oracle.n_kernels(100, 32, 16) == 5 and oracle.n_kernels(47, 32, 16) == 1
    assert oracle.n_kernels(31, 32, 16) == 0 and oracle.n_kernels(32, 32, 16) == 1
    assert np.all(kern[0, 0, 5:] == 0) and np.all(kern[1, 0, 1:] == 0)
    assert np.any(kern[0, 0, 4] != 0) and np.any(kern[1, 0, 0] != 0)


def test_kernel_means_exact_rational():
    rng = np.random.default_rng(2)
    L, d = 160, 4
    k = rand_bf16(rng, (1, 2, L, d), scale=3.0)
    kern, exact = oracle.kernel_pool(k, np.array([L], np.int32), 32, 16, 16)
    kf = BF16_TO_F32(k).astype(np.float64)
    M = oracle.n_kernels(L, 32, 16)
    for h in range(2):
        for j in range(M):
            toks = list(range(16 * j, 16 * j + 32))       # kernel j: 32 tokens from 16*j
            for x in range(d):
                mean = sum(Fraction(float(kf[0, h, i, x])) for i in toks) / 32
                assert exact[0, h, j, x] == float(mean)
                assert int(kern[0, h, j, x]) == bf16_bits_exact(mean)


def test_kernel_pool_ramp():
    # K[i, :] = i/64 (exact in bf16 for i < 256): window mean = (16 j + 15.5) / 64
    L = 256
    ramp = (np.arange(L, dtype=np.float32) / 64.0)[:, None].repeat(2, axis=1)
    k = F32_TO_BF16(ramp)[None, None]
    kern, exact = oracle.kernel_pool(k, np.array([L], np.int32), 32, 16, 15)
    for j in range(15):
        assert exact[0, 0, j, 0] == (16 * j + 15.5) / 64.0
        assert int(kern[0, 0, j, 1]) == bf16_bits_exact(Fraction(32 * j + 31, 128))


# ---------------------------------------------------------------- step 2: block scores

def _one_hot_kernel_setup(M, d, hot, big=8.0):
    kern = np.zeros((1, 1, M, d), dtype=np.uint16)
    kern[0, 0, hot, 0] = F32_TO_BF16(np.array([big], np.float32))[0]
    q = np.zeros((1, 1, 1, d), dtype=np.uint16)
    q[0, 0, 0, 0] = F32_TO_BF16(np.array([1.0], np.float32))[0]
    return q, kern


@pytest.mark.parametrize("bs,hot,blocks", [
    (64, 0, {0}), (64, 3, {0, 1}), (64, 4, {1}), (64, 7, {1, 2}), (64, 8, {2}),
    (128, 7, {0, 1}), (128, 8, {1}), (128, 15, {1, 2}), (128, 3, {0}),
])
def test_block_overlap_hand_cases(bs, hot, blocks):
    # kernel j covers tokens [16 j, 16 j + 31]; it belongs to every block it shares a token with
    L = 1024
    M = oracle.n_kernels(L, 32, 16)
    q, kern = _one_hot_kernel_setup(M, 8, hot)
    S = oracle.block_scores(q, kern, np.array([L], np.int32), 1, params(block_size=bs), tree=True)
    got = {b for b in range(S.shape[-1]) if S[0, 0, 0, b] == 8.0}
    assert got == blocks
    assert np.all(S[0, 0, 0][[b for b in range(S.shape[-1]) if b not in blocks]] == 0.0)


def brute_scores(qf, kf, L, Tq, bs, c, s, G, tree):
    """Token-set brute force: a kernel counts for a block if their token sets meet,
    and for a query if its last token is at or before the query's position."""
    B, _, Hq, d = qf.shape
    Hkv = Hq // G
    M = (L - c) // s + 1 if L >= c else 0
    nblk = (L - 1) // bs + 1
    S = np.full((B, Hkv, Tq, nblk), -np.inf)
    for t in range(Tq):
        pos = L - 1 if tree else L - Tq + t
        for blk in range(pos // bs + 1):
            btoks = set(range(blk * bs, (blk + 1) * bs))
            for j in range(M):
                ktoks = set(range(j * s, j * s + c))
                if not (ktoks & btoks) or max(ktoks) > pos:
                    continue
                for h in range(Hq):
                    v = float(np.dot(qf[0, t, h], kf[0, h // G, j]))
                    S[0, h // G, t, blk] = max(S[0, h // G, t, blk], v)
    return S


@pytest.mark.parametrize("bs,G,tree", [(64, 2, False), (128, 4, False), (64, 2, True)])
def test_block_scores_brute_force(bs, G, tree):
    rng = np.random.default_rng(3 + bs + G)
    L, Tq, Hkv, d = 300, 5 if tree else 40, 2, 8
    Hq = Hkv * G
    q = rand_bf16(rng, (1, Tq, Hq, d))
    M = oracle.n_kernels(L, 32, 16)
    kern = rand_bf16(rng, (1, Hkv, M, d))
    S = oracle.block_scores(q, kern, np.array([L], np.int32), Hkv, params(block_size=bs), tree=tree)
    want = brute_scores(BF16_TO_F32(q).astype(np.float64), BF16_TO_F32(kern).astype(np.float64),
                        L, Tq, bs, 32, 16, G, tree)
    assert S.shape == want.shape
    fin = np.isfinite(want)
    assert np.array_equal(fin, np.isfinite(S))
    np.testing.assert_allclose(S[fin], want[fin], rtol=0, atol=1e-12)


def test_kernel_visibility_in_causal_chunk():
    # query at 70 sits in block 1; kernel 3 (tokens 48..79) ends after it, kernel 2 (32..63) not
    L = 80
    M = oracle.n_kernels(L, 32, 16)
    q, kern = _one_hot_kernel_setup(M, 8, hot=3)
    q = np.repeat(q, 80, axis=1)
    S = oracle.block_scores(q, kern, np.array([L], np.int32), 1, params(block_size=64),
                            t_list=np.array([70, 79]))
    assert S[0, 0, 0, 0] == 0.0                  # hot kernel invisible at 70; kernels 0-2 are
    assert S[0, 0, 0, 1] == -np.inf              # block 1's kernels 3, 4 both end after 70
    assert S[0, 0, 1, 0] == 8.0 and S[0, 0, 1, 1] == 8.0       # visible at 79


def test_group_max_uses_only_own_heads():
    rng = np.random.default_rng(4)
    L, d, G = 256, 8, 4
    M = oracle.n_kernels(L, 32, 16)
    kern = rand_bf16(rng, (1, 2, M, d))
    q = rand_bf16(rng, (1, 1, 2 * G, d))
    S = oracle.block_scores(q, kern, np.array([L], np.int32), 2, params(), tree=True)
    q2 = q.copy()
    q2[0, 0, G:] = rand_bf16(rng, (G, d))          # change group 1's heads only
    S2 = oracle.block_scores(q2, kern, np.array([L], np.int32), 2, params(), tree=True)
    assert np.array_equal(S[0, 0], S2[0, 0]) and not np.array_equal(S[0, 1], S2[0, 1])


# ---------------------------------------------------------------- step 3: selection

def brute_select(row, bt, k, n_i, n_l, dense):
    if dense:
        return list(range(bt + 1))
    forced = {b for b in range(bt + 1) if b < n_i or b >= bt - n_l + 1}
    cands = [b for b in range(bt + 1) if b not in forced]
    ranked = sorted(cands, key=lambda b: (-row[b], b))
    return sorted(forced | set(ranked[:k]))


@pytest.mark.parametrize("k,n_i,n_l", [(4, 1, 2), (1, 0, 1), (7, 2, 3), (40, 1, 2), (0, 1, 1)])
def test_select_brute_force_with_ties(k, n_i, n_l):
    rng = np.random.default_rng(5 + k)
    Tq, nblk = 64, 32
    L = nblk * 64
    # integer-valued scores: many exact ties, which must go to the lower index
    S = rng.integers(-3, 4, size=(1, 1, Tq, nblk)).astype(np.float64)
    S[0, 0, ::7, 3] = -np.inf
    p = params(topk=k, n_init_blocks=n_i, n_local_blocks=n_l)
    t_list = np.arange(Tq) * 32 + 31          # chunk of positions 31, 63, ... in a 2048-token call
    Tcall = L
    idx, counts, kth, nxt = oracle.select(S, np.array([L], np.int32), Tcall, p, t_list=t_list)
    for ti, t in enumerate(t_list):
        bt = t // 64
        want = brute_select(S[0, 0, ti], bt, k, n_i, n_l, False)
        assert counts[0, 0, ti] == len(want)
        assert list(idx[0, 0, ti, :counts[0, 0, ti]]) == want
        assert np.all(idx[0, 0, ti, counts[0, 0, ti]:] == -1)


def test_select_forced_blocks_and_count():
    rng = np.random.default_rng(6)
    nblk, k, n_i, n_l = 50, 5, 2, 3
    S = rng.standard_normal((1, 1, 1, nblk))
    S[0, 0, 0, :n_i] = -100.0           # forced blocks are kept whatever their score
    S[0, 0, 0, -n_l:] = -100.0
    p = params(topk=k, n_init_blocks=n_i, n_local_blocks=n_l)
    idx, counts, _, _ = oracle.select(S, np.array([nblk * 64], np.int32), 1, p)
    sel = list(idx[0, 0, 0, :counts[0, 0, 0]])
    assert counts[0, 0, 0] == n_i + n_l + k
    assert {0, 1, nblk - 3, nblk - 2, nblk - 1} <= set(sel)
    assert sel == sorted(set(sel))


def test_dense_switch():
    rng = np.random.default_rng(8)
    nblk = 20
    S = rng.standard_normal((1, 1, 1, nblk))
    L = nblk * 64
    for dense_len, dense in ((L + 1, True), (L, False), (0, False)):
        p = params(topk=3, dense_len=dense_len)
        idx, counts, _, _ = oracle.select(S, np.array([L], np.int32), 1, p)
        if dense:
            assert counts[0, 0, 0] == nblk and list(idx[0, 0, 0]) == list(range(nblk))
        else:
            assert counts[0, 0, 0] == 3 + 1 + 2


# ---------------------------------------------------------------- step 4: attention

def dense_reference(qf, kf, vf, scale, mask):
    """Textbook masked softmax attention in matrix form: softmax(scale Q K^T + mask) V."""
    z = scale * qf @ kf.T
    z = np.where(mask, z, -np.inf)
    m = z.max(axis=-1, keepdims=True)
    p = np.exp(z - m)
    l = p.sum(axis=-1, keepdims=True)
    return (p / l) @ vf, (m + np.log(l))[..., 0]


def _tiny_inputs(rng, L=200, Tq=30, Hq=4, Hkv=2, d=16):
    q = rand_bf16(rng, (1, Tq, Hq, d))
    k = rand_bf16(rng, (1, Hkv, L, d))
    v = rand_bf16(rng, (1, Hkv, L, d))
    return q, k, v


def test_attention_topk_covering_all_blocks_is_dense_causal():
    rng = np.random.default_rng(9)
    L, Tq, Hq, Hkv, d = 200, 30, 4, 2, 16
    q, k, v = _tiny_inputs(rng, L, Tq, Hq, Hkv, d)
    kv_len = np.array([L], np.int32)
    p = params(topk=1000)
    M = oracle.n_kernels(L, 32, 16)
    kern, _ = oracle.kernel_pool(k, kv_len, 32, 16, M)
    S = oracle.block_scores(q, kern, kv_len, Hkv, p)
    idx, counts, _, _ = oracle.select(S, kv_len, Tq, p)
    o, lse = oracle.attention(q, k, v, kv_len, idx, counts, p)
    qf, kf, vf = (BF16_TO_F32(a).astype(np.float64) for a in (q, k, v))
    for h in range(Hq):
        pos = np.arange(L - Tq, L)
        mask = np.arange(L)[None, :] <= pos[:, None]
        want_o, want_lse = dense_reference(qf[0, :, h], kf[0, h // 2], vf[0, h // 2], 1 / math.sqrt(d), mask)
        np.testing.assert_allclose(o[0, :, h], want_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], want_lse, rtol=0, atol=1e-12)
    # idx=None is the same dense causal attention
    o2, _ = oracle.attention(q, k, v, kv_len, None, None, p)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)


def test_attention_sparse_equals_masked_dense():
    rng = np.random.default_rng(10)
    L, Tq, Hq, Hkv, d = 640, 64, 4, 2, 16
    q, k, v = _tiny_inputs(rng, L, Tq, Hq, Hkv, d)
    kv_len = np.array([L], np.int32)
    p = params(topk=2, n_init_blocks=1, n_local_blocks=1)
    M = oracle.n_kernels(L, 32, 16)
    kern, _ = oracle.kernel_pool(k, kv_len, 32, 16, M)
    S = oracle.block_scores(q, kern, kv_len, Hkv, p)
    idx, counts, _, _ = oracle.select(S, kv_len, Tq, p)
    o, lse = oracle.attention(q, k, v, kv_len, idx, counts, p, scale=0.3)
    qf, kf, vf = (BF16_TO_F32(a).astype(np.float64) for a in (q, k, v))
    tok_block = np.arange(L) // 64
    for h in range(Hq):
        g = h // 2
        mask = np.zeros((Tq, L), bool)
        for t in range(Tq):
            sel = idx[0, g, t, :counts[0, g, t]]
            mask[t] = np.isin(tok_block, sel) & (np.arange(L) <= L - Tq + t)
        want_o, want_lse = dense_reference(qf[0, :, h], kf[0, g], vf[0, g], 0.3, mask)
        np.testing.assert_allclose(o[0, :, h], want_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], want_lse, rtol=0, atol=1e-12)


def test_attention_weights_nonnegative_and_sum_to_one():
    # V rows are one-hot, so the output is the weight vector itself
    rng = np.random.default_rng(11)
    L, d = 64, 64
    q = rand_bf16(rng, (1, 1, 1, d))
    k = rand_bf16(rng, (1, 1, L, d))
    v = np.zeros((1, 1, L, d), np.uint16)
    v[0, 0, np.arange(L), np.arange(L)] = F32_TO_BF16(np.array([1.0], np.float32))[0]
    p = params(topk=10)
    o, _ = oracle.attention(q, k, v, np.array([L], np.int32), None, None, p)
    w = o[0, 0, 0]
    assert np.all(w > 0) and abs(w.sum() - 1.0) < 1e-12
    ones = np.full((1, 1, L, d), F32_TO_BF16(np.array([1.0], np.float32))[0], np.uint16)
    o1, _ = oracle.attention(q, k, ones, np.array([L], np.int32), None, None, p)
    assert np.max(np.abs(o1 - 1.0)) < 1e-12


def test_attention_ragged_cache_tail():
    # kv_len not a multiple of the block: the last block is partial and nothing past kv_len counts
    rng = np.random.default_rng(12)
    L_max, L, d = 256, 150, 16
    q = rand_bf16(rng, (1, 1, 2, d))
    k = rand_bf16(rng, (1, 1, L_max, d))
    v = rand_bf16(rng, (1, 1, L_max, d))
    p = params(topk=100)
    o, _ = oracle.attention(q, k, v, np.array([L], np.int32), None, None, p)
    qf, kf, vf = (BF16_TO_F32(a).astype(np.float64) for a in (q, k, v))
    for h in range(2):
        want, _ = dense_reference(qf[0, :, h], kf[0, 0, :L], vf[0, 0, :L], 1 / 4.0, np.ones((1, L), bool))
        np.testing.assert_allclose(o[0, :, h], want, rtol=0, atol=1e-12)


def test_tree_attention():
    rng = np.random.default_rng(13)
    L, n, Hq, Hkv, d = 320, 6, 4, 2, 16
    q = rand_bf16(rng, (1, n, Hq, d))
    k = rand_bf16(rng, (1, Hkv, L, d))
    v = rand_bf16(rng, (1, Hkv, L, d))
    dk = rand_bf16(rng, (1, Hkv, n, d))
    dv = rand_bf16(rng, (1, Hkv, n, d))
    parent = [-1, 0, 0, 1, 1, 2]
    mask = np.zeros((1, n), np.uint64)
    for i in range(n):
        j = i
        while j >= 0:
            mask[0, i] |= np.uint64(1 << j)
            j = parent[j]
    kv_len = np.array([L], np.int32)
    p = params(topk=1, n_init_blocks=1, n_local_blocks=1)
    M = oracle.n_kernels(L, 32, 16)
    kern, _ = oracle.kernel_pool(k, kv_len, 32, 16, M)
    S = oracle.block_scores(q, kern, kv_len, Hkv, p, tree=True)
    idx, counts, _, _ = oracle.select(S, kv_len, n, p, tree=True)
    o, _ = oracle.attention(q, k, v, kv_len, idx, counts, p, draft_k=dk, draft_v=dv, tree_mask=mask)
    qf, kf, vf, dkf, dvf = (BF16_TO_F32(a).astype(np.float64) for a in (q, k, v, dk, dv))
    tok_block = np.arange(L) // 64
    for i in range(n):
        anc = [j for j in range(n) if (int(mask[0, i]) >> j) & 1]
        assert i in anc and all(j <= i for j in anc)
        for h in range(Hq):
            g = h // 2
            sel = idx[0, g, i, :counts[0, g, i]]
            # the whole last cache block is visible to a draft, plus its ancestors
            assert (L - 1) // 64 in sel and 0 in sel
            keys = np.concatenate([kf[0, g][np.isin(tok_block, sel)], dkf[0, g, anc]])
            vals = np.concatenate([vf[0, g][np.isin(tok_block, sel)], dvf[0, g, anc]])
            want, _ = dense_reference(qf[0, i, h][None], keys, vals, 0.25, np.ones((1, len(keys)), bool))
            np.testing.assert_allclose(o[0, i, h], want[0], rtol=0, atol=1e-12)
    # a mask of self bits only: each draft sees its selected cache blocks and itself
    self_mask = (np.uint64(1) << np.arange(n, dtype=np.uint64))[None]
    o_self, _ = oracle.attention(q, k, v, kv_len, idx, counts, p, draft_k=dk, draft_v=dv,
                                 tree_mask=self_mask)
    for i in range(n):
        for h in range(Hq):
            g = h // 2
            sel = idx[0, g, i, :counts[0, g, i]]
            keys = np.concatenate([kf[0, g][np.isin(tok_block, sel)], dkf[0, g, [i]]])
            vals = np.concatenate([vf[0, g][np.isin(tok_block, sel)], dvf[0, g, [i]]])
            want, _ = dense_reference(qf[0, i, h][None], keys, vals, 0.25, np.ones((1, len(keys)), bool))
            np.testing.assert_allclose(o_self[0, i, h], want[0], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- whole path on planted inputs

def test_planted_blocks_recovered_on_decisive_tiny_inputs():
    w = synth.WORKLOADS["tiny_prefill_2k"]
    inp = synth.make_inputs(w, decisive=True)
    r = oracle.run(inp, w)
    plant = set(inp["plant"][0].tolist())
    for t in range(w.Tq):
        bt = t // w.block_size
        sel = set(r["idx"][0, 0, t, :r["counts"][0, 0, t]].tolist())
        n_cand = max(0, bt + 1 - w.n_init - w.n_local)
        assert {0} | set(range(max(0, bt - 1), bt + 1)) <= sel
        if n_cand > w.topk and all(b <= bt - w.n_local for b in plant):
            assert plant <= sel
    gap = (r["kth"] - r["nxt"]) / np.abs(r["kth"])
    assert np.nanmin(gap) > 1e-3          # no near-ties at the top-k boundary


def test_generator_is_seeded_and_tree_is_valid():
    w = synth.WORKLOADS["tree_verify_64k"].scaled(L=4096, seed=77)
    a = synth.make_inputs(w)
    b = synth.make_inputs(w)
    for key in ("q", "k_cache", "v_cache", "draft_k", "tree_mask", "plant"):
        assert np.array_equal(a[key], b[key])
    parent, dep, mask = a["parent"], a["depth"], a["tree_mask"][0]
    assert parent[0] == -1 and dep.max() <= 5
    assert np.bincount(parent[1:], minlength=w.Tq).max() <= 3
    for i in range(w.Tq):
        assert (int(mask[i]) >> i) & 1
        if i:
            assert int(mask[i]) == int(mask[parent[i]]) | (1 << i)
