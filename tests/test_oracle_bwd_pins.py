"""Pins for the fp64 oracle's backward (CPU only).

The gradients of the oracle are tied to: float64 autograd of the attention
definition (a library routine differentiating the forward), central finite
differences of an independent float64 forward on tiny inputs, the identity
that links the row and the key functions, linearity in dO, conservation of
dO's column sums through dV, and the head-grouping reduction.  A slip such as
a missing softmax-Jacobian term, a wrong soft-cap derivative, a transposed
operand, a missing scale or a wrong head grouping fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def rand_inputs(B, H, Hkv, Sq, Sk, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, Sq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Sk, D), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, Sk, D), generator=g).to(torch.bfloat16)
    do = torch.randn((B, H, Sq, D), generator=g).to(torch.bfloat16)
    return q, k, v, do


def visible_mask(B, Sq, Sk, causal=False, window=0, doc_ids=None, prefix_len=None, q_offset=0):
    """Boolean [B, Sq, Sk] from the mask rules, written element by element."""
    vis = np.ones((B, Sq, Sk), dtype=bool)
    for b in range(B):
        for i in range(Sq):
            qpos = i + q_offset
            for j in range(Sk):
                ok = True
                if causal:
                    ok &= j <= qpos
                if window:
                    ok &= (qpos - window < j <= qpos)
                if doc_ids is not None:
                    ok &= int(doc_ids[b][i]) == int(doc_ids[b][j])
                if prefix_len is not None:
                    ok &= (j <= qpos) or (j < int(prefix_len[b]))
                vis[b, i, j] = ok
    return torch.from_numpy(vis)


def autograd_ref(q, k, v, do, scale, vis, alibi=False, softcap=0.0):
    """float64 autograd of the definition (K/V repeated over the head group)."""
    B, H, Sq, D = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    qd = q.double().requires_grad_(True)
    kd = k.double().requires_grad_(True)
    vd = v.double().requires_grad_(True)
    kr = kd.repeat_interleave(g, dim=1)
    vr = vd.repeat_interleave(g, dim=1)
    s = torch.matmul(qd, kr.transpose(-1, -2)) * float(np.float32(scale))
    if alibi:
        h = torch.arange(H, dtype=torch.float64)
        m = torch.pow(2.0, -8.0 * (h + 1) / H).view(1, H, 1, 1)
        i = torch.arange(Sq, dtype=torch.float64).view(1, 1, Sq, 1)
        j = torch.arange(k.shape[2], dtype=torch.float64).view(1, 1, 1, -1)
        s = s - m * (i - j)
    if softcap:
        cap = float(np.float32(softcap))
        s = cap * torch.tanh(s / cap)
    s = s.masked_fill(~vis.view(B, 1, Sq, -1), float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = torch.matmul(p, vr)
    (o * do.double()).sum().backward()
    return qd.grad.numpy(), kd.grad.numpy(), vd.grad.numpy()


CASES = [
    dict(B=1, H=2, Hkv=2, S=9, D=8, mods={}),
    dict(B=2, H=2, Hkv=1, S=11, D=8, mods=dict(causal=True)),
    dict(B=1, H=4, Hkv=2, S=12, D=4, mods=dict(window=4, causal=True)),
    dict(B=1, H=2, Hkv=2, S=10, D=8, mods=dict(causal=True, alibi=True)),
    dict(B=1, H=2, Hkv=2, S=10, D=8, mods=dict(softcap=2.0)),
    dict(B=1, H=3, Hkv=1, S=10, D=8, mods=dict(causal=True, alibi=True, softcap=3.0)),
    dict(B=2, H=2, Hkv=2, S=10, D=4, mods=dict(doc_ids=[[0, 0, 0, 1, 1, 2, 2, 2, 2, 3],
                                                         [0, 1, 1, 1, 1, 1, 2, 2, 3, 3]],
                                                causal=True)),
    dict(B=2, H=2, Hkv=2, S=9, D=4, mods=dict(prefix_len=[3, 0])),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_backward_equals_float64_autograd(case):
    c = CASES[case]
    B, H, Hkv, S, D, mods = c["B"], c["H"], c["Hkv"], c["S"], c["D"], dict(c["mods"])
    q, k, v, do = rand_inputs(B, H, Hkv, S, S, D, seed=50 + case)
    scale = 1.0 / math.sqrt(D)
    vis = visible_mask(B, S, S, causal=mods.get("causal", False), window=mods.get("window", 0),
                       doc_ids=mods.get("doc_ids"), prefix_len=mods.get("prefix_len"))
    gq, gk, gv = autograd_ref(q, k, v, do, scale, vis, alibi=mods.get("alibi", False),
                              softcap=mods.get("softcap", 0.0))
    okw = dict(mods)
    if "doc_ids" in okw:
        okw["doc_ids"] = np.asarray(okw["doc_ids"], dtype=np.int32)
    if "prefix_len" in okw:
        okw["prefix_len"] = np.asarray(okw["prefix_len"], dtype=np.int32)
    dq = oracle.attn_bwd_rows(q, k, v, do, scale=scale, **okw).reshape(B, H, S, D)
    dk, dv = oracle.attn_bwd_keys(q, k, v, do, scale=scale, **okw)
    np.testing.assert_allclose(dq, gq, rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk.reshape(B, Hkv, S, D), gk, rtol=0, atol=1e-10)
    np.testing.assert_allclose(dv.reshape(B, Hkv, S, D), gv, rtol=0, atol=1e-10)


def forward_np(q, k, v, scale, vis, alibi, softcap):
    """Independent float64 forward of one head (numpy), for finite differences."""
    s = (q @ k.T) * scale
    if alibi is not None:
        i = np.arange(q.shape[0])[:, None]
        j = np.arange(k.shape[0])[None, :]
        s = s - alibi * (i - j)
    if softcap:
        s = softcap * np.tanh(s / softcap)
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    p = np.where(vis, np.exp(s - m), 0.0)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


def test_backward_matches_finite_differences():
    # central differences of L = sum(dO * O) in float64, one head, softcap +
    # ALiBi + window: every entry of Q, K and V
    B, H, S, D = 1, 1, 7, 4
    q, k, v, do = rand_inputs(B, H, H, S, S, D, seed=77)
    scale, cap, slope = 0.5, 2.5, 2.0 ** -8.0
    vis = visible_mask(B, S, S, window=3, causal=True)[0].numpy()
    Q, K, V, G = (x[0, 0].double().numpy() for x in (q, k, v, do))
    sc = float(np.float32(scale))
    cp = float(np.float32(cap))

    def loss(Qx, Kx, Vx):
        return float((forward_np(Qx, Kx, Vx, sc, vis, slope, cp) * G).sum())

    eps = 1e-6
    num = []
    for X in (Q, K, V):
        gnum = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args_p = [Q, K, V]
            args_m = [Q, K, V]
            which = [id(Q), id(K), id(V)].index(id(X))
            args_p[which], args_m[which] = Xp, Xm
            gnum[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        num.append(gnum)
    dq = oracle.attn_bwd_rows(q, k, v, do, scale=scale, window=3, causal=True, alibi=True,
                              softcap=cap).reshape(S, D)
    dk, dv = oracle.attn_bwd_keys(q, k, v, do, scale=scale, window=3, causal=True, alibi=True,
                                  softcap=cap)
    np.testing.assert_allclose(dq, num[0], rtol=0, atol=1e-7)
    np.testing.assert_allclose(dk, num[1], rtol=0, atol=1e-7)
    np.testing.assert_allclose(dv, num[2], rtol=0, atol=1e-7)


def test_rows_and_keys_agree_through_the_score_identity():
    # sum_i q_i . dQ_i = scale * sum_ij dX_ij q_i.k_j = sum_j k_j . dK_j, per
    # K/V head group: ties the row function to the key function
    B, H, Hkv, S, D = 2, 4, 2, 40, 16
    q, k, v, do = rand_inputs(B, H, Hkv, S, S, D, seed=5)
    mods = dict(causal=True, alibi=True, softcap=4.0, window=25)
    dq = oracle.attn_bwd_rows(q, k, v, do, scale=0.25, **mods).reshape(B, H, S, D)
    dk, _ = oracle.attn_bwd_keys(q, k, v, do, scale=0.25, **mods)
    dk = dk.reshape(B, Hkv, S, D)
    Q, K = q.double().numpy(), k.double().numpy()
    g = H // Hkv
    for b in range(B):
        for hk in range(Hkv):
            lhs = sum((Q[b, h] * dq[b, h]).sum() for h in range(hk * g, (hk + 1) * g))
            rhs = (K[b, hk] * dk[b, hk]).sum()
            assert abs(lhs - rhs) <= 1e-10 * (1 + abs(lhs))


def test_linear_in_dout_and_dv_conserves_dout():
    B, H, S, D = 1, 2, 24, 8
    q, k, v, _ = rand_inputs(B, H, H, S, S, D, seed=9)
    g = torch.Generator().manual_seed(10)
    d1 = torch.randint(-1, 2, (B, H, S, D), generator=g).to(torch.bfloat16)
    d2 = torch.randint(-1, 2, (B, H, S, D), generator=g).to(torch.bfloat16)
    mods = dict(causal=True, softcap=3.0)
    a = oracle.attn_bwd_rows(q, k, v, d1, scale=0.3, **mods)
    b = oracle.attn_bwd_rows(q, k, v, d2, scale=0.3, **mods)
    c = oracle.attn_bwd_rows(q, k, v, d1 + d2, scale=0.3, **mods)
    np.testing.assert_allclose(c, a + b, rtol=0, atol=1e-12)
    ka, va = oracle.attn_bwd_keys(q, k, v, d1, scale=0.3, **mods)
    kb, vb = oracle.attn_bwd_keys(q, k, v, d2, scale=0.3, **mods)
    kc, vc = oracle.attn_bwd_keys(q, k, v, d1 + d2, scale=0.3, **mods)
    np.testing.assert_allclose(kc, ka + kb, rtol=0, atol=1e-12)
    np.testing.assert_allclose(vc, va + vb, rtol=0, atol=1e-12)
    # every row sees a key, and each row's probabilities sum to 1, so dV
    # summed over the keys is dO summed over the rows
    np.testing.assert_allclose(va.reshape(B, H, S, D).sum(axis=2),
                               d1.double().numpy().sum(axis=2), rtol=0, atol=1e-10)


def test_rows_without_keys_have_zero_gradient():
    # causal with a negative offset: the first rows see no key
    B, H, S, D = 1, 1, 16, 8
    q, k, v, do = rand_inputs(B, H, H, S, S, D, seed=11)
    dq = oracle.attn_bwd_rows(q, k, v, do, scale=0.3, causal=True, q_offset=-5)
    assert np.all(dq[:5] == 0.0) and np.any(dq[5:] != 0.0)
    dk, dv = oracle.attn_bwd_keys(q, k, v, do, scale=0.3, causal=True, q_offset=-5)
    assert np.all(dk[S - 5:] == 0.0) and np.all(dv[S - 5:] == 0.0)  # keys no row sees


def test_backward_with_rel_bias_and_blocks_equals_autograd():
    # additive relative-position bias and a block map, against float64
    # autograd of the definition (the bias enters the scores, the map the mask)
    B, H, Hkv, S, D = 2, 2, 1, 260, 4
    q, k, v, do = rand_inputs(B, H, Hkv, S, S, D, seed=71)
    R = 5
    g = np.random.default_rng(72)
    table = g.standard_normal((H, 2 * R + 1)).astype(np.float32).astype(np.float64)
    blk = (g.random((B, 3, 3)) < 0.7).astype(np.uint8)
    blk[:, :, 0] = 1
    full = np.stack([np.kron(blk[b], np.ones((128, 128), dtype=np.uint8))[:S, :S]
                     for b in range(B)]).astype(bool)
    causal = np.arange(S)[None, :] <= np.arange(S)[:, None]
    vis = torch.from_numpy(full & causal[None])
    idx = np.clip(np.arange(S)[None, :] - np.arange(S)[:, None], -R, R) + R
    bias = torch.from_numpy(table[:, idx])  # [H, S, S]

    qd = q.double().requires_grad_(True)
    kd = k.double().requires_grad_(True)
    vd = v.double().requires_grad_(True)
    kr, vr = kd.repeat_interleave(H // Hkv, dim=1), vd.repeat_interleave(H // Hkv, dim=1)
    s = torch.matmul(qd, kr.transpose(-1, -2)) * float(np.float32(0.5)) + bias[None]
    s = s.masked_fill(~vis[:, None], float("-inf"))
    o = torch.matmul(torch.softmax(s, dim=-1), vr)
    (o * do.double()).sum().backward()

    mods = dict(causal=True, rel_bias=table, blocks=blk)
    dq = oracle.attn_bwd_rows(q, k, v, do, scale=0.5, **mods).reshape(B, H, S, D)
    dk, dv = oracle.attn_bwd_keys(q, k, v, do, scale=0.5, **mods)
    np.testing.assert_allclose(dq, qd.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk.reshape(B, Hkv, S, D), kd.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dv.reshape(B, Hkv, S, D), vd.grad.numpy(), rtol=0, atol=1e-10)
