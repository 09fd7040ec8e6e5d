"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: a library routine
(``torch.nn.functional.scaled_dot_product_attention`` / ``torch.logsumexp`` in
float64), a closed form, a textbook special case or an invariant that the
definition of attention implies.  They are chosen so that a plausible slip in
the oracle (a dropped term, a wrong sign or index, a transposed operand, a
wrong mask boundary, the wrong head grouping) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def rand_qkv(B, H, Hkv, Sq, Sk, D, seed=0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, Sq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Sk, D), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, Sk, D), generator=g).to(torch.bfloat16)
    return q, k, v


def as_bhsd(x, B, H, S, D):
    return np.asarray(x).reshape(B, H, S, D)


def ref_sdpa(q, k, v, scale, attn_mask=None, is_causal=False):
    """Library reduction: float64 SDPA and float64 logsumexp of the scores."""
    qd, kd, vd = q.double(), k.double(), v.double()
    o = F.scaled_dot_product_attention(qd, kd, vd, attn_mask=attn_mask,
                                       is_causal=is_causal, scale=scale)
    s = torch.matmul(qd, kd.transpose(-1, -2)) * scale
    if is_causal:
        Sq, Sk = s.shape[-2:]
        keep = torch.ones(Sq, Sk, dtype=torch.bool).tril()
        s = s.masked_fill(~keep, float("-inf"))
    if attn_mask is not None:
        s = s.masked_fill(~attn_mask, float("-inf"))
    return o.numpy(), torch.logsumexp(s, dim=-1).numpy()


def f32(x):
    return float(np.float32(x))


# ---------------------------------------------------------------- library ---

def test_dense_equals_sdpa_float64():
    B, H, Sq, Sk, D = 2, 3, 5, 7, 8
    q, k, v = rand_qkv(B, H, H, Sq, Sk, D, seed=1)
    scale = f32(0.37)
    o, lse = oracle.attn_rows(q, k, v, scale=scale)
    ro, rl = ref_sdpa(q, k, v, scale)
    np.testing.assert_allclose(as_bhsd(o, B, H, Sq, D), ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(B, H, Sq), rl, rtol=0, atol=1e-12)


def test_causal_equals_sdpa_is_causal():
    B, H, S, D = 1, 2, 11, 4
    q, k, v = rand_qkv(B, H, H, S, S, D, seed=2)
    scale = f32(0.5)
    o, lse = oracle.attn_rows(q, k, v, scale=scale, causal=True)
    ro, rl = ref_sdpa(q, k, v, scale, is_causal=True)
    np.testing.assert_allclose(as_bhsd(o, B, H, S, D), ro, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(B, H, S), rl, atol=1e-12)


def test_gqa_equals_mha_with_repeated_kv():
    # Consecutive grouping: query head h reads KV head h // (H / H_kv).
    B, H, Hkv, S, D = 2, 6, 2, 9, 4
    q, k, v = rand_qkv(B, H, Hkv, S, S, D, seed=3)
    scale = f32(0.3)
    o, lse = oracle.attn_rows(q, k, v, scale=scale, causal=True)
    kr = k.repeat_interleave(H // Hkv, dim=1)
    vr = v.repeat_interleave(H // Hkv, dim=1)
    ro, rl = ref_sdpa(q, kr, vr, scale, is_causal=True)
    np.testing.assert_allclose(as_bhsd(o, B, H, S, D), ro, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(B, H, S), rl, atol=1e-12)


def test_document_slices_equal_sdpa_on_each_slice():
    # A fully visible document is dense attention on its slice; a causal
    # document is causal attention on its slice.
    S, D = 14, 4
    q, k, v = rand_qkv(1, 2, 2, S, S, D, seed=4)
    docs = torch.tensor([0, 0, 0, 0, 0, 1, 1, 1, 2, 2, 2, 2, 2, 2], dtype=torch.int32)
    scale = f32(0.4)
    for causal in (False, True):
        o, lse = oracle.attn_rows(q, k, v, scale=scale, doc_ids=docs, causal=causal)
        o = as_bhsd(o, 1, 2, S, D)
        lse = lse.reshape(1, 2, S)
        for a, b in ((0, 5), (5, 8), (8, 14)):
            ro, rl = ref_sdpa(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], scale,
                              is_causal=causal)
            np.testing.assert_allclose(o[:, :, a:b], ro, atol=1e-12)
            np.testing.assert_allclose(lse[:, :, a:b], rl, atol=1e-12)


# ----------------------------------------------------------- closed forms ---

def zero_q(B, H, Hkv, S, D, seed=5):
    _, k, v = rand_qkv(B, H, Hkv, S, S, D, seed=seed)
    q = torch.zeros((B, H, S, D), dtype=torch.bfloat16)
    return q, k, v


def check_uniform(o, lse, v, lo_hi, B, H, S, D):
    """With Q = 0 every visible key has score 0: O is the mean of V over the
    visible keys and LSE = ln(#visible)."""
    o = as_bhsd(o, B, H, S, D)
    lse = lse.reshape(B, H, S)
    vd = v.double().numpy()
    for i in range(S):
        lo, hi = lo_hi(i)
        if hi < lo:
            assert np.all(lse[:, :, i] == -np.inf)
            assert np.all(o[:, :, i] == 0)
            continue
        n = hi - lo + 1
        np.testing.assert_allclose(lse[:, :, i], math.log(n), atol=1e-13)
        np.testing.assert_allclose(o[:, :, i], vd[:, :, lo:hi + 1].mean(axis=2), atol=1e-13)


def test_causal_counts_and_means():
    B, H, S, D = 1, 2, 17, 3
    q, k, v = zero_q(B, H, H, S, D)
    o, lse = oracle.attn_rows(q, k, v, scale=1.0, causal=True)
    check_uniform(o, lse, v, lambda i: (0, i), B, H, S, D)


def test_window_counts_and_means():
    B, H, S, D, W = 1, 1, 20, 3, 6
    q, k, v = zero_q(B, H, H, S, D)
    o, lse = oracle.attn_rows(q, k, v, scale=1.0, window=W)
    # key j visible iff i - W < j <= i: exactly min(i + 1, W) keys
    check_uniform(o, lse, v, lambda i: (max(0, i - W + 1), i), B, H, S, D)


def test_window_with_causal_is_the_same_window():
    B, H, S, D, W = 1, 1, 20, 3, 6
    q, k, v = rand_qkv(B, H, H, S, S, D, seed=6)
    a = oracle.attn_rows(q, k, v, scale=0.5, window=W)
    b = oracle.attn_rows(q, k, v, scale=0.5, window=W, causal=True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_prefix_counts_and_means():
    B, H, S, D, P = 1, 1, 15, 3, 6
    q, k, v = zero_q(B, H, H, S, D)
    o, lse = oracle.attn_rows(q, k, v, scale=1.0,
                              prefix_len=torch.tensor([P], dtype=torch.int32))
    # visible iff j <= i or j < P: the keys 0 .. max(i, P - 1)
    check_uniform(o, lse, v, lambda i: (0, max(i, P - 1)), B, H, S, D)


def test_document_causal_counts_and_means():
    B, H, S, D = 1, 1, 12, 3
    q, k, v = zero_q(B, H, H, S, D)
    docs = torch.tensor([0, 0, 0, 1, 1, 1, 1, 1, 2, 3, 3, 3], dtype=torch.int32)
    start = [0, 0, 0, 3, 3, 3, 3, 3, 8, 9, 9, 9]
    o, lse = oracle.attn_rows(q, k, v, scale=1.0, doc_ids=docs, causal=True)
    check_uniform(o, lse, v, lambda i: (start[i], i), B, H, S, D)


def test_rows_without_visible_keys():
    # q_offset < 0 shifts query positions before key 0: those rows see
    # nothing and give O = 0, LSE = -inf.
    B, H, S, D = 1, 1, 8, 3
    q, k, v = zero_q(B, H, H, S, D)
    o, lse = oracle.attn_rows(q, k, v, scale=1.0, causal=True, q_offset=-3)
    check_uniform(o, lse, v, lambda i: (0, i - 3), B, H, S, D)


def test_bottom_right_alignment_with_q_offset():
    # S_q < S_k with q_offset = S_k - S_q: query i sees keys 0 .. i + S_k - S_q
    B, H, Sq, Sk, D = 1, 1, 4, 9, 2
    _, k, v = rand_qkv(B, H, H, Sq, Sk, D, seed=7)
    q = torch.zeros((B, H, Sq, D), dtype=torch.bfloat16)
    o, lse = oracle.attn_rows(q, k, v, scale=1.0, causal=True, q_offset=Sk - Sq)
    vd = v.double().numpy()
    for i in range(Sq):
        n = i + Sk - Sq + 1
        assert lse[i] == pytest.approx(math.log(n), abs=1e-13)
        np.testing.assert_allclose(o[i], vd[0, 0, :n].mean(axis=0), atol=1e-13)


def test_alibi_textbook_slopes_and_geometric_closed_form():
    # ALiBi slopes for 8 heads are the geometric sequence 1/2, 1/4, ..., 1/256.
    # With Q = 0 and causal masking the scores are -m*(i - j), so the softmax
    # over d = i - j is a truncated geometric distribution:
    #   LSE_i = ln((1 - r^(i+1)) / (1 - r)),      r = e^-m
    #   E[d]  = r/(1-r) - (i+1) r^(i+1) / (1 - r^(i+1))
    # and with V[j] = (j, 1) the output is O_i = (i - E[d], 1).
    H, S = 8, 40
    slopes = [0.5 ** (h + 1) for h in range(H)]
    q = torch.zeros((1, H, S, 2), dtype=torch.bfloat16)
    k = torch.zeros((1, H, S, 2), dtype=torch.bfloat16)
    v = torch.stack([torch.arange(S, dtype=torch.float32), torch.ones(S)], -1)
    v = v.to(torch.bfloat16).expand(1, H, S, 2).contiguous()
    o, lse = oracle.attn_rows(q, k, v, scale=1.0, causal=True, alibi=True)
    o = as_bhsd(o, 1, H, S, 2)
    lse = lse.reshape(1, H, S)
    for h in range(H):
        r = math.exp(-slopes[h])
        for i in range(S):
            rn = r ** (i + 1)
            assert lse[0, h, i] == pytest.approx(math.log((1 - rn) / (1 - r)), abs=1e-12)
            ed = r / (1 - r) - (i + 1) * rn / (1 - rn)
            assert o[0, h, i, 0] == pytest.approx(i - ed, abs=1e-10)
            assert o[0, h, i, 1] == pytest.approx(1.0, abs=1e-13)
    # explicit slopes override the default sequence
    o2, lse2 = oracle.attn_rows(q, k, v, scale=1.0, causal=True,
                                alibi_slopes=slopes[::-1])
    np.testing.assert_allclose(lse2.reshape(1, H, S)[0, 0], lse[0, H - 1], atol=1e-13)


def test_causal_first_row_is_v0_and_score():
    B, H, S, D = 2, 2, 6, 8
    q, k, v = rand_qkv(B, H, H, S, S, D, seed=8)
    scale = f32(0.25)
    o, lse = oracle.attn_rows(q, k, v, scale=scale, causal=True)
    o = as_bhsd(o, B, H, S, D)
    lse = lse.reshape(B, H, S)
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    np.testing.assert_array_equal(o[:, :, 0], vd[:, :, 0])
    s00 = scale * np.einsum("bhd,bhd->bh", qd[:, :, 0], kd[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], s00, atol=1e-13)


# -------------------------------------------------------------- invariants ---

def test_probabilities_sum_to_one_and_vanish_on_hidden_keys():
    B, H, S, D = 1, 2, 13, 4
    q, k, v = rand_qkv(B, H, H, S, S, D, seed=9)
    docs = torch.tensor([0] * 5 + [1] * 8, dtype=torch.int32)
    o, lse, p = oracle.attn_rows(q, k, v, scale=0.3, causal=True, doc_ids=docs,
                                 alibi=True, softcap=5.0, want_probs=True)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    for r in range(B * H * S):
        i = r % S
        for j in range(S):
            if j > i or int(docs[j]) != int(docs[i]):
                assert p[r, j] == 0.0
    # and O is exactly P @ V
    vd = v.double().numpy().reshape(H, S, D)
    for r in range(B * H * S):
        h = r // S
        np.testing.assert_allclose(o[r], p[r] @ vd[h], atol=1e-12)


def test_window_and_prefix_limits():
    B, H, S, D = 1, 2, 12, 4
    q, k, v = rand_qkv(B, H, H, S, S, D, seed=10)
    causal = oracle.attn_rows(q, k, v, scale=0.4, causal=True)
    dense = oracle.attn_rows(q, k, v, scale=0.4)
    wide = oracle.attn_rows(q, k, v, scale=0.4, window=S)
    p0 = oracle.attn_rows(q, k, v, scale=0.4, prefix_len=torch.tensor([0], dtype=torch.int32))
    pS = oracle.attn_rows(q, k, v, scale=0.4, prefix_len=torch.tensor([S], dtype=torch.int32))
    for a, b in ((wide, causal), (p0, causal), (pS, dense)):
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


def test_shift_of_every_key_shifts_lse_only():
    # Adding the same vector u to every key adds scale*q_i.u to every score of
    # row i: O is unchanged and LSE moves by that constant.  Small integers
    # keep K + u exact in bf16.
    g = torch.Generator().manual_seed(11)
    B, H, S, D = 1, 2, 9, 4
    q = torch.randint(-3, 4, (B, H, S, D), generator=g).float().to(torch.bfloat16)
    k = torch.randint(-3, 4, (B, H, S, D), generator=g).float().to(torch.bfloat16)
    v = torch.randn((B, H, S, D), generator=g).to(torch.bfloat16)
    u = torch.tensor([1.0, -2.0, 0.0, 3.0])
    k2 = (k.float() + u).to(torch.bfloat16)
    scale = 0.125
    o1, l1 = oracle.attn_rows(q, k, v, scale=scale, causal=True)
    o2, l2 = oracle.attn_rows(q, k2, v, scale=scale, causal=True)
    shift = scale * (q.double().numpy().reshape(-1, D) @ u.double().numpy())
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2, l1 + shift, atol=1e-12)


def test_output_is_linear_in_v():
    g = torch.Generator().manual_seed(12)
    B, H, S, D = 1, 2, 10, 4
    q, k, _ = rand_qkv(B, H, H, S, S, D, seed=12)
    v1 = torch.randint(-4, 5, (B, H, S, D), generator=g).float()
    v2 = torch.randint(-4, 5, (B, H, S, D), generator=g).float()
    va, vb, vc = v1.to(torch.bfloat16), v2.to(torch.bfloat16), (2 * v1 - 3 * v2).to(torch.bfloat16)
    oa, _ = oracle.attn_rows(q, k, va, scale=0.3, window=4)
    ob, _ = oracle.attn_rows(q, k, vb, scale=0.3, window=4)
    oc, _ = oracle.attn_rows(q, k, vc, scale=0.3, window=4)
    np.testing.assert_allclose(oc, 2 * oa - 3 * ob, atol=1e-12)


def test_softcap_limits_and_bounds():
    B, H, S, D = 1, 2, 16, 8
    q, k, v = rand_qkv(B, H, H, S, S, D, seed=13)
    # a huge cap leaves every score unchanged
    a = oracle.attn_rows(q, k, v, scale=0.3, causal=True)
    b = oracle.attn_rows(q, k, v, scale=0.3, causal=True, softcap=1e9)
    np.testing.assert_allclose(b[0], a[0], atol=1e-12)
    np.testing.assert_allclose(b[1], a[1], atol=1e-12)
    # cap 0.5 bounds every modified score in (-0.5, 0.5) even when the scale
    # is large, so every visible probability lies in (e^-1/n, e/n).  Applying
    # the scale after the cap, or dropping the cap, breaks this.
    _, _, p = oracle.attn_rows(q, k, v, scale=100.0, causal=True, softcap=0.5,
                               want_probs=True)
    for r in range(B * H * S):
        n = r % S + 1
        pv = p[r, :n]
        assert np.all(pv > math.exp(-1) / n) and np.all(pv < math.e / n)
    # the cap is monotone: it keeps the order of the probabilities
    _, _, p1 = oracle.attn_rows(q, k, v, scale=0.3, want_probs=True)
    _, _, p2 = oracle.attn_rows(q, k, v, scale=0.3, softcap=2.0, want_probs=True)
    np.testing.assert_array_equal(np.argsort(p1, axis=1, kind="stable"),
                                  np.argsort(p2, axis=1, kind="stable"))


def test_alibi_is_added_before_the_softcap():
    # Q = 0, causal, ALiBi, cap 1: the capped scores lie in (-1, 0], so no
    # probability ratio exceeds e.  Capping first and adding ALiBi after
    # would give ratios up to e^(m*(S-1)).
    H, S, D = 2, 30, 2
    q = torch.zeros((1, H, S, D), dtype=torch.bfloat16)
    k = torch.zeros((1, H, S, D), dtype=torch.bfloat16)
    v = torch.ones((1, H, S, D), dtype=torch.bfloat16)
    _, _, p = oracle.attn_rows(q, k, v, scale=1.0, causal=True, alibi=True,
                               softcap=1.0, want_probs=True)
    for r in range(H * S):
        i = r % S
        pv = p[r, :i + 1]
        assert pv.max() / pv.min() < math.e


# ----------------------------------------------------------- golden cases ---

def _eval_closed_form(expr):
    return float(eval(expr, {"__builtins__": {}}, {"ln": math.log, "exp": math.exp,
                                                   "tanh": math.tanh, "sqrt": math.sqrt}))


@pytest.mark.parametrize("name", sorted(f for f in os.listdir(GOLDEN) if f.endswith(".json")))
def test_golden_worked_examples(name):
    with open(os.path.join(GOLDEN, name)) as f:
        case = json.load(f)
    q = bf16(case["q"])
    k = bf16(case["k"])
    v = bf16(case["v"])
    kw = dict(case.get("mods", {}))
    if "doc_ids" in kw:
        kw["doc_ids"] = torch.tensor(kw["doc_ids"], dtype=torch.int32)
    if "prefix_len" in kw:
        kw["prefix_len"] = torch.tensor(kw["prefix_len"], dtype=torch.int32)
    scale = _eval_closed_form(case["scale"]) if isinstance(case["scale"], str) else case["scale"]
    if isinstance(kw.get("softcap"), str):
        kw["softcap"] = _eval_closed_form(kw["softcap"])
    o, lse = oracle.attn_rows(q, k, v, scale=scale, **kw)
    tol = case["tolerance"]
    for r, exp_row in enumerate(case["expected_o"]):
        for d, e in enumerate(exp_row):
            assert o[r, d] == pytest.approx(_eval_closed_form(e), abs=tol), (r, d)
    for r, e in enumerate(case["expected_lse"]):
        if e == "-inf":
            assert lse[r] == -np.inf
        else:
            assert lse[r] == pytest.approx(_eval_closed_form(e), abs=tol), r


# ------------------------------------------- relative-position bias, blocks ---

def rel_table(H, R, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal((H, 2 * R + 1)).astype(np.float32).astype(np.float64)


def expand_rel(table, S_q, S_k, q_offset=0):
    """bias[h, i, j] = table[h, clip(j - (i + q_offset), -R, R) + R], built by
    explicit indexing (independent of the oracle)."""
    H, W = table.shape
    R = (W - 1) // 2
    i = np.arange(S_q)[:, None] + q_offset
    j = np.arange(S_k)[None, :]
    idx = np.clip(j - i, -R, R) + R
    return table[:, idx]


def test_rel_bias_with_alibi_table_equals_alibi_exactly():
    # a table holding m_h * r reproduces ALiBi's -m_h * (qpos - kpos) term for
    # term (the same products up to sign), so the oracle outputs are identical
    B, H, S, D = 1, 4, 48, 16
    q, k, v = rand_qkv(B, H, H, S, S, D, seed=31)
    R = S
    m = 2.0 ** (-8.0 * (np.arange(H) + 1) / H)
    table = m[:, None] * np.arange(-R, R + 1)[None, :]
    o1, l1 = oracle.attn_rows(q, k, v, scale=0.25, causal=True, alibi=True)
    o2, l2 = oracle.attn_rows(q, k, v, scale=0.25, causal=True, rel_bias=table)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("R,q_offset,causal", [(3, 0, False), (0, 0, True), (7, 5, True), (40, -3, False)])
def test_rel_bias_matches_sdpa_additive_mask(R, q_offset, causal):
    B, H, Sq, Sk, D = 2, 3, 20, 26, 8
    q, k, v = rand_qkv(B, H, H, Sq, Sk, D, seed=32 + R)
    table = rel_table(H, R, seed=R)
    bias = torch.from_numpy(expand_rel(table, Sq, Sk, q_offset))[None]  # [1,H,Sq,Sk]
    if causal:
        i = np.arange(Sq)[:, None] + q_offset
        keep = torch.from_numpy(np.arange(Sk)[None, :] <= i)
        bias = bias.masked_fill(~keep, float("-inf"))
    qd, kd, vd = q.double(), k.double(), v.double()
    sc = f32(0.3)
    o_ref = F.scaled_dot_product_attention(qd, kd, vd, attn_mask=bias, scale=sc).numpy()
    s = torch.matmul(qd, kd.transpose(-1, -2)) * sc + bias
    l_ref = torch.logsumexp(s, dim=-1).numpy()
    o, l = oracle.attn_rows(q, k, v, scale=0.3, rel_bias=table, q_offset=q_offset, causal=causal)
    rows_ok = np.isfinite(l_ref.reshape(-1))
    np.testing.assert_allclose(o[rows_ok], o_ref.reshape(-1, D)[rows_ok], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l[rows_ok], l_ref.reshape(-1)[rows_ok], rtol=0, atol=1e-12)


def random_blocks(Bb, S_q, S_k, seed, p=0.6):
    g = np.random.default_rng(seed)
    nq, nk = -(-S_q // 128), -(-S_k // 128)
    return (g.random((Bb, nq, nk)) < p).astype(np.uint8)


def test_block_map_matches_sdpa_boolean_mask():
    B, H, Sq, Sk, D = 2, 2, 300, 400, 8
    q, k, v = rand_qkv(B, H, H, Sq, Sk, D, seed=40)
    blk = random_blocks(B, Sq, Sk, seed=41)
    blk[:, :, 0] = 1  # every row sees some key
    full = np.stack([np.kron(blk[b], np.ones((128, 128), dtype=np.uint8))[:Sq, :Sk]
                     for b in range(B)]).astype(bool)
    causal = np.arange(Sk)[None, :] <= np.arange(Sq)[:, None]
    mask = torch.from_numpy(full & causal[None])[:, None]
    o_ref, l_ref = ref_sdpa(q, k, v, f32(0.35), attn_mask=mask)
    o, l = oracle.attn_rows(q, k, v, scale=0.35, blocks=blk, causal=True)
    np.testing.assert_allclose(o, o_ref.reshape(-1, D), rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, l_ref.reshape(-1), rtol=0, atol=1e-12)
    # one map shared by the batch, and an all-ones map that changes nothing
    o1, l1 = oracle.attn_rows(q, k, v, scale=0.35, blocks=blk[:1], causal=True)
    full1 = torch.from_numpy(np.kron(blk[0], np.ones((128, 128), dtype=np.uint8))[:Sq, :Sk]
                             .astype(bool) & causal)[None, None]
    o_ref1, _ = ref_sdpa(q, k, v, f32(0.35), attn_mask=full1.expand(B, 1, Sq, Sk))
    np.testing.assert_allclose(o1, o_ref1.reshape(-1, D), rtol=0, atol=1e-12)
    ones = np.ones_like(blk[:1])
    o2, l2 = oracle.attn_rows(q, k, v, scale=0.35, blocks=ones, causal=True)
    o3, l3 = oracle.attn_rows(q, k, v, scale=0.35, causal=True)
    np.testing.assert_array_equal(o2, o3)
    np.testing.assert_array_equal(l2, l3)
