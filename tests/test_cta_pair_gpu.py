"""GPU parity of the CTA-pair forward (option ``cta_pair``): two CTAs of a
cluster issue each score and output product as one 256-row tcgen05 MMA
("FlashAttention-4 explained", "TMEM and 2-CTA MMA", "2-CTA MMA mode").

Every case runs through the C ABI with the option set and is compared with
the fp64 oracle under the same tolerances as the one-CTA forward.  D = 128
problems run on the pair kernel; D = 64 problems run the one-CTA kernel on
the four-tile block mask the option builds, which these cases cover too.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
import test_parity_gpu as tp

pytestmark = pytest.mark.gpu

DEV = tp.DEV


@pytest.fixture(scope="module")
def attn():
    import attention_attn_fwd_04_gb300 as a
    return a


@pytest.fixture
def pair(attn):
    attn.set_option("cta_pair", 1)
    try:
        yield attn
    finally:
        attn.set_option("cta_pair", 0)


# tp.SMALL plus problems spanning several four-tile entries with ragged tails
LARGER = [
    (1, 2, 2, 1000, 1000, 128, {"causal": True}),
    (2, 4, 2, 1536, 1536, 128, {}),
    (1, 2, 2, 1100, 1300, 128, {"window": 300}),
    (1, 4, 4, 1200, 1200, 128, {"causal": True, "alibi": True, "softcap": 20.0}),
    (1, 2, 2, 513, 2000, 128, {"causal": True, "q_offset": 1487}),
]


@pytest.mark.parametrize("case", range(len(tp.SMALL) + len(LARGER)))
def test_pair_shapes(pair, case):
    B, H, Hkv, Sq, Sk, D, mods = (tp.SMALL + LARGER)[case]
    q, k, v = tp.rand_inputs(B, H, Hkv, Sq, Sk, D, seed=700 + case)
    tp.run_and_compare(pair, q, k, v, 1.0 / math.sqrt(D), **mods)


@pytest.mark.parametrize("case", range(len(tp.MODS3)))
def test_pair_rel_bias_and_block_map(pair, case):
    B, H, Hkv, Sq, Sk, D, mods = tp.MODS3[case]
    mods = tp.mods3(B, H, Sq, Sk, mods, seed=800 + case)
    q, k, v = tp.rand_inputs(B, H, Hkv, Sq, Sk, D, seed=800 + case)
    tp.run_and_compare(pair, q, k, v, 1.0 / math.sqrt(D), **mods)


def test_pair_documents_and_prefix(pair):
    B, H, S, D = 2, 2, 1777, 128
    q, k, v = tp.rand_inputs(B, H, H, S, S, D, seed=17)
    docs = torch.stack([workloads.doc_ids_for(S, seed=40 + b, lo=100, hi=700)
                        for b in range(B)]).contiguous()
    tp.run_and_compare(pair, q, k, v, 1 / math.sqrt(D), causal=True, doc_ids=docs)
    prefix = torch.tensor([300, 1500], dtype=torch.int32)
    tp.run_and_compare(pair, q, k, v, 1 / math.sqrt(D), causal=True, prefix_len=prefix)


@pytest.mark.parametrize("seed", range(8))
def test_quad_mask_classes_equal_pair_mask(attn, seed):
    # The tile classes do not depend on how many query tiles an entry groups.
    B, S_q, S_k, mods = tp.random_mask_case(seed)
    S_q, S_k = 3 * S_q, 3 * S_k  # several four-tile entries
    if "prefix_len" in mods:
        mods["prefix_len"] = torch.tensor(mods["prefix_len"], dtype=torch.int32)
    mods = tp.to_dev(mods)
    want = attn.decode_block_mask(attn.build_block_mask(B, 2, S_q, S_k, device=DEV, **mods))
    attn.set_option("cta_pair", 1)
    try:
        got = attn.decode_block_mask(attn.build_block_mask(B, 2, S_q, S_k, device=DEV, **mods))
    finally:
        attn.set_option("cta_pair", 0)
    assert want["tiles_per_entry"] == 2 and got["tiles_per_entry"] == 4
    assert got["nP"] == -(-got["nQ"] // 4)
    np.testing.assert_array_equal(got["cls"], want["cls"])


@pytest.mark.parametrize("mods", [{}, {"causal": True}])
def test_pair_agrees_with_single_cta(attn, mods):
    B, H, S, D = 2, 8, 2048, 128
    q, k, v = tp.rand_inputs(B, H, H, S, S, D, seed=21)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o1, l1 = attn.attn_fwd(qd, kd, vd, **mods)
    attn.set_option("cta_pair", 1)
    try:
        o2, l2 = attn.attn_fwd(qd, kd, vd, **mods)
    finally:
        attn.set_option("cta_pair", 0)
    assert attn.get_device_status(device=DEV) == 0
    d_o = (o1.float() - o2.float()).abs().max().item()
    d_l = (l1 - l2).abs().max().item()
    print("pair vs one CTA: max|dO| %.3g  max|dLSE| %.3g  identical %s"
          % (d_o, d_l, bool(torch.equal(o1, o2) and torch.equal(l1, l2))))
    # both sides are within the oracle bounds; against each other they differ
    # by at most the bf16 rounding of O
    assert d_o <= 2 * tp.TOL_MAX_O and d_l <= tp.TOL_LSE


def test_pair_few_ctas_walk_many_items(pair):
    # one CTA pair walks every item of the persistent schedule
    B, H, S, D = 1, 4, 1100, 128
    q, k, v = tp.rand_inputs(B, H, H, S, S, D, seed=22)
    pair.set_option("num_ctas", 2)
    try:
        tp.run_and_compare(pair, q, k, v, 1 / math.sqrt(D), causal=True)
        pair.set_option("num_ctas", 3)  # rounded to whole pairs
        tp.run_and_compare(pair, q, k, v, 1 / math.sqrt(D))
    finally:
        pair.set_option("num_ctas", 0)


def test_mask_built_for_other_setting_is_reported(attn):
    B, H, S, D = 1, 2, 1024, 128
    q, k, v = tp.rand_inputs(B, H, H, S, S, D, seed=23)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    bm = attn.build_block_mask(B, H, S, S, device=DEV, causal=True)  # two tiles per entry
    attn.set_option("cta_pair", 1)
    try:
        # the one-CTA mask is larger than the pair forward needs, so the size
        # check passes and the kernel's header check catches the mismatch
        attn.attn_fwd(qd, kd, vd, causal=True, block_mask=bm)
        assert attn.get_device_status(device=DEV) == 5  # ATTN_ERR_DEVICE_CHECK
        bm4 = attn.build_block_mask(B, H, S, S, device=DEV, causal=True)
        o, l = attn.attn_fwd(qd, kd, vd, causal=True, block_mask=bm4)
        assert attn.get_device_status(device=DEV) == 0
    finally:
        attn.set_option("cta_pair", 0)
    ro, rl = oracle.attn_rows(q, k, v, scale=1 / math.sqrt(D), causal=True)
    tp.compare(o.float().cpu().numpy().reshape(-1, D), l.cpu().numpy().reshape(-1), ro, rl)


def test_pair_wait_timeout_is_reported_and_context_survives(pair):
    # The issuing CTA's MMA warps wait on a barrier nothing arrives on: both
    # CTAs of every pair must give up (the abort flag reaches the peer),
    # record ATTN_ERR_TIMEOUT and return, and the next call must be correct.
    B, H, S, D = 1, 2, 1024, 128
    q, k, v = tp.rand_inputs(B, H, H, S, S, D, seed=24)
    old_budget = pair.get_option("wait_budget_ms")
    try:
        pair.set_option("wait_budget_ms", 20)
        pair.set_option("debug_stall", 1)
        pair.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
        assert pair.get_device_status(device=DEV) == 4  # ATTN_ERR_TIMEOUT
    finally:
        pair.set_option("debug_stall", 0)
        pair.set_option("wait_budget_ms", old_budget)
    assert pair.get_device_status(device=DEV) == 0
    tp.run_and_compare(pair, q, k, v, 1 / math.sqrt(D), causal=True)


@pytest.mark.parametrize("name", [n for n in workloads.WORKLOADS
                                  if workloads.get(n).D == 128])
def test_pair_workload_parity(pair, name):
    # the full-size workloads, sampled rows against the oracle
    w = workloads.get(name)
    inp = workloads.generate(w)
    rows = workloads.sample_rows(w, 2048, doc_ids=inp.get("doc_ids"))
    kw = dict(causal=w.causal, window=w.window or None, doc_ids=inp.get("doc_ids"),
              prefix_len=inp.get("prefix_len"), alibi=w.alibi, softcap=w.softcap or None,
              q_offset=w.q_offset)
    kw = {k_: v_ for k_, v_ in kw.items() if v_ is not None and v_ is not False}
    msg, _, _ = tp.run_and_compare(pair, inp["q"], inp["k"], inp["v"], w.scale,
                                   rows=rows.numpy(), **kw)
    print(name, msg)


@pytest.mark.parametrize("D", [128, 64])
def test_pair_host_entry_matches_device(pair, D):
    # attn_fwd_host builds its per-chunk block masks under the option too
    B, H, Hkv, S = 2, 4, 2, 900
    q, k, v = tp.rand_inputs(B, H, Hkv, S, S, D, seed=25)
    o_h, l_h = pair.attn_fwd_host(q, k, v, causal=True, alibi=True)
    torch.cuda.synchronize(DEV)
    assert pair.get_device_status(device=DEV) == 0
    o_d, l_d = pair.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, alibi=True)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


def test_backward_does_not_depend_on_the_option(attn):
    # attn_bwd builds its own two-tile masks whatever the option says
    B, H, S, D = 1, 4, 700, 128
    q, k, v = tp.rand_inputs(B, H, H, S, S, D, seed=26)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse = attn.attn_fwd(qd, kd, vd, causal=True)
    g = torch.Generator(device=DEV).manual_seed(5)
    do = torch.randn(o.shape, device=DEV, generator=g).to(torch.bfloat16)
    ref = attn.attn_bwd(qd, kd, vd, o, lse, do, causal=True)
    attn.set_option("cta_pair", 1)
    try:
        got = attn.attn_bwd(qd, kd, vd, o, lse, do, causal=True)
        assert attn.get_device_status(device=DEV) == 0
    finally:
        attn.set_option("cta_pair", 0)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
