"""Backward (attn_bwd) against the fp64 oracle's gradients.

dQ, dK and dV are compared element by element with the oracle on every row
and key of small problems that span several tiles, ragged tails, every mask
and score mod, GQA and both head dimensions; and on sampled rows and keys at
a larger size.  Tolerance (derived in the design notes from the bf16 rounding
of P and dS fed to the tensor cores and of the stored gradients):
|delta| <= 1e-2 * max|ref| + 2^-7 * |ref| per tensor.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads

DEV = torch.device("cuda:0")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import attention_attn_fwd_04_gb300 as a
    return a


def inputs(B, H, Hkv, Sq, Sk, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, Sq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Sk, D), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, Sk, D), generator=g).to(torch.bfloat16)
    do = torch.randn((B, H, Sq, D), generator=g).to(torch.bfloat16)
    return q, k, v, do


def check(name, got, ref):
    got = got.float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    err = np.abs(got - ref)
    bound = 1e-2 * np.abs(ref).max() + 2.0 ** -7 * np.abs(ref)
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), "%s: max err %.3g (ref max %.3g), worst at %s: got %.5g ref %.5g" % (
        name, err.max(), np.abs(ref).max(), np.unravel_index(worst, ref.shape),
        got.flat[worst], ref.flat[worst])


def run_case(attn, B, H, Hkv, S, D, mods, seed):
    q, k, v, do = inputs(B, H, Hkv, S, S, D, seed)
    scale = 1.0 / math.sqrt(D)
    dmods = {n: (t.to(DEV) if isinstance(t, torch.Tensor) else t) for n, t in mods.items()}
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = attn.attn_fwd(qd, kd, vd, scale=scale, **dmods)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dod, scale=scale, **dmods)
    torch.cuda.synchronize()
    assert attn.get_device_status(device=DEV) == 0
    omods = dict(mods)
    if "window" in omods and omods["window"] is None:
        del omods["window"]
    ref_dq = oracle.attn_bwd_rows(q, k, v, do, scale=scale, **omods)
    ref_dk, ref_dv = oracle.attn_bwd_keys(q, k, v, do, scale=scale, **omods)
    check("dQ", dq, ref_dq)
    check("dK", dk, ref_dk)
    check("dV", dv, ref_dv)


def packed_docs(B, S, seed):
    return torch.stack([workloads.doc_ids_for(S, seed=seed + b, lo=40, hi=300)
                        for b in range(B)]).contiguous()


CASES = [
    (1, 2, 2, 256, 128, {}),
    (1, 2, 2, 300, 64, {"causal": True}),
    (2, 4, 2, 384, 128, {"causal": True}),                       # GQA 2:1
    (1, 4, 1, 260, 64, {}),                                     # GQA 4:1, ragged
    (1, 2, 2, 640, 128, {"window": 200, "causal": True, "softcap": 30.0}),
    (1, 2, 2, 520, 64, {"alibi": True, "softcap": 5.0}),
    (1, 4, 4, 600, 128, {"causal": True, "alibi": True}),
    (2, 2, 2, 700, 128, {"doc_ids": "packed", "causal": True}),
    (1, 2, 2, 400, 64, {"doc_ids": "unsorted"}),
    (2, 2, 2, 500, 128, {"prefix_len": [0, 200]}),
    (1, 2, 2, 384, 128, {"causal": True, "q_offset": -100}),    # rows with no key
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_backward_small(attn, case):
    B, H, Hkv, S, D, mods = CASES[case]
    mods = dict(mods)
    if mods.get("doc_ids") == "packed":
        mods["doc_ids"] = packed_docs(B, S, seed=20)
    elif mods.get("doc_ids") == "unsorted":
        g = torch.Generator().manual_seed(21)
        mods["doc_ids"] = torch.randint(0, 3, (B, S), generator=g).to(torch.int32)
    if "prefix_len" in mods:
        mods["prefix_len"] = torch.tensor(mods["prefix_len"], dtype=torch.int32)
    run_case(attn, B, H, Hkv, S, D, mods, seed=300 + case)


def test_backward_explicit_slopes(attn):
    mods = {"causal": True, "alibi_slopes": torch.tensor([0.5, 0.03125], dtype=torch.float32)}
    run_case(attn, 1, 2, 2, 300, 128, mods, seed=400)


def test_backward_sampled_at_size(attn):
    # causal GQA at S = 2048: sampled rows and keys (all tiles of the schedule run)
    B, H, Hkv, S, D = 1, 8, 2, 2048, 128
    q, k, v, do = inputs(B, H, Hkv, S, S, D, seed=500)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = attn.attn_fwd(qd, kd, vd, scale=scale, causal=True)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=True)
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(501)
    rows = torch.randperm(B * H * S, generator=g)[:256].numpy()
    keys = torch.randperm(B * Hkv * S, generator=g)[:64].numpy()
    keys = keys[keys // S < 1]  # one K/V head keeps the oracle's row pass short
    ref_dq = oracle.attn_bwd_rows(q, k, v, do, scale=scale, rows=rows, causal=True)
    ref_dk, ref_dv = oracle.attn_bwd_keys(q, k, v, do, scale=scale, keys=keys, causal=True)
    check("dQ", dq.reshape(-1, D)[torch.from_numpy(rows)], ref_dq)
    check("dK", dk.reshape(-1, D)[torch.from_numpy(keys)], ref_dk)
    check("dV", dv.reshape(-1, D)[torch.from_numpy(keys)], ref_dv)


def test_backward_outputs_aligned_to_16_bytes_only(attn):
    # dQ, dK, dV 16- but not 32-byte aligned take the epilogues' 16-byte
    # stores (32-byte aligned outputs take 32-byte stores): identical results
    B, H, Hkv, S, D = 1, 4, 2, 500, 128
    q, k, v, do = inputs(B, H, Hkv, S, S, D, seed=510)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = attn.attn_fwd(qd, kd, vd, causal=True)
    ref = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=True)

    def off16(shape):
        n = math.prod(shape)
        t = torch.empty(n + 16, dtype=torch.bfloat16, device=DEV)[8:8 + n].view(shape)
        assert t.data_ptr() % 32 == 16
        return t

    bufs = (off16(q.shape), off16(k.shape), off16(v.shape))
    got = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=True, dq=bufs[0], dk=bufs[1], dv=bufs[2])
    torch.cuda.synchronize()
    assert attn.get_device_status(device=DEV) == 0
    for g, b, r in zip(got, bufs, ref):
        assert g is b and torch.equal(g, r)


MODS3 = [
    (1, 2, 2, 300, 128, {"rel": 6, "causal": True}),
    (2, 2, 2, 400, 64, {"blocks": "batched", "rel": 3, "softcap": 8.0}),
    (1, 4, 2, 520, 128, {"blocks": "shared", "causal": True, "alibi": True, "rel": 40}),
]


@pytest.mark.parametrize("case", range(len(MODS3)))
def test_backward_rel_bias_and_block_map(attn, case):
    B, H, Hkv, S, D, mods = MODS3[case]
    mods = dict(mods)
    g = torch.Generator().manual_seed(700 + case)
    if "rel" in mods:
        R = mods.pop("rel")
        mods["rel_bias"] = (torch.randn((H, 2 * R + 1), generator=g) * 0.7).to(torch.float32)
    if "blocks" in mods:
        nb = -(-S // 128)
        Bb = B if mods["blocks"] == "batched" else 1
        mods["blocks"] = (torch.rand((Bb, nb, nb), generator=g) < 0.6).to(torch.uint8)
    run_case(attn, B, H, Hkv, S, D, mods, seed=700 + case)


@pytest.mark.parametrize("kernel", [1, 2])
def test_backward_wait_timeout_is_reported_and_context_survives(attn, kernel):
    # The test hook makes the MMA issuer of one backward kernel (1: dQ,
    # 2: dK/dV) wait on a barrier nothing arrives on: with a 20 ms budget the
    # wait runs out, the kernel records ATTN_ERR_TIMEOUT and returns (its
    # loaders let their copies land, Tensor Memory is freed; no trap, no
    # hang), and the next backward on the same context gives the same
    # gradients, bit for bit, as the one before the stall.
    B, H, S, D = 1, 2, 600, 128
    q, k, v, do = (t.to(DEV) for t in inputs(B, H, H, S, S, D, seed=90 + kernel))
    o, lse = attn.attn_fwd(q, k, v, causal=True)
    ref = attn.attn_bwd(q, k, v, o, lse, do, causal=True)
    assert attn.get_device_status(device=DEV) == 0
    old_budget = attn.get_option("wait_budget_ms")
    try:
        attn.set_option("wait_budget_ms", 20)
        attn.set_option("debug_stall", kernel)
        attn.attn_bwd(q, k, v, o, lse, do, causal=True)
        assert attn.get_device_status(device=DEV) == 4  # ATTN_ERR_TIMEOUT
    finally:
        attn.set_option("debug_stall", 0)
        attn.set_option("wait_budget_ms", old_budget)
    assert attn.get_device_status(device=DEV) == 0
    got = attn.attn_bwd(q, k, v, o, lse, do, causal=True)
    assert attn.get_device_status(device=DEV) == 0
    for g, r in zip(got, ref):
        assert torch.equal(g, r)
