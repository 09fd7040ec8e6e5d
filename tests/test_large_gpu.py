"""GPU parity at the largest sizes the tests can still check against the fp64
oracle: a million-token causal GQA forward, one query against two million
keys, packed documents over a million tokens, a batch of many heads, and the
backward of a short query block against a million keys.

Rows (and keys) are sampled: the first and last rows of every head, rows on
both sides of tile boundaries near the end, and seeded random rows.  At these
lengths a softmax over N(0, 1) scores spreads over so many keys that O
shrinks towards zero, which would let the absolute tolerance pass anything;
the scores here use scale 0.5 (standard deviation about 5.7 at D = 128), so a
handful of keys dominate each row and O stays of order one.  Tolerances are
those of the smaller parity tests.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
import test_parity_gpu as tp
import test_bwd_gpu as tb

pytestmark = pytest.mark.gpu

DEV = tp.DEV
SHARP = 0.5


@pytest.fixture(scope="module")
def attn():
    import attention_attn_fwd_04_gb300 as a
    return a


def edge_rows(B, H, S_q, n_random, seed):
    """Flattened (b*H + h)*S_q + i row indices: each head's first and last
    rows, rows around the last tile boundaries, and seeded random rows."""
    picks = {0, 1, S_q - 1, S_q - 2}
    for t in (128, 256):
        edge = (S_q - 1) // t * t
        picks.update(i for i in (edge - 1, edge, edge + 1) if 0 <= i < S_q)
    g = torch.Generator().manual_seed(seed)
    rows = [(bh * S_q + i) for bh in range(B * H) for i in sorted(picks)]
    rows += torch.randint(0, B * H * S_q, (n_random,), generator=g).tolist()
    return np.unique(np.asarray(rows, dtype=np.int64))


def test_million_token_causal_gqa(attn):
    B, H, Hkv, S, D = 1, 2, 1, 1 << 20, 128
    q, k, v = tp.rand_inputs(B, H, Hkv, S, S, D, seed=900)
    rows = edge_rows(B, H, S, 48, seed=901)
    msg, o, lse = tp.run_and_compare(attn, q, k, v, SHARP, rows=rows, causal=True)
    print("S = 2^20 causal GQA:", msg)
    # a sharp softmax keeps O away from zero, so the comparison has teeth
    assert o.float().abs().mean().item() > 0.05


def test_one_query_two_million_keys(attn):
    # a decode-shaped call: one query row (a single ragged tile) whose one
    # work item walks 16384 key tiles
    B, H, Hkv, S_q, S_k, D = 1, 2, 2, 1, 1 << 21, 64
    q, k, v = tp.rand_inputs(B, H, Hkv, S_q, S_k, D, seed=902)
    msg, _, _ = tp.run_and_compare(attn, q, k, v, SHARP, causal=True, q_offset=S_k - 1)
    print("S_q = 1, S_k = 2^21:", msg)


def test_million_token_documents(attn):
    B, H, S, D = 1, 1, 1 << 20, 128
    q, k, v = tp.rand_inputs(B, H, H, S, S, D, seed=903)
    docs = workloads.doc_ids_for(S, seed=904, lo=256, hi=65536).reshape(1, S).contiguous()
    rows = edge_rows(B, H, S, 64, seed=905)
    msg, _, _ = tp.run_and_compare(attn, q, k, v, SHARP, rows=rows, causal=True, doc_ids=docs,
                                   alibi=True)
    print("S = 2^20 documents + ALiBi:", msg)


def test_many_heads_ragged(attn):
    B, H, Hkv, S, D = 4, 256, 32, 333, 128
    q, k, v = tp.rand_inputs(B, H, Hkv, S, S, D, seed=906)
    rows = edge_rows(1, 1, B * H * S, 512, seed=907)
    msg, _, _ = tp.run_and_compare(attn, q, k, v, 1.0 / math.sqrt(D), rows=rows, causal=True,
                                   softcap=30.0)
    print("B4 H256/32 S333:", msg)


def test_backward_short_block_million_keys(attn):
    # 256 bottom-right queries against 2^20 keys: every dQ row walks 8192 key
    # tiles, and the oracle's per-key pass needs only 256 query rows per head
    B, H, Hkv, S_q, S_k, D = 1, 2, 1, 256, 1 << 20, 128
    g = torch.Generator().manual_seed(908)
    q = torch.randn((B, H, S_q, D), generator=g).to(torch.bfloat16)
    k = torch.randn((B, Hkv, S_k, D), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, S_k, D), generator=g).to(torch.bfloat16)
    do = torch.randn((B, H, S_q, D), generator=g).to(torch.bfloat16)
    mods = {"causal": True, "q_offset": S_k - S_q}
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = attn.attn_fwd(qd, kd, vd, scale=SHARP, **mods)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dod, scale=SHARP, **mods)
    torch.cuda.synchronize()
    assert attn.get_device_status(device=DEV) == 0
    rows = edge_rows(B, H, S_q, 32, seed=909)
    # keys: the first ones, both sides of the diagonal block, the last ones,
    # and random ones, on both K/V heads
    picks = [0, 1, 4095, S_k - S_q - 1, S_k - S_q, S_k - S_q + 1, S_k - 129, S_k - 128,
             S_k - 2, S_k - 1]
    picks += torch.randint(0, S_k, (24,), generator=g).tolist()
    # and the keys that carry most of the softmax weight of a few queries,
    # whose gradients are the large ones (found here on the CPU; this picks
    # which keys to check, the expected values still come from the oracle)
    s = q[0, :, ::32].float().reshape(-1, D) @ k[0, 0, :S_k - S_q].float().T
    picks += s.topk(2, dim=1).indices.flatten().tolist()
    keys = np.unique(np.asarray([hk * S_k + j for hk in range(Hkv) for j in picks],
                                dtype=np.int64))
    ref_dq = oracle.attn_bwd_rows(q, k, v, do, scale=SHARP, rows=rows, **mods)
    ref_dk, ref_dv = oracle.attn_bwd_keys(q, k, v, do, scale=SHARP, keys=keys, **mods)
    tb.check("dQ", dq.reshape(-1, D)[torch.from_numpy(rows)], ref_dq)
    tb.check("dK", dk.reshape(-1, D)[torch.from_numpy(keys)], ref_dk)
    tb.check("dV", dv.reshape(-1, D)[torch.from_numpy(keys)], ref_dv)
