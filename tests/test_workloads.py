"""The seeded input generators both sides read (CPU).

They hold no attention arithmetic, but every parity test and bench line
depends on them: the named problems must be the configurations the metric
is quoted on, document ids must be packed (non-decreasing, lengths in the
drawn range), inputs must be reproducible, and the row samples must cover
the edge rows they promise.
"""
import math

import torch

import workloads


def test_named_workloads_are_the_documented_configurations():
    W = workloads.WORKLOADS
    assert workloads.HEADLINE == "dense_b4_h16_s4096_d128"
    expect = {
        "causal_b1_h2_s128_d64": (1, 2, 2, 128, 64, dict(causal=True)),
        "dense_b4_h16_s4096_d128": (4, 16, 16, 4096, 128, dict()),
        "causal_gqa_b2_h32_hkv8_s8192_d128": (2, 32, 8, 8192, 128, dict(causal=True)),
        "window1024_softcap30_b1_h16_s16384_d128":
            (1, 16, 16, 16384, 128, dict(causal=True, window=1024, softcap=30.0)),
        "docs_alibi_b1_h16_s32768_d128":
            (1, 16, 16, 32768, 128, dict(causal=True, document=True, alibi=True)),
    }
    assert set(W) == set(expect)
    for name, (B, H, Hkv, S, D, mods) in expect.items():
        w = W[name]
        assert (w.B, w.H, w.H_kv, w.S_q, w.S_k, w.D) == (B, H, Hkv, S, S, D), name
        assert w.scale == 1.0 / math.sqrt(D)
        for flag in ("causal", "document", "alibi", "prefix_lm"):
            assert getattr(w, flag) == mods.get(flag, False), (name, flag)
        assert w.window == mods.get("window", 0) and w.softcap == mods.get("softcap", 0.0)
        assert w.q_offset == 0
    # documents: lengths uniform in [256, 4096], seed 1
    d = W["docs_alibi_b1_h16_s32768_d128"]
    assert (d.doc_seed, d.doc_min, d.doc_max) == (1, 256, 4096)


def test_document_ids_are_packed_and_in_range():
    for S, seed, lo, hi in ((32768, 1, 256, 4096), (1777, 40, 100, 700), (5, 3, 10, 20)):
        ids = workloads.doc_ids_for(S, seed=seed, lo=lo, hi=hi)
        assert ids.dtype == torch.int32 and ids.shape == (S,)
        assert bool((ids[1:] - ids[:-1] >= 0).all()) and int(ids[0]) == 0
        assert bool((ids[1:] - ids[:-1] <= 1).all())  # consecutive ids
        lengths = torch.bincount(ids.long()).tolist()
        assert sum(lengths) == S
        assert all(lo <= n <= hi for n in lengths[:-1])
        assert 1 <= lengths[-1] <= hi  # the last one is cut to fit
        assert torch.equal(ids, workloads.doc_ids_for(S, seed=seed, lo=lo, hi=hi))
    assert not torch.equal(workloads.doc_ids_for(4096, seed=1), workloads.doc_ids_for(4096, seed=2))


def test_inputs_are_seeded_bf16_standard_normal():
    w = workloads.Workload(name="t", B=2, H=4, H_kv=2, S_q=300, S_k=500, D=64, scale=0.125,
                           document=True, doc_min=30, doc_max=90, prefix_lm=True)
    a, b = workloads.generate(w), workloads.generate(w)
    assert a["q"].shape == (2, 4, 300, 64) and a["k"].shape == (2, 2, 500, 64)
    assert a["v"].shape == a["k"].shape
    for n in ("q", "k", "v"):
        assert a[n].dtype == torch.bfloat16 and torch.equal(a[n], b[n])
        x = a[n].float()
        assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 1.0) < 0.02
    assert a["doc_ids"].shape == (2, 500) and torch.equal(a["doc_ids"][0], a["doc_ids"][1])
    assert a["prefix_len"].tolist() == [125, 125]
    other = workloads.generate(workloads.Workload(**{**w.__dict__, "seed": 1}))
    assert not torch.equal(a["q"], other["q"])


def test_row_samples_cover_the_edge_rows():
    w = workloads.get("docs_alibi_b1_h16_s32768_d128")
    ids = workloads.doc_ids_for(w.S_k, seed=w.doc_seed, lo=w.doc_min, hi=w.doc_max)
    rows = workloads.sample_rows(w, 4096, doc_ids=ids.reshape(1, -1))
    assert rows.dtype == torch.int64
    assert bool((rows[1:] > rows[:-1]).all())  # sorted, unique
    assert int(rows[0]) >= 0 and int(rows[-1]) < w.B * w.H * w.S_q
    have = set(rows.tolist())
    last = (w.B * w.H - 1) * w.S_q
    for i in (0, 1, 2, 127, 128, w.S_q - 1):
        assert i in have and last + i in have
    starts = torch.nonzero(torch.diff(ids, prepend=ids[:1] - 1)).flatten().tolist()
    for s in starts:
        assert s in have and s + 1 in have and last + s in have
    assert len(rows) >= 4096
    # a small problem is checked on every row
    tiny = workloads.get("causal_b1_h2_s128_d64")
    assert torch.equal(workloads.sample_rows(tiny), torch.arange(2 * 128))
