"""The benchmark's metric arithmetic, on the CPU.

"Useful TFLOPS" counts 4 * D FLOPs per visible (query, key) pair, so the
pair count decides every reported figure.  It is checked against the fp64
oracle's materialised probabilities (a pair is visible exactly when its
probability is non-zero: with these scores no visible exponential
underflows) and against closed forms for the named workloads.  Also: the
algorithmic bytes of the roofline and the quantile helper.
"""
import numpy as np
import pytest

import bench
import oracle
import workloads

CASES = [
    dict(S_q=300, S_k=300),
    dict(S_q=300, S_k=300, causal=True),
    dict(S_q=200, S_k=520, causal=True, q_offset=320),      # bottom-right
    dict(S_q=300, S_k=300, causal=True, q_offset=-50),      # rows with no key
    dict(S_q=300, S_k=300, window=70),
    dict(S_q=400, S_k=400, causal=True, document=True, doc_min=30, doc_max=120),
    dict(S_q=300, S_k=300, prefix_lm=True, prefix_lens=(0, 120)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_visible_pairs_equal_the_oracles_nonzero_probabilities(case):
    w = workloads.Workload(name="t", B=2, H=2, H_kv=2, D=64, scale=0.125, **CASES[case])
    inp = workloads.generate(w)
    _, _, probs = oracle.attn_workload_rows(w, inp, want_probs=True)
    want = int((probs > 0).sum())
    assert want > 0
    assert bench.visible_pairs(w, inp.get("doc_ids"), inp.get("prefix_len")) == want


def test_named_workload_pair_counts_match_closed_forms():
    def tri(n):
        return n * (n + 1) // 2

    got = {}
    for name, w in workloads.WORKLOADS.items():
        inp = workloads.generate(w) if w.document else {}
        got[name] = bench.visible_pairs(w, inp.get("doc_ids"), inp.get("prefix_len"))
    assert got["causal_b1_h2_s128_d64"] == 2 * tri(128)
    assert got["dense_b4_h16_s4096_d128"] == 4 * 16 * 4096 * 4096
    assert got["causal_gqa_b2_h32_hkv8_s8192_d128"] == 2 * 32 * tri(8192)
    # each row sees min(i + 1, W) keys
    W, S = 1024, 16384
    assert got["window1024_softcap30_b1_h16_s16384_d128"] == 16 * (tri(W) + (S - W) * W)
    # causal within each document: one triangle per document
    w = workloads.get("docs_alibi_b1_h16_s32768_d128")
    ids = workloads.generate(w)["doc_ids"][0].numpy()
    lengths = np.unique(ids, return_counts=True)[1]
    assert got["docs_alibi_b1_h16_s32768_d128"] == w.H * sum(tri(int(n)) for n in lengths)


def test_algorithmic_bytes_of_the_headline_shapes():
    # Q, K, V read once (K/V once per K/V head), O and LSE written once
    assert bench.algorithmic_bytes(workloads.get("dense_b4_h16_s4096_d128")) == 269_484_032
    assert bench.algorithmic_bytes(workloads.get("causal_gqa_b2_h32_hkv8_s8192_d128")) == 337_641_472


def test_quantile_interpolates_between_order_statistics():
    xs = [5.0, 1.0, 3.0, 2.0, 4.0]
    assert bench.quantile(xs, 0.0) == 1.0
    assert bench.quantile(xs, 1.0) == 5.0
    assert bench.quantile(xs, 0.5) == 3.0
    assert bench.quantile(xs, 0.1) == pytest.approx(1.4)
    assert bench.quantile(xs, 0.9) == pytest.approx(4.6)
    assert bench.quantile([7.0], 0.9) == 7.0


def test_clock_record_parses_the_sampler_output():
    c = bench.ClockSampler(0)
    c.out = "\n".join([
        "0, 2032, 2070, 910.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1011.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1995, 2070, 1390.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, [N/A], 2070, 1390.2, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ])
    got = c.summary()
    assert got == {"sm_mhz": 2032.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 3}
    c.out = "0, 1500, 2070, 700, 0x8, Active, Not Active, Active, Not Active"
    assert c.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    c.out = ""
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"],
                           "samples": 0}


def test_peaks_come_from_the_measured_file_else_the_fallback(tmp_path, monkeypatch):
    peaks, kind = bench.load_peaks()
    if kind == "measured":
        assert peaks["bf16_tflops"] > 0
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks() == ({"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                                   "bf16_tflops_sustained": 1700.0}, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 7000}')
    assert bench.load_peaks()[1] == "fallback"
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"bf16_tflops": 1850.5}')
    assert bench.load_peaks() == ({"bf16_tflops": 1850.5}, "measured")
