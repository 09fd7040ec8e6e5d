"""attn_fwd_noalloc: the forward for callers that cannot allocate device
memory while they call it (code running under CUDA-graph stream capture,
runtimes whose memory pool owns every device allocation, latency-critical
paths that cannot take cudaMalloc's device-wide synchronisation).

It must give the same results as attn_fwd, call after call, while its
scratch lives in one fixed array inside the library.  This file is named to
be collected last, so a run that stops at the first failure has already run
every other test.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL_MAX_O, TOL_MEAN_O, TOL_LSE = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module")
def api():
    import attention_attn_fwd_04_gb300 as attn
    fn = attn.lib().attn_fwd_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.restype = I
    fn.argtypes = [P, P, P, P, P, I, I, I, I, I, I, ctypes.c_float,
                   ctypes.POINTER(attn.ModDesc), P]
    return attn, fn


def inputs(B, H, Hkv, S, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, S, D), generator=g).to(torch.bfloat16).to(DEV)
    k = torch.randn((B, Hkv, S, D), generator=g).to(torch.bfloat16).to(DEV)
    v = torch.randn((B, Hkv, S, D), generator=g).to(torch.bfloat16).to(DEV)
    return q, k, v


def close(o, lse, ro, rl):
    """The parity tolerance used by the GPU tests (|dO| <= 1e-2 + 2^-8|O|,
    mean |dO| <= 1e-3, |dLSE| <= 1e-3; -inf rows must match)."""
    o, ro = o.float().cpu().numpy(), ro.float().cpu().numpy()
    lse, rl = lse.cpu().numpy(), rl.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(lse), fin)
    d = np.abs(o - ro)
    assert (d - (TOL_MAX_O + 2.0 ** -8 * np.abs(ro))).max() <= 0
    assert d.mean() <= TOL_MEAN_O
    assert np.abs(lse[fin] - rl[fin]).max(initial=0.0) <= TOL_LSE


CASES = [
    # B H Hkv S D  mods
    (1, 4, 2, 700, 128, dict(causal=True, alibi=True)),
    (2, 2, 2, 900, 64, dict(doc_ids="packed", causal=True, softcap=20.0)),
]


def make_case(attn, i):
    B, H, Hkv, S, D, mods = CASES[i]
    q, k, v = inputs(B, H, Hkv, S, D, seed=40 + i)
    mods = dict(mods)
    if mods.get("doc_ids") == "packed":
        ids = torch.zeros((B, S), dtype=torch.int32)
        for b in range(B):
            for cut in (100 + 37 * b, 350, 610 - 11 * b):
                ids[b, cut:] += 1
        mods["doc_ids"] = ids.to(DEV)
    return (q, k, v, B, H, Hkv, S, D, mods)


def call_noalloc(attn, fn, case, out, lse):
    q, k, v, B, H, Hkv, S, D, mods = case
    m, keep = attn._mod_desc(**mods)
    stream = torch.cuda.current_stream(DEV).cuda_stream
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
            B, H, Hkv, S, S, D, 1.0 / math.sqrt(D), ctypes.byref(m), stream)
    del keep
    return st


def test_noalloc_matches_attn_fwd_on_consecutive_calls(api):
    attn, fn = api
    cases = [make_case(attn, 0), make_case(attn, 1)]
    refs = []
    for q, k, v, B, H, Hkv, S, D, mods in cases:
        refs.append(attn.attn_fwd(q, k, v, scale=1.0 / math.sqrt(D), **mods))
    outs = [(torch.empty_like(c[0]), torch.empty(c[0].shape[:3], device=DEV)) for c in cases]
    order = [0, 1, 0]  # different problems back to back, then the first again
    for n, i in enumerate(order):
        o, l = outs[i]
        o.fill_(float("nan"))
        l.fill_(float("nan"))
        torch.cuda.synchronize(DEV)
        free_before = torch.cuda.mem_get_info(DEV)[0]
        assert call_noalloc(attn, fn, cases[i], o, l) == 0
        torch.cuda.synchronize(DEV)
        free_after = torch.cuda.mem_get_info(DEV)[0]
        if n > 0:  # the first call may load the library's array; later ones take nothing
            assert free_after >= free_before, (n, free_before - free_after)
        close(o, l, *refs[i])


def test_noalloc_rejects_what_it_cannot_serve(api):
    attn, fn = api
    big = 1 << 40  # aligned stand-in addresses: rejected before any device use
    P = dict(q=big, k=2 * big, v=3 * big, out=4 * big)
    m = attn.ModDesc()
    m.version = 1
    # S = 2^20: the block mask would need far more than the fixed array
    st = fn(P["q"], P["k"], P["v"], P["out"], None, 1, 1, 1, 1 << 20, 1 << 20, 128, 0.1,
            ctypes.byref(m), None)
    assert st == 2  # ATTN_ERR_UNSUPPORTED
    # a caller-provided block mask is not accepted by this entry point
    m.block_mask = 5 * big
    m.block_mask_bytes = 1 << 20
    st = fn(P["q"], P["k"], P["v"], P["out"], None, 1, 1, 1, 256, 256, 128, 0.1,
            ctypes.byref(m), None)
    assert st == 1  # ATTN_ERR_INVALID_ARG


def test_noalloc_under_cta_pair(api):
    # With the CTA-pair option the fixed scratch holds a four-tile block mask;
    # the results equal attn_fwd's under the same option bit for bit.
    attn, fn = api
    case = make_case(attn, 0)
    q, k, v, B, H, Hkv, S, D, mods = case
    attn.set_option("cta_pair", 1)
    try:
        ro, rl = attn.attn_fwd(q, k, v, scale=1.0 / math.sqrt(D), **mods)
        o, l = torch.empty_like(q), torch.empty(q.shape[:3], device=DEV)
        assert call_noalloc(attn, fn, case, o, l) == 0
        torch.cuda.synchronize(DEV)
        assert attn.get_device_status(device=DEV) == 0
    finally:
        attn.set_option("cta_pair", 0)
    assert torch.equal(o, ro) and torch.equal(l, rl)
