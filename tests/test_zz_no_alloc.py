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

import pytest
import torch

import tolerance

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


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
    """The parity criterion of the GPU tests (tests/tolerance.py), here against
    attn_fwd's own output: |dO| <= 1e-2 (an element above it only within one
    bf16 spacing of the reference, counted and bounded), mean |dO| <= 1e-3,
    |dLSE| <= 1e-3, and the same -inf rows."""
    D = o.shape[-1]
    tolerance.check(o.float().cpu().numpy().reshape(-1, D), lse.cpu().numpy().reshape(-1),
                    ro.double().cpu().numpy().reshape(-1, D), rl.double().cpu().numpy().reshape(-1))


CASES = [
    # B H Hkv S D  mods
    (1, 4, 2, 700, 128, dict(causal=True, alibi=True)),
    (2, 2, 2, 900, 64, dict(doc_ids="packed", causal=True, softcap=20.0)),
]


def lib_const(attn, name):
    """A size the header defines (#define NAME value), read from the header."""
    import os
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "include", "attn.h")
    text = open(hdr).read()
    expr = re.search(r"#define %s \((.*)\)|#define %s (\d+)u" % (name, name), text)
    value = expr.group(1) or expr.group(2)
    return int(eval(value.replace("u", "")))


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
        assert attn.get_noalloc_status(device=DEV) == 0  # synchronises the stream
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
    # documents over three sequences of 131072 tokens: the tile lists alone
    # (3 x 2 MiB) would fit, the per-token document ranges push the mask past
    # the array; the limit is attn_block_mask_bytes against the array's size
    limit = lib_const(attn, "ATTN_NOALLOC_SCRATCH_BYTES") - lib_const(attn, "ATTN_NOALLOC_STATUS_BYTES")
    S, B = 131072, 3
    m.mask_flags = attn.MASK_DOCUMENT | attn.MASK_CAUSAL
    m.doc_ids = 6 * big
    need = attn.lib().attn_block_mask_bytes(B, 1, S, S, ctypes.byref(m))
    assert 4 * B * (S // 256) * (S // 128) <= limit < need
    st = fn(P["q"], P["k"], P["v"], P["out"], None, B, 1, 1, S, S, 128, 0.1, ctypes.byref(m), None)
    assert st == 2  # ATTN_ERR_UNSUPPORTED
    m.mask_flags, m.doc_ids = 0, None
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
        assert attn.get_noalloc_status(device=DEV) == 0
    finally:
        attn.set_option("cta_pair", 0)
    assert torch.equal(o, ro) and torch.equal(l, rl)


def test_noalloc_status_reports_a_timeout_and_the_next_call_is_correct(api):
    # The test hook makes the MMA issuers wait on a barrier nothing arrives
    # on, with a 20 ms budget: the wait runs out, the kernel records
    # ATTN_ERR_TIMEOUT in the fixed array's status word and returns (no trap,
    # no hang).  attn_get_noalloc_status reads it back and clears it, and the
    # next call on the same context is correct.
    attn, fn = api
    case = make_case(attn, 0)
    q, k, v, B, H, Hkv, S, D, mods = case
    ro, rl = attn.attn_fwd(q, k, v, scale=1.0 / math.sqrt(D), **mods)
    o, l = torch.empty_like(q), torch.empty(q.shape[:3], device=DEV)
    old_budget = attn.get_option("wait_budget_ms")
    try:
        attn.set_option("wait_budget_ms", 20)
        attn.set_option("debug_stall", 1)
        assert call_noalloc(attn, fn, case, o, l) == 0
        assert attn.get_noalloc_status(device=DEV) == 4  # ATTN_ERR_TIMEOUT
    finally:
        attn.set_option("debug_stall", 0)
        attn.set_option("wait_budget_ms", old_budget)
    assert attn.get_noalloc_status(device=DEV) == 0  # cleared
    assert attn.get_device_status(device=DEV) == 0   # attn_fwd's word is untouched
    assert call_noalloc(attn, fn, case, o, l) == 0
    assert attn.get_noalloc_status(device=DEV) == 0
    close(o, l, ro, rl)
