"""attn_fwd_host: the forward on host tensors, with the copies and the
compute pipelined by the library.  Its results must equal attn_fwd's on
the same data bit for bit (same kernels), for single and back-to-back
calls, pinned and pageable memory, and problems that grow between calls."""
import math

import pytest
import torch

DEV = torch.device("cuda:0")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import attention_attn_fwd_04_gb300 as a
    return a


def inputs(B, H, H_kv, S, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, S, D), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H_kv, S, D), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H_kv, S, D), generator=g).to(torch.bfloat16)
    return q, k, v


def on_device(attn, q, k, v, mods):
    dm = {n: (t.to(DEV) if isinstance(t, torch.Tensor) else t) for n, t in mods.items()}
    o, lse = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), **dm)
    return o.cpu(), lse.cpu()


def mods_for(B, S, H, seed):
    g = torch.Generator().manual_seed(seed)
    ids = torch.cumsum((torch.rand((B, S), generator=g) < 0.004).to(torch.int32), dim=1)
    ids = ids.to(torch.int32).contiguous()
    slopes = torch.rand((H,), generator=g).to(torch.float32) * 0.1
    return dict(causal=True, doc_ids=ids, alibi_slopes=slopes, softcap=20.0)


@pytest.mark.parametrize("pinned", [True, False])
def test_host_matches_device(attn, pinned):
    B, H, H_kv, S, D = 2, 4, 2, 700, 128
    q, k, v = inputs(B, H, H_kv, S, D, seed=1)
    mods = mods_for(B, S, H, seed=2)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
        mods = {n: (t.pin_memory() if isinstance(t, torch.Tensor) else t) for n, t in mods.items()}
    o, lse = attn.attn_fwd_host(q, k, v, **mods)
    torch.cuda.current_stream(DEV).synchronize()
    assert attn.get_device_status(device=DEV) == 0
    o_ref, lse_ref = on_device(attn, q, k, v, mods)
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)


def test_back_to_back_calls_and_growth(attn):
    # five calls in flight at once (alternating device slots), the third
    # larger than the others so a slot grows; one synchronisation at the end
    shapes = [(1, 2, 2, 300, 64), (2, 4, 4, 512, 128), (2, 8, 4, 1500, 128),
              (1, 2, 2, 300, 64), (1, 4, 1, 260, 128)]
    calls = []
    for i, (B, H, H_kv, S, D) in enumerate(shapes):
        q, k, v = (t.pin_memory() for t in inputs(B, H, H_kv, S, D, seed=10 + i))
        mods = dict(causal=(i % 2 == 0), prefix_len=torch.tensor([S // 3] * B, dtype=torch.int32))
        o, lse = attn.attn_fwd_host(q, k, v, scale=1.0 / math.sqrt(D), **mods)
        calls.append((q, k, v, mods, o, lse, D))
    torch.cuda.current_stream(DEV).synchronize()
    assert attn.get_device_status(device=DEV) == 0
    for q, k, v, mods, o, lse, D in calls:
        o_ref, lse_ref = on_device(attn, q, k, v, dict(mods, scale=1.0 / math.sqrt(D)))
        assert torch.equal(o, o_ref)
        assert torch.equal(lse, lse_ref)


def test_host_call_orders_after_stream_work(attn):
    # the call starts after earlier work on the stream: a device-to-host copy
    # into the pinned input it then reads
    B, H, S, D = 1, 2, 256, 64
    q, k, v = inputs(B, H, H, S, D, seed=30)
    qd = q.to(DEV)
    qh = torch.zeros_like(q).pin_memory()
    s = torch.cuda.current_stream(DEV)
    qh.copy_(qd, non_blocking=True)          # enqueued on s before the call
    o, lse = attn.attn_fwd_host(qh, k.pin_memory(), v.pin_memory(), stream=s)
    s.synchronize()
    o_ref, lse_ref = on_device(attn, q, k, v, {})
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)


def test_default_alibi_slopes_across_head_chunks(attn):
    # 16 heads run as 8 chunks of 2: each chunk must still use the slope of
    # its heads' index among all 16
    B, H, S, D = 1, 16, 384, 64
    q, k, v = (t.pin_memory() for t in inputs(B, H, H, S, D, seed=40))
    mods = dict(alibi=True, causal=True, window=200)
    o, lse = attn.attn_fwd_host(q, k, v, **mods)
    torch.cuda.current_stream(DEV).synchronize()
    o_ref, lse_ref = on_device(attn, q, k, v, mods)
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)


def test_host_rel_bias_and_block_map(attn):
    # a per-batch block map and a bias table across head chunks
    B, H, S, D = 2, 8, 400, 64
    q, k, v = (t.pin_memory() for t in inputs(B, H, H, S, D, seed=50))
    g = torch.Generator().manual_seed(51)
    nb = -(-S // 128)
    mods = dict(causal=True,
                blocks=(torch.rand((B, nb, nb), generator=g) < 0.6).to(torch.uint8),
                rel_bias=(torch.randn((H, 2 * 9 + 1), generator=g) * 0.5).to(torch.float32))
    o, lse = attn.attn_fwd_host(q, k, v, **mods)
    torch.cuda.current_stream(DEV).synchronize()
    o_ref, lse_ref = on_device(attn, q, k, v, mods)
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)
