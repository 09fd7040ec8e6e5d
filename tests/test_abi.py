"""The C-ABI library loads, exports every symbol the header declares, and
rejects bad arguments on the host (no GPU needed: nothing is enqueued)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def attn():
    from attention_attn_fwd_04_gb300 import build as b
    b.build()
    import attention_attn_fwd_04_gb300 as a
    return a


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[a-z_][\w \*]*?\b(attn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "attn_block_mask_bytes", "attn_build_block_mask",
              "attn_get_device_status", "attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(attn):
    lib = ctypes.CDLL(attn.library_path())
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings_and_abi_version(attn):
    lib = attn.lib()
    assert lib.attn_abi_version() == 1
    assert attn.status_string(0) == "ATTN_OK"
    assert attn.status_string(4) == "ATTN_ERR_TIMEOUT"
    assert attn.status_string(99) == "ATTN_ERR_UNKNOWN"


def _call(attn, q=16, k=16, v=16, out=32, lse=None, B=1, H=2, H_kv=2, S_q=128, S_k=128, D=64,
          scale=0.125, mod=None):
    lib = attn.lib()
    return lib.attn_fwd(q, k, v, out, lse, B, H, H_kv, S_q, S_k, D, scale,
                        ctypes.byref(mod) if mod is not None else None, None)


def test_host_validation_rejects_bad_arguments(attn):
    # fake, aligned, non-overlapping "device" addresses: validation fails
    # before any CUDA call, so nothing is dereferenced
    big = 1 << 40
    ok = dict(q=big, k=2 * big, v=3 * big, out=4 * big)
    INVALID, UNSUP = 1, 2
    assert _call(attn, **{**ok, "q": None}) == INVALID
    assert _call(attn, **{**ok, "out": None}) == INVALID
    assert _call(attn, **{**ok, "q": big + 8}) == INVALID          # not 16-byte aligned
    assert _call(attn, **ok, D=96) == UNSUP
    assert _call(attn, **ok, H=3, H_kv=2) == INVALID                # H % H_kv
    assert _call(attn, **ok, S_q=0) == INVALID
    assert _call(attn, **ok, B=-1) == INVALID
    assert _call(attn, **ok, scale=0.0) == INVALID
    assert _call(attn, **ok, scale=float("nan")) == INVALID
    assert _call(attn, **{**ok, "out": big}) == INVALID              # out aliases q
    m = attn.ModDesc()
    m.version = 7
    assert _call(attn, **ok, mod=m) == INVALID                      # bad version
    m.version = 1
    m.mask_flags = attn.MASK_WINDOW
    m.window = 0
    assert _call(attn, **ok, mod=m) == INVALID                      # window <= 0
    m.mask_flags = attn.MASK_DOCUMENT
    assert _call(attn, **ok, mod=m) == INVALID                      # doc_ids NULL
    m.doc_ids = 5 * big
    assert _call(attn, **ok, S_k=256, mod=m) == INVALID             # S_q != S_k
    m.mask_flags = 0
    m.score_flags = attn.SCORE_SOFTCAP
    m.softcap = -1.0
    assert _call(attn, **ok, mod=m) == INVALID                      # softcap <= 0
    m.score_flags = 0
    m.mask_flags = 1 << 9
    assert _call(attn, **ok, mod=m) == INVALID                      # unknown flag
    m.mask_flags = attn.MASK_PREFIX_LM
    assert _call(attn, **ok, mod=m) == INVALID                      # prefix_len NULL


def test_host_entry_point_validation(attn):
    # attn_fwd_host checks its arguments before any CUDA call
    lib = attn.lib()
    buf = [ctypes.create_string_buffer(1 << 16) for _ in range(5)]
    q, k, v, out, lse = (ctypes.addressof(b) for b in buf)
    INVALID, UNSUP = 1, 2

    def call(q=q, k=k, v=v, out=out, lse=lse, D=64, H=2, H_kv=2, mod=None):
        return lib.attn_fwd_host(q, k, v, out, lse, 1, H, H_kv, 64, 64, D, 0.125,
                                 ctypes.byref(mod) if mod is not None else None, None)

    assert call(q=None) == INVALID
    assert call(out=None) == INVALID
    assert call(D=80) == UNSUP
    assert call(H=3, H_kv=2) == INVALID
    assert call(out=q) == INVALID                                   # out aliases q
    m = attn.ModDesc()
    m.version = 1
    m.block_mask = k                                                # not accepted here
    assert call(mod=m) == INVALID


def test_descriptor_versions(attn):
    # version 1 (no block map / bias-table fields) is read without them;
    # unknown versions are rejected.  attn_block_mask_bytes validates the
    # descriptor on the host only (0 = rejected) and touches no memory.
    lib = attn.lib()
    big = 1 << 40

    def nbytes(m):
        return lib.attn_block_mask_bytes(1, 2, 256, 256, ctypes.byref(m))

    m = attn.ModDesc()
    m.version = 2
    m.mask_flags = attn.MASK_BLOCKS
    m.blocks = 5 * big
    assert nbytes(m) > 0
    m.version = 1                       # the v2 field is not part of a v1 descriptor
    assert nbytes(m) == 0
    m.version = 3
    assert nbytes(m) == 0
    m.version = 2
    m.blocks_batched = 2
    assert nbytes(m) == 0               # blocks_batched not 0 or 1
    m.blocks_batched = 0
    m.mask_flags = 0
    m.score_flags = attn.SCORE_RELBIAS
    m.rel_bias = 6 * big
    m.rel_max = -1
    assert nbytes(m) == 0               # rel_max < 0
    m.rel_max = 4
    assert nbytes(m) > 0
    m.rel_bias = None
    assert nbytes(m) == 0               # table missing
    # a v1 descriptor keeps working for the v1 mods
    m1 = attn.ModDesc()
    m1.version = 1
    m1.mask_flags = attn.MASK_CAUSAL
    assert nbytes(m1) > 0


def test_block_mask_bytes_is_host_only(attn):
    lib = attn.lib()
    m = attn.ModDesc()
    m.version = 1
    m.mask_flags = attn.MASK_CAUSAL
    n = lib.attn_block_mask_bytes(2, 32, 8192, 8192, ctypes.byref(m))
    assert n > 0 and n % 16 == 0
    # 64 query tiles -> 32 pairs; 64 key tiles per list entry row
    assert n >= 32 * 64 * 4
    assert lib.attn_block_mask_bytes(0, 1, 8, 8, None) == 0


def test_block_mask_bytes_matches_the_documented_layout(attn):
    # A 144-byte header, order[n] and cnt[n] (int32), list[n][nK] (uint32),
    # each region 16-byte aligned, with n = (B if the mask depends on the
    # batch, else 1) * ceil(S_q / 256); document masks add per-token key
    # ranges [2][B][S_k], per-tile id ranges [2][B][nK] and one flag per
    # 1024 tokens (int32 each).
    lib = attn.lib()

    def a16(x):
        return (x + 15) // 16 * 16

    def want(B, S_q, S_k, per_batch, docs):
        nK = -(-S_k // 128)
        n = (B if per_batch else 1) * -(-S_q // 256)
        total = a16(a16(a16(a16(144) + 4 * n) + 4 * n) + 4 * n * nK)
        if docs:
            bm = B
            total = a16(a16(a16(total + 8 * bm * S_k) + 8 * bm * nK) + 4 * bm * -(-S_k // 1024))
        return total

    m = attn.ModDesc()
    m.version = 1
    for B, S_q, S_k in ((4, 4096, 4096), (2, 300, 1000), (1, 1, 2 ** 21), (3, 5000, 5000)):
        m.mask_flags = 0
        assert lib.attn_block_mask_bytes(B, 8, S_q, S_k, ctypes.byref(m)) == want(B, S_q, S_k, 0, 0)
        m.mask_flags = attn.MASK_CAUSAL
        assert lib.attn_block_mask_bytes(B, 8, S_q, S_k, ctypes.byref(m)) == want(B, S_q, S_k, 0, 0)
    # prefix-LM depends on the batch; documents need S_q == S_k.  The size
    # query only checks that the mask arrays are given (host arrays here;
    # it never reads them).
    prefix = (ctypes.c_int32 * 3)(0, 100, 200)
    docs = (ctypes.c_int32 * (2 * 3000))()
    m.prefix_len = ctypes.cast(prefix, ctypes.c_void_p)
    m.mask_flags = attn.MASK_PREFIX_LM
    assert lib.attn_block_mask_bytes(3, 8, 700, 700, ctypes.byref(m)) == want(3, 700, 700, 1, 0)
    m.prefix_len = None
    m.doc_ids = ctypes.cast(docs, ctypes.c_void_p)
    m.mask_flags = attn.MASK_CAUSAL | attn.MASK_DOCUMENT
    assert lib.attn_block_mask_bytes(2, 8, 3000, 3000, ctypes.byref(m)) == want(2, 3000, 3000, 1, 1)


def test_options_round_trip(attn):
    old = attn.get_option("rescale_threshold")
    attn.set_option("rescale_threshold", 0.0)
    assert attn.get_option("rescale_threshold") == 0.0
    attn.set_option("rescale_threshold", old)
    with pytest.raises(attn.AttnError):
        attn.set_option("exp_poly_fraction", 2.0)
    with pytest.raises(attn.AttnError):
        attn.set_option("force_partial", 0.5)
    with pytest.raises(attn.AttnError):
        attn.set_option("debug_stall", 3)
    with pytest.raises(attn.AttnError):
        attn.set_option("debug_stall", 0.5)
    assert attn.get_option("debug_stall") == 0


def test_cta_pair_option_sets_mask_geometry(attn):
    # With the CTA-pair option a block-mask entry groups four query tiles
    # instead of two: half the entries, the same key-tile rows each.
    lib = attn.lib()
    m = attn.ModDesc()
    m.version = 1
    m.mask_flags = attn.MASK_CAUSAL
    assert attn.get_option("cta_pair") == 0
    n2 = lib.attn_block_mask_bytes(1, 8, 8192, 8192, ctypes.byref(m))
    try:
        attn.set_option("cta_pair", 1)
        assert attn.get_option("cta_pair") == 1
        n4 = lib.attn_block_mask_bytes(1, 8, 8192, 8192, ctypes.byref(m))
    finally:
        attn.set_option("cta_pair", 0)
    # 64 query tiles, 64 key tiles: 32 entries of 64 list slots vs 16
    assert n2 - n4 >= 16 * 64 * 4
    assert lib.attn_block_mask_bytes(1, 8, 8192, 8192, ctypes.byref(m)) == n2
    with pytest.raises(attn.AttnError):
        attn.set_option("cta_pair", 0.5)
    assert attn.get_option("cta_pair") == 0
