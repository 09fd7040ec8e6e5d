"""Host logic of the Python binding (CPU): keyword arguments become the C
descriptor the library validates.  Every keyword sets its flag and field,
the tensors it points at are kept alive for the call, and shapes the
library cannot take are rejected before any call."""
import pytest
import torch

import attention_attn_fwd_04_gb300 as a


def kept(t, keep):
    return any(x is t for x in keep)


def test_no_keywords_is_plain_attention():
    m, keep = a._mod_desc()
    assert m.version == a.MOD_DESC_VERSION
    assert (m.mask_flags, m.score_flags, m.window, m.q_offset, m.softcap) == (0, 0, 0, 0, 0.0)
    assert not m.doc_ids and not m.prefix_len and not m.alibi_slopes and not m.block_mask
    assert keep == ()


def test_interval_masks():
    m, _ = a._mod_desc(causal=True, window=64, q_offset=-5)
    assert m.mask_flags == a.MASK_CAUSAL | a.MASK_WINDOW
    assert (m.window, m.q_offset) == (64, -5)
    m, _ = a._mod_desc(window=0)  # passed through; the library rejects it
    assert m.mask_flags == a.MASK_WINDOW and m.window == 0


def test_mask_arrays_are_pointed_at_and_kept():
    docs = torch.zeros((2, 10), dtype=torch.int32)
    prefix = torch.tensor([3, 4], dtype=torch.int32)
    m, keep = a._mod_desc(doc_ids=docs, prefix_len=prefix)
    assert m.mask_flags == a.MASK_DOCUMENT | a.MASK_PREFIX_LM
    assert m.doc_ids == docs.data_ptr() and m.prefix_len == prefix.data_ptr()
    assert kept(docs, keep) and kept(prefix, keep)


def test_score_mods():
    m, keep = a._mod_desc(alibi=True, softcap=30.0)
    assert m.score_flags == a.SCORE_ALIBI | a.SCORE_SOFTCAP
    assert m.softcap == 30.0 and not m.alibi_slopes and keep == ()
    slopes = torch.rand(4)
    m, keep = a._mod_desc(alibi_slopes=slopes)
    assert m.score_flags == a.SCORE_ALIBI and m.alibi_slopes == slopes.data_ptr()
    assert kept(slopes, keep)
    m, _ = a._mod_desc(softcap=0)
    assert m.score_flags == 0
    table = torch.zeros((4, 2 * 7 + 1), dtype=torch.float32)
    m, keep = a._mod_desc(rel_bias=table)
    assert m.score_flags == a.SCORE_RELBIAS and m.rel_max == 7
    assert m.rel_bias == table.data_ptr() and kept(table, keep)
    with pytest.raises(ValueError):
        a._mod_desc(rel_bias=torch.zeros((4, 6)))  # 2R + 1 columns
    with pytest.raises(ValueError):
        a._mod_desc(rel_bias=torch.zeros(5))


def test_block_maps_one_per_batch_or_shared():
    per_batch = torch.ones((3, 2, 4), dtype=torch.uint8)
    m, keep = a._mod_desc(blocks=per_batch)
    assert m.mask_flags == a.MASK_BLOCKS and m.blocks_batched == 1
    assert m.blocks == per_batch.data_ptr() and kept(per_batch, keep)
    for shared in (torch.ones((1, 2, 4), dtype=torch.uint8), torch.ones((2, 4), dtype=torch.uint8)):
        m, _ = a._mod_desc(blocks=shared)
        assert m.mask_flags == a.MASK_BLOCKS and m.blocks_batched == 0


def test_missing_library_fails_loudly():
    # no fallback: without the compiled library the first call raises
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import attention_attn_fwd_04_gb300 as a\n"
        "a._LIB_PATH = '/nonexistent/libattn_gb300.so'\n"
        "try:\n"
        "    a.status_string(0)\n"
        "except ImportError as e:\n"
        "    print('raised', 'not built' in str(e))\n"
        "else:\n"
        "    print('no error')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=300)
    assert "raised True" in r.stdout, r.stdout + r.stderr
