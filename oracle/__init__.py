"""fp64 CPU oracle for the attention forward and backward -- TEST
INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never imports, links or calls
it, and this package never imports the CUDA library.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, OpenMP
over rows): for every requested query row it materialises all scores, applies
the score modification and the mask literally, and takes the softmax.  This
module builds that file with gcc and marshals numpy arrays into it.

Every function here is pinned by the CPU tests in ``tests/test_oracle_pins.py``
against closed forms, a library routine (``torch.nn.functional.
scaled_dot_product_attention`` in float64) and invariants of the definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_attn.so")
_lock = threading.Lock()
_lib = None

MASK_CAUSAL = 1
MASK_WINDOW = 2
MASK_DOCUMENT = 4
MASK_PREFIX_LM = 8
MASK_BLOCKS = 16
SCORE_ALIBI = 1
SCORE_SOFTCAP = 2
SCORE_RELBIAS = 4
BLOCK = 128  # edge of a block-map tile


class _Mods(ctypes.Structure):
    """Mirror of the C ``or_mods``."""
    _fields_ = [("mask_flags", ctypes.c_uint32), ("score_flags", ctypes.c_uint32),
                ("window", ctypes.c_int), ("q_offset", ctypes.c_int),
                ("doc_ids", ctypes.c_void_p), ("prefix_len", ctypes.c_void_p),
                ("alibi_slopes", ctypes.c_void_p), ("softcap", ctypes.c_double),
                ("blocks", ctypes.c_void_p), ("blocks_batched", ctypes.c_int),
                ("rel_bias", ctypes.c_void_p), ("rel_max", ctypes.c_int)]


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``liboracle_attn.so`` (gcc, -O2, OpenMP).

    No -ffast-math: the oracle keeps IEEE double semantics.
    """
    with _lock:
        fresh = (os.path.exists(_LIB_PATH)
                 and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC))
        if fresh and not force:
            return _LIB_PATH
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    M = ctypes.POINTER(_Mods)
    lib.oracle_attn_rows.restype = ctypes.c_int
    lib.oracle_attn_rows.argtypes = [
        P, P, P,                                   # q k v
        ctypes.c_int, ctypes.c_int, ctypes.c_int,  # B H H_kv
        ctypes.c_int, ctypes.c_int, ctypes.c_int,  # S_q S_k D
        ctypes.c_double, M,                        # scale, mods
        P, ctypes.c_int64,                         # rows n
        P, P, P,                                   # out lse probs
    ]
    for name in ("oracle_attn_bwd_rows", "oracle_attn_bwd_keys"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [
            P, P, P, P,                                # q k v dout
            ctypes.c_int, ctypes.c_int, ctypes.c_int,  # B H H_kv
            ctypes.c_int, ctypes.c_int, ctypes.c_int,  # S_q S_k D
            ctypes.c_double, M,                        # scale, mods
            P, ctypes.c_int64,                         # rows / keys, n
        ] + ([P] if name.endswith("rows") else [P, P])
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    _lib = lib
    return lib


def num_threads() -> int:
    """OpenMP threads the oracle runs on."""
    return int(_load().oracle_num_threads())


def _bits(x) -> np.ndarray:
    """bf16 values as a contiguous uint16 numpy array of their bit patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            assert x.dtype == torch.bfloat16, x.dtype
            return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    assert a.dtype == np.uint16, a.dtype
    return a


def _i32(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _mods(B, H, S_q, S_k, causal=False, window=0, doc_ids=None, prefix_len=None,
          alibi=False, alibi_slopes=None, softcap=0.0, q_offset=0, rel_bias=None,
          blocks=None):
    """The C mods struct and the arrays it points to (keep them alive)."""
    m = _Mods()
    keep = []
    if causal:
        m.mask_flags |= MASK_CAUSAL
    if window and window > 0:
        m.mask_flags |= MASK_WINDOW
        m.window = int(window)
    m.q_offset = int(q_offset)
    if doc_ids is not None:
        m.mask_flags |= MASK_DOCUMENT
        docs = np.ascontiguousarray(np.broadcast_to(_i32(doc_ids).reshape(-1, S_k), (B, S_k)))
        keep.append(docs)
        m.doc_ids = docs.ctypes.data
    if prefix_len is not None:
        m.mask_flags |= MASK_PREFIX_LM
        pref = _i32(prefix_len)
        keep.append(pref)
        m.prefix_len = pref.ctypes.data
    if blocks is not None:
        blk = np.ascontiguousarray(np.asarray(
            blocks.cpu().numpy() if hasattr(blocks, "cpu") else blocks, dtype=np.uint8))
        nq, nk = -(-S_q // BLOCK), -(-S_k // BLOCK)
        blk = blk.reshape(-1, nq, nk)
        assert blk.shape[0] in (1, B)
        m.mask_flags |= MASK_BLOCKS
        m.blocks_batched = 1 if (blk.shape[0] == B and B > 1) else 0
        keep.append(blk)
        m.blocks = blk.ctypes.data
    if alibi or alibi_slopes is not None:
        m.score_flags |= SCORE_ALIBI
        if alibi_slopes is not None:
            sl = np.ascontiguousarray(np.asarray(
                alibi_slopes.cpu().numpy() if hasattr(alibi_slopes, "cpu") else alibi_slopes,
                dtype=np.float64))
            assert sl.shape == (H,)
            keep.append(sl)
            m.alibi_slopes = sl.ctypes.data
    if rel_bias is not None:
        rb = np.ascontiguousarray(np.asarray(
            rel_bias.cpu().numpy() if hasattr(rel_bias, "cpu") else rel_bias, dtype=np.float64))
        assert rb.ndim == 2 and rb.shape[0] == H and rb.shape[1] % 2 == 1
        m.score_flags |= SCORE_RELBIAS
        m.rel_max = (rb.shape[1] - 1) // 2
        keep.append(rb)
        m.rel_bias = rb.ctypes.data
    if softcap and softcap > 0:
        m.score_flags |= SCORE_SOFTCAP
        m.softcap = float(np.float32(softcap))
    return m, keep


def attn_rows(q, k, v, *, scale: float, rows: Optional[Sequence[int]] = None,
              want_probs: bool = False, **mods):
    """Attention forward of the requested rows, in float64.

    ``q`` [B,H,S_q,D] and ``k``/``v`` [B,H_kv,S_k,D] are bf16 torch tensors
    (or uint16 numpy arrays of bf16 bits).  ``scale`` and ``softcap`` are used
    as the float32 values a GPU kernel would receive (the bias-table entries
    as the float32 values given).  ``rows`` are flattened (b*H + h)*S_q + i
    indices (all rows when None).  Mods: ``causal``, ``window``, ``doc_ids``
    [B,S_k], ``prefix_len`` [B], ``alibi`` / ``alibi_slopes`` [H],
    ``softcap``, ``q_offset``, ``rel_bias`` [H, 2R+1] (score += rel_bias[h,
    clamp(kpos - qpos, -R, R) + R]), ``blocks`` [B or 1, ceil(S_q/128),
    ceil(S_k/128)] (0 hides the tile).

    Returns ``(O, LSE)`` as float64 arrays of shapes [n, D] and [n] (and the
    [n, S_k] probability matrix when ``want_probs``).
    """
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, H, S_q, D = qb.shape
    Bk, H_kv, S_k, Dk = kb.shape
    assert (Bk, Dk) == (B, D) and vb.shape == kb.shape
    if rows is None:
        rows_a = np.arange(B * H * S_q, dtype=np.int64)
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows_a.shape[0]
    m, keep = _mods(B, H, S_q, S_k, **mods)
    out = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    probs = np.empty((n, S_k), dtype=np.float64) if want_probs else None
    rc = lib.oracle_attn_rows(
        _ptr(qb), _ptr(kb), _ptr(vb), B, H, H_kv, S_q, S_k, D, float(np.float32(scale)),
        ctypes.byref(m), _ptr(rows_a), n, _ptr(out), _ptr(lse), _ptr(probs))
    del keep
    if rc != 0:
        raise ValueError("oracle_attn_rows rejected its arguments")
    if want_probs:
        return out, lse, probs
    return out, lse


def attn_bwd_rows(q, k, v, dout, *, scale: float, rows: Optional[Sequence[int]] = None,
                  **mods):
    """dQ of the requested query rows (flattened (b*H + h)*S_q + i; all when
    None) for upstream gradient ``dout`` [B,H,S_q,D] (bf16), in float64:
    an array [n, D].  Mods as for :func:`attn_rows`."""
    lib = _load()
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, H, S_q, D = qb.shape
    _, H_kv, S_k, _ = kb.shape
    assert gb.shape == qb.shape and vb.shape == kb.shape
    rows_a = (np.arange(B * H * S_q, dtype=np.int64) if rows is None
              else np.ascontiguousarray(np.asarray(rows, dtype=np.int64)))
    m, keep = _mods(B, H, S_q, S_k, **mods)
    dq = np.empty((rows_a.shape[0], D), dtype=np.float64)
    rc = lib.oracle_attn_bwd_rows(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), B, H, H_kv, S_q, S_k, D,
        float(np.float32(scale)), ctypes.byref(m), _ptr(rows_a), rows_a.shape[0], _ptr(dq))
    del keep
    if rc != 0:
        raise ValueError("oracle_attn_bwd_rows rejected its arguments")
    return dq


def attn_bwd_keys(q, k, v, dout, *, scale: float, keys: Optional[Sequence[int]] = None,
                  **mods):
    """dK and dV of the requested key positions (flattened
    (b*H_kv + hk)*S_k + j; all when None), summed over the query heads that
    share each K/V head, in float64: two arrays [n, D].  Mods as for
    :func:`attn_rows`."""
    lib = _load()
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, H, S_q, D = qb.shape
    _, H_kv, S_k, _ = kb.shape
    assert gb.shape == qb.shape and vb.shape == kb.shape
    keys_a = (np.arange(B * H_kv * S_k, dtype=np.int64) if keys is None
              else np.ascontiguousarray(np.asarray(keys, dtype=np.int64)))
    m, keep = _mods(B, H, S_q, S_k, **mods)
    dk = np.empty((keys_a.shape[0], D), dtype=np.float64)
    dv = np.empty((keys_a.shape[0], D), dtype=np.float64)
    rc = lib.oracle_attn_bwd_keys(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), B, H, H_kv, S_q, S_k, D,
        float(np.float32(scale)), ctypes.byref(m), _ptr(keys_a), keys_a.shape[0], _ptr(dk),
        _ptr(dv))
    del keep
    if rc != 0:
        raise ValueError("oracle_attn_bwd_keys rejected its arguments")
    return dk, dv


def attn_workload_rows(w, inputs, rows=None, want_probs: bool = False):
    """``attn_rows`` for a ``workloads.Workload`` and its generated inputs."""
    return attn_rows(
        inputs["q"], inputs["k"], inputs["v"], scale=w.scale, rows=rows,
        causal=w.causal, window=w.window, doc_ids=inputs.get("doc_ids"),
        prefix_len=inputs.get("prefix_len"), alibi=w.alibi,
        softcap=w.softcap, q_offset=w.q_offset, want_probs=want_probs)
