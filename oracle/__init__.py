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
SCORE_ALIBI = 1
SCORE_SOFTCAP = 2


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
    lib.oracle_attn_rows.restype = ctypes.c_int
    lib.oracle_attn_rows.argtypes = [
        P, P, P,                                   # q k v
        ctypes.c_int, ctypes.c_int, ctypes.c_int,  # B H H_kv
        ctypes.c_int, ctypes.c_int, ctypes.c_int,  # S_q S_k D
        ctypes.c_double,                           # scale
        ctypes.c_uint32, ctypes.c_uint32,          # mask / score flags
        ctypes.c_int, ctypes.c_int,                # window q_offset
        P, P, P,                                   # doc prefix slopes
        ctypes.c_double,                           # softcap
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
            ctypes.c_double,                           # scale
            ctypes.c_uint32, ctypes.c_uint32,          # mask / score flags
            ctypes.c_int, ctypes.c_int,                # window q_offset
            P, P, P,                                   # doc_ids prefix_len slopes
            ctypes.c_double,                           # softcap
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


def attn_rows(q, k, v, *, scale: float, rows: Optional[Sequence[int]] = None,
              causal: bool = False, window: int = 0, doc_ids=None,
              prefix_len=None, alibi: bool = False,
              alibi_slopes: Optional[Sequence[float]] = None,
              softcap: float = 0.0, q_offset: int = 0,
              want_probs: bool = False):
    """Attention forward of the requested rows, in float64.

    ``q`` [B,H,S_q,D] and ``k``/``v`` [B,H_kv,S_k,D] are bf16 torch tensors
    (or uint16 numpy arrays of bf16 bits).  ``scale`` and ``softcap`` are used
    as the float32 values a GPU kernel would receive.  ``rows`` are flattened
    (b*H + h)*S_q + i indices (all rows when None).

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
    mask = 0
    if causal:
        mask |= MASK_CAUSAL
    if window and window > 0:
        mask |= MASK_WINDOW
    if doc_ids is not None:
        mask |= MASK_DOCUMENT
    if prefix_len is not None:
        mask |= MASK_PREFIX_LM
    score = 0
    if alibi or alibi_slopes is not None:
        score |= SCORE_ALIBI
    if softcap and softcap > 0:
        score |= SCORE_SOFTCAP
    docs = _i32(doc_ids)
    if docs is not None:
        docs = np.ascontiguousarray(np.broadcast_to(docs.reshape(-1, S_k), (B, S_k)))
    pref = _i32(prefix_len)
    slopes = None
    if alibi_slopes is not None:
        slopes = np.ascontiguousarray(np.asarray(alibi_slopes, dtype=np.float64))
        assert slopes.shape == (H,)
    out = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    probs = np.empty((n, S_k), dtype=np.float64) if want_probs else None
    scale32 = float(np.float32(scale))
    cap32 = float(np.float32(softcap)) if softcap else 0.0
    rc = lib.oracle_attn_rows(
        _ptr(qb), _ptr(kb), _ptr(vb), B, H, H_kv, S_q, S_k, D, scale32,
        mask, score, int(window or 0), int(q_offset), _ptr(docs), _ptr(pref),
        _ptr(slopes), cap32, _ptr(rows_a), n, _ptr(out), _ptr(lse), _ptr(probs))
    if rc != 0:
        raise ValueError("oracle_attn_rows rejected its arguments")
    if want_probs:
        return out, lse, probs
    return out, lse


def _mod_args(B, H, S_k, causal, window, doc_ids, prefix_len, alibi, alibi_slopes,
              softcap):
    mask = 0
    if causal:
        mask |= MASK_CAUSAL
    if window and window > 0:
        mask |= MASK_WINDOW
    if doc_ids is not None:
        mask |= MASK_DOCUMENT
    if prefix_len is not None:
        mask |= MASK_PREFIX_LM
    score = 0
    if alibi or alibi_slopes is not None:
        score |= SCORE_ALIBI
    if softcap and softcap > 0:
        score |= SCORE_SOFTCAP
    docs = _i32(doc_ids)
    if docs is not None:
        docs = np.ascontiguousarray(np.broadcast_to(docs.reshape(-1, S_k), (B, S_k)))
    pref = _i32(prefix_len)
    slopes = None
    if alibi_slopes is not None:
        slopes = np.ascontiguousarray(np.asarray(alibi_slopes, dtype=np.float64))
        assert slopes.shape == (H,)
    cap32 = float(np.float32(softcap)) if softcap else 0.0
    return mask, score, docs, pref, slopes, cap32


def attn_bwd_rows(q, k, v, dout, *, scale: float, rows: Optional[Sequence[int]] = None,
                  causal: bool = False, window: int = 0, doc_ids=None, prefix_len=None,
                  alibi: bool = False, alibi_slopes: Optional[Sequence[float]] = None,
                  softcap: float = 0.0, q_offset: int = 0):
    """dQ of the requested query rows (flattened (b*H + h)*S_q + i; all when
    None) for upstream gradient ``dout`` [B,H,S_q,D] (bf16), in float64:
    an array [n, D]."""
    lib = _load()
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, H, S_q, D = qb.shape
    _, H_kv, S_k, _ = kb.shape
    assert gb.shape == qb.shape and vb.shape == kb.shape
    rows_a = (np.arange(B * H * S_q, dtype=np.int64) if rows is None
              else np.ascontiguousarray(np.asarray(rows, dtype=np.int64)))
    mask, score, docs, pref, slopes, cap32 = _mod_args(
        B, H, S_k, causal, window, doc_ids, prefix_len, alibi, alibi_slopes, softcap)
    dq = np.empty((rows_a.shape[0], D), dtype=np.float64)
    rc = lib.oracle_attn_bwd_rows(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), B, H, H_kv, S_q, S_k, D,
        float(np.float32(scale)), mask, score, int(window or 0), int(q_offset), _ptr(docs),
        _ptr(pref), _ptr(slopes), cap32, _ptr(rows_a), rows_a.shape[0], _ptr(dq))
    if rc != 0:
        raise ValueError("oracle_attn_bwd_rows rejected its arguments")
    return dq


def attn_bwd_keys(q, k, v, dout, *, scale: float, keys: Optional[Sequence[int]] = None,
                  causal: bool = False, window: int = 0, doc_ids=None, prefix_len=None,
                  alibi: bool = False, alibi_slopes: Optional[Sequence[float]] = None,
                  softcap: float = 0.0, q_offset: int = 0):
    """dK and dV of the requested key positions (flattened
    (b*H_kv + hk)*S_k + j; all when None), summed over the query heads that
    share each K/V head, in float64: two arrays [n, D]."""
    lib = _load()
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, H, S_q, D = qb.shape
    _, H_kv, S_k, _ = kb.shape
    assert gb.shape == qb.shape and vb.shape == kb.shape
    keys_a = (np.arange(B * H_kv * S_k, dtype=np.int64) if keys is None
              else np.ascontiguousarray(np.asarray(keys, dtype=np.int64)))
    mask, score, docs, pref, slopes, cap32 = _mod_args(
        B, H, S_k, causal, window, doc_ids, prefix_len, alibi, alibi_slopes, softcap)
    dk = np.empty((keys_a.shape[0], D), dtype=np.float64)
    dv = np.empty((keys_a.shape[0], D), dtype=np.float64)
    rc = lib.oracle_attn_bwd_keys(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), B, H, H_kv, S_q, S_k, D,
        float(np.float32(scale)), mask, score, int(window or 0), int(q_offset), _ptr(docs),
        _ptr(pref), _ptr(slopes), cap32, _ptr(keys_a), keys_a.shape[0], _ptr(dk), _ptr(dv))
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
