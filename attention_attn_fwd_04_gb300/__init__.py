"""GB300 (sm_103a) fused attention forward -- Python binding.

A thin ctypes layer over the C ABI in ``include/attn.h``: it marshals torch
tensors (device memory and the current stream) into the library's plain
pointers and sizes.  Every step of the computation runs in the CUDA library
``libattn_gb300.so``; there is no CPU or PyTorch fallback.  If the library
is missing, importing this package raises: build it first with
``python -m attention_attn_fwd_04_gb300.build``.

    from attention_attn_fwd_04_gb300 import attn_fwd
    O, LSE = attn_fwd(q, k, v, causal=True)        # q [B,H,S,D] bf16 on cuda

Semantics (see ``include/attn.h``): scale first, then ALiBi, then the soft
cap; masks combine with AND; a row with no visible key yields O = 0 and
LSE = -inf; LSE uses the natural log.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

__all__ = [
    "AttnError",
    "BlockMask",
    "attn_fwd",
    "attn_fwd_into",
    "attn_fwd_host",
    "attn_bwd",
    "build_block_mask",
    "block_mask_bytes",
    "block_mask_stats",
    "get_device_status",
    "get_noalloc_status",
    "set_option",
    "get_option",
    "status_string",
    "library_path",
    "MASK_CAUSAL", "MASK_WINDOW", "MASK_DOCUMENT", "MASK_PREFIX_LM", "MASK_BLOCKS",
    "SCORE_ALIBI", "SCORE_SOFTCAP", "SCORE_RELBIAS", "BLOCK",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libattn_gb300.so")

MOD_DESC_VERSION = 2
MASK_CAUSAL, MASK_WINDOW, MASK_DOCUMENT, MASK_PREFIX_LM, MASK_BLOCKS = 1, 2, 4, 8, 16
SCORE_ALIBI, SCORE_SOFTCAP, SCORE_RELBIAS = 1, 2, 4
BLOCK = 128  # edge of a block-map tile

OPT_RESCALE_THRESHOLD = 1
OPT_FORCE_PARTIAL = 2
OPT_WAIT_BUDGET_MS = 3
OPT_NUM_CTAS = 4
OPT_EXP_POLY_FRACTION = 5
OPT_DEBUG_STALL = 6
OPT_CTA_PAIR = 7
_OPTIONS = {
    "rescale_threshold": OPT_RESCALE_THRESHOLD,
    "force_partial": OPT_FORCE_PARTIAL,
    "wait_budget_ms": OPT_WAIT_BUDGET_MS,
    "num_ctas": OPT_NUM_CTAS,
    "exp_poly_fraction": OPT_EXP_POLY_FRACTION,
    "debug_stall": OPT_DEBUG_STALL,
    "cta_pair": OPT_CTA_PAIR,
}

STATUS_NAMES = {
    0: "ATTN_OK",
    1: "ATTN_ERR_INVALID_ARG",
    2: "ATTN_ERR_UNSUPPORTED",
    3: "ATTN_ERR_CUDA",
    4: "ATTN_ERR_TIMEOUT",
    5: "ATTN_ERR_DEVICE_CHECK",
}


class AttnError(RuntimeError):
    """A non-OK status returned by the C library."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s" % (what, STATUS_NAMES.get(status, str(status))))


class ModDesc(ctypes.Structure):
    """Mirror of ``attn_mod_desc``."""

    _fields_ = [
        ("version", ctypes.c_uint32),
        ("mask_flags", ctypes.c_uint32),
        ("score_flags", ctypes.c_uint32),
        ("window", ctypes.c_int32),
        ("q_offset", ctypes.c_int32),
        ("softcap", ctypes.c_float),
        ("doc_ids", ctypes.c_void_p),
        ("prefix_len", ctypes.c_void_p),
        ("alibi_slopes", ctypes.c_void_p),
        ("block_mask", ctypes.c_void_p),
        ("block_mask_bytes", ctypes.c_size_t),
        ("blocks", ctypes.c_void_p),
        ("blocks_batched", ctypes.c_int32),
        ("rel_max", ctypes.c_int32),
        ("rel_bias", ctypes.c_void_p),
    ]


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            "libattn_gb300.so is not built (%s). Build it with "
            "`python -m attention_attn_fwd_04_gb300.build`." % _LIB_PATH)
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd.restype = I
    lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F,
                             ctypes.POINTER(ModDesc), P]
    lib.attn_bwd.restype = I
    lib.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F,
                             ctypes.POINTER(ModDesc), P]
    lib.attn_fwd_host.restype = I
    lib.attn_fwd_host.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F,
                                  ctypes.POINTER(ModDesc), P]
    lib.attn_block_mask_bytes.restype = ctypes.c_size_t
    lib.attn_block_mask_bytes.argtypes = [I, I, I, I, ctypes.POINTER(ModDesc)]
    lib.attn_build_block_mask.restype = I
    lib.attn_build_block_mask.argtypes = [I, I, I, I, ctypes.POINTER(ModDesc), P,
                                          ctypes.c_size_t, P]
    lib.attn_block_mask_stats.restype = I
    lib.attn_block_mask_stats.argtypes = [P, ctypes.c_size_t, P] + \
        [ctypes.POINTER(ctypes.c_int64)] * 4
    lib.attn_get_device_status.restype = I
    lib.attn_get_device_status.argtypes = [P]
    lib.attn_get_noalloc_status.restype = I
    lib.attn_get_noalloc_status.argtypes = [P]
    lib.attn_set_option.restype = I
    lib.attn_set_option.argtypes = [I, ctypes.c_double]
    lib.attn_get_option.restype = I
    lib.attn_get_option.argtypes = [I, ctypes.POINTER(ctypes.c_double)]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_status_string.argtypes = [I]
    lib.attn_abi_version.restype = I
    lib.attn_abi_version.argtypes = []
    return lib


class _LazyLib:
    """Loads ``libattn_gb300.so`` on first use, so the build module can be
    imported before the library exists.  A missing library raises."""

    _cdll = None

    def __getattr__(self, name):
        if _LazyLib._cdll is None:
            cdll = _load()
            if cdll.attn_abi_version() != 1:
                raise ImportError("libattn_gb300.so ABI version mismatch")
            _LazyLib._cdll = cdll
        return getattr(_LazyLib._cdll, name)


_lib = _LazyLib()


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded C library (for callers that want the raw ABI)."""
    _lib.attn_abi_version  # force the load
    return _LazyLib._cdll


def status_string(status: int) -> str:
    return _lib.attn_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != 0:
        raise AttnError(status, what)


def _stream_ptr(stream: Optional[torch.cuda.Stream], device: torch.device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


class BlockMask:
    """A device block mask built for one problem (opaque bytes + the mask
    arrays it was built from, kept alive while the mask is)."""

    def __init__(self, buf: torch.Tensor, B: int, H: int, S_q: int, S_k: int, mod: ModDesc,
                 keep: tuple):
        self.buf = buf
        self.B, self.H, self.S_q, self.S_k = B, H, S_q, S_k
        self.mask_flags = mod.mask_flags
        self._mod = mod
        self._keep = keep

    @property
    def nbytes(self) -> int:
        return self.buf.numel()

    def rebuild(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        """Rebuild in place (same buffer, same mask arrays) on ``stream``."""
        _check(_lib.attn_build_block_mask(self.B, self.H, self.S_q, self.S_k,
                                          ctypes.byref(self._mod), self.buf.data_ptr(),
                                          self.nbytes, _stream_ptr(stream, self.buf.device)),
               "attn_build_block_mask")


def _mod_desc(*, causal=False, window=None, doc_ids=None, prefix_len=None, alibi=False,
              alibi_slopes=None, softcap=None, q_offset=0, block_mask=None, blocks=None,
              rel_bias=None) -> Tuple[ModDesc, tuple]:
    m = ModDesc()
    m.version = MOD_DESC_VERSION
    keep = []
    if causal:
        m.mask_flags |= MASK_CAUSAL
    if window is not None:  # window <= 0 is rejected by the library
        m.mask_flags |= MASK_WINDOW
        m.window = int(window)
    if doc_ids is not None:
        m.mask_flags |= MASK_DOCUMENT
        m.doc_ids = _ptr(doc_ids)
        keep.append(doc_ids)
    if prefix_len is not None:
        m.mask_flags |= MASK_PREFIX_LM
        m.prefix_len = _ptr(prefix_len)
        keep.append(prefix_len)
    if alibi or alibi_slopes is not None:
        m.score_flags |= SCORE_ALIBI
        if alibi_slopes is not None:
            m.alibi_slopes = _ptr(alibi_slopes)
            keep.append(alibi_slopes)
    if softcap is not None and softcap != 0:
        m.score_flags |= SCORE_SOFTCAP
        m.softcap = float(softcap)
    if blocks is not None:
        # [B, nQ, nK] (one map per batch entry) or [nQ, nK] / [1, nQ, nK]
        m.mask_flags |= MASK_BLOCKS
        m.blocks = _ptr(blocks)
        m.blocks_batched = 1 if (blocks.dim() == 3 and blocks.shape[0] > 1) else 0
        keep.append(blocks)
    if rel_bias is not None:
        if rel_bias.dim() != 2 or rel_bias.shape[1] % 2 != 1:
            raise ValueError("rel_bias must be [H, 2R+1]")
        m.score_flags |= SCORE_RELBIAS
        m.rel_bias = _ptr(rel_bias)
        m.rel_max = (rel_bias.shape[1] - 1) // 2
        keep.append(rel_bias)
    m.q_offset = int(q_offset)
    if block_mask is not None:
        m.block_mask = _ptr(block_mask.buf)
        m.block_mask_bytes = block_mask.nbytes
        keep.append(block_mask)
    return m, tuple(keep)


def _check_mask_arrays(device, doc_ids, prefix_len, alibi_slopes, blocks=None, rel_bias=None):
    for name, t, dt in (("doc_ids", doc_ids, torch.int32), ("prefix_len", prefix_len, torch.int32),
                        ("alibi_slopes", alibi_slopes, torch.float32),
                        ("blocks", blocks, torch.uint8), ("rel_bias", rel_bias, torch.float32)):
        if t is None:
            continue
        if t.device != device or t.dtype != dt or not t.is_contiguous():
            raise ValueError("%s must be a contiguous %s tensor on %s" % (name, dt, device))


def block_mask_bytes(B: int, H: int, S_q: int, S_k: int, **mods) -> int:
    m, _ = _mod_desc(**mods)
    return int(_lib.attn_block_mask_bytes(B, H, S_q, S_k, ctypes.byref(m)))


def build_block_mask(B: int, H: int, S_q: int, S_k: int, *, device=None,
                     stream: Optional[torch.cuda.Stream] = None, **mods) -> BlockMask:
    """Build the tile classification for a problem on the device.  ``mods``
    take the same keywords as :func:`attn_fwd` (score mods are ignored)."""
    device = torch.device(device if device is not None else "cuda")
    _check_mask_arrays(device, mods.get("doc_ids"), mods.get("prefix_len"), None,
                       mods.get("blocks"))
    m, keep = _mod_desc(**mods)
    n = int(_lib.attn_block_mask_bytes(B, H, S_q, S_k, ctypes.byref(m)))
    if n == 0:
        raise AttnError(1, "attn_block_mask_bytes")
    buf = torch.empty(n, dtype=torch.uint8, device=device)
    _check(_lib.attn_build_block_mask(B, H, S_q, S_k, ctypes.byref(m), buf.data_ptr(), n,
                                      _stream_ptr(stream, device)), "attn_build_block_mask")
    return BlockMask(buf, B, H, S_q, S_k, m, keep)


def block_mask_stats(bm: BlockMask, stream: Optional[torch.cuda.Stream] = None) -> dict:
    """Counts of computed entries and FULL / PARTIAL / EMPTY tiles (syncs)."""
    vals = [ctypes.c_int64() for _ in range(4)]
    _check(_lib.attn_block_mask_stats(bm.buf.data_ptr(), bm.nbytes,
                                      _stream_ptr(stream, bm.buf.device),
                                      *[ctypes.byref(x) for x in vals]), "attn_block_mask_stats")
    return dict(zip(("entries", "full", "partial", "empty"), (x.value for x in vals)))


def attn_fwd_into(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                  lse: Optional[torch.Tensor], *, scale: Optional[float] = None,
                  causal: bool = False, window: Optional[int] = None,
                  doc_ids: Optional[torch.Tensor] = None,
                  prefix_len: Optional[torch.Tensor] = None, alibi: bool = False,
                  alibi_slopes: Optional[torch.Tensor] = None, softcap: Optional[float] = None,
                  q_offset: int = 0, block_mask: Optional[BlockMask] = None,
                  blocks: Optional[torch.Tensor] = None,
                  rel_bias: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None) -> None:
    """Attention forward into caller-provided ``out`` (and ``lse``).
    ``blocks``: uint8 block map [B or 1, ceil(S_q/128), ceil(S_k/128)]
    (0 hides the 128 x 128 tile); ``rel_bias``: float32 [H, 2R+1] added as
    rel_bias[h, clamp(kpos - qpos, -R, R) + R]."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, S, D]")
    B, H, S_q, D = q.shape
    Bk, H_kv, S_k, Dk = k.shape
    if (Bk, Dk) != (B, D) or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k and v")
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.device != dev or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous bfloat16 tensor on %s" % (name, dev))
    if tuple(out.shape) != (B, H, S_q, D):
        raise ValueError("out must be [B, H, S_q, D]")
    if lse is not None and (lse.device != dev or lse.dtype != torch.float32
                            or not lse.is_contiguous() or tuple(lse.shape) != (B, H, S_q)):
        raise ValueError("lse must be a contiguous float32 [B, H, S_q] tensor on %s" % dev)
    _check_mask_arrays(dev, doc_ids, prefix_len, alibi_slopes, blocks, rel_bias)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    m, keep = _mod_desc(causal=causal, window=window, doc_ids=doc_ids, prefix_len=prefix_len,
                        alibi=alibi, alibi_slopes=alibi_slopes, softcap=softcap,
                        q_offset=q_offset, block_mask=block_mask, blocks=blocks,
                        rel_bias=rel_bias)
    with torch.cuda.device(dev):
        st = _lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), _ptr(lse),
                           B, H, H_kv, S_q, S_k, D, float(scale), ctypes.byref(m),
                           _stream_ptr(stream, dev))
    del keep
    _check(st, "attn_fwd")


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, return_lse: bool = True,
             stream: Optional[torch.cuda.Stream] = None, **kw):
    """Fused attention forward.  Returns ``(O, LSE)`` (or ``O`` when
    ``return_lse`` is False).  Keywords: ``scale`` (default 1/sqrt(D)),
    ``causal``, ``window``, ``doc_ids`` [B,S] int32, ``prefix_len`` [B]
    int32, ``alibi`` / ``alibi_slopes`` [H] fp32, ``softcap``, ``q_offset``,
    ``block_mask`` (from :func:`build_block_mask`)."""
    B, H, S_q, D = q.shape
    out = torch.empty((B, H, S_q, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, S_q), dtype=torch.float32, device=q.device) if return_lse else None
    attn_fwd_into(q, k, v, out, lse, stream=stream, **kw)
    return (out, lse) if return_lse else out


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
             lse: torch.Tensor, dout: torch.Tensor, *, scale: Optional[float] = None,
             stream: Optional[torch.cuda.Stream] = None, dq: Optional[torch.Tensor] = None,
             dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None, **mods):
    """Gradients of :func:`attn_fwd`: returns ``(dQ, dK, dV)`` (bf16, shapes
    of q, k, v) for the upstream gradient ``dout`` of ``out``.  ``out`` and
    ``lse`` are the forward's results for the same inputs, scale and mods
    (keywords as for :func:`attn_fwd`, without ``block_mask``).  ``dq``,
    ``dk``, ``dv``: caller-provided outputs (contiguous bf16, the shapes of
    q, k, v), written and returned instead of new tensors."""
    B, H, S_q, D = q.shape
    _, H_kv, S_k, _ = k.shape
    dev = q.device
    for name, t, shape, dt in (("q", q, (B, H, S_q, D), torch.bfloat16),
                               ("k", k, (B, H_kv, S_k, D), torch.bfloat16),
                               ("v", v, (B, H_kv, S_k, D), torch.bfloat16),
                               ("out", out, (B, H, S_q, D), torch.bfloat16),
                               ("lse", lse, (B, H, S_q), torch.float32),
                               ("dout", dout, (B, H, S_q, D), torch.bfloat16)):
        if (t.device != dev or t.dtype != dt or not t.is_contiguous()
                or tuple(t.shape) != shape):
            raise ValueError("%s must be a contiguous %s %s tensor on %s" % (name, dt, shape, dev))
    _check_mask_arrays(dev, mods.get("doc_ids"), mods.get("prefix_len"), mods.get("alibi_slopes"),
                       mods.get("blocks"), mods.get("rel_bias"))
    if "block_mask" in mods:
        raise ValueError("attn_bwd builds its own block masks")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, shape in (("dq", dq, (B, H, S_q, D)), ("dk", dk, (B, H_kv, S_k, D)),
                           ("dv", dv, (B, H_kv, S_k, D))):
        if (t.device != dev or t.dtype != torch.bfloat16 or not t.is_contiguous()
                or tuple(t.shape) != shape):
            raise ValueError("%s must be a contiguous bfloat16 %s tensor on %s" % (name, shape, dev))
    m, keep = _mod_desc(**mods)
    with torch.cuda.device(dev):
        st = _lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                           dv.data_ptr(), B, H, H_kv, S_q, S_k, D, float(scale),
                           ctypes.byref(m), _stream_ptr(stream, dev))
    del keep
    _check(st, "attn_bwd")
    return dq, dk, dv


def attn_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *,
                  out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  return_lse: bool = True, scale: Optional[float] = None, device=None,
                  stream: Optional[torch.cuda.Stream] = None, **mods):
    """Attention forward on tensors in host memory (the library copies them
    in and the results out).  ``q``, ``k``, ``v`` and the mask arrays
    (``doc_ids``, ``prefix_len``, ``alibi_slopes``) are CPU tensors --
    page-locked (``pin_memory()``) for full copy speed.  Returns CPU
    ``(O, LSE)`` (or ``O``), written into ``out`` / ``lse`` when given.

    Asynchronous: the call is ordered on ``stream`` (default: the current
    stream of ``device``, default ``cuda``); synchronise it before reading
    the results or changing the inputs.  Consecutive calls overlap their
    copies with each other's compute."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, S, D]")
    B, H, S_q, D = q.shape
    Bk, H_kv, S_k, Dk = k.shape
    if (Bk, Dk) != (B, D) or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k and v")
    cpu = torch.device("cpu")
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((B, H, S_q, D), dtype=torch.bfloat16, pin_memory=pin)
    if lse is None and return_lse:
        lse = torch.empty((B, H, S_q), dtype=torch.float32, pin_memory=pin)
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.device != cpu or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous bfloat16 CPU tensor" % name)
    if tuple(out.shape) != (B, H, S_q, D):
        raise ValueError("out must be [B, H, S_q, D]")
    if lse is not None and (lse.device != cpu or lse.dtype != torch.float32
                            or not lse.is_contiguous() or tuple(lse.shape) != (B, H, S_q)):
        raise ValueError("lse must be a contiguous float32 [B, H, S_q] CPU tensor")
    _check_mask_arrays(cpu, mods.get("doc_ids"), mods.get("prefix_len"), mods.get("alibi_slopes"),
                       mods.get("blocks"), mods.get("rel_bias"))
    if "block_mask" in mods:
        raise ValueError("attn_fwd_host builds its own block mask")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    m, keep = _mod_desc(**mods)
    dev = torch.device(device if device is not None else "cuda")
    with torch.cuda.device(dev):
        st = _lib.attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                _ptr(lse), B, H, H_kv, S_q, S_k, D, float(scale),
                                ctypes.byref(m), _stream_ptr(stream, dev))
    del keep
    _check(st, "attn_fwd_host")
    return (out, lse) if return_lse else out


def get_device_status(stream: Optional[torch.cuda.Stream] = None, device=None) -> int:
    """Synchronise and return (then clear) the device status word."""
    device = torch.device(device if device is not None else "cuda")
    with torch.cuda.device(device):
        return int(_lib.attn_get_device_status(_stream_ptr(stream, device)))


def get_noalloc_status(stream: Optional[torch.cuda.Stream] = None, device=None) -> int:
    """Synchronise and return (then clear) the status word of the
    allocation-free entry point's fixed scratch array."""
    device = torch.device(device if device is not None else "cuda")
    with torch.cuda.device(device):
        return int(_lib.attn_get_noalloc_status(_stream_ptr(stream, device)))


def set_option(name: str, value: float) -> None:
    _check(_lib.attn_set_option(_OPTIONS[name], float(value)), "attn_set_option(%s)" % name)


def get_option(name: str) -> float:
    v = ctypes.c_double()
    _check(_lib.attn_get_option(_OPTIONS[name], ctypes.byref(v)), "attn_get_option(%s)" % name)
    return v.value


_HDR_FMT = "<IIiiiiiiiiIiiiiiQQQQQQQiiQQ"  # mirrors the device block-mask header


def decode_block_mask(bm: BlockMask) -> dict:
    """Host copy of a block mask for inspection: header fields, per-entry
    counts, work order, key-tile lists, the class grid
    ``cls[mask_batch][q_tile][k_tile]`` (0 EMPTY, 1 PARTIAL, 2 FULL) and, with
    a document mask, ``doc_lo`` / ``doc_hi[mask_batch][token]`` (the run of
    equal ids holding each token).  Synchronises the device."""
    import struct

    import numpy as np

    raw = bm.buf.cpu().numpy()
    hsz = struct.calcsize(_HDR_FMT)
    f = struct.unpack(_HDR_FMT, raw[:hsz].tobytes())
    keys = ("magic", "version", "B", "S_q", "S_k", "nQ", "nK", "nP", "bm", "n_entries",
            "mask_flags", "window", "q_offset", "force_partial", "uniform", "max_cnt",
            "doc_ptr", "prefix_ptr", "order_off", "cnt_off", "list_off", "total_bytes",
            "doc_off", "docs_sorted", "tiles_per_entry", "blocks_ptr", "pad2")
    h = dict(zip(keys, f))
    n, nK, nP, nQ = h["n_entries"], h["nK"], h["nP"], h["nQ"]
    order = raw[h["order_off"]:h["order_off"] + 4 * n].view(np.int32).copy()
    cnt = raw[h["cnt_off"]:h["cnt_off"] + 4 * n].view(np.int32).copy()
    lst = raw[h["list_off"]:h["list_off"] + 4 * n * nK].view(np.uint32).reshape(n, nK).copy()
    tpe = h["tiles_per_entry"]  # query tiles per entry: 2, or 4 for the CTA-pair forward
    cls = np.zeros((h["bm"], nQ, nK), dtype=np.int8)
    for e in range(n):
        b, p = divmod(e, nP)
        for x in lst[e, :cnt[e]]:
            kt = int(x) & 0xFFFFFF
            for t in range(tpe):
                if tpe * p + t < nQ:
                    cls[b, tpe * p + t, kt] = (int(x) >> (24 + 2 * t)) & 3
    h.update(order=order, cnt=cnt, list=lst, cls=cls)
    if h["doc_off"]:  # document mask: first / last key of each token's run of equal ids
        bm_, S = h["bm"], h["S_k"]
        d = raw[h["doc_off"]:h["doc_off"] + 8 * bm_ * S].view(np.int32).reshape(2, bm_, S)
        h.update(doc_lo=d[0].copy(), doc_hi=d[1].copy())
    return h
