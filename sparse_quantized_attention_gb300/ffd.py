"""Thin Python binding of libffd.so (ctypes): argument marshalling only.

Every entry point has the name of its C counterpart in include/ffd.h and forwards torch tensors
as raw device pointers. Nothing here computes any step of the method; a missing or unloadable
library raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import NamedTuple

import torch

from . import _build

_lock = threading.Lock()
_lib = None

FFD_OK = 0
FFD_ERR_CUDA = 4
STATUS_NAMES = {0: "FFD_OK", 1: "FFD_ERR_INVALID_ARG", 2: "FFD_ERR_UNSUPPORTED",
                3: "FFD_ERR_WORKSPACE", 4: "FFD_ERR_CUDA", 5: "FFD_ERR_BOUNDS",
                6: "FFD_ERR_RANGE", 7: "FFD_ERR_TIMEOUT"}
HEAD_DIM = 128
PAGE = 64
SCHEDULE_FUSED = 0        # FFD_SCHEDULE_FUSED
SCHEDULE_SCAN_REFINE = 1  # FFD_SCHEDULE_SCAN_REFINE


class FFDError(RuntimeError):
    def __init__(self, status: int, where: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        extra = f" (cudaError_t {cuda_error})" if cuda_error else ""
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}{extra}")


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32)]


class DecodeParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("sink_tokens", ctypes.c_int32),
                ("local_tokens", ctypes.c_int32), ("delta", ctypes.c_float),
                ("sm_scale", ctypes.c_float), ("num_splits", ctypes.c_int32),
                ("wait_limit_us", ctypes.c_int32), ("schedule", ctypes.c_int32)]


def make_params(batch, num_q_heads, num_kv_heads, num_pages, max_blocks_per_seq, *, sink=64,
                local=1024, delta=5.0, sm_scale=None, num_splits=0,
                wait_limit_us=0, schedule=0) -> DecodeParams:
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    return DecodeParams(batch, num_q_heads, num_kv_heads, HEAD_DIM, PAGE, num_pages,
                        max_blocks_per_seq, sink, local, delta, sm_scale, num_splits,
                        wait_limit_us, schedule)


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libffd.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"{_build.LIB} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(_build.LIB)
            P = ctypes.c_void_p
            st = ctypes.c_int
            L.ffd_status_string.argtypes = [st]
            L.ffd_status_string.restype = ctypes.c_char_p
            L.ffd_version.argtypes = []
            L.ffd_version.restype = ctypes.c_int32
            L.ffd_last_cuda_error.argtypes = []
            L.ffd_last_cuda_error.restype = ctypes.c_int32
            L.ffd_suggest_schedule.argtypes = [ctypes.c_int64, ctypes.c_int64]
            L.ffd_suggest_schedule.restype = ctypes.c_int32
            L.ffd_quantize_keys.argtypes = [ctypes.POINTER(CacheDesc), P, P, P, P,
                                            ctypes.c_int32, P, P]
            L.ffd_quantize_keys.restype = st
            L.ffd_append_kv.argtypes = [ctypes.POINTER(CacheDesc), ctypes.c_int32,
                                        ctypes.c_int32] + [P] * 10
            L.ffd_append_kv.restype = st
            L.ffd_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeParams)]
            L.ffd_decode_workspace_size.restype = ctypes.c_size_t
            L.ffd_dense_workspace_size.argtypes = [ctypes.POINTER(DecodeParams)]
            L.ffd_dense_workspace_size.restype = ctypes.c_size_t
            L.ffd_decode_attention.argtypes = [ctypes.POINTER(DecodeParams)] + [P] * 10 + \
                [ctypes.c_size_t, P]
            L.ffd_decode_attention.restype = st
            L.ffd_dense_decode.argtypes = [ctypes.POINTER(DecodeParams)] + [P] * 7 + \
                [ctypes.c_size_t, P]
            L.ffd_dense_decode.restype = st
            L.ffd_decode_attention_static.argtypes = [ctypes.POINTER(DecodeParams)] + \
                [P] * 11
            L.ffd_decode_attention_static.restype = st
            L.ffd_select_workspace_size.argtypes = [ctypes.POINTER(DecodeParams)]
            L.ffd_select_workspace_size.restype = ctypes.c_size_t
            L.ffd_select_blocks.argtypes = [ctypes.POINTER(DecodeParams), ctypes.c_int32,
                                            ctypes.c_float] + [P] * 6 + [ctypes.c_size_t, P]
            L.ffd_select_blocks.restype = st
            L.ffd_decode_attention_masked.argtypes = [ctypes.POINTER(DecodeParams)] + \
                [P] * 11 + [ctypes.c_size_t, P]
            L.ffd_decode_attention_masked.restype = st
            L.ffd_art_workspace_size.argtypes = [ctypes.POINTER(DecodeParams)]
            L.ffd_art_workspace_size.restype = ctypes.c_size_t
            L.ffd_art_attention.argtypes = [ctypes.POINTER(DecodeParams), ctypes.c_float,
                                            ctypes.c_float, ctypes.c_int32] + [P] * 10 + \
                [ctypes.c_size_t, P]
            L.ffd_art_attention.restype = st
            L.ffd_set_profile_events.argtypes = [P, P]
            L.ffd_set_profile_events.restype = st
            L.ffd_get_error.argtypes = [P, P]
            L.ffd_get_error.restype = st
            _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status: int, where: str):
    if status != FFD_OK:
        raise FFDError(status, where,
                       ffd_last_cuda_error() if status == FFD_ERR_CUDA else 0)


THUMB_RECORD_BYTES = 3072
RESID_RECORD_BYTES = 8704


class QuantizedCache(NamedTuple):
    """The stored key cache, one record pair per (page, KV head), byte layouts in include/ffd.h:
    thumb u8 [P, Hkv, 3072] (2-bit codes, thumbnail scales, zeros); resid u8 [P, Hkv, 8704]
    (int8 residual codes in the kernel's chunk order, residual scales)."""
    thumb: torch.Tensor
    resid: torch.Tensor


def alloc_quantized_cache(num_pages: int, num_kv_heads: int, device="cuda") -> QuantizedCache:
    shp = (num_pages, num_kv_heads)
    return QuantizedCache(
        torch.empty(shp + (THUMB_RECORD_BYTES,), dtype=torch.uint8, device=device),
        torch.empty(shp + (RESID_RECORD_BYTES,), dtype=torch.uint8, device=device))


def ffd_status_string(status: int) -> str:
    return lib().ffd_status_string(status).decode()


def ffd_version() -> int:
    return int(lib().ffd_version())


def ffd_suggest_schedule(total_blocks: int, kept_blocks: int) -> int:
    """SCHEDULE_FUSED or SCHEDULE_SCAN_REFINE for a step like the previous one (host only)."""
    return int(lib().ffd_suggest_schedule(int(total_blocks), int(kept_blocks)))


def ffd_last_cuda_error() -> int:
    """The cudaError_t behind this thread's latest FFD_ERR_CUDA (0 if none)."""
    return int(lib().ffd_last_cuda_error())


def ffd_quantize_keys(k: torch.Tensor, cache: QuantizedCache, *, page_ids=None,
                      error_word=None, stream=None) -> None:
    """Quantise bf16 keys k [P,Hkv,64,128] into ``cache`` (all pages, or ``page_ids``)."""
    desc = CacheDesc(k.shape[0], k.shape[1], k.shape[3], k.shape[2])
    n_ids = 0 if page_ids is None else int(page_ids.numel())
    _check(lib().ffd_quantize_keys(ctypes.byref(desc), _ptr(k), *map(_ptr, cache),
                                   _ptr(page_ids), n_ids, _ptr(error_word), _stream(stream)),
           "ffd_quantize_keys")


def ffd_append_kv(k_new, v_new, positions, block_table, cache: QuantizedCache, v_cache, *,
                  k_cache=None, error_word=None, stream=None) -> None:
    """Append one token per sequence: k_new, v_new bf16 [B,Hkv,128] go to row p % 64 of page
    block_table[b, p // 64], p = positions[b] (negative: nothing for that sequence)."""
    P, Hkv = v_cache.shape[0], v_cache.shape[1]
    desc = CacheDesc(P, Hkv, v_cache.shape[3], v_cache.shape[2])
    _check(lib().ffd_append_kv(ctypes.byref(desc), k_new.shape[0], block_table.shape[1],
                               _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(block_table),
                               *map(_ptr, cache), _ptr(v_cache), _ptr(k_cache),
                               _ptr(error_word), _stream(stream)), "ffd_append_kv")


def ffd_decode_workspace_size(params: DecodeParams) -> int:
    return int(lib().ffd_decode_workspace_size(ctypes.byref(params)))


def ffd_dense_workspace_size(params: DecodeParams) -> int:
    return int(lib().ffd_dense_workspace_size(ctypes.byref(params)))


def alloc_workspace(params: DecodeParams, *, dense=False, device="cuda") -> torch.Tensor:
    """Zero-filled workspace of the size the library asks for (torch allocates it)."""
    n = ffd_dense_workspace_size(params) if dense else ffd_decode_workspace_size(params)
    if n == 0:
        raise FFDError(1, "workspace size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def ffd_decode_attention(params: DecodeParams, q, cache: QuantizedCache, v, seq_lens,
                         block_table, out, workspace, *, keep_mask=None, m_tilde=None,
                         stream=None) -> None:
    _check(lib().ffd_decode_attention(
        ctypes.byref(params), _ptr(q), *map(_ptr, cache), _ptr(v), _ptr(seq_lens),
        _ptr(block_table), _ptr(out), _ptr(keep_mask), _ptr(m_tilde), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)), "ffd_decode_attention")


def ffd_decode_attention_static(params: DecodeParams, q, cache: QuantizedCache, v, seq_lens,
                                block_table, out, *, keep_mask=None, m_tilde=None,
                                error_word=None, stream=None) -> None:
    """ffd_decode_attention without a workspace, for callers that cannot allocate device memory:
    the library's own 4 MiB static device scratch is used instead (calls that overlap on the GPU
    race on it; the first call on a device should precede any stream capture)."""
    _check(lib().ffd_decode_attention_static(
        ctypes.byref(params), _ptr(q), *map(_ptr, cache), _ptr(v), _ptr(seq_lens),
        _ptr(block_table), _ptr(out), _ptr(keep_mask), _ptr(m_tilde), _ptr(error_word),
        _stream(stream)), "ffd_decode_attention_static")


SELECT_TOPK = 1
SELECT_TOPP = 2


def ffd_select_workspace_size(params: DecodeParams) -> int:
    return int(lib().ffd_select_workspace_size(ctypes.byref(params)))


def alloc_select_workspace(params: DecodeParams, device="cuda") -> torch.Tensor:
    n = ffd_select_workspace_size(params)
    if n == 0:
        raise FFDError(1, "select workspace size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def ffd_select_blocks(params: DecodeParams, selector: int, budget: float, q, cache: QuantizedCache,
                      seq_lens, block_table, keep_mask, workspace, *, stream=None) -> None:
    """Top-k (selector 1, budget = k) or Top-p (selector 2, budget = p) block mask."""
    _check(lib().ffd_select_blocks(
        ctypes.byref(params), selector, budget, _ptr(q), _ptr(cache.thumb), _ptr(seq_lens),
        _ptr(block_table), _ptr(keep_mask), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)), "ffd_select_blocks")


def ffd_decode_attention_masked(params: DecodeParams, q, cache: QuantizedCache, v, seq_lens,
                                block_table, keep_in, out, workspace, *, keep_mask=None,
                                m_tilde=None, stream=None) -> None:
    """Exact attention over the blocks a given mask selects (the decode workspace)."""
    _check(lib().ffd_decode_attention_masked(
        ctypes.byref(params), _ptr(q), *map(_ptr, cache), _ptr(v), _ptr(seq_lens),
        _ptr(block_table), _ptr(keep_in), _ptr(out), _ptr(keep_mask), _ptr(m_tilde),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
        "ffd_decode_attention_masked")


def ffd_art_workspace_size(params: DecodeParams) -> int:
    return int(lib().ffd_art_workspace_size(ctypes.byref(params)))


def alloc_art_workspace(params: DecodeParams, device="cuda") -> torch.Tensor:
    n = ffd_art_workspace_size(params)
    if n == 0:
        raise FFDError(1, "ART workspace size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def ffd_art_attention(params: DecodeParams, tau: float, phi: float, patience: int, q,
                      cache: QuantizedCache, v, seq_lens, block_table, out, workspace, *,
                      keep_in=None, blocks_used=None, stream=None) -> None:
    """Attention with run-time termination (ART) over block 0 and the blocks of ``keep_in`` (all
    blocks when None), most recent first; ``blocks_used`` [B, Hkv] int32 receives the count."""
    _check(lib().ffd_art_attention(
        ctypes.byref(params), tau, phi, patience, _ptr(q), *map(_ptr, cache), _ptr(v),
        _ptr(seq_lens), _ptr(block_table), _ptr(keep_in), _ptr(out), _ptr(blocks_used),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
        "ffd_art_attention")


def ffd_dense_decode(params: DecodeParams, q, k, v, seq_lens, block_table, out, workspace, *,
                     stream=None) -> None:
    _check(lib().ffd_dense_decode(
        ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), _ptr(block_table),
        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "ffd_dense_decode")


def ffd_get_error(error_word, *, stream=None) -> int:
    """Synchronise, read and clear a device error word; returns the status code."""
    return int(lib().ffd_get_error(_ptr(error_word), _stream(stream)))


def ffd_set_profile_events(start=None, stop=None) -> None:
    """Record ``start`` / ``stop`` (torch.cuda.Event, created) around the main kernel of the
    following decode calls; ``None, None`` turns it off."""
    def raw(ev):
        if ev is None:
            return None
        return ctypes.c_void_p(ev.cuda_event)
    _check(lib().ffd_set_profile_events(raw(start), raw(stop)), "ffd_set_profile_events")
