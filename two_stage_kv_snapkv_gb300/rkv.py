"""Thin Python binding of librkv (include/rkv.h).

Argument marshalling only: every step of the hot path runs in the CUDA library.
torch tensors provide device memory and streams.  Importing this module loads
``_build/librkv.so`` and raises if it has not been built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import functools
import math
import os
from typing import Optional, Sequence

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "librkv.so")

RKV_OK = 0
RKV_ERR_INVALID_ARG = 1
RKV_ERR_UNSUPPORTED = 2
RKV_ERR_WORKSPACE = 3
RKV_ERR_CUDA = 4
RKV_ERR_DEVICE_DATA = 5
RKV_ERR_TIMEOUT = 6
DEVERR_PAGE_ID = 0x1
DEVERR_CAPACITY = 0x2
DEVERR_TIMEOUT = 0x4
DEVERR_SEQ_LEN = 0x8
HEAD_DIM = 128
MAX_BATCH = 256


class RkvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"rkv status {status}: {msg}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"librkv.so is not built ({_LIB_PATH}); run `python -c 'import __graft_entry__ as g; g.build()'`")
    return ctypes.CDLL(_LIB_PATH)


_lib = _load()


class RkvSplit(ctypes.Structure):
    _fields_ = [("c", ctypes.c_double), ("r", ctypes.c_double), ("c1", ctypes.c_double), ("c2", ctypes.c_double),
                ("keep1", ctypes.c_int32), ("k1", ctypes.c_int32), ("k2", ctypes.c_int32),
                ("pool_kernel", ctypes.c_int32)]


class RkvCacheStruct(ctypes.Structure):
    _fields_ = [("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("seq_len", ctypes.c_void_p), ("kmax", ctypes.c_void_p), ("kmin", ctypes.c_void_p),
                ("error_word", ctypes.c_void_p), ("step_sync", ctypes.c_void_p), ("B", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("num_phys_pages", ctypes.c_int32)]


_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
_i32p = ctypes.POINTER(ctypes.c_int32)
_lib.rkv_split_ratio.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(RkvSplit)]
_lib.rkv_split_ratio.restype = _i32
_lib.rkv_split_ratio_mt.argtypes = [_i32, _i32, _i32, _i32, _i32, ctypes.POINTER(RkvSplit)]
_lib.rkv_split_ratio_mt.restype = _i32
_lib.rkv_prefill_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32]
_lib.rkv_prefill_workspace_size.restype = _sz
_lib.rkv_prefill_evict.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32p, _i32p, _i32p, _f32,
                                   ctypes.POINTER(RkvCacheStruct), _vp, _i32, _vp, _vp, _sz, _vp]
_lib.rkv_prefill_evict.restype = _i32
_lib.rkv_prefill_chunk_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32]
_lib.rkv_prefill_chunk_workspace_size.restype = _sz
_lib.rkv_prefill_chunk.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32p, _i32p, _i32p, _i32p, _f32,
                                   ctypes.POINTER(RkvCacheStruct), _vp, _i32, _vp, _sz, _vp]
_lib.rkv_prefill_chunk.restype = _i32
_lib.rkv_append_page_summary.argtypes = [ctypes.POINTER(RkvCacheStruct), _vp, _vp, _i32, _vp]
_lib.rkv_append_page_summary.restype = _i32
_lib.rkv_decode_workspace_size.argtypes = [_i32, _i32, _i32, _i32]
_lib.rkv_decode_workspace_size.restype = _sz
_lib.rkv_decode_hsa.argtypes = [ctypes.POINTER(RkvCacheStruct), _vp, _i32, _i32p, _i32p, _f32, _vp, _vp, _vp, _i32,
                                _vp, _sz, _vp]
_lib.rkv_decode_hsa.restype = _i32
_lib.rkv_decode_step.argtypes = [ctypes.POINTER(RkvCacheStruct), _vp, _vp, _vp, _i32, _i32p, _i32p, _f32, _vp, _vp,
                                 _vp, _i32, _vp, _sz, _vp]
_lib.rkv_decode_step.restype = _i32
_lib.rkv_decode_path.argtypes = [_i32]
_lib.rkv_decode_path.restype = _i32
_lib.rkv_decode_hsa_noalloc.argtypes = [ctypes.POINTER(RkvCacheStruct), _vp, _i32, _i32p, _i32p, _f32, _vp, _vp,
                                        _vp, _i32, _vp]
_lib.rkv_decode_hsa_noalloc.restype = _i32
_lib.rkv_step_host_staging_size.argtypes = [_i32, _i32, _i32]
_lib.rkv_step_host_staging_size.restype = _sz
_lib.rkv_decode_step_host.argtypes = [ctypes.POINTER(RkvCacheStruct), _vp, _vp, _i32, _i32p, _i32p, _f32, _vp, _sz,
                                      _vp, _sz, _vp]
_lib.rkv_decode_step_host.restype = _i32
_lib.rkv_sparq_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32]
_lib.rkv_sparq_workspace_size.restype = _sz
_lib.rkv_decode_sparq.argtypes = [ctypes.POINTER(RkvCacheStruct), _vp, _i32, _i32p, _i32p, _f32, _vp, _vp, _vp, _i32,
                                  _vp, _sz, _vp, _sz, _vp]
_lib.rkv_sparq_keys_size.argtypes = [_i32, _i32, _i32, _i32]
_lib.rkv_sparq_keys_size.restype = _sz
_lib.rkv_decode_sparq.restype = _i32
_lib.rkv_exact_topk_recall.argtypes = [ctypes.POINTER(RkvCacheStruct), _vp, _i32, _vp, _i32, _i32p, _f32, _vp, _vp,
                                       _vp]
_lib.rkv_exact_topk_recall.restype = _i32
_lib.rkv_selftest_bounded_wait.argtypes = [ctypes.POINTER(RkvCacheStruct), ctypes.c_int64, _vp]
_lib.rkv_selftest_bounded_wait.restype = _i32
_lib.rkv_get_device_status.argtypes = [ctypes.POINTER(RkvCacheStruct), _vp, _i32p]
_lib.rkv_get_device_status.restype = _i32
_lib.rkv_last_error.argtypes = []
_lib.rkv_last_error.restype = ctypes.c_char_p
_lib.rkv_launch_count.argtypes = []
_lib.rkv_launch_count.restype = ctypes.c_int64
_lib.rkv_profile_enable.argtypes = [_i32]
_lib.rkv_profile_enable.restype = None
_lib.rkv_profile_reset.argtypes = []
_lib.rkv_profile_reset.restype = None
_lib.rkv_profile_accumulate.argtypes = []
_lib.rkv_profile_accumulate.restype = None
_lib.rkv_profile_release.argtypes = []
_lib.rkv_profile_release.restype = None
_lib.rkv_profile_read.argtypes = [_i32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)]
_lib.rkv_profile_read.restype = ctypes.c_char_p

EXPORTED = ["rkv_split_ratio", "rkv_split_ratio_mt", "rkv_prefill_workspace_size", "rkv_prefill_evict",
            "rkv_prefill_chunk_workspace_size", "rkv_prefill_chunk", "rkv_append_page_summary",
            "rkv_decode_workspace_size", "rkv_decode_hsa", "rkv_decode_hsa_noalloc", "rkv_decode_step",
            "rkv_decode_path", "rkv_step_host_staging_size", "rkv_decode_step_host", "rkv_sparq_workspace_size", "rkv_decode_sparq", "rkv_sparq_keys_size",
            "rkv_exact_topk_recall", "rkv_selftest_bounded_wait", "rkv_get_device_status", "rkv_last_error",
            "rkv_launch_count", "rkv_profile_enable", "rkv_profile_accumulate", "rkv_profile_release",
            "rkv_profile_reset", "rkv_profile_read"]


def lib() -> ctypes.CDLL:
    return _lib


def _check(status: int):
    if status != RKV_OK:
        raise RkvError(status, _lib.rkv_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to librkv must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@functools.lru_cache(maxsize=256)
def _host_i32_cached(values: tuple):
    return (ctypes.c_int32 * len(values))(*values)


def _host_i32(values: Sequence[int]):
    """Host int32 array for the C call; the library only reads it during the call, so
    arrays of the same values are built once and shared."""
    return _host_i32_cached(tuple(int(v) for v in values))


# ------------------------------------------------------------------ cache
class PagedCache:
    """Device memory of one layer's compressed paged cache (see rkv_cache in rkv.h)."""

    def __init__(self, B: int, Hkv: int, page_size: int, max_pages: int, device="cuda",
                 page_table: Optional[torch.Tensor] = None, num_phys_pages: Optional[int] = None,
                 fill: Optional[float] = None):
        max_pages = (max_pages + 7) // 8 * 8
        if page_table is None:
            page_table = torch.arange(B * max_pages, dtype=torch.int32, device=device).view(B, max_pages)
        assert page_table.shape == (B, max_pages) and page_table.dtype == torch.int32
        if num_phys_pages is None:
            num_phys_pages = int(page_table.max().item()) + 1
        self.B, self.Hkv, self.page_size, self.max_pages = B, Hkv, page_size, max_pages
        self.num_phys_pages = num_phys_pages
        self.page_table = page_table.to(device).contiguous()
        shape = (num_phys_pages, Hkv, page_size, HEAD_DIM)
        self.k_pages = torch.empty(shape, dtype=torch.bfloat16, device=device)
        self.v_pages = torch.empty(shape, dtype=torch.bfloat16, device=device)
        self.kmax = torch.empty((B, Hkv, HEAD_DIM, max_pages), dtype=torch.bfloat16, device=device)
        self.kmin = torch.empty((B, Hkv, HEAD_DIM, max_pages), dtype=torch.bfloat16, device=device)
        if fill is not None:
            for t in (self.k_pages, self.v_pages, self.kmax, self.kmin):
                t.fill_(fill)
        self.seq_len = torch.zeros(B, dtype=torch.int32, device=device)
        self.error_word = torch.zeros(4, dtype=torch.int32, device=device)
        self.step_sync = torch.zeros(B, dtype=torch.int32, device=device)
        self._struct = RkvCacheStruct(
            self.k_pages.data_ptr(), self.v_pages.data_ptr(), self.page_table.data_ptr(), self.seq_len.data_ptr(),
            self.kmax.data_ptr(), self.kmin.data_ptr(), self.error_word.data_ptr(), self.step_sync.data_ptr(), B, Hkv,
            HEAD_DIM, page_size, max_pages, num_phys_pages)

    @property
    def struct(self) -> RkvCacheStruct:
        return self._struct

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in
                   (self.k_pages, self.v_pages, self.kmax, self.kmin, self.page_table, self.seq_len))

    def token_kv(self, b: int, n: Optional[int] = None):
        """(K, V) of sequence b's first n tokens, [Hkv, n, 128] (gathered by torch; for checks)."""
        if n is None:
            n = int(self.seq_len[b].item())
        P = self.page_size
        npg = -(-n // P)
        phys = self.page_table[b, :npg].long()
        K = self.k_pages[phys].permute(1, 0, 2, 3).reshape(self.Hkv, npg * P, HEAD_DIM)[:, :n]
        V = self.v_pages[phys].permute(1, 0, 2, 3).reshape(self.Hkv, npg * P, HEAD_DIM)[:, :n]
        return K, V


# ------------------------------------------------------------------ entry points
def rkv_split_ratio(prompt_len: int, budget: int, head_dim: int = HEAD_DIM, page_size: int = 16, window: int = 32,
                    k1_override: int = 0) -> dict:
    out = RkvSplit()
    _check(_lib.rkv_split_ratio(prompt_len, budget, head_dim, page_size, window, k1_override, ctypes.byref(out)))
    return dict(c=out.c, r=out.r, c1=out.c1, c2=out.c2, keep1=out.keep1, k1=out.k1, k2=out.k2,
                pool_kernel=out.pool_kernel)


def rkv_split_ratio_mt(prompt_len: int, budget: int, head_dim: int = HEAD_DIM, page_size: int = 16,
                       k1_override: int = 0) -> dict:
    """RocketKV-MT's split: nothing evicted (keep1 = prompt_len), HSA takes the whole ratio."""
    out = RkvSplit()
    _check(_lib.rkv_split_ratio_mt(prompt_len, budget, head_dim, page_size, k1_override, ctypes.byref(out)))
    return dict(c=out.c, r=out.r, c1=out.c1, c2=out.c2, keep1=out.keep1, k1=out.k1, k2=out.k2,
                pool_kernel=out.pool_kernel)


def prefill_workspace(B: int, Hq: int, Hkv: int, window: int, max_prompt_len: int, device="cuda") -> torch.Tensor:
    n = _lib.rkv_prefill_workspace_size(B, Hq, Hkv, window, max_prompt_len)
    return torch.empty(n, dtype=torch.uint8, device=device)


def decode_workspace(B: int, Hq: int, Hkv: int, max_pages: int, device="cuda") -> torch.Tensor:
    n = _lib.rkv_decode_workspace_size(B, Hq, Hkv, max_pages)
    return torch.empty(n, dtype=torch.uint8, device=device)


def rkv_prefill_evict(q_win: torch.Tensor, k: torch.Tensor, v: torch.Tensor, prompt_len: Sequence[int],
                      keep1: Sequence[int], pool_kernel: Sequence[int], cache: PagedCache, kept_idx: torch.Tensor,
                      pooled_scores: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None):
    B, Hq, w, d = q_win.shape
    Lmax = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = prefill_workspace(B, Hq, cache.Hkv, w, Lmax, q_win.device)
    _check(_lib.rkv_prefill_evict(_ptr(q_win), _ptr(k), _ptr(v), B, Hq, w, Lmax, _host_i32(prompt_len),
                                  _host_i32(keep1), _host_i32(pool_kernel), scale, ctypes.byref(cache.struct),
                                  _ptr(kept_idx), kept_idx.shape[-1], _ptr(pooled_scores), _ptr(workspace),
                                  workspace.numel(), _stream(stream)))


def prefill_chunk_workspace(B: int, Hq: int, Hkv: int, window: int, max_total_len: int,
                            device="cuda") -> torch.Tensor:
    n = _lib.rkv_prefill_chunk_workspace_size(B, Hq, Hkv, window, max_total_len)
    return torch.empty(n, dtype=torch.uint8, device=device)


def rkv_prefill_chunk(q_win: torch.Tensor, k_chunk: torch.Tensor, v_chunk: torch.Tensor, chunk_len: Sequence[int],
                      held_len: Sequence[int], keep1: Sequence[int], pool_kernel: Sequence[int], cache: PagedCache,
                      kept_idx: torch.Tensor, scale: Optional[float] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None):
    """One chunk of a chunked prefill; held_len is the cache's seq_len before the call."""
    B, Hq, w, d = q_win.shape
    chunk_max = k_chunk.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        total = max(int(h) + int(m) for h, m in zip(held_len, chunk_len))
        workspace = prefill_chunk_workspace(B, Hq, cache.Hkv, w, total, q_win.device)
    _check(_lib.rkv_prefill_chunk(_ptr(q_win), _ptr(k_chunk), _ptr(v_chunk), B, Hq, w, chunk_max,
                                  _host_i32(chunk_len), _host_i32(held_len), _host_i32(keep1),
                                  _host_i32(pool_kernel), scale, ctypes.byref(cache.struct), _ptr(kept_idx),
                                  kept_idx.shape[-1], _ptr(workspace), workspace.numel(), _stream(stream)))


def rkv_append_page_summary(cache: PagedCache, k_new: Optional[torch.Tensor] = None,
                            v_new: Optional[torch.Tensor] = None, n_new: Optional[int] = None, stream=None):
    if n_new is None:
        n_new = 1 if k_new is None or k_new.dim() == 3 else k_new.shape[2]
    _check(_lib.rkv_append_page_summary(ctypes.byref(cache.struct), _ptr(k_new), _ptr(v_new), n_new,
                                        _stream(stream)))


def rkv_decode_hsa(cache: PagedCache, q: torch.Tensor, k1: Sequence[int], k2: Sequence[int], out: torch.Tensor,
                   sel_channels: Optional[torch.Tensor] = None, sel_pages: Optional[torch.Tensor] = None,
                   scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    B, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = decode_workspace(B, Hq, cache.Hkv, cache.max_pages, q.device)
    stride = sel_pages.shape[-1] if sel_pages is not None else 0
    _check(_lib.rkv_decode_hsa(ctypes.byref(cache.struct), _ptr(q), Hq, _host_i32(k1), _host_i32(k2), scale,
                               _ptr(out), _ptr(sel_channels), _ptr(sel_pages), stride, _ptr(workspace),
                               workspace.numel(), _stream(stream)))


def rkv_decode_step(cache: PagedCache, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                    k1: Sequence[int], k2: Sequence[int], out: torch.Tensor,
                    sel_channels: Optional[torch.Tensor] = None, sel_pages: Optional[torch.Tensor] = None,
                    scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Append one token ([B, Hkv, 128] k_new / v_new) and run the HSA step, as one launch."""
    B, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = decode_workspace(B, Hq, cache.Hkv, cache.max_pages, q.device)
    stride = sel_pages.shape[-1] if sel_pages is not None else 0
    _check(_lib.rkv_decode_step(ctypes.byref(cache.struct), _ptr(q), _ptr(k_new), _ptr(v_new), Hq, _host_i32(k1),
                                _host_i32(k2), scale, _ptr(out), _ptr(sel_channels), _ptr(sel_pages), stride,
                                _ptr(workspace), workspace.numel(), _stream(stream)))


def step_host_staging(B: int, Hq: int, Hkv: int, device="cuda") -> torch.Tensor:
    n = _lib.rkv_step_host_staging_size(B, Hq, Hkv)
    return torch.empty(n, dtype=torch.uint8, device=device)


def rkv_decode_step_host(cache: PagedCache, host_in: torch.Tensor, host_out: torch.Tensor, Hq: int,
                         k1: Sequence[int], k2: Sequence[int], staging: torch.Tensor, workspace: torch.Tensor,
                         scale: Optional[float] = None, stream=None):
    """rkv_decode_step from host buffers: host_in packs q, k_new, v_new (bf16, in that
    order); host_out [B, Hq, 128] fp32 receives the output.  Pinned host tensors keep
    the two copies asynchronous."""
    if scale is None:
        scale = 1.0 / math.sqrt(HEAD_DIM)
    if host_in.is_cuda or host_out.is_cuda:
        raise ValueError("host_in and host_out are host tensors")
    _check(_lib.rkv_decode_step_host(ctypes.byref(cache.struct), _ptr(host_in), _ptr(host_out), Hq, _host_i32(k1),
                                     _host_i32(k2), scale, _ptr(staging), staging.numel(), _ptr(workspace),
                                     workspace.numel(), _stream(stream)))


def sparq_workspace(B: int, Hq: int, Hkv: int, max_pages: int, page_size: int, device="cuda") -> torch.Tensor:
    n = _lib.rkv_sparq_workspace_size(B, Hq, Hkv, max_pages, page_size)
    return torch.empty(n, dtype=torch.uint8, device=device)


def sparq_keys(cache: "PagedCache", device="cuda") -> torch.Tensor:
    """A zero-filled (empty) channel-major key copy for rkv_decode_sparq's keys_t."""
    n = _lib.rkv_sparq_keys_size(cache.B, cache.Hkv, cache.max_pages, cache.page_size)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def rkv_decode_sparq(cache: PagedCache, q: torch.Tensor, k1: Sequence[int], k_tokens: Sequence[int],
                     out: torch.Tensor, sel_channels: Optional[torch.Tensor] = None,
                     sel_tokens: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                     workspace: Optional[torch.Tensor] = None, keys_t: Optional[torch.Tensor] = None, stream=None):
    """SparQ-only step (HSA with one-token pages): k_tokens tokens by their partial dot
    products over the top-k1 channels, then exact attention over them.  keys_t (from
    sparq_keys) is the channel-major key copy to score from, kept between calls."""
    B, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = sparq_workspace(B, Hq, cache.Hkv, cache.max_pages, cache.page_size, q.device)
    stride = sel_tokens.shape[-1] if sel_tokens is not None else 0
    kt_bytes = keys_t.numel() * keys_t.element_size() if keys_t is not None else 0
    _check(_lib.rkv_decode_sparq(ctypes.byref(cache.struct), _ptr(q), Hq, _host_i32(k1), _host_i32(k_tokens), scale,
                                 _ptr(out), _ptr(sel_channels), _ptr(sel_tokens), stride, _ptr(keys_t), kt_bytes,
                                 _ptr(workspace), workspace.numel(), _stream(stream)))


def rkv_exact_topk_recall(cache: PagedCache, q: torch.Tensor, sel_pages: torch.Tensor, k_tokens: Sequence[int],
                          recall: Optional[torch.Tensor] = None, mass: Optional[torch.Tensor] = None,
                          scale: Optional[float] = None, stream=None) -> tuple:
    """Exact-TopK recall of a page selection, per (sequence, KV head): the share of the
    exact top-k_tokens[b] tokens (attention summed over the GQA group) and of their
    attention mass that lies in sel_pages ([B, Hkv, stride] as rkv_decode_hsa writes it).
    Returns (recall, mass), [B, Hkv] fp32 device tensors."""
    B, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if recall is None:
        recall = torch.empty((B, cache.Hkv), dtype=torch.float32, device=q.device)
    if mass is None:
        mass = torch.empty((B, cache.Hkv), dtype=torch.float32, device=q.device)
    _check(_lib.rkv_exact_topk_recall(ctypes.byref(cache.struct), _ptr(q), Hq, _ptr(sel_pages), sel_pages.shape[-1],
                                      _host_i32(k_tokens), scale, _ptr(recall), _ptr(mass), _stream(stream)))
    return recall, mass


def rkv_decode_path(path: int = -1) -> int:
    """0 auto (fused when it fits), 1 four-kernel path, 2 fused; -1 only reads the setting."""
    return int(_lib.rkv_decode_path(path))


def rkv_selftest_bounded_wait(cache: PagedCache, limit_ns: int, stream=None) -> None:
    _check(_lib.rkv_selftest_bounded_wait(ctypes.byref(cache.struct), int(limit_ns), _stream(stream)))


def rkv_get_device_status(cache: PagedCache, stream=None) -> tuple:
    bits = ctypes.c_int32(0)
    st = _lib.rkv_get_device_status(ctypes.byref(cache.struct), _stream(stream), ctypes.byref(bits))
    return st, bits.value


def rkv_last_error() -> str:
    return _lib.rkv_last_error().decode()


def rkv_launch_count() -> int:
    return int(_lib.rkv_launch_count())


def profile_enable(on: bool = True):
    _lib.rkv_profile_enable(1 if on else 0)


def profile_reset():
    _lib.rkv_profile_reset()


def profile_accumulate():
    _lib.rkv_profile_accumulate()


def profile_release():
    _lib.rkv_profile_release()


def profile_read() -> dict:
    """{kernel name: (launches, total ms)} for every kernel kind."""
    res = {}
    kind = 0
    while True:
        n = ctypes.c_int64(0)
        ms = ctypes.c_double(0.0)
        name = _lib.rkv_profile_read(kind, ctypes.byref(n), ctypes.byref(ms))
        if name is None:
            break
        res[name.decode()] = (int(n.value), float(ms.value))
        kind += 1
    return res
