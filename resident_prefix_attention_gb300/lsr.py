"""Thin Python binding of ``liblsr.so`` (the C ABI in include/lsr.h and
include/lsr_latent.h).

Argument marshalling only: every step of the replay path runs in the
library's CUDA kernels.  Tensors supply device memory, and
``torch.cuda.current_stream()`` supplies the stream.  The functions keep
the C names.  Status codes other than LSR_OK raise ``LsrError`` carrying
the library's error text.  There is no fallback: if the library is missing
the import of this module fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblsr.so")

LSR_OK = 0
LSR_ERR_INVALID_ARG = 1
LSR_ERR_UNSUPPORTED = 2
LSR_ERR_CUDA = 3
LSR_ERR_DEVICE = 4
LSR_ERR_STALE = 5
LSR_ERR_DUPLICATE = 6
LSR_ERR_STATE = 7
LSR_DEV_WAIT_TIMEOUT = 1
LSR_DEV_BAD_PAGE = 2
LSR_DEV_BOUNDS = 4

# Every function the header declares, with (restype, argtypes).
_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_PZ = ctypes.POINTER(ctypes.c_size_t)
_PI = ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "lsr_page_pool_create": (_I, [_I, _I, _I, _I, _P, _P, _P, ctypes.POINTER(_P)]),
    "lsr_page_pool_destroy": (_I, [_P]),
    "lsr_write_prefix_pages": (_I, [_P, _P, _P, _I, _I, _P, _I, _P]),
    "lsr_replay_attn_fwd": (_I, [_P, _P, _I, _I, _I, _I, _P, _I, _I, _F,
                                 _P, _P, _P, _P]),
    "lsr_lse_merge": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "lsr_bwd_workspace_size": (_I, [_I, _I, _I, _I, _PZ]),
    "lsr_replay_attn_bwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _I,
                                 _I, _F, _P, _P, _P, _P, _Z, _P]),
    "lsr_replay_attn_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I,
                                         _P, _I, _I, _F, _P, _P, _P, _P]),
    "lsr_replay_workspace_size": (_I, [_I, _I, _I, _I, _I, _PZ]),
    "lsr_replay_response": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _I, _I, _F,
                                 _P, _P, _P, _P, _P, _P, _Z, _P]),
    "lsr_pool_device_status": (_I, [_P, _PI, _P]),
    "lsr_selftest_bounded_wait": (_I, [_P, _I, _P]),
    "lsr_pool_set_wait_limit": (_I, [_P, _I]),
    "lsr_group_rows": (_I, [_I, _I, _I, _P, _P]),
    "lsr_group_workspace_size": (_I, [_I, _I, _I, _I, _PZ]),
    "lsr_replay_group": (_I, [_P, _I, _P, _P, _P, _P, _P, _I, _I, _P, _I, _I,
                              _F, _P, _P, _P, _P, _P, _I, _P, _Z, _P]),
    "lsr_pool_set_version": (_I, [_P, ctypes.c_uint64]),
    "lsr_pool_version": (_I, [_P, ctypes.POINTER(ctypes.c_uint64)]),
    "lsr_window_create": (_I, [ctypes.c_uint64, ctypes.POINTER(_P)]),
    "lsr_window_destroy": (_I, [_P]),
    "lsr_window_begin_replay": (_I, [_P, ctypes.c_uint64, ctypes.c_uint64]),
    "lsr_window_commit_replay": (_I, [_P, ctypes.c_uint64,
                                      ctypes.c_longlong]),
    "lsr_window_abort_replay": (_I, [_P, ctypes.c_uint64]),
    "lsr_window_close": (_I, [_P, ctypes.c_uint64,
                              ctypes.POINTER(ctypes.c_longlong),
                              ctypes.POINTER(ctypes.c_longlong)]),
    "lsr_score_shards": (_I, [_P, _I, _I, _I, _PI]),
    "lsr_score_workspace_size": (_I, [_I, _I, _I, _I, _PZ]),
    "lsr_score_fwd": (_I, [_P, _P, _I, _I, _I, _I, _P, _I, _I, _F, _P, _P,
                           _P, _Z, _P]),
    "lsr_profile_set": (_I, [_I]),
    "lsr_profile_read": (_I, [_I, ctypes.POINTER(ctypes.c_longlong),
                              ctypes.POINTER(ctypes.c_double)]),
    "lsr_kernel_name": (ctypes.c_char_p, [_I]),
    "lsr_last_error": (ctypes.c_char_p, []),
    # include/lsr_latent.h
    "lsr_latent_pool_create": (_I, [_I, _I, _I, _I, _P, _P,
                                    ctypes.POINTER(_P)]),
    "lsr_latent_write_pages": (_I, [_P, _P, _I, _I, _P, _I, _P]),
    "lsr_latent_attn_fwd": (_I, [_P, _P, _I, _I, _I, _I, _P, _I, _I, _F,
                                 _P, _P, _P, _P]),
    "lsr_latent_bwd_workspace_size": (_I, [_I, _I, _I, _PZ]),
    "lsr_latent_attn_bwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _I,
                                 _I, _F, _P, _P, _P, _Z, _P]),
    "lsr_latent_replay_workspace_size": (_I, [_I, _I, _I, _I, _PZ]),
    "lsr_latent_replay_response": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _I,
                                        _I, _F, _P, _P, _P, _P, _P, _Z, _P]),
    "lsr_latent_group_workspace_size": (_I, [_I, _I, _I, _PZ]),
    "lsr_latent_replay_group": (_I, [_P, _I, _P, _P, _P, _P, _P, _I, _I, _P,
                                     _I, _I, _F, _P, _P, _P, _P, _I, _P, _Z,
                                     _P]),
}

# Kernel ids of the profiling calls.
LSR_K_WRITE_PAGES, LSR_K_ATTN_FWD, LSR_K_LSE_MERGE, LSR_K_BWD_PREPROCESS, \
    LSR_K_ATTN_BWD_DQ, LSR_K_DQ_REDUCE, LSR_K_ATTN_BWD_DKDV, \
    LSR_K_LATENT_BWD_DQ, LSR_K_LATENT_BWD_DLAT = range(9)
LSR_K_COUNT = 9


class LsrError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"lsr status {status}: {msg}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _check(status: int):
    if status != LSR_OK:
        raise LsrError(status, _lib.lsr_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    """Device address of a contiguous CUDA tensor (the library's kernels
    read and write it directly, so host tensors are refused here)."""
    if t is None:
        return None
    if t.device.type != "cuda":
        raise ValueError("tensors passed to the library must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _table(t: torch.Tensor):
    """Device address of a page table (int32, logical -> physical page)."""
    if t.dtype != torch.int32:
        raise TypeError("page_table must be int32")
    return _ptr(t)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _bf16(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")


def _f32(t: torch.Tensor, name: str):
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")


class Pool:
    """Opaque handle of a paged K/V pool; holds references to its tensors."""

    def __init__(self, handle, k_pages, v_pages, status):
        self.handle = handle
        self.k_pages, self.v_pages, self.status = k_pages, v_pages, status
        self.num_pages, self.num_kv_heads, self.page_size, self.head_dim = \
            k_pages.shape

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.lsr_page_pool_destroy(h)
            self.handle = None


def lsr_page_pool_create(k_pages: torch.Tensor, v_pages: torch.Tensor,
                         dev_status: torch.Tensor) -> Pool:
    """k_pages, v_pages: bf16 [num_pages, Hkv, page_size, d]; dev_status:
    int32 [1] (zeroed)."""
    _bf16(k_pages, "k_pages")
    _bf16(v_pages, "v_pages")
    if dev_status.dtype != torch.int32:
        raise TypeError("dev_status must be int32")
    npg, hkv, ps, d = k_pages.shape
    h = ctypes.c_void_p()
    _check(_lib.lsr_page_pool_create(npg, ps, hkv, d, _ptr(k_pages),
                                     _ptr(v_pages), _ptr(dev_status),
                                     ctypes.byref(h)))
    return Pool(h, k_pages, v_pages, dev_status)


def lsr_page_pool_destroy(pool: Pool):
    if pool.handle is not None:
        _check(_lib.lsr_page_pool_destroy(pool.handle))
        pool.handle = None


def lsr_write_prefix_pages(pool: Pool, k: torch.Tensor, v: torch.Tensor,
                           pos0: int, page_table: torch.Tensor, stream=None):
    _bf16(k, "k")
    _bf16(v, "v")
    _check(_lib.lsr_write_prefix_pages(pool.handle, _ptr(k), _ptr(v),
                                       k.shape[0], pos0, _table(page_table),
                                       page_table.numel(), _stream(stream)))


def lsr_replay_attn_fwd(pool: Pool, q: torch.Tensor, P: int, resp_pos0: int,
                        page_table: torch.Tensor, num_shards: int,
                        scale: float, m: torch.Tensor, l: torch.Tensor,
                        o_part: torch.Tensor, stream=None):
    _bf16(q, "q")
    for t, n in ((m, "m"), (l, "l"), (o_part, "o_part")):
        _f32(t, n)
    R_b, Hq, _ = q.shape
    _check(_lib.lsr_replay_attn_fwd(pool.handle, _ptr(q), Hq, R_b, P,
                                    resp_pos0, _table(page_table),
                                    page_table.numel(), num_shards, scale,
                                    _ptr(m), _ptr(l), _ptr(o_part),
                                    _stream(stream)))


def lsr_lse_merge(m: torch.Tensor, l: torch.Tensor, o_part: torch.Tensor,
                  o: torch.Tensor, lse: torch.Tensor, stream=None):
    for t, n in ((m, "m"), (l, "l"), (o_part, "o_part"), (lse, "lse")):
        _f32(t, n)
    _f32(o, "o")
    parts, R_b, Hq, d = o_part.shape
    _check(_lib.lsr_lse_merge(_ptr(m), _ptr(l), _ptr(o_part), parts, Hq, R_b,
                              d, _ptr(o), _ptr(lse), _stream(stream)))


def lsr_bwd_workspace_size(num_shards: int, Hq: int, R_b: int,
                           head_dim: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.lsr_bwd_workspace_size(num_shards, Hq, R_b, head_dim,
                                       ctypes.byref(n)))
    return n.value


def lsr_replay_attn_bwd(pool: Pool, q, o, dO, lse, P: int, resp_pos0: int,
                        page_table, num_shards: int, scale: float, dq, dk_resp,
                        dv_resp, workspace: torch.Tensor, stream=None):
    for t, n in ((q, "q"), (dO, "dO")):
        _bf16(t, n)
    for t, n in ((o, "o"), (lse, "lse"), (dq, "dq"), (dk_resp, "dk_resp"),
                 (dv_resp, "dv_resp")):
        _f32(t, n)
    R_b, Hq, _ = q.shape
    _check(_lib.lsr_replay_attn_bwd(
        pool.handle, _ptr(q), _ptr(o), _ptr(dO), _ptr(lse), Hq, R_b, P,
        resp_pos0, _table(page_table), page_table.numel(), num_shards, scale,
        _ptr(dq), _ptr(dk_resp), _ptr(dv_resp), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def lsr_replay_attn_bwd_noalloc(pool: Pool, q, o, dO, lse, P: int,
                                resp_pos0: int, page_table, num_shards: int,
                                scale: float, dq, dk_resp, dv_resp,
                                stream=None):
    """lsr_replay_attn_bwd without a workspace argument: for callers that
    cannot allocate device memory at this point; the library's built-in
    64 MiB scratch is used instead (shared by all calls, so calls that
    overlap on the GPU race)."""
    for t, n in ((q, "q"), (dO, "dO")):
        _bf16(t, n)
    for t, n in ((o, "o"), (lse, "lse"), (dq, "dq"), (dk_resp, "dk_resp"),
                 (dv_resp, "dv_resp")):
        _f32(t, n)
    R_b, Hq, _ = q.shape
    _check(_lib.lsr_replay_attn_bwd_noalloc(
        pool.handle, _ptr(q), _ptr(o), _ptr(dO), _ptr(lse), Hq, R_b, P,
        resp_pos0, _table(page_table), page_table.numel(), num_shards, scale,
        _ptr(dq), _ptr(dk_resp), _ptr(dv_resp), _stream(stream)))


def lsr_replay_workspace_size(num_shards: int, Hq: int, R: int,
                              num_blocks: int, head_dim: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.lsr_replay_workspace_size(num_shards, Hq, R, num_blocks,
                                          head_dim, ctypes.byref(n)))
    return n.value


def lsr_replay_response(pool: Pool, q, dO, num_blocks: int, P: int,
                        page_table, num_shards: int, scale: float, o, lse, dq,
                        dk_resp, dv_resp, workspace: torch.Tensor,
                        stream=None):
    _bf16(q, "q")
    _bf16(dO, "dO")
    _f32(o, "o")
    R, Hq, _ = q.shape
    _check(_lib.lsr_replay_response(
        pool.handle, _ptr(q), _ptr(dO), Hq, R, num_blocks, P,
        _table(page_table), page_table.numel(), num_shards, scale, _ptr(o),
        _ptr(lse), _ptr(dq), _ptr(dk_resp), _ptr(dv_resp), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def lsr_pool_device_status(pool: Pool, stream=None) -> int:
    v = ctypes.c_int()
    st = _lib.lsr_pool_device_status(pool.handle, ctypes.byref(v),
                                     _stream(stream))
    if st not in (LSR_OK, LSR_ERR_DEVICE):
        _check(st)
    return v.value


def lsr_profile_set(enable: bool):
    _check(_lib.lsr_profile_set(1 if enable else 0))


def lsr_profile_read(kernel: int):
    """(launches, total_ms) of one kernel id since the last profile_set."""
    n = ctypes.c_longlong()
    ms = ctypes.c_double()
    _check(_lib.lsr_profile_read(kernel, ctypes.byref(n), ctypes.byref(ms)))
    return n.value, ms.value


def lsr_kernel_name(kernel: int) -> str:
    return _lib.lsr_kernel_name(kernel).decode()


def _ints(vals):
    arr = (ctypes.c_int * len(vals))(*[int(v) for v in vals])
    return arr


def lsr_group_rows(Hq: int, num_kv_heads: int, R):
    """row0[0..K]: response k occupies rows [row0[k], row0[k+1])."""
    row0 = (ctypes.c_int * (len(R) + 1))()
    _check(_lib.lsr_group_rows(Hq, num_kv_heads, len(R), _ints(R), row0))
    return list(row0)


def lsr_group_workspace_size(num_shards: int, Hq: int, total_rows: int,
                             head_dim: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.lsr_group_workspace_size(num_shards, Hq, total_rows, head_dim,
                                         ctypes.byref(n)))
    return n.value


def lsr_replay_group(pool: Pool, R, resp_page0, grad_page0, q, dO, P: int,
                     page_table, num_shards: int, scale: float, o, lse, dq,
                     dk, dv, workspace, stream=None):
    for t, n in ((q, "q"), (dO, "dO")):
        _bf16(t, n)
    for t, n in ((o, "o"), (lse, "lse"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        _f32(t, n)
    _check(_lib.lsr_replay_group(
        pool.handle, len(R), _ints(R), _ints(resp_page0), _ints(grad_page0),
        _ptr(q), _ptr(dO), q.shape[1], P, _table(page_table),
        page_table.numel(), num_shards, scale, _ptr(o), _ptr(lse), _ptr(dq),
        _ptr(dk), _ptr(dv), dk.shape[0], _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def lsr_pool_set_version(pool: Pool, version: int):
    _check(_lib.lsr_pool_set_version(pool.handle, version))


def lsr_pool_version(pool: Pool) -> int:
    v = ctypes.c_uint64()
    _check(_lib.lsr_pool_version(pool.handle, ctypes.byref(v)))
    return v.value


class Window:
    """Host handle of an accumulation window (closed by an optimizer step)."""

    def __init__(self, handle):
        self.handle = handle

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.lsr_window_destroy(h)
            self.handle = None


def lsr_window_create(model_version: int) -> Window:
    h = ctypes.c_void_p()
    _check(_lib.lsr_window_create(model_version, ctypes.byref(h)))
    return Window(h)


def lsr_window_destroy(window: Window):
    if window.handle is not None:
        _check(_lib.lsr_window_destroy(window.handle))
        window.handle = None


def lsr_window_begin_replay(window: Window, resident_version: int,
                            replay_id: int):
    _check(_lib.lsr_window_begin_replay(window.handle, resident_version,
                                        replay_id))


def lsr_window_commit_replay(window: Window, replay_id: int, n_tokens: int):
    _check(_lib.lsr_window_commit_replay(window.handle, replay_id, n_tokens))


def lsr_window_abort_replay(window: Window, replay_id: int):
    _check(_lib.lsr_window_abort_replay(window.handle, replay_id))


def lsr_window_close(window: Window, next_version: int):
    """Returns (replays counted, tokens counted) and opens the next version."""
    n = ctypes.c_longlong()
    t = ctypes.c_longlong()
    _check(_lib.lsr_window_close(window.handle, next_version, ctypes.byref(n),
                                 ctypes.byref(t)))
    return n.value, t.value


def lsr_score_shards(pool: Pool, Hq: int, R_b: int, P: int) -> int:
    n = ctypes.c_int()
    _check(_lib.lsr_score_shards(pool.handle, Hq, R_b, P, ctypes.byref(n)))
    return n.value


def lsr_score_workspace_size(num_shards: int, Hq: int, R_b: int,
                             head_dim: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.lsr_score_workspace_size(num_shards, Hq, R_b, head_dim,
                                         ctypes.byref(n)))
    return n.value


def lsr_score_fwd(pool: Pool, q, P: int, resp_pos0: int, page_table,
                  num_shards: int, scale: float, o, lse, workspace,
                  stream=None):
    _bf16(q, "q")
    _f32(o, "o")
    _f32(lse, "lse")
    R_b, Hq, _ = q.shape
    _check(_lib.lsr_score_fwd(
        pool.handle, _ptr(q), Hq, R_b, P, resp_pos0, _table(page_table),
        page_table.numel(), num_shards, scale, _ptr(o), _ptr(lse),
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def lsr_selftest_bounded_wait(dev_status: torch.Tensor, limit_us: int,
                              stream=None):
    """Launch a wait that must time out and set LSR_DEV_WAIT_TIMEOUT."""
    if dev_status.dtype != torch.int32:
        raise TypeError("dev_status must be int32")
    _check(_lib.lsr_selftest_bounded_wait(_ptr(dev_status), limit_us,
                                          _stream(stream)))


def lsr_pool_set_wait_limit(pool, limit_us: int):
    """Limit (microseconds, 0 = default 4 s) of the attention kernels'
    pipeline waits for later calls on `pool`."""
    _check(_lib.lsr_pool_set_wait_limit(pool.handle, limit_us))


def lsr_last_error() -> str:
    return _lib.lsr_last_error().decode()


# ---------------------------------------------------------------- latent pages
class LatentPool(Pool):
    """Opaque handle of a latent page pool [num_pages, page_size, d_c + d_r]."""

    def __init__(self, handle, pages, status, d_c, d_r):
        self.handle = handle
        self.k_pages = self.v_pages = pages
        self.status = status
        self.num_pages, self.page_size, _ = pages.shape
        self.num_kv_heads, self.head_dim = 1, d_c + d_r
        self.d_c, self.d_r = d_c, d_r


def lsr_latent_pool_create(pages: torch.Tensor, dev_status: torch.Tensor,
                           d_c: int = 128, d_r: int = 64) -> LatentPool:
    """pages: bf16 [num_pages, page_size, d_c + d_r]; dev_status: int32."""
    _bf16(pages, "pages")
    if dev_status.dtype != torch.int32:
        raise TypeError("dev_status must be int32")
    npg, ps, dl = pages.shape
    if dl != d_c + d_r:
        raise ValueError("pages' last dimension must be d_c + d_r")
    h = ctypes.c_void_p()
    _check(_lib.lsr_latent_pool_create(npg, ps, d_c, d_r, _ptr(pages),
                                       _ptr(dev_status), ctypes.byref(h)))
    return LatentPool(h, pages, dev_status, d_c, d_r)


def lsr_latent_write_pages(pool: LatentPool, lat: torch.Tensor, pos0: int,
                           page_table: torch.Tensor, stream=None):
    _bf16(lat, "lat")
    _check(_lib.lsr_latent_write_pages(pool.handle, _ptr(lat), lat.shape[0],
                                       pos0, _table(page_table),
                                       page_table.numel(), _stream(stream)))


def lsr_latent_attn_fwd(pool: LatentPool, q: torch.Tensor, P: int,
                        resp_pos0: int, page_table: torch.Tensor,
                        num_shards: int, scale: float, m: torch.Tensor,
                        l: torch.Tensor, o_part: torch.Tensor, stream=None):
    _bf16(q, "q")
    for t, n in ((m, "m"), (l, "l"), (o_part, "o_part")):
        _f32(t, n)
    R_b, Hq, _ = q.shape
    _check(_lib.lsr_latent_attn_fwd(pool.handle, _ptr(q), Hq, R_b, P,
                                    resp_pos0, _table(page_table),
                                    page_table.numel(), num_shards, scale,
                                    _ptr(m), _ptr(l), _ptr(o_part),
                                    _stream(stream)))


def lsr_latent_bwd_workspace_size(num_shards: int, Hq: int, R_b: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.lsr_latent_bwd_workspace_size(num_shards, Hq, R_b,
                                              ctypes.byref(n)))
    return n.value


def lsr_latent_attn_bwd(pool: LatentPool, q, o, dO, lse, P: int,
                        resp_pos0: int, page_table, num_shards: int,
                        scale: float, dq, dlat, workspace: torch.Tensor,
                        stream=None):
    for t, n in ((q, "q"), (dO, "dO")):
        _bf16(t, n)
    for t, n in ((o, "o"), (lse, "lse"), (dq, "dq"), (dlat, "dlat")):
        _f32(t, n)
    R_b, Hq, _ = q.shape
    _check(_lib.lsr_latent_attn_bwd(
        pool.handle, _ptr(q), _ptr(o), _ptr(dO), _ptr(lse), Hq, R_b, P,
        resp_pos0, _table(page_table), page_table.numel(), num_shards, scale,
        _ptr(dq), _ptr(dlat), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def lsr_latent_replay_workspace_size(num_shards: int, Hq: int, R: int,
                                     num_blocks: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.lsr_latent_replay_workspace_size(num_shards, Hq, R,
                                                 num_blocks, ctypes.byref(n)))
    return n.value


def lsr_latent_replay_response(pool: LatentPool, q, dO, num_blocks: int,
                               P: int, page_table, num_shards: int,
                               scale: float, o, lse, dq, dlat,
                               workspace: torch.Tensor, stream=None):
    _bf16(q, "q")
    _bf16(dO, "dO")
    for t, n in ((o, "o"), (lse, "lse"), (dq, "dq"), (dlat, "dlat")):
        _f32(t, n)
    R, Hq, _ = q.shape
    _check(_lib.lsr_latent_replay_response(
        pool.handle, _ptr(q), _ptr(dO), Hq, R, num_blocks, P,
        _table(page_table), page_table.numel(), num_shards, scale, _ptr(o),
        _ptr(lse), _ptr(dq), _ptr(dlat), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def lsr_latent_group_workspace_size(num_shards: int, Hq: int,
                                    total_rows: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.lsr_latent_group_workspace_size(num_shards, Hq, total_rows,
                                                ctypes.byref(n)))
    return n.value


def lsr_latent_replay_group(pool: LatentPool, R, resp_page0, grad_page0, q,
                            dO, P: int, page_table, num_shards: int,
                            scale: float, o, lse, dq, dlat, workspace,
                            stream=None):
    for t, n in ((q, "q"), (dO, "dO")):
        _bf16(t, n)
    for t, n in ((o, "o"), (lse, "lse"), (dq, "dq"), (dlat, "dlat")):
        _f32(t, n)
    _check(_lib.lsr_latent_replay_group(
        pool.handle, len(R), _ints(R), _ints(resp_page0), _ints(grad_page0),
        _ptr(q), _ptr(dO), q.shape[1], P, _table(page_table),
        page_table.numel(), num_shards, scale, _ptr(o), _ptr(lse), _ptr(dq),
        _ptr(dlat), dlat.shape[0], _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
