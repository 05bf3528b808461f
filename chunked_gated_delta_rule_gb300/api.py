"""ctypes binding of ``include/gdr.h``: argument marshalling only.

Every step of the forward and backward passes runs in the CUDA library; these
functions pass tensor pointers, sizes and the current CUDA stream across the
C ABI.  If the library has not been built (``__graft_entry__.build()``),
every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

from . import build as _build

GDR_F32, GDR_BF16, GDR_F16 = 0, 1, 2


class gdr_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64),
                ("K", ctypes.c_int64), ("V", ctypes.c_int64), ("N", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("max_len", ctypes.c_int64),
                ("q_stride", ctypes.c_int64 * 2), ("k_stride", ctypes.c_int64 * 2),
                ("v_stride", ctypes.c_int64 * 2), ("o_stride", ctypes.c_int64 * 2)]


class gdr_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("bv", ctypes.c_int32),
                ("n_segments", ctypes.c_int32), ("compose", ctypes.c_int32)]


class gdr_options(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("force_path", ctypes.c_int32),
                ("force_bv", ctypes.c_int32), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("status", ctypes.c_void_p),
                ("events", ctypes.c_void_p), ("max_launches", ctypes.c_int32),
                ("launch_ids", ctypes.c_void_p), ("n_launches", ctypes.c_void_p),
                ("grid_limit", ctypes.c_int32)]


# Diagnostic entry points declared in include/gdr_selftest.h.
SELFTEST_EXPORTS = ("gdr_selftest_umma", "gdr_selftest_tma", "gdr_selftest_inverse",
                    "gdr_selftest_timeout")

# Every symbol include/gdr.h declares.
EXPORTS = ("gdr_chunk_fwd", "gdr_chunk_fwd_ex", "gdr_chunk_fwd_host", "gdr_chunk_fwd_noalloc",
           "gdr_workspace_size", "gdr_plan_query", "gdr_recurrent_fwd", "gdr_kernel_name", "gdr_error_string",
           "gdr_release_cached", "gdr_version", "gdr_chunk_bwd", "gdr_bwd_workspace_size")

_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Open ``libgdr.so``.  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        vp, i32p = ctypes.c_void_p, ctypes.c_void_p
        dims_p = ctypes.POINTER(gdr_dims)
        fwd_args = [dims_p, vp, vp, vp, vp, vp, i32p, vp, vp, vp, ctypes.c_int]
        lib.gdr_chunk_fwd.argtypes = fwd_args + [vp]
        lib.gdr_chunk_fwd.restype = ctypes.c_int
        lib.gdr_chunk_fwd_ex.argtypes = fwd_args + [ctypes.POINTER(gdr_options), vp]
        lib.gdr_chunk_fwd_ex.restype = ctypes.c_int
        lib.gdr_chunk_fwd_host.argtypes = fwd_args + [vp]
        lib.gdr_chunk_fwd_host.restype = ctypes.c_int
        lib.gdr_chunk_fwd_noalloc.argtypes = fwd_args + [vp]
        lib.gdr_chunk_fwd_noalloc.restype = ctypes.c_int
        lib.gdr_recurrent_fwd.argtypes = [dims_p, vp, vp, vp, vp, vp, i32p, vp, ctypes.c_int64,
                                          i32p, vp, vp, vp]
        lib.gdr_recurrent_fwd.restype = ctypes.c_int
        lib.gdr_chunk_bwd.argtypes = [dims_p, vp, vp, vp, vp, vp, i32p, vp, vp, vp, vp, vp, vp,
                                      vp, vp, vp, ctypes.c_int, ctypes.POINTER(gdr_options), vp]
        lib.gdr_chunk_bwd.restype = ctypes.c_int
        lib.gdr_bwd_workspace_size.argtypes = [dims_p, ctypes.c_int, ctypes.c_int]
        lib.gdr_bwd_workspace_size.restype = ctypes.c_size_t
        lib.gdr_workspace_size.argtypes = [dims_p, ctypes.c_int, ctypes.c_int]
        lib.gdr_workspace_size.restype = ctypes.c_size_t
        lib.gdr_plan_query.argtypes = [dims_p, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(gdr_plan)]
        lib.gdr_plan_query.restype = ctypes.c_int
        lib.gdr_kernel_name.argtypes = [ctypes.c_int]
        lib.gdr_kernel_name.restype = ctypes.c_char_p
        lib.gdr_error_string.argtypes = [ctypes.c_int]
        lib.gdr_error_string.restype = ctypes.c_char_p
        lib.gdr_selftest_umma.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, vp, vp]
        lib.gdr_selftest_umma.restype = ctypes.c_int
        lib.gdr_selftest_tma.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp]
        lib.gdr_selftest_tma.restype = ctypes.c_int
        lib.gdr_selftest_timeout.argtypes = [vp, ctypes.c_uint64, vp, vp]
        lib.gdr_selftest_timeout.restype = ctypes.c_int
        lib.gdr_selftest_inverse.argtypes = [vp, vp, vp]
        lib.gdr_selftest_inverse.restype = ctypes.c_int
        lib.gdr_release_cached.argtypes = []
        lib.gdr_release_cached.restype = ctypes.c_int
        lib.gdr_version.argtypes = []
        lib.gdr_version.restype = ctypes.c_int
        _lib = lib
        return lib


class GdrError(RuntimeError):
    def __init__(self, code: int):
        msg = load_library().gdr_error_string(code).decode()
        super().__init__(f"gdr error {code}: {msg}")
        self.code = code


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return GDR_F32
    if t == torch.bfloat16:
        return GDR_BF16
    if t == torch.float16:
        return GDR_F16
    raise TypeError(f"unsupported dtype {t}: q, k, v must be float32, bfloat16 or float16")


GDR_SEQLENS_I64 = 1  # gdr_dims.flags: cu_seqlens holds int64 offsets
GDR_STATE_VK = 2     # gdr_dims.flags: h0 / ht / state pool are S [.., V, K]


def make_dims(B, T, H, K, V, N=0, dtype=GDR_BF16, flags=0, max_len=0) -> gdr_dims:
    return gdr_dims(B, T, H, K, V, N, dtype, flags, max_len)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _row_strides(t):
    """(token, head) element strides of a [B, T, H, D] tensor, or (0, 0)
    when it is contiguous.  The last dimension must be contiguous and B, T
    must flatten into one token dimension."""
    if t.is_contiguous():
        return (0, 0)
    B, T = t.shape[0], t.shape[1]
    if t.stride(-1) != 1 or (B > 1 and t.stride(0) != T * t.stride(1)):
        raise ValueError("q, k, v and o need a contiguous last dimension and batch rows "
                         "T token strides apart")
    return (t.stride(1), t.stride(2))


def _dims_of(q, v, cu_seqlens, state_layout="kv", max_seqlen=None, k=None, o=None) -> gdr_dims:
    """Sizes and flags: int64 cu_seqlens sets GDR_SEQLENS_I64; state_layout
    "vk" (states as S, [.., V, K]) sets GDR_STATE_VK; ``max_seqlen`` (the
    longest sequence's token count, a planning hint; None = unknown) goes
    to gdr_dims.max_len; the token / head strides of q, k, v, o (views of a
    larger tensor) go to the stride fields."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    N = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    if state_layout not in ("kv", "vk"):
        raise ValueError(f"state_layout must be 'kv' or 'vk', got {state_layout!r}")
    flags = (GDR_SEQLENS_I64 if cu_seqlens is not None and cu_seqlens.dtype == torch.int64
             else 0) | (GDR_STATE_VK if state_layout == "vk" else 0)
    dims = make_dims(B, T, H, K, V, N, _dtype_code(q.dtype), flags,
                     0 if max_seqlen is None else int(max_seqlen))
    for name, t in (("q_stride", q), ("k_stride", k), ("v_stride", v), ("o_stride", o)):
        if t is not None:
            getattr(dims, name)[:] = _row_strides(t)
    return dims


def _state_dims(dims, state_layout):
    return (dims.V, dims.K) if state_layout == "vk" else (dims.K, dims.V)


def _check_cu(t, device=None):
    if t is not None and t.dtype not in (torch.int32, torch.int64):
        raise TypeError(f"cu_seqlens must be int32 or int64, got {t.dtype}")
    _check("cu_seqlens", t, None, device)


def _check(name, t, dtype, device=None, strided=False):
    """dtype / device checks; contiguous unless ``strided`` (q, k, v, o of
    the device entry points, whose token and head strides go to the
    library)."""
    if t is None:
        return
    if strided:
        _row_strides(t)
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


class LaunchTimer:
    """Caller-side CUDA events for the per-launch timing hook of
    gdr_chunk_fwd_ex (benchmarks).  After a call, ``ids[:count]`` are the
    kernel ids launched and ``elapsed_ms(i)`` the duration of launch i once
    the stream has been synchronised."""

    def __init__(self, max_launches=16):
        self.max = max_launches
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * max_launches)]
        for e in self.events:  # torch creates the CUDA event on first record
            e.record()
        torch.cuda.current_stream().synchronize()
        self._handles = (ctypes.c_void_p * (2 * max_launches))(
            *[ctypes.c_void_p(e.cuda_event) for e in self.events])
        self._ids = (ctypes.c_int32 * max_launches)()
        self._count = ctypes.c_int32(0)

    @property
    def count(self):
        return int(self._count.value)

    @property
    def ids(self):
        return [int(self._ids[i]) for i in range(min(self.count, self.max))]

    def elapsed_ms(self, i):
        return self.events[2 * i].elapsed_time(self.events[2 * i + 1])


def gdr_chunk_fwd(q, k, v, g, beta=None, cu_seqlens=None, h0=None, *, n_segments=0,
                  state_layout="kv", max_seqlen=None,
                  output_final_state=True, o=None, ht=None, scale=0.0, force_path=0,
                  force_bv=0, workspace=None, status=None, stream=None, timer=None,
                  grid_limit=0):
    """Forward pass on CUDA tensors (layouts of include/gdr.h).  Returns
    ``(o, ht)``; ``ht`` is None unless ``output_final_state``.  Work is
    enqueued on ``stream`` (default: torch's current stream) and not
    synchronised.  ``max_seqlen`` is the longest sequence's token count when
    the caller knows it (a planning hint: cu_seqlens stays on the device).
    ``timer`` (a :class:`LaunchTimer`) records events around every kernel
    launch; ``grid_limit`` caps the CTAs of the persistent kernels."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("gdr_chunk_fwd takes CUDA tensors; use gdr_chunk_fwd_host for host buffers")
    _check("q", q, None, dev, strided=True)
    for name, t in (("k", k), ("v", v)):
        _check(name, t, q.dtype, dev, strided=True)
    _check("g", g, torch.float32, dev)
    _check("beta", beta, torch.float32, dev)
    _check_cu(cu_seqlens, dev)
    _check("h0", h0, torch.float32, dev)
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=dev)
    _check("o", o, q.dtype, dev, strided=True)
    dims = _dims_of(q, v, cu_seqlens, state_layout, max_seqlen, k=k, o=o)
    nseq = dims.N if dims.N else dims.B
    if ht is None and output_final_state:
        ht = torch.empty(nseq, dims.H, *_state_dims(dims, state_layout), dtype=torch.float32,
                         device=dev)
    _check("ht", ht, torch.float32, dev)
    opt = gdr_options(float(scale), int(force_path), int(force_bv),
                      None if workspace is None else workspace.data_ptr(),
                      0 if workspace is None else workspace.numel() * workspace.element_size(),
                      None if status is None else status.data_ptr())
    opt.grid_limit = int(grid_limit)
    if timer is not None:
        opt.events = ctypes.cast(timer._handles, ctypes.c_void_p)
        opt.max_launches = timer.max
        opt.launch_ids = ctypes.cast(timer._ids, ctypes.c_void_p)
        opt.n_launches = ctypes.cast(ctypes.pointer(timer._count), ctypes.c_void_p)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        rc = lib.gdr_chunk_fwd_ex(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                  _ptr(beta), _ptr(cu_seqlens), _ptr(h0), _ptr(o), _ptr(ht),
                                  int(n_segments), ctypes.byref(opt),
                                  ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise GdrError(rc)
    return o, ht


def gdr_chunk_bwd(q, k, v, g, beta, do, cu_seqlens=None, h0=None, dht=None, *, n_segments=0,
                  state_layout="kv", want_dh0=True, scale=0.0, workspace=None, status=None,
                  dq=None, dk=None, dv=None, dg=None, dbeta=None, dh0=None, stream=None,
                  timer=None, force_path=0, grid_limit=0):
    """Backward pass on CUDA tensors: the gradients of ``<do, o> + <dht, ht>``
    for the forward pass on the same inputs.  Returns ``(dq, dk, dv, dg,
    dbeta, dh0)``: dq, dk, dv in the input dtype, the rest float32; ``dbeta``
    is None in the beta-free mode and ``dh0`` None unless ``want_dh0``.  Work
    is enqueued on ``stream`` (default: torch's current stream).
    ``force_path`` 1 takes the CUDA-core route (FP32 arithmetic), 2 the
    tensor-core route (BF16, K = V = 128, delta rule, serial), 0 the plan's."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("gdr_chunk_bwd takes CUDA tensors")
    _check("q", q, None, dev, strided=True)
    for name, t in (("k", k), ("v", v)):
        _check(name, t, q.dtype, dev, strided=True)
    _check("do", do, q.dtype, dev)
    if do.shape != v.shape:
        raise ValueError("do must have v's shape")
    _check("g", g, torch.float32, dev)
    _check("beta", beta, torch.float32, dev)
    _check_cu(cu_seqlens, dev)
    _check("h0", h0, torch.float32, dev)
    _check("dht", dht, torch.float32, dev)
    dims = _dims_of(q, v, cu_seqlens, state_layout, k=k)
    nseq = dims.N if dims.N else dims.B
    dq = torch.empty(q.shape, dtype=q.dtype, device=dev) if dq is None else dq
    dk = torch.empty(k.shape, dtype=q.dtype, device=dev) if dk is None else dk
    dv = torch.empty(v.shape, dtype=q.dtype, device=dev) if dv is None else dv
    dg = torch.empty(g.shape, dtype=torch.float32, device=dev) if dg is None else dg
    if beta is not None and dbeta is None:
        dbeta = torch.empty(beta.shape, dtype=torch.float32, device=dev)
    if want_dh0 and dh0 is None:
        dh0 = torch.empty(nseq, dims.H, *_state_dims(dims, state_layout), dtype=torch.float32,
                          device=dev)
    for name, t, dt in (("dq", dq, q.dtype), ("dk", dk, q.dtype), ("dv", dv, q.dtype),
                        ("dg", dg, torch.float32), ("dbeta", dbeta, torch.float32),
                        ("dh0", dh0, torch.float32)):
        _check(name, t, dt, dev)
    opt = gdr_options(float(scale), int(force_path), 0,
                      None if workspace is None else workspace.data_ptr(),
                      0 if workspace is None else workspace.numel() * workspace.element_size(),
                      None if status is None else status.data_ptr())
    opt.grid_limit = int(grid_limit)
    if timer is not None:
        opt.events = ctypes.cast(timer._handles, ctypes.c_void_p)
        opt.max_launches = timer.max
        opt.launch_ids = ctypes.cast(timer._ids, ctypes.c_void_p)
        opt.n_launches = ctypes.cast(ctypes.pointer(timer._count), ctypes.c_void_p)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        rc = lib.gdr_chunk_bwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                               _ptr(beta), _ptr(cu_seqlens), _ptr(h0), _ptr(do), _ptr(dht),
                               _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0),
                               int(n_segments), ctypes.byref(opt),
                               ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise GdrError(rc)
    return dq, dk, dv, dg, dbeta, dh0


def gdr_bwd_workspace_size(B, T, H, K, V, N=0, dtype=GDR_BF16, beta_free=False, flags=0,
                           n_segments=0) -> int:
    return int(load_library().gdr_bwd_workspace_size(
        ctypes.byref(make_dims(B, T, H, K, V, N, dtype, flags)), int(beta_free),
        int(n_segments)))


def gdr_recurrent_fwd(q, k, v, g, beta=None, cu_seqlens=None, *, state, state_indices=None,
                      state_layout="kv",
                      o=None, status=None, stream=None):
    """Per-token recurrence from rows of the state pool ``state`` ([P, H, K,
    V] float32, updated in place): sequence n starts from row
    ``state_indices[n]`` (row n if None) and writes its final state back
    there.  Returns ``o``.  Work is enqueued on ``stream`` and not
    synchronised."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("gdr_recurrent_fwd takes CUDA tensors")
    _check("q", q, None, dev, strided=True)
    for name, t in (("k", k), ("v", v)):
        _check(name, t, q.dtype, dev, strided=True)
    _check("g", g, torch.float32, dev)
    _check("beta", beta, torch.float32, dev)
    _check_cu(cu_seqlens, dev)
    _check("state", state, torch.float32, dev)
    _check("state_indices", state_indices, torch.int32, dev)
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=dev)
    _check("o", o, q.dtype, dev, strided=True)
    dims = _dims_of(q, v, cu_seqlens, state_layout, k=k, o=o)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        rc = lib.gdr_recurrent_fwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                   _ptr(beta), _ptr(cu_seqlens), _ptr(state),
                                   ctypes.c_int64(state.shape[0]), _ptr(state_indices), _ptr(o),
                                   _ptr(status), ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise GdrError(rc)
    return o


def gdr_chunk_fwd_host(q, k, v, g, beta=None, cu_seqlens=None, h0=None, *, n_segments=0,
                       state_layout="kv",
                       output_final_state=True, o=None, ht=None, stream=None):
    """Forward pass on HOST (CPU) tensors through ``gdr_chunk_fwd_host``: the
    library copies inputs in, runs, copies o / ht out and synchronises.
    Pinned tensors give asynchronous copies."""
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta),
                    ("cu_seqlens", cu_seqlens), ("h0", h0)):
        if t is not None and t.device.type != "cpu":
            raise ValueError(f"{name} must be a host tensor")
    _check("k", k, q.dtype)
    _check("v", v, q.dtype)
    _check("g", g, torch.float32)
    _check("beta", beta, torch.float32)
    _check_cu(cu_seqlens)
    _check("h0", h0, torch.float32)
    dims = _dims_of(q, v, cu_seqlens, state_layout)
    nseq = dims.N if dims.N else dims.B
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype)
    if ht is None and output_final_state:
        ht = torch.empty(nseq, dims.H, *_state_dims(dims, state_layout), dtype=torch.float32)
    if stream is None:
        stream = torch.cuda.current_stream()
    rc = lib.gdr_chunk_fwd_host(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                _ptr(beta), _ptr(cu_seqlens), _ptr(h0), _ptr(o), _ptr(ht),
                                int(n_segments), ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise GdrError(rc)
    return o, ht


NOALLOC_SCRATCH_BYTES = 64 << 20


def gdr_chunk_fwd_noalloc(q, k, v, g, beta=None, cu_seqlens=None, h0=None, *, n_segments=0,
                          state_layout="kv", max_seqlen=None,
                          output_final_state=True, o=None, ht=None, stream=None):
    """Forward pass through ``gdr_chunk_fwd_noalloc``: the library uses a
    fixed 64 MiB device array as scratch and allocates nothing, for callers
    that must not allocate device memory during the call.  ``o`` and ``ht``
    should be passed in by such callers (this wrapper creates them with
    torch only when they are omitted).  Calls that overlap on the GPU share
    the one scratch array and must be ordered by the caller; the first call
    on a device should happen outside CUDA graph capture."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("gdr_chunk_fwd_noalloc takes CUDA tensors")
    _check("q", q, None, dev, strided=True)
    for name, t in (("k", k), ("v", v)):
        _check(name, t, q.dtype, dev, strided=True)
    _check("g", g, torch.float32, dev)
    _check("beta", beta, torch.float32, dev)
    _check_cu(cu_seqlens, dev)
    _check("h0", h0, torch.float32, dev)
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, device=dev)
    _check("o", o, q.dtype, dev, strided=True)
    dims = _dims_of(q, v, cu_seqlens, state_layout, max_seqlen, k=k, o=o)
    nseq = dims.N if dims.N else dims.B
    if ht is None and output_final_state:
        ht = torch.empty(nseq, dims.H, *_state_dims(dims, state_layout), dtype=torch.float32,
                         device=dev)
    _check("ht", ht, torch.float32, dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        rc = lib.gdr_chunk_fwd_noalloc(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                       _ptr(beta), _ptr(cu_seqlens), _ptr(h0), _ptr(o), _ptr(ht),
                                       int(n_segments), ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise GdrError(rc)
    return o, ht


def gdr_workspace_size(B, T, H, K, V, N=0, dtype=GDR_BF16, beta_free=False, n_segments=0,
                       max_len=0) -> int:
    return int(load_library().gdr_workspace_size(
        ctypes.byref(make_dims(B, T, H, K, V, N, dtype, max_len=max_len)), int(bool(beta_free)),
        int(n_segments)))


def gdr_plan_query(B, T, H, K, V, N=0, dtype=GDR_BF16, beta_free=False, n_segments=0,
                   max_len=0) -> dict:
    plan = gdr_plan()
    rc = load_library().gdr_plan_query(ctypes.byref(make_dims(B, T, H, K, V, N, dtype,
                                                              max_len=max_len)),
                                       int(bool(beta_free)), int(n_segments), ctypes.byref(plan))
    if rc != 0:
        raise GdrError(rc)
    return dict(path=plan.path, bv=plan.bv, n_segments=plan.n_segments, compose=plan.compose)


def gdr_selftest_umma(A, B, a_mn, b_mn, status=None):
    """D = A @ B^T (A [128, Kd], B [N, Kd] BF16 CUDA tensors) computed by one
    tcgen05 MMA chain with the given operand layouts; returns D (FP32)."""
    N, Kd = B.shape
    D = torch.full((A.shape[0], N), float("nan"), dtype=torch.float32, device=A.device)
    rc = load_library().gdr_selftest_umma(_ptr(A), _ptr(B), _ptr(D), N, Kd, int(a_mn), int(b_mn),
                                          _ptr(status),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc != 0:
        raise GdrError(rc)
    return D


def gdr_selftest_tma(src, t0, h, k0, status=None):
    """One 64x64 box of src [T, H, K] (BF16 CUDA) through TMA + the swizzle
    address map; returns the [64, 64] box."""
    T, H, K = src.shape
    out = torch.full((64, 64), float("nan"), dtype=torch.bfloat16, device=src.device)
    rc = load_library().gdr_selftest_tma(_ptr(src), T, H, K, int(t0), int(h), int(k0), _ptr(out),
                                         _ptr(status),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc != 0:
        raise GdrError(rc)
    return out


def gdr_selftest_inverse(A):
    """(I + tril(A, -1))^-1 for a 64x64 FP32 CUDA tensor, by the device routine
    of the tensor-core path."""
    A = A.contiguous()
    T = torch.full_like(A, float("nan"))
    rc = load_library().gdr_selftest_inverse(_ptr(A), _ptr(T),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc != 0:
        raise GdrError(rc)
    return T


def gdr_selftest_timeout(limit_ns=1_000_000):
    """Runs the bounded-wait failure path once; returns (status, done)."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    done = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = load_library().gdr_selftest_timeout(_ptr(status), int(limit_ns), _ptr(done),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc != 0:
        raise GdrError(rc)
    torch.cuda.synchronize()
    return int(status.item()), int(done.item())


def gdr_kernel_name(kid: int) -> str:
    return load_library().gdr_kernel_name(int(kid)).decode()


def gdr_error_string(code: int) -> str:
    return load_library().gdr_error_string(int(code)).decode()


def gdr_release_cached() -> None:
    """Return the device memory the library keeps between calls (its
    stream-ordered scratch pools) to the driver."""
    rc = load_library().gdr_release_cached()
    if rc != 0:
        raise GdrError(rc)


def gdr_version() -> int:
    return int(load_library().gdr_version())
