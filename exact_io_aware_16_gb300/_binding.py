"""ctypes binding of libfa.so: argument marshalling only.

Names and argument order follow ``include/fa.h``.  Tensors must be CUDA bf16
(inputs/outputs) or fp32 (lse, D) and contiguous; the functions allocate the
outputs with PyTorch when they are not given.  Calls are asynchronous on the
current PyTorch stream of the tensors' device unless ``stream`` is given.  All
tensors of one call must live on one GPU; that GPU is made current for the
call (the library launches on the current device).
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = os.path.join(_HERE, "_build", "libfa.so")
_lock = threading.Lock()
_lib = None

FA_OK = 0
STATUS_NAMES = {
    0: "FA_OK", -1: "FA_ERR_NULL", -2: "FA_ERR_SHAPE", -3: "FA_ERR_HEADDIM", -4: "FA_ERR_ALIGN",
    -5: "FA_ERR_ARCH", -6: "FA_ERR_WORKSPACE", -7: "FA_ERR_CUDA", -8: "FA_ERR_DEVICE_TIMEOUT",
}


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({fa_status_string(status)})")


def library_path() -> str:
    return _LIB


def library():
    """Load libfa.so (raises if it has not been built: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB):
            raise ImportError(f"libfa.so not built ({_LIB}); run exact_io_aware_16_gb300/build.py")
        lib = ctypes.CDLL(_LIB)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_forward.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        lib.fa_forward.restype = i
        lib.fa_backward_workspace_size.argtypes = [i, i, i, i]
        lib.fa_backward_workspace_size.restype = sz
        lib.fa_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz,
                                    vp]
        lib.fa_backward.restype = i
        ll = ctypes.c_longlong
        lib.fa_forward_blocksparse.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, ll, vp]
        lib.fa_forward_blocksparse.restype = i
        lib.fa_backward_blocksparse.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f,
                                                i, vp, ll, vp, sz, vp]
        lib.fa_backward_blocksparse.restype = i
        u64, u32 = ctypes.c_ulonglong, ctypes.c_uint
        lib.fa_forward_dropout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, f, u64, u32, vp,
                                           ll, vp]
        lib.fa_forward_dropout.restype = i
        lib.fa_backward_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i,
                                            f, u64, u32, vp, ll, vp, sz, vp]
        lib.fa_backward_dropout.restype = i
        lib.fa_forward_fp8.argtypes = [vp, vp, vp, f, f, f, vp, vp, i, i, i, i, f, i, vp]
        lib.fa_forward_fp8.restype = i
        lib.fa_host_plan_create.argtypes = [i, i, i, i, f, i, ctypes.POINTER(vp)]
        lib.fa_host_plan_create.restype = i
        lib.fa_host_step.argtypes = [vp] * 10
        lib.fa_host_step.restype = i
        lib.fa_host_wait.argtypes = [vp]
        lib.fa_host_wait.restype = i
        lib.fa_host_plan_destroy.argtypes = [vp]
        lib.fa_host_plan_destroy.restype = i
        lib.fa_decode_workspace_size.argtypes = [i, i, i, i, i]
        lib.fa_decode_workspace_size.restype = sz
        lib.fa_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
        lib.fa_decode.restype = i
        lib.fa_backward_preprocess.argtypes = [vp, vp, vp, i, i, i, i, vp]
        lib.fa_backward_preprocess.restype = i
        lib.fa_backward_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i,
                                             vp]
        lib.fa_backward_noalloc.restype = i
        lib.fa_backward_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        lib.fa_backward_dkdv.restype = i
        lib.fa_backward_dq.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        lib.fa_selftest_wait_timeout.argtypes = [vp]
        lib.fa_selftest_wait_timeout.restype = i
        lib.fa_backward_dq.restype = i
        lib.fa_get_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.fa_get_device_error.restype = i
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_forward_tile_count.argtypes = [i, i]
        lib.fa_forward_tile_count.restype = ctypes.c_longlong
        _lib = lib
        return lib


def fa_status_string(status: int) -> str:
    return library().fa_status_string(int(status)).decode()


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _on_device(t) -> bool:
    return bool(t.is_cuda)


def _device_index(t) -> int:
    return t.get_device()


def _one_device(*named):
    """The device index shared by every (tensor, name) given (None entries
    skipped): a tensor on another GPU would be read or written through an
    address the launching GPU may not map."""
    dev = _device_index(named[0][0])
    for t, nm in named[1:]:
        if t is not None and _device_index(t) != dev:
            raise ValueError(f"{nm} is on device {_device_index(t)}, the call's other tensors "
                             f"on device {dev}")
    return dev


def _device_guard(dev: int):
    """Makes device `dev` current for a library call when it is not already."""
    if dev < 0 or dev == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(dev)


def _check(t, name, dtype, shape=None):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not _on_device(t):
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _check_grads(dq, dk, dv, shape):
    for t, nm in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, nm, torch.bfloat16, shape)


def _check_workspace(ws):
    if not isinstance(ws, torch.Tensor) or not _on_device(ws) or not ws.is_contiguous() \
            or ws.dtype != torch.uint8:
        raise TypeError("workspace must be a contiguous uint8 CUDA tensor")


def fa_forward_tile_count(N: int, causal: bool) -> int:
    return int(library().fa_forward_tile_count(int(N), int(bool(causal))))


def fa_forward(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None,
               stream=None):
    """O = softmax(scale q k^T) v and the per-row lse; q, k, v bf16 [B,H,N,d]."""
    B, H, N, d = q.shape
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, nm, torch.bfloat16, (B, H, N, d))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check(o, "o", torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    dev = _one_device((q, "q"), (k, "k"), (v, "v"), (o, "o"), (lse, "lse"))
    with _device_guard(dev):
        st = library().fa_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                  float(scale), int(bool(causal)),
                                  ctypes.c_void_p(_stream_handle(stream, q.device)))
    if st != FA_OK:
        raise FaError(st, "fa_forward")
    return o, lse


def _mask_args(mask, B, H, N):
    """(pointer, head stride) of a uint8 CUDA block mask [nt,nt] or [B*H,nt,nt]."""
    nt = -(-N // 128)
    if mask.dtype != torch.uint8 or not _on_device(mask) or not mask.is_contiguous():
        raise TypeError("block mask must be a contiguous uint8 CUDA tensor")
    if tuple(mask.shape) == (nt, nt):
        return ctypes.c_void_p(mask.data_ptr()), 0
    if tuple(mask.shape) == (B * H, nt, nt):
        return ctypes.c_void_p(mask.data_ptr()), nt * nt
    raise ValueError(f"block mask must be [{nt},{nt}] or [{B * H},{nt},{nt}]")


def fa_forward_blocksparse(q, k, v, block_mask, causal: bool = False, scale: float | None = None,
                           o=None, lse=None, stream=None):
    """fa_forward restricted to the 128x128 tiles a uint8 block mask keeps."""
    B, H, N, d = q.shape
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, nm, torch.bfloat16, (B, H, N, d))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(o, "o", torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    mp, ms = _mask_args(block_mask, B, H, N)
    dev = _one_device((q, "q"), (k, "k"), (v, "v"), (o, "o"), (lse, "lse"),
                      (block_mask, "block_mask"))
    with _device_guard(dev):
        st = library().fa_forward_blocksparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                              N, d, float(scale), int(bool(causal)), mp, ms,
                                              ctypes.c_void_p(_stream_handle(stream, q.device)))
    if st != FA_OK:
        raise FaError(st, "fa_forward_blocksparse")
    return o, lse


def fa_backward_blocksparse(q, k, v, o, dO, lse, block_mask, causal: bool = False,
                            scale: float | None = None, dq=None, dk=None, dv=None,
                            workspace=None, stream=None):
    """fa_backward restricted to the 128x128 tiles a uint8 block mask keeps."""
    B, H, N, d = q.shape
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO")):
        _check(t, nm, torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_grads(dq, dk, dv, (B, H, N, d))
    need = fa_backward_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check_workspace(workspace)
    mp, ms = _mask_args(block_mask, B, H, N)
    dev = _one_device((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO"), (lse, "lse"),
                      (dq, "dq"), (dk, "dk"), (dv, "dv"), (workspace, "workspace"),
                      (block_mask, "block_mask"))
    with _device_guard(dev):
        st = library().fa_backward_blocksparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO),
                                               _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N,
                                               d, float(scale), int(bool(causal)), mp, ms,
                                               _ptr(workspace), workspace.numel(),
                                               ctypes.c_void_p(_stream_handle(stream, q.device)))
    if st != FA_OK:
        raise FaError(st, "fa_backward_blocksparse")
    return dq, dk, dv


def fa_forward_dropout(q, k, v, p_drop: float, seed: int, offset: int = 0,
                       causal: bool = False, scale: float | None = None, block_mask=None,
                       o=None, lse=None, stream=None):
    """O = (softmax(scale q k^T) o Z / (1 - p_drop)) v and the lse of the
    undropped softmax; Z is replayed from Philox4x32-10 at (seed, offset).
    block_mask: None (dense) or a uint8 CUDA block mask as for
    fa_forward_blocksparse."""
    B, H, N, d = q.shape
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, nm, torch.bfloat16, (B, H, N, d))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(o, "o", torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    mp, ms = (None, 0) if block_mask is None else _mask_args(block_mask, B, H, N)
    dev = _one_device((q, "q"), (k, "k"), (v, "v"), (o, "o"), (lse, "lse"),
                      (block_mask, "block_mask"))
    with _device_guard(dev):
        st = library().fa_forward_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N,
                                          d, float(scale), int(bool(causal)), float(p_drop),
                                          int(seed) & (2**64 - 1), int(offset) & 0xFFFFFFFF, mp,
                                          ms, ctypes.c_void_p(_stream_handle(stream, q.device)))
    if st != FA_OK:
        raise FaError(st, "fa_forward_dropout")
    return o, lse


def fa_backward_dropout(q, k, v, o, dO, lse, p_drop: float, seed: int, offset: int = 0,
                        causal: bool = False, scale: float | None = None, block_mask=None,
                        dq=None, dk=None, dv=None, workspace=None, stream=None):
    """(dq, dk, dv) of fa_forward_dropout with the same p_drop, seed, offset."""
    B, H, N, d = q.shape
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO")):
        _check(t, nm, torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_grads(dq, dk, dv, (B, H, N, d))
    need = fa_backward_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check_workspace(workspace)
    mp, ms = (None, 0) if block_mask is None else _mask_args(block_mask, B, H, N)
    dev = _one_device((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO"), (lse, "lse"),
                      (dq, "dq"), (dk, "dk"), (dv, "dv"), (workspace, "workspace"),
                      (block_mask, "block_mask"))
    with _device_guard(dev):
        st = library().fa_backward_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO),
                                           _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                                           float(scale), int(bool(causal)), float(p_drop),
                                           int(seed) & (2**64 - 1), int(offset) & 0xFFFFFFFF, mp,
                                           ms, _ptr(workspace), workspace.numel(),
                                           ctypes.c_void_p(_stream_handle(stream, q.device)))
    if st != FA_OK:
        raise FaError(st, "fa_backward_dropout")
    return dq, dk, dv


def fa_forward_fp8(q8, k8, vt8, q_descale: float, k_descale: float, v_descale: float,
                   causal: bool = False, scale: float | None = None, o=None, lse=None,
                   stream=None):
    """O and lse of the attention of the dequantised e4m3 inputs.

    q8, k8: torch.float8_e4m3fn (or uint8 holding e4m3) [B,H,N,d]; vt8: V
    transposed per head, [B,H,d,N]; the descales map stored values to real
    ones.  d = 128, N a multiple of 16.
    """
    B, H, N, d = q8.shape
    for t, nm, shp in ((q8, "q8", (B, H, N, d)), (k8, "k8", (B, H, N, d)),
                       (vt8, "vt8", (B, H, d, N))):
        if t.element_size() != 1 or not _on_device(t) or not t.is_contiguous():
            raise TypeError(f"{nm} must be a contiguous one-byte (e4m3) CUDA tensor")
        if tuple(t.shape) != shp:
            raise ValueError(f"{nm} has shape {tuple(t.shape)}, expected {shp}")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    _check(o, "o", torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    dev = _one_device((q8, "q8"), (k8, "k8"), (vt8, "vt8"), (o, "o"), (lse, "lse"))
    with _device_guard(dev):
        st = library().fa_forward_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), float(q_descale),
                                      float(k_descale), float(v_descale), _ptr(o), _ptr(lse), B,
                                      H, N, d, float(scale), int(bool(causal)),
                                      ctypes.c_void_p(_stream_handle(stream, q8.device)))
    if st != FA_OK:
        raise FaError(st, "fa_forward_fp8")
    return o, lse


class HostPlan:
    """Training steps on HOST tensors through the library's host runtime
    (fa_host_plan_create / fa_host_step / fa_host_wait).

    step() enqueues one fa_forward + fa_backward whose inputs q, k, v, dO and
    outputs o, lse, dq, dk, dv are CPU tensors (bf16 [B,H,N,d], lse fp32
    [B,H,N]; pin them for the copies to overlap the kernels) and returns at
    once; the tensors must stay untouched until wait().
    """

    def __init__(self, B: int, H: int, N: int, d: int, causal: bool = False,
                 scale: float | None = None, device=None):
        self.shape = (B, H, N, d)
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        dev = torch.device("cuda") if device is None else torch.device(device)
        lib = library()
        h = ctypes.c_void_p()
        with torch.cuda.device(dev):
            st = lib.fa_host_plan_create(B, H, N, d, float(scale), int(bool(causal)),
                                         ctypes.byref(h))
        if st != FA_OK:
            raise FaError(st, "fa_host_plan_create")
        self._h = h
        self._keep = []

    def step(self, q, k, v, dO, o, lse, dq, dk, dv):
        B, H, N, d = self.shape
        for t, nm in ((q, "q"), (k, "k"), (v, "v"), (dO, "dO"), (o, "o"), (dq, "dq"),
                      (dk, "dk"), (dv, "dv")):
            if t.device.type != "cpu" or t.dtype != torch.bfloat16 or not t.is_contiguous() \
                    or tuple(t.shape) != (B, H, N, d):
                raise TypeError(f"{nm} must be a contiguous bf16 CPU tensor of shape "
                                f"{(B, H, N, d)}")
        if lse.device.type != "cpu" or lse.dtype != torch.float32 or not lse.is_contiguous() \
                or tuple(lse.shape) != (B, H, N):
            raise TypeError(f"lse must be a contiguous fp32 CPU tensor of shape {(B, H, N)}")
        ts = (q, k, v, dO, o, lse, dq, dk, dv)
        st = library().fa_host_step(self._h, *(ctypes.c_void_p(t.data_ptr()) for t in ts))
        if st != FA_OK:
            raise FaError(st, "fa_host_step")
        self._keep.append(ts)  # the buffers stay referenced until wait()

    def wait(self):
        st = library().fa_host_wait(self._h)
        self._keep.clear()
        if st != FA_OK:
            raise FaError(st, "fa_host_wait")

    def close(self):
        if getattr(self, "_h", None):
            st = library().fa_host_plan_destroy(self._h)
            self._h = None
            self._keep.clear()
            if st != FA_OK:
                raise FaError(st, "fa_host_plan_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fa_decode_workspace_size(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return int(library().fa_decode_workspace_size(B, H, Nq, Nk, d))


def fa_decode(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None,
              workspace=None, stream=None):
    """Nq (<= 16) query rows q [B,H,Nq,d] against a key/value cache k, v [B,H,Nk,d]."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    _check(q, "q", torch.bfloat16)
    _check(k, "k", torch.bfloat16, (B, H, Nk, d))
    _check(v, "v", torch.bfloat16, (B, H, Nk, d))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(o, "o", torch.bfloat16, (B, H, Nq, d))
    _check(lse, "lse", torch.float32, (B, H, Nq))
    need = fa_decode_workspace_size(B, H, Nq, Nk, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check_workspace(workspace)
    dev = _one_device((q, "q"), (k, "k"), (v, "v"), (o, "o"), (lse, "lse"),
                      (workspace, "workspace"))
    with _device_guard(dev):
        st = library().fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                                 float(scale), int(bool(causal)), _ptr(workspace),
                                 workspace.numel(),
                                 ctypes.c_void_p(_stream_handle(stream, q.device)))
    if st != FA_OK:
        raise FaError(st, "fa_decode")
    return o, lse


def fa_backward_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(library().fa_backward_workspace_size(B, H, N, d))


def fa_backward_preprocess(o, dO, D=None, stream=None):
    B, H, N, d = o.shape
    _check(o, "o", torch.bfloat16)
    _check(dO, "dO", torch.bfloat16, (B, H, N, d))
    if D is None:
        D = torch.empty((B, H, N), dtype=torch.float32, device=o.device)
    _check(D, "D", torch.float32, (B, H, N))
    dev = _one_device((o, "o"), (dO, "dO"), (D, "D"))
    with _device_guard(dev):
        st = library().fa_backward_preprocess(_ptr(o), _ptr(dO), _ptr(D), B, H, N, d,
                                              ctypes.c_void_p(_stream_handle(stream, o.device)))
    if st != FA_OK:
        raise FaError(st, "fa_backward_preprocess")
    return D


def fa_backward(q, k, v, o, dO, lse, causal: bool = False, scale: float | None = None,
                dq=None, dk=None, dv=None, workspace=None, stream=None):
    """(dq, dk, dv) of the attention; workspace is a uint8 CUDA tensor or None."""
    B, H, N, d = q.shape
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO")):
        _check(t, nm, torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_grads(dq, dk, dv, (B, H, N, d))
    need = fa_backward_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check_workspace(workspace)
    dev = _one_device((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO"), (lse, "lse"),
                      (dq, "dq"), (dk, "dk"), (dv, "dv"), (workspace, "workspace"))
    with _device_guard(dev):
        st = library().fa_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse),
                                   _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                   int(bool(causal)), _ptr(workspace), workspace.numel(),
                                   ctypes.c_void_p(_stream_handle(stream, q.device)))
    if st != FA_OK:
        raise FaError(st, "fa_backward")
    return dq, dk, dv


def fa_backward_noalloc(q, k, v, o, dO, lse, causal: bool = False, scale: float | None = None,
                        dq=None, dk=None, dv=None, stream=None):
    """fa_backward for callers that cannot allocate: the library's built-in
    8 MiB workspace replaces the caller's (B*H*N <= 2,097,152)."""
    B, H, N, d = q.shape
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO")):
        _check(t, nm, torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_grads(dq, dk, dv, (B, H, N, d))
    dev = _one_device((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO"), (lse, "lse"),
                      (dq, "dq"), (dk, "dk"), (dv, "dv"))
    with _device_guard(dev):
        st = library().fa_backward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO),
                                           _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                                           float(scale), int(bool(causal)),
                                           ctypes.c_void_p(_stream_handle(stream, q.device)))
    if st != FA_OK:
        raise FaError(st, "fa_backward_noalloc")
    return dq, dk, dv


def fa_backward_dkdv(q, k, v, dO, lse, D, causal: bool = False, scale: float | None = None,
                     dk=None, dv=None, stream=None):
    """dk, dv from the D pre-pass output D (fp32 [B,H,N])."""
    B, H, N, d = q.shape
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (dO, "dO")):
        _check(t, nm, torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    _check(D, "D", torch.float32, (B, H, N))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(dk, "dk", torch.bfloat16, (B, H, N, d))
    _check(dv, "dv", torch.bfloat16, (B, H, N, d))
    dev = _one_device((q, "q"), (k, "k"), (v, "v"), (dO, "dO"), (lse, "lse"), (D, "D"),
                      (dk, "dk"), (dv, "dv"))
    with _device_guard(dev):
        st = library().fa_backward_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(D),
                                        _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                        int(bool(causal)),
                                        ctypes.c_void_p(_stream_handle(stream, q.device)))
    if st != FA_OK:
        raise FaError(st, "fa_backward_dkdv")
    return dk, dv


def fa_backward_dq(q, k, v, dO, lse, D, causal: bool = False, scale: float | None = None,
                   dq=None, stream=None):
    """dq from the D pre-pass output D (fp32 [B,H,N])."""
    B, H, N, d = q.shape
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (dO, "dO")):
        _check(t, nm, torch.bfloat16, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    _check(D, "D", torch.float32, (B, H, N))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    _check(dq, "dq", torch.bfloat16, (B, H, N, d))
    dev = _one_device((q, "q"), (k, "k"), (v, "v"), (dO, "dO"), (lse, "lse"), (D, "D"),
                      (dq, "dq"))
    with _device_guard(dev):
        st = library().fa_backward_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(D),
                                      _ptr(dq), B, H, N, d, float(scale), int(bool(causal)),
                                      ctypes.c_void_p(_stream_handle(stream, q.device)))
    if st != FA_OK:
        raise FaError(st, "fa_backward_dq")
    return dq


def fa_selftest_wait_timeout(stream=None):
    """Launch the library's failure-reporting self-test: a wait that can never
    complete gives up after its limit; fa_get_device_error then reports it."""
    dev = torch.cuda.current_device()
    st = library().fa_selftest_wait_timeout(ctypes.c_void_p(_stream_handle(stream, dev)))
    if st != FA_OK:
        raise FaError(st, "fa_selftest_wait_timeout")


def fa_get_device_error(stream=None):
    """(status, raw detail word); synchronises the stream."""
    detail = ctypes.c_uint32(0)
    dev = torch.cuda.current_device()
    st = library().fa_get_device_error(ctypes.c_void_p(_stream_handle(stream, dev)),
                                       ctypes.byref(detail))
    return st, int(detail.value)
