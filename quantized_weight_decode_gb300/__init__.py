"""Python binding of libnq.so, the groupwise-quantized small-T GEMV library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI of ``include/nq.h``.  PyTorch is used for device
memory and streams (tensors pass their ``data_ptr()``, streams their
``cuda_stream`` handle).  The library must have been built (``build()`` below
or ``python quantized_weight_decode_gb300/buildlib.py``); importing works without
it, but every call raises if it is missing -- there is no fallback path.

Names follow the C ABI: ``gemv`` is ``nq_gemv``, ``pack`` is ``nq_pack`` ...
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

__all__ = [
    "NQError", "ROUTE_AUTO", "ROUTE_MMA", "ROUTE_FFMA", "lib", "lib_path", "build",
    "packed_bytes", "pack", "pack_gate_up", "unpack", "pack_device", "quantize_rtn", "quantize_search", "gemv", "gemv_swiglu", "mlp", "mlp_one_launch_ok", "interleave_gate_up", "gemv_head",
    "head_workspace_bytes", "gemv_head_noalloc", "gemv_head_topk", "head_topk_workspace_bytes",
    "dequant",
    "last_device_error", "plan", "selftest_wait_timeout", "status_string", "layout_version",
    "QuantizedWeight", "EXPORTED",
]

ROUTE_AUTO, ROUTE_MMA, ROUTE_FFMA = 0, 1, 2
# x placement of a plan (nq_x_place)
X_PLACES = ("smem", "regs", "regs2", "hybrid")
OK, EINVAL, EALIGN, ERANGE, ECUDA, ETIMEOUT, EUNSUPPORTED = 0, -1, -2, -3, -4, -5, -6

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libnq.so")
_lib = None
_lock = threading.Lock()

# Every symbol declared in include/nq.h, with its ctypes signature.
_i64, _i32, _vp, _szp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)
_ip = ctypes.POINTER(ctypes.c_int)
_SIGS = {
    "nq_packed_bytes": (_i32, [_i64, _i64, _i32, _szp, _szp]),
    "nq_pack": (_i32, [_vp, _vp, _i64, _i64, _i32, _vp, _vp]),
    "nq_pack_gate_up": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp]),
    "nq_unpack": (_i32, [_vp, _vp, _i64, _i64, _i32, _vp, _vp]),
    "nq_pack_device": (_i32, [_vp, _vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "nq_quantize_rtn": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "nq_quantize_search": (_i32, [_vp, _vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "nq_gemv": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _vp]),
    "nq_gemv_ex": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _i32, _vp]),
    "nq_gemv_swiglu": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _vp]),
    "nq_mlp": (_i32, [_vp, _vp, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp]),
    "nq_mlp_ex": (_i32, [_vp, _vp, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32,
                         _vp]),
    "nq_mlp_one_launch_ok": (_i32, [_i64, _i64, _i64, _i32, _i32, _i32, _ip]),
    "nq_gemv_head": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp, _vp,
                            ctypes.c_size_t, _vp]),
    "nq_head_workspace_bytes": (_i32, [_szp]),
    "nq_gemv_head_topk": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp, _vp, _vp,
                                 _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "nq_head_topk_workspace_bytes": (_i32, [_szp]),
    "nq_gemv_head_noalloc": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp,
                                    _vp]),
    "nq_dequant": (_i32, [_vp, _vp, _vp, _i64, _i64, _i32, _vp]),
    "nq_last_device_error": (_i32, [_vp]),
    "nq_gemv_plan": (_i32, [_i64, _i64, _i32, _i32, _i32, _i32, _ip, _ip, _ip, _ip, _ip]),
    "nq_gemv_plan_x": (_i32, [_i64, _i64, _i32, _i32, _i32, _i32, _ip]),
    "nq_selftest_wait_timeout": (_i32, [_i32, _vp]),
    "nq_status_string": (ctypes.c_char_p, [_i32]),
    "nq_layout_version": (_i32, []),
}
EXPORTED = tuple(_SIGS)


class NQError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


def lib_path() -> str:
    return _LIB_PATH


def build(force: bool = False) -> str:
    """Compile libnq.so for sm_103a in-tree (needs nvcc)."""
    from . import buildlib as _b
    return _b.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with quantized_weight_decode_gb300.build() "
                    "(there is no fallback implementation)")
            h = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(h, name)
                f.restype = res
                f.argtypes = args
            _lib = h
    return _lib


def status_string(code: int) -> str:
    return lib().nq_status_string(int(code)).decode()


def layout_version() -> int:
    return int(lib().nq_layout_version())


def _check(rc: int, where: str) -> None:
    if rc != OK:
        raise NQError(rc, where)


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _dptr(t):
    return None if t is None else int(t.data_ptr())


# ---------------------------------------------------------------- host side
def packed_bytes(K: int, N: int, bits: int) -> tuple[int, int]:
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().nq_packed_bytes(K, N, bits, ctypes.byref(cb), ctypes.byref(sb)), "nq_packed_bytes")
    return cb.value, sb.value


def pack(codes: np.ndarray, scales: np.ndarray, bits: int) -> tuple[np.ndarray, np.ndarray]:
    """Host packer: int8 codes [N, K] and FP16 scale bits [N, K/64] -> packed
    codes (uint8) and packed scales (uint16), as numpy arrays."""
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    scales = np.ascontiguousarray(scales).view(np.uint16)
    N, K = codes.shape
    cb, sb = packed_bytes(K, N, bits)
    out = np.empty(cb, dtype=np.uint8)
    sout = np.empty(sb // 2, dtype=np.uint16)
    _check(lib().nq_pack(codes.ctypes.data, scales.ctypes.data, K, N, bits,
                         out.ctypes.data, sout.ctypes.data), "nq_pack")
    return out, sout


def pack_gate_up(codes_gate: np.ndarray, scales_gate: np.ndarray, codes_up: np.ndarray,
                 scales_up: np.ndarray, bits: int) -> tuple[np.ndarray, np.ndarray]:
    """Host packer of a gate+up matrix in nq_gemv_swiglu's row order
    (nq_pack_gate_up): gate and up int8 codes [I, K], FP16 scale bits
    [I, K/64] -> packed codes and scales of the [2 I, K] matrix."""
    cg = np.ascontiguousarray(codes_gate, dtype=np.int8)
    cu = np.ascontiguousarray(codes_up, dtype=np.int8)
    sg = np.ascontiguousarray(scales_gate).view(np.uint16)
    su = np.ascontiguousarray(scales_up).view(np.uint16)
    I, K = cg.shape
    cb, sb = packed_bytes(K, 2 * I, bits)
    out = np.empty(cb, dtype=np.uint8)
    sout = np.empty(sb // 2, dtype=np.uint16)
    _check(lib().nq_pack_gate_up(cg.ctypes.data, sg.ctypes.data, cu.ctypes.data, su.ctypes.data,
                                 K, I, bits, out.ctypes.data, sout.ctypes.data), "nq_pack_gate_up")
    return out, sout


def unpack(packed: np.ndarray, scales_packed: np.ndarray, K: int, N: int,
           bits: int) -> tuple[np.ndarray, np.ndarray]:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scales_packed = np.ascontiguousarray(scales_packed).view(np.uint16)
    codes = np.empty((N, K), dtype=np.int8)
    scales = np.empty((N, K // 64), dtype=np.uint16)
    _check(lib().nq_unpack(packed.ctypes.data, scales_packed.ctypes.data, K, N, bits,
                           codes.ctypes.data, scales.ctypes.data), "nq_unpack")
    return codes, scales


# ---------------------------------------------------------------- device side
def pack_device(codes, scales, bits: int, packed=None, scales_packed=None, stream=None):
    """Device packer.  codes: int8 cuda [N, K]; scales: 16-bit cuda [N, K/64].
    Returns (packed uint8 tensor, packed scales int16 tensor)."""
    import torch
    N, K = codes.shape
    cb, sb = packed_bytes(K, N, bits)
    if packed is None:
        packed = torch.empty(cb, dtype=torch.uint8, device=codes.device)
    if scales_packed is None:
        scales_packed = torch.empty(sb // 2, dtype=torch.int16, device=codes.device)
    _check(lib().nq_pack_device(_dptr(codes), _dptr(scales), K, N, bits, _dptr(packed),
                                _dptr(scales_packed), _stream_handle(stream)), "nq_pack_device")
    return packed, scales_packed


def quantize_rtn(w, bits: int, codes=None, scales=None, stream=None):
    """Device round-to-nearest encoder: fp32 cuda w [N, K] -> (int8 codes [N, K],
    int16 FP16-scale bits [N, K/64])."""
    import torch
    N, K = w.shape
    if codes is None:
        codes = torch.empty((N, K), dtype=torch.int8, device=w.device)
    if scales is None:
        scales = torch.empty((N, K // 64), dtype=torch.int16, device=w.device)
    _check(lib().nq_quantize_rtn(_dptr(w), K, N, bits, _dptr(codes), _dptr(scales),
                                 _stream_handle(stream)), "nq_quantize_rtn")
    return codes, scales


def quantize_search(w, bits: int, imatrix=None, codes=None, scales=None, stream=None):
    """Searched encoder on the device: w fp32 [N, K] (device tensor), imatrix
    fp32 [K] or None -> (codes int8 [N, K], scales int16 FP16 bits [N, K/64])."""
    import torch
    N, K = w.shape
    if codes is None:
        codes = torch.empty((N, K), dtype=torch.int8, device=w.device)
    if scales is None:
        scales = torch.empty((N, K // 64), dtype=torch.int16, device=w.device)
    _check(lib().nq_quantize_search(_dptr(w), _dptr(imatrix), K, N, bits, _dptr(codes),
                                    _dptr(scales), _stream_handle(stream)), "nq_quantize_search")
    return codes, scales


def gemv(packed, scales, x, y, K: int, N: int, T: int, bits: int, route: int = ROUTE_AUTO,
         ksplit: int = 0, stream=None) -> None:
    """y[T, N] (fp32 cuda) = x[T, K] (bf16 cuda) @ dequant(W)^T, asynchronous."""
    if route == ROUTE_AUTO and ksplit == 0:
        rc = lib().nq_gemv(_dptr(packed), _dptr(scales), _dptr(x), _dptr(y), K, N, T, bits,
                           _stream_handle(stream))
    else:
        rc = lib().nq_gemv_ex(_dptr(packed), _dptr(scales), _dptr(x), _dptr(y), K, N, T, bits,
                              route, ksplit, _stream_handle(stream))
    _check(rc, "nq_gemv")


def interleave_gate_up(gate, up):
    """Rows of the gate+up matrix in the order nq_gemv_swiglu expects: row
    16 r + m = gate row 8 r + m, row 16 r + 8 + m = up row 8 r + m (m < 8).
    Works on numpy arrays or torch tensors [I, ...] (I a multiple of 8)."""
    i = gate.shape[0]
    rest = tuple(gate.shape[1:])
    g = gate.reshape((i // 8, 1, 8) + rest)
    u = up.reshape((i // 8, 1, 8) + rest)
    try:
        import torch
        if isinstance(gate, torch.Tensor):
            return torch.cat([g, u], dim=1).reshape((2 * i,) + rest)
    except ImportError:
        pass
    import numpy as np
    return np.concatenate([g, u], axis=1).reshape((2 * i,) + rest)


def gemv_swiglu(packed_gu, scales_gu, x, act, K: int, N: int, T: int, bits: int, stream=None):
    """act[T, N/2] (bf16 tensor) = silu(gate) * up from a gate+up matrix packed
    with interleave_gate_up's row order."""
    _check(lib().nq_gemv_swiglu(_dptr(packed_gu), _dptr(scales_gu), _dptr(x), _dptr(act), K, N, T,
                                bits, _stream_handle(stream)), "nq_gemv_swiglu")


def mlp(gu, down, x, act, y, T: int, launches: int = 0, stream=None):
    """The layer MLP: gu, down are QuantizedWeight (gu packed interleaved);
    act [T, I] bf16 scratch, y [T, H_out] fp32.  launches: 0 = the library's
    choice, 1 = one launch (nq_mlp_ex), 2 = two launches."""
    _check(lib().nq_mlp_ex(_dptr(gu.packed), _dptr(gu.scales), gu.bits, _dptr(down.packed),
                           _dptr(down.scales), down.bits, _dptr(x), _dptr(act), _dptr(y), gu.K,
                           gu.N // 2, down.N, T, launches, _stream_handle(stream)), "nq_mlp_ex")


def mlp_one_launch_ok(H: int, I: int, H_out: int, T: int, bits_gu: int, bits_down: int) -> bool:
    """Whether nq_mlp_ex(launches=1) supports this layer shape here."""
    v = ctypes.c_int()
    _check(lib().nq_mlp_one_launch_ok(H, I, H_out, T, bits_gu, bits_down, ctypes.byref(v)),
           "nq_mlp_one_launch_ok")
    return bool(v.value)


def head_workspace_bytes() -> int:
    """Workspace bytes nq_gemv_head needs on the current device."""
    v = ctypes.c_size_t()
    _check(lib().nq_head_workspace_bytes(ctypes.byref(v)), "nq_head_workspace_bytes")
    return int(v.value)


def gemv_head(packed, scales, x, K: int, N: int, T: int, bits: int, y=None, workspace=None,
              argmax=None, maxval=None, lse=None, stream=None):
    """Fused verify head: y = x W^T (stored if `y` is given) and, per token,
    the argmax, the maximum and the logsumexp of the N outputs.  Returns
    (argmax int32 [T], maxval fp32 [T], lse fp32 [T]) device tensors; the
    workspace is allocated here if not passed (torch memory)."""
    import torch
    dev = x.device
    if workspace is None:
        workspace = torch.empty(head_workspace_bytes(), dtype=torch.uint8, device=dev)
    if argmax is None:
        argmax = torch.empty(T, dtype=torch.int32, device=dev)
    if maxval is None:
        maxval = torch.empty(T, dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty(T, dtype=torch.float32, device=dev)
    _check(lib().nq_gemv_head(_dptr(packed), _dptr(scales), _dptr(x), _dptr(y), K, N, T, bits,
                              _dptr(argmax), _dptr(maxval), _dptr(lse), _dptr(workspace),
                              workspace.numel() * workspace.element_size(),
                              _stream_handle(stream)), "nq_gemv_head")
    return argmax, maxval, lse


def head_topk_workspace_bytes() -> int:
    """Workspace bytes nq_gemv_head_topk needs on the current device."""
    v = ctypes.c_size_t()
    _check(lib().nq_head_topk_workspace_bytes(ctypes.byref(v)), "nq_head_topk_workspace_bytes")
    return int(v.value)


def gemv_head_topk(packed, scales, x, K: int, N: int, T: int, bits: int, k: int, y=None,
                   workspace=None, topk_idx=None, topk_val=None, argmax=None, maxval=None,
                   lse=None, stream=None):
    """gemv_head plus the k largest logits of every token (larger value
    first, equal values by smaller index).  Returns (topk_idx int32 [T, k],
    topk_val fp32 [T, k], argmax, maxval, lse) device tensors; the workspace
    and outputs not passed are allocated here (torch memory)."""
    import torch
    dev = x.device
    if workspace is None:
        workspace = torch.empty(head_topk_workspace_bytes(), dtype=torch.uint8, device=dev)
    kk = max(k, 1)          # a bad k is the library's to reject
    if topk_idx is None:
        topk_idx = torch.empty((T, kk), dtype=torch.int32, device=dev)
    if topk_val is None:
        topk_val = torch.empty((T, kk), dtype=torch.float32, device=dev)
    if argmax is None:
        argmax = torch.empty(T, dtype=torch.int32, device=dev)
    if maxval is None:
        maxval = torch.empty(T, dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty(T, dtype=torch.float32, device=dev)
    _check(lib().nq_gemv_head_topk(_dptr(packed), _dptr(scales), _dptr(x), _dptr(y), K, N, T, bits,
                                   k, _dptr(topk_idx), _dptr(topk_val), _dptr(argmax),
                                   _dptr(maxval), _dptr(lse), _dptr(workspace),
                                   workspace.numel() * workspace.element_size(),
                                   _stream_handle(stream)), "nq_gemv_head_topk")
    return topk_idx, topk_val, argmax, maxval, lse


def gemv_head_noalloc(packed, scales, x, K: int, N: int, T: int, bits: int, y=None,
                      argmax=None, maxval=None, lse=None, stream=None):
    """gemv_head through the entry point that allocates nothing: the library
    uses its own fixed device scratch instead of a workspace.  Calls must not
    overlap on the GPU.  Returns (argmax, maxval, lse); output tensors the
    caller does not pass are created here (torch memory)."""
    import torch
    dev = x.device
    if argmax is None:
        argmax = torch.empty(T, dtype=torch.int32, device=dev)
    if maxval is None:
        maxval = torch.empty(T, dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty(T, dtype=torch.float32, device=dev)
    _check(lib().nq_gemv_head_noalloc(_dptr(packed), _dptr(scales), _dptr(x), _dptr(y), K, N, T,
                                      bits, _dptr(argmax), _dptr(maxval), _dptr(lse),
                                      _stream_handle(stream)), "nq_gemv_head_noalloc")
    return argmax, maxval, lse


def dequant(packed, scales, K: int, N: int, bits: int, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=packed.device)
    _check(lib().nq_dequant(_dptr(packed), _dptr(scales), _dptr(out), K, N, bits,
                            _stream_handle(stream)), "nq_dequant")
    return out


def last_device_error(stream=None) -> int:
    """Synchronise the stream, return and clear the device status word."""
    return int(lib().nq_last_device_error(_stream_handle(stream)))


def plan(K: int, N: int, T: int, bits: int, route: int = ROUTE_AUTO, ksplit: int = 0) -> dict:
    vals = [ctypes.c_int() for _ in range(5)]
    _check(lib().nq_gemv_plan(K, N, T, bits, route, ksplit, *[ctypes.byref(v) for v in vals]),
           "nq_gemv_plan")
    keys = ("route", "ksplit", "clusters", "stages", "smem")
    out = {k: v.value for k, v in zip(keys, vals)}
    xp = ctypes.c_int()
    _check(lib().nq_gemv_plan_x(K, N, T, bits, route, ksplit, ctypes.byref(xp)), "nq_gemv_plan_x")
    out["x"] = X_PLACES[xp.value]
    return out


def selftest_wait_timeout(limit_us: int, stream=None) -> None:
    _check(lib().nq_selftest_wait_timeout(limit_us, _stream_handle(stream)),
           "nq_selftest_wait_timeout")


class QuantizedWeight:
    """A packed weight W[N, K] resident on the device, with its GEMV."""

    def __init__(self, packed, scales, K: int, N: int, bits: int):
        self.packed, self.scales, self.K, self.N, self.bits = packed, scales, K, N, bits

    @classmethod
    def from_fp32(cls, w, bits: int, stream=None) -> "QuantizedWeight":
        codes, scales = quantize_rtn(w, bits, stream=stream)
        packed, sp = pack_device(codes, scales, bits, stream=stream)
        N, K = w.shape
        return cls(packed, sp, K, N, bits)

    @property
    def nbytes(self) -> int:
        return self.packed.numel() + 2 * self.scales.numel()

    def gemv(self, x, y=None, route: int = ROUTE_AUTO, ksplit: int = 0, stream=None):
        import torch
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.N), dtype=torch.float32, device=x.device)
        gemv(self.packed, self.scales, x, y, self.K, self.N, T, self.bits, route, ksplit, stream)
        return y
