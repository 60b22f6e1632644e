"""Python binding of libw4a16.so (the W4A16 linear layer on GB300): argument marshalling only.

Every function here checks tensor devices, dtypes and shapes, takes raw device pointers and the
current CUDA stream from PyTorch, and calls the C entry point of the same name. All computation runs
in the library's CUDA kernels; there is no fallback. If the shared library is missing the import of
the ``lib`` handle fails loudly: build it with ``python -m w4a16_int4_weight_group_gb300.build``.

The facade mirrors ``triton_w4a16_gemm(a, b_q, scales, qzeros, group_size, zp_bias=8)`` from the
PR #51453 report (key source snippets), extended by ``bias`` and an optional ``out``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a16.so")

W4A16_F16, W4A16_BF16 = 0, 1
STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "MISALIGNED", 4: "CUDA", 5: "TIMEOUT"}
PATHS = {0: "none", 1: "generic", 2: "decode", 3: "prefill"}


class W4A16Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("k_blocks_per_stage", ctypes.c_int32), ("m_tile", ctypes.c_int32),
                ("n_tile", ctypes.c_int32), ("k_split", ctypes.c_int32), ("warps", ctypes.c_int32),
                ("grid", ctypes.c_int64), ("smem_bytes", ctypes.c_int32), ("stream_k", ctypes.c_int32)]

    def as_dict(self):
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["path_name"] = PATHS.get(self.path, str(self.path))
        return d


_lib = None
_c_i64, _c_int, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p

# (name, restype, argtypes) of every entry point declared in include/w4a16.h
SIGNATURES = [
    ("w4a16_pack", _c_int, [_vp, _vp, _c_i64, _c_i64, _vp]),
    ("w4a16_unpack", _c_int, [_vp, _vp, _c_i64, _c_i64, _vp]),
    ("w4a16_repack_k_to_n", _c_int, [_vp, _vp, _c_i64, _c_i64, _vp]),
    ("w4a16_dequant", _c_int, [_vp, _vp, _vp, _c_i64, _c_i64, _c_int, _c_int, _c_int, _vp, _vp]),
    ("w4a16_gemm", _c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _vp, _vp, _c_i64, _c_i64, _c_i64, _c_int, _vp]),
    ("w4a16_gemm_ws", _c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _vp, _vp, _c_i64, _c_i64, _c_i64, _c_int, _vp,
                               ctypes.c_size_t, _vp]),
    ("w4a16_gemm_workspace_size", ctypes.c_size_t, [_c_i64, _c_i64, _c_i64, _c_int, _c_int]),
    ("w4a16_layer_create", _c_int, [_vp, _vp, _vp, _c_int, _c_int, _vp, _c_i64, _c_i64, _c_int,
                                    ctypes.POINTER(_vp)]),
    ("w4a16_layer_create_prepacked", _c_int, [_vp, _vp, _vp, _c_int, _c_int, _vp, _c_i64, _c_i64, _c_int,
                                              ctypes.POINTER(_vp)]),
    ("w4a16_prepack_bytes", ctypes.c_size_t, [_c_i64, _c_i64]),
    ("w4a16_prepack", _c_int, [_vp, _vp, _c_i64, _c_i64, _vp]),
    ("w4a16_layer_gemm", _c_int, [_vp, _vp, _vp, _c_i64, _vp, ctypes.c_size_t, _vp]),
    ("w4a16_layer_workspace_size", ctypes.c_size_t, [_vp, _c_i64]),
    ("w4a16_layer_destroy", _c_int, [_vp]),
    ("w4a16_gemm_noalloc", _c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _vp, _vp, _c_i64, _c_i64, _c_i64, _c_int,
                                    _vp]),
    ("w4a16_can_implement", _c_int, [_c_i64, _c_i64, _c_int, _c_int, _c_int]),
    ("w4a16_plan", _c_int, [_c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_int, _c_int, _c_int, ctypes.POINTER(Plan)]),
    ("w4a16_last_error", ctypes.c_char_p, []),
    ("w4a16_get_device_error", _c_int, []),
    ("w4a16_debug_selected_path", _c_int, [_c_i64, _c_i64, _c_i64, _c_int]),
    ("w4a16_debug_force_path", _c_int, [_c_int]),
    ("w4a16_debug_decode_override", _c_int, [_c_int, _c_int, _c_int]),
    ("w4a16_debug_set_wait_limit_ns", _c_int, [ctypes.c_uint64]),
    ("w4a16_debug_inject_stall", _c_int, [_c_int]),
    ("w4a16_debug_launch_count", ctypes.c_uint64, []),
    ("w4a16_version", ctypes.c_char_p, []),
]


def lib() -> ctypes.CDLL:
    """The loaded libw4a16.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m w4a16_int4_weight_group_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def last_error() -> str:
    return lib().w4a16_last_error().decode()


def _check(status: int):
    if status != 0:
        raise W4A16Error(status, last_error())


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float16:
        return W4A16_F16
    if dt == torch.bfloat16:
        return W4A16_BF16
    raise W4A16Error(2, f"Only float16/bfloat16 activations are supported (got {dt})")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _layer_gemm_fn():
    """The prepared-layer call: the CPython marshalling module when it was built (it converts the
    integer arguments with less host time per call than ctypes), else the ctypes function."""
    L = lib()
    try:
        from . import _w4a16_call
    except ImportError:
        return L.w4a16_layer_gemm
    _w4a16_call.bind(ctypes.cast(L.w4a16_layer_gemm, ctypes.c_void_p).value)
    return _w4a16_call.layer_gemm


def _stream(device: torch.device):
    """The current CUDA stream of `device` as a raw handle (without building a Stream object when
    the runtime offers the raw query)."""
    if _raw_stream is not None:
        return ctypes.c_void_p(_raw_stream(device.index if device.index is not None else torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _require_cuda(*ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous (row-major)")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("all tensors must be on the same device")
    return dev


def w4a16_pack(q: torch.Tensor, packed: Optional[torch.Tensor] = None) -> torch.Tensor:
    """uint8 [rows, n] (values 0..15) -> int32 [rows, n/8]; nibble j of word c <- column 8c+j."""
    if q.dtype != torch.uint8 or q.dim() != 2:
        raise ValueError("q must be a 2-D uint8 tensor")
    rows, n = q.shape
    if packed is None:
        packed = torch.empty((rows, n // 8), dtype=torch.int32, device=q.device)
    dev = _require_cuda(q, packed)
    _check(lib().w4a16_pack(_ptr(q), _ptr(packed), rows, n, _stream(dev)))
    return packed


def w4a16_unpack(packed: torch.Tensor, n: Optional[int] = None, q: Optional[torch.Tensor] = None) -> torch.Tensor:
    """int32 [rows, n/8] -> uint8 [rows, n]."""
    if packed.dtype != torch.int32 or packed.dim() != 2:
        raise ValueError("packed must be a 2-D int32 tensor")
    rows = packed.shape[0]
    n = packed.shape[1] * 8 if n is None else n
    if q is None:
        q = torch.empty((rows, n), dtype=torch.uint8, device=packed.device)
    dev = _require_cuda(q, packed)
    _check(lib().w4a16_unpack(_ptr(packed), _ptr(q), rows, n, _stream(dev)))
    return q


def w4a16_repack_k_to_n(k_packed: torch.Tensor, b_q: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Weights packed along K, int32 [n, k/8] -> this library's b_q, int32 [k, n/8] (nibble j of a
    K-packed word is row 8c+j; see the C header)."""
    if k_packed.dtype != torch.int32 or k_packed.dim() != 2:
        raise ValueError("k_packed must be a 2-D int32 tensor")
    n, k = k_packed.shape[0], k_packed.shape[1] * 8
    if b_q is None:
        b_q = torch.empty((k, n // 8), dtype=torch.int32, device=k_packed.device)
    dev = _require_cuda(k_packed, b_q)
    _check(lib().w4a16_repack_k_to_n(_ptr(k_packed), _ptr(b_q), k, n, _stream(dev)))
    return b_q


def w4a16_prepack(b_q: torch.Tensor, b_pp: Optional[torch.Tensor] = None) -> torch.Tensor:
    """b_q int32 [K, N/8] -> the prepacked layout (a flat int32 tensor of w4a16_prepack_bytes / 4
    words; see the C header)."""
    if b_q.dtype != torch.int32 or b_q.dim() != 2:
        raise ValueError("b_q must be a 2-D int32 tensor")
    k, n = b_q.shape[0], b_q.shape[1] * 8
    nbytes = int(lib().w4a16_prepack_bytes(k, n))
    if b_pp is None:
        b_pp = torch.empty(nbytes // 4, dtype=torch.int32, device=b_q.device)
    if b_pp.numel() * 4 < nbytes:
        raise ValueError(f"b_pp holds {b_pp.numel() * 4} bytes, {nbytes} needed")
    dev = _require_cuda(b_q, b_pp)
    _check(lib().w4a16_prepack(_ptr(b_q), _ptr(b_pp), k, n, _stream(dev)))
    return b_pp


def w4a16_dequant(b_q: torch.Tensor, scales: torch.Tensor, qzeros: Optional[torch.Tensor], group_size: int,
                  zp_bias: int = 8, w_out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """dequant(W)[k, n] = RNE_dtype((q - zp) * scale) as a [K, N] tensor of the scales' dtype."""
    k, nw = b_q.shape
    n = nw * 8
    if w_out is None:
        w_out = torch.empty((k, n), dtype=scales.dtype, device=b_q.device)
    dev = _require_cuda(b_q, scales, qzeros, w_out)
    _check(lib().w4a16_dequant(_ptr(b_q), _ptr(scales), _ptr(qzeros), k, n, group_size, zp_bias,
                               _dtype_code(scales.dtype), _ptr(w_out), _stream(dev)))
    return w_out


_workspaces = {}


# workspace bytes per (device, m, k, n, group_size, dtype): a pure function of the shape and the device
_ws_need: dict = {}


def workspace_for(device: torch.device, stream, nbytes: int) -> torch.Tensor:
    """A scratch buffer of at least nbytes, kept per (device, stream) and grown on demand.

    It is zero-filled when (re)allocated; the library leaves its flag area (the first 4 KiB) zero
    after every call and needs nothing else of the rest between calls.
    """
    key = (device.index, int(stream))
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = buf
    return buf


def w4a16_gemm(a: torch.Tensor, b_q: torch.Tensor, scales: torch.Tensor, qzeros: Optional[torch.Tensor],
               group_size: int, zp_bias: int = 8, bias: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None, use_workspace: bool = True) -> torch.Tensor:
    """out[M, N] = cast(a[M, K] @ dequant(b_q, scales, qzeros|zp_bias) + bias), fp32 accumulation.

    Output shape (M, b_q.shape[1] * 8), dtype and device of ``a`` (PR #51453 report, fake impl).
    With ``use_workspace`` a per-(device, stream) scratch buffer is passed to ``w4a16_gemm_ws`` so
    that large-M shapes can use stream-K; otherwise ``w4a16_gemm`` (no scratch) is called.
    """
    if a.dim() != 2 or b_q.dim() != 2:
        raise ValueError("a and b_q must be 2-D")
    m, k = a.shape
    n = b_q.shape[1] * 8
    if b_q.shape[0] != k:
        raise ValueError(f"b_q has {b_q.shape[0]} rows, a has K={k}")
    if out is None:
        out = torch.empty((m, n), dtype=a.dtype, device=a.device)
    dev = _require_cuda(a, b_q, scales, qzeros, bias, out)
    if scales.dtype != a.dtype or out.dtype != a.dtype or (bias is not None and bias.dtype != a.dtype):
        raise ValueError("scales, bias and out must have the dtype of a")
    if b_q.dtype != torch.int32 or (qzeros is not None and qzeros.dtype != torch.int32):
        raise ValueError("b_q and qzeros must be int32")
    stream = _stream(dev)
    code = _dtype_code(a.dtype)
    need = 0
    if use_workspace:
        key = (dev.index, m, k, n, group_size, code)
        need = _ws_need.get(key)
        if need is None:
            need = _ws_need[key] = int(lib().w4a16_gemm_workspace_size(m, k, n, group_size, code))
    if need:
        ws = workspace_for(dev, stream.value or 0, need)
        _check(lib().w4a16_gemm_ws(_ptr(a), _ptr(b_q), _ptr(scales), _ptr(qzeros), group_size, zp_bias,
                                   _ptr(bias), _ptr(out), m, k, n, code, _ptr(ws), ws.numel(),
                                   stream))
    else:
        _check(lib().w4a16_gemm(_ptr(a), _ptr(b_q), _ptr(scales), _ptr(qzeros), group_size, zp_bias, _ptr(bias),
                                _ptr(out), m, k, n, code, stream))
    return out


class W4A16Linear:
    """A prepared W4A16 layer: out[M, N] = a[M, K] @ dequant(W) (+ bias), as w4a16_gemm.

    Wraps the library's prepared-layer handle (w4a16_layer_create): the weights (b_q, scales, qzeros or
    zp_bias, bias) are checked once, and the dispatcher's plan and the weight descriptors are kept per
    call shape inside the library, so each call checks and encodes only the activations and the output.
    The layer keeps references to its tensors (the handle stores their pointers).
    """

    def __init__(self, b_q: torch.Tensor, scales: torch.Tensor, qzeros: Optional[torch.Tensor], group_size: int,
                 zp_bias: int = 8, bias: Optional[torch.Tensor] = None, use_workspace: bool = True,
                 prepacked: bool = False):
        """prepacked: keep the weights in the library's prepacked layout (w4a16_prepack, made here
        from b_q on the current stream) and run the layer on it; b_q is not kept."""
        if b_q.dim() != 2 or b_q.dtype != torch.int32:
            raise ValueError("b_q must be a 2-D int32 tensor [K, N/8]")
        if qzeros is not None and qzeros.dtype != torch.int32:
            raise ValueError("qzeros must be int32")
        if bias is not None and bias.dtype != scales.dtype:
            raise ValueError("bias must have the dtype of scales")
        self._handle = None
        self.device = _require_cuda(b_q, scales, qzeros, bias)
        self.k, self.n = b_q.shape[0], b_q.shape[1] * 8
        self.dtype = scales.dtype
        self.code = _dtype_code(scales.dtype)
        self.group_size, self.zp_bias = int(group_size), int(zp_bias)
        self.use_workspace = use_workspace
        self._need = {}
        L = lib()
        h = ctypes.c_void_p()
        self.prepacked = prepacked
        with torch.cuda.device(self.device):
            if prepacked:
                b_pp = w4a16_prepack(b_q)
                self._tensors = (b_pp, scales, qzeros, bias)
                _check(L.w4a16_layer_create_prepacked(b_pp.data_ptr(), scales.data_ptr(),
                                                      None if qzeros is None else qzeros.data_ptr(), self.group_size,
                                                      self.zp_bias, None if bias is None else bias.data_ptr(),
                                                      self.k, self.n, self.code, ctypes.byref(h)))
            else:
                self._tensors = (b_q, scales, qzeros, bias)
                _check(L.w4a16_layer_create(b_q.data_ptr(), scales.data_ptr(),
                                            None if qzeros is None else qzeros.data_ptr(), self.group_size,
                                            self.zp_bias, None if bias is None else bias.data_ptr(),
                                            self.k, self.n, self.code, ctypes.byref(h)))
        self._handle = h.value
        self._lib = L
        self._gemm = _layer_gemm_fn()
        self._dev_index = self.device.index if self.device.index is not None else torch.cuda.current_device()

    def __del__(self):
        h = getattr(self, "_handle", None)
        if h and _lib is not None:
            _lib.w4a16_layer_destroy(h)
            self._handle = None

    def __call__(self, a: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        # the checks use the cheapest tensor queries, each shape read once (every `.shape` builds a new
        # size object; a decode call takes a few microseconds)
        dev = self._dev_index
        sa = a.shape
        if (a.dtype is not self.dtype or len(sa) != 2 or sa[1] != self.k or a.get_device() != dev
                or not a.is_contiguous()):
            raise ValueError(f"a must be a contiguous [M, {self.k}] {self.dtype} tensor on {self.device}")
        m = sa[0]
        if out is None:
            out = torch.empty((m, self.n), dtype=self.dtype, device=self.device)
        else:
            so = out.shape
            if (out.dtype is not self.dtype or len(so) != 2 or so[0] != m or so[1] != self.n
                    or out.get_device() != dev or not out.is_contiguous()):
                raise ValueError(f"out must be a contiguous [{m}, {self.n}] {self.dtype} tensor on {self.device}")
        stream = _raw_stream(dev) if _raw_stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        need = 0
        if self.use_workspace:
            need = self._need.get(m)
            if need is None:
                need = self._need[m] = int(self._lib.w4a16_layer_workspace_size(self._handle, m))
        if need:
            ws = workspace_for(self.device, stream, need)
            st = self._gemm(self._handle, a.data_ptr(), out.data_ptr(), m, ws.data_ptr(), ws.numel(), stream)
        else:
            st = self._gemm(self._handle, a.data_ptr(), out.data_ptr(), m, None, 0, stream)
        if st != 0:
            raise W4A16Error(st, last_error())
        return out


def w4a16_can_implement(k: int, n: int, group_size: int, dtype, has_g_idx: bool = False):
    """(True, "") or (False, reason), like the pages' can_implement."""
    code = dtype if isinstance(dtype, int) else ({torch.float16: 0, torch.bfloat16: 1}.get(dtype, 99))
    st = lib().w4a16_can_implement(k, n, group_size, code, int(bool(has_g_idx)))
    return (True, "") if st == 0 else (False, last_error())


def w4a16_plan(m: int, k: int, n: int, group_size: int, dtype=W4A16_F16, has_zp: bool = False,
               num_sms: int = 0, with_workspace: bool = True) -> dict:
    p = Plan()
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    _check(lib().w4a16_plan(m, k, n, group_size, code, int(bool(has_zp)), num_sms, int(bool(with_workspace)),
                            ctypes.byref(p)))
    return p.as_dict()


def w4a16_gemm_workspace_size(m: int, k: int, n: int, group_size: int, dtype=W4A16_F16) -> int:
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    return int(lib().w4a16_gemm_workspace_size(m, k, n, group_size, code))


def w4a16_get_device_error() -> int:
    """The library's device-side error status (read and cleared). After a TIMEOUT a stream-K call may
    have stopped with partial-tile flags still set in its workspace, so the flag area of every
    workspace this module keeps is zeroed again before any further call can use it."""
    st = lib().w4a16_get_device_error()
    if st == 5:
        for buf in _workspaces.values():
            buf[:4096].zero_()
        torch.cuda.synchronize()
    return st


def w4a16_debug_selected_path(m: int, k: int, n: int, group_size: int) -> int:
    return lib().w4a16_debug_selected_path(m, k, n, group_size)


def w4a16_debug_force_path(path):
    """Restrict the dispatcher to a path ("generic", "decode", "prefill"), or lift it (None)."""
    code = {None: -1, "generic": 1, "decode": 2, "prefill": 3}[path]
    _check(lib().w4a16_debug_force_path(code))


def w4a16_debug_decode_override(consumer_groups: int = 0, k_split: int = 0, k_blocks_per_stage: int = 0):
    """Fix the decode plan's consumer groups, split-K factor and stage size (0: automatic)."""
    _check(lib().w4a16_debug_decode_override(consumer_groups, k_split, k_blocks_per_stage))


def w4a16_debug_set_wait_limit_ns(ns: int):
    _check(lib().w4a16_debug_set_wait_limit_ns(ns))


def w4a16_debug_inject_stall(on: bool):
    _check(lib().w4a16_debug_inject_stall(int(bool(on))))


def w4a16_debug_launch_count() -> int:
    return int(lib().w4a16_debug_launch_count())


def w4a16_version() -> str:
    return lib().w4a16_version().decode()


__all__ = ["w4a16_pack", "w4a16_unpack", "w4a16_prepack", "w4a16_dequant", "w4a16_gemm", "w4a16_can_implement", "w4a16_plan",
           "w4a16_gemm_workspace_size", "workspace_for",
           "w4a16_get_device_error", "w4a16_debug_selected_path", "w4a16_debug_force_path",
           "w4a16_debug_decode_override",
           "w4a16_debug_set_wait_limit_ns",
           "w4a16_debug_inject_stall",
           "w4a16_debug_launch_count", "w4a16_version", "W4A16Error", "lib", "last_error", "LIB_PATH",
           "SIGNATURES", "PATHS"]
