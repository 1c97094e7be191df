"""moeq4 for GB300: a 4-bit (Q4_0 family) MoE expert-FFN layer.

Thin Python binding of the C ABI in ``include/moeq4.h``.  Functions carry the
same names as the C entry points and only marshal arguments (device pointers,
sizes, the current CUDA stream); every step of the layer runs in the CUDA
library ``libmoeq4.so``.  PyTorch provides device memory and streams.  There is
no fallback: if the library is missing or the device is not sm_103a, calls
raise ``MoeError``.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB_PATH, build

__all__ = [
    "MoeError", "MoeDebug", "load_library", "build",
    "moe_version", "moe_q4_packed_bytes", "moe_q4_pack", "moe_q4_quantize", "moe_route_topk",
    "moe_workspace_bytes", "moe_q4_forward_prefill", "moe_w4a8_forward_decode",
    "moe_w4a8_forward_decode_stack", "moe_q4_forward_prefill_stack_streamed", "moe_q8_packed_bytes",
    "moe_q8_pack", "moe_w8a8_forward_decode", "moe_get_device_status",
    "moe_clear_device_status", "make_debug", "EXPORTED_SYMBOLS",
]

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_SHAPE = -2
MOE_ERR_ALIGN = -3
MOE_ERR_UNSUPPORTED = -4
MOE_ERR_CUDA = -5
MOE_ERR_TIMEOUT = -6
MOE_ERR_WORKSPACE = -7
MOE_Q4_CODES = 0
MOE_Q4_BLOCK18 = 1
MOE_SRC_F32 = 0
MOE_SRC_BF16 = 1
MOE_OUT_FP32 = 1
MOE_STACKED_PRENORM = 2
MOE_MODE_PREFILL = 0
MOE_MODE_DECODE = 1
MOE_MODE_PREFILL_STREAMED = 2
MOE_DECODE_MAX_T = 32
MOE_W8_DECODE_MAX_T = 16

EXPORTED_SYMBOLS = (
    "moe_version", "moe_last_error_string", "moe_get_device_status", "moe_clear_device_status",
    "moe_q4_packed_bytes", "moe_q4_pack", "moe_route_topk", "moe_workspace_bytes",
    "moe_q4_forward_prefill", "moe_w4a8_forward_decode", "moe_w4a8_forward_decode_noalloc",
    "moe_q4_quantize", "moe_w4a8_forward_decode_stack", "moe_q4_forward_prefill_stack_streamed",
    "moe_q8_packed_bytes", "moe_q8_pack", "moe_w8a8_forward_decode",
)
MOE_DECODE_MAX_LAYERS = 64
MOE_NOALLOC_SCRATCH_BYTES = 8 << 20


class MoeError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"moeq4 error {code}: {message}")
        self.code = code


_DEBUG_FIELDS = ("logits", "topk_idx", "topk_w", "expert_offsets", "bucket_token", "bucket_slot",
                 "h", "q_x", "d_x", "dots_gu", "q_h", "d_h", "dots_d", "stage_events")
MOE_NUM_STAGE_EVENTS = 7


class MoeDebug(ctypes.Structure):
    """Mirror of ``struct moe_debug``: device pointers, each may be NULL."""
    _fields_ = [(name, ctypes.c_void_p) for name in _DEBUG_FIELDS]


_lib = None
_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t


def load_library(path: str | None = None):
    """Loads ``libmoeq4.so`` (raises MoeError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise MoeError(MOE_ERR_UNSUPPORTED,
                       f"{p} is missing; build it with bit_quantized_moe_q4_gb300.build()")
    lib = ctypes.CDLL(p)
    sig = {
        "moe_version": (_i, []),
        "moe_last_error_string": (ctypes.c_char_p, []),
        "moe_get_device_status": (_i, [_vp, ctypes.POINTER(_i)]),
        "moe_clear_device_status": (_i, [_vp]),
        "moe_q4_packed_bytes": (_sz, [_i, _i, _i]),
        "moe_q4_pack": (_i, [_i, _vp, _vp, _i, _i, _i, _vp, _sz, _vp]),
        "moe_q8_packed_bytes": (_sz, [_i, _i, _i]),
        "moe_q8_pack": (_i, [_vp, _vp, _i, _i, _i, _vp, _sz, _vp]),
        "moe_w8a8_forward_decode": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_uint,
                                         _vp, _vp, _sz, ctypes.POINTER(MoeDebug), _vp]),
        "moe_q4_quantize": (_i, [_i, _vp, ctypes.c_longlong, _i, _i, _vp, _vp, _vp]),
        "moe_route_topk": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp]),
        "moe_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
        "moe_q4_forward_prefill": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_uint,
                                        _vp, _vp, _sz, ctypes.POINTER(MoeDebug), _vp]),
        "moe_w4a8_forward_decode": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_uint,
                                         _vp, _vp, _sz, ctypes.POINTER(MoeDebug), _vp]),
        "moe_w4a8_forward_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                                 ctypes.c_uint, _vp, ctypes.POINTER(MoeDebug),
                                                 _vp]),
        "moe_w4a8_forward_decode_stack": (_i, [_vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                               ctypes.c_uint, _vp, _vp, _sz, _vp]),
        "moe_q4_forward_prefill_stack_streamed": (_i, [_vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                                       ctypes.c_uint, _vp, _vp, _sz, _vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc: int) -> None:
    if rc != MOE_OK:
        msg = load_library().moe_last_error_string().decode(errors="replace")
        raise MoeError(rc, msg)


def _host_ptr(t: torch.Tensor):
    if t.is_cuda or not t.is_pinned():
        raise MoeError(MOE_ERR_INVALID_ARG, "streamed expert weights must be pinned CPU tensors")
    if not t.is_contiguous():
        raise MoeError(MOE_ERR_INVALID_ARG, "tensor arguments must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise MoeError(MOE_ERR_INVALID_ARG, "tensor arguments must live on a CUDA device")
    if not t.is_contiguous():
        raise MoeError(MOE_ERR_INVALID_ARG, "tensor arguments must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def moe_version() -> int:
    return load_library().moe_version()


def moe_get_device_status(stream=None) -> int:
    v = _i(0)
    _check(load_library().moe_get_device_status(_stream(stream), ctypes.byref(v)))
    return v.value


def moe_clear_device_status(stream=None) -> None:
    _check(load_library().moe_clear_device_status(_stream(stream)))


def moe_q4_packed_bytes(E: int, N: int, K: int) -> int:
    return load_library().moe_q4_packed_bytes(E, N, K)


def moe_q4_pack(src: torch.Tensor, src_scales: torch.Tensor | None, E: int, N: int, K: int,
                fmt: int = MOE_Q4_CODES, out: torch.Tensor | None = None, stream=None):
    """Packs canonical Q4_0 weights (uint8 codes [E,N,K] + fp16 scales
    [E,N,K/32], or 18-byte blocks) into the packed layout; returns the packed
    uint8 tensor."""
    nbytes = moe_q4_packed_bytes(E, N, K)
    if out is None:
        out = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=src.device)
    _check(load_library().moe_q4_pack(fmt, _ptr(src), _ptr(src_scales), E, N, K, _ptr(out),
                                      out.numel() * out.element_size(), _stream(stream)))
    return out


def moe_q8_packed_bytes(E: int, N: int, K: int) -> int:
    return int(load_library().moe_q8_packed_bytes(E, N, K))


def moe_q8_pack(codes: torch.Tensor, scales: torch.Tensor, E: int, N: int, K: int,
                out: torch.Tensor | None = None, stream=None):
    """Packs 8-bit weights (int8 codes [E,N,K] + fp16 scales [E,N,K/32] as
    int16 bits) into 8-bit tiles; returns the packed uint8 tensor."""
    nbytes = moe_q8_packed_bytes(E, N, K)
    if out is None:
        out = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=codes.device)
    _check(load_library().moe_q8_pack(_ptr(codes), _ptr(scales), E, N, K, _ptr(out),
                                      out.numel() * out.element_size(), _stream(stream)))
    return out


def moe_q4_quantize(w: torch.Tensor, fmt: int = MOE_Q4_CODES, stream=None):
    """Encodes float weights [..., K] (fp32 or bf16, K % 32 == 0) as Q4_0
    blocks on the GPU.  Returns (codes uint8 [..., K], scales fp16 [..., K/32])
    for MOE_Q4_CODES, or the 18-byte blocks uint8 [..., K/32, 18] for
    MOE_Q4_BLOCK18."""
    if w.dtype == torch.float32:
        src_type = MOE_SRC_F32
    elif w.dtype == torch.bfloat16:
        src_type = MOE_SRC_BF16
    else:
        raise MoeError(MOE_ERR_INVALID_ARG, f"weights must be float32 or bfloat16, not {w.dtype}")
    *lead, K = w.shape
    rows = int(w.numel() // K) if K else 0
    if fmt == MOE_Q4_CODES:
        codes = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
        scales = torch.empty((*lead, K // 32), dtype=torch.float16, device=w.device)
        _check(load_library().moe_q4_quantize(src_type, _ptr(w), rows, K, fmt, _ptr(codes),
                                              _ptr(scales), _stream(stream)))
        return codes, scales
    blocks = torch.empty((*lead, K // 32, 18), dtype=torch.uint8, device=w.device)
    _check(load_library().moe_q4_quantize(src_type, _ptr(w), rows, K, fmt, _ptr(blocks), None,
                                          _stream(stream)))
    return blocks


def moe_route_topk(x: torch.Tensor, wr: torch.Tensor, k: int, logits: torch.Tensor | None = None,
                   idx: torch.Tensor | None = None, w: torch.Tensor | None = None, stream=None):
    """Router top-k.  x: bf16 [T,H]; wr: fp32 [E,H].  Returns (idx int32
    [T,k], w fp32 [T,k]); fills ``logits`` (fp32 [T,E]) when given."""
    T, H = x.shape
    E = wr.shape[0]
    if idx is None:
        idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
    if w is None:
        w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    _check(load_library().moe_route_topk(_ptr(x), _ptr(wr), T, H, E, k, _ptr(idx), _ptr(w),
                                         _ptr(logits), _stream(stream)))
    return idx, w


def moe_workspace_bytes(mode: int, T: int, H: int, I: int, E: int, k: int) -> int:
    return load_library().moe_workspace_bytes(mode, T, H, I, E, k)


def make_debug(mode: int, T: int, H: int, I: int, E: int, k: int, device="cuda"):
    """Allocates every stage output of a forward call; returns (dict of
    tensors, MoeDebug pointing at them)."""
    Tk = T * k
    G, GI = H // 32, I // 32
    d = {
        "logits": torch.empty((T, E), dtype=torch.float32, device=device),
        "topk_idx": torch.empty((T, k), dtype=torch.int32, device=device),
        "topk_w": torch.empty((T, k), dtype=torch.float32, device=device),
        "expert_offsets": torch.empty(E + 1, dtype=torch.int32, device=device),
        "bucket_token": torch.empty(Tk, dtype=torch.int32, device=device),
        "bucket_slot": torch.empty(Tk, dtype=torch.int32, device=device),
    }
    if mode == MOE_MODE_PREFILL:
        d["h"] = torch.empty((Tk, I), dtype=torch.float16, device=device)
    else:
        d["q_x"] = torch.empty((T, H), dtype=torch.int8, device=device)
        d["d_x"] = torch.empty((T, G), dtype=torch.int16, device=device)
        d["dots_gu"] = torch.empty((Tk, 2 * I, G), dtype=torch.int32, device=device)
        d["q_h"] = torch.empty((Tk, I), dtype=torch.int8, device=device)
        d["d_h"] = torch.empty((Tk, GI), dtype=torch.int16, device=device)
        d["dots_d"] = torch.empty((Tk, H, GI), dtype=torch.int32, device=device)
    dbg = MoeDebug(**{name: (t.data_ptr() if t.numel() else None) for name, t in d.items()})
    return d, dbg


def _forward(fn_name, x, wr, wgu_packed, wd_packed, I, k, out, out_fp32, workspace, debug,
             stream, prenorm=False):
    T, H = x.shape
    E = wr.shape[0]
    mode = MOE_MODE_PREFILL if fn_name == "moe_q4_forward_prefill" else MOE_MODE_DECODE
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=x.device)
    if workspace is None:
        workspace = torch.empty(max(moe_workspace_bytes(mode, T, H, I, E, k), 1),
                                dtype=torch.uint8, device=x.device)
    flags = (MOE_OUT_FP32 if out_fp32 else 0) | (MOE_STACKED_PRENORM if prenorm else 0)
    fn = getattr(load_library(), fn_name)
    _check(fn(_ptr(x), _ptr(wr), _ptr(wgu_packed), _ptr(wd_packed), T, H, I, E, k, flags,
              _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
              ctypes.byref(debug) if debug is not None else None, _stream(stream)))
    return out


def moe_w8a8_forward_decode(x, wr, wgu_q8, wd_q8, I: int, k: int, out=None, out_fp32: bool = True,
                            workspace=None, debug: MoeDebug | None = None, stream=None,
                            prenorm: bool = False):
    """One decode MoE layer with 8-bit expert weights (packed by moe_q8_pack)."""
    return _forward("moe_w8a8_forward_decode", x, wr, wgu_q8, wd_q8, I, k, out, out_fp32,
                    workspace, debug, stream, prenorm)


def moe_q4_forward_prefill(x, wr, wgu_packed, wd_packed, I: int, k: int, out=None,
                           out_fp32: bool = True, workspace=None, debug: MoeDebug | None = None,
                           stream=None, prenorm: bool = False):
    """One prefill MoE layer.  x bf16 [T,H]; wr fp32 [E,H]; packed gate/up
    ([E,2I,H]) and down ([E,H,I]) weights.  Returns out [T,H] (fp32 or bf16).
    ``prenorm`` sets MOE_STACKED_PRENORM (route and multiply RMSNorm(x))."""
    return _forward("moe_q4_forward_prefill", x, wr, wgu_packed, wd_packed, I, k, out, out_fp32,
                    workspace, debug, stream, prenorm)


def moe_w4a8_forward_decode(x, wr, wgu_packed, wd_packed, I: int, k: int, out=None,
                            out_fp32: bool = True, workspace=None,
                            debug: MoeDebug | None = None, stream=None, prenorm: bool = False):
    """One decode MoE layer on the W4A8 integer path (T <= 32)."""
    return _forward("moe_w4a8_forward_decode", x, wr, wgu_packed, wd_packed, I, k, out, out_fp32,
                    workspace, debug, stream, prenorm)


def moe_w4a8_forward_decode_stack(x, layers, I: int, k: int, out=None, out_fp32: bool = True,
                                  workspace=None, stream=None, prenorm: bool = True):
    """L stacked decode layers from one call.  ``layers``: a sequence of
    (wr, wgu_packed, wd_packed) per layer; layer l + 1 reads layer l's output
    rounded to bf16.  Returns the last layer's output [T, H]."""
    T, H = x.shape
    L = len(layers)
    E = layers[0][0].shape[0] if L else 0
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=x.device)
    if workspace is None:
        workspace = torch.empty(max(moe_workspace_bytes(MOE_MODE_DECODE, T, H, I, E, k), 1),
                                dtype=torch.uint8, device=x.device)
    arrs = [(ctypes.c_void_p * max(L, 1))(*[_ptr(layer[j]).value for layer in layers])
            for j in range(3)]
    flags = (MOE_OUT_FP32 if out_fp32 else 0) | (MOE_STACKED_PRENORM if prenorm else 0)
    _check(load_library().moe_w4a8_forward_decode_stack(
        _ptr(x), L, arrs[0], arrs[1], arrs[2], T, H, I, E, k, flags, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def moe_q4_forward_prefill_stack_streamed(x, layers, I: int, k: int, out=None,
                                          out_fp32: bool = True, workspace=None, stream=None,
                                          prenorm: bool = True):
    """L stacked prefill layers whose packed experts stay in pinned host memory
    and are copied to the GPU layer by layer, overlapped with compute.
    ``layers``: a sequence of (wr on the device, wgu_packed and wd_packed as
    pinned CPU tensors) per layer; layer l + 1 reads layer l's output rounded
    to bf16.  Returns the last layer's output [T, H]."""
    T, H = x.shape
    L = len(layers)
    E = layers[0][0].shape[0] if L else 0
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=x.device)
    if workspace is None:
        workspace = torch.empty(max(moe_workspace_bytes(MOE_MODE_PREFILL_STREAMED, T, H, I, E, k), 1),
                                dtype=torch.uint8, device=x.device)
    arrs = [(ctypes.c_void_p * max(L, 1))(*[(_ptr(layer[j]) if j == 0 else _host_ptr(layer[j])).value
                                            for layer in layers])
            for j in range(3)]
    flags = (MOE_OUT_FP32 if out_fp32 else 0) | (MOE_STACKED_PRENORM if prenorm else 0)
    _check(load_library().moe_q4_forward_prefill_stack_streamed(
        _ptr(x), L, arrs[0], arrs[1], arrs[2], T, H, I, E, k, flags, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


class StageEvents:
    """Caller-owned CUDA events the forward calls record at their stage
    boundaries (``moe_debug.stage_events``); ``ms(i, j)`` is the time from
    boundary i to boundary j of the last recorded call."""

    def __init__(self):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(MOE_NUM_STAGE_EVENTS)]
        for e in self.events:  # torch creates the CUDA event on first record
            e.record()
        self._arr = (ctypes.c_void_p * MOE_NUM_STAGE_EVENTS)(*[e.cuda_event for e in self.events])
        self.debug = MoeDebug()
        self.debug.stage_events = ctypes.cast(self._arr, ctypes.c_void_p)

    def ms(self, i: int, j: int) -> float:
        return self.events[i].elapsed_time(self.events[j])


def moe_w4a8_forward_decode_noalloc(x, wr, wgu_packed, wd_packed, I: int, k: int, out=None,
                                    out_fp32: bool = True, debug: MoeDebug | None = None,
                                    stream=None, prenorm: bool = False):
    """The decode layer with the library's fixed scratch array instead of a
    caller workspace, for callers that cannot allocate device memory (see
    include/moeq4.h).  ``out`` should be preallocated by such callers; this
    wrapper only creates it when it is not given."""
    T, H = x.shape
    E = wr.shape[0]
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=x.device)
    flags = (MOE_OUT_FP32 if out_fp32 else 0) | (MOE_STACKED_PRENORM if prenorm else 0)
    _check(load_library().moe_w4a8_forward_decode_noalloc(
        _ptr(x), _ptr(wr), _ptr(wgu_packed), _ptr(wd_packed), T, H, I, E, k, flags, _ptr(out),
        ctypes.byref(debug) if debug is not None else None, _stream(stream)))
    return out
