"""ctypes binding of the C ABI in ``include/conv3d_fp8.h`` (argument marshalling only).

Every entry point keeps its C name. Tensors are passed as raw device pointers (``data_ptr()``);
torch is only used for device memory and streams. There is no fallback of any kind: if the CUDA
library has not been built, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

CONV3D_OK = 0
CONV3D_EINVAL = 1
CONV3D_EUNSUPPORTED = 2
CONV3D_ENOMEM = 3
CONV3D_ECUDA = 4
CONV3D_EDEVICE = 5

_lock = threading.Lock()
_lib = None


class Conv3dFp8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {conv3d_fp8_strerror(status)} (status {status})")


class Options(ctypes.Structure):
    _fields_ = [("splits", ctypes.c_int), ("block_n", ctypes.c_int), ("max_ctas", ctypes.c_int),
                ("wait_timeout_ms", ctypes.c_int), ("debug_flags", ctypes.c_int),
                ("route", ctypes.c_int), ("cta_pair", ctypes.c_int),
                ("input_layout", ctypes.c_int), ("epilogue", ctypes.c_int),
                ("overlap", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("Do", ctypes.c_int), ("Ho", ctypes.c_int), ("Wo", ctypes.c_int),
                ("npq", ctypes.c_longlong), ("k_gemm", ctypes.c_int), ("block_m", ctypes.c_int),
                ("block_n", ctypes.c_int), ("m_tiles", ctypes.c_int), ("n_tiles", ctypes.c_int),
                ("k_blocks", ctypes.c_int), ("splits", ctypes.c_int),
                ("k_blocks_per_split", ctypes.c_int), ("stages", ctypes.c_int),
                ("row_chk", ctypes.c_int), ("grid", ctypes.c_int), ("sm_count", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t), ("route", ctypes.c_int),
                ("cta_pair", ctypes.c_int), ("full_tiles", ctypes.c_int),
                ("epilogue", ctypes.c_int), ("overlap_planes", ctypes.c_int),
                ("overlap_units", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load the in-tree CUDA library. Raises if it is missing: there is no other code path."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is not built; run `python -m fp8_implicit_gemm_gb300.build`"
                    " (or __graft_entry__.build()) first")
            lib = ctypes.CDLL(path)
            ci, vp = ctypes.c_int, ctypes.c_void_p
            i3 = ctypes.POINTER(ctypes.c_int)
            lib.conv3d_fp8_plan.restype = ci
            lib.conv3d_fp8_plan.argtypes = [ctypes.POINTER(vp)] + [ci] * 9 + [i3, i3, ci]
            lib.conv3d_fp8_plan_ex.restype = ci
            lib.conv3d_fp8_plan_ex.argtypes = ([ctypes.POINTER(vp)] + [ci] * 9 + [i3, i3, ci]
                                               + [ctypes.POINTER(Options)])
            lib.conv3d_fp8_run.restype = ci
            lib.conv3d_fp8_run.argtypes = [vp, vp, vp, vp, vp, vp, i3, i3, vp]
            lib.conv3d_fp8_set_timing_events.restype = ci
            lib.conv3d_fp8_set_timing_events.argtypes = [vp, vp, vp]
            lib.conv3d_fp8_set_pack_timing_event.restype = ci
            lib.conv3d_fp8_set_pack_timing_event.argtypes = [vp, vp]
            lib.conv3d_fp8_set_write_counter.restype = ci
            lib.conv3d_fp8_set_write_counter.argtypes = [vp, vp]
            lib.conv3d_fp8_run_noalloc.restype = ci
            lib.conv3d_fp8_run_noalloc.argtypes = [ci] * 9 + [i3, i3, vp, vp, vp, vp, vp, vp]
            lib.conv3d_fp8_noalloc_check.restype = ci
            lib.conv3d_fp8_noalloc_check.argtypes = []
            lib.conv3d_fp8_check.restype = ci
            lib.conv3d_fp8_check.argtypes = [vp]
            lib.conv3d_fp8_get_info.restype = ci
            lib.conv3d_fp8_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
            lib.conv3d_fp8_describe.restype = ci
            lib.conv3d_fp8_describe.argtypes = ([ci] * 9 + [i3, i3, ci, ctypes.POINTER(Options),
                                                            ctypes.POINTER(PlanInfo)])
            lib.conv3d_bf16_plan.restype = ci
            lib.conv3d_bf16_plan.argtypes = [ctypes.POINTER(vp)] + [ci] * 9 + [i3, i3, ci]
            lib.conv3d_bf16_plan_ex.restype = ci
            lib.conv3d_bf16_plan_ex.argtypes = ([ctypes.POINTER(vp)] + [ci] * 9 + [i3, i3, ci]
                                                + [ctypes.POINTER(Options)])
            lib.conv3d_bf16_run.restype = ci
            lib.conv3d_bf16_run.argtypes = [vp, vp, vp, vp, i3, i3, vp]
            lib.conv3d_fp8_run_host.restype = ci
            lib.conv3d_fp8_run_host.argtypes = [vp, vp, vp, vp, vp, i3, i3, vp]
            lib.conv3d_bf16_run_host.restype = ci
            lib.conv3d_bf16_run_host.argtypes = [vp, vp, vp, vp, i3, i3, vp]
            lib.conv3d_bf16_describe.restype = ci
            lib.conv3d_bf16_describe.argtypes = ([ci] * 9 + [i3, i3, ci, ctypes.POINTER(Options),
                                                             ctypes.POINTER(PlanInfo)])
            lib.conv3d_fp8_quantize.restype = ci
            lib.conv3d_fp8_quantize.argtypes = [vp, ci, ctypes.c_longlong, vp, vp, vp]
            lib.conv3d_fp8_run_quantize_x.restype = ci
            lib.conv3d_fp8_run_quantize_x.argtypes = [vp, vp, ci, vp, vp, vp, i3, i3, vp, vp]
            lib.conv3d_fp8_workspace_size.restype = ctypes.c_size_t
            lib.conv3d_fp8_workspace_size.argtypes = [vp]
            lib.conv3d_fp8_out_dims.restype = ci
            lib.conv3d_fp8_out_dims.argtypes = [vp, i3, i3, i3]
            lib.conv3d_fp8_destroy.restype = None
            lib.conv3d_fp8_destroy.argtypes = [vp]
            lib.conv3d_fp8_strerror.restype = ctypes.c_char_p
            lib.conv3d_fp8_strerror.argtypes = [ci]
            _lib = lib
    return _lib


def _int3(v):
    if isinstance(v, int):
        v = (v, v, v)
    v = tuple(int(i) for i in v)
    if len(v) != 3:
        raise ValueError("expected an int or 3 ints (d, h, w)")
    return (ctypes.c_int * 3)(*v)


def _options(**kw) -> Options | None:
    if not kw:
        return None
    o = Options()
    for k, v in kw.items():
        if v is not None:
            setattr(o, k, int(v))
    return o


def _ptr(t) -> int:
    """Device address of a torch tensor (or an int address, passed through)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _host_ptr(t) -> int:
    """Host address of a CPU torch tensor (or an int address, passed through)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if t.is_cuda:
        raise ValueError("expected a CPU tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _raise(status: int, where: str):
    if status != CONV3D_OK:
        raise Conv3dFp8Error(status, where)


def conv3d_fp8_strerror(status: int) -> str:
    return load().conv3d_fp8_strerror(int(status)).decode()


def conv3d_fp8_plan(N, C, D, H, W, K, T, R, S, stride, pad, device=0, **options) -> int:
    """Create a plan; returns its handle. Keyword options (0 = the library's choice): splits,
    block_n, max_ctas, wait_timeout_ms, debug_flags, route, cta_pair, input_layout (1 = x is
    NDHWC), epilogue (2 = TMA-store epilogue), overlap (-1 = never pack beside the GEMM, P > 0 =
    pack P input planes before it); see conv3d_fp8_options in include/conv3d_fp8.h."""
    lib = load()
    h = ctypes.c_void_p()
    o = _options(**options)
    if o is None:
        st = lib.conv3d_fp8_plan(ctypes.byref(h), N, C, D, H, W, K, T, R, S, _int3(stride),
                                 _int3(pad), device)
    else:
        st = lib.conv3d_fp8_plan_ex(ctypes.byref(h), N, C, D, H, W, K, T, R, S, _int3(stride),
                                    _int3(pad), device, ctypes.byref(o))
    _raise(st, "conv3d_fp8_plan")
    return h.value


def conv3d_fp8_run(plan, x, w, scale_x, scale_w, y, stride, pad, stream=None) -> None:
    st = load().conv3d_fp8_run(plan, _ptr(x), _ptr(w), _ptr(scale_x), _ptr(scale_w), _ptr(y),
                               _int3(stride), _int3(pad), _stream(stream))
    _raise(st, "conv3d_fp8_run")


def conv3d_fp8_run_status(plan, x, w, scale_x, scale_w, y, stride, pad, stream=None) -> int:
    """As conv3d_fp8_run, but returns the status code instead of raising."""
    return load().conv3d_fp8_run(plan, _ptr(x), _ptr(w), _ptr(scale_x), _ptr(scale_w), _ptr(y),
                                 _int3(stride), _int3(pad), _stream(stream))


def conv3d_fp8_run_host_status(plan, x_host, w_host, scales_host, y_host, stride, pad,
                               stream=None) -> int:
    """conv3d_fp8_run_host: CPU tensors (page-locked for asynchronous copies); scales_host holds
    (scale_x, scale_w) as fp32. Returns the status code."""
    return load().conv3d_fp8_run_host(plan, _host_ptr(x_host), _host_ptr(w_host),
                                      _host_ptr(scales_host), _host_ptr(y_host), _int3(stride),
                                      _int3(pad), _stream(stream))


def conv3d_fp8_run_host(plan, x_host, w_host, scales_host, y_host, stride, pad,
                        stream=None) -> None:
    _raise(conv3d_fp8_run_host_status(plan, x_host, w_host, scales_host, y_host, stride, pad,
                                      stream), "conv3d_fp8_run_host")


def conv3d_fp8_run_noalloc_status(N, C, D, H, W, K, T, R, S, stride, pad, x, w, scale_x,
                                  scale_w, y, stream=None) -> int:
    """Allocation-free run (no plan; scratch in a fixed device array of the library, see
    include/conv3d_fp8.h). Returns the status code."""
    return load().conv3d_fp8_run_noalloc(N, C, D, H, W, K, T, R, S, _int3(stride), _int3(pad),
                                         _ptr(x), _ptr(w), _ptr(scale_x), _ptr(scale_w), _ptr(y),
                                         _stream(stream))


def conv3d_fp8_noalloc_check() -> int:
    """Synchronise the current device, then report (and clear) the status word of its latest
    allocation-free call: CONV3D_OK or CONV3D_EDEVICE."""
    return int(load().conv3d_fp8_noalloc_check())


def conv3d_fp8_run_noalloc(N, C, D, H, W, K, T, R, S, stride, pad, x, w, scale_x, scale_w, y,
                           stream=None) -> None:
    _raise(conv3d_fp8_run_noalloc_status(N, C, D, H, W, K, T, R, S, stride, pad, x, w, scale_x,
                                         scale_w, y, stream), "conv3d_fp8_run_noalloc")


def _raw_event(ev):
    if ev is None:
        return None
    if isinstance(ev, int):
        return ev
    if not ev.cuda_event:       # torch creates its event lazily, on first record
        ev.record()
    return ev.cuda_event


def conv3d_fp8_set_timing_events(plan, ev_begin, ev_end) -> None:
    """Record the given events (torch.cuda.Event or raw cudaEvent_t ints; None to clear) around
    the main kernel of every later run of the plan."""
    _raise(load().conv3d_fp8_set_timing_events(plan, _raw_event(ev_begin), _raw_event(ev_end)),
           "conv3d_fp8_set_timing_events")


def conv3d_fp8_set_write_counter_status(plan, counts) -> int:
    """Count the stores to each output element into `counts` (a zeroed uint32/int32 device
    tensor of N*K*Do*Ho*Wo elements; None stops); only a library built with C3D_COUNT_WRITES
    counts, the product build returns CONV3D_EUNSUPPORTED."""
    return load().conv3d_fp8_set_write_counter(plan, _ptr(counts) if counts is not None else None)


def conv3d_fp8_set_pack_timing_event(plan, ev_pack) -> None:
    """Record the given event (None to clear) right before the pack kernel of every later run
    of the plan; with the begin event of conv3d_fp8_set_timing_events it brackets the pack."""
    _raise(load().conv3d_fp8_set_pack_timing_event(plan, _raw_event(ev_pack)),
           "conv3d_fp8_set_pack_timing_event")


def conv3d_fp8_check(plan) -> int:
    """Synchronise and return (and clear) the plan's device status: CONV3D_OK or CONV3D_EDEVICE."""
    return load().conv3d_fp8_check(plan)


def conv3d_fp8_get_info(plan) -> dict:
    info = PlanInfo()
    _raise(load().conv3d_fp8_get_info(plan, ctypes.byref(info)), "conv3d_fp8_get_info")
    return info.as_dict()


def conv3d_fp8_describe(N, C, D, H, W, K, T, R, S, stride, pad, sm_count, **options) -> dict:
    """Host-only planning decision (no device access)."""
    info = PlanInfo()
    o = _options(**options)
    st = load().conv3d_fp8_describe(N, C, D, H, W, K, T, R, S, _int3(stride), _int3(pad),
                                    sm_count, ctypes.byref(o) if o is not None else None,
                                    ctypes.byref(info))
    _raise(st, "conv3d_fp8_describe")
    return info.as_dict()


def conv3d_fp8_describe_status(N, C, D, H, W, K, T, R, S, stride, pad, sm_count, **options) -> int:
    info = PlanInfo()
    o = _options(**options)
    return load().conv3d_fp8_describe(N, C, D, H, W, K, T, R, S, _int3(stride), _int3(pad),
                                      sm_count, ctypes.byref(o) if o is not None else None,
                                      ctypes.byref(info))


def conv3d_fp8_workspace_size(plan) -> int:
    return int(load().conv3d_fp8_workspace_size(plan))


def conv3d_fp8_out_dims(plan) -> tuple[int, int, int]:
    d, h, w = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _raise(load().conv3d_fp8_out_dims(plan, ctypes.byref(d), ctypes.byref(h), ctypes.byref(w)),
           "conv3d_fp8_out_dims")
    return d.value, h.value, w.value


def conv3d_fp8_destroy(plan) -> None:
    if plan:
        load().conv3d_fp8_destroy(plan)


# ------------------------------------------------------------------------- BF16-input twin
def conv3d_bf16_plan(N, C, D, H, W, K, T, R, S, stride, pad, device=0, **options) -> int:
    """Create a plan of the BF16-input twin (same options as conv3d_fp8_plan)."""
    lib = load()
    h = ctypes.c_void_p()
    o = _options(**options)
    if o is None:
        st = lib.conv3d_bf16_plan(ctypes.byref(h), N, C, D, H, W, K, T, R, S, _int3(stride),
                                  _int3(pad), device)
    else:
        st = lib.conv3d_bf16_plan_ex(ctypes.byref(h), N, C, D, H, W, K, T, R, S, _int3(stride),
                                     _int3(pad), device, ctypes.byref(o))
    _raise(st, "conv3d_bf16_plan")
    return h.value


def conv3d_bf16_run_status(plan, x, w, y, stride, pad, stream=None) -> int:
    return load().conv3d_bf16_run(plan, _ptr(x), _ptr(w), _ptr(y), _int3(stride), _int3(pad),
                                  _stream(stream))


def conv3d_bf16_run(plan, x, w, y, stride, pad, stream=None) -> None:
    _raise(conv3d_bf16_run_status(plan, x, w, y, stride, pad, stream), "conv3d_bf16_run")


def conv3d_bf16_run_host_status(plan, x_host, w_host, y_host, stride, pad, stream=None) -> int:
    return load().conv3d_bf16_run_host(plan, _host_ptr(x_host), _host_ptr(w_host),
                                       _host_ptr(y_host), _int3(stride), _int3(pad),
                                       _stream(stream))


def conv3d_bf16_run_host(plan, x_host, w_host, y_host, stride, pad, stream=None) -> None:
    _raise(conv3d_bf16_run_host_status(plan, x_host, w_host, y_host, stride, pad, stream),
           "conv3d_bf16_run_host")


def conv3d_bf16_describe_status(N, C, D, H, W, K, T, R, S, stride, pad, sm_count,
                                **options) -> int:
    info = PlanInfo()
    o = _options(**options)
    return load().conv3d_bf16_describe(N, C, D, H, W, K, T, R, S, _int3(stride), _int3(pad),
                                       sm_count, ctypes.byref(o) if o is not None else None,
                                       ctypes.byref(info))


def conv3d_bf16_describe(N, C, D, H, W, K, T, R, S, stride, pad, sm_count, **options) -> dict:
    """Host-only planning decision of the BF16-input twin (no device access)."""
    info = PlanInfo()
    o = _options(**options)
    st = load().conv3d_bf16_describe(N, C, D, H, W, K, T, R, S, _int3(stride), _int3(pad),
                                     sm_count, ctypes.byref(o) if o is not None else None,
                                     ctypes.byref(info))
    _raise(st, "conv3d_bf16_describe")
    return info.as_dict()


# ------------------------------------------------------------------------------- quantiser
CONV3D_SRC_F32 = 1
CONV3D_SRC_BF16 = 2


def _src_type(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return CONV3D_SRC_F32
    if t.dtype == torch.bfloat16:
        return CONV3D_SRC_BF16
    raise ValueError(f"the quantiser takes fp32 or bfloat16 values, not {t.dtype}")


def conv3d_fp8_quantize_status(src, dst, scale_out, stream=None) -> int:
    """Quantise a CUDA fp32/bfloat16 tensor into uint8 e4m3 codes (dst) and a device scale."""
    return load().conv3d_fp8_quantize(_ptr(src), _src_type(src), src.numel(), _ptr(dst),
                                      _ptr(scale_out), _stream(stream))


def conv3d_fp8_quantize(src, dst, scale_out, stream=None) -> None:
    _raise(conv3d_fp8_quantize_status(src, dst, scale_out, stream), "conv3d_fp8_quantize")


def conv3d_fp8_run_quantize_x_status(plan, x_src, w, scale_w, y, stride, pad, scale_x_out=None,
                                     stream=None) -> int:
    return load().conv3d_fp8_run_quantize_x(plan, _ptr(x_src), _src_type(x_src), _ptr(w),
                                            _ptr(scale_w), _ptr(y), _int3(stride), _int3(pad),
                                            _ptr(scale_x_out), _stream(stream))


def conv3d_fp8_run_quantize_x(plan, x_src, w, scale_w, y, stride, pad, scale_x_out=None,
                              stream=None) -> None:
    _raise(conv3d_fp8_run_quantize_x_status(plan, x_src, w, scale_w, y, stride, pad, scale_x_out,
                                            stream), "conv3d_fp8_run_quantize_x")
