"""ctypes binding over libssm's C ABI (include/ssm.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their data pointers and torch's current CUDA stream are passed to
the C entry points, and every step of the computation runs in libssm's CUDA
kernels.  A missing or unloadable library raises SsmError; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssm.so")

SSM_OK = 0
SSM_ERR_INVALID_ARG = 1
SSM_ERR_UNSUPPORTED = 2
SSM_ERR_CUDA = 3
SSM_ERR_DEVICE_TIMEOUT = 4

DTYPE_F32 = 0
DTYPE_BF16 = 1

DISC_ZOH = 0
DISC_EULER = 1
_DISC = {"zoh": DISC_ZOH, "euler": DISC_EULER, DISC_ZOH: DISC_ZOH, DISC_EULER: DISC_EULER}

ALGO_AUTO = 0
ALGO_CHANNEL = 1
ALGO_CHUNK = 2
ALGO_CHANNEL_L1 = 3
ALGO_CHANNEL_L2 = 4
ALGO_CHANNEL_L4 = 5
ALGO_SEGMENTED = 6
ALGO_CHANNEL_MIXED = 7
_ALGOS = {"auto": ALGO_AUTO, "channel": ALGO_CHANNEL, "chunk": ALGO_CHUNK,
          "channel_l1": ALGO_CHANNEL_L1, "channel_l2": ALGO_CHANNEL_L2,
          "channel_l4": ALGO_CHANNEL_L4, "segmented": ALGO_SEGMENTED,
          "channel_mixed": ALGO_CHANNEL_MIXED}
_ALGOS.update({v: v for v in list(_ALGOS.values())})

# every symbol include/ssm.h declares
EXPORTED = ("ssm_scan_fwd_workspace_size", "ssm_scan_fwd_algo_workspace_size", "ssm_scan_fwd",
            "ssm_scan_fwd_algo", "ssm_scan_fwd_ex", "ssm_state_update_ex", "ssm_conv1d_fwd",
            "ssm_conv1d_update", "ssm_scan_bwd_workspace_size", "ssm_scan_bwd",
            "ssm_scan_bwd_ex_workspace_size", "ssm_scan_bwd_ex", "ssm_selftest_wait",
            "ssm_scan_fwd_host_workspace_size", "ssm_scan_fwd_host",
            "ssm_scan_fwd_noalloc", "ssm_state_update", "ssm_read_device_status",
            "ssm_status_string", "ssm_last_cuda_error", "ssm_last_plan", "ssm_version",
            "ssm_scan_ckpt_bytes", "ssm_scan_fwd_train", "ssm_scan_bwd_ckpt_workspace_size",
            "ssm_scan_bwd_ckpt")


class SsmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(what)


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int


def library(path: Optional[str] = None):
    """Load libssm.so (building it first if the sources are newer)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if path is None:
            from . import build as _build
            if not _build.up_to_date():
                try:
                    _build.build()
                except Exception as e:  # noqa: BLE001
                    if not os.path.exists(p):
                        raise SsmError(SSM_ERR_CUDA, f"libssm.so is not built and building it "
                                                     f"failed: {e}") from e
        if not os.path.exists(p):
            raise SsmError(SSM_ERR_CUDA, f"libssm.so not found at {p}")
        lib = ctypes.CDLL(p)
        lib.ssm_scan_fwd_workspace_size.restype = ctypes.c_size_t
        lib.ssm_scan_fwd_workspace_size.argtypes = [_i64, _i64, _i64, _i64]
        lib.ssm_scan_fwd_algo_workspace_size.restype = ctypes.c_size_t
        lib.ssm_scan_fwd_algo_workspace_size.argtypes = [_i64, _i64, _i64, _i64, _int]
        scan_args = [_i64, _i64, _i64, _i64, _int, _vp, _vp, _vp, _int, _vp, _vp, _vp, _vp, _vp,
                     _vp, _vp, _vp, _vp, ctypes.c_size_t]
        lib.ssm_scan_fwd.restype = _int
        lib.ssm_scan_fwd.argtypes = scan_args + [_vp]
        lib.ssm_scan_fwd_algo.restype = _int
        lib.ssm_scan_fwd_algo.argtypes = scan_args + [_int, _vp]
        lib.ssm_scan_fwd_noalloc.restype = _int
        lib.ssm_scan_fwd_noalloc.argtypes = scan_args[:17] + [_vp]
        lib.ssm_scan_fwd_ex.restype = _int
        lib.ssm_scan_fwd_ex.argtypes = scan_args + [_int, _int, _vp]
        lib.ssm_scan_ckpt_bytes.restype = ctypes.c_size_t
        lib.ssm_scan_ckpt_bytes.argtypes = [_i64, _i64, _i64, _i64]
        lib.ssm_scan_fwd_train.restype = _int
        lib.ssm_scan_fwd_train.argtypes = (scan_args[:17] + [_vp, ctypes.c_size_t]
                                           + scan_args[17:] + [_int, _int, _vp])
        lib.ssm_state_update.restype = _int
        lib.ssm_state_update.argtypes = [_i64, _i64, _i64, _int, _vp, _vp, _vp, _vp, _int, _vp,
                                         _vp, _vp, _vp, _vp, _vp, _vp]
        lib.ssm_state_update_ex.restype = _int
        lib.ssm_state_update_ex.argtypes = [_i64, _i64, _i64, _int, _vp, _vp, _vp, _vp, _int,
                                            _vp, _vp, _vp, _vp, _vp, _vp, _int, _vp]
        lib.ssm_conv1d_fwd.restype = _int
        lib.ssm_conv1d_fwd.argtypes = [_i64, _i64, _i64, _i64, _int, _vp, _vp, _vp, _vp, _int,
                                       _vp, _vp, _vp]
        lib.ssm_conv1d_update.restype = _int
        lib.ssm_conv1d_update.argtypes = [_i64, _i64, _i64, _int, _vp, _vp, _vp, _vp, _int, _vp,
                                          _vp]
        lib.ssm_scan_bwd_workspace_size.restype = ctypes.c_size_t
        lib.ssm_scan_bwd_workspace_size.argtypes = [_i64, _i64, _i64, _i64]
        lib.ssm_scan_bwd.restype = _int
        lib.ssm_scan_bwd.argtypes = ([_i64, _i64, _i64, _i64, _int, _vp, _vp, _vp, _int]
                                     + [_vp] * 18 + [ctypes.c_size_t, _int, _vp])
        lib.ssm_scan_bwd_ex_workspace_size.restype = ctypes.c_size_t
        lib.ssm_scan_bwd_ex_workspace_size.argtypes = [_i64, _i64, _i64, _i64, _int]
        lib.ssm_scan_bwd_ex.restype = _int
        lib.ssm_scan_bwd_ex.argtypes = ([_i64, _i64, _i64, _i64, _int, _vp, _vp, _vp, _int]
                                        + [_vp] * 18 + [ctypes.c_size_t, _int, _int, _vp])
        lib.ssm_scan_bwd_ckpt_workspace_size.restype = ctypes.c_size_t
        lib.ssm_scan_bwd_ckpt_workspace_size.argtypes = [_i64, _i64, _i64, _i64, _int]
        lib.ssm_scan_bwd_ckpt.restype = _int
        lib.ssm_scan_bwd_ckpt.argtypes = ([_i64, _i64, _i64, _i64, _int, _vp, _vp, _vp, _int]
                                          + [_vp] * 19 + [ctypes.c_size_t, _int, _int, _vp])
        lib.ssm_scan_fwd_host_workspace_size.restype = ctypes.c_size_t
        lib.ssm_scan_fwd_host_workspace_size.argtypes = [_i64, _i64, _i64, _i64, _int, _int,
                                                         _int, _int, _int]
        lib.ssm_scan_fwd_host.restype = _int
        lib.ssm_scan_fwd_host.argtypes = ([_i64, _i64, _i64, _i64, _int, _vp, _vp, _vp, _int]
                                          + [_vp] * 9 + [ctypes.c_size_t, _int, _int])
        lib.ssm_selftest_wait.restype = _int
        lib.ssm_selftest_wait.argtypes = [_vp, ctypes.c_size_t, _i64, _int, _vp]
        lib.ssm_read_device_status.restype = _int
        lib.ssm_read_device_status.argtypes = [_vp, _vp]
        lib.ssm_status_string.restype = ctypes.c_char_p
        lib.ssm_status_string.argtypes = [_int]
        lib.ssm_last_cuda_error.restype = ctypes.c_char_p
        lib.ssm_last_cuda_error.argtypes = []
        lib.ssm_last_plan.restype = ctypes.c_char_p
        lib.ssm_last_plan.argtypes = []
        lib.ssm_version.restype = _int
        lib.ssm_version.argtypes = []
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return library().ssm_status_string(int(status)).decode()


def last_plan() -> str:
    """The kernels the last scan-forward call on this thread launched (ssm_last_plan)."""
    return library().ssm_last_plan().decode()


def _check(status: int, what: str):
    if status != SSM_OK:
        lib = library()
        msg = f"{what}: {status_string(status)}"
        if status == SSM_ERR_CUDA:
            msg += f" ({lib.ssm_last_cuda_error().decode()})"
        raise SsmError(status, msg)


def _io_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise SsmError(SSM_ERR_UNSUPPORTED, f"io dtype must be float32 or bfloat16, got {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: Optional[torch.Tensor], name: str, shape, dtype, device, optional=False):
    if t is None:
        if optional:
            return
        raise SsmError(SSM_ERR_INVALID_ARG, f"{name} is required")
    if t.device != device:
        raise SsmError(SSM_ERR_INVALID_ARG, f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise SsmError(SSM_ERR_INVALID_ARG, f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise SsmError(SSM_ERR_INVALID_ARG, f"{name} has shape {tuple(t.shape)}, expected "
                                            f"{tuple(shape)}")
    if not t.is_contiguous():
        raise SsmError(SSM_ERR_INVALID_ARG, f"{name} must be contiguous")


_ws_cache = {}


def scan_fwd_workspace_size(batch: int, dim: int, dstate: int, seqlen: int) -> int:
    return int(library().ssm_scan_fwd_workspace_size(batch, dim, dstate, seqlen))


def _workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    """The scan workspace of a device: one buffer per device, grown to the largest
    size asked for so far, so that its status words are the ones the last scan on
    that device wrote (zero-filled when allocated)."""
    key = device.index
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True, h0=None,
             return_last_state=False, algo="auto", out=None, workspace=None,
             discretization="zoh", ckpt=None):
    """Selective-scan forward on torch CUDA tensors.

    u, delta, z, out: [batch, dim, seqlen] (float32 or bfloat16); B, C: [batch, dstate, seqlen]
    (same dtype); A: [dim, dstate] float32; D, delta_bias: [dim] float32; h0: [batch, dim,
    dstate] float32.  Returns y (and h_last [batch, dim, dstate] float32 when asked).
    discretization: "zoh" (default) or "euler" (input term dt * B).
    ckpt (training forward, ssm_scan_fwd_train): a float32 tensor [ceil(seqlen / 8), batch,
    dim, dstate] that receives the state entering every block of 8 positions, for
    scan_bwd(..., ckpt=...)."""
    if not isinstance(u, torch.Tensor) or not u.is_cuda:
        raise SsmError(SSM_ERR_INVALID_ARG, "u must be a CUDA tensor")
    if u.dim() != 3:
        raise SsmError(SSM_ERR_INVALID_ARG, "u must be [batch, dim, seqlen]")
    batch, dim, seqlen = u.shape
    dstate = A.shape[-1]
    dev = u.device
    io = _io_dtype(u)
    _need(u, "u", (batch, dim, seqlen), u.dtype, dev)
    _need(delta, "delta", (batch, dim, seqlen), u.dtype, dev)
    _need(z, "z", (batch, dim, seqlen), u.dtype, dev, optional=True)
    _need(B, "B", (batch, dstate, seqlen), u.dtype, dev)
    _need(C, "C", (batch, dstate, seqlen), u.dtype, dev)
    _need(A, "A", (dim, dstate), torch.float32, dev)
    _need(D, "D", (dim,), torch.float32, dev, optional=True)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev, optional=True)
    _need(h0, "h0", (batch, dim, dstate), torch.float32, dev, optional=True)
    y = torch.empty_like(u) if out is None else out
    _need(y, "out", (batch, dim, seqlen), u.dtype, dev)
    h_last = (torch.empty((batch, dim, dstate), dtype=torch.float32, device=dev)
              if return_last_state else None)
    lib = library()
    nbytes = int(lib.ssm_scan_fwd_algo_workspace_size(batch, dim, dstate, seqlen, _ALGOS[algo]))
    ws = _workspace(dev, nbytes) if workspace is None else workspace
    stream = torch.cuda.current_stream(dev).cuda_stream
    if ckpt is not None:
        _need(ckpt, "ckpt", ((seqlen + 7) // 8, batch, dim, dstate), torch.float32, dev)
        with torch.cuda.device(dev):
            st = lib.ssm_scan_fwd_train(batch, dim, dstate, seqlen, io, _ptr(u), _ptr(delta),
                                        _ptr(delta_bias), int(bool(delta_softplus)), _ptr(A),
                                        _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(h0),
                                        _ptr(h_last), _ptr(y), _ptr(ckpt),
                                        ckpt.numel() * 4, _ptr(ws), ws.numel(),
                                        _DISC[discretization], _ALGOS[algo],
                                        ctypes.c_void_p(stream))
        _check(st, "ssm_scan_fwd_train")
        return (y, h_last) if return_last_state else y
    with torch.cuda.device(dev):
        st = lib.ssm_scan_fwd_ex(batch, dim, dstate, seqlen, io, _ptr(u), _ptr(delta),
                                 _ptr(delta_bias), int(bool(delta_softplus)), _ptr(A), _ptr(B),
                                 _ptr(C), _ptr(D), _ptr(z), _ptr(h0), _ptr(h_last), _ptr(y),
                                 _ptr(ws), ws.numel(), _DISC[discretization], _ALGOS[algo],
                                 ctypes.c_void_p(stream))
    _check(st, "ssm_scan_fwd")
    return (y, h_last) if return_last_state else y


def ckpt_shape(batch: int, dim: int, dstate: int, seqlen: int):
    """Shape of the training forward's checkpoint tensor (float32)."""
    return ((seqlen + 7) // 8, batch, dim, dstate)


_bwd_ws_cache = {}


def scan_bwd_workspace_size(batch: int, dim: int, dstate: int, seqlen: int) -> int:
    return int(library().ssm_scan_bwd_workspace_size(batch, dim, dstate, seqlen))


def scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, delta_softplus=True,
             h0=None, dh_last=None, want_dh0=True, discretization="zoh", workspace=None,
             segments=0, ckpt=None):
    """Gradient of scan_fwd for the upstream gradient dy [batch, dim, seqlen] (and
    dh_last [batch, dim, dstate] float32 for the final state).  Takes the forward's
    inputs as passed to scan_fwd.  Returns a dict: du, ddelta, dz (io dtype,
    [batch, dim, seqlen]); dB, dC (io dtype, [batch, dstate, seqlen]); dA [dim, dstate],
    dD [dim] (when D), ddelta_bias [dim] (when delta_bias), dh0 [batch, dim, dstate]
    (when want_dh0), all float32.  segments: split of the sequence (0: the
    library's choice).  ckpt: the training forward's checkpoints (scan_fwd(...,
    ckpt=...)) for the same inputs; the gradient then runs no forward pass of its own
    (ssm_scan_bwd_ckpt)."""
    if not isinstance(u, torch.Tensor) or not u.is_cuda:
        raise SsmError(SSM_ERR_INVALID_ARG, "u must be a CUDA tensor")
    if u.dim() != 3:
        raise SsmError(SSM_ERR_INVALID_ARG, "u must be [batch, dim, seqlen]")
    batch, dim, seqlen = u.shape
    dstate = A.shape[-1]
    dev = u.device
    io = _io_dtype(u)
    for t, name, shape in ((delta, "delta", (batch, dim, seqlen)), (dy, "dy", (batch, dim, seqlen)),
                           (B, "B", (batch, dstate, seqlen)), (C, "C", (batch, dstate, seqlen))):
        _need(t, name, shape, u.dtype, dev)
    _need(z, "z", (batch, dim, seqlen), u.dtype, dev, optional=True)
    _need(A, "A", (dim, dstate), torch.float32, dev)
    _need(D, "D", (dim,), torch.float32, dev, optional=True)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev, optional=True)
    _need(h0, "h0", (batch, dim, dstate), torch.float32, dev, optional=True)
    _need(dh_last, "dh_last", (batch, dim, dstate), torch.float32, dev, optional=True)
    f32 = dict(dtype=torch.float32, device=dev)
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
         "dz": torch.empty_like(u) if z is not None else None,
         "dB": torch.empty_like(B), "dC": torch.empty_like(C),
         "dA": torch.empty((dim, dstate), **f32),
         "dD": torch.empty((dim,), **f32) if D is not None else None,
         "ddelta_bias": torch.empty((dim,), **f32) if delta_bias is not None else None,
         "dh0": torch.empty((batch, dim, dstate), **f32) if want_dh0 else None}
    lib = library()
    if ckpt is not None:
        _need(ckpt, "ckpt", ((seqlen + 7) // 8, batch, dim, dstate), torch.float32, dev)
    with torch.cuda.device(dev):
        size_fn = (lib.ssm_scan_bwd_ckpt_workspace_size if ckpt is not None
                   else lib.ssm_scan_bwd_ex_workspace_size)
        nbytes = int(size_fn(batch, dim, dstate, seqlen, int(segments)))
    if workspace is None:
        ws = _bwd_ws_cache.get(dev.index)
        if ws is None or ws.numel() < nbytes:
            ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
            _bwd_ws_cache[dev.index] = ws
    else:
        ws = workspace
    stream = torch.cuda.current_stream(dev).cuda_stream
    grads = (_ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
             _ptr(g["dD"]), _ptr(g["dz"]), _ptr(g["ddelta_bias"]), _ptr(g["dh0"]))
    with torch.cuda.device(dev):
        if ckpt is not None:
            st = lib.ssm_scan_bwd_ckpt(batch, dim, dstate, seqlen, io, _ptr(u), _ptr(delta),
                                       _ptr(delta_bias), int(bool(delta_softplus)), _ptr(A),
                                       _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(h0),
                                       _ptr(ckpt), _ptr(dy), _ptr(dh_last), *grads, _ptr(ws),
                                       ws.numel(), _DISC[discretization], int(segments),
                                       ctypes.c_void_p(stream))
        else:
            st = lib.ssm_scan_bwd_ex(batch, dim, dstate, seqlen, io, _ptr(u), _ptr(delta),
                                     _ptr(delta_bias), int(bool(delta_softplus)), _ptr(A),
                                     _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(h0), _ptr(dy),
                                     _ptr(dh_last), *grads, _ptr(ws), ws.numel(),
                                     _DISC[discretization], int(segments),
                                     ctypes.c_void_p(stream))
    _check(st, "ssm_scan_bwd_ckpt" if ckpt is not None else "ssm_scan_bwd")
    return g


_host_ws_cache = {}


def scan_fwd_host(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                  h0=None, return_last_state=False, out=None, algo="auto",
                  discretization="zoh", device=None):
    """The scan on HOST tensors (CPU, ideally pinned): the library streams the batch
    through device staging buffers in pieces, overlapping copy-in, scan and
    copy-out, and returns once the outputs are in host memory.  Shapes and dtypes as
    scan_fwd; A, D, delta_bias, h0 float32 host tensors too.  Returns y (host; `out`
    if given) and h_last (host) when asked."""
    for name, t in (("u", u), ("delta", delta), ("A", A), ("B", B), ("C", C)):
        if not isinstance(t, torch.Tensor) or t.is_cuda:
            raise SsmError(SSM_ERR_INVALID_ARG, f"{name} must be a host (CPU) tensor")
    batch, dim, seqlen = u.shape
    dstate = A.shape[-1]
    io = _io_dtype(u)
    cpu = torch.device("cpu")
    _need(delta, "delta", (batch, dim, seqlen), u.dtype, cpu)
    _need(z, "z", (batch, dim, seqlen), u.dtype, cpu, optional=True)
    _need(B, "B", (batch, dstate, seqlen), u.dtype, cpu)
    _need(C, "C", (batch, dstate, seqlen), u.dtype, cpu)
    _need(A, "A", (dim, dstate), torch.float32, cpu)
    _need(D, "D", (dim,), torch.float32, cpu, optional=True)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, cpu, optional=True)
    _need(h0, "h0", (batch, dim, dstate), torch.float32, cpu, optional=True)
    y = torch.empty_like(u) if out is None else out
    _need(y, "out", (batch, dim, seqlen), u.dtype, cpu)
    h_last = torch.empty((batch, dim, dstate), dtype=torch.float32) if return_last_state else None
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    lib = library()
    with torch.cuda.device(dev):
        nbytes = int(lib.ssm_scan_fwd_host_workspace_size(
            batch, dim, dstate, seqlen, io, int(z is not None), int(h0 is not None),
            int(return_last_state), _ALGOS[algo]))
        ws = _host_ws_cache.get(dev.index)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
            _host_ws_cache[dev.index] = ws
        st = lib.ssm_scan_fwd_host(batch, dim, dstate, seqlen, io, _ptr(u), _ptr(delta),
                                   _ptr(delta_bias), int(bool(delta_softplus)), _ptr(A), _ptr(B),
                                   _ptr(C), _ptr(D), _ptr(z), _ptr(h0), _ptr(h_last), _ptr(y),
                                   _ptr(ws), ws.numel(), _DISC[discretization], _ALGOS[algo])
    _check(st, "ssm_scan_fwd_host")
    return (y, h_last) if return_last_state else y


def selftest_wait(limit_ns: int, arrive: bool, device=None) -> int:
    """Run the device-side timeout check on a fresh status buffer of its own and
    return its status: SSM_OK when `arrive`, SSM_ERR_DEVICE_TIMEOUT otherwise."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    lib = library()
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        _check(lib.ssm_selftest_wait(_ptr(ws), ws.numel(), int(limit_ns), int(bool(arrive)),
                                     ctypes.c_void_p(stream)), "ssm_selftest_wait")
        return int(lib.ssm_read_device_status(_ptr(ws), ctypes.c_void_p(stream)))


def read_device_status(workspace: Optional[torch.Tensor] = None, device=None) -> int:
    """Synchronise the current stream and return the status recorded in a scan workspace."""
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        workspace = _workspace(dev, 256)
    stream = torch.cuda.current_stream(workspace.device).cuda_stream
    return int(library().ssm_read_device_status(_ptr(workspace), ctypes.c_void_p(stream)))


def state_update(h, u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 out=None, discretization="zoh"):
    """One decode step; h [batch, dim, dstate] float32 is updated in place.

    u, delta, z, out: [batch, dim]; B, C: [batch, dstate]; A: [dim, dstate] float32.
    Returns y [batch, dim]."""
    if not isinstance(h, torch.Tensor) or not h.is_cuda:
        raise SsmError(SSM_ERR_INVALID_ARG, "h must be a CUDA tensor")
    batch, dim, dstate = h.shape
    dev = h.device
    io = _io_dtype(u)
    _need(h, "h", (batch, dim, dstate), torch.float32, dev)
    _need(u, "u", (batch, dim), u.dtype, dev)
    _need(delta, "delta", (batch, dim), u.dtype, dev)
    _need(z, "z", (batch, dim), u.dtype, dev, optional=True)
    _need(B, "B", (batch, dstate), u.dtype, dev)
    _need(C, "C", (batch, dstate), u.dtype, dev)
    _need(A, "A", (dim, dstate), torch.float32, dev)
    _need(D, "D", (dim,), torch.float32, dev, optional=True)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev, optional=True)
    y = torch.empty_like(u) if out is None else out
    _need(y, "out", (batch, dim), u.dtype, dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        st = library().ssm_state_update_ex(batch, dim, dstate, io, _ptr(h), _ptr(u),
                                           _ptr(delta), _ptr(delta_bias),
                                           int(bool(delta_softplus)), _ptr(A), _ptr(B), _ptr(C),
                                           _ptr(D), _ptr(z), _ptr(y), _DISC[discretization],
                                           ctypes.c_void_p(stream))
    _check(st, "ssm_state_update")
    return y


def conv1d_fwd(x, weight, bias=None, conv_state=None, apply_silu=True, return_state=False,
               out=None):
    """Causal depthwise convolution over time (+ silu) on torch CUDA tensors.

    x, out: [batch, dim, seqlen] (float32 or bfloat16); weight [dim, width] float32;
    bias [dim] float32; conv_state [batch, dim, width - 1] (x's dtype): the inputs
    before position 0.  Returns out (and the last width - 1 inputs when asked)."""
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dim() != 3:
        raise SsmError(SSM_ERR_INVALID_ARG, "x must be a [batch, dim, seqlen] CUDA tensor")
    batch, dim, seqlen = x.shape
    width = weight.shape[-1]
    dev = x.device
    io = _io_dtype(x)
    _need(x, "x", (batch, dim, seqlen), x.dtype, dev)
    _need(weight, "weight", (dim, width), torch.float32, dev)
    _need(bias, "bias", (dim,), torch.float32, dev, optional=True)
    _need(conv_state, "conv_state", (batch, dim, width - 1), x.dtype, dev, optional=True)
    y = torch.empty_like(x) if out is None else out
    _need(y, "out", (batch, dim, seqlen), x.dtype, dev)
    st_out = torch.empty((batch, dim, width - 1), dtype=x.dtype, device=dev) \
        if return_state else None
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        st = library().ssm_conv1d_fwd(batch, dim, seqlen, width, io, _ptr(x), _ptr(weight),
                                      _ptr(bias), _ptr(conv_state), int(bool(apply_silu)),
                                      _ptr(y), _ptr(st_out), ctypes.c_void_p(stream))
    _check(st, "ssm_conv1d_fwd")
    return (y, st_out) if return_state else y


def conv1d_update(conv_state, x, weight, bias=None, apply_silu=True, out=None):
    """One decode position of conv1d_fwd; conv_state [batch, dim, width - 1] is
    updated in place.  x, out: [batch, dim].  Returns out."""
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dim() != 2:
        raise SsmError(SSM_ERR_INVALID_ARG, "x must be a [batch, dim] CUDA tensor")
    batch, dim = x.shape
    width = weight.shape[-1]
    dev = x.device
    io = _io_dtype(x)
    _need(weight, "weight", (dim, width), torch.float32, dev)
    _need(bias, "bias", (dim,), torch.float32, dev, optional=True)
    _need(conv_state, "conv_state", (batch, dim, width - 1), x.dtype, dev)
    y = torch.empty_like(x) if out is None else out
    _need(y, "out", (batch, dim), x.dtype, dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        st = library().ssm_conv1d_update(batch, dim, width, io, _ptr(conv_state), _ptr(x),
                                         _ptr(weight), _ptr(bias), int(bool(apply_silu)),
                                         _ptr(y), ctypes.c_void_p(stream))
    _check(st, "ssm_conv1d_update")
    return y
