"""ctypes binding of ``liblrscan.so`` (the C ABI in ``include/lrscan.h``).

Two layers, both argument marshalling only -- every step of every scan runs
in the library's CUDA kernels:

* ``lr_*`` functions with the C names and signatures (pointers as ints);
* torch conveniences (:func:`selective_scan`, :func:`rglru_scan`,
  :func:`hgrn2`) that check shapes and dtypes, allocate outputs and the
  workspace with torch, pass the current CUDA stream and raise
  :class:`LrError` on a non-zero status.  Given host tensors they copy the
  inputs to the current CUDA device and the outputs back (the end-to-end
  path); given device tensors they stay on the device.

There is no fallback: if the library is missing this module raises at import.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import build as _build

LR_F32, LR_BF16 = 0, 1
LR_OK = 0
LR_ERR_INVALID_ARG, LR_ERR_UNSUPPORTED, LR_ERR_MISALIGNED = -1, -2, -3
LR_ERR_WORKSPACE, LR_ERR_CUDA, LR_ERR_TIMEOUT, LR_ERR_RANGE = -4, -5, -6, -7

_IO = {torch.float32: LR_F32, torch.bfloat16: LR_BF16}

# (name, restype, argtypes) of every exported C symbol
_P, _I64, _F, _I, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "lr_status_string": (ctypes.c_char_p, [_I]),
    "lr_version": (_I, []),
    "lr_check_status": (_I, [_P, _P]),
    "lr_set_split_override": (_I, [_I]),
    "lr_test_withhold_split": (_I, [_I, _I]),
    "lr_set_host_chunk_steps": (_I64, [_I64]),
    "lr_set_selective_warmup": (_I64, [_I64]),
    "lr_selective_scan_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I]),
    "lr_selective_scan_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _I64, _I64, _I64, _I64, _I, _I, _P, _SZ, _P]),
    "lr_rglru_scan_workspace_size": (_SZ, [_I64, _I64, _I64, _I]),
    "lr_rglru_scan_fwd": (_I, [_P, _P, _P, _P, _F, _P, _P, _P,
                               _I64, _I64, _I64, _I, _P, _SZ, _P]),
    "lr_rglru_scan_fwd_noalloc": (_I, [_P, _P, _P, _P, _F, _P, _P, _P,
                                       _I64, _I64, _I64, _I, _P]),
    "lr_hgrn2_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I64, _I]),
    "lr_hgrn2_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                          _I64, _I64, _I, _P, _SZ, _P]),
    "lr_rglru_scan_preact_fwd": (_I, [_P, _P, _P, _P, _F, _P, _P, _P,
                                      _I64, _I64, _I64, _I, _P, _SZ, _P]),
    "lr_hgrn2_preact_fwd": (_I, [_P, _P, _P, _P, _F, _P, _P, _P, _I64, _I64, _I64, _I64,
                                 _I64, _I64, _I, _P, _SZ, _P]),
    "lr_minmax_scan_workspace_size": (_SZ, [_I64, _I64, _I64, _I]),
    "lr_minmax_scan_fwd": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _P, _SZ, _P]),
    "lr_selective_scan_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                    _I64, _I64, _I64, _I, _I, _P]),
    "lr_rglru_scan_step": (_I, [_P, _P, _P, _P, _F, _P, _P, _P, _I64, _I64, _I, _P]),
    "lr_hgrn2_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I, _P]),
    "lr_minmax_scan_step": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I, _P]),
    "lr_selective_scan_fwd_host_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I]),
    "lr_selective_scan_fwd_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        _I64, _I64, _I64, _I64, _I, _I, _P, _SZ, _P]),
    "lr_rglru_scan_fwd_host_workspace_size": (_SZ, [_I64, _I64, _I64, _I]),
    "lr_rglru_scan_fwd_host": (_I, [_P, _P, _P, _P, _F, _P, _P, _P,
                                    _I64, _I64, _I64, _I, _P, _SZ, _P]),
    "lr_hgrn2_fwd_host_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I64, _I]),
    "lr_hgrn2_fwd_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                               _I64, _I64, _I, _P, _SZ, _P]),
    "lr_minmax_scan_fwd_host_workspace_size": (_SZ, [_I64, _I64, _I64, _I]),
    "lr_minmax_scan_fwd_host": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _P, _SZ, _P]),
    "lr_selective_scan_fwd_host_async": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                              _I64, _I64, _I64, _I64, _I, _I, _P, _SZ, _P]),
    "lr_rglru_scan_fwd_host_async": (_I, [_P, _P, _P, _P, _F, _P, _P, _P,
                                          _I64, _I64, _I64, _I, _P, _SZ, _P]),
    "lr_hgrn2_fwd_host_async": (_I, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                     _I64, _I64, _I, _P, _SZ, _P]),
    "lr_minmax_scan_fwd_host_async": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _P, _SZ, _P]),
    "lr_host_sync": (_I, []),
}


def _load():
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with selective_state_space_chunked_gb300."
            "build.build() (nvcc, sm_103a). There is no CPU fallback.")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
LIB_PATH = _build.LIB_PATH


class LrError(RuntimeError):
    """A non-zero lrscan status."""

    def __init__(self, code: int, where: str = ""):
        self.code = int(code)
        msg = lr_status_string(code)
        super().__init__(f"{where}: {msg}" if where else msg)


# ---------------------------------------------------------------- C names
def lr_status_string(code: int) -> str:
    return _lib.lr_status_string(int(code)).decode()


def lr_version() -> int:
    return int(_lib.lr_version())


def lr_check_status(workspace, stream: int = 0) -> int:
    """Status of the latest call that used ``workspace`` (a device pointer;
    None = the built-in scratch of lr_rglru_scan_fwd_noalloc); synchronises
    ``stream`` and resets the status."""
    return int(_lib.lr_check_status(workspace or None, stream or None))


def lr_set_split_override(splits: int) -> int:
    return int(_lib.lr_set_split_override(int(splits)))


def lr_set_host_chunk_steps(steps: int) -> int:
    """Chunk length of the host-buffer path (0 = automatic); returns the previous."""
    return int(_lib.lr_set_host_chunk_steps(int(steps)))


def lr_set_selective_warmup(max_steps: int) -> int:
    """Longest warm-up of the selective scan's pieces in steps (0 = carries
    by look-back only, negative = automatic: 2048 for bf16 I/O, 0 for fp32);
    returns the previous setting (-1 = automatic)."""
    return int(_lib.lr_set_selective_warmup(int(max_steps)))


def lr_test_withhold_split(split: int, timeout_ms: int = 1000) -> int:
    return int(_lib.lr_test_withhold_split(int(split), int(timeout_ms)))


def lr_selective_scan_workspace_size(B, L, D, N, io) -> int:
    return int(_lib.lr_selective_scan_workspace_size(B, L, D, N, io))


def lr_selective_scan_fwd(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final,
                          B, L, D, N, io, dt_softplus, workspace, ws_bytes,
                          stream) -> int:
    return int(_lib.lr_selective_scan_fwd(x, dt, z, Bm, Cm, A_log, Dskip, h0, y,
                                          h_final, B, L, D, N, io, dt_softplus,
                                          workspace, ws_bytes, stream))


def lr_rglru_scan_workspace_size(B, L, D, io) -> int:
    return int(_lib.lr_rglru_scan_workspace_size(B, L, D, io))


def lr_rglru_scan_fwd(x, r, i, a_log, c, h0, y, h_final, B, L, D, io,
                      workspace, ws_bytes, stream) -> int:
    return int(_lib.lr_rglru_scan_fwd(x, r, i, a_log, c, h0, y, h_final, B, L, D,
                                      io, workspace, ws_bytes, stream))


def lr_rglru_scan_fwd_noalloc(x, r, i, a_log, c, h0, y, h_final, B, L, D, io,
                              stream) -> int:
    """RG-LRU scan using the library's built-in scratch (no workspace)."""
    return int(_lib.lr_rglru_scan_fwd_noalloc(x, r, i, a_log, c, h0, y, h_final, B, L,
                                              D, io, stream))


def lr_hgrn2_workspace_size(B, L, H, dk, dv, io) -> int:
    return int(_lib.lr_hgrn2_workspace_size(B, L, H, dk, dv, io))


def lr_hgrn2_fwd(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, chunk, io,
                 workspace, ws_bytes, stream) -> int:
    return int(_lib.lr_hgrn2_fwd(q, k, v, g, S0, o, S_final, B, L, H, dk, dv,
                                 chunk, io, workspace, ws_bytes, stream))


def lr_rglru_scan_preact_fwd(x, r_pre, i_pre, a_log, c, h0, y, h_final, B, L, D, io,
                             workspace, ws_bytes, stream) -> int:
    return int(_lib.lr_rglru_scan_preact_fwd(x, r_pre, i_pre, a_log, c, h0, y, h_final, B, L, D,
                                             io, workspace, ws_bytes, stream))


def lr_hgrn2_preact_fwd(q, k, v, f, lb, S0, o, S_final, B, L, H, dk, dv, chunk, io,
                        workspace, ws_bytes, stream) -> int:
    return int(_lib.lr_hgrn2_preact_fwd(q, k, v, f, lb, S0, o, S_final, B, L, H, dk, dv, chunk,
                                        io, workspace, ws_bytes, stream))


def lr_minmax_scan_workspace_size(B, L, D, io) -> int:
    return int(_lib.lr_minmax_scan_workspace_size(B, L, D, io))


def lr_minmax_scan_fwd(r, s, x0, y, x_final, B, L, D, io, workspace, ws_bytes, stream) -> int:
    return int(_lib.lr_minmax_scan_fwd(r, s, x0, y, x_final, B, L, D, io, workspace, ws_bytes,
                                       stream))


def lr_selective_scan_step(x, dt, z, Bm, Cm, A_log, Dskip, h_in, h_out, y, B, D, N,
                           io, dt_softplus, stream) -> int:
    return int(_lib.lr_selective_scan_step(x, dt, z, Bm, Cm, A_log, Dskip, h_in, h_out,
                                           y, B, D, N, io, dt_softplus, stream))


def lr_rglru_scan_step(x, r, i, a_log, c, h_in, h_out, y, B, D, io, stream) -> int:
    return int(_lib.lr_rglru_scan_step(x, r, i, a_log, c, h_in, h_out, y, B, D, io,
                                       stream))


def lr_minmax_scan_step(r, s, x_in, x_out, y, B, D, io, stream) -> int:
    return int(_lib.lr_minmax_scan_step(r, s, x_in, x_out, y, B, D, io, stream))


def lr_hgrn2_step(q, k, v, g, S_in, S_out, o, B, H, dk, dv, io, stream) -> int:
    return int(_lib.lr_hgrn2_step(q, k, v, g, S_in, S_out, o, B, H, dk, dv, io,
                                  stream))


def lr_selective_scan_fwd_host_workspace_size(B, L, D, N, io) -> int:
    return int(_lib.lr_selective_scan_fwd_host_workspace_size(B, L, D, N, io))


def lr_selective_scan_fwd_host(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final, B, L, D, N, io,
                               dt_softplus, workspace, ws_bytes, stream) -> int:
    """Selective scan on host buffers (device workspace only)."""
    return int(_lib.lr_selective_scan_fwd_host(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final,
                                               B, L, D, N, io, dt_softplus, workspace, ws_bytes,
                                               stream))


def lr_rglru_scan_fwd_host_workspace_size(B, L, D, io) -> int:
    return int(_lib.lr_rglru_scan_fwd_host_workspace_size(B, L, D, io))


def lr_rglru_scan_fwd_host(x, r, i, a_log, c, h0, y, h_final, B, L, D, io, workspace, ws_bytes,
                           stream) -> int:
    """RG-LRU scan on host buffers (device workspace only)."""
    return int(_lib.lr_rglru_scan_fwd_host(x, r, i, a_log, c, h0, y, h_final, B, L, D, io,
                                           workspace, ws_bytes, stream))


def lr_hgrn2_fwd_host_workspace_size(B, L, H, dk, dv, io) -> int:
    return int(_lib.lr_hgrn2_fwd_host_workspace_size(B, L, H, dk, dv, io))


def lr_hgrn2_fwd_host(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, chunk, io, workspace, ws_bytes,
                      stream) -> int:
    """HGRN2 on host buffers (device workspace only)."""
    return int(_lib.lr_hgrn2_fwd_host(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, chunk, io,
                                      workspace, ws_bytes, stream))


def lr_minmax_scan_fwd_host_workspace_size(B, L, D, io) -> int:
    return int(_lib.lr_minmax_scan_fwd_host_workspace_size(B, L, D, io))


def lr_minmax_scan_fwd_host(r, s, x0, y, x_final, B, L, D, io, workspace, ws_bytes, stream) -> int:
    """MinMax scan on host buffers (device workspace only)."""
    return int(_lib.lr_minmax_scan_fwd_host(r, s, x0, y, x_final, B, L, D, io, workspace, ws_bytes,
                                            stream))


def lr_selective_scan_fwd_host_async(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final, B, L, D, N, io,
                                     dt_softplus, workspace, ws_bytes, stream) -> int:
    """As lr_selective_scan_fwd_host, returning once the work is queued."""
    return int(_lib.lr_selective_scan_fwd_host_async(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final,
                                                     B, L, D, N, io, dt_softplus, workspace, ws_bytes,
                                                     stream))


def lr_rglru_scan_fwd_host_async(x, r, i, a_log, c, h0, y, h_final, B, L, D, io, workspace, ws_bytes,
                                 stream) -> int:
    """As lr_rglru_scan_fwd_host, returning once the work is queued."""
    return int(_lib.lr_rglru_scan_fwd_host_async(x, r, i, a_log, c, h0, y, h_final, B, L, D, io,
                                                 workspace, ws_bytes, stream))


def lr_hgrn2_fwd_host_async(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, chunk, io, workspace, ws_bytes,
                            stream) -> int:
    """As lr_hgrn2_fwd_host, returning once the work is queued."""
    return int(_lib.lr_hgrn2_fwd_host_async(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, chunk, io,
                                            workspace, ws_bytes, stream))


def lr_minmax_scan_fwd_host_async(r, s, x0, y, x_final, B, L, D, io, workspace, ws_bytes, stream) -> int:
    """As lr_minmax_scan_fwd_host, returning once the work is queued."""
    return int(_lib.lr_minmax_scan_fwd_host_async(r, s, x0, y, x_final, B, L, D, io, workspace, ws_bytes,
                                                  stream))


def lr_host_sync() -> int:
    """Waits for every host-buffer call queued on the current device."""
    return int(_lib.lr_host_sync())


# ------------------------------------------------------------ torch helpers
def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _dev(t: Optional[torch.Tensor], device) -> Optional[torch.Tensor]:
    if t is None:
        return None
    if t.device.type != "cuda":
        t = t.to(device, non_blocking=True)
    return t.contiguous()


def _check(rc: int, where: str):
    if rc != LR_OK:
        _tls.ws = None   # a call that failed on the host recorded no device status
        raise LrError(rc, where)


def _io_of(t: torch.Tensor) -> int:
    if t.dtype not in _IO:
        raise TypeError(f"unsupported I/O dtype {t.dtype}; use float32 or bfloat16")
    return _IO[t.dtype]


def _same(ref: torch.Tensor, *ts):
    for t in ts:
        if t is not None and t.dtype != ref.dtype:
            raise TypeError("all activation tensors must share one dtype")


# The workspace of this thread's latest call through the torch helpers: its
# first bytes hold that call's device-side status (see status()).
_tls = threading.local()


def last_workspace() -> Optional[torch.Tensor]:
    """Workspace tensor of this thread's latest call through a torch helper."""
    return getattr(_tls, "ws", None)


def _workspace(nbytes: int, device, given: Optional[torch.Tensor]):
    if nbytes == (1 << 64) - 1:
        raise LrError(LR_ERR_CUDA, "workspace size query")
    if nbytes == 0:
        _tls.ws = None
        return None, 0
    if given is not None:
        ws, n = given, given.numel() * given.element_size()
    else:
        ws, n = torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes
    _tls.ws = ws
    return ws, n


def _target_device(*ts):
    for t in ts:
        if t is not None and t.device.type == "cuda":
            return t.device
    return torch.device("cuda", torch.cuda.current_device())


def _back(out: torch.Tensor, host: bool) -> torch.Tensor:
    if not host:
        return out
    h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h.copy_(out, non_blocking=True)
    return h


def _outputs(out, specs, dev):
    """Device buffers the kernel writes, and the caller's host destinations.

    ``out`` is None or a tuple of tensors matching ``specs`` (shape, dtype):
    all on the GPU (the kernel writes them in place) or all on the host
    (results are copied into them; pinned memory keeps the copy
    asynchronous and avoids allocating a pinned buffer per call)."""
    if out is None:
        return [torch.empty(sh, dtype=dt, device=dev) for sh, dt in specs], None
    if len(out) != len(specs):
        raise ValueError(f"out must hold {len(specs)} tensors")
    for o, (sh, dt) in zip(out, specs):
        if tuple(o.shape) != tuple(sh) or o.dtype != dt or not o.is_contiguous():
            raise ValueError(f"out tensor {tuple(o.shape)} {o.dtype} does not match "
                             f"{tuple(sh)} {dt} (contiguous)")
    on_gpu = [o.device.type == "cuda" for o in out]
    if all(on_gpu):
        if any(o.device != dev for o in out):
            raise ValueError("out tensors must be on the inputs' GPU")
        return list(out), None
    if any(on_gpu):
        raise ValueError("out tensors must be all on the GPU or all on the host")
    return [torch.empty(sh, dtype=dt, device=dev) for sh, dt in specs], list(out)


# ---- host buffers: the library's chunked host path (lr_*_fwd_host)
_HOST_WS = {}


def _host_route(acts, out) -> bool:
    """True when every activation and every given result tensor is in host
    memory: the call then goes to the library's host-buffer entry point."""
    if any(t is not None and t.device.type == "cuda" for t in acts):
        return False
    return out is None or all(o.device.type != "cuda" for o in out)


def _h(t: Optional[torch.Tensor], dtype=None) -> Optional[torch.Tensor]:
    if t is None:
        return None
    if t.device.type == "cuda":
        t = t.cpu()
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous()


def _host_outputs(out, specs):
    """Host result tensors: the caller's, or new pinned ones."""
    if out is None:
        return [torch.empty(sh, dtype=dt, pin_memory=True) for sh, dt in specs]
    if len(out) != len(specs):
        raise ValueError(f"out must hold {len(specs)} tensors")
    for o, (sh, dt) in zip(out, specs):
        if tuple(o.shape) != tuple(sh) or o.dtype != dt or not o.is_contiguous():
            raise ValueError(f"out tensor {tuple(o.shape)} {o.dtype} does not match "
                             f"{tuple(sh)} {dt} (contiguous)")
    return list(out)


def _host_workspace(nbytes: int, given: Optional[torch.Tensor]):
    """Device staging for a host-buffer call: the caller's tensor, or one
    kept per device and grown as needed."""
    if nbytes == (1 << 64) - 1:
        raise LrError(LR_ERR_CUDA, "workspace size query")
    if nbytes == 0:
        return None, 0
    if given is not None:
        _tls.ws = given
        return given, given.numel() * given.element_size()
    dev = torch.cuda.current_device()
    ws = _HOST_WS.get(dev)
    if ws is None or ws.numel() < nbytes:
        _HOST_WS.pop(dev, None)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=torch.device("cuda", dev))
        _HOST_WS[dev] = ws
    _tls.ws = ws
    return ws, nbytes


# tensors that host-buffer calls queued with sync_host=False still read or
# write (inputs, results, workspaces), per device, until host_sync()
_ASYNC_KEEP = {}


def _async_workspace(nbytes: int, given: Optional[torch.Tensor]):
    """Device staging for a queued host-buffer call: the caller's tensor, or a
    new one (calls in flight must not share one)."""
    if nbytes == (1 << 64) - 1:
        raise LrError(LR_ERR_CUDA, "workspace size query")
    if nbytes == 0:
        return None, 0
    if given is not None:
        _tls.ws = given
        return given, given.numel() * given.element_size()
    ws = torch.empty(nbytes, dtype=torch.uint8, device=torch.device("cuda", torch.cuda.current_device()))
    _tls.ws = ws
    return ws, nbytes


def _host_entry(sync_fn, async_fn, nbytes, workspace, sync_host: bool, keep):
    """The host-buffer entry point and its workspace: synchronous, or queued
    (its tensors kept alive until host_sync())."""
    if sync_host:
        ws, wsb = _host_workspace(nbytes, workspace)
        return sync_fn, ws, wsb
    ws, wsb = _async_workspace(nbytes, workspace)
    _ASYNC_KEEP.setdefault(torch.cuda.current_device(), []).extend(
        [t for t in list(keep) + [ws] if t is not None])
    return async_fn, ws, wsb


def host_sync() -> None:
    """Waits for every host-buffer call queued with ``sync_host=False`` on the
    current device; their results are then in host memory (read each call's
    device-side status afterwards with ``status(workspace)``)."""
    _check(lr_host_sync(), "lr_host_sync")
    _ASYNC_KEEP.pop(torch.cuda.current_device(), None)


def _host_stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _finish(bufs, host_out, host: bool, dev, sync_host: bool):
    if host_out is not None:
        for dst, src in zip(host_out, bufs):
            dst.copy_(src, non_blocking=True)
        res = host_out
    else:
        res = [_back(b, host) for b in bufs]
    if (host or host_out is not None) and sync_host:
        torch.cuda.current_stream(dev).synchronize()
    return tuple(res)


def selective_scan(x, dt, Bm, Cm, A_log, z=None, Dskip=None, h0=None,
                   dt_softplus: bool = True, workspace=None, out=None,
                   sync_host: bool = True) -> Tuple[torch.Tensor, torch.Tensor]:
    """Selective SSM scan.  x, dt, z: (B, L, D); Bm, Cm: (B, L, 16), all one
    dtype (float32 or bfloat16); A_log: (D, 16) fp32; Dskip: (D,) fp32;
    h0: (B, D, 16) fp32.  Returns (y (B, L, D) in the I/O dtype, h_final
    (B, D, 16) fp32); ``out=(y, h_final)`` gives the result tensors (GPU or
    host).  Host inputs with host (or no) ``out`` run the library's
    host-buffer path (chunked, copies overlapping the scan; pinned memory
    keeps the copies asynchronous); ``workspace`` is then its device
    staging buffer.  With ``sync_host=False`` a host-buffer call returns once
    its work is queued, so consecutive calls overlap; ``host_sync()`` waits
    for it (each queued call without a ``workspace`` gets a new one)."""
    if _host_route((x, dt, z, Bm, Cm), out):
        x, dt, z, Bm, Cm = (_h(t) for t in (x, dt, z, Bm, Cm))
        A_log, Dskip, h0 = (_h(t, torch.float32) for t in (A_log, Dskip, h0))
        _same(x, dt, z, Bm, Cm)
        io = _io_of(x)
        B, L, D = x.shape
        N = Bm.shape[-1]
        y, hf = _host_outputs(out, [((B, L, D), x.dtype), ((B, D, N), torch.float32)])
        fn, ws, wsb = _host_entry(lr_selective_scan_fwd_host, lr_selective_scan_fwd_host_async,
                                  lr_selective_scan_fwd_host_workspace_size(B, L, D, N, io), workspace,
                                  sync_host, (x, dt, z, Bm, Cm, A_log, Dskip, h0, y, hf))
        _check(fn(_ptr(x), _ptr(dt), _ptr(z), _ptr(Bm), _ptr(Cm), _ptr(A_log), _ptr(Dskip), _ptr(h0),
                  _ptr(y), _ptr(hf), B, L, D, N, io, int(bool(dt_softplus)), _ptr(ws), wsb,
                  _host_stream()), fn.__name__)
        return y, hf
    host = x.device.type != "cuda"
    dev = _target_device(x)
    x, dt, z, Bm, Cm = (_dev(t, dev) for t in (x, dt, z, Bm, Cm))
    A_log, Dskip, h0 = (_dev(None if t is None else t.float(), dev) for t in (A_log, Dskip, h0))
    _same(x, dt, z, Bm, Cm)
    io = _io_of(x)
    B, L, D = x.shape
    N = Bm.shape[-1]
    (y, hf), host_out = _outputs(out, [((B, L, D), x.dtype), ((B, D, N), torch.float32)], dev)
    ws, wsb = _workspace(lr_selective_scan_workspace_size(B, L, D, N, io), dev, workspace)
    stream = torch.cuda.current_stream(dev).cuda_stream
    _check(lr_selective_scan_fwd(_ptr(x), _ptr(dt), _ptr(z), _ptr(Bm), _ptr(Cm),
                                 _ptr(A_log), _ptr(Dskip), _ptr(h0), _ptr(y),
                                 _ptr(hf), B, L, D, N, io, int(bool(dt_softplus)),
                                 _ptr(ws), wsb, stream), "lr_selective_scan_fwd")
    return _finish((y, hf), host_out, host, dev, sync_host)


def rglru_scan(x, r, i, a_log, c: float = 8.0, h0=None, workspace=None, out=None,
               sync_host: bool = True, gates_preact: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """RG-LRU scan.  x, r, i: (B, L, D) (r, i after their sigmoid, or before
    it with ``gates_preact=True``: the kernel applies it), one dtype;
    a_log: (D,) fp32; h0: (B, D) fp32.  Returns (y (B, L, D), h_final (B, D)
    fp32); ``out=(y, h_final)`` gives the result tensors (GPU or host).  Host
    inputs with host (or no) ``out`` run the library's host-buffer path
    (activated gates only; ``sync_host=False`` queues it, as for
    ``selective_scan``)."""
    if not gates_preact and _host_route((x, r, i), out):
        x, r, i = (_h(t) for t in (x, r, i))
        a_log, h0 = (_h(t, torch.float32) for t in (a_log, h0))
        _same(x, r, i)
        io = _io_of(x)
        B, L, D = x.shape
        y, hf = _host_outputs(out, [((B, L, D), x.dtype), ((B, D), torch.float32)])
        fn, ws, wsb = _host_entry(lr_rglru_scan_fwd_host, lr_rglru_scan_fwd_host_async,
                                  lr_rglru_scan_fwd_host_workspace_size(B, L, D, io), workspace, sync_host,
                                  (x, r, i, a_log, h0, y, hf))
        _check(fn(_ptr(x), _ptr(r), _ptr(i), _ptr(a_log), float(c), _ptr(h0), _ptr(y), _ptr(hf),
                  B, L, D, io, _ptr(ws), wsb, _host_stream()), fn.__name__)
        return y, hf
    host = x.device.type != "cuda"
    dev = _target_device(x)
    x, r, i = (_dev(t, dev) for t in (x, r, i))
    a_log, h0 = (_dev(None if t is None else t.float(), dev) for t in (a_log, h0))
    _same(x, r, i)
    io = _io_of(x)
    B, L, D = x.shape
    (y, hf), host_out = _outputs(out, [((B, L, D), x.dtype), ((B, D), torch.float32)], dev)
    ws, wsb = _workspace(lr_rglru_scan_workspace_size(B, L, D, io), dev, workspace)
    stream = torch.cuda.current_stream(dev).cuda_stream
    fwd = lr_rglru_scan_preact_fwd if gates_preact else lr_rglru_scan_fwd
    _check(fwd(_ptr(x), _ptr(r), _ptr(i), _ptr(a_log), float(c), _ptr(h0), _ptr(y), _ptr(hf),
               B, L, D, io, _ptr(ws), wsb, stream), fwd.__name__)
    return _finish((y, hf), host_out, host, dev, sync_host)


def hgrn2(q, k, v, g, H: int, S0=None, chunk: int = 64, workspace=None, out=None,
          sync_host: bool = True, gate_lb: Optional[float] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """HGRN2 matrix-state recurrence.  q, k: (B, L, H*dk); v, g: (B, L, H*dv)
    (g after its activation and lower bound; with ``gate_lb`` set, g is the
    pre-activation f and the kernel forms lb + (1 - lb) sigmoid(f)), one
    dtype (bfloat16 or float32); S0: (B, H, dv, dk) fp32.  Returns (o (B, L, H*dv), S_final
    (B, H, dv, dk) fp32); ``out=(o, S_final)`` gives the result tensors (GPU
    or host).  Host inputs with host (or no) ``out`` run the library's
    host-buffer path (activated gates only; ``sync_host=False`` queues it, as
    for ``selective_scan``).  Raises ValueError when the hidden size is not
    divisible by the head count."""
    if q.shape[-1] % H or v.shape[-1] % H:
        raise ValueError(f"hidden size {q.shape[-1]} is not divisible by {H} heads")
    if gate_lb is None and _host_route((q, k, v, g), out):
        q, k, v, g = (_h(t) for t in (q, k, v, g))
        S0 = _h(S0, torch.float32)
        _same(q, k, v, g)
        io = _io_of(q)
        B, L, HK = q.shape
        dk, dv = HK // H, v.shape[-1] // H
        o, Sf = _host_outputs(out, [((B, L, H * dv), q.dtype), ((B, H, dv, dk), torch.float32)])
        fn, ws, wsb = _host_entry(lr_hgrn2_fwd_host, lr_hgrn2_fwd_host_async,
                                  lr_hgrn2_fwd_host_workspace_size(B, L, H, dk, dv, io), workspace, sync_host,
                                  (q, k, v, g, S0, o, Sf))
        _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(S0), _ptr(o), _ptr(Sf),
                  B, L, H, dk, dv, chunk, io, _ptr(ws), wsb, _host_stream()), fn.__name__)
        return o, Sf
    host = q.device.type != "cuda"
    dev = _target_device(q)
    q, k, v, g = (_dev(t, dev) for t in (q, k, v, g))
    S0 = _dev(None if S0 is None else S0.float(), dev)
    _same(q, k, v, g)
    io = _io_of(q)
    B, L, HK = q.shape
    dk, dv = HK // H, v.shape[-1] // H
    (o, Sf), host_out = _outputs(out, [((B, L, H * dv), q.dtype), ((B, H, dv, dk), torch.float32)],
                                 dev)
    ws, wsb = _workspace(lr_hgrn2_workspace_size(B, L, H, dk, dv, io), dev, workspace)
    stream = torch.cuda.current_stream(dev).cuda_stream
    if gate_lb is None:
        _check(lr_hgrn2_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(S0), _ptr(o),
                            _ptr(Sf), B, L, H, dk, dv, chunk, io, _ptr(ws), wsb,
                            stream), "lr_hgrn2_fwd")
    else:
        _check(lr_hgrn2_preact_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), float(gate_lb), _ptr(S0),
                                   _ptr(o), _ptr(Sf), B, L, H, dk, dv, chunk, io, _ptr(ws), wsb,
                                   stream), "lr_hgrn2_preact_fwd")
    return _finish((o, Sf), host_out, host, dev, sync_host)


def minmax_scan(r, s, x0=None, workspace=None, out=None,
                sync_host: bool = True) -> Tuple[torch.Tensor, torch.Tensor]:
    """MinMax recurrence x_t = max(min(r_t, x_{t-1}), s_t).  r, s: (B, L, D),
    one dtype (float32 or bfloat16); x0: (B, D) fp32 or None (zero).
    Returns (y (B, L, D) = the state after every step, x_final (B, D) fp32);
    ``out=(y, x_final)`` gives the result tensors (GPU or host).  Host inputs
    with host (or no) ``out`` run the library's host-buffer path
    (``sync_host=False`` queues it, as for ``selective_scan``)."""
    if _host_route((r, s), out):
        r, s = (_h(t) for t in (r, s))
        x0 = _h(x0, torch.float32)
        _same(r, s)
        io = _io_of(r)
        B, L, D = r.shape
        y, xf = _host_outputs(out, [((B, L, D), r.dtype), ((B, D), torch.float32)])
        fn, ws, wsb = _host_entry(lr_minmax_scan_fwd_host, lr_minmax_scan_fwd_host_async,
                                  lr_minmax_scan_fwd_host_workspace_size(B, L, D, io), workspace, sync_host,
                                  (r, s, x0, y, xf))
        _check(fn(_ptr(r), _ptr(s), _ptr(x0), _ptr(y), _ptr(xf), B, L, D, io, _ptr(ws), wsb,
                  _host_stream()), fn.__name__)
        return y, xf
    host = r.device.type != "cuda"
    dev = _target_device(r)
    r, s = (_dev(t, dev) for t in (r, s))
    x0 = _dev(None if x0 is None else x0.float(), dev)
    _same(r, s)
    io = _io_of(r)
    B, L, D = r.shape
    (y, xf), host_out = _outputs(out, [((B, L, D), r.dtype), ((B, D), torch.float32)], dev)
    ws, wsb = _workspace(lr_minmax_scan_workspace_size(B, L, D, io), dev, workspace)
    stream = torch.cuda.current_stream(dev).cuda_stream
    _check(lr_minmax_scan_fwd(_ptr(r), _ptr(s), _ptr(x0), _ptr(y), _ptr(xf), B, L, D, io, _ptr(ws),
                              wsb, stream), "lr_minmax_scan_fwd")
    return _finish((y, xf), host_out, host, dev, sync_host)


def _step_state(state, shape, dev, state_out):
    """(state before the step or None, state buffer the step writes)."""
    h_in = None if state is None else _dev(state.float(), dev)
    if state_out is None:
        state_out = torch.empty(shape, dtype=torch.float32, device=dev)
    elif (tuple(state_out.shape) != tuple(shape) or state_out.dtype != torch.float32
          or state_out.device != dev or not state_out.is_contiguous()):
        raise ValueError(f"state_out must be a contiguous fp32 GPU tensor of shape {tuple(shape)}")
    return h_in, state_out


def selective_scan_step(x, dt, Bm, Cm, A_log, z=None, Dskip=None, h=None,
                        dt_softplus: bool = True, h_out=None):
    """One decode step of the selective SSM.  x, dt, z: (B, D); Bm, Cm: (B, 16),
    one dtype on the GPU; A_log: (D, 16); Dskip: (D,); h: (B, D, 16) fp32 or
    None (zero).  Returns (y (B, D), h_new (B, D, 16) fp32); ``h_out`` gives
    the buffer h_new is written to (it may be ``h`` itself)."""
    dev = _target_device(x)
    x, dt, z, Bm, Cm = (_dev(t, dev) for t in (x, dt, z, Bm, Cm))
    A_log, Dskip = (_dev(None if t is None else t.float(), dev) for t in (A_log, Dskip))
    _same(x, dt, z, Bm, Cm)
    B, D = x.shape
    N = Bm.shape[-1]
    h_in, h_new = _step_state(h, (B, D, N), dev, h_out)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev).cuda_stream
    _check(lr_selective_scan_step(_ptr(x), _ptr(dt), _ptr(z), _ptr(Bm), _ptr(Cm), _ptr(A_log),
                                  _ptr(Dskip), _ptr(h_in), _ptr(h_new), _ptr(y), B, D, N,
                                  _io_of(x), int(bool(dt_softplus)), stream),
           "lr_selective_scan_step")
    return y, h_new


def rglru_scan_step(x, r, i, a_log, c: float = 8.0, h=None, h_out=None):
    """One decode step of the RG-LRU.  x, r, i: (B, D) on the GPU; a_log: (D,);
    h: (B, D) fp32 or None.  Returns (y (B, D), h_new (B, D) fp32)."""
    dev = _target_device(x)
    x, r, i = (_dev(t, dev) for t in (x, r, i))
    a_log = _dev(a_log.float(), dev)
    _same(x, r, i)
    B, D = x.shape
    h_in, h_new = _step_state(h, (B, D), dev, h_out)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev).cuda_stream
    _check(lr_rglru_scan_step(_ptr(x), _ptr(r), _ptr(i), _ptr(a_log), float(c), _ptr(h_in),
                              _ptr(h_new), _ptr(y), B, D, _io_of(x), stream), "lr_rglru_scan_step")
    return y, h_new


def minmax_scan_step(r, s, x=None, x_out=None):
    """One decode step of the MinMax recurrence.  r, s: (B, D) on the GPU;
    x: (B, D) fp32 or None (zero).  Returns (y (B, D), x_new (B, D) fp32)."""
    dev = _target_device(r)
    r, s = (_dev(t, dev) for t in (r, s))
    _same(r, s)
    B, D = r.shape
    x_in, x_new = _step_state(x, (B, D), dev, x_out)
    y = torch.empty_like(r)
    stream = torch.cuda.current_stream(dev).cuda_stream
    _check(lr_minmax_scan_step(_ptr(r), _ptr(s), _ptr(x_in), _ptr(x_new), _ptr(y), B, D, _io_of(r),
                               stream), "lr_minmax_scan_step")
    return y, x_new


def hgrn2_step(q, k, v, g, H: int, S=None, S_out=None):
    """One decode step of HGRN2.  q, k: (B, H*dk); v, g: (B, H*dv) on the GPU;
    S: (B, H, dv, dk) fp32 or None.  Returns (o (B, H*dv), S_new)."""
    if q.shape[-1] % H or v.shape[-1] % H:
        raise ValueError(f"hidden size {q.shape[-1]} is not divisible by {H} heads")
    dev = _target_device(q)
    q, k, v, g = (_dev(t, dev) for t in (q, k, v, g))
    _same(q, k, v, g)
    B = q.shape[0]
    dk, dv = q.shape[-1] // H, v.shape[-1] // H
    S_in, S_new = _step_state(S, (B, H, dv, dk), dev, S_out)
    o = torch.empty(B, H * dv, dtype=q.dtype, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    _check(lr_hgrn2_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(S_in), _ptr(S_new), _ptr(o),
                         B, H, dk, dv, _io_of(q), stream), "lr_hgrn2_step")
    return o, S_new


def status(workspace=None, stream=None) -> int:
    """Device-side status code of the latest call that used ``workspace`` (a
    tensor; default: the workspace of this thread's latest call through the
    torch helpers); synchronises the stream (default: current) and resets
    the status to LR_OK."""
    ws = workspace if workspace is not None else last_workspace()
    if ws is None:
        return LR_OK
    s = (stream if stream is not None else torch.cuda.current_stream(ws.device)).cuda_stream
    return lr_check_status(ws.data_ptr(), s)


def check_status(workspace=None, stream=None) -> None:
    """As :func:`status`, raising :class:`LrError` on a non-zero code."""
    _check(status(workspace, stream), "device status")
