"""Python binding of libfd, the C-ABI split-KV decode attention library.

Argument marshalling only: every function below checks tensor dtypes,
shapes, devices and contiguity, allocates outputs and workspace with torch
when the caller did not pass them, and calls the C entry point of the same
name (declared in include/fd.h) on the current CUDA stream.  All arithmetic
runs in the library's CUDA kernels; there is no fallback.  A missing or
unloadable libfd.so raises an error.
"""
from __future__ import annotations

import ctypes
import functools
import math
import os
import re

import torch

__all__ = [
    "FdError", "load", "open_library", "header_symbols", "fd_abi_version", "fd_status_string", "fd_num_splits",
    "fd_decode_workspace_size", "fd_decode_dense", "fd_decode_paged", "fd_quantize_keys",
    "fd_topdelta_workspace_size", "fd_decode_topdelta", "fd_device_status", "fd_decode_dense_noalloc",
    "fd_quantize_kv_fp8", "fd_num_splits_fp8", "fd_decode_fp8_workspace_size", "fd_decode_dense_fp8",
    "fd_decode_paged_fp8", "fd_quantize_kv_fp4", "fd_num_splits_fp4", "fd_decode_fp4_workspace_size",
    "fd_decode_dense_fp4", "fd_decode_paged_fp4", "fd_decode_dense_unified", "fd_decode_paged_unified",
    "fd_decode_topdelta_group_union", "fd_debug_inject_wait_timeout", "fd_quantize_v_fp4",
    "FD_OK", "FD_ERR_INVALID_ARG", "FD_ERR_UNSUPPORTED", "FD_ERR_WORKSPACE_TOO_SMALL",
    "FD_ERR_BAD_PAGE_TABLE", "FD_ERR_CUDA", "FD_ERR_DEVICE_TIMEOUT", "FD_OUT_F32", "FD_OUT_BF16",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfd.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "fd.h")

FD_OK = 0
FD_ERR_INVALID_ARG = 1
FD_ERR_UNSUPPORTED = 2
FD_ERR_WORKSPACE_TOO_SMALL = 3
FD_ERR_BAD_PAGE_TABLE = 4
FD_ERR_CUDA = 5
FD_ERR_DEVICE_TIMEOUT = 6
FD_OUT_F32 = 0
FD_OUT_BF16 = 1

_lib = None


class FdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        msg = fd_status_string(status) if _lib is not None else str(status)
        super().__init__(f"{where}: {msg}")


def load():
    """The process-wide libfd handle (loaded on first use); raises if the
    library has not been built."""
    global _lib
    if _lib is None:
        _lib = open_library(LIB_PATH)
    return _lib


def open_library(path: str):
    """Open libfd at `path` and declare its C signatures."""
    if not os.path.exists(path):
        raise ImportError(f"libfd.so not built at {path}; run long_context_decode_split_gb300._build.build()")
    lib = ctypes.CDLL(path)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "fd_abi_version": (I, []),
        "fd_status_string": (ctypes.c_char_p, [I]),
        "fd_num_splits": (I, [I, I, I, I, I, I, I]),
        "fd_decode_workspace_size": (S, [I, I, I, I, I, I, I]),
        "fd_decode_dense": (I, [P, P, P, P, I, I, I, I, I, F, I, P, I, P, P, S, P]),
        "fd_decode_paged": (I, [P, P, P, P, I, I, P, I, I, I, I, I, F, I, P, I, P, P, S, P]),
        "fd_decode_dense_unified": (I, [P, P, P, P, I, I, I, I, I, F, F, I, P, I, P, P, S, P]),
        "fd_decode_paged_unified": (I, [P, P, P, P, I, I, P, I, I, I, I, I, F, F, I, P, I, P, P, S, P]),
        "fd_quantize_keys": (I, [P, P, I, I, I, I, P, P, P, P, P]),
        "fd_topdelta_workspace_size": (S, [I, I, I, I, I, I]),
        "fd_decode_topdelta": (I, [P, P, P, P, P, P, P, I, I, I, I, I, F, F, I, I, I, P, I, P, P, P, P, S, P]),
        "fd_decode_topdelta_group_union": (I, [P, P, P, P, P, P, P, I, I, I, I, I, F, F, I, I, I, P, I, P, P, P, P,
                                               S, P]),
        "fd_device_status": (I, [I, P]),
        "fd_debug_inject_wait_timeout": (I, [ctypes.c_ulonglong, I]),
        "fd_decode_dense_noalloc": (I, [P, P, P, P, I, I, I, I, I, F, I, P, I, P, P]),
        "fd_quantize_kv_fp8": (I, [P, P, I, I, I, I, P, P, P]),
        "fd_num_splits_fp8": (I, [I, I, I, I, I, I, I]),
        "fd_decode_fp8_workspace_size": (S, [I, I, I, I, I, I, I]),
        "fd_decode_dense_fp8": (I, [P, P, P, P, P, P, I, I, I, I, I, F, I, P, I, P, P, S, P]),
        "fd_decode_paged_fp8": (I, [P, P, P, P, P, P, I, I, P, I, I, I, I, I, F, I, P, I, P, P, S, P]),
        "fd_quantize_kv_fp4": (I, [P, P, I, I, I, I, P, P, P]),
        "fd_quantize_v_fp4": (I, [P, P, I, I, I, I, P, P, P]),
        "fd_num_splits_fp4": (I, [I, I, I, I, I, I, I]),
        "fd_decode_fp4_workspace_size": (S, [I, I, I, I, I, I, I]),
        "fd_decode_dense_fp4": (I, [P, P, P, P, P, P, I, I, I, I, I, F, I, P, I, P, P, S, P]),
        "fd_decode_paged_fp4": (I, [P, P, P, P, P, P, I, I, P, I, I, I, I, I, F, I, P, I, P, P, S, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def header_symbols(path: str = HEADER):
    """Names of the functions include/fd.h declares."""
    with open(path) as f:
        text = f.read()
    return sorted(set(re.findall(r"^FD_API\s+[\w\s\*]+?\b(fd_\w+)\s*\(", text, flags=re.M)))


def _p(t):
    # the pointer as a Python int: every pointer parameter is declared c_void_p
    return None if t is None else t.data_ptr()


def _stream(stream):
    """The stream handle for a call on the current device: `stream`, which must
    belong to that device, or the device's current torch stream."""
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    dev = torch.cuda.current_device()
    if stream.device.index != dev:
        raise ValueError(f"stream is on {stream.device}, the tensors on cuda:{dev}")
    return stream.cuda_stream


def _on_device_of_first_tensor(fn):
    """Run a wrapper with its leading tensor's device current, so the
    library's planner, its scratch lookup and the default stream all refer to
    the device that holds the data (every other tensor is checked against it)."""
    @functools.wraps(fn)
    def wrapper(t, *args, **kwargs):
        if not (isinstance(t, torch.Tensor) and t.is_cuda):
            raise ValueError(f"{fn.__name__}: the first argument must be a CUDA tensor")
        if t.device.index == torch.cuda.current_device():
            return fn(t, *args, **kwargs)
        with torch.cuda.device(t.device):
            return fn(t, *args, **kwargs)
    return wrapper


def _need(cond, what):
    if not cond:
        raise ValueError(what)


def _check_cuda(t, name, dtype=None, shape=None):
    # messages are built only on failure: this runs several times per call
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    dev = torch.cuda.current_device()
    if t.device.index != dev:
        raise ValueError(f"{name} is on {t.device}, expected cuda:{dev} (the first tensor's device)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _raise(st, where):
    if st != FD_OK:
        raise FdError(st, where)


def _out_code(out_dtype):
    if out_dtype in ("bf16", torch.bfloat16, FD_OUT_BF16):
        return FD_OUT_BF16, torch.bfloat16
    if out_dtype in ("f32", "fp32", torch.float32, FD_OUT_F32):
        return FD_OUT_F32, torch.float32
    raise ValueError(f"out_dtype {out_dtype!r}")


def fd_abi_version() -> int:
    return int(load().fd_abi_version())


def fd_status_string(status: int) -> str:
    return load().fd_status_string(int(status)).decode()


def fd_num_splits(B, Hq, Hkv, L_max, d, num_splits=0, ragged=False) -> int:
    r = int(load().fd_num_splits(B, Hq, Hkv, L_max, d, num_splits, int(bool(ragged))))
    if r < 0:
        raise FdError(-r, "fd_num_splits")
    return r


_WS_SIZES = {}


def fd_decode_workspace_size(B, Hq, Hkv, L_max, d, num_splits=0, ragged=False) -> int:
    # the plan depends on the shape and the current device only: remembered per both
    key = (torch.cuda.current_device() if torch.cuda.is_available() else -1, B, Hq, Hkv, L_max, d, num_splits,
           bool(ragged))
    n = _WS_SIZES.get(key)
    if n is None:
        n = int(load().fd_decode_workspace_size(B, Hq, Hkv, L_max, d, num_splits, int(bool(ragged))))
        _WS_SIZES[key] = n
    return n


def fd_topdelta_workspace_size(B, Hq, Hkv, L_max, d, num_splits=0) -> int:
    return int(load().fd_topdelta_workspace_size(B, Hq, Hkv, L_max, d, num_splits))


def _workspace(nbytes, device, workspace):
    if nbytes == 0:
        return workspace
    if workspace is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    _check_cuda(workspace, "workspace")
    _need(workspace.numel() * workspace.element_size() >= nbytes, "workspace too small")
    return workspace


def _outputs(B, Hq, d, device, out, lse, out_dtype, want_lse):
    code, tdt = _out_code(out_dtype)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=tdt, device=device)
    _check_cuda(out, "out", tdt, (B, Hq, d))
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=device)
    if lse is not None:
        _check_cuda(lse, "lse", torch.float32, (B, Hq))
    return code, out, lse


@_on_device_of_first_tensor
def fd_decode_dense(q, k, v, seq_lens=None, scale=None, num_splits=0, out=None, lse=None,
                    out_dtype="bf16", want_lse=True, workspace=None, stream=None, _unified_phi=None):
    """Dense split-KV decode.  q [B,Hq,d] bf16; k, v [B,Hkv,L_max,d] bf16;
    seq_lens [B] int32 or None.  Returns (out [B,Hq,d], lse [B,Hq] or None)."""
    lib = load()
    _check_cuda(q, "q", torch.bfloat16)
    B, Hq, d = q.shape
    _check_cuda(k, "k", torch.bfloat16)
    _need(k.dim() == 4 and k.shape[0] == B and k.shape[3] == d, "k must be [B, Hkv, L_max, d]")
    _, Hkv, L_max, _ = k.shape
    _check_cuda(v, "v", torch.bfloat16, k.shape)
    if seq_lens is not None:
        _check_cuda(seq_lens, "seq_lens", torch.int32, (B,))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    code, out, lse = _outputs(B, Hq, d, q.device, out, lse, out_dtype, want_lse)
    need = fd_decode_workspace_size(B, Hq, Hkv, L_max, d, num_splits, seq_lens is not None)
    ws = _workspace(need, q.device, workspace)
    head = (_p(q), _p(k), _p(v), _p(seq_lens), B, Hq, Hkv, L_max, d, scale)
    tail = (int(num_splits), _p(out), code, _p(lse), _p(ws), 0 if ws is None else ws.numel() * ws.element_size(),
            _stream(stream))
    if _unified_phi is None:
        st = lib.fd_decode_dense(*head, *tail)
        _raise(st, "fd_decode_dense")
    else:
        st = lib.fd_decode_dense_unified(*head, _unified_phi, *tail)
        _raise(st, "fd_decode_dense_unified")
    return out, lse


@_on_device_of_first_tensor
def fd_decode_dense_unified(q, k, v, seq_lens=None, scale=None, phi=6.5, num_splits=0, out=None, lse=None,
                            out_dtype="bf16", want_lse=True, workspace=None, stream=None):
    """fd_decode_dense with one fixed max value `phi` (natural-log units of
    the scaled score) for every chunk, falling back to the running maximum
    where scores leave [phi - 60, phi].  Same result up to fp32 rounding."""
    return fd_decode_dense(q, k, v, seq_lens, scale, num_splits, out, lse, out_dtype, want_lse, workspace,
                           stream, _unified_phi=float(phi))


@_on_device_of_first_tensor
def fd_decode_paged_unified(q, k_pages, v_pages, page_table, num_pages, seq_lens, scale=None, phi=6.5,
                            num_splits=0, out=None, lse=None, out_dtype="bf16", want_lse=True, workspace=None,
                            stream=None):
    """fd_decode_paged with the unified max value `phi` (see
    fd_decode_dense_unified)."""
    return fd_decode_paged(q, k_pages, v_pages, page_table, num_pages, seq_lens, scale, num_splits, out, lse,
                           out_dtype, want_lse, workspace, stream, _unified_phi=float(phi))


@_on_device_of_first_tensor
def fd_decode_paged(q, k_pages, v_pages, page_table, num_pages, seq_lens, scale=None, num_splits=0,
                    out=None, lse=None, out_dtype="bf16", want_lse=True, workspace=None, stream=None,
                    _unified_phi=None):
    """Paged split-KV decode.  k_pages/v_pages [P,Hkv,64,d] bf16,
    page_table [B,max_pages] int32, seq_lens [B] int32."""
    lib = load()
    _check_cuda(q, "q", torch.bfloat16)
    B, Hq, d = q.shape
    _check_cuda(k_pages, "k_pages", torch.bfloat16)
    _need(k_pages.dim() == 4 and k_pages.shape[3] == d, "k_pages must be [P, Hkv, page, d]")
    _, Hkv, page_size, _ = k_pages.shape
    _check_cuda(v_pages, "v_pages", torch.bfloat16, k_pages.shape)
    _check_cuda(page_table, "page_table", torch.int32)
    _need(page_table.dim() == 2 and page_table.shape[0] == B, "page_table must be [B, max_pages]")
    max_pages = page_table.shape[1]
    _check_cuda(seq_lens, "seq_lens", torch.int32, (B,))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    code, out, lse = _outputs(B, Hq, d, q.device, out, lse, out_dtype, want_lse)
    need = fd_decode_workspace_size(B, Hq, Hkv, max_pages * page_size, d, num_splits, True)
    ws = _workspace(need, q.device, workspace)
    head = (_p(q), _p(k_pages), _p(v_pages), _p(page_table), max_pages, int(num_pages), _p(seq_lens), page_size,
            B, Hq, Hkv, d, scale)
    tail = (int(num_splits), _p(out), code, _p(lse), _p(ws), 0 if ws is None else ws.numel() * ws.element_size(),
            _stream(stream))
    if _unified_phi is None:
        st = lib.fd_decode_paged(*head, *tail)
        _raise(st, "fd_decode_paged")
    else:
        st = lib.fd_decode_paged_unified(*head, _unified_phi, *tail)
        _raise(st, "fd_decode_paged_unified")
    return out, lse


@_on_device_of_first_tensor
def fd_quantize_keys(k, seq_lens=None, codes=None, mn_scale=None, res=None, res_scale=None, stream=None):
    """Key encoder.  Returns (codes u8 [B,Hkv,L,d/4], mn_scale fp16 [B,Hkv,L,d/32,2],
    res int8 [B,Hkv,L,d], res_scale fp16 [B,Hkv,L,d/32])."""
    lib = load()
    _check_cuda(k, "k", torch.bfloat16)
    B, Hkv, L_max, d = k.shape
    dev = k.device
    if codes is None:
        codes = torch.zeros((B, Hkv, L_max, d // 4), dtype=torch.uint8, device=dev)
    if mn_scale is None:
        mn_scale = torch.zeros((B, Hkv, L_max, d // 32, 2), dtype=torch.float16, device=dev)
    if res is None:
        res = torch.zeros((B, Hkv, L_max, d), dtype=torch.int8, device=dev)
    if res_scale is None:
        res_scale = torch.zeros((B, Hkv, L_max, d // 32), dtype=torch.float16, device=dev)
    _check_cuda(codes, "codes", torch.uint8, (B, Hkv, L_max, d // 4))
    _check_cuda(mn_scale, "mn_scale", torch.float16, (B, Hkv, L_max, d // 32, 2))
    _check_cuda(res, "res", torch.int8, (B, Hkv, L_max, d))
    _check_cuda(res_scale, "res_scale", torch.float16, (B, Hkv, L_max, d // 32))
    if seq_lens is not None:
        _check_cuda(seq_lens, "seq_lens", torch.int32, (B,))
    st = lib.fd_quantize_keys(_p(k), _p(seq_lens), B, Hkv, L_max, d, _p(codes), _p(mn_scale), _p(res),
                              _p(res_scale), _stream(stream))
    _raise(st, "fd_quantize_keys")
    return codes, mn_scale, res, res_scale


@_on_device_of_first_tensor
def fd_decode_topdelta(q, codes, mn_scale, res, res_scale, v, seq_lens=None, scale=None, delta=5.0,
                       n_sink=4, window=64, num_splits=0, out=None, lse=None, out_dtype="bf16",
                       want_lse=True, sel_mask=None, sel_count=None, want_selection=False,
                       workspace=None, stream=None, group_union=False):
    """Top-delta sparse decode over fd_quantize_keys' outputs.  Returns
    (out, lse, sel_mask or None, sel_count or None).  group_union=True calls
    fd_decode_topdelta_group_union: every head of a KV group attends to the
    union of the group's candidate sets."""
    lib = load()
    _check_cuda(q, "q", torch.bfloat16)
    B, Hq, d = q.shape
    _check_cuda(v, "v", torch.bfloat16)
    _need(v.dim() == 4 and v.shape[0] == B and v.shape[3] == d, "v must be [B, Hkv, L_max, d]")
    _, Hkv, L_max, _ = v.shape
    _check_cuda(codes, "codes", torch.uint8, (B, Hkv, L_max, d // 4))
    _check_cuda(mn_scale, "mn_scale", torch.float16, (B, Hkv, L_max, d // 32, 2))
    _check_cuda(res, "res", torch.int8, (B, Hkv, L_max, d))
    _check_cuda(res_scale, "res_scale", torch.float16, (B, Hkv, L_max, d // 32))
    if seq_lens is not None:
        _check_cuda(seq_lens, "seq_lens", torch.int32, (B,))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    delta = math.inf if delta is None else float(delta)
    code, out, lse = _outputs(B, Hq, d, q.device, out, lse, out_dtype, want_lse)
    words = (L_max + 31) // 32
    if want_selection and sel_mask is None:
        sel_mask = torch.empty((B, Hq, words), dtype=torch.int32, device=q.device)
    if want_selection and sel_count is None:
        sel_count = torch.empty((B, Hq), dtype=torch.int32, device=q.device)
    if sel_mask is not None:
        _check_cuda(sel_mask, "sel_mask", torch.int32, (B, Hq, words))
    if sel_count is not None:
        _check_cuda(sel_count, "sel_count", torch.int32, (B, Hq))
    need = fd_topdelta_workspace_size(B, Hq, Hkv, L_max, d, num_splits)
    ws = _workspace(need, q.device, workspace)
    name = "fd_decode_topdelta_group_union" if group_union else "fd_decode_topdelta"
    st = getattr(lib, name)(_p(q), _p(codes), _p(mn_scale), _p(res), _p(res_scale), _p(v), _p(seq_lens),
                            B, Hq, Hkv, L_max, d, scale, delta, int(n_sink), int(window), int(num_splits),
                            _p(out), code, _p(lse), _p(sel_mask), _p(sel_count), _p(ws),
                            0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _raise(st, name)
    return out, lse, sel_mask, sel_count


@_on_device_of_first_tensor
def fd_decode_dense_noalloc(q, k, v, out, seq_lens=None, scale=None, num_splits=0, lse=None, stream=None):
    """fd_decode_dense for callers that cannot allocate: the library's fixed
    device scratch array stands in for the workspace, and this wrapper
    allocates nothing either (the caller passes `out` and, optionally,
    `lse`).  Raises FdError(FD_ERR_WORKSPACE_TOO_SMALL) when the plan needs
    more than FD_NOALLOC_SCRATCH_BYTES of scratch."""
    lib = load()
    _check_cuda(q, "q", torch.bfloat16)
    B, Hq, d = q.shape
    _check_cuda(k, "k", torch.bfloat16)
    _need(k.dim() == 4 and k.shape[0] == B and k.shape[3] == d, "k must be [B, Hkv, L_max, d]")
    _, Hkv, L_max, _ = k.shape
    _check_cuda(v, "v", torch.bfloat16, k.shape)
    if seq_lens is not None:
        _check_cuda(seq_lens, "seq_lens", torch.int32, (B,))
    code, _ = _out_code(out.dtype)
    _check_cuda(out, "out", None, (B, Hq, d))
    if lse is not None:
        _check_cuda(lse, "lse", torch.float32, (B, Hq))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib.fd_decode_dense_noalloc(_p(q), _p(k), _p(v), _p(seq_lens), B, Hq, Hkv, L_max, d, scale,
                                     int(num_splits), _p(out), code, _p(lse), _stream(stream))
    _raise(st, "fd_decode_dense_noalloc")
    return out, lse


# Quantized KV caches: code bytes per row and the scale entries per row, with their dtype.
#   fp8: d codes (e4m3), one float32 scale per row
#   fp4: d/2 codes (two e2m1 per byte), d/32 uint8 block exponents per row; the fp4 VALUE
#        cache holds d codes per pair of rows (_v_code_shape)
_QCACHE = {
    "fp8": (lambda d: d, lambda d: (), torch.float32),
    "fp4": (lambda d: d // 2, lambda d: (d // 32,), torch.uint8),
}


def _v_code_shape(kind, lead, rows, d):
    """Shape of the value codes: as the keys', except fp4 values in token pairs."""
    if kind == "fp4":
        return tuple(lead) + ((rows + 1) // 2, d)
    return tuple(lead) + (rows, _QCACHE[kind][0](d))


def _quantize_kv(kind, x, seq_lens, codes, scales, stream, values=False):
    code_bytes, scale_shape, scale_dtype = _QCACHE[kind]
    name = "fd_quantize_v_fp4" if values else "fd_quantize_kv_" + kind
    lib = load()
    _check_cuda(x, "x", torch.bfloat16)
    _need(x.dim() == 4, "x must be [B, H, L_max, d]")
    B, H, L_max, d = x.shape
    cshape = _v_code_shape(kind, (B, H), L_max, d) if values else (B, H, L_max, code_bytes(d))
    sshape = (B, H, L_max) + scale_shape(d)
    if codes is None:
        codes = torch.zeros(cshape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.zeros(sshape, dtype=scale_dtype, device=x.device)
    _check_cuda(codes, "codes", torch.uint8, cshape)
    _check_cuda(scales, "scales", scale_dtype, sshape)
    if seq_lens is not None:
        _check_cuda(seq_lens, "seq_lens", torch.int32, (B,))
    st = getattr(lib, name)(_p(x), _p(seq_lens), B, H, L_max, d, _p(codes), _p(scales), _stream(stream))
    _raise(st, name)
    return codes, scales


def _num_splits_q(kind, B, Hq, Hkv, L_max, d, num_splits, ragged):
    name = "fd_num_splits_" + kind
    r = int(getattr(load(), name)(B, Hq, Hkv, L_max, d, num_splits, int(bool(ragged))))
    if r < 0:
        raise FdError(-r, name)
    return r


def _workspace_size_q(kind, B, Hq, Hkv, L_max, d, num_splits, ragged):
    fn = getattr(load(), "fd_decode_%s_workspace_size" % kind)
    return int(fn(B, Hq, Hkv, L_max, d, num_splits, int(bool(ragged))))


def _decode_dense_q(kind, q, k_codes, k_scales, v_codes, v_scales, seq_lens, scale, num_splits, out, lse,
                    out_dtype, want_lse, workspace, stream):
    code_bytes, scale_shape, scale_dtype = _QCACHE[kind]
    name = "fd_decode_dense_" + kind
    lib = load()
    _check_cuda(q, "q", torch.bfloat16)
    B, Hq, d = q.shape
    _check_cuda(k_codes, "k_codes", torch.uint8)
    _need(k_codes.dim() == 4 and k_codes.shape[0] == B and k_codes.shape[3] == code_bytes(d),
          "k_codes must be [B, Hkv, L_max, %s]" % ("d" if kind == "fp8" else "d/2"))
    _, Hkv, L_max, _ = k_codes.shape
    _check_cuda(v_codes, "v_codes", torch.uint8, _v_code_shape(kind, (B, Hkv), L_max, d))
    _check_cuda(k_scales, "k_scales", scale_dtype, (B, Hkv, L_max) + scale_shape(d))
    _check_cuda(v_scales, "v_scales", scale_dtype, (B, Hkv, L_max) + scale_shape(d))
    if seq_lens is not None:
        _check_cuda(seq_lens, "seq_lens", torch.int32, (B,))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    code, out, lse = _outputs(B, Hq, d, q.device, out, lse, out_dtype, want_lse)
    need = _workspace_size_q(kind, B, Hq, Hkv, L_max, d, num_splits, seq_lens is not None)
    ws = _workspace(need, q.device, workspace)
    st = getattr(lib, name)(_p(q), _p(k_codes), _p(k_scales), _p(v_codes), _p(v_scales), _p(seq_lens),
                            B, Hq, Hkv, L_max, d, scale, int(num_splits), _p(out), code, _p(lse), _p(ws),
                            0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _raise(st, name)
    return out, lse


def _decode_paged_q(kind, q, k_pages, k_page_scales, v_pages, v_page_scales, page_table, num_pages, seq_lens,
                    scale, num_splits, out, lse, out_dtype, want_lse, workspace, stream):
    code_bytes, scale_shape, scale_dtype = _QCACHE[kind]
    name = "fd_decode_paged_" + kind
    lib = load()
    _check_cuda(q, "q", torch.bfloat16)
    B, Hq, d = q.shape
    _check_cuda(k_pages, "k_pages", torch.uint8)
    _need(k_pages.dim() == 4 and k_pages.shape[3] == code_bytes(d),
          "k_pages must be [P, Hkv, page, %s]" % ("d" if kind == "fp8" else "d/2"))
    P, Hkv, page_size, _ = k_pages.shape
    _check_cuda(v_pages, "v_pages", torch.uint8, _v_code_shape(kind, (P, Hkv), page_size, d))
    _check_cuda(k_page_scales, "k_page_scales", scale_dtype, (P, Hkv, page_size) + scale_shape(d))
    _check_cuda(v_page_scales, "v_page_scales", scale_dtype, (P, Hkv, page_size) + scale_shape(d))
    _check_cuda(page_table, "page_table", torch.int32)
    _need(page_table.dim() == 2 and page_table.shape[0] == B, "page_table must be [B, max_pages]")
    max_pages = page_table.shape[1]
    _check_cuda(seq_lens, "seq_lens", torch.int32, (B,))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    code, out, lse = _outputs(B, Hq, d, q.device, out, lse, out_dtype, want_lse)
    need = _workspace_size_q(kind, B, Hq, Hkv, max_pages * page_size, d, num_splits, True)
    ws = _workspace(need, q.device, workspace)
    st = getattr(lib, name)(_p(q), _p(k_pages), _p(k_page_scales), _p(v_pages), _p(v_page_scales),
                            _p(page_table), max_pages, int(num_pages), _p(seq_lens), page_size, B, Hq, Hkv,
                            d, scale, int(num_splits), _p(out), code, _p(lse), _p(ws),
                            0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _raise(st, name)
    return out, lse


@_on_device_of_first_tensor
def fd_quantize_kv_fp8(x, seq_lens=None, codes=None, scales=None, stream=None):
    """fp8 cache encoder.  x [B,H,L_max,d] bf16 -> (codes uint8 [B,H,L_max,d],
    scales float32 [B,H,L_max]).  Rows past seq_lens[b] are left as passed
    (zero when this wrapper allocates them)."""
    return _quantize_kv("fp8", x, seq_lens, codes, scales, stream)


def fd_num_splits_fp8(B, Hq, Hkv, L_max, d, num_splits=0, ragged=False) -> int:
    return _num_splits_q("fp8", B, Hq, Hkv, L_max, d, num_splits, ragged)


def fd_decode_fp8_workspace_size(B, Hq, Hkv, L_max, d, num_splits=0, ragged=False) -> int:
    return _workspace_size_q("fp8", B, Hq, Hkv, L_max, d, num_splits, ragged)


@_on_device_of_first_tensor
def fd_decode_dense_fp8(q, k_codes, k_scales, v_codes, v_scales, seq_lens=None, scale=None, num_splits=0,
                        out=None, lse=None, out_dtype="bf16", want_lse=True, workspace=None, stream=None):
    """Split-KV decode over an fp8 cache.  q [B,Hq,d] bf16; k_codes, v_codes
    [B,Hkv,L_max,d] uint8; k_scales, v_scales [B,Hkv,L_max] float32."""
    return _decode_dense_q("fp8", q, k_codes, k_scales, v_codes, v_scales, seq_lens, scale, num_splits, out, lse,
                           out_dtype, want_lse, workspace, stream)


@_on_device_of_first_tensor
def fd_decode_paged_fp8(q, k_pages, k_page_scales, v_pages, v_page_scales, page_table, num_pages, seq_lens,
                        scale=None, num_splits=0, out=None, lse=None, out_dtype="bf16", want_lse=True,
                        workspace=None, stream=None):
    """Paged split-KV decode over an fp8 cache.  k_pages/v_pages [P,Hkv,64,d]
    uint8, k_page_scales/v_page_scales [P,Hkv,64] float32."""
    return _decode_paged_q("fp8", q, k_pages, k_page_scales, v_pages, v_page_scales, page_table, num_pages,
                           seq_lens, scale, num_splits, out, lse, out_dtype, want_lse, workspace, stream)


@_on_device_of_first_tensor
def fd_quantize_kv_fp4(x, seq_lens=None, codes=None, scales=None, stream=None):
    """fp4 KEY cache encoder.  x [B,H,L_max,d] bf16 -> (codes uint8 [B,H,L_max,d/2],
    scales uint8 [B,H,L_max,d/32]).  Rows past seq_lens[b] are left as passed
    (zero when this wrapper allocates them)."""
    return _quantize_kv("fp4", x, seq_lens, codes, scales, stream)


@_on_device_of_first_tensor
def fd_quantize_v_fp4(x, seq_lens=None, codes=None, scales=None, stream=None):
    """fp4 VALUE cache encoder (token pairs).  x [B,H,L_max,d] bf16 -> (codes
    uint8 [B,H,(L_max+1)//2,d], scales uint8 [B,H,L_max,d/32])."""
    return _quantize_kv("fp4", x, seq_lens, codes, scales, stream, values=True)


def fd_num_splits_fp4(B, Hq, Hkv, L_max, d, num_splits=0, ragged=False) -> int:
    return _num_splits_q("fp4", B, Hq, Hkv, L_max, d, num_splits, ragged)


def fd_decode_fp4_workspace_size(B, Hq, Hkv, L_max, d, num_splits=0, ragged=False) -> int:
    return _workspace_size_q("fp4", B, Hq, Hkv, L_max, d, num_splits, ragged)


@_on_device_of_first_tensor
def fd_decode_dense_fp4(q, k_codes, k_scales, v_codes, v_scales, seq_lens=None, scale=None, num_splits=0,
                        out=None, lse=None, out_dtype="bf16", want_lse=True, workspace=None, stream=None):
    """Split-KV decode over an fp4 cache.  q [B,Hq,d] bf16; k_codes [B,Hkv,L_max,d/2]
    uint8 (fd_quantize_kv_fp4); v_codes [B,Hkv,(L_max+1)//2,d] uint8 (fd_quantize_v_fp4);
    k_scales, v_scales [B,Hkv,L_max,d/32] uint8."""
    return _decode_dense_q("fp4", q, k_codes, k_scales, v_codes, v_scales, seq_lens, scale, num_splits, out, lse,
                           out_dtype, want_lse, workspace, stream)


@_on_device_of_first_tensor
def fd_decode_paged_fp4(q, k_pages, k_page_scales, v_pages, v_page_scales, page_table, num_pages, seq_lens,
                        scale=None, num_splits=0, out=None, lse=None, out_dtype="bf16", want_lse=True,
                        workspace=None, stream=None):
    """Paged split-KV decode over an fp4 cache.  k_pages [P,Hkv,64,d/2] uint8,
    v_pages [P,Hkv,32,d] uint8 (token pairs), k_page_scales/v_page_scales
    [P,Hkv,64,d/32] uint8."""
    return _decode_paged_q("fp4", q, k_pages, k_page_scales, v_pages, v_page_scales, page_table, num_pages,
                           seq_lens, scale, num_splits, out, lse, out_dtype, want_lse, workspace, stream)


def fd_debug_inject_wait_timeout(wait_limit_ns=0, withhold_tile=-1) -> int:
    """Test-only fault injection for the bf16 dense/paged decode: a pipeline
    wait limit in ns (0 = the default 2 s) and a tile index whose copies the
    producer withholds (-1 = none).  See include/fd.h."""
    return int(load().fd_debug_inject_wait_timeout(int(wait_limit_ns), int(withhold_tile)))


def fd_device_status(clear=True, stream=None) -> int:
    """Synchronises the stream and returns the device status (FD_OK or an FD_ERR_* code)."""
    return int(load().fd_device_status(int(bool(clear)), _stream(stream)))
