"""Python binding of ``libditattn.so`` (ctypes; argument marshalling only).

The functions named like the C entry points (``dit_attn_fwd``,
``dit_attn_fwd_partials``, ``dit_attn_merge``, ``cfg_combine``) take torch CUDA
tensors for every buffer, check dtype / shape / contiguity / device, and pass
raw pointers plus the current torch stream to the C ABI.  All arithmetic runs
in the library's CUDA kernels.  There is no CPU fallback: if the library is
missing or a call fails, a ``RuntimeError`` is raised.

Convenience wrappers ``attention``, ``attention_partials``, ``merge`` and
``combine`` allocate the outputs with torch and return them.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libditattn.so")

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p

SIGNATURES = {
    "dit_attn_fwd": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      ctypes.c_int, _vp], ctypes.c_int),
    "dit_attn_fwd_partials": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, _vp], ctypes.c_int),
    "dit_attn_merge": ([_vp, _vp, ctypes.c_int, _vp, _vp, ctypes.c_longlong, ctypes.c_int, _vp],
                       ctypes.c_int),
    "dit_attn_fwd_range": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                            ctypes.c_int, ctypes.c_int, _vp], ctypes.c_int),
    "dit_attn_fwd_torus": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int,
                            ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp], ctypes.c_int),
    "dit_attn_fwd_split": ([_vp, _vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                            ctypes.c_int, _vp, ctypes.c_size_t, _vp], ctypes.c_int),
    "dit_attn_split_workspace_bytes": ([ctypes.c_int] * 5, ctypes.c_size_t),
    "cfg_combine": ([_vp, _vp, ctypes.c_float, _vp, ctypes.c_longlong, _vp], ctypes.c_int),
    "cfg_combine_relmae": ([_vp, _vp, ctypes.c_float, _vp, ctypes.c_longlong, _vp, _vp], ctypes.c_int),
    "cfg_combine_relmae_static": ([_vp, _vp, ctypes.c_float, _vp, ctypes.c_longlong, _vp, _vp], ctypes.c_int),
    "dit_last_device_status": ([_vp], ctypes.c_int),
    "dit_selftest_bounded_wait": ([_vp], ctypes.c_int),
    "dit_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "dit_abi_version": ([], ctypes.c_int),
}

STATUS = {
    0: "DIT_OK", -1: "DIT_ERR_INVALID_ARG", -2: "DIT_ERR_UNSUPPORTED_SHAPE", -3: "DIT_ERR_MISALIGNED",
    -4: "DIT_ERR_UNSUPPORTED_DEVICE", -5: "DIT_ERR_LAUNCH", -6: "DIT_ERR_DEVICE_TIMEOUT",
    -7: "DIT_ERR_CUDA",
}


class DitError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


def lib() -> ctypes.CDLL:
    """Load ``libditattn.so`` (built in-tree); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m sequence_attention_attn_b300.build` (no CPU fallback exists)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (argtypes, restype) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = argtypes
                fn.restype = restype
            _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().dit_status_string(int(status)).decode()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise DitError(rc, what)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# ----------------------------------------------------------- C-named calls
def dit_attn_fwd(q, k, v, out, lse, n_kv_chunks: int = 1, stream=None) -> None:
    """Blockwise attention; q, k, v, out bf16 [B, H, S, D]; lse fp32 [B, H, S] or None."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, S, D]")
    B, H, S, D = q.shape
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(out, "out", torch.bfloat16, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, S))
    rc = lib().dit_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            None if lse is None else lse.data_ptr(), B, H, S, D, int(n_kv_chunks),
                            _stream(stream))
    _check(rc, "dit_attn_fwd")


def dit_attn_fwd_partials(q, k, v, partials, lses, n_kv_chunks: int, stream=None) -> None:
    """Per-chunk partials: partials fp32 [n, B*H*S, D], lses fp32 [n, B*H*S]."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, S, D]")
    B, H, S, D = q.shape
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    n = int(n_kv_chunks)
    _need(partials, "partials", torch.float32, (n, B * H * S, D))
    _need(lses, "lses", torch.float32, (n, B * H * S))
    rc = lib().dit_attn_fwd_partials(q.data_ptr(), k.data_ptr(), v.data_ptr(), partials.data_ptr(),
                                     lses.data_ptr(), B, H, S, D, n, _stream(stream))
    _check(rc, "dit_attn_fwd_partials")


def dit_attn_split_workspace_bytes(B: int, H: int, S: int, D: int, n_split: int) -> int:
    """Bytes of workspace dit_attn_fwd_split needs (0 for invalid sizes)."""
    return int(lib().dit_attn_split_workspace_bytes(int(B), int(H), int(S), int(D), int(n_split)))


def dit_attn_fwd_split(q, k, v, out, lse, n_split: int, workspace, stream=None) -> None:
    """Chunk-parallel attention: q, k, v, out bf16 [B, H, S, D]; lse fp32
    [B, H, S] or None; workspace a uint8 CUDA tensor of at least
    dit_attn_split_workspace_bytes(...) bytes."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, S, D]")
    B, H, S, D = q.shape
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(out, "out", torch.bfloat16, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, H, S))
    _need(workspace, "workspace", torch.uint8)
    rc = lib().dit_attn_fwd_split(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  None if lse is None else lse.data_ptr(), B, H, S, D, int(n_split),
                                  workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check(rc, "dit_attn_fwd_split")


def dit_attn_merge(partials, lses, out, lse_out=None, stream=None) -> None:
    """LSE merge: partials fp32 [n, rows, D], lses fp32 [n, rows] -> out [rows, D]."""
    _need(partials, "partials", torch.float32)
    if partials.dim() != 3:
        raise ValueError("partials must be [n, rows, D]")
    n, rows, D = partials.shape
    _need(lses, "lses", torch.float32, (n, rows))
    _need(out, "out", torch.float32, (rows, D))
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32, (rows,))
    rc = lib().dit_attn_merge(partials.data_ptr(), lses.data_ptr(), n, out.data_ptr(),
                              None if lse_out is None else lse_out.data_ptr(), rows, D,
                              _stream(stream))
    _check(rc, "dit_attn_merge")


def cfg_combine(eps_c, eps_u, w: float, out, stream=None) -> None:
    """out = eps_u + w (eps_c - eps_u); fp32, same shapes; out may be eps_c or eps_u."""
    _need(eps_c, "eps_c", torch.float32)
    _need(eps_u, "eps_u", torch.float32, eps_c.shape)
    _need(out, "out", torch.float32, eps_c.shape)
    rc = lib().cfg_combine(eps_c.data_ptr(), eps_u.data_ptr(), float(w), out.data_ptr(), eps_c.numel(),
                           _stream(stream))
    _check(rc, "cfg_combine")


def dit_attn_fwd_range(q, k, v, out, lse, j0: int, j1: int, stream=None) -> None:
    """Attention over keys [j0, j1): out fp32 [B*H*S, D], lse fp32 [B*H*S]."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, S, D]")
    B, H, S, D = q.shape
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(out, "out", torch.float32, (B * H * S, D))
    _need(lse, "lse", torch.float32, (B * H * S,))
    rc = lib().dit_attn_fwd_range(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                  B, H, S, D, int(j0), int(j1), _stream(stream))
    _check(rc, "dit_attn_fwd_range")


def dit_attn_fwd_torus(q, k_src, v_src, k, v, partials, lses, out, lse_out, n_kv_chunks: int, stream=None,
                       copy_stream=None) -> None:
    """Torus-style chunked attention: K/V chunks copied from k_src / v_src (pinned
    host or device tensors) into k / v on copy_stream while earlier chunks are
    computed on stream; partials fp32 [n, B*H*S, D], lses fp32 [n, B*H*S], out fp32
    [B*H*S, D], lse_out fp32 [B*H*S] or None."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, S, D]")
    B, H, S, D = q.shape
    n = int(n_kv_chunks)
    rows = B * H * S
    for t, name in ((k_src, "k_src"), (v_src, "v_src")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or tuple(t.shape) != tuple(q.shape) \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(partials, "partials", torch.float32, (n, rows, D))
    _need(lses, "lses", torch.float32, (n, rows))
    _need(out, "out", torch.float32, (rows, D))
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32, (rows,))
    cs = None if copy_stream is None else _stream(copy_stream)
    rc = lib().dit_attn_fwd_torus(q.data_ptr(), k_src.data_ptr(), v_src.data_ptr(), k.data_ptr(), v.data_ptr(),
                                  partials.data_ptr(), lses.data_ptr(), out.data_ptr(),
                                  None if lse_out is None else lse_out.data_ptr(), B, H, S, D, n,
                                  _stream(stream), cs)
    _check(rc, "dit_attn_fwd_torus")


def cfg_combine_relmae(eps_c, eps_u, w: float, out, sums, stream=None) -> None:
    """cfg_combine plus sums = [sum |eps_c - eps_u|, sum |eps_u|, rel-MAE] (fp64 [3]
    on the device); the library computes the rel-MAE discrepancy of the two
    guidance paths, sums[0] / sums[1], on the device."""
    _need(eps_c, "eps_c", torch.float32)
    _need(eps_u, "eps_u", torch.float32, eps_c.shape)
    _need(out, "out", torch.float32, eps_c.shape)
    _need(sums, "sums", torch.float64, (3,))
    rc = lib().cfg_combine_relmae(eps_c.data_ptr(), eps_u.data_ptr(), float(w), out.data_ptr(), eps_c.numel(),
                                  sums.data_ptr(), _stream(stream))
    _check(rc, "cfg_combine_relmae")


# Largest numel cfg_combine_relmae_static accepts (DIT_RELMAE_STATIC_MAX_NUMEL).
RELMAE_STATIC_MAX_NUMEL = 1 << 28


def cfg_combine_relmae_static(eps_c, eps_u, w: float, out, sums, stream=None) -> None:
    """cfg_combine_relmae with the per-block sums in the library's fixed
    device array (no workspace, nothing allocated) and a fixed summation
    order; numel <= RELMAE_STATIC_MAX_NUMEL.  Calls on one device must not
    overlap (they share that array)."""
    _need(eps_c, "eps_c", torch.float32)
    _need(eps_u, "eps_u", torch.float32, eps_c.shape)
    _need(out, "out", torch.float32, eps_c.shape)
    _need(sums, "sums", torch.float64, (3,))
    rc = lib().cfg_combine_relmae_static(eps_c.data_ptr(), eps_u.data_ptr(), float(w), out.data_ptr(),
                                         eps_c.numel(), sums.data_ptr(), _stream(stream))
    if rc == -1 and eps_c.numel() > RELMAE_STATIC_MAX_NUMEL:
        raise DitError(rc, f"cfg_combine_relmae_static: numel {eps_c.numel()} is above the maximum "
                           f"{RELMAE_STATIC_MAX_NUMEL}")
    _check(rc, "cfg_combine_relmae_static")


def dit_last_device_status(stream=None) -> int:
    """Synchronise the stream, read and clear the device status word."""
    return int(lib().dit_last_device_status(_stream(stream)))


def dit_selftest_bounded_wait(stream=None) -> None:
    """Launch the bounded-wait self test (its wait runs out after ~1 s)."""
    _check(lib().dit_selftest_bounded_wait(_stream(stream)), "dit_selftest_bounded_wait")


# --------------------------------------------------------- conveniences
def attention(q, k, v, n_kv_chunks: int = 1, with_lse: bool = True, stream=None):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device) if with_lse else None
    dit_attn_fwd(q, k, v, out, lse, n_kv_chunks, stream)
    return out, lse


def attention_split(q, k, v, n_split: int, with_lse: bool = True, stream=None):
    """dit_attn_fwd_split with the outputs and the workspace allocated by torch; returns (out, lse)."""
    B, H, S, D = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if with_lse else None
    nbytes = dit_attn_split_workspace_bytes(B, H, S, D, n_split)
    if nbytes == 0:
        raise ValueError("invalid sizes for the split launch")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    dit_attn_fwd_split(q, k, v, out, lse, n_split, ws, stream)
    return out, lse


def attention_partials(q, k, v, n_kv_chunks: int, stream=None):
    B, H, S, D = q.shape
    partials = torch.empty((n_kv_chunks, B * H * S, D), dtype=torch.float32, device=q.device)
    lses = torch.empty((n_kv_chunks, B * H * S), dtype=torch.float32, device=q.device)
    dit_attn_fwd_partials(q, k, v, partials, lses, n_kv_chunks, stream)
    return partials, lses


def merge(partials, lses, stream=None):
    n, rows, D = partials.shape
    out = torch.empty((rows, D), dtype=torch.float32, device=partials.device)
    lse = torch.empty((rows,), dtype=torch.float32, device=partials.device)
    dit_attn_merge(partials, lses, out, lse, stream)
    return out, lse


def combine(eps_c, eps_u, w: float, stream=None):
    out = torch.empty_like(eps_c)
    cfg_combine(eps_c, eps_u, w, out, stream)
    return out


def attention_range(q, k, v, j0: int, j1: int, stream=None):
    B, H, S, D = q.shape
    out = torch.empty((B * H * S, D), dtype=torch.float32, device=q.device)
    lse = torch.empty((B * H * S,), dtype=torch.float32, device=q.device)
    dit_attn_fwd_range(q, k, v, out, lse, j0, j1, stream)
    return out, lse


def attention_torus(q, k_src, v_src, n_kv_chunks: int, stream=None, copy_stream=None):
    """Returns (out fp32 [B*H*S, D], lse fp32 [B*H*S]); allocates the device K/V
    landing buffers and the partials with torch."""
    B, H, S, D = q.shape
    rows = B * H * S
    k = torch.empty_like(q)
    v = torch.empty_like(q)
    partials = torch.empty((n_kv_chunks, rows, D), dtype=torch.float32, device=q.device)
    lses = torch.empty((n_kv_chunks, rows), dtype=torch.float32, device=q.device)
    out = torch.empty((rows, D), dtype=torch.float32, device=q.device)
    lse = torch.empty((rows,), dtype=torch.float32, device=q.device)
    dit_attn_fwd_torus(q, k_src, v_src, k, v, partials, lses, out, lse, n_kv_chunks, stream, copy_stream)
    # The buffers were allocated on torch's current stream; keep the caching
    # allocator from handing them out again before the other streams finish.
    for s_ in (stream, copy_stream):
        if isinstance(s_, torch.cuda.Stream):
            for t in (k, v, partials, lses, out, lse):
                t.record_stream(s_)
    return out, lse


def combine_relmae(eps_c, eps_u, w: float, stream=None):
    """Returns (out, rel_mae): rel_mae = sum |eps_c - eps_u| / sum |eps_u| as the
    library computed it, read back as a Python float (reading waits for the stream)."""
    out = torch.empty_like(eps_c)
    sums = torch.empty(3, dtype=torch.float64, device=eps_c.device)
    cfg_combine_relmae(eps_c, eps_u, w, out, sums, stream)
    return out, sums[2].item()
