"""fp64 CPU oracle for the DiT blockwise-attention path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``sequence_attention_attn_b300``) never imports, loads or calls it, and the two
share no code: this package holds the definitions written out in plain C
(``attn_ref.c``, compiled here with gcc) and an independent NumPy twin
(``brute.py``) used to pin the C code on small inputs.

Definitions (the pages print no formula; each is the plainest reading of what
they describe, see ``attn_ref.c`` for the page citations):

* attention over keys [j0, j1) of one (batch, head)::

      score_ij = q_i . k_j / sqrt(D)
      LSE_i    = max_j score_ij + ln sum_j exp(score_ij - max_j score_ij)
      O_i      = sum_j exp(score_ij - LSE_i) v_j

* chunked attention: the keys are split into contiguous chunks, each chunk
  gives (O_c, LSE_c) by the formula above, and the chunks are merged by
  ``lse_merge`` -- the per-device computation and the recombination of ring /
  Torus sequence-parallel attention ("SwiftFusion: Scalable Sequence
  Parallelism ...", ideas 1 and 2);
* ``lse_merge``: LSE = M + ln sum_c exp(LSE_c - M), O = sum_c exp(LSE_c - LSE) O_c;
* ``cfg_combine``: out = eps_u + w (eps_c - eps_u) ("Accelerating Diffusion via
  Hybrid Data-Pipeline Parallelism Based on Conditional Guidance Scheduling",
  Technische Zusammenfassung 2A).

All arithmetic is fp64.  Inputs are widened exactly to float64 by the callers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib_handle = None

_dptr = ctypes.POINTER(ctypes.c_double)
_i64ptr = ctypes.POINTER(ctypes.c_longlong)


def _compile(src_path: str, so_path: str) -> None:
    tmp = so_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-o", tmp, src_path, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, so_path)


def build(force: bool = False) -> str:
    """Compile ``attn_ref.c`` into ``liboracle.so`` (plain gcc, OpenMP)."""
    stale = (not os.path.exists(_SO)) or os.path.getmtime(_SO) < os.path.getmtime(_SRC)
    if force or stale:
        _compile(_SRC, _SO)
    return _SO


def _as_f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dptr)


def _qkv(q, k, v):
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    if q.ndim < 2 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one shape [..., S, D]")
    lead = q.shape[:-2]
    S, D = q.shape[-2], q.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    return q, k, v, lead, BH, S, D


class OracleLib:
    """The compiled oracle: one instance per shared object."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        lib.oracle_attn_range.argtypes = [_dptr, _dptr, _dptr, ctypes.c_longlong,
                                          ctypes.c_longlong, ctypes.c_int,
                                          ctypes.c_longlong, ctypes.c_longlong,
                                          _dptr, _dptr]
        lib.oracle_attn_range.restype = ctypes.c_int
        lib.oracle_attn_rows.argtypes = [_dptr, _dptr, _dptr, ctypes.c_longlong,
                                         ctypes.c_longlong, ctypes.c_int, _i64ptr,
                                         ctypes.c_longlong, ctypes.c_longlong,
                                         ctypes.c_longlong, _dptr, _dptr]
        lib.oracle_attn_rows.restype = ctypes.c_int
        lib.oracle_lse_merge.argtypes = [_dptr, _dptr, ctypes.c_int, ctypes.c_longlong,
                                         ctypes.c_int, _dptr, _dptr]
        lib.oracle_lse_merge.restype = ctypes.c_int
        lib.oracle_cfg_combine.argtypes = [_dptr, _dptr, ctypes.c_double, _dptr,
                                           ctypes.c_longlong]
        lib.oracle_cfg_combine.restype = ctypes.c_int
        lib.oracle_cfg_relmae.argtypes = [_dptr, _dptr, ctypes.c_double, _dptr,
                                          ctypes.c_longlong, _dptr]
        lib.oracle_cfg_relmae.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        self._lib = lib

    def num_threads(self) -> int:
        """OpenMP threads the oracle's loops run on."""
        return int(self._lib.oracle_num_threads())

    def attention(self, q, k, v, j0: int = 0, j1: int | None = None):
        """Attention of all queries over keys [j0, j1).  q, k, v: [..., S, D].

        Returns (O [..., S, D], LSE [..., S]) in float64, LSE in natural log."""
        q, k, v, lead, BH, S, D = _qkv(q, k, v)
        j1 = S if j1 is None else j1
        out = np.empty((BH, S, D), dtype=np.float64)
        lse = np.empty((BH, S), dtype=np.float64)
        rc = self._lib.oracle_attn_range(_p(q), _p(k), _p(v), BH, S, D, j0, j1,
                                         _p(out), _p(lse))
        if rc != 0:
            raise ValueError(f"bad key range [{j0}, {j1}) for S={S}")
        return out.reshape(*lead, S, D), lse.reshape(*lead, S)

    def attention_rows(self, q, k, v, rows, j0: int = 0, j1: int | None = None):
        """Attention for sampled flat rows (row = bh * S + i) over keys [j0, j1).

        Returns (O [len(rows), D], LSE [len(rows)])."""
        q, k, v, _lead, BH, S, D = _qkv(q, k, v)
        j1 = S if j1 is None else j1
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        out = np.empty((rows.size, D), dtype=np.float64)
        lse = np.empty((rows.size,), dtype=np.float64)
        rc = self._lib.oracle_attn_rows(_p(q), _p(k), _p(v), BH, S, D,
                                        rows.ctypes.data_as(_i64ptr), rows.size, j0, j1,
                                        _p(out), _p(lse))
        if rc != 0:
            raise ValueError("bad rows or key range")
        return out, lse

    def lse_merge(self, partials, lses):
        """Merge n partials.  partials: [n, rows, D], lses: [n, rows].

        Returns (O [rows, D], LSE [rows])."""
        partials, lses = _as_f64(partials), _as_f64(lses)
        if partials.ndim != 3 or lses.shape != partials.shape[:2]:
            raise ValueError("partials must be [n, rows, D] and lses [n, rows]")
        n, rows, D = partials.shape
        out = np.empty((rows, D), dtype=np.float64)
        lse = np.empty((rows,), dtype=np.float64)
        rc = self._lib.oracle_lse_merge(_p(partials), _p(lses), n, rows, D, _p(out), _p(lse))
        if rc != 0:
            raise ValueError("bad merge arguments")
        return out, lse

    def cfg_combine(self, eps_c, eps_u, w: float):
        """out = eps_u + w (eps_c - eps_u), elementwise, same shape as the inputs."""
        eps_c, eps_u = _as_f64(eps_c), _as_f64(eps_u)
        if eps_c.shape != eps_u.shape:
            raise ValueError("eps_c and eps_u must share one shape")
        out = np.empty_like(eps_c)
        self._lib.oracle_cfg_combine(_p(eps_c), _p(eps_u), float(w), _p(out), eps_c.size)
        return out

    def cfg_relmae(self, eps_c, eps_u, w: float):
        """CFG combine plus the rel-MAE sums.  Returns (out, (sum |eps_c - eps_u|,
        sum |eps_u|)); the rel-MAE is their ratio (``cfg_relmae_ratio``)."""
        eps_c, eps_u = _as_f64(eps_c), _as_f64(eps_u)
        if eps_c.shape != eps_u.shape:
            raise ValueError("eps_c and eps_u must share one shape")
        out = np.empty_like(eps_c)
        sums = np.zeros(3, dtype=np.float64)
        self._lib.oracle_cfg_relmae(_p(eps_c), _p(eps_u), float(w), _p(out), eps_c.size, _p(sums))
        return out, (float(sums[0]), float(sums[1]))

    def cfg_relmae_ratio(self, eps_c, eps_u):
        """The rel-MAE sum |eps_c - eps_u| / sum |eps_u| as the oracle computes it
        (0 when both sums are 0, +inf when only the base sum is)."""
        eps_c, eps_u = _as_f64(eps_c), _as_f64(eps_u)
        if eps_c.shape != eps_u.shape:
            raise ValueError("eps_c and eps_u must share one shape")
        out = np.empty_like(eps_c)
        sums = np.zeros(3, dtype=np.float64)
        self._lib.oracle_cfg_relmae(_p(eps_c), _p(eps_u), 0.0, _p(out), eps_c.size, _p(sums))
        return float(sums[2])

    def attention_chunked(self, q, k, v, bounds):
        """Chunked attention: (O_c, LSE_c) per key range in ``bounds``, then the
        log-sum-exp merge.  Returns (O, LSE) shaped like ``attention``."""
        q, k, v, lead, BH, S, D = _qkv(q, k, v)
        parts, lses = [], []
        for j0, j1 in bounds:
            o_c, l_c = self.attention(q.reshape(BH, S, D), k.reshape(BH, S, D),
                                      v.reshape(BH, S, D), j0, j1)
            parts.append(o_c.reshape(BH * S, D))
            lses.append(l_c.reshape(BH * S))
        out, lse = self.lse_merge(np.stack(parts), np.stack(lses))
        return out.reshape(*lead, S, D), lse.reshape(*lead, S)


def default() -> OracleLib:
    """The oracle built from ``attn_ref.c`` (compiled on first use)."""
    global _lib_handle
    with _lock:
        if _lib_handle is None:
            build()
            _lib_handle = OracleLib(_SO)
    return _lib_handle


def load_variant(c_source: str, workdir: str) -> OracleLib:
    """Compile a modified copy of the oracle's C source (tests plant mistakes
    in copies of the oracle to show that its pins catch them)."""
    os.makedirs(workdir, exist_ok=True)
    tag = abs(hash(c_source)) % (1 << 40)
    src_path = os.path.join(workdir, f"variant_{tag}.c")
    so_path = os.path.join(workdir, f"libvariant_{tag}.so")
    with open(src_path, "w") as f:
        f.write(c_source)
    _compile(src_path, so_path)
    return OracleLib(so_path)


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def attention(q, k, v, j0: int = 0, j1: int | None = None):
    return default().attention(q, k, v, j0, j1)


def attention_rows(q, k, v, rows, j0: int = 0, j1: int | None = None):
    return default().attention_rows(q, k, v, rows, j0, j1)


def lse_merge(partials, lses):
    return default().lse_merge(partials, lses)


def cfg_combine(eps_c, eps_u, w: float):
    return default().cfg_combine(eps_c, eps_u, w)


def cfg_relmae(eps_c, eps_u, w: float):
    return default().cfg_relmae(eps_c, eps_u, w)


def cfg_relmae_ratio(eps_c, eps_u):
    return default().cfg_relmae_ratio(eps_c, eps_u)


def attention_chunked(q, k, v, bounds):
    return default().attention_chunked(q, k, v, bounds)


def chunk_bounds(S: int, n: int):
    """Balanced contiguous partition of [0, S) into n chunks:
    chunk c = [floor(c S / n), floor((c + 1) S / n)).  Requires 1 <= n <= S."""
    if not (1 <= n <= S):
        raise ValueError(f"need 1 <= n <= S, got n={n}, S={S}")
    return [((c * S) // n, ((c + 1) * S) // n) for c in range(n)]
