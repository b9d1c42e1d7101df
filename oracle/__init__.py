"""fp64 CPU oracle for the chunked Gated DeltaNet prefill.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never imports, links or calls it, and it imports nothing from the library.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, POSIX threads over
(sequence, head) units); this module compiles it with gcc and marshals numpy
arrays through ctypes.  What each entry point computes, and which passage of
the pages it follows, is stated in the C file's header:

* :func:`gdn_sequential` -- the per-token gated delta rule recurrence
  ("GDN 与 Chunked Prefill", section "GDN 是什么": the decaying form
  S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = scale S_t q_t).
* :func:`gdn_chunked` -- the same result through the 64-token chunk algebra
  (log-space gate sums, triangular solve, W/U, Delta, chunk output, state
  pass), optionally returning the per-chunk G, W and U.
* :func:`chunk_map` -- the flat chunk -> (sequence, chunk) table
  ("GDN 与 Chunked Prefill", section "chunked prefill 有两层含义").

Every function is pinned by ``tests/test_oracle_pins.py`` to facts the pages
and the mathematics fix (the 4-token expansion table, closed forms, erasure
and linear-attention special cases, chunk-map and checkpoint-count examples).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


class _Args(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int64),
        ("N", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p),
        ("hq", ctypes.c_int32),
        ("hk", ctypes.c_int32),
        ("hv", ctypes.c_int32),
        ("D", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p),
        ("beta", ctypes.c_void_p),
        ("scale", ctypes.c_double),
        ("l2norm", ctypes.c_int32),
        ("initial_state", ctypes.c_void_p),
        ("state_indices", ctypes.c_void_p),
        ("output", ctypes.c_void_p),
        ("final_state", ctypes.c_void_p),
        ("ckpt_n", ctypes.c_int32),
        ("ckpt_cu_starts", ctypes.c_void_p),
        ("checkpoints", ctypes.c_void_p),
        ("chunk", ctypes.c_int32),
        ("dump_g", ctypes.c_void_p),
        ("dump_w", ctypes.c_void_p),
        ("dump_u", ctypes.c_void_p),
        ("threads", ctypes.c_int32),
    ]


def build(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle into a shared library (gcc, -O2, no -march)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, src, "-lpthread", "-lm"],
                   check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` loads another build of it."""
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
        _declare(lib)
        return lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            _declare(lib)
            _lib = lib
    return _lib


def _declare(lib):
    lib.oracle_gdn_sequential.argtypes = [ctypes.POINTER(_Args)]
    lib.oracle_gdn_sequential.restype = ctypes.c_int
    lib.oracle_gdn_chunked.argtypes = [ctypes.POINTER(_Args)]
    lib.oracle_gdn_chunked.restype = ctypes.c_int
    lib.oracle_chunk_map.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_int64]
    lib.oracle_chunk_map.restype = ctypes.c_int64


def _f64(x):
    return None if x is None else np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x):
    return None if x is None else np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _run(fn_name, q, k, v, g, beta, cu_seqlens, scale, initial_state, state_indices, output_final_state,
         l2norm, checkpoint_every_n_tokens, checkpoint_cu_starts, chunk, dump, threads, lib):
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, hq, D = q.shape
    hk, hv = k.shape[1], v.shape[1]
    H = max(hq, hv)
    cu = _i64(cu_seqlens if cu_seqlens is not None else [0, T])
    N = cu.shape[0] - 1
    g, beta = _f64(g), _f64(beta)
    s0 = _f64(initial_state)
    idx = _i64(state_indices)
    out = np.zeros((T, H, D), dtype=np.float64)
    final = None
    if output_final_state:
        if idx is not None:
            # the pool itself is the result: untouched rows keep their values
            final = s0.copy() if s0 is not None else np.zeros((int(idx.max()) + 1 if N else 0, H, D, D))
        else:
            final = np.zeros((N, H, D, D), dtype=np.float64)
    n = int(checkpoint_every_n_tokens or 0)
    ccs, ckpts = None, None
    if n > 0:
        ccs = _i64(checkpoint_cu_starts)
        ckpts = np.zeros((int(ccs[-1]), H, D, D), dtype=np.float64)
    dumps = {}
    if dump:
        lens = np.diff(cu)
        nflat = int(((lens + chunk - 1) // chunk).sum())
        dumps = {"G": np.zeros((nflat, H, chunk)), "W": np.zeros((nflat, H, chunk, D)),
                 "U": np.zeros((nflat, H, chunk, D))}
    a = _Args(T=T, N=N, cu_seqlens=_ptr(cu), hq=hq, hk=hk, hv=hv, D=D, q=_ptr(q), k=_ptr(k), v=_ptr(v),
              g=_ptr(g), beta=_ptr(beta), scale=float(D ** -0.5 if scale is None else scale),
              l2norm=int(bool(l2norm)), initial_state=_ptr(s0), state_indices=_ptr(idx), output=_ptr(out),
              final_state=_ptr(final), ckpt_n=n, ckpt_cu_starts=_ptr(ccs), checkpoints=_ptr(ckpts),
              chunk=int(chunk), dump_g=_ptr(dumps.get("G")), dump_w=_ptr(dumps.get("W")),
              dump_u=_ptr(dumps.get("U")), threads=int(threads or default_threads()))
    rc = getattr(lib, fn_name)(ctypes.byref(a))
    if rc != 0:
        raise ValueError(f"oracle {fn_name} rejected its arguments (code {rc})")
    res = {"output": out, "final_state": final, "checkpoints": ckpts}
    res.update(dumps)
    return res


def gdn_sequential(q, k, v, g=None, beta=None, cu_seqlens=None, scale=None, initial_state=None,
                   state_indices=None, output_final_state=False, l2norm=False, checkpoint_every_n_tokens=0,
                   checkpoint_cu_starts=None, threads=None, lib=None):
    """Per-token recurrence.  Returns dict(output [T,H,D], final_state, checkpoints).

    With ``state_indices`` the returned final_state is the whole pool (rows not
    named by ``state_indices`` keep their initial values), as the pages' API
    returns the pool itself.
    """
    return _run("oracle_gdn_sequential", q, k, v, g, beta, cu_seqlens, scale, initial_state, state_indices,
                output_final_state, l2norm, checkpoint_every_n_tokens, checkpoint_cu_starts, 1, False, threads,
                lib)


def gdn_chunked(q, k, v, g=None, beta=None, cu_seqlens=None, scale=None, initial_state=None,
                state_indices=None, output_final_state=False, l2norm=False, checkpoint_every_n_tokens=0,
                checkpoint_cu_starts=None, chunk=64, return_intermediates=False, threads=None, lib=None):
    """Chunk form (chunk length ``chunk``).  Same returns as :func:`gdn_sequential`,
    plus G [n_chunks,H,C], W and U [n_chunks,H,C,D] when ``return_intermediates``."""
    return _run("oracle_gdn_chunked", q, k, v, g, beta, cu_seqlens, scale, initial_state, state_indices,
                output_final_state, l2norm, checkpoint_every_n_tokens, checkpoint_cu_starts, chunk,
                return_intermediates, threads, lib)


def chunk_map(cu_seqlens, chunk=64, map_rows=None, lib=None):
    """Returns (offsets [N+1] int32, map [map_rows, 2] int32 padded with -1, n_chunks)."""
    lib = lib or load()
    cu = _i64(cu_seqlens)
    N = cu.shape[0] - 1
    if map_rows is None:
        map_rows = int(((np.diff(cu) + chunk - 1) // chunk).clip(min=0).sum())
    offsets = np.zeros(N + 1, dtype=np.int32)
    mp = np.zeros((max(map_rows, 0), 2), dtype=np.int32)
    n = lib.oracle_chunk_map(N, _ptr(cu), int(chunk), _ptr(offsets), _ptr(mp), int(map_rows))
    if n < 0:
        raise ValueError("oracle chunk_map: decreasing cu_seqlens or map too small")
    return offsets, mp, int(n)
