"""Chunked Gated DeltaNet prefill on one GB300 GPU.

A thin ctypes binding over the C ABI in ``include/gdn_prefill.h``: it only
marshals arguments.  Every step of the prefill runs in the CUDA kernels of
``libgdn_prefill.so`` (built in-tree by :func:`build`); PyTorch provides device
memory and the current stream.  There is no CPU fallback: if the library is
missing, every call raises.

The Python entry point mirrors the pages' API ("FlashInfer GDN Prefill 完全指南",
section "chunk_gated_delta_rule API 全参数解析"):

    chunk_gated_delta_rule(q, k, v, g=None, beta=None, scale=None,
                           initial_state=None, output_final_state=False,
                           cu_seqlens=None, use_qk_l2norm_in_kernel=False,
                           output=None, output_state=None,
                           state_checkpoints=None, checkpoint_cu_starts=None,
                           checkpoint_every_n_tokens=0, state_indices=None,
                           max_seqlen=None)

returning ``output`` or ``(output, final_state)``; with ``state_indices`` the
final state is the pool itself.  ``use_cp`` allows context parallelism inside
the GPU (long sequences cut into segments chosen on the device); the pages'
``_cp_chunk_len`` and ``backend`` arguments select among other libraries'
kernels and have no counterpart here.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import _build

__all__ = [
    "build", "lib", "chunk_gated_delta_rule", "gated_delta_rule_decode", "gdn_prefill_plan", "gdn_prefill_run",
    "gdn_prefill_prepare", "gdn_decode_run",
    "gdn_prefill_chunks", "gdn_prefill_run_static", "gdn_prefill_read_status",
    "gdn_prefill_workspace_layout", "gdn_prefill_plan_destroy", "gdn_status_string", "Desc", "Args", "Layout",
    "GdnError", "STATUS", "DEVICE_ERR", "FLAGS",
]

STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_CUDA",
          4: "GDN_ERR_DEVICE_INPUT", 5: "GDN_ERR_DEVICE_TIMEOUT"}
DTYPE_F32, DTYPE_BF16, DTYPE_F16 = 0, 1, 2
_QKV_DTYPES = {torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16, torch.float32: DTYPE_F32}
DTYPE_F8E4M3, DTYPE_F8E5M2 = 3, 4
# states and checkpoints may also be stored in fp8 (widened on load, rounded to nearest and saturated on store)
_STATE_DTYPES = {**_QKV_DTYPES, torch.float8_e4m3fn: DTYPE_F8E4M3, torch.float8_e5m2: DTYPE_F8E5M2}
FLAGS = {
    "HAS_G": 1 << 0, "HAS_BETA": 1 << 1, "HAS_SCALE": 1 << 2, "QK_L2NORM": 1 << 3, "HAS_INITIAL_STATE": 1 << 4,
    "OUTPUT_FINAL_STATE": 1 << 5, "HAS_STATE_INDICES": 1 << 6, "CU_SEQLENS_I64": 1 << 7,
    "STATE_INDICES_I64": 1 << 8, "CHECKPOINT_STARTS_I64": 1 << 9, "CONTEXT_PARALLEL": 1 << 10,
}
DEVICE_ERR = {"CU_SEQLENS": 1 << 0, "CHECKPOINT_STARTS": 1 << 1, "STATE_INDEX_RANGE": 1 << 2,
              "STATE_INDEX_DUP": 1 << 3, "MAX_SEQLEN": 1 << 4, "TIMEOUT": 1 << 5}
HEAD_SIZE = 128
CHUNK = 64


class GdnError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


class Desc(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_size", ctypes.c_int32), ("qkv_dtype", ctypes.c_int32), ("state_dtype", ctypes.c_int32),
                ("max_total_tokens", ctypes.c_int64), ("max_num_seqs", ctypes.c_int32),
                ("max_pool_rows", ctypes.c_int32), ("checkpoint_every_n_tokens", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("checkpoint_dtype", ctypes.c_int32)]


class Args(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("g", ctypes.c_void_p),
                ("beta", ctypes.c_void_p), ("scale", ctypes.c_float), ("cu_seqlens", ctypes.c_void_p),
                ("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int64), ("max_seqlen", ctypes.c_int64),
                ("initial_state", ctypes.c_void_p), ("output_state", ctypes.c_void_p),
                ("state_strides", ctypes.c_int64 * 3), ("n_pool", ctypes.c_int32),
                ("state_indices", ctypes.c_void_p), ("state_checkpoints", ctypes.c_void_p),
                ("num_checkpoints", ctypes.c_int64), ("checkpoint_cu_starts", ctypes.c_void_p),
                ("output", ctypes.c_void_p), ("device_status", ctypes.c_void_p), ("intra_g", ctypes.c_void_p),
                ("intra_w", ctypes.c_void_p), ("intra_u", ctypes.c_void_p)]


class Layout(ctypes.Structure):
    _fields_ = [("status", ctypes.c_size_t), ("n_chunks", ctypes.c_size_t), ("chunk_offsets", ctypes.c_size_t),
                ("chunk_map", ctypes.c_size_t), ("seq_order", ctypes.c_size_t), ("max_chunks", ctypes.c_int64)]


_lib = None
_lib_lock = threading.Lock()


def build() -> str:
    """Compile ``csrc/*.cu`` for sm_103a into ``libgdn_prefill.so`` (in-tree)."""
    return _build.build()


def lib():
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lib_lock:
            if _lib is None:
                if not os.path.exists(_build.LIB_PATH):
                    raise RuntimeError(f"{_build.LIB_PATH} is missing: build it with "
                                       "gated_deltanet_chunked_device_gb300.build() (nvcc, sm_103a)")
                L = ctypes.CDLL(_build.LIB_PATH)
                L.gdn_prefill_plan.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(ctypes.c_void_p),
                                               ctypes.POINTER(ctypes.c_size_t)]
                L.gdn_prefill_plan.restype = ctypes.c_int
                L.gdn_prefill_run.argtypes = [ctypes.c_void_p, ctypes.POINTER(Args), ctypes.c_void_p, ctypes.c_size_t,
                                              ctypes.c_void_p]
                L.gdn_prefill_run.restype = ctypes.c_int
                for name in ("gdn_prefill_prepare", "gdn_prefill_chunks"):
                    fn = getattr(L, name)
                    fn.argtypes = L.gdn_prefill_run.argtypes
                    fn.restype = ctypes.c_int
                L.gdn_decode_run.argtypes = [ctypes.c_void_p, ctypes.POINTER(Args), ctypes.c_int32, ctypes.c_void_p]
                L.gdn_decode_run.restype = ctypes.c_int
                L.gdn_prefill_run_static.argtypes = [ctypes.c_void_p, ctypes.POINTER(Args), ctypes.c_void_p]
                L.gdn_prefill_run_static.restype = ctypes.c_int
                L.gdn_prefill_read_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                      ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
                L.gdn_prefill_read_status.restype = ctypes.c_int
                L.gdn_prefill_workspace_layout.argtypes = [ctypes.c_void_p, ctypes.POINTER(Layout)]
                L.gdn_prefill_workspace_layout.restype = ctypes.c_int
                L.gdn_prefill_plan_destroy.argtypes = [ctypes.c_void_p]
                L.gdn_prefill_cp_segments.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32,
                                                      ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
                L.gdn_prefill_cp_segments.restype = ctypes.c_int32
                L.gdn_prefill_plan_destroy.restype = None
                L.gdn_status_string.argtypes = [ctypes.c_int]
                L.gdn_status_string.restype = ctypes.c_char_p
                _lib = L
    return _lib


# ---------------------------------------------------------------------------
# C ABI, one Python function per entry point (same names, same arguments)
# ---------------------------------------------------------------------------

def gdn_prefill_plan(desc: Desc):
    """Returns (status, plan handle, workspace bytes)."""
    plan = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib().gdn_prefill_plan(ctypes.byref(desc), ctypes.byref(plan), ctypes.byref(ws))
    return st, plan, ws.value


def gdn_prefill_run(plan, args: Args, workspace_ptr: int, workspace_bytes: int, stream_ptr: int) -> int:
    return lib().gdn_prefill_run(plan, ctypes.byref(args), ctypes.c_void_p(workspace_ptr), workspace_bytes,
                                 ctypes.c_void_p(stream_ptr))


def gdn_prefill_prepare(plan, args: Args, workspace_ptr: int, workspace_bytes: int, stream_ptr: int) -> int:
    return lib().gdn_prefill_prepare(plan, ctypes.byref(args), ctypes.c_void_p(workspace_ptr), workspace_bytes,
                                     ctypes.c_void_p(stream_ptr))


def gdn_prefill_chunks(plan, args: Args, workspace_ptr: int, workspace_bytes: int, stream_ptr: int) -> int:
    return lib().gdn_prefill_chunks(plan, ctypes.byref(args), ctypes.c_void_p(workspace_ptr), workspace_bytes,
                                    ctypes.c_void_p(stream_ptr))


def gdn_decode_run(plan, args: Args, tokens_per_seq: int, stream_ptr: int) -> int:
    return lib().gdn_decode_run(plan, ctypes.byref(args), int(tokens_per_seq), ctypes.c_void_p(stream_ptr))


def gdn_prefill_run_static(plan, args: Args, stream_ptr: int) -> int:
    """The run that allocates nothing: its workspace is a fixed array in the
    library's device globals (see include/gdn_prefill.h)."""
    return lib().gdn_prefill_run_static(plan, ctypes.byref(args), ctypes.c_void_p(stream_ptr))


def gdn_prefill_read_status(plan, workspace_ptr, device_status_ptr, stream_ptr):
    """Returns (status, bits).  Synchronises the stream."""
    bits = ctypes.c_int32()
    st = lib().gdn_prefill_read_status(plan, ctypes.c_void_p(workspace_ptr), ctypes.c_void_p(device_status_ptr),
                                       ctypes.c_void_p(stream_ptr), ctypes.byref(bits))
    return st, bits.value


def gdn_prefill_workspace_layout(plan) -> Layout:
    lay = Layout()
    st = lib().gdn_prefill_workspace_layout(plan, ctypes.byref(lay))
    if st != 0:
        raise GdnError(st, "gdn_prefill_workspace_layout")
    return lay


def gdn_prefill_cp_segments(plan, seq_lens, sm_count_hint: int = 0):
    """Returns (largest segment count or 0, per-sequence counts): the
    context-parallel choice a run of this plan makes for these host lengths."""
    n = len(seq_lens)
    lens = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in seq_lens])
    segs = (ctypes.c_int32 * max(n, 1))()
    most = lib().gdn_prefill_cp_segments(plan, lens, n, int(sm_count_hint), segs)
    return int(most), [int(segs[i]) for i in range(n)]


def gdn_prefill_plan_destroy(plan) -> None:
    lib().gdn_prefill_plan_destroy(plan)


def gdn_status_string(status: int) -> str:
    return lib().gdn_status_string(status).decode()


# ---------------------------------------------------------------------------
# Plans and workspaces, cached per shape class
# ---------------------------------------------------------------------------

class _Plan:
    def __init__(self, desc: Desc):
        st, handle, nbytes = gdn_prefill_plan(desc)
        if st != 0:
            raise GdnError(st, "gdn_prefill_plan")
        self.desc = desc
        self.handle = handle
        self.workspace_bytes = nbytes
        self.workspaces = {}

    def workspace(self, device: torch.device) -> torch.Tensor:
        key = (device.type, device.index)
        ws = self.workspaces.get(key)
        if ws is None:
            ws = torch.empty(self.workspace_bytes, dtype=torch.uint8, device=device)
            self.workspaces[key] = ws
        return ws

    def __del__(self):
        try:
            if self.handle:
                gdn_prefill_plan_destroy(self.handle)
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass


_plans = {}
_plans_lock = threading.Lock()


def _pow2_at_least(x: int, lo: int = 1) -> int:
    x = max(int(x), lo)
    return 1 << (x - 1).bit_length()


def get_plan(hq, hk, hv, qkv_dtype, flags, ckpt_n, total_tokens, num_seqs, pool_rows, state_dtype=DTYPE_F32,
             checkpoint_dtype=DTYPE_F32) -> _Plan:
    key = (hq, hk, hv, qkv_dtype, flags, ckpt_n, state_dtype, checkpoint_dtype)
    with _plans_lock:
        p = _plans.get(key)
        d = p.desc if p else None
        if p is None or d.max_total_tokens < total_tokens or d.max_num_seqs < num_seqs or d.max_pool_rows < pool_rows:
            desc = Desc(num_q_heads=hq, num_k_heads=hk, num_v_heads=hv, head_size=HEAD_SIZE, qkv_dtype=qkv_dtype,
                        state_dtype=state_dtype, max_total_tokens=_pow2_at_least(total_tokens, 64),
                        max_num_seqs=_pow2_at_least(num_seqs), max_pool_rows=_pow2_at_least(pool_rows) if pool_rows else 0,
                        checkpoint_every_n_tokens=ckpt_n, flags=flags, checkpoint_dtype=checkpoint_dtype)
            p = _Plan(desc)
            _plans[key] = p
        return p


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_dev(name, t, device, dtype=None):
    if t is None:
        return
    if t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")


def _state_layout(initial_state, output_state, device):
    """State dtype code and element strides of [row][head][v] shared by the
    initial and output states (k contiguous); (DTYPE_F32, (0, 0, 0)) without
    either.  The C side checks the strides for overlap."""
    states = [t for t in (initial_state, output_state) if t is not None]
    if not states:
        return DTYPE_F32, (0, 0, 0)
    t0 = states[0]
    for name, t in zip(("initial_state", "output_state"), (initial_state, output_state)):
        if t is None:
            continue
        if t.device != device:
            raise ValueError(f"{name} must be on {device}")
        if t.dim() != 4 or t.shape[2:] != (HEAD_SIZE, HEAD_SIZE) or t.stride(3) != 1:
            raise ValueError(f"{name} must be [rows, heads, 128, 128] with contiguous rows of 128")
        if t.dtype != t0.dtype or t.stride() != t0.stride():
            raise ValueError("initial_state and output_state must share dtype and strides")
    dt = _STATE_DTYPES.get(t0.dtype)
    if dt is None:
        raise ValueError(f"unsupported state dtype {t0.dtype}")
    strides = (0, 0, 0) if t0.is_contiguous() else tuple(int(x) for x in t0.stride()[:3])
    return dt, strides


def chunk_gated_delta_rule(q, k, v, g=None, beta=None, scale=None, initial_state=None, output_final_state=False,
                           cu_seqlens=None, use_qk_l2norm_in_kernel=False, output=None, output_state=None,
                           state_checkpoints=None, checkpoint_cu_starts=None, checkpoint_every_n_tokens=0,
                           state_indices=None, max_seqlen=None, num_seqs=None, intermediates=None,
                           device_status=None, return_plan=False, use_cp=False):
    """Chunked GDN prefill through the C ABI (see the module docstring).

    ``num_seqs`` may be given to avoid reading the length of ``cu_seqlens``
    (it is its length minus one).  ``intermediates``, when a dict, receives
    the intra-chunk outputs G, W and U per flat chunk (fp32).  With
    ``return_plan`` the plan and workspace are returned as well (for status
    and chunk-map reads).  ``use_cp`` allows context parallelism: the
    sequences that set the run's time run as segments on more SMs, chosen on
    the device (a larger workspace; the same results within rounding).
    """
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be [total_tokens, heads, head_size]")
    device = q.device
    if device.type != "cuda":
        raise ValueError("q, k, v must be CUDA tensors: this library has no CPU path")
    T, hq, D = q.shape
    hk, hv = k.shape[1], v.shape[1]
    if D != HEAD_SIZE or k.shape[2] != D or v.shape[2] != D or k.shape[0] != T or v.shape[0] != T:
        raise ValueError("q, k, v must share total_tokens and have head_size 128")
    qkv_dtype = _QKV_DTYPES.get(q.dtype)
    if qkv_dtype is None:
        raise ValueError(f"unsupported q/k/v dtype {q.dtype}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_dev(name, t, device, q.dtype)
    H = max(hq, hv)
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=device)
    _check_dev("cu_seqlens", cu_seqlens, device)
    N = int(num_seqs) if num_seqs is not None else cu_seqlens.numel() - 1
    flags = 0
    if g is not None:
        _check_dev("g", g, device, torch.float32)
        flags |= FLAGS["HAS_G"]
    if beta is not None:
        _check_dev("beta", beta, device, torch.float32)
        flags |= FLAGS["HAS_BETA"]
    if scale is not None:
        flags |= FLAGS["HAS_SCALE"]
    if use_qk_l2norm_in_kernel:
        flags |= FLAGS["QK_L2NORM"]
    if use_cp:  # the library segments the sequences that its load model says gain from it
        flags |= FLAGS["CONTEXT_PARALLEL"]
    if cu_seqlens.dtype == torch.int64:
        flags |= FLAGS["CU_SEQLENS_I64"]
    elif cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32 or int64")
    n_pool = 0
    if state_indices is not None:
        _check_dev("state_indices", state_indices, device)
        flags |= FLAGS["HAS_STATE_INDICES"]
        if state_indices.dtype == torch.int64:
            flags |= FLAGS["STATE_INDICES_I64"]
        if initial_state is None and output_state is None:
            raise ValueError("state_indices needs a state pool (initial_state and/or output_state)")
        n_pool = (initial_state if initial_state is not None else output_state).shape[0]
    if initial_state is not None:
        flags |= FLAGS["HAS_INITIAL_STATE"]
    if output_final_state:
        if output_state is None:
            if state_indices is not None:
                raise ValueError("output_final_state with state_indices requires the output_state pool")
            st_dtype = initial_state.dtype if initial_state is not None else torch.float32
            output_state = torch.empty(N, H, D, D, dtype=st_dtype, device=device)
            if initial_state is not None and not initial_state.is_contiguous():
                output_state = torch.empty_strided(initial_state.shape, initial_state.stride(), dtype=st_dtype,
                                                   device=device)
        flags |= FLAGS["OUTPUT_FINAL_STATE"]
    state_dtype, state_strides = _state_layout(initial_state, output_state if output_final_state else None, device)
    n = int(checkpoint_every_n_tokens or 0)
    if (state_checkpoints is None) != (checkpoint_cu_starts is None):
        raise ValueError("state_checkpoints and checkpoint_cu_starts must be given together")
    if n > 0 and state_checkpoints is None:
        raise ValueError("checkpoint_every_n_tokens > 0 needs state_checkpoints and checkpoint_cu_starts")
    num_ck = 0
    if checkpoint_cu_starts is not None:
        _check_dev("checkpoint_cu_starts", checkpoint_cu_starts, device)
        _check_dev("state_checkpoints", state_checkpoints, device)
        if state_checkpoints.dtype not in _STATE_DTYPES:
            raise ValueError(f"unsupported checkpoint dtype {state_checkpoints.dtype}")
        if checkpoint_cu_starts.dtype == torch.int64:
            flags |= FLAGS["CHECKPOINT_STARTS_I64"]
        num_ck = state_checkpoints.shape[0]
    if output is None:
        output = torch.empty(T, H, D, dtype=q.dtype, device=device)
    _check_dev("output", output, device, q.dtype)
    ckpt_dtype = _STATE_DTYPES[state_checkpoints.dtype] if state_checkpoints is not None else DTYPE_F32
    plan = get_plan(hq, hk, hv, qkv_dtype, flags, n, T, N, n_pool, state_dtype, ckpt_dtype)
    ws = plan.workspace(device)
    args = Args(q=_ptr(q), k=_ptr(k), v=_ptr(v), g=_ptr(g), beta=_ptr(beta),
                scale=float(scale) if scale is not None else 0.0, cu_seqlens=_ptr(cu_seqlens), num_seqs=N,
                total_tokens=T, max_seqlen=int(max_seqlen or 0), initial_state=_ptr(initial_state),
                output_state=_ptr(output_state) if output_final_state else None,
                state_strides=(ctypes.c_int64 * 3)(*state_strides), n_pool=n_pool,
                state_indices=_ptr(state_indices), state_checkpoints=_ptr(state_checkpoints), num_checkpoints=num_ck,
                checkpoint_cu_starts=_ptr(checkpoint_cu_starts), output=_ptr(output),
                device_status=_ptr(device_status))
    if isinstance(intermediates, dict):
        F = (T + CHUNK - 1) // CHUNK + N
        intermediates["G"] = torch.zeros(F, H, CHUNK, dtype=torch.float32, device=device)
        intermediates["W"] = torch.zeros(F, H, CHUNK, D, dtype=torch.float32, device=device)
        intermediates["U"] = torch.zeros(F, H, CHUNK, D, dtype=torch.float32, device=device)
        args.intra_g = intermediates["G"].data_ptr()
        args.intra_w = intermediates["W"].data_ptr()
        args.intra_u = intermediates["U"].data_ptr()
    stream = torch.cuda.current_stream(device).cuda_stream
    st = gdn_prefill_run(plan.handle, args, ws.data_ptr(), plan.workspace_bytes, stream)
    if st != 0:
        raise GdnError(st, "gdn_prefill_run")
    res = (output, output_state) if output_final_state else output
    if return_plan:
        return res, plan, ws
    return res


def gated_delta_rule_decode(q, k, v, g=None, beta=None, scale=None, initial_state=None, state_indices=None,
                            output_final_state=True, output_state=None, use_qk_l2norm_in_kernel=False,
                            tokens_per_seq=1, output=None, device_status=None):
    """Decode step (or a short run of tokens) for N sequences of ``tokens_per_seq``
    tokens each, rows i * tokens_per_seq + j of q, k, v [N * m, heads, 128],
    g and beta [N * m, H].  Reads each sequence's state (its pool row with
    ``state_indices``), carries it through the tokens and writes it back to
    ``output_state`` (the pool itself, in place, with ``state_indices``).
    Returns ``output`` or ``(output, final_state)``."""
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be [N * tokens_per_seq, heads, head_size]")
    device = q.device
    if device.type != "cuda":
        raise ValueError("q, k, v must be CUDA tensors: this library has no CPU path")
    T, hq, D = q.shape
    hk, hv = k.shape[1], v.shape[1]
    m = int(tokens_per_seq)
    if D != HEAD_SIZE or k.shape[2] != D or v.shape[2] != D or k.shape[0] != T or v.shape[0] != T or m < 1 or T % m:
        raise ValueError("q, k, v must share N * tokens_per_seq rows and have head_size 128")
    N = T // m
    qkv_dtype = _QKV_DTYPES.get(q.dtype)
    if qkv_dtype is None:
        raise ValueError(f"unsupported q/k/v dtype {q.dtype}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_dev(name, t, device, q.dtype)
    H = max(hq, hv)
    flags = 0
    if g is not None:
        _check_dev("g", g, device, torch.float32)
        flags |= FLAGS["HAS_G"]
    if beta is not None:
        _check_dev("beta", beta, device, torch.float32)
        flags |= FLAGS["HAS_BETA"]
    if scale is not None:
        flags |= FLAGS["HAS_SCALE"]
    if use_qk_l2norm_in_kernel:
        flags |= FLAGS["QK_L2NORM"]
    n_pool = 0
    if state_indices is not None:
        _check_dev("state_indices", state_indices, device)
        flags |= FLAGS["HAS_STATE_INDICES"]
        if state_indices.dtype == torch.int64:
            flags |= FLAGS["STATE_INDICES_I64"]
        if initial_state is None:
            raise ValueError("state_indices needs the state pool as initial_state")
        n_pool = initial_state.shape[0]
        if output_final_state and output_state is None:
            output_state = initial_state
    if initial_state is not None:
        flags |= FLAGS["HAS_INITIAL_STATE"]
    if output_final_state:
        if output_state is None:
            st_dtype = initial_state.dtype if initial_state is not None else torch.float32
            output_state = torch.empty(N, H, D, D, dtype=st_dtype, device=device)
            if initial_state is not None and not initial_state.is_contiguous():
                output_state = torch.empty_strided(initial_state.shape, initial_state.stride(), dtype=st_dtype,
                                                   device=device)
        flags |= FLAGS["OUTPUT_FINAL_STATE"]
    state_dtype, state_strides = _state_layout(initial_state, output_state if output_final_state else None, device)
    if output is None:
        output = torch.empty(T, H, D, dtype=q.dtype, device=device)
    _check_dev("output", output, device, q.dtype)
    plan = get_plan(hq, hk, hv, qkv_dtype, flags, 0, T, N, n_pool, state_dtype)
    args = Args(q=_ptr(q), k=_ptr(k), v=_ptr(v), g=_ptr(g), beta=_ptr(beta),
                scale=float(scale) if scale is not None else 0.0, num_seqs=N, total_tokens=T,
                initial_state=_ptr(initial_state), output_state=_ptr(output_state) if output_final_state else None,
                state_strides=(ctypes.c_int64 * 3)(*state_strides),
                n_pool=n_pool, state_indices=_ptr(state_indices), output=_ptr(output),
                device_status=_ptr(device_status))
    st = gdn_decode_run(plan.handle, args, m, torch.cuda.current_stream(device).cuda_stream)
    if st != 0:
        raise GdnError(st, "gdn_decode_run")
    return (output, output_state) if output_final_state else output


def read_status(plan: _Plan, ws: torch.Tensor, device_status=None):
    """Device status bits of the last run (synchronises the current stream)."""
    stream = torch.cuda.current_stream(ws.device).cuda_stream
    st, bits = gdn_prefill_read_status(plan.handle, ws.data_ptr(), _ptr(device_status), stream)
    if st not in (0, 4, 5):
        raise GdnError(st, "gdn_prefill_read_status")
    return bits


def read_chunk_map(plan: _Plan, ws: torch.Tensor, num_seqs: int):
    """(chunk_offsets [N+1], chunk_map [n_chunks, 2], n_chunks, seq_order [N]) written by the prepare step."""
    lay = gdn_prefill_workspace_layout(plan.handle)
    raw = ws.cpu()

    def i32(off, count):
        return raw[off: off + 4 * count].view(torch.int32).clone()

    n_chunks = int(i32(lay.n_chunks, 1)[0])
    offsets = i32(lay.chunk_offsets, num_seqs + 1)
    cmap = i32(lay.chunk_map, 2 * max(n_chunks, 0)).view(-1, 2)
    order = i32(lay.seq_order, num_seqs)
    return offsets, cmap, n_chunks, order
