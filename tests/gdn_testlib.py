"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the fp64 oracle on the same (rounded) inputs, and compare."""
import json
import os

import numpy as np
import torch

import oracle
import gated_deltanet_chunked_device_gb300 as gdn
from gated_deltanet_chunked_device_gb300 import workloads as wl

# Tolerances of the parity bar: elementwise |gpu - ref| <= tol + tol * |ref|
# fp16 inputs take the 16-bit bound the pages give for bf16 (their only 16-bit figure)
TOL = {torch.bfloat16: 2e-2, torch.float16: 2e-2, torch.float32: 1e-3}

# Storage of a state or a checkpoint in a narrower type (the reading: the fp32 value is rounded to nearest,
# ties to even; fp8 saturated to its finite range): mantissa bits m and half the subnormal spacing.  A
# stored value r of a computed value x obeys |r - x| <= 2^-(m+1) |x| + half_sub, so a stored result carries
# that much on top of the parity bar.
STORED = {torch.bfloat16: (7, 2.0 ** -134), torch.float16: (10, 2.0 ** -25), torch.float8_e4m3fn: (3, 2.0 ** -10),
          torch.float8_e5m2: (2, 2.0 ** -17)}


def rounding_bound(x, dtype):
    """Largest |round(x) - x| of storage type `dtype` at values x (numpy), normal and subnormal ranges."""
    m, half_sub = STORED[dtype]
    return 2.0 ** -(m + 1) * np.abs(x) + half_sub


def to_device(inp, device="cuda"):
    out = dict(inp)
    for key in ("q", "k", "v", "g", "beta", "cu_seqlens", "initial_state", "state_indices", "checkpoint_cu_starts"):
        if out.get(key) is not None:
            out[key] = out[key].to(device).contiguous()
    return out


def run_gpu(inp, intermediates=None, return_plan=False, check_status=True, ckpt_dtype=torch.float32, **override):
    """Run the CUDA path on device inputs `inp` (from to_device).  With
    check_status the device status word must come back clear: no input flag
    and no timed-out wait inside a kernel."""
    d = inp["q"].device
    H = inp["H"]
    T = inp["T"]
    lens = inp["seq_lens"]
    kw = dict(g=inp["g"], beta=inp["beta"], scale=inp["scale"], cu_seqlens=inp["cu_seqlens"],
              use_qk_l2norm_in_kernel=inp["use_qk_l2norm_in_kernel"], output_final_state=inp["output_final_state"])
    pool = inp.get("state_indices") is not None
    if inp.get("initial_state") is not None:
        st = inp["initial_state"].clone()
        kw["initial_state"] = st
        if pool:
            kw["state_indices"] = inp["state_indices"]
            kw["output_state"] = st  # in place, as the pages' pool example
    n = inp.get("checkpoint_every_n_tokens") or 0
    if n:
        nck = wl.num_checkpoints(lens, n)
        kw["checkpoint_every_n_tokens"] = n
        kw["checkpoint_cu_starts"] = inp["checkpoint_cu_starts"]
        kw["state_checkpoints"] = torch.full((max(nck, 1), H, 128, 128), float("nan"), device=d).to(ckpt_dtype)
    kw.update(override)
    res = gdn.chunk_gated_delta_rule(inp["q"], inp["k"], inp["v"], intermediates=intermediates,
                                     return_plan=True, **kw)
    res, plan, ws = res
    if check_status:
        bits = gdn.read_status(plan, ws)
        assert bits == 0, f"device status bits {bits:#x}"
    if kw.get("output_final_state"):
        out, fin = res
    else:
        out, fin = res, None
    torch.cuda.synchronize()
    r = {"output": out, "final_state": fin, "checkpoints": kw.get("state_checkpoints")}
    if return_plan:
        r["plan"], r["ws"] = plan, ws
    return r


def _np(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def run_oracle(inp, heads=None, threads=None):
    """fp64 oracle on CPU inputs `inp` (from workloads.generate).  With `heads`
    (a list of state heads) only those heads are computed, as an equal-head
    problem on the gathered q/k/v/g/beta heads."""
    H = inp["H"]
    hq, hk, hv = inp["q"].shape[1], inp["k"].shape[1], inp["v"].shape[1]
    q, k, v = _np(inp["q"]), _np(inp["k"]), _np(inp["v"])
    g, b = _np(inp["g"]), _np(inp["beta"])
    s0 = _np(inp.get("initial_state"))
    idx = None if inp.get("state_indices") is None else inp["state_indices"].numpy().astype(np.int64)
    if heads is not None:
        hs = list(heads)
        q = q[:, [h // (H // hq) for h in hs]]
        k = k[:, [h // (H // hk) for h in hs]]
        v = v[:, [h // (H // hv) for h in hs]]
        g, b = g[:, hs], b[:, hs]
        if s0 is not None:
            s0 = s0[:, hs]
    n = inp.get("checkpoint_every_n_tokens") or 0
    ccs = None if not n else inp["checkpoint_cu_starts"].numpy().astype(np.int64)
    return oracle.gdn_sequential(q, k, v, g, b, inp["cu_seqlens"].numpy().astype(np.int64), scale=inp["scale"],
                                 initial_state=s0, state_indices=idx, output_final_state=inp["output_final_state"],
                                 l2norm=inp["use_qk_l2norm_in_kernel"], checkpoint_every_n_tokens=n,
                                 checkpoint_cu_starts=ccs, threads=threads)


# Accuracy guard.  Besides the parity bar (the pages' tolerance), each GPU parity case must stay within four
# times the largest error max|d| / max|ref| it showed when the table was taken (floor 1e-4): a loss of accuracy
# that still passes the bar fails here.  The table holds errors of the CUDA path against the oracle, measured;
# it is a guard, not a reference (no expected value comes from it).  GDN_RECORD_MARGINS=<file> appends the
# errors of a run to <file> (JSON lines) instead of checking them; tests/accuracy_margins.py turns such a file
# into the table.
MARGINS_FILE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "accuracy_margins.json")
_margins = None


def _current_case():
    node = os.environ.get("PYTEST_CURRENT_TEST", "")
    return node.rsplit(" (", 1)[0]


def _accuracy_guard(name, stats):
    global _margins
    case = _current_case()
    rec = os.environ.get("GDN_RECORD_MARGINS")
    if rec:
        with open(rec, "a") as f:
            f.write(json.dumps({"case": case, "quantity": name, **stats}) + "\n")
        return
    if _margins is None:
        try:
            with open(MARGINS_FILE) as f:
                _margins = json.load(f)["margins"]
        except FileNotFoundError:
            _margins = {}
    m = _margins.get(case, {}).get(name)
    if m is not None:
        assert stats["rel_to_max"] <= m, (f"{name}: error max|d|/max|ref| = {stats['rel_to_max']:.3g} above the "
                                          f"accuracy guard {m:.3g} of {case}")


def compare(name, gpu, ref, tol, stored=None):
    """Elementwise |gpu - ref| <= tol + tol*|ref| (plus the fp8 rounding bound when the GPU result is stored
    in a narrower type `stored`: bf16, fp16 or fp8); returns stats, raises on failure."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, f"{name}: shape {gpu.shape} vs {ref.shape}"
    assert np.isfinite(gpu).all(), f"{name}: non-finite values from the CUDA path"
    d = np.abs(gpu - ref)
    bound = tol + tol * np.abs(ref)
    if stored in STORED:
        bound = bound + rounding_bound(np.abs(ref) + bound, stored)
    bad = d > bound
    stats = {"max_abs": float(d.max()) if d.size else 0.0,
             "rel_to_max": float(d.max() / max(np.abs(ref).max(), 1e-30)) if d.size else 0.0,
             "n_bad": int(bad.sum())}
    if bad.any():
        i = np.unravel_index(np.argmax(d - bound), d.shape)
        raise AssertionError(f"{name}: {stats['n_bad']} of {d.size} elements outside tol {tol}; worst at {i}: "
                             f"gpu={gpu[i]:.6g} ref={ref[i]:.6g}; max_abs={stats['max_abs']:.3g}")
    _accuracy_guard(name, stats)
    return stats


def check_against_oracle(inp_cpu, gpu_res, heads=None, tol=None):
    """Compare output / final state / checkpoints of a GPU run with the oracle."""
    tol = tol or TOL[inp_cpu["q"].dtype]
    ref = run_oracle(inp_cpu, heads=heads)
    H = inp_cpu["H"]
    hs = list(range(H)) if heads is None else list(heads)
    stats = {}
    stats["output"] = compare("output", _np(gpu_res["output"])[:, hs], ref["output"], tol)
    if inp_cpu["output_final_state"]:
        fin = _np(gpu_res["final_state"])[:, hs]
        stats["final_state"] = compare("final_state", fin, ref["final_state"], tol,
                                       stored=gpu_res["final_state"].dtype)
    if inp_cpu.get("checkpoint_every_n_tokens"):
        nck = ref["checkpoints"].shape[0]
        stats["checkpoints"] = compare("checkpoints", _np(gpu_res["checkpoints"])[:nck][:, hs], ref["checkpoints"],
                                       tol, stored=gpu_res["checkpoints"].dtype)
    return stats
