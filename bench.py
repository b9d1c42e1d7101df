#!/usr/bin/env python3
"""Benchmark of the chunked Gated DeltaNet prefill on GB300.

One step = one full prefill (prepare + chunk kernel: intra-chunk solve, state
pass, output, checkpoints) over the benchmark workload, inputs resident in HBM.
Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--seed S] [--no-cpu-baseline] [--op prefill|decode]

* value: tokens/s of the whole job (all ranks), device-timed with CUDA events,
  L2 flushed (256 MiB write) between steps, outside the timed events.
* roofline: the chunk kernel (the dominant kernel), timed alone with events on
  its own stream; algorithmic bytes per launch / its mean duration, against the
  measured HBM copy bandwidth.
* e2e: the same metric through the public API with host buffers: pinned-host
  inputs copied in and results copied out inside the timed region.
* cpu_baseline: the fp64 oracle (sequential recurrence, all host cores) on a
  bounded sample of the same workload (a subset of state heads), scaled to
  tokens/s of the whole workload.
* --impl reference: the oracle as the reference arm (host cores only).

--op decode times the decode step (gdn_decode_run) on a decode workload
(default decode_gva_512seq_bf16: 512 sequences, one token each, a pool of
1024 states) instead; its JSON line carries the same roofline and
cpu_baseline objects.

Multi-GPU: launched by torch.distributed.run, every rank runs its own replica
of the workload (units are independent: no data-path collective); only a
barrier and a max-reduction of the step time cross ranks ("scaling": "weak").
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gated_deltanet_chunked_device_gb300 as gdn  # noqa: E402
from gated_deltanet_chunked_device_gb300 import workloads as wl  # noqa: E402

METRIC = "GDN prefill tokens/s and TFLOP/s as % of GB300 dense BF16 roofline, 1 GPU"
FLOP_DENSE = 180224       # per token per state head: 10*C*D + 6*D^2, dense 64/128 tiles
FLOP_TRI = 140630         # per token per state head: triangular-aware count
# the arithmetic type each input type computes in, and the chunk kernel instance that runs it
DTYPE_NAMES = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}
CHUNK_KERNEL_NAMES = {torch.bfloat16: "gdn_chunk_kernel<__nv_bfloat16, false, false>",
                      torch.float16: "gdn_chunk_kernel<__half, false, false>",
                      torch.float32: "gdn_chunk_f32_kernel"}
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = ["gated_deltanet_chunked_device_gb300/csrc/gdn_chunk_bf16.cu",
                  "gated_deltanet_chunked_device_gb300/csrc/sm103_ptx.cuh",
                  "gated_deltanet_chunked_device_gb300/csrc/gdn_internal.cuh"]
DECODE_SOURCES = ["gated_deltanet_chunked_device_gb300/csrc/gdn_decode.cu",
                  "gated_deltanet_chunked_device_gb300/csrc/sm103_ptx.cuh",
                  "gated_deltanet_chunked_device_gb300/csrc/gdn_internal.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, dist=None, device=None):
    """The largest value of x over all ranks (x itself without a process group):
    the job's time is its slowest rank's."""
    if dist is None:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(copies, tokens_per_copy, ms):
    """Whole-job throughput: the job processes `copies` whole batches per step (replicas: every rank prefills its
    own copy, so copies = world; a head-split batch is one copy spread over the ranks)."""
    return copies * tokens_per_copy / (ms / 1e3)


def head_shard(H, hq, hk, hv, rank, world):
    """The heads rank `rank` of `world` takes when one batch is split by state head (the (sequence, head) units
    are independent: no exchange).  State heads [a, b) with b - a = H / world, and the q, k and v heads those
    read under the grouped head mapping (state head h reads q head h / (H / hq), and so on): each a contiguous
    range, so every rank runs the same problem shape with hq, hk, hv and H divided by `world`.  Raises when the
    head counts do not divide."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    for name, n in (("state", H), ("q", hq), ("k", hk), ("v", hv)):
        if n % world:
            raise ValueError(f"{n} {name} heads do not split over {world} ranks")
    per = {"h": H // world, "q": hq // world, "k": hk // world, "v": hv // world}
    return {key: (rank * n, (rank + 1) * n) for key, n in per.items()}


def shard_heads(w, inp, rank, world):
    """This rank's part of a head-split batch: the workload with its head counts divided and the inputs sliced
    (contiguous copies) to this rank's heads."""
    import dataclasses
    r = head_shard(inp["H"], w.hq, w.hk, w.hv, rank, world)
    out = dict(inp)
    for key, hk_ in (("q", "q"), ("k", "k"), ("v", "v")):
        a, b = r[hk_]
        out[key] = inp[key][:, a:b].contiguous()
    a, b = r["h"]
    out["g"] = inp["g"][:, a:b].contiguous()
    out["beta"] = inp["beta"][:, a:b].contiguous()
    if inp.get("initial_state") is not None:
        out["initial_state"] = inp["initial_state"][:, a:b].contiguous()
    out["H"] = b - a
    return dataclasses.replace(w, hq=w.hq // world, hk=w.hk // world, hv=w.hv // world), out


def algorithmic_bytes(w, inp):
    """Bytes the method must move once: q, k, v read, g and beta read, o written,
    initial / final states, checkpoints."""
    T, H, D = inp["T"], inp["H"], 128
    esz = inp["q"].element_size()
    b = T * (w.hq + w.hk + w.hv) * D * esz      # q, k, v
    b += T * H * 4 * 2                          # g, beta (fp32)
    b += T * H * D * esz                        # output
    N = len(inp["seq_lens"])
    state = H * D * D * storage_bytes(inp, "state_dtype")
    if inp.get("initial_state") is not None:
        b += N * state                          # rows read (pool: only the indexed rows)
    if inp["output_final_state"]:
        b += N * state
    n = inp.get("checkpoint_every_n_tokens") or 0
    if n:
        b += wl.num_checkpoints(inp["seq_lens"], n) * H * D * D * storage_bytes(inp, "checkpoint_dtype")
    return b


STORAGE_DTYPES = {"float32": torch.float32, "bfloat16": torch.bfloat16, "float16": torch.float16,
                  "float8_e4m3fn": torch.float8_e4m3fn, "float8_e5m2": torch.float8_e5m2}


def storage_bytes(inp, key):
    """Bytes per element of the states or checkpoints as stored (fp32 unless the run chose another type)."""
    return torch.empty(0, dtype=inp.get(key, torch.float32)).element_size()


def with_storage_types(inp, state_dtype=None, checkpoint_dtype=None):
    """The workload with its initial state (or pool) rounded to `state_dtype` and the final states and
    checkpoints to be stored in the given types; the oracle then reads the same rounded state."""
    inp = dict(inp)
    if state_dtype is not None:
        inp["state_dtype"] = STORAGE_DTYPES[state_dtype]
        if inp.get("initial_state") is not None:
            inp["initial_state"] = inp["initial_state"].to(inp["state_dtype"])
    if checkpoint_dtype is not None:
        inp["checkpoint_dtype"] = STORAGE_DTYPES[checkpoint_dtype]
    return inp


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:  # noqa: BLE001
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash(sources=KERNEL_SOURCES):
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, sources=KERNEL_SOURCES):
    """dram read+write bytes per launch of the workload's kernel from the
    committed ncu summary, if it was taken on the current kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        e = rec.get(workload)
        if e and e.get("kernel_source_hash") == kernel_source_hash(sources):
            return float(e["dram_bytes_per_launch"]), e.get("note")
    except Exception:  # noqa: BLE001
        pass
    return None, None


class ClockSampler:
    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        self.t_start = self.t_end = None
        try:
            props = torch.cuda.get_device_properties(device_index)
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
        except Exception:  # noqa: BLE001
            bus = None
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits", "-lms", "100"]
        if bus:
            cmd += ["-i", bus]
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:  # noqa: BLE001
            self.proc = None

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:  # noqa: BLE001
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) != len(self.FIELDS):
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[5:]))
                except Exception:  # noqa: BLE001
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        lo, hi = (self.t_start or 0) - 1.0, (self.t_end or 1e30) + 1.0
        inside = [r for r in rows if lo <= r[0] <= hi] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


def make_call(inp, device, use_cp=False):
    """Device buffers and C-ABI arguments for one prefill of `inp`."""
    d = {k: (v.to(device).contiguous() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    T, H = inp["T"], inp["H"]
    N = len(inp["seq_lens"])
    out = torch.empty(T, H, 128, dtype=d["q"].dtype, device=device)
    fin = (torch.empty(N, H, 128, 128, dtype=inp.get("state_dtype", torch.float32), device=device)
           if inp["output_final_state"] else None)
    n = inp.get("checkpoint_every_n_tokens") or 0
    ck = torch.empty(max(wl.num_checkpoints(inp["seq_lens"], n), 1), H, 128, 128,
                     dtype=inp.get("checkpoint_dtype", torch.float32), device=device) if n else None
    kw = dict(g=d["g"], beta=d["beta"], scale=inp["scale"], cu_seqlens=d["cu_seqlens"],
              use_qk_l2norm_in_kernel=inp["use_qk_l2norm_in_kernel"], output=out,
              initial_state=d.get("initial_state"), output_final_state=inp["output_final_state"], output_state=fin,
              state_indices=d.get("state_indices"), checkpoint_every_n_tokens=n,
              checkpoint_cu_starts=d.get("checkpoint_cu_starts"), state_checkpoints=ck, use_cp=use_cp)
    if d.get("state_indices") is not None:
        kw["output_state"] = d["initial_state"]
    # One eager call builds the plan and the workspace, and checks the device status.
    _, plan, ws = gdn.chunk_gated_delta_rule(d["q"], d["k"], d["v"], return_plan=True, **kw)
    bits = gdn.read_status(plan, ws)
    if bits:
        raise RuntimeError(f"device status bits {bits:#x} on the benchmark input")
    st = inp.get("initial_state")
    args = gdn.Args(q=d["q"].data_ptr(), k=d["k"].data_ptr(), v=d["v"].data_ptr(), g=d["g"].data_ptr(),
                    beta=d["beta"].data_ptr(), scale=float(inp["scale"]), cu_seqlens=d["cu_seqlens"].data_ptr(),
                    num_seqs=N, total_tokens=T, max_seqlen=max(inp["seq_lens"]) if N else 0,
                    initial_state=d["initial_state"].data_ptr() if st is not None else None,
                    output_state=(kw["output_state"].data_ptr() if inp["output_final_state"] else None),
                    n_pool=(st.shape[0] if d.get("state_indices") is not None else 0),
                    state_indices=d["state_indices"].data_ptr() if d.get("state_indices") is not None else None,
                    state_checkpoints=ck.data_ptr() if ck is not None else None,
                    num_checkpoints=ck.shape[0] if ck is not None else 0,
                    checkpoint_cu_starts=d["checkpoint_cu_starts"].data_ptr() if n else None,
                    output=out.data_ptr())
    return {"dev": d, "out": out, "fin": fin, "ck": ck, "plan": plan, "ws": ws, "args": args, "kw": kw}


def cpu_baseline(inp, budget_s=15.0):
    """Time the fp64 oracle on a sample of state heads (all sequences, all tokens)."""
    import oracle
    import numpy as np

    H = inp["H"]
    threads = oracle.default_threads()

    def run_heads(nh):
        hs = list(range(nh))
        hq, hk, hv = inp["q"].shape[1], inp["k"].shape[1], inp["v"].shape[1]
        f64 = lambda t: t.to(torch.float64).numpy()
        q = f64(inp["q"])[:, [h // (H // hq) for h in hs]]
        k = f64(inp["k"])[:, [h // (H // hk) for h in hs]]
        v = f64(inp["v"])[:, [h // (H // hv) for h in hs]]
        g, b = f64(inp["g"])[:, hs], f64(inp["beta"])[:, hs]
        s0, idx = None, None
        if inp.get("initial_state") is not None:
            st = inp["initial_state"]
            if inp.get("state_indices") is not None:  # only the named pool rows, renumbered in order
                st = st[inp["state_indices"].long()]
                idx = np.arange(st.shape[0], dtype=np.int64)
            s0 = f64(st[:, hs])
        n = inp.get("checkpoint_every_n_tokens") or 0
        ccs = None if not n else inp["checkpoint_cu_starts"].numpy().astype(np.int64)
        t0 = time.perf_counter()
        oracle.gdn_sequential(q, k, v, g, b, inp["cu_seqlens"].numpy().astype(np.int64), scale=inp["scale"],
                              initial_state=s0, state_indices=idx, output_final_state=inp["output_final_state"],
                              l2norm=inp["use_qk_l2norm_in_kernel"], checkpoint_every_n_tokens=n,
                              checkpoint_cu_starts=ccs, threads=threads)
        return time.perf_counter() - t0

    t1 = run_heads(1)
    nh = max(1, min(H, int(budget_s / max(t1, 1e-3))))
    # repeat the sampled heads until the sample holds about `budget_s` of CPU work
    reps, t = 0, 0.0
    while reps == 0 or (t < budget_s and reps < 64):
        t += run_heads(nh)
        reps += 1
    value = inp["T"] * nh * reps / t / H
    return {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{nh} of {H} state heads x {reps} repetitions, all {len(inp['seq_lens'])} sequences "
                      f"({inp['T']} tokens), fp64 sequential recurrence, {t:.1f} s; scaled to whole-workload "
                      f"tokens/s (x {H}/{nh} heads)"}


def run_reference(args, w, inp):
    """The oracle as the reference arm: host cores only, bounded samples."""
    steps, warmup = args.steps, args.warmup
    H = inp["H"]
    import oracle
    import numpy as np
    threads = oracle.default_threads()
    hq, hk, hv = inp["q"].shape[1], inp["k"].shape[1], inp["v"].shape[1]
    f64 = lambda t: t.to(torch.float64).numpy()
    qa, ka, va, ga, ba = f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["g"]), f64(inp["beta"])
    n = inp.get("checkpoint_every_n_tokens") or 0
    ccs = None if not n else inp["checkpoint_cu_starts"].numpy().astype(np.int64)
    cu = inp["cu_seqlens"].numpy().astype(np.int64)

    def one(nh, h0=0):
        hs = [(h0 + i) % H for i in range(nh)]
        t0 = time.perf_counter()
        oracle.gdn_sequential(qa[:, [h // (H // hq) for h in hs]], ka[:, [h // (H // hk) for h in hs]],
                              va[:, [h // (H // hv) for h in hs]], ga[:, hs], ba[:, hs], cu, scale=inp["scale"],
                              output_final_state=inp["output_final_state"], l2norm=inp["use_qk_l2norm_in_kernel"],
                              checkpoint_every_n_tokens=n, checkpoint_cu_starts=ccs, threads=threads)
        return time.perf_counter() - t0

    t1 = one(1)
    budget = float(os.environ.get("GDN_REFERENCE_STEP_SECONDS", "6"))
    nh = max(1, min(H, int(budget / max(t1, 1e-3))))
    for i in range(warmup):
        one(nh, i)
    times = [one(nh, warmup + i) for i in range(steps)]
    step_s = sum(times) / len(times)
    value = inp["T"] * nh / step_s / H
    sample = f"{nh} of {H} state heads per step, all sequences, fp64 sequential recurrence"
    line = {"metric": METRIC, "impl": "reference", "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": warmup, "ms_per_step": step_s * 1e3 * H / nh, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, inp, args),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def decode_bytes(w, inp):
    """Bytes a decode step must move: every named state read and written,
    q, k, v and g, beta read, o written, the pool indices read."""
    T, H, D = inp["T"], inp["H"], 128
    N = len(inp["seq_lens"])
    esz = inp["q"].element_size()
    return (2 * N * H * D * D * storage_bytes(inp, "state_dtype") + T * (w.hq + w.hk + w.hv) * D * esz
            + T * H * 8 + T * H * D * esz
            + (N * 4 if inp.get("state_indices") is not None else 0))


def run_decode_bench(args, w, inp, device):
    m = inp["seq_lens"][0]
    if any(x != m for x in inp["seq_lens"]):
        raise SystemExit("--op decode needs a workload whose sequences all have the same length")
    d = {k: (v.to(device).contiguous() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    status = torch.zeros(1, dtype=torch.int32, device=device)
    pool = d["initial_state"]
    out, _ = gdn.gated_delta_rule_decode(d["q"], d["k"], d["v"], g=d["g"], beta=d["beta"], scale=inp["scale"],
                                         initial_state=pool, state_indices=d.get("state_indices"),
                                         use_qk_l2norm_in_kernel=inp["use_qk_l2norm_in_kernel"],
                                         tokens_per_seq=m, device_status=status)
    torch.cuda.synchronize(device)
    if int(status.item()):
        raise RuntimeError(f"device status bits {int(status.item()):#x} on the decode workload")
    N, T, H = len(inp["seq_lens"]), inp["T"], inp["H"]
    plan = gdn.get_plan(w.hq, w.hk, w.hv, gdn.DTYPE_BF16 if inp["q"].dtype == torch.bfloat16 else gdn.DTYPE_F32,
                        gdn.FLAGS["HAS_G"] | gdn.FLAGS["HAS_BETA"] | gdn.FLAGS["HAS_SCALE"] |
                        (gdn.FLAGS["QK_L2NORM"] if inp["use_qk_l2norm_in_kernel"] else 0) |
                        gdn.FLAGS["HAS_INITIAL_STATE"] | gdn.FLAGS["OUTPUT_FINAL_STATE"] |
                        gdn.FLAGS["HAS_STATE_INDICES"], 0, T, N, pool.shape[0],
                        state_dtype=gdn._STATE_DTYPES[pool.dtype])
    cargs = gdn.Args(q=d["q"].data_ptr(), k=d["k"].data_ptr(), v=d["v"].data_ptr(), g=d["g"].data_ptr(),
                     beta=d["beta"].data_ptr(), scale=float(inp["scale"]), num_seqs=N, total_tokens=T,
                     initial_state=pool.data_ptr(), output_state=pool.data_ptr(), n_pool=pool.shape[0],
                     state_indices=d["state_indices"].data_ptr(), output=out.data_ptr(),
                     device_status=status.data_ptr())
    stream = torch.cuda.Stream(device)
    sp = stream.cuda_stream

    def step():
        st = gdn.gdn_decode_run(plan.handle, cargs, m, sp)
        if st:
            raise RuntimeError(f"gdn_decode_run returned {st}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    sampler = ClockSampler(device.index or 0)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark_start()
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    sampler.mark_end()
    ms = e0.elapsed_time(e1) / K
    clocks = sampler.stop()
    if int(status.item()):
        raise RuntimeError(f"device status bits {int(status.item()):#x} after the timed steps")
    hbm, _, src = measured_peaks()
    abytes = decode_bytes(w, inp)
    achieved = abytes / (ms / 1e3) / 1e9
    line = {"metric": "GDN decode step tokens/s, 1 GPU", "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
            "steps": K, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if inp["q"].dtype == torch.bfloat16 else "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "op": "decode", "num_seqs": N, "tokens_per_seq": m,
                       "num_q_heads": w.hq, "num_k_heads": w.hk, "num_v_heads": w.hv, "state_heads": H,
                       "pool_rows": pool.shape[0], "qk_l2norm_in_kernel": w.l2norm_in_kernel,
                       **storage_config(inp),
                       "l2": f"inputs larger than L2 ({abytes / 2**20:.0f} MiB moved per step), no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": (None if "state_dtype" in inp
                                     else recorded_traffic(w.name, DECODE_SOURCES)[0]),
                         "kernel": "gdn_decode_kernel",
                         "kernel_ms": ms,
                         "algorithmic_bytes": abytes, "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)"},
            "gpu_launches": K}
    if clocks:
        line["clocks"] = clocks
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp)
    print(json.dumps(line), flush=True)


def storage_config(inp):
    """Config keys for storage types other than the default fp32 (absent otherwise)."""
    return {k: str(inp[k]).replace("torch.", "") for k in ("state_dtype", "checkpoint_dtype") if k in inp}


def workload_config(w, inp, args):
    return {"workload": w.name, "total_tokens": inp["T"], "num_seqs": len(inp["seq_lens"]),
            "seq_lens": inp["seq_lens"] if len(inp["seq_lens"]) <= 16 else f"{len(inp['seq_lens'])} sequences",
            "num_q_heads": w.hq, "num_k_heads": w.hk, "num_v_heads": w.hv, "state_heads": inp["H"],
            "head_size": 128, "chunk": 64, "checkpoint_every_n_tokens": w.checkpoint_every,
            "qk_l2norm_in_kernel": w.l2norm_in_kernel, "seed": args.seed,
            "l2": "flushed between steps (256 MiB write outside the timed events)", **storage_config(inp)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.BENCH_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--op", choices=["prefill", "decode"], default="prefill")
    ap.add_argument("--cp", action="store_true", help="allow context parallelism (few (sequence, head) units)")
    ap.add_argument("--shard", choices=["replica", "heads"], default="replica",
                    help="multi-GPU: every rank runs its own copy of the batch (weak scaling), or the ranks split "
                         "one batch's state heads (strong scaling); no data-path collective either way")
    ap.add_argument("--state-dtype", choices=sorted(STORAGE_DTYPES), default=None,
                    help="store the initial / final states (or the pool) in this type (default fp32)")
    ap.add_argument("--checkpoint-dtype", choices=sorted(STORAGE_DTYPES), default=None,
                    help="store the checkpoints in this type (default fp32)")
    args = ap.parse_args()
    world, rank, local = dist_env()
    if args.op == "decode" and args.workload == wl.BENCH_WORKLOAD:
        args.workload = "decode_gva_512seq_bf16"
    w = wl.WORKLOADS[args.workload]
    inp = with_storage_types(wl.generate(w, seed=args.seed), args.state_dtype, args.checkpoint_dtype)
    full_batches = world if args.shard == "replica" else 1  # copies of the whole batch the job runs per step
    tokens_batch = inp["T"]
    if args.shard == "heads" and world > 1 and args.impl == "ours":
        w, inp = shard_heads(w, inp, rank, world)

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w, inp)
        return

    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        pg = dist
    gdn.build()
    if args.op == "decode":
        if rank == 0:
            run_decode_bench(args, w, inp, device)
        return
    call = make_call(inp, device, use_cp=args.cp)
    plan, ws, cargs = call["plan"], call["ws"], call["args"]
    cp_segments = gdn.gdn_prefill_cp_segments(plan.handle, inp["seq_lens"], 0)[0] if args.cp else 0
    # the context-parallel launches run whenever the plan allows them, unless max_seqlen (passed by make_call)
    # already rules out any gain: 0.85 ceil(max_seqlen / 64) <= H T / (64 S), as the header states
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    cmax = -(-max(inp["seq_lens"]) // 64) if inp["seq_lens"] else 0
    cp_route = bool(args.cp and w.dtype != torch.float32 and 85 * cmax * 64 * sms > 100 * inp["H"] * inp["T"])
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)
    sp = stream.cuda_stream

    def step(e0=None, e1=None, e2=None):
        if e0 is not None:
            e0.record(stream)
        st = gdn.gdn_prefill_prepare(plan.handle, cargs, ws.data_ptr(), plan.workspace_bytes, sp)
        if e1 is not None:
            e1.record(stream)
        st |= gdn.gdn_prefill_chunks(plan.handle, cargs, ws.data_ptr(), plan.workspace_bytes, sp)
        if e2 is not None:
            e2.record(stream)
        if st:
            raise RuntimeError(f"gdn_prefill returned {st}")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1.0)
            step()
    torch.cuda.synchronize(device)

    sampler = ClockSampler(local) if rank == 0 else None
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize(device)
    if sampler:
        sampler.mark_start()
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush.fill_(float(i))
            step(*ev[i])
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - wall0
    if pg:
        pg.barrier()
    if sampler:
        sampler.mark_end()
    step_ms = [ev[i][0].elapsed_time(ev[i][2]) for i in range(K)]
    chunk_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    ms_per_step = sum(step_ms) / K
    chunk_avg_ms = sum(chunk_ms) / K
    ms_per_step = max_over_ranks(ms_per_step, pg, device)
    bits = gdn.read_status(plan, ws)
    if bits:
        raise RuntimeError(f"device status bits {bits:#x} after the timed steps")
    # the same steps back to back without the L2 flush (inputs partly L2-resident), outside the timed region
    Ku = min(K, 50)
    evu = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(Ku)]
    with torch.cuda.stream(stream):
        for i in range(Ku):
            step(*evu[i])
    torch.cuda.synchronize(device)
    unflushed_ms = sum(evu[i][0].elapsed_time(evu[i][2]) for i in range(Ku)) / Ku

    # ---- end to end through the public API, host buffers: every step copies its inputs in from pinned host
    #      memory and its results out.  Two sets of device buffers and three streams (copy in, compute, copy
    #      out) let step i's copy-in and step i-1's copy-out run while step i-1 / step i compute: the two
    #      directions and the compute overlap, the computes stay in order on one stream (one workspace).
    e2e = None
    if not args.no_e2e:
        sets = [call, make_call(inp, device, use_cp=args.cp)]
        in_keys = [k for k in ("q", "k", "v", "g", "beta", "cu_seqlens", "checkpoint_cu_starts", "initial_state",
                               "state_indices") if inp.get(k) is not None]
        host_in = {k: inp[k].pin_memory() for k in in_keys}

        def outs(c):
            o = {"output": c["out"]}
            if c["ck"] is not None:
                o["checkpoints"] = c["ck"]
            if c["fin"] is not None or inp.get("state_indices") is not None:
                o["final_state"] = c["kw"]["output_state"]
            return o

        host_out = {k: torch.empty_like(t, device="cpu").pin_memory() for k, t in outs(call).items()}
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
        ev_in = [torch.cuda.Event() for _ in sets]
        ev_done = [torch.cuda.Event() for _ in sets]
        ev_free = [torch.cuda.Event() for _ in sets]
        for e in ev_free:
            e.record(stream)
        Ke = max(3, min(K, 50))

        def e2e_step(i):
            b = i % 2
            c = sets[b]
            s_in.wait_event(ev_free[b])                 # set b's previous results have been copied out
            with torch.cuda.stream(s_in):
                for k2, t in host_in.items():
                    c["dev"][k2].copy_(t, non_blocking=True)
            ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            st = gdn.gdn_prefill_prepare(c["plan"].handle, c["args"], c["ws"].data_ptr(),
                                         c["plan"].workspace_bytes, sp)
            st |= gdn.gdn_prefill_chunks(c["plan"].handle, c["args"], c["ws"].data_ptr(),
                                         c["plan"].workspace_bytes, sp)
            if st:
                raise RuntimeError(f"gdn_prefill returned {st}")
            ev_done[b].record(stream)
            s_out.wait_event(ev_done[b])
            with torch.cuda.stream(s_out):
                for k2, t in outs(c).items():
                    host_out[k2].copy_(t, non_blocking=True)
            ev_free[b].record(s_out)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(device)
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        es.record(s_in)
        for i in range(Ke):
            e2e_step(i)
        ee.record(s_out)
        torch.cuda.synchronize(device)
        e2e_ms = es.elapsed_time(ee) / Ke
        e2e_ms = max_over_ranks(e2e_ms, pg, device)
        e2e = {"value": job_tokens_per_s(full_batches, tokens_batch, e2e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "link_gb_per_s": (h2d + d2h) / (e2e_ms / 1e3) / 1e9,
               "pipelined": "two buffer sets; copy-in, compute and copy-out streams overlap"}

    clocks = sampler.stop() if sampler else None
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return
    T, H = inp["T"], inp["H"]
    hbm, bf16, src = measured_peaks()
    abytes = algorithmic_bytes(w, inp)
    achieved = abytes / (chunk_avg_ms / 1e3) / 1e9
    traffic, tnote = recorded_traffic(w.name) if not storage_config(inp) else (None, None)
    tflops_dense = T * H * FLOP_DENSE / (ms_per_step / 1e3) / 1e12
    tflops_tri = T * H * FLOP_TRI / (ms_per_step / 1e3) / 1e12
    roof_time = max(abytes / (hbm * 1e9), T * H * FLOP_DENSE / (bf16 * 1e12))
    line = {
        "metric": METRIC, "value": job_tokens_per_s(full_batches, tokens_batch, ms_per_step), "unit": "tokens/s",
        "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak" if args.shard == "replica" else "strong",
        "vs_baseline": None, "dtype": DTYPE_NAMES[w.dtype], "data": "synthetic",
        "config": dict(workload_config(w, inp, args), context_parallel_segments=cp_segments,
                       parallelism=(f"replicas{world}" if args.shard == "replica" else f"heads{world}")),
        "tflops": {"dense_tile_count": tflops_dense, "triangular_aware": tflops_tri,
                   "pct_of_bf16_peak": 100 * tflops_dense / bf16, "peak_tflops": bf16, "peak_source": src},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic if not cp_segments else None,
                     "kernel": (CHUNK_KERNEL_NAMES[w.dtype] if not cp_segments
                                else "chunk stage with context parallelism (transfer pass, scan, segment pass)"),
                     "kernel_ms": chunk_avg_ms,
                     "algorithmic_bytes": abytes, "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)"
                     if src == "measured" else "fallback 6800 GB/s",
                     "step_frac_of_roofline_time": roof_time / (ms_per_step / 1e3)},
        # prepare + chunk kernel; on the context-parallel route the chunk stage is cp_prepare, the transfer
        # pass, the scan, the segment prepare, the segment pass and (with a final state) the state copy
        "gpu_launches": K * ((6 + (1 if inp["output_final_state"] else 0)) if cp_route else 2),
        "wall_s_timed_region": wall,
        "step_ms_stats": {"mean": sum(step_ms) / K, "median": statistics.median(step_ms), "min": min(step_ms),
                          "max": max(step_ms), "unflushed_mean": unflushed_ms, "unflushed_steps": Ku},
    }
    if tnote:
        line["roofline"]["traffic_note"] = tnote
    if e2e:
        line["e2e"] = e2e
    if clocks:
        line["clocks"] = clocks
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp)
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
