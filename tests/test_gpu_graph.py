"""CUDA-Graph capture and replay of the prefill and decode calls.

gdn_prefill_run and gdn_decode_run only enqueue kernels: no allocation, no
synchronisation and no host read of device memory, so a serving loop can
capture them once and replay them with new data in the same buffers.  These
tests capture each call into a graph, refill the inputs in place, replay, and
require the replay to equal an eager call on the new inputs bit for bit (each
(sequence, head) unit is computed the same way whichever CTA takes it), and
the replayed results to match the fp64 oracle on those inputs.  The
context-parallel path (transfer pass, scan, segment pass, final copy) is
captured the same way ("FlashInfer GDN Prefill 完全指南", the section on plan
caching, address rebinding and CUDA Graph replay)."""
import pytest
import torch

import gated_deltanet_chunked_device_gb300 as gdn
from gated_deltanet_chunked_device_gb300 import workloads as wl
from gdn_testlib import check_against_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.build()


def _refill(dst, src):
    for key in ("q", "k", "v", "g", "beta", "state_indices"):
        if dst.get(key) is not None:
            dst[key].copy_(src[key])


def test_prefill_graph_replay_matches_eager():
    w = wl.custom(seq_lens=[300, 0, 77, 130], hq=4, hk=4, hv=8, initial_state="dense", l2norm_in_kernel=True,
                  qk_prenorm=False, checkpoint_every=64)
    b_cpu = wl.generate(w, seed=41)
    a, b = to_device(wl.generate(w, seed=40)), to_device(b_cpu)
    ck = torch.zeros(wl.num_checkpoints(a["seq_lens"], 64), a["H"], 128, 128, device="cuda")
    out = torch.empty(a["T"], a["H"], 128, dtype=a["q"].dtype, device="cuda")
    fin = torch.empty_like(a["initial_state"])

    def call(d, stream_out, stream_fin, stream_ck):
        return gdn.chunk_gated_delta_rule(
            d["q"], d["k"], d["v"], g=d["g"], beta=d["beta"], scale=d["scale"], initial_state=d["initial_state"],
            output_final_state=True, cu_seqlens=d["cu_seqlens"], use_qk_l2norm_in_kernel=True, output=stream_out,
            output_state=stream_fin, state_checkpoints=stream_ck, checkpoint_cu_starts=d["checkpoint_cu_starts"],
            checkpoint_every_n_tokens=64)

    live = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in a.items()}
    call(live, out, fin, ck)  # eager warm-up: plan, workspace, one-time kernel attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(live, out, fin, ck)
    _refill(live, b)
    live["initial_state"].copy_(b["initial_state"])
    g.replay()
    torch.cuda.synchronize()
    out_e, fin_e, ck_e = torch.empty_like(out), torch.empty_like(fin), torch.zeros_like(ck)
    call(b, out_e, fin_e, ck_e)
    torch.cuda.synchronize()
    assert torch.equal(out, out_e)
    assert torch.equal(fin, fin_e)
    assert torch.equal(ck, ck_e)
    check_against_oracle(b_cpu, {"output": out, "final_state": fin, "checkpoints": ck})


def test_context_parallel_graph_replay_matches_eager_and_oracle():
    # one long sequence beside a short one: the long one runs as segments, the short one whole, and all the
    # launches go into one graph.  The replay swaps the two lengths (same total): the segments are cut on the
    # device from cu_seqlens, so the captured graph follows the new batch without being captured again.
    w = wl.custom(seq_lens=[1500, 70], hq=2, hk=2, hv=2, initial_state="dense", l2norm_in_kernel=True,
                  qk_prenorm=False, checkpoint_every=128)
    w2 = wl.custom(seq_lens=[70, 1500], hq=2, hk=2, hv=2, initial_state="dense", l2norm_in_kernel=True,
                   qk_prenorm=False, checkpoint_every=128)
    b_cpu = wl.generate(w2, seed=48)
    a, b = to_device(wl.generate(w, seed=47)), to_device(b_cpu)
    ck = torch.zeros(wl.num_checkpoints(a["seq_lens"], 128), a["H"], 128, 128, device="cuda")
    out = torch.empty(a["T"], a["H"], 128, dtype=a["q"].dtype, device="cuda")
    fin = torch.empty_like(a["initial_state"])

    def call(d, out_, fin_, ck_, return_plan=False):
        return gdn.chunk_gated_delta_rule(
            d["q"], d["k"], d["v"], g=d["g"], beta=d["beta"], scale=d["scale"], initial_state=d["initial_state"],
            output_final_state=True, cu_seqlens=d["cu_seqlens"], use_qk_l2norm_in_kernel=True, output=out_,
            output_state=fin_, state_checkpoints=ck_, checkpoint_cu_starts=d["checkpoint_cu_starts"],
            checkpoint_every_n_tokens=128, use_cp=True, return_plan=return_plan)

    live = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in a.items()}
    _, plan, _ = call(live, out, fin, ck, return_plan=True)  # eager: plan, workspace, kernel attributes
    assert gdn.gdn_prefill_cp_segments(plan.handle, a["seq_lens"], 0)[1][1] == 1
    assert gdn.gdn_prefill_cp_segments(plan.handle, a["seq_lens"], 0)[1][0] >= 2
    assert gdn.gdn_prefill_cp_segments(plan.handle, b["seq_lens"], 0)[1][0] == 1
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(live, out, fin, ck)
    _refill(live, b)
    for key in ("initial_state", "cu_seqlens", "checkpoint_cu_starts"):
        live[key].copy_(b[key])
    g.replay()
    torch.cuda.synchronize()
    out_e, fin_e, ck_e = torch.empty_like(out), torch.empty_like(fin), torch.zeros_like(ck)
    call(b, out_e, fin_e, ck_e)
    torch.cuda.synchronize()
    assert torch.equal(out, out_e) and torch.equal(fin, fin_e) and torch.equal(ck, ck_e)
    check_against_oracle(b_cpu, {"output": out, "final_state": fin, "checkpoints": ck})


def test_decode_graph_replay_matches_eager():
    w = wl.custom(seq_lens=[1] * 40, hq=8, hk=8, hv=16, initial_state="pool", n_pool=64, l2norm_in_kernel=True,
                  qk_prenorm=False)
    b_cpu = wl.generate(w, seed=43)
    a, b = to_device(wl.generate(w, seed=42)), to_device(b_cpu)
    pool = a["initial_state"].clone()
    out = torch.empty(a["T"], a["H"], 128, dtype=a["q"].dtype, device="cuda")
    live = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in a.items()}

    def call(d, pool_, out_):
        return gdn.gated_delta_rule_decode(d["q"], d["k"], d["v"], g=d["g"], beta=d["beta"], scale=d["scale"],
                                           initial_state=pool_, state_indices=d["state_indices"],
                                           use_qk_l2norm_in_kernel=True, output=out_)

    call(live, pool, out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(live, pool, out)
    _refill(live, b)
    pool.copy_(b["initial_state"])
    g.replay()
    torch.cuda.synchronize()
    pool_e, out_e = b["initial_state"].clone(), torch.empty_like(out)
    call(b, pool_e, out_e)
    torch.cuda.synchronize()
    assert torch.equal(out, out_e)
    assert torch.equal(pool, pool_e)
    check_against_oracle(b_cpu, {"output": out, "final_state": pool})


def test_one_plan_serves_rotating_buffers_and_smaller_batches():
    # The plan holds shapes and flags only: the same plan runs over two rotating sets of buffers (different
    # addresses) and over a smaller batch that fits its bounds, each result equal to the oracle's.
    from gdn_testlib import check_against_oracle, run_gpu
    gdn._plans.clear()
    big = wl.custom(seq_lens=[200, 64, 7], hq=2, hk=2, hv=4, initial_state="dense", l2norm_in_kernel=True,
                    qk_prenorm=False)
    small = wl.custom(seq_lens=[90, 3], hq=2, hk=2, hv=4, initial_state="dense", l2norm_in_kernel=True,
                      qk_prenorm=False)
    cases = [wl.generate(big, seed=44), wl.generate(big, seed=45), wl.generate(small, seed=46)]
    plans, live = set(), []
    for inp in cases:
        live.append(to_device(inp))  # kept alive: every run sees buffers at new addresses
        check_against_oracle(inp, run_gpu(live[-1]))
        plans.update(id(p) for p in gdn._plans.values())
    assert len(gdn._plans) == 1 and len(plans) == 1
    assert len({d["q"].data_ptr() for d in live}) == 3
