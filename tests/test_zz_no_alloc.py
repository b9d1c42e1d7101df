"""The entry point that allocates nothing (gdn_prefill_run_static).

Some callers cannot allocate device memory when they run the prefill (code
inside an allocator or memory-pool callback, or under a framework that owns
every allocation), so they cannot pass a workspace.  gdn_prefill_run_static
takes its workspace from a fixed array in the library's device globals.  This
file checks, through the C ABI, that two calls in a row give the same results
as the allocating entry point, and that a plan too large for the array is
refused before anything runs.  It sits last in collection order so that a run
stopping at the first failure has already run every other test.
"""
import pytest
import torch

import gated_deltanet_chunked_device_gb300 as gdn
from gated_deltanet_chunked_device_gb300 import workloads as wl
from gdn_testlib import TOL, compare

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else t.data_ptr()


def _args(inp, out, pool_out, ckpt, status):
    lens = inp["seq_lens"]
    return gdn.Args(q=_ptr(inp["q"]), k=_ptr(inp["k"]), v=_ptr(inp["v"]), g=_ptr(inp["g"]), beta=_ptr(inp["beta"]),
                    scale=float(inp["scale"]), cu_seqlens=_ptr(inp["cu_seqlens"]), num_seqs=len(lens),
                    total_tokens=inp["T"], max_seqlen=0, initial_state=_ptr(inp["initial_state"]),
                    output_state=_ptr(pool_out), n_pool=inp["initial_state"].shape[0],
                    state_indices=_ptr(inp["state_indices"]), state_checkpoints=_ptr(ckpt),
                    num_checkpoints=ckpt.shape[0], checkpoint_cu_starts=_ptr(inp["checkpoint_cu_starts"]),
                    output=_ptr(out), device_status=_ptr(status))


def test_static_workspace_matches_allocating_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.build()
    w = wl.custom(seq_lens=[130, 0, 20, 300, 64], hq=4, hk=4, hv=8, l2norm_in_kernel=True, qk_prenorm=False,
                  initial_state="pool", n_pool=9, checkpoint_every=64)
    cpu = wl.generate(w, seed=21)
    inp = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
    H, T = inp["H"], inp["T"]
    nck = wl.num_checkpoints(inp["seq_lens"], 64)

    def buffers():
        return (torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda"),
                inp["initial_state"].clone(), torch.zeros(nck, H, 128, 128, device="cuda"),
                torch.zeros(1, dtype=torch.int32, device="cuda"))

    # reference: the allocating entry point, out of place so the pool input stays as drawn
    out_ref, pool_ref, ck_ref, _ = buffers()
    (_, _), plan, _ws = gdn.chunk_gated_delta_rule(
        inp["q"], inp["k"], inp["v"], g=inp["g"], beta=inp["beta"], scale=inp["scale"],
        cu_seqlens=inp["cu_seqlens"], use_qk_l2norm_in_kernel=True, initial_state=inp["initial_state"],
        output_state=pool_ref, state_indices=inp["state_indices"], output_final_state=True, output=out_ref,
        checkpoint_every_n_tokens=64, checkpoint_cu_starts=inp["checkpoint_cu_starts"],
        state_checkpoints=ck_ref, return_plan=True)
    torch.cuda.synchronize()
    assert plan.workspace_bytes <= (1 << 20)  # fits GDN_PREFILL_STATIC_WORKSPACE_BYTES
    stream = torch.cuda.current_stream().cuda_stream
    tol = TOL[torch.bfloat16]
    for call in range(2):
        out, pool, ck, status = buffers()
        st = gdn.gdn_prefill_run_static(plan.handle, _args(inp, out, pool, ck, status), stream)
        assert st == 0, f"call {call}: {gdn.STATUS.get(st, st)}"
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        compare(f"output (call {call})", out.double().cpu().numpy(), out_ref.double().cpu().numpy(), tol)
        compare(f"pool (call {call})", pool.double().cpu().numpy(), pool_ref.double().cpu().numpy(), tol)
        compare(f"checkpoints (call {call})", ck.double().cpu().numpy(), ck_ref.double().cpu().numpy(), tol)


def test_static_workspace_refuses_plans_larger_than_the_array():
    gdn.build()
    desc = gdn.Desc(num_q_heads=4, num_k_heads=4, num_v_heads=4, head_size=128, qkv_dtype=gdn.DTYPE_BF16,
                    state_dtype=gdn.DTYPE_F32, max_total_tokens=1 << 27, max_num_seqs=1 << 16, max_pool_rows=0,
                    checkpoint_every_n_tokens=0, flags=0)
    st, plan, nbytes = gdn.gdn_prefill_plan(desc)
    assert st == 0 and nbytes > (1 << 20)
    try:
        args = gdn.Args(num_seqs=1, total_tokens=64)
        assert gdn.gdn_prefill_run_static(plan, args, 0) == 2  # GDN_ERR_UNSUPPORTED, before any launch
    finally:
        gdn.gdn_prefill_plan_destroy(plan)


def test_static_workspace_refuses_context_parallel_plans():
    # a plan that allows context parallelism needs its segment scratch (tens of MiB): the static entry
    # refuses it before any launch, as any plan above the array
    gdn.build()
    desc = gdn.Desc(num_q_heads=4, num_k_heads=4, num_v_heads=4, head_size=128, qkv_dtype=gdn.DTYPE_BF16,
                    state_dtype=gdn.DTYPE_F32, max_total_tokens=1 << 12, max_num_seqs=4, max_pool_rows=0,
                    checkpoint_every_n_tokens=0, flags=gdn.FLAGS["CONTEXT_PARALLEL"])
    st, plan, nbytes = gdn.gdn_prefill_plan(desc)
    assert st == 0 and nbytes > (1 << 20)
    try:
        args = gdn.Args(num_seqs=1, total_tokens=64)
        assert gdn.gdn_prefill_run_static(plan, args, 0) == 2  # GDN_ERR_UNSUPPORTED, before any launch
    finally:
        gdn.gdn_prefill_plan_destroy(plan)
