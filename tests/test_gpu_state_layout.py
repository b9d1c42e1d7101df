"""GPU parity of the state layouts: bf16 and fp16 states, and state pools with
strides other than the contiguous [rows][H][128][128].

FlashInfer GDN Prefill 完全指南 (requirements section) lists fp16/bf16 inputs
with fp32, fp16 or bf16 states and fp32 checkpoints.  A 16-bit state is read
into the fp32 recurrence and the final state is rounded back to its type; the
oracle runs on the same rounded initial values.  Strided pools (head-major,
padded rows) hold the same values as a contiguous one, and the results,
read back through the strides, must match the oracle's; rows the batch does
not name stay bit-identical.
"""
import pytest
import torch

import gated_deltanet_chunked_device_gb300 as gdn
from gated_deltanet_chunked_device_gb300 import workloads as wl
from gdn_testlib import TOL, check_against_oracle, compare, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.build()


@pytest.mark.parametrize("state_dtype", [torch.bfloat16, torch.float16])
def test_16bit_state_pool_prefill(state_dtype):
    w = wl.custom(seq_lens=[130, 0, 77, 64, 5], hq=2, hk=2, hv=4, initial_state="pool", n_pool=12,
                  l2norm_in_kernel=True, qk_prenorm=False, checkpoint_every=64)
    inp = wl.generate(w, seed=50)
    inp["initial_state"] = inp["initial_state"].to(state_dtype)
    res = run_gpu(to_device(inp))
    assert res["final_state"].dtype == state_dtype
    assert res["checkpoints"].dtype == torch.float32
    check_against_oracle(inp, res)
    named = set(inp["state_indices"].tolist())
    pool = res["final_state"].cpu()
    for r in range(pool.shape[0]):
        if r not in named:
            assert torch.equal(pool[r], inp["initial_state"][r])


@pytest.mark.parametrize("state_dtype", [torch.bfloat16, torch.float16])
def test_16bit_dense_state_prefill_new_output(state_dtype):
    # dense initial state, a new final-state tensor of the same type (allocated by the wrapper)
    w = wl.custom(seq_lens=[200, 3, 64], hq=4, hk=4, hv=4, initial_state="dense", alpha="exp_softplus16")
    inp = wl.generate(w, seed=51)
    inp["initial_state"] = inp["initial_state"].to(state_dtype)
    res = run_gpu(to_device(inp))
    assert res["final_state"].dtype == state_dtype
    check_against_oracle(inp, res)


@pytest.mark.parametrize("state_dtype", [torch.bfloat16, torch.float16])
def test_16bit_state_pool_decode(state_dtype):
    w = wl.custom(seq_lens=[2] * 30, hq=4, hk=4, hv=8, initial_state="pool", n_pool=40, l2norm_in_kernel=True,
                  qk_prenorm=False)
    inp = wl.generate(w, seed=52)
    inp["initial_state"] = inp["initial_state"].to(state_dtype)
    d = to_device(inp)
    pool = d["initial_state"].clone()
    out, fin = gdn.gated_delta_rule_decode(d["q"], d["k"], d["v"], g=d["g"], beta=d["beta"], scale=inp["scale"],
                                           initial_state=pool, state_indices=d["state_indices"],
                                           use_qk_l2norm_in_kernel=True, tokens_per_seq=2)
    torch.cuda.synchronize()
    assert fin.dtype == state_dtype and fin.data_ptr() == pool.data_ptr()
    check_against_oracle(inp, {"output": out, "final_state": fin})


def _strided_pool(values, layout):
    """A device pool with the given layout holding `values` [rows, H, 128, 128]."""
    rows, H = values.shape[:2]
    if layout == "head_major":
        base = torch.empty(H, rows, 128, 128, dtype=values.dtype, device="cuda")
        pool = base.permute(1, 0, 2, 3)
    elif layout == "padded_rows":
        base = torch.full((rows, H, 128, 136), float("nan"), dtype=values.dtype, device="cuda")
        pool = base[..., :128]
    else:
        raise ValueError(layout)
    pool.copy_(values.to("cuda"))
    assert not pool.is_contiguous()
    return base, pool


@pytest.mark.parametrize("layout", ["head_major", "padded_rows"])
@pytest.mark.parametrize("op", ["prefill", "decode"])
def test_strided_state_pool(layout, op):
    m = 3 if op == "decode" else None
    lens = [m] * 20 if op == "decode" else [150, 0, 64, 33]
    w = wl.custom(seq_lens=lens, hq=2, hk=2, hv=4, initial_state="pool", n_pool=24, l2norm_in_kernel=True,
                  qk_prenorm=False)
    inp = wl.generate(w, seed=53)
    d = to_device(inp)
    base, pool = _strided_pool(inp["initial_state"], layout)
    if op == "prefill":
        out, fin = gdn.chunk_gated_delta_rule(d["q"], d["k"], d["v"], g=d["g"], beta=d["beta"], scale=inp["scale"],
                                              initial_state=pool, output_state=pool, output_final_state=True,
                                              state_indices=d["state_indices"], cu_seqlens=d["cu_seqlens"],
                                              use_qk_l2norm_in_kernel=True)
    else:
        out, fin = gdn.gated_delta_rule_decode(d["q"], d["k"], d["v"], g=d["g"], beta=d["beta"], scale=inp["scale"],
                                               initial_state=pool, state_indices=d["state_indices"],
                                               use_qk_l2norm_in_kernel=True, tokens_per_seq=m)
    torch.cuda.synchronize()
    ref = run_oracle(inp)
    tol = TOL[torch.bfloat16]
    compare("output", out.cpu().double().numpy(), ref["output"], tol)
    compare("pool", pool.cpu().double().numpy(), ref["final_state"], tol)
    if layout == "padded_rows":  # the padding between rows is never written
        assert torch.isnan(base[..., 128:]).all()
    named = set(inp["state_indices"].tolist())
    for r in range(pool.shape[0]):
        if r not in named:
            assert torch.equal(pool[r].cpu(), inp["initial_state"][r])


# fp8 states and typed checkpoints ("FlashInfer GDN Prefill 完全指南": the initial_state row of the API table
# and the dtype requirement of "中间状态检查点" list float8_e4m3fn and float8_e5m2).  The fp8 initial values
# reach the fp32 recurrence exactly; a stored final state or checkpoint is the fp32 result rounded to nearest
# (ties to even, saturated), so its check adds the fp8 rounding bound to the parity bar.
FP8_TYPES = [torch.float8_e4m3fn, torch.float8_e5m2]


@pytest.mark.parametrize("state_dtype", FP8_TYPES)
def test_fp8_state_pool_prefill_with_fp8_checkpoints(state_dtype):
    w = wl.custom(seq_lens=[300, 0, 90, 64], hq=2, hk=2, hv=4, initial_state="pool", n_pool=10,
                  l2norm_in_kernel=True, qk_prenorm=False, checkpoint_every=64)
    inp = wl.generate(w, seed=54)
    inp["initial_state"] = inp["initial_state"].to(state_dtype)
    res = run_gpu(to_device(inp), ckpt_dtype=state_dtype)
    assert res["final_state"].dtype == state_dtype and res["checkpoints"].dtype == state_dtype
    check_against_oracle(inp, res)
    named = set(inp["state_indices"].tolist())
    pool = res["final_state"].cpu()
    for r in range(pool.shape[0]):
        if r not in named:  # rows the batch does not name keep their bytes
            assert torch.equal(pool[r].view(torch.uint8), inp["initial_state"][r].view(torch.uint8))


@pytest.mark.parametrize("ckpt_dtype", [torch.bfloat16, torch.float16] + FP8_TYPES)
def test_checkpoint_types_dense_state(ckpt_dtype):
    w = wl.custom(seq_lens=[260, 128, 7], hq=4, hk=4, hv=4, initial_state="dense", alpha="exp_softplus16",
                  checkpoint_every=128)
    inp = wl.generate(w, seed=55)
    res = run_gpu(to_device(inp), ckpt_dtype=ckpt_dtype)
    assert res["checkpoints"].dtype == ckpt_dtype and res["final_state"].dtype == torch.float32
    check_against_oracle(inp, res)


@pytest.mark.parametrize("state_dtype", FP8_TYPES)
def test_fp8_state_dense_new_output(state_dtype):
    w = wl.custom(seq_lens=[200, 3, 64], hq=4, hk=2, hv=2, initial_state="dense", alpha="u(0.9,1.0)")
    inp = wl.generate(w, seed=56)
    inp["initial_state"] = inp["initial_state"].to(state_dtype)
    res = run_gpu(to_device(inp))
    assert res["final_state"].dtype == state_dtype
    check_against_oracle(inp, res)


@pytest.mark.parametrize("state_dtype", FP8_TYPES)
def test_fp8_state_pool_decode(state_dtype):
    w = wl.custom(seq_lens=[3] * 24, hq=4, hk=4, hv=8, initial_state="pool", n_pool=32, l2norm_in_kernel=True,
                  qk_prenorm=False)
    inp = wl.generate(w, seed=57)
    inp["initial_state"] = inp["initial_state"].to(state_dtype)
    d = to_device(inp)
    pool = d["initial_state"].clone()
    out, fin = gdn.gated_delta_rule_decode(d["q"], d["k"], d["v"], g=d["g"], beta=d["beta"], scale=inp["scale"],
                                           initial_state=pool, state_indices=d["state_indices"],
                                           use_qk_l2norm_in_kernel=True, tokens_per_seq=3)
    torch.cuda.synchronize()
    assert fin.dtype == state_dtype and fin.data_ptr() == pool.data_ptr()
    check_against_oracle(inp, {"output": out, "final_state": fin})


def test_fp32_inputs_fp8_state_and_bf16_checkpoints():
    # the fp32-input kernel shares the typed state and checkpoint stores
    w = wl.custom(seq_lens=[192, 70], hq=2, hk=2, hv=2, dtype=torch.float32, initial_state="dense",
                  checkpoint_every=64, qk_prenorm=True)
    inp = wl.generate(w, seed=58)
    inp["initial_state"] = inp["initial_state"].to(torch.float8_e4m3fn)
    res = run_gpu(to_device(inp), ckpt_dtype=torch.bfloat16)
    assert res["final_state"].dtype == torch.float8_e4m3fn and res["checkpoints"].dtype == torch.bfloat16
    check_against_oracle(inp, res)  # the fp32 bar, plus each stored type's own rounding
