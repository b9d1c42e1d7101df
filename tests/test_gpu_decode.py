"""GPU parity of the decode step (gdn_decode_run) against the fp64 oracle.

A decode batch is N sequences of m tokens each; the oracle runs the per-token
recurrence on the same seeded inputs with cu_seqlens = [0, m, 2m, ...].
Covered: one token and several tokens per sequence, GVA and GQA head
mappings, the state pool in place (untouched rows bit-identical), a dense
initial state, a zero state, the in-kernel L2 norm, fp32 inputs, decode after
a prefill against the oracle on the whole sequence, and an out-of-range pool
index (skipped, flagged in the status word).
"""
import numpy as np
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


def run_decode(inp, m, check_status=True):
    d = to_device(inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = d.get("state_indices") is not None
    st = d["initial_state"].clone() if d.get("initial_state") is not None else None
    out, fin = gdn.gated_delta_rule_decode(
        d["q"], d["k"], d["v"], g=d["g"], beta=d["beta"], scale=inp["scale"], initial_state=st,
        state_indices=d.get("state_indices"), output_final_state=True,
        use_qk_l2norm_in_kernel=inp["use_qk_l2norm_in_kernel"], tokens_per_seq=m, device_status=status)
    torch.cuda.synchronize()
    if check_status:
        assert int(status.item()) == 0
    return {"output": out, "final_state": fin, "pool": pool, "status": int(status.item())}


@pytest.mark.parametrize("m", [1, 3])
@pytest.mark.parametrize("hq,hk,hv", [(16, 16, 32), (32, 16, 16), (4, 4, 4)])
def test_decode_pool_in_place(m, hq, hk, hv):
    n = 37
    w = wl.custom(seq_lens=[m] * n, hq=hq, hk=hk, hv=hv, initial_state="pool", n_pool=64, l2norm_in_kernel=True,
                  qk_prenorm=False)
    inp = wl.generate(w, seed=20 + m)
    res = run_decode(inp, m)
    check_against_oracle(inp, res)
    pool = res["final_state"].cpu()
    untouched = torch.ones(pool.shape[0], dtype=torch.bool)
    untouched[inp["state_indices"].long()] = False
    assert torch.equal(pool[untouched], inp["initial_state"][untouched])


@pytest.mark.parametrize("init", ["dense", "none"])
def test_decode_dense_and_zero_state(init):
    w = wl.custom(seq_lens=[2] * 50, hq=8, hk=8, hv=8, initial_state=init, alpha="exp_softplus16")
    inp = wl.generate(w, seed=30)
    check_against_oracle(inp, run_decode(inp, 2))


def test_decode_fp32_inputs():
    w = wl.custom(seq_lens=[4] * 20, hq=2, hk=2, hv=4, dtype=torch.float32, initial_state="dense",
                  l2norm_in_kernel=True, qk_prenorm=False)
    inp = wl.generate(w, seed=31)
    check_against_oracle(inp, run_decode(inp, 4))


@pytest.mark.parametrize("m", [1, 3])
def test_decode_fp16_inputs(m):
    w = wl.custom(seq_lens=[m] * 24, hq=4, hk=4, hv=8, dtype=torch.float16, initial_state="pool", n_pool=32,
                  l2norm_in_kernel=True, qk_prenorm=False)
    inp = wl.generate(w, seed=34 + m)
    res = run_decode(inp, m)
    assert res["output"].dtype == torch.float16
    check_against_oracle(inp, res)


def test_decode_after_prefill_matches_the_whole_sequence():
    # prefill 300 tokens of 6 sequences, then decode one more token each from the prefill's final states
    L, n = 300, 6
    w = wl.custom(seq_lens=[L + 1] * n, hq=4, hk=4, hv=8, initial_state="dense", l2norm_in_kernel=True,
                  qk_prenorm=False)
    inp = wl.generate(w, seed=32)
    rows = torch.arange(n * (L + 1)).view(n, L + 1)
    pre_rows, dec_rows = rows[:, :L].reshape(-1), rows[:, L]
    pre = dict(inp, seq_lens=[L] * n, T=n * L,
               cu_seqlens=torch.arange(0, n * L + 1, L, dtype=torch.int32))
    for key in ("q", "k", "v", "g", "beta"):
        pre[key] = inp[key][pre_rows].contiguous()
    pre_res = run_gpu(to_device(pre))
    dec = dict(inp, seq_lens=[1] * n, T=n, cu_seqlens=torch.arange(0, n + 1, dtype=torch.int32),
               initial_state=pre_res["final_state"].cpu())
    for key in ("q", "k", "v", "g", "beta"):
        dec[key] = inp[key][dec_rows].contiguous()
    dec_res = run_decode(dec, 1)
    ref = run_oracle(inp)
    tol = TOL[torch.bfloat16]
    compare("decode output", dec_res["output"].cpu().double().numpy(), ref["output"][dec_rows.numpy()], tol)
    compare("final state", dec_res["final_state"].cpu().double().numpy(), ref["final_state"], tol)


def test_decode_out_of_range_pool_index_is_skipped_and_flagged():
    w = wl.custom(seq_lens=[1] * 8, hq=2, hk=2, hv=2, initial_state="pool", n_pool=16)
    inp = wl.generate(w, seed=33)
    bad = inp["state_indices"].clone()
    bad[3] = 16                                   # one past the pool
    inp_bad = dict(inp, state_indices=bad)
    res = run_decode(inp_bad, 1, check_status=False)
    assert res["status"] & gdn.DEVICE_ERR["STATE_INDEX_RANGE"]
    pool = res["final_state"].cpu()
    others = [i for i in range(8) if i != 3]
    good = dict(inp, seq_lens=[1] * 7, T=7, cu_seqlens=torch.arange(0, 8, dtype=torch.int32),
                state_indices=inp["state_indices"][others].contiguous())
    for key in ("q", "k", "v", "g", "beta"):
        good[key] = inp[key][others].contiguous()
    ref = run_oracle(good)
    compare("output", res["output"][others].cpu().double().numpy(), ref["output"], TOL[torch.bfloat16])
    # the whole pool: the skipped sequence's row and the unnamed rows keep their initial values
    compare("pool", pool.double().numpy(), ref["final_state"], TOL[torch.bfloat16])
    assert torch.equal(pool[int(inp["state_indices"][3])], inp["initial_state"][int(inp["state_indices"][3])])
