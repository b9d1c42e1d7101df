"""GPU parity of context parallelism inside the GPU (use_cp): a batch with few
(sequence, head) units is cut into segments whose start states come from a
transfer pass (each segment run from zero and, with U = 0, from the
identity) and an fp32 scan, then the segments run as sequences of their own
("FlashInfer GDN Prefill 完全指南", the CP routing of the API table).  Every
case is checked against the fp64 sequential oracle: outputs, final states
(pool rows in place, 16-bit states) and checkpoints, which must land where
the unsegmented sequence puts them."""
import pytest
import torch

import gated_deltanet_chunked_device_gb300 as gdn
from gated_deltanet_chunked_device_gb300 import workloads as wl
from gdn_testlib import check_against_oracle, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.build()


def _cp_segments(res, inp):
    return gdn.lib().gdn_prefill_cp_segments(res["plan"].handle, len(inp["seq_lens"]), inp["T"], 0)


def test_cp_one_long_sequence_with_checkpoints():
    w = wl.custom(seq_lens=[1500], hq=2, hk=2, hv=4, initial_state="dense", l2norm_in_kernel=True,
                  qk_prenorm=False, checkpoint_every=128)
    inp = wl.generate(w, seed=60)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    assert _cp_segments(res, inp) >= 2
    check_against_oracle(inp, res)


def test_cp_pool_zero_length_and_short_sequences():
    w = wl.custom(seq_lens=[700, 0, 5, 64, 333], hq=2, hk=2, hv=2, initial_state="pool", n_pool=9,
                  l2norm_in_kernel=True, qk_prenorm=False, checkpoint_every=64)
    inp = wl.generate(w, seed=61)
    check_against_oracle(inp, run_gpu(to_device(inp), use_cp=True))


@pytest.mark.parametrize("dtype,state_dtype", [(torch.float16, torch.float32), (torch.bfloat16, torch.bfloat16)])
def test_cp_input_and_state_types(dtype, state_dtype):
    w = wl.custom(seq_lens=[900, 260], hq=4, hk=2, hv=2, dtype=dtype, initial_state="dense", alpha="exp_softplus16")
    inp = wl.generate(w, seed=62)
    inp["initial_state"] = inp["initial_state"].to(state_dtype)
    check_against_oracle(inp, run_gpu(to_device(inp), use_cp=True))


def test_cp_steep_gates_and_zero_initial_state():
    # strong decay: the segment transfers are close to zero and the pairwise decay path runs
    w = wl.custom(seq_lens=[640, 130], hq=1, hk=1, hv=2, alpha="u(0.05,0.3)", l2norm_in_kernel=True,
                  qk_prenorm=False)
    inp = wl.generate(w, seed=63)
    check_against_oracle(inp, run_gpu(to_device(inp), use_cp=True))


def test_cp_full_size_single_long_sequence_sampled_heads():
    # the one-sequence workload (32768 tokens, 32 state heads): 32 units on a 152-SM GPU, so the run takes
    # segments; heads sampled for the oracle, every output row finite
    inp = wl.generate(wl.WORKLOADS["gqa_long_32768_bf16"], seed=0)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    assert _cp_segments(res, inp) >= 2
    check_against_oracle(inp, res, heads=[0, 13, 31])
    assert torch.isfinite(res["output"]).all()


@pytest.mark.parametrize("state_dtype", [torch.float8_e4m3fn, torch.float8_e5m2])
def test_cp_fp8_state_pool_and_fp8_checkpoints(state_dtype):
    # context parallelism reads the fp8 pool into the fp32 scan and writes the last segments' states back in fp8
    w = wl.custom(seq_lens=[1100, 40], hq=2, hk=2, hv=2, initial_state="pool", n_pool=5, l2norm_in_kernel=True,
                  qk_prenorm=False, checkpoint_every=128)
    inp = wl.generate(w, seed=64)
    inp["initial_state"] = inp["initial_state"].to(state_dtype)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True, ckpt_dtype=state_dtype)
    assert _cp_segments(res, inp) >= 2
    check_against_oracle(inp, res)


def test_cp_eight_segments_long_sequence():
    # one sequence, two state heads: N * H = 2 on a 152-SM GPU gives the plan's maximum of eight segments,
    # whose start states come from seven chained transfers (each rounded through the 16-bit state operand)
    w = wl.custom(seq_lens=[4096], hq=2, hk=2, hv=2, initial_state="dense", l2norm_in_kernel=True,
                  qk_prenorm=False, alpha="u(0.95,1.0)", checkpoint_every=256)
    inp = wl.generate(w, seed=65)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    if torch.cuda.get_device_properties(0).multi_processor_count >= 30:
        assert _cp_segments(res, inp) == 8
    check_against_oracle(inp, res)
