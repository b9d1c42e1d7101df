"""GPU parity of context parallelism inside the GPU (use_cp): the sequences
that set a run's time are cut into segments whose start states come from a
transfer pass (each segment run from zero and, with U = 0, from the
identity) and an fp32 scan; then the segments and the sequences left whole
run as one batch ("FlashInfer GDN Prefill 完全指南", the CP routing of the
API table).  The device picks the segments from cu_seqlens; each case first
asks the host mirror of that choice which sequences it cuts, so that the
case covers what it names.  Every case is checked against the fp64
sequential oracle: outputs, final states (pool rows in place, 16-bit and
fp8 states) and checkpoints, which must land where the unsegmented sequence
puts them."""
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
    return gdn.gdn_prefill_cp_segments(res["plan"].handle, inp["seq_lens"], 0)[0]


def _cp_per_seq(res, inp):
    return gdn.gdn_prefill_cp_segments(res["plan"].handle, inp["seq_lens"], 0)[1]


def test_cp_one_long_sequence_with_checkpoints():
    w = wl.custom(seq_lens=[1500], hq=2, hk=2, hv=4, initial_state="dense", l2norm_in_kernel=True,
                  qk_prenorm=False, checkpoint_every=128)
    inp = wl.generate(w, seed=60)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    assert _cp_segments(res, inp) >= 2
    check_against_oracle(inp, res)


def test_cp_pool_zero_length_and_short_sequences():
    # a mixed batch on a pool: the long sequence runs as segments; the empty and short ones run whole, in the
    # same launch, reading and writing their own pool rows in place
    w = wl.custom(seq_lens=[2800, 0, 5, 64, 333], hq=2, hk=2, hv=2, initial_state="pool", n_pool=9,
                  l2norm_in_kernel=True, qk_prenorm=False, checkpoint_every=64)
    inp = wl.generate(w, seed=61)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    segs = _cp_per_seq(res, inp)
    assert segs[0] >= 2 and segs[1:] == [1, 1, 1, 1]
    check_against_oracle(inp, res)


@pytest.mark.parametrize("dtype,state_dtype", [(torch.float16, torch.float32), (torch.bfloat16, torch.bfloat16)])
def test_cp_input_and_state_types(dtype, state_dtype):
    # the 16-bit state is read by the fp32 scan (segmented sequence) and by the chunk kernel (whole sequence)
    w = wl.custom(seq_lens=[3000, 260], hq=4, hk=2, hv=2, dtype=dtype, initial_state="dense", alpha="exp_softplus16")
    inp = wl.generate(w, seed=62)
    inp["initial_state"] = inp["initial_state"].to(state_dtype)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    segs = _cp_per_seq(res, inp)
    assert segs[0] >= 2 and segs[1] == 1
    check_against_oracle(inp, res)


def test_cp_steep_gates_and_zero_initial_state():
    # strong decay: the segment transfers are close to zero and the pairwise decay path runs
    w = wl.custom(seq_lens=[2560, 130], hq=1, hk=1, hv=2, alpha="u(0.05,0.3)", l2norm_in_kernel=True,
                  qk_prenorm=False)
    inp = wl.generate(w, seed=63)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    assert _cp_segments(res, inp) >= 2
    check_against_oracle(inp, res)


def test_cp_several_segmented_sequences_among_whole_ones():
    # two long sequences cut (one of them into fewer segments), five short ones whole, a pool with gaps,
    # checkpoints every 128 tokens: segment starts, transfer rows and start rows of two sequences interleave
    w = wl.custom(seq_lens=[150, 2600, 40, 1400, 0, 300, 90], hq=2, hk=2, hv=2, initial_state="pool", n_pool=12,
                  l2norm_in_kernel=True, qk_prenorm=False, checkpoint_every=128)
    inp = wl.generate(w, seed=66)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    segs = _cp_per_seq(res, inp)
    assert segs[1] >= 2 and segs[3] >= 2 and segs[3] < segs[1]
    assert [segs[i] for i in (0, 2, 4, 5, 6)] == [1] * 5
    check_against_oracle(inp, res)


def test_cp_declined_runs_every_sequence_whole():
    # a balanced batch: the load model takes no segments, and the context-parallel launches still give the
    # one-pass results (every unit on the caller's state in the segment pass, nothing to scan or copy)
    w = wl.custom(seq_lens=[400, 380, 410, 350], hq=2, hk=2, hv=2, initial_state="dense", l2norm_in_kernel=True,
                  qk_prenorm=False, checkpoint_every=64)
    inp = wl.generate(w, seed=67)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    assert _cp_segments(res, inp) == 0
    check_against_oracle(inp, res)


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
    w = wl.custom(seq_lens=[3000, 40], hq=2, hk=2, hv=2, initial_state="pool", n_pool=5, l2norm_in_kernel=True,
                  qk_prenorm=False, checkpoint_every=128)
    inp = wl.generate(w, seed=64)
    inp["initial_state"] = inp["initial_state"].to(state_dtype)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True, ckpt_dtype=state_dtype)
    assert _cp_segments(res, inp) >= 2
    check_against_oracle(inp, res)


def test_cp_eight_segments_long_sequence():
    # one sequence of 64 chunks, two state heads: eight segments of 8 chunks (27 chunk periods against 64 for
    # one pass) -- the plan's maximum, whose start states come from seven chained transfers, each rounded
    # through the 16-bit state operand
    w = wl.custom(seq_lens=[4096], hq=2, hk=2, hv=2, initial_state="dense", l2norm_in_kernel=True,
                  qk_prenorm=False, alpha="u(0.95,1.0)", checkpoint_every=256)
    inp = wl.generate(w, seed=65)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    if torch.cuda.get_device_properties(0).multi_processor_count >= 30:
        assert _cp_segments(res, inp) == 8
    check_against_oracle(inp, res)


def test_cp_state_carried_across_segments():
    # gates near one and small beta: a segment's transfer M stays close to the identity (alpha^512 ~ 0.77,
    # the erasure (I - beta k k^T) weak), so the start state of every segment -- the fp32 scan S M + N over up
    # to seven transfers -- shows in that segment's outputs and in the final state instead of decaying away
    w = wl.custom(seq_lens=[4096, 300], hq=2, hk=2, hv=2, initial_state="dense", l2norm_in_kernel=True,
                  qk_prenorm=False, alpha="u(0.999,1.0)", checkpoint_every=256)
    inp = wl.generate(w, seed=68)
    inp["beta"] = inp["beta"] * 0.02
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    segs = _cp_per_seq(res, inp)
    assert segs[0] >= 4 and segs[1] == 1
    check_against_oracle(inp, res)


def test_cp_many_sequences_cross_the_segmentation_tiles():
    # 600 sequences: the segmentation's block scans run over three tiles of 256; one long sequence early and
    # one late are cut, the others run whole, and every offset after the first cut shifts
    lens = [5 + (37 * i) % 90 for i in range(600)]
    lens[3] = 5000
    lens[520] = 4000
    w = wl.custom(seq_lens=lens, hq=1, hk=1, hv=1, initial_state="pool", n_pool=640, l2norm_in_kernel=True,
                  qk_prenorm=False, checkpoint_every=64)
    inp = wl.generate(w, seed=69)
    res = run_gpu(to_device(inp), use_cp=True, return_plan=True)
    segs = _cp_per_seq(res, inp)
    assert segs[3] >= 2 and segs[520] >= 2
    assert sum(1 for x in segs if x > 1) == 2
    check_against_oracle(inp, res, heads=[0])
