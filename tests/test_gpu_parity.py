"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.

* every workload of the benchmark suite (small ones on all heads and extra
  seeds; the full-size ones on sampled state heads, in the launch
  configuration the benchmark times);
* integer outputs of the prepare step (chunk offsets, flat chunk map, LPT
  order) bit-exact against the oracle's chunk map;
* pool routing (untouched rows bit-identical), zero-length and empty batches,
  chunk-boundary lengths, head mappings, defaults, int64 indices, resume;
* the intra-chunk stage's G, W and U against the oracle's chunk intermediates;
* device-checked input errors land in the status word without hanging.
"""
import numpy as np
import pytest
import torch

import oracle
import gated_deltanet_chunked_device_gb300 as gdn
from gated_deltanet_chunked_device_gb300 import workloads as wl
from gdn_testlib import TOL, check_against_oracle, compare, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn.build()


SMALL = ["single_L128_fp32", "varlen_pool_bf16", "two_seq_2048_bf16"]
LARGE = {  # full-size workloads: state heads sampled for the oracle
    "gva_8seq_ckpt512_bf16": [0, 1, 17, 30, 31],
    "gqa_long_32768_bf16": [0, 13, 31],
    "gqa_batch_64x1024_bf16": [0, 1, 22, 31],
    "gqa_long_plus_batch_bf16": [5, 6],
}


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_small_workloads_all_heads(name, seed):
    inp = wl.generate(wl.WORKLOADS[name], seed=seed)
    res = run_gpu(to_device(inp))
    check_against_oracle(inp, res)


@pytest.mark.parametrize("name", list(LARGE))
def test_full_size_workloads_sampled_heads(name):
    inp = wl.generate(wl.WORKLOADS[name], seed=0)
    res = run_gpu(to_device(inp))
    check_against_oracle(inp, res, heads=LARGE[name])
    # all heads: finite, and outputs of every row were written (NaN-free)
    assert torch.isfinite(res["output"]).all()


def test_pool_routing_in_place_untouched_rows_bit_identical():
    inp = wl.generate(wl.WORKLOADS["varlen_pool_bf16"], seed=3)
    dev = to_device(inp)
    res = run_gpu(dev)
    pool = res["final_state"].cpu()
    idx = inp["state_indices"].long()
    untouched = torch.ones(pool.shape[0], dtype=torch.bool)
    untouched[idx] = False
    assert torch.equal(pool[untouched], inp["initial_state"][untouched])
    # the zero-length sequence (index 1) passes its row through bit-identically
    assert torch.equal(pool[idx[1]], inp["initial_state"][idx[1]])
    check_against_oracle(inp, res)


@pytest.mark.parametrize("lens", [[1], [63], [64], [65], [127], [128], [1, 63, 64, 65, 127, 128, 0, 200]])
def test_chunk_boundary_lengths(lens):
    w = wl.custom(seq_lens=lens, hq=2, hk=2, hv=2, l2norm_in_kernel=True, qk_prenorm=False, initial_state="dense",
                  checkpoint_every=64)
    inp = wl.generate(w, seed=4)
    check_against_oracle(inp, run_gpu(to_device(inp)))


def test_all_sequences_empty():
    w = wl.custom(seq_lens=[0, 0, 0], hq=2, hk=2, hv=2, initial_state="dense")
    inp = wl.generate(w, seed=5)
    res = run_gpu(to_device(inp))
    assert res["output"].shape[0] == 0
    assert torch.equal(res["final_state"].cpu(), inp["initial_state"])


def test_runs_of_empty_sequences_between_chunks():
    # several zero-length sequences in a row between non-empty ones: every role must step over them
    # without waiting for the next non-empty unit early (the status word must stay clear: no timed-out wait)
    w = wl.custom(seq_lens=[100, 0, 0, 0, 70, 0, 0, 130, 0, 0, 0, 0, 5, 0, 0], hq=2, hk=2, hv=2,
                  initial_state="dense", checkpoint_every=64)
    inp = wl.generate(w, seed=17)
    check_against_oracle(inp, run_gpu(to_device(inp)))


def test_zero_initial_state_and_no_final_state():
    w = wl.custom(seq_lens=[100, 0, 37], hq=4, hk=4, hv=4, output_final_state=False)
    inp = wl.generate(w, seed=6)
    check_against_oracle(inp, run_gpu(to_device(inp)))


@pytest.mark.parametrize("hq,hk,hv", [(8, 2, 2), (2, 2, 8), (4, 4, 4), (4, 1, 1), (1, 1, 4)])
def test_head_mappings(hq, hk, hv):
    w = wl.custom(seq_lens=[150, 70], hq=hq, hk=hk, hv=hv, initial_state="dense")
    inp = wl.generate(w, seed=7)
    check_against_oracle(inp, run_gpu(to_device(inp)))


def test_defaults_g_beta_scale():
    w = wl.custom(seq_lens=[90], hq=2, hk=2, hv=2)
    inp = wl.generate(w, seed=8)
    dev = to_device(inp)
    res = run_gpu(dev, g=None, beta=None, scale=None)
    ones = inp["g"] * 0 + 1
    ref_inp = dict(inp, g=ones, beta=ones, scale=128 ** -0.5)
    check_against_oracle(ref_inp, res)


def test_int64_indices_everywhere():
    w = wl.custom(seq_lens=[130, 0, 20, 300], hq=4, hk=4, hv=4, initial_state="pool", n_pool=9,
                  checkpoint_every=128, l2norm_in_kernel=True, qk_prenorm=False)
    inp = wl.generate(w, seed=9, index_dtype=torch.int64)
    assert inp["cu_seqlens"].dtype == torch.int64 and inp["state_indices"].dtype == torch.int64
    check_against_oracle(inp, run_gpu(to_device(inp)))


@pytest.mark.parametrize("split", [256, 200])
def test_resume_from_final_state(split):
    w = wl.custom(seq_lens=[500], hq=2, hk=2, hv=2, initial_state="dense")
    inp = wl.generate(w, seed=10)
    dev = to_device(inp)
    full = run_gpu(dev)
    first = {k: v for k, v in dev.items()}
    second = {k: v for k, v in dev.items()}
    for key in ("q", "k", "v", "g", "beta"):
        first[key] = dev[key][:split].contiguous()
        second[key] = dev[key][split:].contiguous()
    first.update(T=split, seq_lens=[split], cu_seqlens=torch.tensor([0, split], dtype=torch.int32, device="cuda"))
    a = run_gpu(first)
    second.update(T=500 - split, seq_lens=[500 - split], initial_state=a["final_state"],
                  cu_seqlens=torch.tensor([0, 500 - split], dtype=torch.int32, device="cuda"))
    b = run_gpu(second)
    tol = TOL[torch.bfloat16]
    compare("output", torch.cat([a["output"], b["output"]]).cpu().double().numpy(),
            full["output"].cpu().double().numpy(), tol)
    compare("final_state", b["final_state"].cpu().double().numpy(), full["final_state"].cpu().double().numpy(), tol)


def test_prepare_chunk_map_bit_exact():
    rng = np.random.default_rng(11)
    lens = [130, 0, 20, 300] + list(rng.integers(0, 700, size=60)) + [0, 0, 4096]
    w = wl.custom(seq_lens=lens, hq=1, hk=1, hv=1)
    inp = wl.generate(w, seed=11)
    res = run_gpu(to_device(inp), return_plan=True)
    N = len(lens)
    offsets, cmap, n_chunks, order = gdn.read_chunk_map(res["plan"], res["ws"], N)
    ref_off, ref_map, ref_n = oracle.chunk_map(inp["cu_seqlens"].numpy(), 64)
    assert n_chunks == ref_n
    assert np.array_equal(offsets.numpy(), ref_off)
    assert np.array_equal(cmap.numpy(), ref_map[:ref_n])
    # LPT order: a permutation, chunk counts non-increasing, ties by index
    counts = np.diff(ref_off)
    o = order.numpy()
    assert sorted(o.tolist()) == list(range(N))
    keys = [(-counts[i], i) for i in o]
    assert keys == sorted(keys)
    assert gdn.read_status(res["plan"], res["ws"]) == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_intra_stage_matches_oracle_intermediates(dtype):
    w = wl.custom(seq_lens=[130, 0, 20, 100], hq=2, hk=2, hv=4, l2norm_in_kernel=False, qk_prenorm=True, dtype=dtype)
    inp = wl.generate(w, seed=12)
    inter = {}
    run_gpu(to_device(inp), intermediates=inter)
    q, k, v = (inp[x].double().numpy() for x in ("q", "k", "v"))
    ref = oracle.gdn_chunked(q, k, v, inp["g"].double().numpy(), inp["beta"].double().numpy(),
                             inp["cu_seqlens"].numpy(), scale=inp["scale"], chunk=64, return_intermediates=True)
    F = ref["G"].shape[0]
    tol = TOL[dtype]
    compare("G", inter["G"][:F].cpu().double().numpy(), ref["G"], 1e-4)
    compare("W", inter["W"][:F].cpu().double().numpy(), ref["W"], tol)
    compare("U", inter["U"][:F].cpu().double().numpy(), ref["U"], tol)


def _status_after(inp_dev, **override):
    res = run_gpu(inp_dev, return_plan=True, check_status=False, **override)
    return gdn.read_status(res["plan"], res["ws"])


def test_device_status_flags_bad_inputs():
    w = wl.custom(seq_lens=[100, 50, 70], hq=2, hk=2, hv=2, initial_state="pool", n_pool=8, checkpoint_every=64)
    inp = wl.generate(w, seed=13)
    dev = to_device(inp)
    E = gdn.DEVICE_ERR
    assert _status_after(dev) == 0
    bad_cu = torch.tensor([0, 100, 90, 220], dtype=torch.int32, device="cuda")   # decreasing
    assert _status_after(dict(dev, cu_seqlens=bad_cu)) & E["CU_SEQLENS"]
    short_cu = torch.tensor([0, 100, 150, 219], dtype=torch.int32, device="cuda")  # ends before T
    assert _status_after(dict(dev, cu_seqlens=short_cu)) & E["CU_SEQLENS"]
    bad_ccs = torch.tensor([0, 1, 1, 3], dtype=torch.int32, device="cuda")       # 70 // 64 = 1, not 2
    assert _status_after(dict(dev, checkpoint_cu_starts=bad_ccs)) & E["CHECKPOINT_STARTS"]
    out_of_range = torch.tensor([1, 8, 2], dtype=torch.int32, device="cuda")
    assert _status_after(dict(dev, state_indices=out_of_range)) & E["STATE_INDEX_RANGE"]
    dup = torch.tensor([3, 5, 3], dtype=torch.int32, device="cuda")
    assert _status_after(dict(dev, state_indices=dup)) & E["STATE_INDEX_DUP"]
    assert _status_after(dev, max_seqlen=90) & E["MAX_SEQLEN"]
    # a clean run afterwards works and clears the word
    assert _status_after(dev) == 0


@pytest.mark.parametrize("l2", [False, True])
def test_fp32_inputs_tails_heads_pool_checkpoints(l2):
    w = wl.custom(seq_lens=[200, 0, 65, 128], hq=4, hk=2, hv=2, dtype=torch.float32, qk_prenorm=not l2,
                  l2norm_in_kernel=l2, initial_state="pool", n_pool=6, checkpoint_every=64)
    inp = wl.generate(w, seed=14)
    check_against_oracle(inp, run_gpu(to_device(inp)))


@pytest.mark.parametrize("per_sm", [0.25, 0.5, 1.0, 1.2])
def test_fp32_inputs_every_slice_count(per_sm):
    # the fp32 kernel cuts each (sequence, head) unit into 16, 8, 4 or 2 slices of the state rows, the most that
    # keep the grid within about four CTAs per SM: a quarter, a half, one and 1.2 times the SM count in units take
    # each instance once (rows of every slice, tails, checkpoints and the final state against the oracle)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = max(1, int(sms * per_sm) // 4)
    lens = [70 + (13 * i) % 60 for i in range(n)]
    w = wl.custom(seq_lens=lens, hq=2, hk=2, hv=4, dtype=torch.float32, l2norm_in_kernel=True, qk_prenorm=False,
                  initial_state="dense", checkpoint_every=64)
    inp = wl.generate(w, seed=70)
    check_against_oracle(inp, run_gpu(to_device(inp)))


def test_steep_gates_take_the_pairwise_decay_path():
    # alpha ~ U(0.05, 0.3): log alpha ~ -1.2 .. -3 per token, so a chunk's gate range is far above the
    # limit of the row x column factorisation and every A / P entry takes e^{G_i - G_j} pairwise
    w = wl.custom(seq_lens=[200, 64, 5, 130], hq=2, hk=2, hv=4, alpha="u(0.05,0.3)", l2norm_in_kernel=True,
                  qk_prenorm=False, initial_state="dense", checkpoint_every=64)
    inp = wl.generate(w, seed=15)
    check_against_oracle(inp, run_gpu(to_device(inp)))


@pytest.mark.parametrize("l2norm", [True, False])
def test_moderate_gates_scale_q_in_place(l2norm):
    # alpha ~ U(0.75, 0.95): log alpha ~ -0.05 .. -0.29 per token, so G leaves [-8, 8] inside most full chunks
    # (those rescale Q in shared memory) while short tails stay inside it (those keep Q and fold gamma into P
    # and the output factor); the gate range stays small enough for the row x column factorisation
    w = wl.custom(seq_lens=[300, 64, 5, 130, 20], hq=2, hk=2, hv=4, alpha="u(0.75,0.95)", l2norm_in_kernel=l2norm,
                  qk_prenorm=not l2norm, initial_state="dense", checkpoint_every=64)
    inp = wl.generate(w, seed=17)
    check_against_oracle(inp, run_gpu(to_device(inp)))


@pytest.mark.parametrize("case", ["gva_l2norm_pool_ckpt", "gqa_prenorm_dense"])
def test_fp16_inputs(case):
    # fp16 q/k/v: the fp16 instance of the tensor-core kernel (every 16-bit operand in fp16), output in fp16
    if case == "gva_l2norm_pool_ckpt":
        w = wl.custom(seq_lens=[300, 0, 77, 130, 64], hq=2, hk=2, hv=4, dtype=torch.float16, initial_state="pool",
                      n_pool=8, l2norm_in_kernel=True, qk_prenorm=False, checkpoint_every=64)
    else:
        w = wl.custom(seq_lens=[200, 5, 129], hq=4, hk=2, hv=2, dtype=torch.float16, initial_state="dense",
                      alpha="exp_softplus16")
    inp = wl.generate(w, seed=18)
    res = run_gpu(to_device(inp))
    assert res["output"].dtype == torch.float16
    check_against_oracle(inp, res)


def test_more_sequences_than_the_on_chip_sort():
    # 9000 sequences (above the 8192 the prepare kernel sorts on chip; the rest keep their order), most of
    # them a few tokens long, a few of them several chunks long
    rng = np.random.default_rng(16)
    lens = rng.integers(0, 4, size=9000)
    lens[::997] = rng.integers(60, 300, size=len(lens[::997]))
    w = wl.custom(seq_lens=[int(x) for x in lens], hq=1, hk=1, hv=1, initial_state="dense")
    inp = wl.generate(w, seed=16)
    res = run_gpu(to_device(inp), return_plan=True)
    check_against_oracle(inp, res)
    offsets, cmap, n_chunks, order = gdn.read_chunk_map(res["plan"], res["ws"], len(lens))
    ref_off, ref_map, ref_n = oracle.chunk_map(inp["cu_seqlens"].numpy(), 64)
    assert n_chunks == ref_n
    assert np.array_equal(offsets.numpy(), ref_off)
    assert np.array_equal(cmap.numpy(), ref_map[:ref_n])
    assert sorted(order.numpy().tolist()) == list(range(len(lens)))
