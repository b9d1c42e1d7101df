"""The benchmark's roofline numerator: algorithmic bytes per launch, written out in closed form.

The bytes the method must move once are q, k and v read at their own head counts, g and beta read (fp32), the
output written, the states read and written where asked, and the checkpoints, with states and checkpoints at
their stored size.  These tests rebuild those sums by hand for the benchmark workload (8 sequences, T = 33408,
16 q/k heads, 32 v heads, 62 checkpoints of 32 heads) and for the decode workload (512 sequences of one token on a
pool), so that a change to the accounting or to a workload's shape shows up here and not as a silent change of
the reported fraction.
"""
import torch

import bench
from gated_deltanet_chunked_device_gb300 import workloads as wl

PLANE = 128 * 128  # elements of one (sequence, head) state


def _bench_input(name):
    w = wl.WORKLOADS[name]
    return w, wl.generate(w, seed=0)


def test_benchmark_workload_bytes_in_closed_form():
    w, inp = _bench_input("gva_8seq_ckpt512_bf16")
    T, H = 33408, 32
    assert inp["T"] == T and inp["H"] == H
    n_ck = sum(L // 512 for L in inp["seq_lens"])
    assert n_ck == 62
    qkv = T * (16 + 16 + 32) * 128 * 2
    gates = T * H * 8
    out = T * H * 128 * 2
    ckpt = n_ck * H * PLANE * 4
    assert bench.algorithmic_bytes(w, inp) == qkv + gates + out + ckpt == 959_610_880


def test_checkpoint_storage_type_scales_only_the_checkpoint_bytes():
    w, inp = _bench_input("gva_8seq_ckpt512_bf16")
    full = bench.algorithmic_bytes(w, inp)
    ckpt32 = 62 * 32 * PLANE * 4
    for name, size in (("bfloat16", 2), ("float16", 2), ("float8_e4m3fn", 1), ("float8_e5m2", 1)):
        typed = bench.with_storage_types(inp, checkpoint_dtype=name)
        assert bench.algorithmic_bytes(w, typed) == full - ckpt32 + ckpt32 * size // 4


def test_decode_bytes_in_closed_form_and_with_a_narrow_pool():
    w, inp = _bench_input("decode_gva_512seq_bf16")
    N, H = 512, 32
    tokens = N * (16 + 16 + 32) * 128 * 2 + N * H * 8 + N * H * 128 * 2 + N * 4
    assert bench.decode_bytes(w, inp) == 2 * N * H * PLANE * 4 + tokens == 2_160_199_680
    for name, size in (("bfloat16", 2), ("float8_e4m3fn", 1)):
        typed = bench.with_storage_types(inp, state_dtype=name)
        assert typed["initial_state"].dtype == bench.STORAGE_DTYPES[name]
        assert bench.decode_bytes(w, typed) == 2 * N * H * PLANE * size + tokens


def test_state_storage_type_counts_initial_and_final_states():
    w, inp = _bench_input("two_seq_2048_bf16")  # dense initial state and final state, 16 heads
    T, N, H = 4096, 2, 16
    base = T * 3 * 16 * 128 * 2 + T * H * 8 + T * H * 128 * 2
    assert bench.algorithmic_bytes(w, inp) == base + 2 * N * H * PLANE * 4
    typed = bench.with_storage_types(inp, state_dtype="bfloat16")
    assert bench.algorithmic_bytes(w, typed) == base + 2 * N * H * PLANE * 2
    # the oracle and the GPU both read the rounded state
    assert torch.equal(typed["initial_state"].float(), inp["initial_state"].to(torch.bfloat16).float())


def test_config_keys_appear_only_for_a_chosen_storage_type():
    _, inp = _bench_input("gva_8seq_ckpt512_bf16")
    assert bench.storage_config(inp) == {}
    assert bench.storage_config(bench.with_storage_types(inp, "float16", "float8_e5m2")) == {
        "state_dtype": "float16", "checkpoint_dtype": "float8_e5m2"}
