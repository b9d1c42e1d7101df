"""Mutation check of the oracle pins.

Each case plants one plausible mistake in a copy of the oracle's C source (on
the CPU, in a temporary directory), builds it, and runs the pins of
``test_oracle_pins`` against that build.  At least one pin must fail for every
planted mistake; otherwise the pins would not be able to tell a wrong oracle
from a right one.
"""
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

MUTANTS = [
    ("erase with + instead of -", "S[r * D + c] - be * Sk[r] * kt[c]", "S[r * D + c] + be * Sk[r] * kt[c]"),
    ("gate on the state only", "al * (S[r * D + c] - be * Sk[r] * kt[c])", "al * S[r * D + c] - be * Sk[r] * kt[c]"),
    ("S^T k instead of S k", "acc += S[r * D + c] * kt[c];", "acc += S[c * D + r] * kt[c];"),
    ("write without beta", "+ be * vt[r] * kt[c];", "+ vt[r] * kt[c];"),
    ("read with S^T", "acc += S[r * D + c] * qt[c];", "acc += S[c * D + r] * qt[c];"),
    ("k head by modulo", "hk_i = h / (H / a->hk)", "hk_i = h % a->hk"),
    # stays in bounds: p = j*n + 1 still maps to slot j - 1
    ("checkpoint one token late", "p % a->ckpt_n != 0) return;", "(p - 1) % a->ckpt_n != 0 || p == 1) return;"),
    ("checkpoint written to head 0", "a->checkpoints + ((size_t)slot * H + h)", "a->checkpoints + ((size_t)slot * H + 0)"),
    ("decay exponent reversed in A", "val = B[r] * exp(G[r] - G[j]) * kk;", "val = B[r] * exp(G[j] - G[r]) * kk;"),
    ("W without gamma", "w += Tm[r * C + j] * B[j] * exp(G[j]) * K[j * D + d];",
     "w += Tm[r * C + j] * B[j] * K[j * D + d];"),
    ("strict causal mask in output", "for (int32_t j = 0; j <= r; ++j) {", "for (int32_t j = 0; j < r; ++j) {"),
    ("state update without per-row decay", "acc += exp(glast - G[j]) * Dl[j * D + vv]",
     "acc += exp(glast) * Dl[j * D + vv]"),
    ("forward substitution sign", "val -= A[r * C + m] * Tm[m * C + j];", "val += A[r * C + m] * Tm[m * C + j];"),
    ("exclusive gate cumsum", "G[r] = run; /* G_r",
     "G[r] = run - (r < Lc ? log(gate_alpha(a, t0 + start + r, h)) : 0.0); /* G_r"),
    ("final state never written", "if (!a->final_state) return;", "if (!a->final_state || 1) return;"),
    ("initial state ignored", "if (!a->initial_state) {", "if (1) {"),
    ("chunk map drops zero-length offset", "offsets[i] = (int32_t)total;", "offsets[i] = (int32_t)total + (L == 0);"),
]

PIN_CALLS = [
    pins.test_chunk_map_matches_printed_example,
    pins.test_chunk_map_zero_length_and_padding,
    pins.test_checkpoint_count_matches_printed_example,
    pins.test_four_token_expansion_table,
    lambda: pins.test_beta_zero_is_pure_decay("sequential"),
    lambda: pins.test_beta_zero_is_pure_decay("chunked"),
    pins.test_alpha_one_beta_zero_keeps_state,
    pins.test_delta_rule_erasure,
    pins.test_key_response_general,
    lambda: pins.test_orthonormal_keys_reduce_to_decayed_linear_attention("sequential"),
    lambda: pins.test_orthonormal_keys_reduce_to_decayed_linear_attention("chunked"),
    pins.test_explicit_matrix_products_tiny,
    lambda: pins.test_chunked_equals_sequential([130, 0, 20, 300], 64, (2, 2, 2), True),
    lambda: pins.test_chunked_equals_sequential([200, 33], 8, (4, 2, 2), True),
    pins.test_zero_length_sequences_pass_state_through,
    pins.test_pool_routing_matches_dense_run,
    pins.test_checkpoints_equal_truncated_runs,
    lambda: pins.test_head_mapping_by_explicit_expansion(4, 1, 1),
    lambda: pins.test_head_mapping_by_explicit_expansion(6, 3, 3),
    lambda: pins.test_head_mapping_by_explicit_expansion(2, 2, 6),
    pins.test_chunk_intermediates_against_delta_residual,
]


@pytest.fixture(scope="module")
def tmpdir_mod():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


def test_pins_pass_on_unmodified_oracle():
    for call in PIN_CALLS:
        call()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, tmpdir_mod, monkeypatch):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    tag = "".join(ch if ch.isalnum() else "_" for ch in name)
    msrc = os.path.join(tmpdir_mod, f"{tag}.c")
    with open(msrc, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.load(oracle.build(src=msrc, out=os.path.join(tmpdir_mod, f"{tag}.so")))
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    with np.errstate(all="ignore"):
        for call in PIN_CALLS:
            try:
                call()
            except Exception as e:  # noqa: BLE001 - any failure of a pin counts
                caught.append(type(e).__name__)
    assert caught, f"no pin fails when the oracle has the mistake: {name}"
