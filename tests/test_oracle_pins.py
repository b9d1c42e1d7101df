"""Pins for the fp64 oracle: facts fixed by the pages or by the mathematics.

None of these re-types the oracle's own formula.  Each test checks the oracle
against a worked example the pages print (fixtures in ``tests/golden``), a
closed form, an invariant, or a special case that reduces to a different,
textbook computation:

* the 4-token expansion table of "GDN 与 Chunked Prefill" (exact when every
  S_{t-1} k_t vanishes);
* beta = 0 (pure decay) and alpha = 1, beta = 0 (constant state);
* delta-rule erasure (alpha = beta = 1, unit key => S_t k_t = v_t) and the
  general key response S_t k = a (1 - b|k|^2) S_{t-1} k + b |k|^2 v;
* orthonormal keys => causal decayed linear attention, computed as a masked
  attention matrix (read-after-update, decay indexing);
* the chunk map and checkpoint counts the pages print;
* chunked form == per-token form, checkpoints == truncated runs, resume,
  pool routing, head mapping by explicit head expansion, L2 norm, defaults;
* the chunk intermediates W and U against the delta-rule residual
  beta_i (v_i - alpha_i S_{i-1} k_i) obtained from truncated per-token runs;
* the segment transfer (S_end = S0 M + N, N from zero, M from the identity
  with v = 0) that context parallelism relies on.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _rand_inputs(rng, lens, D=8, hq=1, hk=1, hv=1, unit_keys=True):
    T = int(sum(lens))
    q = rng.standard_normal((T, hq, D))
    k = rng.standard_normal((T, hk, D))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, hv, D))
    H = max(hq, hv)
    g = rng.uniform(0.7, 1.0, (T, H))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return q, k, v, g, b, cu


# ---------------------------------------------------------------------------
# Values the pages print
# ---------------------------------------------------------------------------

def test_chunk_map_matches_printed_example():
    rows = _read_fixture("chunk_map_example.txt")
    chunk = int(rows[0][1])
    lens = [int(x) for x in rows[1][1:]]
    counts = [int(x) for x in rows[2][1:]]
    printed = [tuple(int(x) for x in r[1:]) for r in rows[3:]]
    cu = np.concatenate([[0], np.cumsum(lens)])
    offsets, mp, n = oracle.chunk_map(cu, chunk)
    assert list(np.diff(offsets)) == counts
    assert n == sum(counts)
    for flat, seq, c in printed:
        assert (mp[flat, 0], mp[flat, 1]) == (seq, c)
    # every flat chunk appears once, in sequence order, chunk ids counting up
    expect = [(s, c) for s, cnt in enumerate(counts) for c in range(cnt)]
    assert [tuple(r) for r in mp[:n]] == expect


def test_chunk_map_zero_length_and_padding():
    offsets, mp, n = oracle.chunk_map([0, 130, 130, 150, 450], 64, map_rows=16)
    assert list(offsets) == [0, 3, 3, 4, 9] and n == 9
    assert [tuple(r) for r in mp[:n]] == [(0, 0), (0, 1), (0, 2), (2, 0), (3, 0), (3, 1), (3, 2), (3, 3), (3, 4)]
    assert (mp[n:] == -1).all()
    # chunk boundaries: 63, 64, 65 tokens
    offsets, _, n = oracle.chunk_map([0, 63, 127, 192], 64)
    assert list(np.diff(offsets)) == [1, 1, 2] and n == 4


def test_checkpoint_count_matches_printed_example():
    from gated_deltanet_chunked_device_gb300 import workloads as wl
    rows = _read_fixture("checkpoint_count_example.txt")
    every = int(rows[0][1])
    lens = [int(x) for x in rows[1][1:]]
    total = int(rows[2][1])
    starts = [int(x) for x in rows[3][1:]]
    w = wl.custom(seq_lens=lens, hq=1, hk=1, hv=1, checkpoint_every=every, head_size=8)
    inp = wl.generate(w, seed=0)
    assert inp["checkpoint_cu_starts"].tolist() == starts
    assert wl.num_checkpoints(lens, every) == total
    # the oracle fills exactly those slots, each with the state at p = j * every
    rng = np.random.default_rng(1)
    q, k, v, g, b, cu = _rand_inputs(rng, lens, D=4)
    res = oracle.gdn_sequential(q, k, v, g, b, cu, checkpoint_every_n_tokens=every,
                                checkpoint_cu_starts=np.array(starts), output_final_state=True)
    assert res["checkpoints"].shape[0] == total
    np.testing.assert_array_equal(res["checkpoints"][7], res["final_state"][0])
    np.testing.assert_array_equal(res["checkpoints"][15], res["final_state"][1])


def _parse_coef(token, g):
    if token == "1":
        return 1.0
    val = 1.0
    for f in token.split("*"):
        val *= g[int(f[1:])]
    return val


def test_four_token_expansion_table():
    """Keys e_1..e_4 and S0 with zero columns 1..4 make S_{t-1} k_t = 0, so the
    recurrence reduces to S_t = g_t S_{t-1} + u_t with u_t = beta_t v_t k_t^T and
    the printed table must hold exactly."""
    rows = _read_fixture("expansion_table_4token.txt")
    rng = np.random.default_rng(2)
    D = 8
    q = rng.standard_normal((4, 1, D))
    k = np.zeros((4, 1, D))
    for t in range(4):
        k[t, 0, t] = 1.0
    v = rng.standard_normal((4, 1, D))
    g = rng.uniform(0.3, 1.0, (4, 1))
    b = rng.uniform(0.1, 1.0, (4, 1))
    S0 = rng.standard_normal((1, 1, D, D))
    S0[..., :4] = 0.0
    gi = {t + 1: g[t, 0] for t in range(4)}
    u = {j + 1: b[j, 0] * np.outer(v[j, 0], k[j, 0]) for j in range(4)}
    for t, row in enumerate(rows, start=1):
        expect = np.prod([gi[m] for m in range(1, t + 1)]) * S0[0, 0]
        for j, tok in enumerate(row[1:], start=1):
            expect = expect + _parse_coef(tok, gi) * u[j]
        res = oracle.gdn_sequential(q[:t], k[:t], v[:t], g[:t], b[:t], [0, t], scale=0.5, initial_state=S0,
                                    output_final_state=True)
        np.testing.assert_allclose(res["final_state"][0, 0], expect, rtol=0, atol=1e-14)
        np.testing.assert_allclose(res["output"][t - 1, 0], 0.5 * expect @ q[t - 1, 0], rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# Closed forms and special cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("form", ["sequential", "chunked"])
def test_beta_zero_is_pure_decay(form):
    rng = np.random.default_rng(3)
    q, k, v, g, b, cu = _rand_inputs(rng, [37], D=8, unit_keys=False)
    b[:] = 0.0
    S0 = rng.standard_normal((1, 1, 8, 8))
    fn = oracle.gdn_sequential if form == "sequential" else (lambda *a, **kw: oracle.gdn_chunked(*a, chunk=8, **kw))
    res = fn(q, k, v, g, b, cu, scale=0.3, initial_state=S0, output_final_state=True)
    cum = np.cumprod(g[:, 0])
    np.testing.assert_allclose(res["final_state"][0, 0], cum[-1] * S0[0, 0], rtol=1e-13, atol=1e-15)
    expect_o = 0.3 * cum[:, None] * (q[:, 0] @ S0[0, 0].T)
    np.testing.assert_allclose(res["output"][:, 0], expect_o, rtol=1e-12, atol=1e-14)


def test_alpha_one_beta_zero_keeps_state():
    rng = np.random.default_rng(4)
    q, k, v, g, b, cu = _rand_inputs(rng, [50], D=8)
    g[:] = 1.0
    b[:] = 0.0
    S0 = rng.standard_normal((1, 1, 8, 8))
    for fn in (oracle.gdn_sequential, lambda *a, **kw: oracle.gdn_chunked(*a, chunk=16, **kw)):
        res = fn(q, k, v, g, b, cu, scale=1.0, initial_state=S0, output_final_state=True)
        np.testing.assert_array_equal(res["final_state"], S0)
        np.testing.assert_allclose(res["output"][:, 0], q[:, 0] @ S0[0, 0].T, rtol=1e-13, atol=1e-14)


def test_delta_rule_erasure():
    """alpha = beta = 1 and |k| = 1: the write replaces the value stored under k."""
    rng = np.random.default_rng(5)
    D, L = 8, 12
    q, k, v, g, b, cu = _rand_inputs(rng, [L], D=D)
    g[:] = 1.0
    b[:] = 1.0
    S0 = rng.standard_normal((1, 1, D, D))
    for t in range(1, L + 1):
        res = oracle.gdn_sequential(q[:t], k[:t], v[:t], g[:t], b[:t], [0, t], initial_state=S0,
                                    output_final_state=True)
        np.testing.assert_allclose(res["final_state"][0, 0] @ k[t - 1, 0], v[t - 1, 0], rtol=0, atol=1e-12)


def test_key_response_general():
    """S_t k_t = a (1 - b |k|^2) S_{t-1} k_t + b |k|^2 v_t, for keys of any length;
    directions orthogonal to k_t are only decayed: S_t x = a S_{t-1} x for x . k_t = 0."""
    rng = np.random.default_rng(6)
    D, L = 8, 9
    q, k, v, g, b, cu = _rand_inputs(rng, [L], D=D, unit_keys=False)
    S0 = rng.standard_normal((1, 1, D, D))
    prev = S0[0, 0]
    for t in range(1, L + 1):
        res = oracle.gdn_sequential(q[:t], k[:t], v[:t], g[:t], b[:t], [0, t], initial_state=S0,
                                    output_final_state=True)
        cur = res["final_state"][0, 0]
        kt, vt, a, bb = k[t - 1, 0], v[t - 1, 0], g[t - 1, 0], b[t - 1, 0]
        n2 = kt @ kt
        np.testing.assert_allclose(cur @ kt, a * (1 - bb * n2) * (prev @ kt) + bb * n2 * vt, rtol=1e-12, atol=1e-12)
        x = rng.standard_normal(D)
        x -= (x @ kt) / n2 * kt
        np.testing.assert_allclose(cur @ x, a * (prev @ x), rtol=1e-12, atol=1e-12)
        prev = cur


@pytest.mark.parametrize("form", ["sequential", "chunked"])
def test_orthonormal_keys_reduce_to_decayed_linear_attention(form):
    """With orthonormal keys and S0 = 0, every S_{t-1} k_t vanishes, so
    o_t = scale * sum_{j <= t} (prod_{m=j+1..t} a_m) b_j (k_j . q_t) v_j:
    a causal, decay-weighted attention matrix times diag(b) V."""
    rng = np.random.default_rng(7)
    D = L = 16
    Qo, _ = np.linalg.qr(rng.standard_normal((D, D)))
    q = rng.standard_normal((L, 1, D))
    k = Qo.T[:L, None, :].copy()
    v = rng.standard_normal((L, 1, D))
    g = rng.uniform(0.5, 1.0, (L, 1))
    b = rng.uniform(0.1, 1.0, (L, 1))
    fn = oracle.gdn_sequential if form == "sequential" else (lambda *a, **kw: oracle.gdn_chunked(*a, chunk=4, **kw))
    res = fn(q, k, v, g, b, [0, L], scale=0.7)
    logc = np.cumsum(np.log(g[:, 0]))
    decay = np.exp(logc[:, None] - logc[None, :]) * np.tril(np.ones((L, L)))
    attn = decay * (q[:, 0] @ k[:, 0].T)
    expect = 0.7 * attn @ (b[:, 0:1] * v[:, 0])
    np.testing.assert_allclose(res["output"][:, 0], expect, rtol=1e-12, atol=1e-13)


def test_explicit_matrix_products_tiny():
    """L = 8, D = 8: state as the product of explicit D x D step matrices,
    S_L = S0 M_1 ... M_L + sum_t beta_t v_t k_t^T M_{t+1} ... M_L with
    M_t = a_t (I - b_t k_t k_t^T): the (M, N) transfer composition of
    "GDN与线性注意力GPU并行实现" section 2.1, in right-multiplying form."""
    rng = np.random.default_rng(8)
    D = L = 8
    q, k, v, g, b, cu = _rand_inputs(rng, [L], D=D, unit_keys=False)
    S0 = rng.standard_normal((1, 1, D, D))
    M = np.eye(D)
    N = np.zeros((D, D))
    for t in range(L):
        Mt = g[t, 0] * (np.eye(D) - b[t, 0] * np.outer(k[t, 0], k[t, 0]))
        Nt = b[t, 0] * np.outer(v[t, 0], k[t, 0])
        M, N = M @ Mt, N @ Mt + Nt  # compose left segment (M, N) with step t
    res = oracle.gdn_sequential(q, k, v, g, b, cu, initial_state=S0, output_final_state=True)
    np.testing.assert_allclose(res["final_state"][0, 0], S0[0, 0] @ M + N, rtol=1e-12, atol=1e-12)


def test_state_is_affine_in_initial_state():
    rng = np.random.default_rng(9)
    q, k, v, g, b, cu = _rand_inputs(rng, [70], D=8)
    X = rng.standard_normal((1, 1, 8, 8))
    Y = rng.standard_normal((1, 1, 8, 8))
    run = lambda s: oracle.gdn_chunked(q, k, v, g, b, cu, initial_state=s, output_final_state=True, chunk=16)
    z, fx, fy, fxy = run(np.zeros_like(X)), run(X), run(Y), run(2 * X - 3 * Y)
    for key in ("final_state", "output"):
        lin = 2 * (fx[key] - z[key]) - 3 * (fy[key] - z[key])
        np.testing.assert_allclose(fxy[key] - z[key], lin, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("split", [64, 128, 200])
def test_segment_transfer_from_zero_and_identity(split):
    # The segment decomposition behind context parallelism ("GDN与线性注意力GPU并行实现", section 3.3): over
    # the segment [0, split) the state map is S_end = S0 M + N, where N is the segment run from zero and M
    # the run from the identity with v = 0; the rest of the sequence then continues from S0 M + N.
    rng = np.random.default_rng(12)
    L = 300
    q, k, v, g, b, cu = _rand_inputs(rng, [L], D=8)
    S0 = rng.standard_normal((1, 1, 8, 8))
    seg = slice(0, split)
    one = np.array([0, split], dtype=np.int64)
    run = lambda vv, s0: oracle.gdn_sequential(q[seg], k[seg], vv, g[seg], b[seg], one, initial_state=s0,
                                               output_final_state=True)["final_state"]
    N = run(v[seg], np.zeros_like(S0))[0, 0]
    M = run(np.zeros_like(v[seg]), np.eye(8)[None, None])[0, 0]
    whole = oracle.gdn_sequential(q, k, v, g, b, cu, initial_state=S0, output_final_state=True)
    head = oracle.gdn_sequential(q[seg], k[seg], v[seg], g[seg], b[seg], one, initial_state=S0,
                                 output_final_state=True)
    np.testing.assert_allclose(head["final_state"][0, 0], S0[0, 0] @ M + N, rtol=1e-11, atol=1e-12)
    rest = slice(split, L)
    tail = oracle.gdn_sequential(q[rest], k[rest], v[rest], g[rest], b[rest], np.array([0, L - split]),
                                 initial_state=(S0[0, 0] @ M + N)[None, None], output_final_state=True)
    np.testing.assert_allclose(tail["output"], whole["output"][rest], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(tail["final_state"], whole["final_state"], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------
# Chunk form against the per-token form; routing features
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("lens,chunk,heads,l2", [
    ([1], 64, (1, 1, 1), False),
    ([63, 64, 65], 64, (2, 2, 2), False),
    ([130, 0, 20, 300], 64, (2, 2, 2), True),
    ([127, 128, 5], 16, (2, 2, 4), False),   # GVA
    ([200, 33], 8, (4, 2, 2), True),         # GQA
    ([17, 0, 0, 40], 3, (1, 1, 1), False),
    ([9], 1, (1, 1, 1), False),
])
def test_chunked_equals_sequential(lens, chunk, heads, l2):
    rng = np.random.default_rng(10 + len(lens) + chunk)
    hq, hk, hv = heads
    D = 16
    q, k, v, g, b, cu = _rand_inputs(rng, lens, D=D, hq=hq, hk=hk, hv=hv, unit_keys=not l2)
    H = max(hq, hv)
    S0 = 0.1 * rng.standard_normal((len(lens), H, D, D))
    kw = dict(cu_seqlens=cu, scale=0.25, initial_state=S0, output_final_state=True, l2norm=l2)
    a = oracle.gdn_sequential(q, k, v, g, b, **kw)
    c = oracle.gdn_chunked(q, k, v, g, b, chunk=chunk, **kw)
    np.testing.assert_allclose(c["output"], a["output"], rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(c["final_state"], a["final_state"], rtol=1e-10, atol=1e-11)


def test_zero_length_sequences_pass_state_through():
    rng = np.random.default_rng(11)
    lens = [0, 5, 0]
    q, k, v, g, b, cu = _rand_inputs(rng, lens, D=8)
    pool = rng.standard_normal((6, 1, 8, 8))
    idx = np.array([4, 1, 2])
    for fn in (oracle.gdn_sequential, oracle.gdn_chunked):
        res = fn(q, k, v, g, b, cu, initial_state=pool, state_indices=idx, output_final_state=True)
        out = res["final_state"]
        np.testing.assert_array_equal(out[4], pool[4])
        np.testing.assert_array_equal(out[2], pool[2])
        np.testing.assert_array_equal(out[[0, 3, 5]], pool[[0, 3, 5]])
        assert not np.array_equal(out[1], pool[1])
        dense = fn(q, k, v, g, b, cu, initial_state=pool[idx], output_final_state=True)
        np.testing.assert_array_equal(dense["final_state"][0], pool[4])
        none = fn(q, k, v, g, b, cu, output_final_state=True)
        np.testing.assert_array_equal(none["final_state"][2], 0.0)


def test_pool_routing_matches_dense_run():
    rng = np.random.default_rng(12)
    lens = [30, 70, 1]
    q, k, v, g, b, cu = _rand_inputs(rng, lens, D=8, hq=2, hk=2, hv=2)
    pool = rng.standard_normal((10, 2, 8, 8))
    idx = np.array([7, 0, 3])
    for fn in (oracle.gdn_sequential, oracle.gdn_chunked):
        pooled = fn(q, k, v, g, b, cu, initial_state=pool, state_indices=idx, output_final_state=True)
        dense = fn(q, k, v, g, b, cu, initial_state=pool[idx], output_final_state=True)
        np.testing.assert_array_equal(pooled["output"], dense["output"])
        np.testing.assert_array_equal(pooled["final_state"][idx], dense["final_state"])
        untouched = np.setdiff1d(np.arange(10), idx)
        np.testing.assert_array_equal(pooled["final_state"][untouched], pool[untouched])


def test_checkpoints_equal_truncated_runs():
    rng = np.random.default_rng(13)
    lens = [40, 7, 33]
    n = 8
    q, k, v, g, b, cu = _rand_inputs(rng, lens, D=8, hq=2, hk=2, hv=2)
    ccs = np.concatenate([[0], np.cumsum([l // n for l in lens])])
    seq = oracle.gdn_sequential(q, k, v, g, b, cu, checkpoint_every_n_tokens=n, checkpoint_cu_starts=ccs,
                                output_final_state=True)
    chk = oracle.gdn_chunked(q, k, v, g, b, cu, checkpoint_every_n_tokens=n, checkpoint_cu_starts=ccs,
                             output_final_state=True, chunk=4)
    np.testing.assert_allclose(chk["checkpoints"], seq["checkpoints"], rtol=1e-10, atol=1e-12)
    for i, L in enumerate(lens):
        for j in range(1, L // n + 1):
            t0 = cu[i]
            p = j * n
            trunc = oracle.gdn_sequential(q[t0:t0 + p], k[t0:t0 + p], v[t0:t0 + p], g[t0:t0 + p], b[t0:t0 + p],
                                          [0, p], output_final_state=True)
            np.testing.assert_array_equal(seq["checkpoints"][ccs[i] + j - 1], trunc["final_state"][0])


@pytest.mark.parametrize("split", [64, 100])
def test_resume_from_state_equals_uninterrupted_run(split):
    rng = np.random.default_rng(14)
    L = 200
    q, k, v, g, b, cu = _rand_inputs(rng, [L], D=8, hq=2, hk=2, hv=2)
    S0 = rng.standard_normal((1, 2, 8, 8))
    full = oracle.gdn_chunked(q, k, v, g, b, cu, initial_state=S0, output_final_state=True)
    a = oracle.gdn_chunked(q[:split], k[:split], v[:split], g[:split], b[:split], [0, split], initial_state=S0,
                           output_final_state=True)
    bb = oracle.gdn_chunked(q[split:], k[split:], v[split:], g[split:], b[split:], [0, L - split],
                            initial_state=a["final_state"], output_final_state=True)
    np.testing.assert_allclose(np.concatenate([a["output"], bb["output"]]), full["output"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(bb["final_state"], full["final_state"], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("hq,hk,hv", [(2, 2, 6), (6, 3, 3), (4, 1, 1), (3, 3, 3)])
def test_head_mapping_by_explicit_expansion(hq, hk, hv):
    """Grouped heads equal an equal-head run whose q/k/v heads were repeated in
    contiguous blocks (state head h reads q head h // (H // hq), etc.)."""
    rng = np.random.default_rng(15)
    lens = [20, 45]
    q, k, v, g, b, cu = _rand_inputs(rng, lens, D=8, hq=hq, hk=hk, hv=hv)
    H = max(hq, hv)
    grouped = oracle.gdn_chunked(q, k, v, g, b, cu, output_final_state=True, chunk=8)
    rep = lambda x, h: np.repeat(x, H // h, axis=1)
    equal = oracle.gdn_chunked(rep(q, hq), rep(k, hk), rep(v, hv), g, b, cu, output_final_state=True, chunk=8)
    np.testing.assert_array_equal(grouped["output"], equal["output"])
    np.testing.assert_array_equal(grouped["final_state"], equal["final_state"])
    # state heads fed identical inputs produce identical results
    if hv > hq:
        v2 = v.copy()
        v2[:, 1] = v2[:, 0]
        g2, b2 = g.copy(), b.copy()
        g2[:, 1], b2[:, 1] = g2[:, 0], b2[:, 0]
        r = oracle.gdn_sequential(q, k, v2, g2, b2, cu, output_final_state=True)
        if (H // hq) > 1:  # heads 0 and 1 share a q/k head
            np.testing.assert_array_equal(r["output"][:, 0], r["output"][:, 1])


def test_l2norm_matches_prenormalised_inputs():
    rng = np.random.default_rng(16)
    q, k, v, g, b, cu = _rand_inputs(rng, [50], D=16, unit_keys=False)
    q *= 3.0
    k *= 0.5
    on = oracle.gdn_sequential(q, k, v, g, b, cu, l2norm=True, output_final_state=True)
    qn = q / np.sqrt((q * q).sum(-1, keepdims=True))
    kn = k / np.sqrt((k * k).sum(-1, keepdims=True))
    off = oracle.gdn_sequential(qn, kn, v, g, b, cu, l2norm=False, output_final_state=True)
    # eps = 1e-6 inside the square root moves results by about 1e-6 / |x|^2 relative
    np.testing.assert_allclose(on["output"], off["output"], rtol=1e-5, atol=1e-6)
    # scaling a row by a positive constant leaves the normalised result unchanged up to eps
    on2 = oracle.gdn_sequential(q * 2.0, k * 4.0, v, g, b, cu, l2norm=True, output_final_state=True)
    np.testing.assert_allclose(on2["output"], on["output"], rtol=1e-5, atol=1e-6)


def test_defaults_and_scale():
    rng = np.random.default_rng(17)
    D = 16
    q, k, v, g, b, cu = _rand_inputs(rng, [30], D=D)
    ones = np.ones_like(g)
    dflt = oracle.gdn_sequential(q, k, v, None, None, cu, scale=None)
    expl = oracle.gdn_sequential(q, k, v, ones, ones, cu, scale=1.0 / np.sqrt(D))
    np.testing.assert_array_equal(dflt["output"], expl["output"])
    s1 = oracle.gdn_sequential(q, k, v, g, b, cu, scale=1.0)
    s3 = oracle.gdn_sequential(q, k, v, g, b, cu, scale=3.0)
    np.testing.assert_allclose(s3["output"], 3.0 * s1["output"], rtol=1e-13, atol=0)


def test_chunk_intermediates_against_delta_residual():
    """Delta = U - W S0^T for every S0, and Delta_i is the delta-rule residual
    beta_i (v_i - alpha_i S_{i-1} k_i).  U is therefore the residual at S0 = 0
    and W S0^T its S0-dependent part; both are checked against states taken
    from truncated per-token runs.  G is the running sum of log alpha."""
    rng = np.random.default_rng(18)
    C, D, L = 8, 8, 8
    q, k, v, g, b, cu = _rand_inputs(rng, [L], D=D)
    X = rng.standard_normal((1, 1, D, D))
    res = oracle.gdn_chunked(q, k, v, g, b, cu, chunk=C, return_intermediates=True)
    W, U, G = res["W"][0, 0], res["U"][0, 0], res["G"][0, 0]
    np.testing.assert_allclose(np.exp(G), np.cumprod(g[:, 0]), rtol=1e-13)

    def prev_state(i, s0):
        if i == 0:
            return s0[0, 0]
        r = oracle.gdn_sequential(q[:i], k[:i], v[:i], g[:i], b[:i], [0, i], initial_state=s0,
                                  output_final_state=True)
        return r["final_state"][0, 0]

    Z = np.zeros_like(X)
    for i in range(L):
        s_z, s_x = prev_state(i, Z), prev_state(i, X)
        resid_z = b[i, 0] * (v[i, 0] - g[i, 0] * s_z @ k[i, 0])
        np.testing.assert_allclose(U[i], resid_z, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(W[i] @ X[0, 0].T, b[i, 0] * g[i, 0] * (s_x - s_z) @ k[i, 0], rtol=1e-11,
                                   atol=1e-12)
