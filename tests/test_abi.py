"""The C ABI on the host: the library loads, exports every declared entry
point, and rejects host-checkable bad arguments before launching anything.
None of these tests needs a GPU (every rejection happens before the first
CUDA call)."""
import ctypes
import os
import re

import pytest

import gated_deltanet_chunked_device_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn_prefill.h")
OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def L():
    gdn.build()
    return gdn.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert {"gdn_prefill_plan", "gdn_prefill_run", "gdn_prefill_read_status", "gdn_prefill_plan_destroy",
            "gdn_status_string", "gdn_prefill_workspace_layout"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in gdn_prefill.h but not exported"


def _desc(**kw):
    d = dict(num_q_heads=16, num_k_heads=16, num_v_heads=32, head_size=128, qkv_dtype=gdn.DTYPE_BF16,
             state_dtype=gdn.DTYPE_F32, max_total_tokens=1 << 16, max_num_seqs=64, max_pool_rows=0,
             checkpoint_every_n_tokens=0, flags=0)
    d.update(kw)
    return gdn.Desc(**d)


@pytest.mark.parametrize("kw,expect", [
    ({}, OK),
    (dict(head_size=64), UNSUPPORTED),
    (dict(num_q_heads=4, num_k_heads=2, num_v_heads=8), INVALID),       # neither GQA nor GVA
    (dict(num_q_heads=32, num_k_heads=16, num_v_heads=16), OK),         # GQA
    (dict(num_q_heads=6, num_k_heads=4, num_v_heads=4), INVALID),       # hq % hk != 0
    (dict(num_q_heads=16, num_k_heads=16, num_v_heads=24), INVALID),    # hv % hq != 0
    (dict(num_q_heads=0), INVALID),
    (dict(checkpoint_every_n_tokens=100), INVALID),
    (dict(checkpoint_every_n_tokens=512), OK),
    (dict(checkpoint_every_n_tokens=-64), INVALID),
    (dict(state_dtype=gdn.DTYPE_BF16), OK),
    (dict(state_dtype=gdn.DTYPE_F16), OK),
    (dict(state_dtype=9), UNSUPPORTED),
    (dict(state_dtype=gdn.DTYPE_F8E4M3), OK),                          # fp8 states (storage only)
    (dict(state_dtype=gdn.DTYPE_F8E5M2), OK),
    (dict(state_dtype=5), UNSUPPORTED),
    (dict(checkpoint_every_n_tokens=64, checkpoint_dtype=gdn.DTYPE_BF16), OK),
    (dict(checkpoint_every_n_tokens=64, checkpoint_dtype=gdn.DTYPE_F16), OK),
    (dict(checkpoint_every_n_tokens=64, checkpoint_dtype=gdn.DTYPE_F8E4M3), OK),
    (dict(checkpoint_every_n_tokens=64, checkpoint_dtype=gdn.DTYPE_F8E5M2), OK),
    (dict(checkpoint_every_n_tokens=64, checkpoint_dtype=5), UNSUPPORTED),
    (dict(qkv_dtype=gdn.DTYPE_F8E4M3), UNSUPPORTED),                   # fp8 is not an input type
    (dict(qkv_dtype=7), UNSUPPORTED),
    (dict(qkv_dtype=gdn.DTYPE_F16), OK),
    (dict(qkv_dtype=gdn.DTYPE_F32), OK),
    (dict(flags=1 << 20), INVALID),
    (dict(max_total_tokens=-1), INVALID),
    (dict(max_total_tokens=1 << 31), UNSUPPORTED),
    (dict(flags=gdn.FLAGS["HAS_STATE_INDICES"], max_pool_rows=0), INVALID),
    (dict(flags=gdn.FLAGS["HAS_STATE_INDICES"], max_pool_rows=64), OK),
])
def test_plan_validation(L, kw, expect):
    st, plan, nbytes = gdn.gdn_prefill_plan(_desc(**kw))
    assert st == expect, gdn.STATUS.get(st)
    if st == OK:
        assert nbytes > 0 and nbytes % 16 == 0
        lay = gdn.gdn_prefill_workspace_layout(plan)
        assert lay.max_chunks == (1 << 16) // 64 + 64
        gdn.gdn_prefill_plan_destroy(plan)
    else:
        assert not plan.value


_CP = gdn.FLAGS["CONTEXT_PARALLEL"]


_H64 = dict(num_q_heads=64, num_k_heads=16, num_v_heads=16)
_H128 = dict(num_q_heads=128, num_k_heads=16, num_v_heads=16)
_H1 = dict(num_q_heads=1, num_k_heads=1, num_v_heads=1)
_H2 = dict(num_q_heads=2, num_k_heads=2, num_v_heads=2)


# Expected choices worked by hand from the load model (chunk periods; S SMs, H state heads, c_i chunks):
# transfer ceil(2 H nA / S) tau + segment pass max(ceil(H nS / S) tau, ceil(H sum c / S), longest whole)
# + (P - 1) + 4, taken when at most 85 % of one pass max(c_max, ceil(H sum c / S)).
@pytest.mark.parametrize("desc_kw,lens,sms,expect,per_seq", [
    # 512 chunks, 32 heads: P = 3 costs 171 + 171 + 6 = 348 of 512; P = 4 needs two waves of transfers (391)
    (dict(flags=_CP), [32768], 152, 3, [3]),
    # the same sequence beside four short ones: they run whole in the segment pass
    (dict(flags=_CP), [32768, 1024, 1024, 1024, 1024], 152, 3, [3, 1, 1, 1, 1]),
    # ... beside 64 of them: the batch alone fills 324 periods of the 512, CP would cost 501 > 435
    (dict(flags=_CP), [32768] + [1024] * 64, 152, 0, None),
    # eight sequences up to 118 chunks on 32 heads: P = 2 already needs two transfer waves (118); P >= 3 does
    # not fit the 256 transfer planes
    (dict(flags=_CP), [7528, 6000, 5000, 4000, 3000, 2000, 1000, 500], 152, 0, None),
    # one head, 79 chunks: eight segments of 10 chunks cost 10 + 10 + 11 = 31
    (dict(flags=_CP, **_H1), [5000], 152, 8, [8]),
    # checkpoints every 1024 tokens: segments are multiples of 16 chunks, so 4 x 16 (39) beats 2 x 32 (69)
    (dict(flags=_CP, checkpoint_every_n_tokens=1024, **_H2), [4096], 152, 4, [4]),
    (dict(flags=_CP, checkpoint_every_n_tokens=512, **_H2), [4096], 152, 8, [8]),
    # 64 heads: two transfer segments fill the 256 planes, so at most three segments (53 + 53 + 6 of 157)
    (dict(flags=_CP, **_H64), [10000], 1024, 3, [3]),
    (dict(flags=_CP, **_H64), [10000], 152, 0, None),     # ... but on 152 SMs two waves each: 218 > 157
    (dict(flags=_CP, **_H128), [10000], 1024, 0, None),   # 128 heads: three segments do not fit, two cannot gain
    ({}, [32768], 152, 0, None),                          # the plan does not allow it
    (dict(flags=_CP, qkv_dtype=gdn.DTYPE_F32), [32768], 152, 0, None),  # fp32 inputs: one pass
    (dict(flags=_CP), [0], 152, 0, None),                 # no tokens
    (dict(flags=_CP), [0, 32768, 0], 152, 3, [1, 3, 1]),  # empty sequences run whole (their state passes through)
])
def test_context_parallel_segment_choice(L, desc_kw, lens, sms, expect, per_seq):
    st, plan, nbytes = gdn.gdn_prefill_plan(_desc(**desc_kw))
    assert st == OK
    try:
        most, segs = gdn.gdn_prefill_cp_segments(plan, lens, sms)
        assert most == expect
        assert segs == (per_seq if per_seq is not None else [1] * len(lens))
    finally:
        gdn.gdn_prefill_plan_destroy(plan)


def test_context_parallel_choice_on_large_batches(L):
    # the host query walks any number of sequences; a batch of many short ones never segments, and one long
    # sequence among them is cut while the rest stay whole
    st, plan, _ = gdn.gdn_prefill_plan(_desc(flags=_CP, max_num_seqs=5000, **_H1))
    assert st == OK
    try:
        most, segs = gdn.gdn_prefill_cp_segments(plan, [100] * 3000, 152)
        assert most == 0 and set(segs) == {1}
        lens = [30] * 3000
        lens[1234] = 20000
        most, segs = gdn.gdn_prefill_cp_segments(plan, lens, 152)
        assert most >= 2 and segs[1234] == most and segs.count(1) == 2999
    finally:
        gdn.gdn_prefill_plan_destroy(plan)


def test_context_parallel_plan_reserves_its_scratch(L):
    st, p0, base = gdn.gdn_prefill_plan(_desc())
    st1, p1, with_cp = gdn.gdn_prefill_plan(_desc(flags=_CP))
    assert st == OK and st1 == OK
    gdn.gdn_prefill_plan_destroy(p0)
    gdn.gdn_prefill_plan_destroy(p1)
    assert with_cp >= base + 2 * 256 * 128 * 128 * 4  # transfer and start planes, fp32


def _valid_args(**kw):
    # fake, 256-byte aligned device addresses: never dereferenced, because every
    # case below is rejected (or needs no launch) before the first CUDA call
    fake = 0x7f0000000000
    a = dict(q=fake, k=fake + 0x100000, v=fake + 0x200000, g=None, beta=None, scale=0.0, cu_seqlens=fake + 0x300000,
             num_seqs=2, total_tokens=100, max_seqlen=0, initial_state=None, output_state=None, n_pool=0,
             state_indices=None, state_checkpoints=None, num_checkpoints=0, checkpoint_cu_starts=None,
             output=fake + 0x400000, device_status=None)
    strides = kw.pop("state_strides", (0, 0, 0))
    a.update(kw)
    return gdn.Args(state_strides=(ctypes.c_int64 * 3)(*strides), **a)


@pytest.mark.parametrize("desc_kw,args_kw,ws,expect", [
    ({}, dict(q=None), 1 << 20, INVALID),
    ({}, dict(q=0x7f0000000008), 1 << 20, INVALID),                     # q not 16-byte aligned
    ({}, dict(num_seqs=65), 1 << 20, INVALID),                          # above max_num_seqs
    ({}, dict(total_tokens=(1 << 16) + 1), 1 << 20, INVALID),           # above max_total_tokens
    ({}, dict(num_seqs=0, total_tokens=5), 1 << 20, INVALID),
    ({}, dict(num_seqs=0, total_tokens=0), 1 << 20, OK),                # nothing to do, nothing launched
    ({}, dict(cu_seqlens=None), 1 << 20, INVALID),
    ({}, dict(max_seqlen=101), 1 << 20, INVALID),                       # > T
    ({}, dict(max_seqlen=49), 1 << 20, INVALID),                        # < ceil(T / N)
    ({}, {}, 16, INVALID),                                              # workspace too small
    (dict(flags=gdn.FLAGS["HAS_G"]), {}, 1 << 20, INVALID),             # g flag without g
    (dict(flags=gdn.FLAGS["HAS_INITIAL_STATE"]), {}, 1 << 20, INVALID),
    (dict(flags=gdn.FLAGS["OUTPUT_FINAL_STATE"] | gdn.FLAGS["HAS_STATE_INDICES"], max_pool_rows=8),
     dict(state_indices=0x7f0000500000, n_pool=8), 1 << 20, INVALID),  # pool output required with indices
    (dict(flags=gdn.FLAGS["HAS_STATE_INDICES"], max_pool_rows=8),
     dict(state_indices=0x7f0000500000, n_pool=9), 1 << 20, INVALID),  # n_pool above the plan's bound
    (dict(checkpoint_every_n_tokens=64), dict(state_checkpoints=0x7f0000600000), 1 << 20, INVALID),  # starts missing
    ({}, dict(checkpoint_cu_starts=0x7f0000600000), 1 << 20, INVALID),  # checkpoints without an interval
    (dict(qkv_dtype=gdn.DTYPE_F32, num_q_heads=2, num_k_heads=2, num_v_heads=2), dict(q=None), 1 << 20, INVALID),
    # state strides [row, head, v] (elements; the plan has H = 32 heads, N = 2 rows): one of them zero
    ({}, dict(state_strides=(0, 128 * 128, 128)), 1 << 20, INVALID),
    ({}, dict(state_strides=(32 * 128 * 128, 128 * 128, 130)), 1 << 20, INVALID),   # 520 bytes: not 16-aligned
    ({}, dict(state_strides=(32 * 128 * 128, 128 * 128, 64)), 1 << 20, INVALID),    # v rows overlap
    ({}, dict(state_strides=(32 * 128 * 128, 127 * 128, 128)), 1 << 20, INVALID),   # heads overlap
    ({}, dict(state_strides=(31 * 128 * 128, 128 * 128, 128)), 1 << 20, INVALID),   # rows overlap
    # fp8 states: strides are multiples of 16 bytes = 16 elements
    (dict(state_dtype=gdn.DTYPE_F8E4M3), dict(state_strides=(32 * 128 * 128, 128 * 128, 136)), 1 << 20, INVALID),
])
def test_run_rejects_before_launch(L, desc_kw, args_kw, ws, expect):
    st, plan, nbytes = gdn.gdn_prefill_plan(_desc(**desc_kw))
    assert st == OK
    try:
        args = _valid_args(**args_kw)
        st = gdn.gdn_prefill_run(plan, args, 0x7f0000700000, ws, 0)
        assert st == expect, gdn.STATUS.get(st)
    finally:
        gdn.gdn_prefill_plan_destroy(plan)


def test_status_strings(L):
    for code in range(6):
        assert gdn.gdn_status_string(code) and gdn.gdn_status_string(code) != "unknown status"


def test_python_wrapper_refuses_cpu_tensors():
    import torch
    q = torch.zeros(4, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        gdn.chunk_gated_delta_rule(q, q, q)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(gdn._build, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(gdn, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        gdn.lib()


@pytest.mark.parametrize("desc_kw,args_kw,m,expect", [
    ({}, dict(num_seqs=4, total_tokens=4), 0, INVALID),                 # no tokens per sequence
    ({}, dict(num_seqs=1, total_tokens=65), 65, INVALID),               # above the decode limit
    ({}, dict(num_seqs=4, total_tokens=5), 1, INVALID),                 # total != N * m
    ({}, dict(num_seqs=0, total_tokens=0), 1, OK),                      # nothing to do, nothing launched
    ({}, dict(num_seqs=4, total_tokens=8, q=None), 2, INVALID),
    ({}, dict(num_seqs=4, total_tokens=4, q=0x7f0000000008), 1, INVALID),  # q not 16-byte aligned
    (dict(checkpoint_every_n_tokens=64), dict(num_seqs=4, total_tokens=4), 1, UNSUPPORTED),
    ({}, dict(num_seqs=4, total_tokens=4, state_checkpoints=0x7f0000600000), 1, INVALID),
    (dict(flags=gdn.FLAGS["HAS_BETA"]), dict(num_seqs=4, total_tokens=4), 1, INVALID),  # beta flag without beta
    (dict(flags=gdn.FLAGS["HAS_STATE_INDICES"] | gdn.FLAGS["HAS_INITIAL_STATE"], max_pool_rows=8),
     dict(num_seqs=4, total_tokens=4, initial_state=0x7f0000500000, state_indices=0x7f0000500000, n_pool=0), 1,
     INVALID),                                                           # pool without rows
])
def test_decode_rejects_before_launch(L, desc_kw, args_kw, m, expect):
    st, plan, nbytes = gdn.gdn_prefill_plan(_desc(**desc_kw))
    assert st == OK
    try:
        st = gdn.gdn_decode_run(plan, _valid_args(cu_seqlens=None, **args_kw), m, 0)
        assert st == expect, gdn.STATUS.get(st)
    finally:
        gdn.gdn_prefill_plan_destroy(plan)


def test_decode_wrapper_refuses_cpu_tensors():
    import torch
    q = torch.zeros(4, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        gdn.gated_delta_rule_decode(q, q, q)
