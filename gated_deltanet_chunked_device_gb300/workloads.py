"""Seeded synthetic workloads for the chunked Gated DeltaNet prefill.

This module only draws inputs.  It holds none of the method's arithmetic, so
both the CUDA path (tests, benchmark) and the fp64 oracle (tests) take their
inputs from here.  Every tensor is drawn on the CPU from
``torch.Generator().manual_seed(seed)`` in a fixed order:

    lengths -> q -> k -> v -> alpha -> beta -> initial state / pool -> state_indices

and cast to the workload's dtype; the oracle is fed the same rounded values.

The workloads follow the shapes the pages use: the FlashInfer API example
(2 sequences x 2048 tokens, 16 heads, head size 128), the varlen batch with a
zero-length sequence, the state pool with ``state_indices``, checkpoints every
n tokens with ``checkpoint_cu_starts = [0] + cumsum(len // n)``, and GQA / GVA
head mappings ("FlashInfer GDN Prefill 完全指南", API table and the sections on
the state pool and on checkpoints).  No dataset is involved.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

HEAD_SIZE = 128
CHUNK = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seq_lens: Optional[tuple]          # fixed lengths, or None to draw them
    num_seqs: int
    hq: int
    hk: int
    hv: int
    dtype: torch.dtype
    qk_prenorm: bool                   # q, k drawn N(0,1) then divided by their norm per head
    l2norm_in_kernel: bool
    alpha: str                         # "u(lo,hi)" or "exp_softplus16"
    initial_state: str                 # "none" | "dense" (std 0.02) | "pool"
    n_pool: int = 0
    output_final_state: bool = True
    checkpoint_every: int = 0
    max_len: int = 0                   # when seq_lens is None: lengths ~ randint(1, max_len + 1)
    head_size: int = HEAD_SIZE

    @property
    def H(self) -> int:
        return max(self.hq, self.hv)


def _alpha_range(spec: str):
    lo, hi = spec[2:-1].split(",")
    return float(lo), float(hi)


WORKLOADS = {
    # 1: one sequence of 128 tokens (2 chunks), 2 heads, fp32 inputs
    "single_L128_fp32": Workload("single_L128_fp32", (128,), 1, 2, 2, 2, torch.float32, True, False,
                                 "u(0.9,1.0)", "none", output_final_state=True),
    # 2: varlen batch with a zero-length sequence, in-place pool update
    "varlen_pool_bf16": Workload("varlen_pool_bf16", (130, 0, 20, 300), 4, 16, 16, 16, torch.bfloat16, False,
                                 True, "u(0.8,1.0)", "pool", n_pool=64, output_final_state=True),
    # 3: the pages' API example: 2 x 2048 tokens, 16 heads
    "two_seq_2048_bf16": Workload("two_seq_2048_bf16", (2048, 2048), 2, 16, 16, 16, torch.bfloat16, True, False,
                                  "exp_softplus16", "dense", output_final_state=True),
    # 4: GVA 16 q/k heads, 32 v heads, 8 sequences of random length, checkpoints every 512 tokens
    "gva_8seq_ckpt512_bf16": Workload("gva_8seq_ckpt512_bf16", None, 8, 16, 16, 32, torch.bfloat16, False, True,
                                      "u(0.9,1.0)", "none", output_final_state=False, checkpoint_every=512,
                                      max_len=8192),
    # 5a: GQA long prefill, one sequence of 32768 tokens (512 chunks)
    "gqa_long_32768_bf16": Workload("gqa_long_32768_bf16", (32768,), 1, 32, 16, 16, torch.bfloat16, True, False,
                                    "exp_softplus16", "none", output_final_state=True),
    # 5b: GQA batch of 64 sequences x 1024 tokens
    "gqa_batch_64x1024_bf16": Workload("gqa_batch_64x1024_bf16", (1024,) * 64, 64, 32, 16, 16, torch.bfloat16, True,
                                       False, "exp_softplus16", "none", output_final_state=True),
    # 5 as one call: the long sequence plus the 64 x 1024 batch (65 sequences)
    "gqa_long_plus_batch_bf16": Workload("gqa_long_plus_batch_bf16", (32768,) + (1024,) * 64, 65, 32, 16, 16,
                                         torch.bfloat16, True, False, "exp_softplus16", "none",
                                         output_final_state=True),
    # decode steps on a state pool (one token per sequence, and four speculative tokens), GVA heads
    "decode_gva_512seq_bf16": Workload("decode_gva_512seq_bf16", (1,) * 512, 512, 16, 16, 32, torch.bfloat16, False,
                                       True, "u(0.9,1.0)", "pool", n_pool=1024, output_final_state=True),
    "decode4_gva_512seq_bf16": Workload("decode4_gva_512seq_bf16", (4,) * 512, 512, 16, 16, 32, torch.bfloat16,
                                        False, True, "u(0.9,1.0)", "pool", n_pool=1024, output_final_state=True),
}

# The benchmark workload (the configuration the headline metric is quoted on).
BENCH_WORKLOAD = "gva_8seq_ckpt512_bf16"


def custom(name="custom", seq_lens=(64,), hq=2, hk=2, hv=2, dtype=torch.bfloat16, qk_prenorm=True,
           l2norm_in_kernel=False, alpha="u(0.9,1.0)", initial_state="none", n_pool=0, output_final_state=True,
           checkpoint_every=0, head_size=HEAD_SIZE) -> Workload:
    """A workload of explicit shape, for edge-case tests."""
    return Workload(name, tuple(seq_lens), len(seq_lens), hq, hk, hv, dtype, qk_prenorm, l2norm_in_kernel, alpha,
                    initial_state, n_pool=n_pool, output_final_state=output_final_state,
                    checkpoint_every=checkpoint_every, head_size=head_size)


def _normal(shape, gen):
    return torch.randn(shape, generator=gen, dtype=torch.float32)


def generate(w: Workload, seed: int = 0, index_dtype=torch.int32) -> dict:
    """Draw the inputs of workload ``w`` on the CPU.

    Returns a dict of CPU tensors: q, k, v (w.dtype), g and beta (fp32, [T, H]),
    cu_seqlens ([N+1], ``index_dtype``), scale (float), initial_state (fp32 or
    None), state_indices (or None), checkpoint_cu_starts (or None) and the
    flags the call needs.
    """
    gen = torch.Generator().manual_seed(seed)
    if w.seq_lens is None:
        lens = torch.randint(1, w.max_len + 1, (w.num_seqs,), generator=gen).tolist()
    else:
        lens = list(w.seq_lens)
    T = int(sum(lens))
    D = w.head_size
    H = w.H
    cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0)

    def qk(h):
        x = _normal((T, h, D), gen)
        if w.qk_prenorm:
            x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)
        return x.to(w.dtype)

    q = qk(w.hq)
    k = qk(w.hk)
    v = _normal((T, w.hv, D), gen).to(w.dtype)
    if w.alpha.startswith("u("):
        lo, hi = _alpha_range(w.alpha)
        g = lo + (hi - lo) * torch.rand((T, H), generator=gen, dtype=torch.float32)
    elif w.alpha == "exp_softplus16":
        g = torch.exp(-torch.nn.functional.softplus(_normal((T, H), gen)) / 16.0)
    else:
        raise ValueError(w.alpha)
    beta = torch.sigmoid(_normal((T, H), gen))
    initial_state = None
    state_indices = None
    if w.initial_state == "dense":
        initial_state = 0.02 * _normal((len(lens), H, D, D), gen)
    elif w.initial_state == "pool":
        initial_state = 0.02 * _normal((w.n_pool, H, D, D), gen)
        state_indices = torch.randperm(w.n_pool, generator=gen)[: len(lens)].to(index_dtype)
    ccs = None
    if w.checkpoint_every:
        n = w.checkpoint_every
        ccs = torch.zeros(len(lens) + 1, dtype=torch.int64)
        ccs[1:] = torch.cumsum(torch.tensor([l // n for l in lens], dtype=torch.int64), 0)
        ccs = ccs.to(index_dtype)
    return {
        "q": q, "k": k, "v": v, "g": g, "beta": beta,
        "cu_seqlens": cu.to(index_dtype), "seq_lens": lens, "T": T, "H": H,
        "scale": 1.0 / math.sqrt(D),
        "initial_state": initial_state, "state_indices": state_indices,
        "output_final_state": w.output_final_state,
        "use_qk_l2norm_in_kernel": w.l2norm_in_kernel,
        "checkpoint_every_n_tokens": w.checkpoint_every, "checkpoint_cu_starts": ccs,
    }


def num_checkpoints(lens, n) -> int:
    return int(sum(l // n for l in lens)) if n else 0
