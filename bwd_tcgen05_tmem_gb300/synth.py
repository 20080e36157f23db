"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no attention arithmetic: it only draws numbers.  Values are
drawn as float32 N(0, 1) from a seeded CPU ``torch.Generator`` and then cast to
the storage type (TransformerEngine PR #3527 review notes: inputs are generated
in float32 and cast down).  Seeds: 0 for Q, 1 for K, 2 for V, 3 for dO, 4 for the
varlen document-length draw.

Workload shapes are the ones the attention pages measure: 32K-token causal
attention with 32 heads and QK/V head dims 192/128 (TransformerEngine PR #3510,
validation table), packed THD with 32 query / 8 key-value heads at head dim 128
(PR #3699 timing tables), and symmetric head dim 512 / head dim 256 with a
sliding window (PR #3527 scope).
"""
from __future__ import annotations

import dataclasses
import math

import torch

SEED_Q, SEED_K, SEED_V, SEED_DO, SEED_LEN = 0, 1, 2, 3, 4


def normal(shape, seed, dtype=torch.bfloat16):
    """float32 N(0,1) from ``seed`` on the CPU, cast to ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32).to(dtype)


def varlen_lengths(total, lo, hi, seed=SEED_LEN):
    """Document lengths drawn uniformly from [lo, hi] until they reach ``total``.

    The last document is cut so the lengths sum to exactly ``total`` (it may
    come out shorter than ``lo``).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out, acc = [], 0
    while acc < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def cu_from_lengths(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int            # dense batch, or number of documents for THD
    seqlen: int           # dense sequence length, or max document length for THD
    heads_q: int
    heads_kv: int
    d_qk: int
    d_v: int
    dtype: str = "bf16"
    causal: bool = True
    window: tuple = (-1, -1)
    thd_total: int = 0    # > 0: packed varlen THD with this many tokens
    thd_len: tuple = (512, 8192)

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d_qk)

    @property
    def torch_dtype(self):
        return {"bf16": torch.bfloat16, "fp16": torch.float16}[self.dtype]

    @property
    def is_thd(self):
        return self.thd_total > 0

    def lengths(self):
        if self.is_thd:
            return varlen_lengths(self.thd_total, *self.thd_len)
        return [self.seqlen] * self.batch

    def with_(self, **kw):
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_b1_h2_s256_d64", 1, 256, 2, 2, 64, 64),
        # the benchmark's head dims at a size the oracle checks in a moment
        Workload("tiny_b1_h2_s256_d192_128", 1, 256, 2, 2, 192, 128),
        Workload("b2_h32_s4096_d192_128", 2, 4096, 32, 32, 192, 128),
        Workload("b1_h32_s32768_d192_128", 1, 32768, 32, 32, 192, 128),
        # the same heads at 8K: a profiling case (64 tiles per head, so the
        # grid runs in the same tile-major order as 32K; inputs above L2)
        Workload("b1_h32_s8192_d192_128", 1, 8192, 32, 32, 192, 128),
        Workload("thd_h32_kv8_t65536_d128_fp16", 0, 0, 32, 8, 128, 128, dtype="fp16",
                 thd_total=65536),
        Workload("thd_h32_kv8_t65536_d128_bf16", 0, 0, 32, 8, 128, 128, dtype="bf16",
                 thd_total=65536),
        Workload("b1_h16_kv4_s16384_d512", 1, 16384, 16, 4, 512, 512),
        # the same heads at 4K: a profiling case (inputs above L2, ~2 GB of P/dS)
        Workload("b1_h16_kv4_s4096_d512", 1, 4096, 16, 4, 512, 512),
        Workload("b1_h16_kv4_s16384_d256_w1024", 1, 16384, 16, 4, 256, 256,
                 window=(1023, 0)),
    ]
}


def make_inputs(w: Workload, *, with_dout=True, lengths=None):
    """Q, K, V (and dO) as CPU tensors of the workload's storage type.

    Dense workloads give [B, S, H, d]; THD workloads give [T, H, d] and the
    int32 ``cu_seqlens``.  Returns a dict.
    """
    dt = w.torch_dtype
    if w.is_thd or lengths is not None:
        lens = list(lengths) if lengths is not None else w.lengths()
        t = sum(lens)
        out = {
            "q": normal((t, w.heads_q, w.d_qk), SEED_Q, dt),
            "k": normal((t, w.heads_kv, w.d_qk), SEED_K, dt),
            "v": normal((t, w.heads_kv, w.d_v), SEED_V, dt),
            "cu_seqlens": cu_from_lengths(lens),
            "max_seqlen": max(lens) if lens else 0,
        }
        if with_dout:
            out["dout"] = normal((t, w.heads_q, w.d_v), SEED_DO, dt)
        return out
    b, s = w.batch, w.seqlen
    out = {
        "q": normal((b, s, w.heads_q, w.d_qk), SEED_Q, dt),
        "k": normal((b, s, w.heads_kv, w.d_qk), SEED_K, dt),
        "v": normal((b, s, w.heads_kv, w.d_v), SEED_V, dt),
    }
    if with_dout:
        out["dout"] = normal((b, s, w.heads_q, w.d_v), SEED_DO, dt)
    return out
