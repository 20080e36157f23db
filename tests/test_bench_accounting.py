"""The benchmark's work accounting, pinned against the oracle.

``bench.visible_pairs`` is the denominator of every TFLOP/s the benchmark
reports.  With Q = K = 0 every key a query row can see gets the same score,
so the oracle's natural-log LSE of that row is log(number of visible keys);
summing exp(LSE) over rows and heads counts the visible (query, key) pairs
through the oracle's own mask, which follows the causal and sliding-window
definition of TransformerEngine PR #3527 (review notes on sliding windows and
causal alignment).  Keyless rows have LSE = -inf and count zero.
"""
import numpy as np
import pytest

import bench
import oracle
from bwd_tcgen05_tmem_gb300 import synth

BASE = synth.WORKLOADS["tiny_b1_h2_s256_d64"]

CASES = [
    ([1], (-1, 0), 1),
    ([37], (-1, 0), 2),
    ([130, 1, 64], (-1, 0), 3),
    ([100], (0, 0), 1),       # window of the diagonal only
    ([100, 7], (9, 0), 2),    # window shorter than some sequences
    ([50], (1023, 0), 1),     # window longer than the sequence
]


@pytest.mark.parametrize("lengths,window,hq", CASES)
def test_visible_pairs_match_oracle_mask(lengths, window, hq):
    w = BASE.with_(heads_q=hq, heads_kv=1, window=window)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    t = int(cu[-1])
    q = np.zeros((t, hq, 8))
    k = np.zeros((t, 1, 8))
    v = np.zeros((t, 1, 8))
    _, lse = oracle.fwd(q, k, v, cu, cu, scale=1.0, causal=True, window=window)
    counted = float(np.exp(lse).sum())
    assert round(counted) == bench.visible_pairs(w, lengths)
    assert abs(counted - round(counted)) < 1e-6 * max(1.0, counted)


def test_visible_pairs_closed_forms():
    # full causal: S (S + 1) / 2 per sequence and head
    w = synth.WORKLOADS["b1_h32_s32768_d192_128"]
    assert bench.visible_pairs(w) == 32 * 32768 * 32769 // 2
    # causal window of W keys (W - 1 to the left plus the diagonal): the first
    # W - 1 rows see 1..W-1 keys, every later row W
    w = synth.WORKLOADS["b1_h16_kv4_s16384_d256_w1024"]
    s, wk = 16384, 1024
    assert bench.visible_pairs(w) == 16 * ((wk - 1) * wk // 2 + (s - (wk - 1)) * wk)


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_flop_attribution_sums_to_total(name):
    w = synth.WORKLOADS[name]
    f = bench.flops(w)
    nv = f["n_visible"]
    assert f["fwd"] == 2 * nv * (w.d_qk + w.d_v)
    assert f["bwd"] == 2 * nv * (3 * w.d_qk + 2 * w.d_v)
    assert sum(f["kernel"].values()) == f["total"] == f["fwd"] + f["bwd"]


@pytest.mark.parametrize("b,s,window", [(1, 1, (-1, 0)), (2, 300, (-1, 0)), (1, 1000, (200, 0)),
                                        (3, 256, (127, 0)), (1, 4096, (-1, 0))])
def test_score_blocks_match_the_library_plan(b, s, window):
    """``bench.score_blocks`` (the dS bytes the benchmark credits to the dK/dV
    kernel and the dQ GEMM) counts the 128 x 128 blocks the library sizes its
    dS workspace for, and every block it counts holds a visible pair."""
    import ctypes
    import torch
    from bwd_tcgen05_tmem_gb300 import attn, build
    build.build()
    lib = attn.load()
    hq = 4
    w = BASE.with_(batch=b, seqlen=s, heads_q=hq, heads_kv=2, d_qk=192, d_v=128, window=window)
    meta = lambda *shape: torch.empty(shape, dtype=torch.bfloat16, device="meta")  # noqa: E731
    q, k, v = meta(b, s, hq, 192), meta(b, s, 2, 192), meta(b, s, 2, 128)
    p = attn.make_params(q, k, v, o=meta(b, s, hq, 128), causal=True, window=window, bwd_ds=1)
    assert lib.attn_bwd_path(ctypes.byref(p)) == attn.BWD_DS
    base = 256 + -(-(b * s * hq * 8) // 256) * 256
    blk_off = -(-(base + (b + 1) * 8) // 1024) * 1024
    blocks = (lib.attn_bwd_workspace_size(ctypes.byref(p)) - blk_off) // 32768
    assert bench.score_blocks(w) == blocks
    # brute force over the blocks of one sequence and head: a block counts iff
    # some query row of its tile sees some key of it (causal, left window)
    wl = window[0]
    n = 0
    for qt in range((s + 127) // 128):
        for kb in range((s + 127) // 128):
            n += any(kb * 128 <= j <= min(kb * 128 + 127, i) and (wl < 0 or j >= i - wl)
                     for i in range(qt * 128, min(qt * 128 + 128, s))
                     for j in range(kb * 128, min(kb * 128 + 128, s)))
    assert bench.score_blocks(w) == n * b * hq
