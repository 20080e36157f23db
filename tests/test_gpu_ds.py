"""GPU parity of the two backward paths at head dims 128/128 and 192/128.

ATTN_BWD_DS: the key-stationary dK/dV kernel also writes dS (16-bit, one
32 KiB block per visible 128 x 128 tile and query head) and dQ = scale dS K
is a GEMM over those blocks.  ATTN_BWD_RECOMPUTE: a query-stationary dQ
kernel computes S and dP again.  Both are checked against the FP64 oracle on
the masks whose block tables have corners: causal and bottom-right, sliding
windows whose key tiles are seen by only one 64-row half of a 128-row query
tile (those halves hold zeros in the block), non-causal attention (key rows
past the sequence end are visible there and must hold zero dS), packed THD
documents (the K rows past a document belong to the next one), GQA, FP16 and
FP32 accumulation; and for reproducibility, stage order and the no-allocation
entry point.
"""
import math

import pytest
import torch

from bwd_tcgen05_tmem_gb300 import attn, synth
from parity import Reference, gate, rel_l2
from test_gpu_parity import dense_inputs, run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from bwd_tcgen05_tmem_gb300 import build
    build.build()
    attn.load()


CASES = [
    # b, sq, sk, hq, hkv, dqk, dv, dtype, causal, window, bottom_right
    (2, 300, 300, 2, 2, 192, 128, "bf16", True, (-1, -1), False),
    (2, 300, 300, 8, 2, 128, 128, "fp16", True, (-1, -1), False),
    (1, 700, 700, 4, 2, 192, 128, "bf16", True, (129, 0), False),     # upper-half gaps
    (1, 300, 300, 2, 2, 192, 128, "bf16", False, (30, 20), False),    # lower and upper gaps
    (1, 300, 300, 2, 2, 128, 128, "fp16", False, (30, 20), False),
    (1, 200, 333, 2, 2, 128, 128, "bf16", True, (-1, -1), True),
    (1, 333, 200, 6, 2, 192, 128, "bf16", True, (-1, -1), True),      # keyless rows
    (1, 300, 300, 2, 2, 192, 128, "bf16", False, (-1, -1), False),    # past-the-end key rows
    (1, 130, 130, 2, 2, 128, 128, "bf16", True, (0, 0), False),
]


def _id(c):
    return f"b{c[0]}q{c[1]}k{c[2]}h{c[3]}/{c[4]}d{c[5]}-{c[6]}{c[7]}c{int(c[8])}w{c[9][0]},{c[9][1]}br{int(c[10])}"


@pytest.mark.parametrize("mode", [1, -1], ids=["ds", "recompute"])
@pytest.mark.parametrize("case", CASES, ids=_id)
def test_dense_both_paths(case, mode):
    b, sq, sk, hq, hkv, dqk, dv, dtype, causal, window, br = case
    q, k, v, do = dense_inputs(b, sq, sk, hq, hkv, dqk, dv, dtype)
    kw = dict(causal=causal, window=window, bottom_right=br)
    want = attn.BWD_DS if mode == 1 else attn.BWD_RECOMPUTE
    assert attn.bwd_path(q, k, v, bwd_ds=mode, **kw) == want
    run_and_check(q, k, v, do, dtype=dtype, bwd_ds=mode, **kw)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dims", [(128, 128), (192, 128)])
def test_thd_varlen_ds(dims, causal):
    lens = [0, 1, 129, 300, 64, 200, 0]
    w = synth.Workload("t", 0, 0, 8, 2, dims[0], dims[1], dtype="bf16", thd_total=1)
    inp = synth.make_inputs(w, lengths=lens)
    run_and_check(inp["q"], inp["k"], inp["v"], inp["dout"], dtype="bf16", causal=causal,
                  cu=inp["cu_seqlens"], max_len=inp["max_seqlen"], bwd_ds=1)


def _fwd(dims, s=500, hq=4, hkv=2):
    q, k, v, do = dense_inputs(1, s, s, hq, hkv, dims[0], dims[1], "bf16")
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn.fwd(qd, kd, vd)
    return (q, k, v, do), (qd, kd, vd, dod, o, lse)


@pytest.mark.parametrize("dims", [(128, 128), (192, 128)])
def test_ds_bitwise_reproducible_and_stages_in_order(dims):
    """Two calls give identical gradients; preprocess, dkdv, dq called one by
    one (the order attn_bwd uses on this path) give the one-call result."""
    _, (qd, kd, vd, dod, o, lse) = _fwd(dims)
    g1 = attn.bwd(qd, kd, vd, o, dod, lse, bwd_ds=1)
    g2 = attn.bwd(qd, kd, vd, o, dod, lse, bwd_ds=1)
    ws = torch.empty(attn.workspace_size("bwd", qd, kd, vd, bwd_ds=1), dtype=torch.uint8,
                     device="cuda")
    g3 = [torch.full_like(t, float("nan")) for t in (qd, kd, vd)]
    for st in ("preprocess", "dkdv", "dq"):
        attn.bwd(qd, kd, vd, o, dod, lse, dq=g3[0], dk=g3[1], dv=g3[2], workspace=ws, stage=st,
                 bwd_ds=1)
    attn.query_status(ws)
    torch.cuda.synchronize()
    for a, b_, c in zip(g1, g2, g3):
        assert torch.equal(a, b_) and torch.equal(a, c)


def test_ds_and_recompute_agree_and_dkdv_identical():
    """The paths differ only in how dQ is formed: dK and dV come from the same
    kernel and are bit-identical; dQ agrees to rounding."""
    (q, k, v, do), (qd, kd, vd, dod, o, lse) = _fwd((192, 128), s=700)
    a = attn.bwd(qd, kd, vd, o, dod, lse, bwd_ds=1)
    b_ = attn.bwd(qd, kd, vd, o, dod, lse, bwd_ds=-1)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b_[1]) and torch.equal(a[2], b_[2])
    d = (a[0].float() - b_[0].float()).norm() / b_[0].float().norm()
    assert d < 1e-2, float(d)


def test_ds_fp32_accumulate_adds_into_gradients():
    (q, k, v, do), (qd, kd, vd, dod, o, lse) = _fwd((128, 128))
    fresh = attn.bwd(qd, kd, vd, o, dod, lse, grad_dtype=torch.float32, bwd_ds=1)
    g = torch.Generator(device="cuda").manual_seed(3)
    prev = [torch.randn(t.shape, generator=g, device="cuda") for t in fresh]
    acc = [p.clone() for p in prev]
    attn.bwd(qd, kd, vd, o, dod, lse, dq=acc[0], dk=acc[1], dv=acc[2], grad_dtype=torch.float32,
             accumulate=True, bwd_ds=1)
    torch.cuda.synchronize()
    for a, p, f in zip(acc, prev, fresh):
        assert torch.allclose(a, p + f, rtol=1e-6, atol=1e-6)


def test_noalloc_takes_the_recompute_path():
    """attn_bwd_noalloc (8 MiB static scratch) runs the recompute backward
    under bwd_ds = 0, and gives attn_bwd's results on that path."""
    _, (qd, kd, vd, dod, o, lse) = _fwd((192, 128), s=300)
    a = attn.bwd_noalloc(qd, kd, vd, o, dod, lse)
    b_ = attn.bwd(qd, kd, vd, o, dod, lse, bwd_ds=-1)
    torch.cuda.synchronize()
    for x, y in zip(a, b_):
        assert torch.equal(x, y)


def test_ds_gqa_group_and_oracle_rel_l2():
    """GQA 8:1 at 192/128 over several query tiles of a longer sequence."""
    q, k, v, do = dense_inputs(1, 1100, 1100, 8, 1, 192, 128, "bf16")
    scale = 1.0 / math.sqrt(192)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn.fwd(qd, kd, vd)
    dq, dk, dv = attn.bwd(qd, kd, vd, o, dod, lse, bwd_ds=1)
    torch.cuda.synchronize()
    ref = Reference(q, k, v, do, causal=True, scale=scale, dtype="bf16")
    for name, got, ex in (("dq", dq, ref.dq), ("dk", dk, ref.dk), ("dv", dv, ref.dv)):
        gate(name, got, ex, ref.floor[name])
        rel_l2(name, got, ex)
