"""Bounded waits: a wait that runs out unwinds the kernel instead of hanging it.

Every mbarrier wait in the attention kernels has a wall-clock limit; when one
expires the CTA raises ATTN_ERR_TIMEOUT in the status word, lets its in-flight
copies land, drains its MMAs, frees its TMEM and returns.  This is the guard
against the class of bug TransformerEngine PR #3699's review found in a
backward kernel (a "missing wait" on a reused barrier phase): with it such a
bug shows up as a status, not as a hung GPU.

Each case arms the library's test-only fault injection (attn_debug_inject) so
that the first CTA of one kernel leaves out one of its loads and waits at most
20 ms.  The test checks that the call then reports ATTN_ERR_TIMEOUT through
attn_query_status (so the kernel returned and the stream synchronised), and
that the next, normal call on the same device and workspace gives results
bit-identical to a call made before the fault, which themselves pass the
2x-naive parity gate against the FP64 oracle.  No wait here is endless and
nothing traps: the dropped load only makes one bounded wait run out.
"""
import math

import pytest
import torch

from bwd_tcgen05_tmem_gb300 import attn
from parity import Reference, check_lse, gate, rel_l2
from test_gpu_parity import dense_inputs

pytestmark = pytest.mark.gpu

WAIT_NS = 20_000_000  # 20 ms wait limit while a load is left out

CASES = [
    # id, (dqk, dv), hq, hkv, seqlen, kernel bit, dropped load, bwd_ds
    ("fwd-192", (192, 128), 2, 2, 300, attn.DEBUG_FWD, 1, 0),
    ("ds-dq-gemm-192", (192, 128), 2, 2, 300, attn.DEBUG_DQ, 1, 0),
    ("ds-dkdv-192", (192, 128), 2, 2, 300, attn.DEBUG_DKDV, 1, 0),
    ("dq-192", (192, 128), 2, 2, 300, attn.DEBUG_DQ, 1, -1),
    ("dkdv-192", (192, 128), 2, 2, 300, attn.DEBUG_DKDV, 1, -1),
    ("ds-dkdv-128-gqa", (128, 128), 4, 2, 300, attn.DEBUG_DKDV, 3, 1),
    # at head dim 128 the dQ GEMM has a K producer warp of its own, which must
    # unwind too when a dS copy is missing
    ("ds-dq-gemm-128-gqa", (128, 128), 4, 2, 300, attn.DEBUG_DQ, 1, 1),
    ("dkdv-128-gqa", (128, 128), 4, 2, 300, attn.DEBUG_DKDV, 3, -1),
    ("fwd-512", (512, 512), 4, 1, 300, attn.DEBUG_FWD, 1, 0),
    ("scores-512", (512, 512), 4, 1, 300, attn.DEBUG_SCORES, 5, 0),
    ("wide-dq-512", (512, 512), 4, 1, 300, attn.DEBUG_DQ, 1, 0),
    ("wide-dkdv-512", (512, 512), 4, 1, 300, attn.DEBUG_DKDV, 1, 0),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from bwd_tcgen05_tmem_gb300 import build
    build.build()
    attn.load()


def _expect_timeout(ws):
    with pytest.raises(attn.AttnError) as e:
        attn.query_status(ws)
    assert e.value.code == 6, str(e.value)  # ATTN_ERR_TIMEOUT


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_expired_wait_reports_timeout_and_device_recovers(case):
    _, dims, hq, hkv, s, bit, drop, mode = case
    q, k, v, do = dense_inputs(1, s, s, hq, hkv, dims[0], dims[1], "bf16")
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    fws = torch.empty(attn.workspace_size("fwd", qd, kd, vd), dtype=torch.uint8, device="cuda")
    bws = torch.empty(attn.workspace_size("bwd", qd, kd, vd, bwd_ds=mode), dtype=torch.uint8,
                      device="cuda")
    # results before the fault
    o, lse = attn.fwd(qd, kd, vd, workspace=fws)
    g = attn.bwd(qd, kd, vd, o, dod, lse, workspace=bws, bwd_ds=mode)
    attn.query_status(bws)
    o, lse, g = o.clone(), lse.clone(), [t.clone() for t in g]

    nan = float("nan")
    o2 = torch.full_like(o, nan)
    lse2 = torch.full_like(lse, nan)
    g2 = [torch.full_like(t, nan) for t in (qd, kd, vd)]
    if bit == attn.DEBUG_FWD:
        attn.debug_inject(bit, drop, WAIT_NS)
        attn.fwd(qd, kd, vd, out=o2, lse=lse2, workspace=fws)
        _expect_timeout(fws)
        attn.fwd(qd, kd, vd, out=o2, lse=lse2, workspace=fws)  # normal again
        attn.query_status(fws)
    else:
        attn.debug_inject(bit, drop, WAIT_NS)
        attn.bwd(qd, kd, vd, o, dod, lse, dq=g2[0], dk=g2[1], dv=g2[2], workspace=bws,
                 bwd_ds=mode)
        _expect_timeout(bws)
        attn.fwd(qd, kd, vd, out=o2, lse=lse2, workspace=fws)
        attn.bwd(qd, kd, vd, o, dod, lse, dq=g2[0], dk=g2[1], dv=g2[2], workspace=bws,
                 bwd_ds=mode)
        attn.query_status(bws)
    torch.cuda.synchronize()
    assert torch.equal(o2, o) and torch.equal(lse2, lse)
    if bit != attn.DEBUG_FWD:
        for a, b in zip(g2, g):
            assert torch.equal(a, b)
    # and those results pass parity against the oracle
    ref = Reference(q, k, v, do, causal=True, scale=1.0 / math.sqrt(dims[0]), dtype="bf16")
    gate("o", o2, ref.o, ref.floor["o"])
    check_lse(lse2, ref.lse)
    if bit != attn.DEBUG_FWD:
        for name, got, ex in zip(("dq", "dk", "dv"), g2, (ref.dq, ref.dk, ref.dv)):
            gate(name, got, ex, ref.floor[name])
            rel_l2(name, got, ex)


def test_injection_is_cleared_after_one_call():
    """The injection arms exactly one call: the call after it is normal."""
    q, k, v, _ = dense_inputs(1, 300, 300, 2, 2, 192, 128, "bf16")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    attn.debug_inject(attn.DEBUG_FWD, 1, WAIT_NS)
    attn.fwd(qd, kd, vd, workspace=ws)
    _expect_timeout(ws)
    o, lse = attn.fwd(qd, kd, vd, workspace=ws)
    attn.query_status(ws)
    ref_o, ref_l = attn.fwd(qd, kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
