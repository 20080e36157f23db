"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (latency-bound serving loops, plugin hosts that plan all device
memory in advance, code inside another runtime's callbacks) may not call
cudaMalloc mid-run and often have no allocator to carve a workspace from, so
this entry point uses the library's fixed 8 MiB static scratch area instead of
a caller workspace.  The test calls it through the C ABI twice in a row, with
different inputs, and checks each result against attn_bwd's (the backward is
deterministic, so the results must match exactly).  It sits in a file that
pytest collects last, and it also passes when run alone in a fresh process.
"""
import ctypes
import math

import pytest
import torch

from bwd_tcgen05_tmem_gb300 import attn, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from bwd_tcgen05_tmem_gb300 import build
    build.build()
    attn.load()


def _problem(seed_shift, s=333, hq=4, hkv=2, dqk=192, dv=128):
    dt = torch.bfloat16
    q = synth.normal((1, s, hq, dqk), synth.SEED_Q + seed_shift, dt).cuda()
    k = synth.normal((1, s, hkv, dqk), synth.SEED_K + seed_shift, dt).cuda()
    v = synth.normal((1, s, hkv, dv), synth.SEED_V + seed_shift, dt).cuda()
    do = synth.normal((1, s, hq, dv), synth.SEED_DO + seed_shift, dt).cuda()
    return q, k, v, do


@pytest.mark.parametrize("shape", [dict(s=333, hq=4, hkv=2, dqk=192, dv=128),
                                   dict(s=200, hq=4, hkv=1, dqk=512, dv=512)],
                         ids=["fused-192-128", "materialising-d512-gqa"])
def test_noalloc_backward_matches_attn_bwd_twice(shape):
    # the d512 case runs the materialising backward, whose P/dS blocks
    # (768 KiB here) also live in the static scratch area
    for call, shift in enumerate((0, 10)):
        q, k, v, do = _problem(shift, **shape)
        scale = 1.0 / math.sqrt(q.shape[-1])
        o, lse = attn.fwd(q, k, v, scale=scale)
        ref = attn.bwd(q, k, v, o, do, lse, scale=scale)
        got = attn.bwd_noalloc(q, k, v, o, do, lse, scale=scale)
        torch.cuda.synchronize()
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(a).all(), (call, name)
            assert torch.equal(a, b), (call, name, (a.float() - b.float()).abs().max().item())


def test_noalloc_refuses_problems_beyond_its_scratch():
    # 2 x 4096 x 300 (rows x query heads) x 8 bytes of row statistics exceed the 8 MiB area
    q = torch.empty((2, 4096, 300, 64), dtype=torch.bfloat16, device="meta")
    p = attn.make_params(q, q, q)
    lib = attn.load()
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) > (8 << 20)
    rc = lib.attn_bwd_noalloc(ctypes.byref(p), *([None] * 10))
    assert rc == 4  # ATTN_ERR_WORKSPACE, nothing launched
