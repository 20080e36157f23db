"""attn_lse_merge on the GPU against the oracle's merge, edge cases included.

The merge is the context-parallel ring correction (TransformerEngine PR #3527
description: partial results are combined by exponentiating LSE differences):
LSE = ln sum_p exp(LSE_p), O = sum_p exp(LSE_p - LSE) O_p over the parts that
cover a row.  Cases: parts that cover only part of the rows, a part that is
-inf everywhere (its O is NaN-poisoned: a -inf part must not be read), rows
whose parts are all -inf (O = 0, LSE = -inf), LSE values large enough that an
unshifted exponential would overflow FP32, and all three output types.

The oracle takes every part over all rows, so a part that does not cover a row
is given to it as LSE = -inf there (weight 0 by the definition above).

Tolerance, from the arithmetic: the kernel merges in FP32 (fast exponential
and logarithm, a few ulp of relative error for arguments down to -90) and
rounds O to the output type once, so |O - exact| <= u * |exact| + 1e-5 * max|O|
with u the output type's unit roundoff (2^-8 BF16, 2^-11 FP16, 1e-5 FP32);
LSE within the 1e-4 gate the attention tests use.
"""
import numpy as np
import pytest
import torch

import oracle
from bwd_tcgen05_tmem_gb300 import attn
from parity import LSE_ATOL

pytestmark = pytest.mark.gpu

UNIT = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11, torch.float32: 1e-5}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from bwd_tcgen05_tmem_gb300 import build
    build.build()
    attn.load()


def make_parts(rows, heads, dv, seed):
    g = torch.Generator().manual_seed(seed)
    # (first row, rows) of each part
    ranges = [(0, rows), (0, 120), (100, 150), (250, rows - 250), (0, rows), (37, 1)]
    o_parts, lse_parts = [], []
    for i, (r0, n) in enumerate(ranges):
        o = torch.randn(n, heads, dv, generator=g)
        lse = torch.randn(heads, n, generator=g) * 3.0
        if i == 2:
            lse += 85.0  # exp(LSE) overflows FP32 unless the maximum is subtracted
        if i == 4:  # -inf everywhere; its O must not be read
            lse.fill_(float("-inf"))
            o.fill_(float("nan"))
        o_parts.append(o)
        lse_parts.append(lse)
    # rows [280, rows) see no key in any part: -inf in every part covering them
    for (r0, n), lse in zip(ranges, lse_parts):
        lo, hi = max(280, r0), min(rows, r0 + n)
        if lo < hi:
            lse[:, lo - r0:hi - r0] = float("-inf")
    # one row where every part but one is -inf
    for i, ((r0, n), lse) in enumerate(zip(ranges, lse_parts)):
        if i != 1 and r0 <= 50 < r0 + n:
            lse[:, 50 - r0] = float("-inf")
    return ranges, o_parts, lse_parts


def oracle_merge(ranges, o_parts, lse_parts, rows, heads, dv):
    n = len(ranges)
    op = np.zeros((n, rows, heads, dv))
    lp = np.full((n, heads, rows), -np.inf)
    for i, ((r0, nr), o, lse) in enumerate(zip(ranges, o_parts, lse_parts)):
        ov = o.double().numpy()
        lv = lse.double().numpy()
        # a -inf entry has weight 0: give the oracle a finite O there
        ov = np.where(np.isneginf(lv).T[:, :, None], 0.0, ov)
        op[i, r0:r0 + nr] = ov
        lp[i, :, r0:r0 + nr] = lv
    return oracle.lse_merge(op, lp)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("dv", [128, 64, 12])
def test_lse_merge_matches_oracle(out_dtype, dv):
    rows, heads = 300, 3
    ranges, o_parts, lse_parts = make_parts(rows, heads, dv, seed=40 + dv)
    eo, el = oracle_merge(ranges, o_parts, lse_parts, rows, heads, dv)
    out, lse = attn.lse_merge([o.cuda() for o in o_parts], [l.cuda() for l in lse_parts],
                              [r[0] for r in ranges], [r[1] for r in ranges], rows,
                              out_dtype=out_dtype)
    torch.cuda.synchronize()
    got_o = out.double().cpu().numpy()
    got_l = lse.double().cpu().numpy()
    assert np.array_equal(np.isneginf(got_l), np.isneginf(el))
    assert np.isneginf(el[:, 280:]).all()
    fin = np.isfinite(el)
    assert np.max(np.abs(got_l[fin] - el[fin])) <= LSE_ATOL
    assert np.all(np.isfinite(got_o))
    assert np.all(got_o[280:] == 0)
    tol = UNIT[out_dtype] * np.abs(eo) + 1e-5 * np.max(np.abs(eo))
    err = np.abs(got_o - eo)
    assert np.all(err <= tol), float(np.max(err - tol))


def test_lse_merge_single_part_is_identity_in_fp32():
    """One part covering every row: LSE unchanged and O equal to it up to the
    FP32 rounding of the weight exp(LSE - LSE) = 1."""
    rows, heads, dv = 257, 2, 128
    g = torch.Generator().manual_seed(3)
    o = torch.randn(rows, heads, dv, generator=g).cuda()
    lse = (torch.randn(heads, rows, generator=g) * 5).cuda()
    out, l2 = attn.lse_merge([o], [lse], [0], [rows], rows, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.allclose(l2, lse, atol=1e-6, rtol=0)
    assert torch.allclose(out, o, atol=0, rtol=1e-6)
