"""The C-ABI library (CPU-side checks only; nothing here computes on a GPU).

* libattn.so builds for sm_103a and exports every function include/attn.h
  declares;
* the host-side validation refuses bad requests with the documented status
  codes before anything is launched (TransformerEngine PR #3527: unsupported
  configurations are refused rather than approximated).
"""
import ctypes
import os
import re

import pytest
import torch

from bwd_tcgen05_tmem_gb300 import attn, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return attn.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(attn.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), n


def fake(shape, dtype=torch.bfloat16):
    # meta tensors give shapes and strides without memory; pointers are never used
    return torch.empty(shape, dtype=dtype, device="meta")


def call_fwd(lib, p, q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, ws=0x6000,
             ws_bytes=1 << 20):
    return lib.attn_fwd(ctypes.byref(p), ctypes.c_void_p(q), ctypes.c_void_p(k),
                        ctypes.c_void_p(v), ctypes.c_void_p(o), ctypes.c_void_p(lse),
                        ctypes.c_void_p(ws), ws_bytes, None)


def base_params(**kw):
    q = fake((2, 256, 4, 128))
    k = fake((2, 256, 2, 128))
    v = fake((2, 256, 2, 128))
    o = fake((2, 256, 4, 128))
    return attn.make_params(q, k, v, o=o, **kw)


@pytest.mark.parametrize("mutate,code", [
    (lambda p: setattr(p, "d_qk", 96), 2),            # unsupported head dim
    (lambda p: setattr(p, "d_qk", 100), 1),           # not a multiple of 8
    (lambda p: setattr(p, "heads_kv", 3), 1),         # GQA divisibility
    (lambda p: setattr(p, "window_left", -2), 1),     # window must be >= -1
    (lambda p: setattr(p, "softmax_scale", 0.0), 1),  # scale must be positive
    (lambda p: setattr(p, "dtype", 2), 2),            # FP32 inputs refused
    (lambda p: setattr(p, "o_dtype", 1), 2),          # O dtype mix refused
    (lambda p: p.stride_q.__setitem__(1, 4 * 128 + 4), 3),  # stride not 16-byte multiple
])
def test_validation_refuses(lib, mutate, code):
    p = base_params()
    mutate(p)
    assert call_fwd(lib, p) == code
    assert lib.attn_last_error()


def test_misaligned_pointer_and_workspace(lib):
    p = base_params()
    assert call_fwd(lib, p, q=0x1008) == 3
    assert call_fwd(lib, p, ws=0) == 4
    assert call_fwd(lib, p, ws_bytes=16) == 4
    assert call_fwd(lib, p, ws=0x6010) == 3


def test_output_overlapping_input_refused(lib):
    p = base_params()
    assert call_fwd(lib, p, o=0x1000) == 1


def test_workspace_sizes(lib):
    p = base_params()
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) >= 256
    need = lib.attn_bwd_workspace_size(ctypes.byref(p))
    assert need >= 256 + 2 * 4 * 256 * 8  # status word + {LSE log2 e, D} for every query row


def test_merge_validation(lib):
    n = 2
    vp = (ctypes.c_void_p * n)(0x1000, 0x2000)
    lp = (ctypes.c_void_p * n)(0x3000, 0x4000)
    r0 = (ctypes.c_int64 * n)(0, 5)
    nr = (ctypes.c_int64 * n)(10, 10)  # second part exceeds rows
    rc = lib.attn_lse_merge(n, vp, lp, r0, nr, 12, 2, 64, ctypes.c_void_p(0x9000), 0,
                            ctypes.c_void_p(0xA000), None)
    assert rc == 1
    rc = lib.attn_lse_merge(0, vp, lp, r0, nr, 12, 2, 64, ctypes.c_void_p(0x9000), 0,
                            ctypes.c_void_p(0xA000), None)
    assert rc == 1


def _visible_blocks(sq, sk, causal, wl, wr, bottom_right):
    """Brute force: 128x128 (query tile, key block) pairs holding a visible key."""
    off = sk - sq if bottom_right else 0
    n = 0
    for qt in range((sq + 127) // 128):
        blocks = set()
        for i in range(qt * 128, min(qt * 128 + 128, sq)):
            lo = 0 if wl < 0 else max(0, i + off - wl)
            hi = sk - 1
            if causal:
                hi = min(hi, i + off)
            elif wr >= 0:
                hi = min(hi, i + off + wr)
            for j in range(lo, hi + 1, 1):
                blocks.add(j // 128)
        n += len(blocks)
    return n


@pytest.mark.parametrize("sq,sk,causal,wl,wr,br", [
    (300, 300, True, -1, -1, False), (200, 333, True, -1, -1, True),
    (333, 200, True, -1, -1, True), (300, 300, False, 100, 30, False),
    (700, 700, True, 129, 0, False), (260, 260, False, -1, -1, False)])
def test_wide_backward_workspace_counts_visible_blocks(lib, sq, sk, causal, wl, wr, br):
    """Head dim 512: one 64 KiB block of P/dS per visible (query tile, key block)."""
    b, hq, hkv = 2, 4, 2
    q, k = fake((b, sq, hq, 512)), fake((b, sk, hkv, 512))
    p = attn.make_params(q, k, k, o=q, causal=causal, window=(wl, wr), bottom_right=br)
    base = 256 + -(-(b * sq * hq * 8) // 256) * 256
    blk_off = -(-(base + (b + 1) * 8) // 1024) * 1024
    blocks = b * hq * _visible_blocks(sq, sk, causal, wl, wr, br)
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == blk_off + blocks * 65536


def test_cp_relayout_validation(lib):
    arr = ctypes.c_int64 * 3
    # contiguous [cp, 2*chunk, heads, d] sequence side and [cp, S, heads/cp, d] head side;
    # every call below is refused before anything is launched (the pointers are fake)
    seq_s, head_s = arr(256 * 8 * 64, 8 * 64, 64), arr(1024 * 2 * 64, 2 * 64, 64)

    def call(to_heads=1, cp=4, seqlen=1024, heads=8, d=64, eb=2, src=0x100000, dst=0x40000000):
        return lib.attn_cp_relayout(to_heads, cp, seqlen, heads, d, eb, ctypes.c_void_p(src),
                                    seq_s, ctypes.c_void_p(dst), head_s, None)
    assert call(seqlen=1001) == 1          # not 2*cp chunks
    assert call(heads=6) == 1              # heads % cp
    assert call(eb=3) == 1                 # element size
    assert call(cp=0) == 1
    assert call(src=0x100001) == 3         # misaligned
    assert call(dst=0x100000 + 64) == 1    # overlapping src/dst


def test_seqused_validation(lib):
    p = base_params()
    p.seqused_q = 0x7000  # dense tensors: seqused needs THD
    p.seqused_k = 0x7000
    assert call_fwd(lib, p) == 1
    q = fake((64, 4, 128))
    cu = torch.zeros(3, dtype=torch.int32)  # host tensor: only its address is read
    p = attn.make_params(q, fake((64, 2, 128)), fake((64, 2, 128)), o=q, cu_seqlens_q=cu,
                         max_seqlen_q=64, max_seqlen_k=64)
    p.seqused_q = 0x7000  # only one of the pair
    assert call_fwd(lib, p) == 1
    p.seqused_k = 0x7002  # misaligned
    assert call_fwd(lib, p) == 3


@pytest.mark.parametrize("s,window,wide", [(700, (-1, -1), True), (700, (100, 0), True),
                                           (65536, (-1, -1), False), (65536, (1023, 0), True)])
def test_d256_backward_route_by_block_bytes(lib, s, window, wide):
    """Head dim 256 materialises P/dS while the blocks take at most 16 GiB (the
    fused path would need two recomputing dK/dV launches); beyond that the
    workspace is the status word and D alone."""
    b, hq, hkv = 1, 4, 1
    q, k = fake((b, s, hq, 256)), fake((b, s, hkv, 256))
    p = attn.make_params(q, k, k, o=q, causal=True, window=window)
    base = 256 + -(-(b * s * hq * 8) // 256) * 256
    need = lib.attn_bwd_workspace_size(ctypes.byref(p))
    if not wide:
        assert need == base
    else:
        blk_off = -(-(base + (b + 1) * 8) // 1024) * 1024
        nq, nk = (s + 127) // 128, (s + 127) // 128
        if s <= 2048:
            blocks = b * hq * _visible_blocks(s, s, True, window[0], window[1], False)
        else:  # closed form: causal with a window of 1024 -> 9 blocks per query tile at most
            blocks = b * hq * sum(min(qt, (1023 + 127) // 128 + 1) if qt > 8 else qt + 1
                                  for qt in range(nq))
        assert need == blk_off + blocks * 65536


def host_step_params():
    q, k, v = fake((2, 256, 4, 128)), fake((2, 256, 2, 128)), fake((2, 256, 2, 128))
    o, do = fake((2, 256, 4, 128)), fake((2, 256, 4, 128))
    dq, dk, dv = (fake(t.shape, torch.float32) for t in (q, k, v))
    return attn.make_params(q, k, v, o=o, dout=do, dq=dq, dk=dk, dv=dv,
                            grad_dtype=torch.float32), (q, k, v, do, o, dq, dk, dv)


def test_host_arena_size_is_workspaces_plus_tensor_copies(lib):
    """attn_fwd_bwd_host's arena: forward workspace, backward workspace, then
    the nine tensors, each rounded up to 256 bytes (include/attn.h)."""
    p, ts = host_step_params()
    up = lambda x: (x + 255) // 256 * 256
    nbytes = [t.numel() * t.element_size() for t in ts]  # contiguous: span = numel
    lse = 2 * 4 * 256 * 4
    want = (up(lib.attn_fwd_workspace_size(ctypes.byref(p))) +
            up(lib.attn_bwd_workspace_size(ctypes.byref(p))) + sum(up(b) for b in nbytes) + up(lse))
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) == 256  # status word at arena + 0
    assert lib.attn_host_arena_size(ctypes.byref(p)) == want
    bad, _ = host_step_params()
    bad.d_qk = 96
    assert lib.attn_host_arena_size(ctypes.byref(bad)) == 0


def test_host_step_refuses_bad_arena(lib):
    p, _ = host_step_params()
    need = lib.attn_host_arena_size(ctypes.byref(p))

    def call(arena, nbytes):
        ptrs = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(9)]
        return lib.attn_fwd_bwd_host(ctypes.byref(p), *ptrs, ctypes.c_void_p(arena), nbytes, None)

    assert call(0, need) == 4
    assert call(0x7000100, need - 1) == 4
    assert call(0x7000010, need) == 3
    p.heads_kv = 3
    assert call(0x7000100, need) == 1


def test_host_stages_mask_validated(lib):
    p, _ = host_step_params()
    need = lib.attn_host_arena_size(ctypes.byref(p))
    ptrs = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(9)]
    for bad in (0, 8, 15):
        assert lib.attn_fwd_bwd_host_stages(ctypes.byref(p), *ptrs, ctypes.c_void_p(0x7000100),
                                            need, bad, None) == 1


@pytest.mark.parametrize("dims,sq,sk,causal,wl,wr,br", [
    ((192, 128), 300, 300, True, -1, -1, False), ((128, 128), 200, 333, True, -1, -1, True),
    ((192, 128), 333, 200, True, -1, -1, True), ((128, 128), 300, 300, False, 100, 30, False),
    ((192, 128), 700, 700, True, 129, 0, False), ((128, 128), 260, 260, False, -1, -1, False)])
def test_ds_backward_workspace_counts_visible_blocks(lib, dims, sq, sk, causal, wl, wr, br):
    """Head dims 128/128 and 192/128 keep dS: one 32 KiB block per visible
    (query tile, key block) and query head, after the status word, D and the
    per-sequence block prefix; bwd_ds = -1 leaves the status word and D."""
    b, hq, hkv = 2, 4, 2
    q, k, v = fake((b, sq, hq, dims[0])), fake((b, sk, hkv, dims[0])), fake((b, sk, hkv, dims[1]))
    o = fake((b, sq, hq, dims[1]))
    kw = dict(o=o, causal=causal, window=(wl, wr), bottom_right=br)
    base = 256 + -(-(b * sq * hq * 8) // 256) * 256
    blk_off = -(-(base + (b + 1) * 8) // 1024) * 1024
    blocks = b * hq * _visible_blocks(sq, sk, causal, wl, wr, br)
    p = attn.make_params(q, k, v, bwd_ds=1, **kw)
    assert lib.attn_bwd_path(ctypes.byref(p)) == attn.BWD_DS
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == blk_off + blocks * 32768
    p = attn.make_params(q, k, v, **kw)  # auto keeps dS at both head dims
    assert lib.attn_bwd_path(ctypes.byref(p)) == attn.BWD_DS
    p = attn.make_params(q, k, v, bwd_ds=-1, **kw)
    assert lib.attn_bwd_path(ctypes.byref(p)) == attn.BWD_RECOMPUTE
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == base


@pytest.mark.parametrize("b,s,dims,mode,path", [
    (1, 32768, (192, 128), 0, 1),    # 32 heads: 1,052,672 blocks, 34.5 GB: kept
    (8, 32768, (192, 128), 0, 0),    # 276 GB of blocks: above the 64 GiB cap, recompute
    (8, 32768, (192, 128), 1, 1),    # ... unless forced
    (1, 32768, (128, 128), 0, 1),    # 128/128 keeps dS as well
    (1, 32768, (128, 128), -1, 0),
    (1, 300, (64, 64), 0, 0),        # 64/64 always recomputes (cheaper than streaming dS)
    (1, 300, (64, 64), 1, 0),
    (1, 300, (256, 256), 0, 2),      # P and dS (the wide path)
    (1, 300, (512, 512), -1, 2),
    (1, 300, (192, 128), 2, -1),     # invalid bwd_ds
])
def test_bwd_path_selection(lib, b, s, dims, mode, path):
    hq = 32
    q, k = fake((b, s, hq, dims[0])), fake((b, s, hq, dims[0]))
    v, o = fake((b, s, hq, dims[1])), fake((b, s, hq, dims[1]))
    p = attn.make_params(q, k, v, o=o, causal=True, bwd_ds=mode)
    assert lib.attn_bwd_path(ctypes.byref(p)) == path
    if path == attn.BWD_DS:
        nq = (s + 127) // 128
        blocks = b * hq * nq * (nq + 1) // 2
        base = 256 + -(-(b * s * hq * 8) // 256) * 256
        blk_off = -(-(base + (b + 1) * 8) // 1024) * 1024
        assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == blk_off + blocks * 32768


@pytest.mark.parametrize("dims,causal,order", [
    ((192, 128), True, ("dkdv", "dq")),    # dS path: the dkdv stage writes the blocks
    ((128, 128), False, ("dkdv", "dq")),
    ((64, 64), True, ("dq", "dkdv")),      # recompute
    ((512, 512), False, ("dq", "dkdv")),   # P/dS: the scores kernel runs in the dq stage
])
def test_cp_stage_order_follows_the_path(lib, dims, causal, order):
    """The CP schedules run each call's stages in the order its path needs."""
    from bwd_tcgen05_tmem_gb300 import cp as cpmod
    q, k = fake((1, 4096, 8, dims[0])), fake((1, 2048, 8, dims[0]))
    v = fake((1, 2048, 8, dims[1]))
    assert cpmod.stage_order(q, k, v, causal=causal) == order
