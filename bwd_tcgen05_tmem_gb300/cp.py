"""One-GPU emulation of context-parallel (CP) causal attention with the
dual-chunk-swap load balance, forward and backward.

The sequence is cut into 2*cp chunks; rank r holds chunks r and 2cp-1-r
(TransformerEngine PR #3527: ``DUAL_CHUNK_SWAP`` CP layout).  In the p2p ring,
at step s rank r sees the key/value chunks of rank r' = (r - s) mod cp; the
per-step kernel window is causal ``(-1, 0)`` at step 0 and full ``(-1, -1)``
otherwise (PR #3527 review notes on the p2p path), and the partial results are
combined through their LSE (the ring correction):

* s = 0:   both local query chunks vs both local key chunks, causal over the
           rank's local concatenation;
* r' < r:  both query chunks vs key chunk r' only, full;
* r' > r:  query chunk 2cp-1-r only vs both key chunks, full.

Every rank's data lives on this one GPU, so the "exchange" of step s is the
address of rank r''s shard; there are no collectives.  All arithmetic runs in
the library's kernels: ``attn_fwd`` writes FP32 partials, ``attn_lse_merge``
combines them, and ``attn_bwd`` (FP32 gradients, ``accumulate``) adds each
step's dQ into the rank's rows and its dK/dV into the source rank's rows.
"""
from __future__ import annotations

import dataclasses

import torch

from . import attn

# The ring and all-gather schedules run the backward's stages themselves (the
# dkdv stages that add into shared dK/dV run one after another, the dq stages
# of different calls overlap on their streams) and keep one workspace per
# query-row set across ring steps.  Each call takes the path the library picks
# for its shape (attn_bwd_path): on the dS path the dkdv stage writes the dS
# blocks that the dq stage of the same call then reads, so dkdv goes first.


def stage_order(q, k, v, **kw):
    """The dq / dkdv stages of one attn_bwd call in the order its path needs."""
    return ("dkdv", "dq") if attn.bwd_path(q, k, v, **kw) == attn.BWD_DS else ("dq", "dkdv")


@dataclasses.dataclass
class Piece:
    rank: int
    src: int
    q_rows: tuple   # (first, count) rows of the rank's local query shard
    k_rows: tuple   # (first, count) rows of the source rank's local key shard
    causal: bool


def ring_pieces(cp: int, chunk: int):
    """The (rank, step) pieces of the dual-chunk-swap p2p ring, per rank."""
    out = []
    for r in range(cp):
        pcs = []
        for s in range(cp):
            src = (r - s) % cp
            if s == 0:
                pcs.append(Piece(r, src, (0, 2 * chunk), (0, 2 * chunk), True))
            elif src < r:
                pcs.append(Piece(r, src, (0, 2 * chunk), (0, chunk), False))
            else:
                pcs.append(Piece(r, src, (chunk, chunk), (0, 2 * chunk), False))
        out.append(pcs)
    return out


def shard(x, cp):
    """[B, S, H, d] -> list of cp local shards [B, 2c, H, d] (chunks r, 2cp-1-r)."""
    s = x.shape[1]
    c = s // (2 * cp)
    assert c * 2 * cp == s, "sequence must split into 2*cp equal chunks"
    return [torch.cat([x[:, r * c:(r + 1) * c], x[:, (2 * cp - 1 - r) * c:(2 * cp - r) * c]],
                      dim=1).contiguous() for r in range(cp)]


def unshard(shards, cp):
    """Inverse of ``shard`` along dim 1."""
    c = shards[0].shape[1] // 2
    parts = [None] * (2 * cp)
    for r, t in enumerate(shards):
        parts[r] = t[:, :c]
        parts[2 * cp - 1 - r] = t[:, c:]
    return torch.cat(parts, dim=1)


def unshard_lse(shards, cp):
    """LSE shards [B, H, 2c] -> [B, H, S]."""
    c = shards[0].shape[2] // 2
    parts = [None] * (2 * cp)
    for r, t in enumerate(shards):
        parts[r] = t[:, :, :c]
        parts[2 * cp - 1 - r] = t[:, :, c:]
    return torch.cat(parts, dim=2)


class _Streams:
    """One CUDA stream per emulated rank, forked from and joined back into the
    caller's current stream, so the ranks' launches overlap on the GPU."""

    def __init__(self, n, device):
        self.s = [torch.cuda.Stream(device=device) for _ in range(n)]

    def fork(self):
        cur = torch.cuda.current_stream()
        for st in self.s:
            st.wait_stream(cur)

    def join(self):
        cur = torch.cuda.current_stream()
        for st in self.s:
            cur.wait_stream(st)


class CPRing:
    """Holds per-rank shards and the buffers of one emulated CP fwd+bwd.

    q/k/v/dout: dense [1, S, H, d] device tensors (batch 1, as the pages'
    32K benchmark).  Buffers are allocated once; ``forward``/``backward`` only
    launch kernels, each rank on its own stream (each with its own workspace).
    """

    def __init__(self, q, k, v, dout, cp=8, scale=None):
        assert q.shape[0] == 1, "the ring emulation runs batch 1"
        self.cp = cp
        self.scale = scale
        self.chunk = q.shape[1] // (2 * cp)
        self.q, self.k, self.v, self.do = (shard(t, cp) for t in (q, k, v, dout))
        self.pieces = ring_pieces(cp, self.chunk)
        dev = q.device
        hq, dv = q.shape[2], v.shape[3]
        rows = 2 * self.chunk
        # FP32 partials per (rank, step), merged outputs, FP32 gradients per rank
        self.o_part = [[torch.empty((1, pc.q_rows[1], hq, dv), dtype=torch.float32, device=dev)
                        for pc in pcs] for pcs in self.pieces]
        self.lse_part = [[torch.empty((1, hq, pc.q_rows[1]), dtype=torch.float32, device=dev)
                          for pc in pcs] for pcs in self.pieces]
        self.o = [torch.empty((1, rows, hq, dv), dtype=q.dtype, device=dev) for _ in range(cp)]
        self.lse = [torch.empty((1, hq, rows), dtype=torch.float32, device=dev)
                    for _ in range(cp)]
        self.dq = [torch.zeros((1, rows, *q.shape[2:]), dtype=torch.float32, device=dev)
                   for _ in range(cp)]
        self.dk = [torch.zeros((1, rows, *k.shape[2:]), dtype=torch.float32, device=dev)
                   for _ in range(cp)]
        self.dv = [torch.zeros((1, rows, *v.shape[2:]), dtype=torch.float32, device=dev)
                   for _ in range(cp)]
        self.fwd_ws = [torch.empty(256, dtype=torch.uint8, device=dev) for _ in range(cp)]
        # one backward workspace per rank and query-row set: D (the preprocess)
        # depends only on the query rows, so it is computed once per rank for
        # all of its rows and once for its second chunk, and every ring step
        # then runs only the dq and dkdv stages on the matching workspace
        c = self.chunk
        shapes = (((0, 2 * c), (0, 2 * c), True), ((0, 2 * c), (0, c), False),
                  ((c, c), (0, 2 * c), False))
        need = max(256, *(attn.workspace_size("bwd", self.q[0][:, q0:q0 + nq],
                                              self.k[0][:, k0:k0 + nk], self.v[0][:, k0:k0 + nk],
                                              causal=cz) for (q0, nq), (k0, nk), cz in shapes))
        order = {(qr, kr[1], cz): stage_order(self.q[0][:, qr[0]:qr[0] + qr[1]],
                                              self.k[0][:, kr[0]:kr[0] + kr[1]],
                                              self.v[0][:, kr[0]:kr[0] + kr[1]], causal=cz)
                 for qr, kr, cz in shapes}
        self.order = [[order[(pc.q_rows, pc.k_rows[1], pc.causal)] for pc in pcs]
                      for pcs in self.pieces]
        self.bwd_ws = [{rq: torch.empty(need, dtype=torch.uint8, device=dev)
                        for rq in ((0, 2 * c), (c, c))} for _ in range(cp)]
        self.streams = _Streams(cp, dev)
        self.launches = 0

    def forward(self):
        """Partials per ring step, then one LSE merge per rank (rank r on stream r)."""
        n = 0
        self.streams.fork()
        for r, pcs in enumerate(self.pieces):
            st = self.streams.s[r]
            for i, pc in enumerate(pcs):
                q0, nq = pc.q_rows
                k0, nk = pc.k_rows
                attn.fwd(self.q[r][:, q0:q0 + nq], self.k[pc.src][:, k0:k0 + nk],
                         self.v[pc.src][:, k0:k0 + nk], causal=pc.causal, scale=self.scale,
                         out=self.o_part[r][i], lse=self.lse_part[r][i],
                         workspace=self.fwd_ws[r], stream=st)
                n += attn.last_launch_count()
            n += self.merge(r, st)
        self.streams.join()
        self.launches = n
        return self.o, self.lse

    def merge(self, r, stream=None):
        """LSE-merge rank r's ring-step partials into its O / LSE; returns the
        number of kernels launched."""
        pcs = self.pieces[r]
        attn.lse_merge([t[0] for t in self.o_part[r]], [t[0] for t in self.lse_part[r]],
                       [pc.q_rows[0] for pc in pcs], [pc.q_rows[1] for pc in pcs],
                       2 * self.chunk, out=self.o[r][0], lse_out=self.lse[r][0], stream=stream)
        return attn.last_launch_count()

    def merge_all(self):
        """Every rank's merge, in order on the current stream (to time the merge
        kernel alone)."""
        for r in range(self.cp):
            self.merge(r)

    def backward(self):
        """Per ring step the dq and dkdv stages of attn_bwd with the merged
        LSE/O and FP32 gradients; D = rowsum(dO * O) of the merged O comes from
        one preprocess per rank and query-row set.

        Step 0 of every rank covers all of its query rows and all of its own key
        rows, so the step-0 calls (run first) overwrite every gradient element
        and the later steps accumulate into them: no zero fill is needed.

        Rank r runs on stream r.  Its step s adds into the dK/dV shard of rank
        (r - s) mod cp, which rank r - 1 added into at step s - 1, so each call
        waits for that one call (an event) and nothing else."""
        n = 0
        rows = 2 * self.chunk
        cp = self.cp
        done = [[None] * cp for _ in range(cp)]
        self.streams.fork()

        def call(r, pc, stage, accumulate):
            q0, nq = pc.q_rows
            k0, nk = pc.k_rows
            lse = self.lse[r][:, :, q0:]  # rows q0.. of the merged LSE, head stride `rows`
            attn.bwd(self.q[r][:, q0:q0 + nq], self.k[pc.src][:, k0:k0 + nk],
                     self.v[pc.src][:, k0:k0 + nk], self.o[r][:, q0:q0 + nq],
                     self.do[r][:, q0:q0 + nq], lse, causal=pc.causal, scale=self.scale,
                     dq=self.dq[r][:, q0:q0 + nq], dk=self.dk[pc.src][:, k0:k0 + nk],
                     dv=self.dv[pc.src][:, k0:k0 + nk], grad_dtype=torch.float32,
                     accumulate=accumulate, lse_strides=(0, rows),
                     workspace=self.bwd_ws[r][pc.q_rows], stream=self.streams.s[r], stage=stage)
            return attn.last_launch_count()

        for r in range(cp):  # D of every query-row set the rank's steps use, once
            seen = set()
            for pc in self.pieces[r]:
                if pc.q_rows not in seen:
                    seen.add(pc.q_rows)
                    n += call(r, pc, "preprocess", False)
        for s in range(cp):
            for r in range(cp):
                st = self.streams.s[r]
                if s > 0:
                    st.wait_event(done[s - 1][(r - 1) % cp])
                pc = self.pieces[r][s]
                for stage in self.order[r][s]:
                    n += call(r, pc, stage, s > 0)
                    if stage == "dkdv":  # the next step's writer of this shard waits here
                        done[s][r] = torch.cuda.Event()
                        done[s][r].record(st)
        self.streams.join()
        self.launches += n
        return self.dq, self.dk, self.dv


def allgather_pieces(cp: int, chunk: int, window_left: int = -1):
    """The per-rank calls of the all-gather CP variant: (rank, local query
    rows (first, count), global key range (first, end)).

    After the all-gather every rank holds all of K/V; for its query chunk c
    (global rows [c*chunk, (c+1)*chunk)) it keeps only the keys the chunk can
    see, [max(0, c*chunk - L), (c+1)*chunk) with L = window_left (unbounded if
    < 0), and runs one call with BOTTOM-RIGHT causal alignment, which places the
    diagonal at the end of that trimmed range (TransformerEngine PR #3527 review
    notes on all_gather: KV gathered and trimmed, a per-step window causal
    relative to the trimmed range, no LSE correction).  The window's left bound
    counts from the diagonal, so it is the same in the trimmed frame."""
    out = []
    for r in range(cp):
        pcs = []
        for local, c in enumerate((r, 2 * cp - 1 - r)):
            k_end = (c + 1) * chunk
            k_first = 0 if window_left < 0 else max(0, c * chunk - window_left)
            pcs.append((r, (local * chunk, chunk), (k_first, k_end)))
        out.append(pcs)
    return out


class CPAllGather:
    """One-GPU emulation of the all-gather CP variant with the dual-chunk-swap
    layout: rank r holds query chunks r and 2cp-1-r, gathers the whole K/V
    (here: the full tensors are already on this GPU) and calls attn_fwd /
    attn_bwd once per local chunk on the trimmed keys.  dQ of a chunk is
    complete after its call; the dK/dV of the trimmed range are partial sums
    that a real system reduce-scatters to the owners; here every call adds
    them (FP32, ``accumulate``) into full-sequence dK/dV buffers.

    q/k/v/dout: dense [1, S, H, d] device tensors.  ``window`` = (left, right)
    with right 0 or -1 (causal); left -1 = unbounded."""

    def __init__(self, q, k, v, dout, cp=8, scale=None, window=(-1, 0)):
        assert q.shape[0] == 1, "the emulation runs batch 1"
        self.cp = cp
        self.scale = scale
        self.window = (window[0], 0)
        self.chunk = q.shape[1] // (2 * cp)
        self.k_full, self.v_full = k, v
        self.q, self.do = shard(q, cp), shard(dout, cp)
        self.pieces = allgather_pieces(cp, self.chunk, window[0])
        dev = q.device
        hq, dv = q.shape[2], v.shape[3]
        rows = 2 * self.chunk
        self.o = [torch.empty((1, rows, hq, dv), dtype=q.dtype, device=dev) for _ in range(cp)]
        self.lse = [torch.empty((1, hq, rows), dtype=torch.float32, device=dev) for _ in range(cp)]
        self.dq = [torch.empty((1, rows, *q.shape[2:]), dtype=torch.float32, device=dev)
                   for _ in range(cp)]
        self.dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
        self.dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
        self.fwd_ws = [torch.empty(256, dtype=torch.uint8, device=dev) for _ in range(cp)]
        kw = dict(causal=True, bottom_right=True, window=self.window)
        qc = self.q[0][:, :self.chunk]
        # one workspace per call, sized for its own key range: the calls'
        # preprocess and dq stages overlap
        self.bwd_ws = [[torch.empty(max(attn.workspace_size("bwd", qc, k[:, k0:k1], v[:, k0:k1],
                                                            **kw), 256),
                                    dtype=torch.uint8, device=dev)
                        for _, _, (k0, k1) in pcs] for pcs in self.pieces]
        self.order = [[stage_order(qc, k[:, k0:k1], v[:, k0:k1], **kw) for _, _, (k0, k1) in pcs]
                      for pcs in self.pieces]
        self.streams = _Streams(cp, dev)
        self.launches = 0

    def forward(self):
        """One call per local query chunk; rank r runs on stream r, so the
        ranks' calls overlap (each writes only its own O and LSE rows)."""
        n = 0
        self.streams.fork()
        for r, pcs in enumerate(self.pieces):
            for _, (q0, nq), (k0, k1) in pcs:
                attn.fwd(self.q[r][:, q0:q0 + nq], self.k_full[:, k0:k1], self.v_full[:, k0:k1],
                         causal=True, bottom_right=True, window=self.window, scale=self.scale,
                         out=self.o[r][:, q0:q0 + nq], lse=self.lse[r][:, :, q0:q0 + nq],
                         lse_strides=(0, 2 * self.chunk), workspace=self.fwd_ws[r],
                         stream=self.streams.s[r])
                n += attn.last_launch_count()
        self.streams.join()
        self.launches = n
        return self.o, self.lse

    def backward(self):
        """dQ per chunk; dK/dV summed over every chunk's trimmed range.  The
        library's accumulate flag covers all three gradients, so the FP32
        buffers start from zero.  Rank r runs on stream r: the preprocess and
        dq stages of all calls overlap; every dkdv stage adds into the shared
        dK/dV, so those run one after another (each waits for the previous
        one through an event)."""
        for t in (*self.dq, self.dk, self.dv):
            t.zero_()
        n = 0
        rows = 2 * self.chunk
        self.streams.fork()
        prev = None
        for r, pcs in enumerate(self.pieces):
            st = self.streams.s[r]

            def call(i, stage):
                _, (q0, nq), (k0, k1) = pcs[i]
                attn.bwd(self.q[r][:, q0:q0 + nq], self.k_full[:, k0:k1], self.v_full[:, k0:k1],
                         self.o[r][:, q0:q0 + nq], self.do[r][:, q0:q0 + nq],
                         self.lse[r][:, :, q0:], causal=True, bottom_right=True,
                         window=self.window, scale=self.scale, dq=self.dq[r][:, q0:q0 + nq],
                         dk=self.dk[:, k0:k1], dv=self.dv[:, k0:k1], grad_dtype=torch.float32,
                         accumulate=True, lse_strides=(0, rows), workspace=self.bwd_ws[r][i],
                         stream=st, stage=stage)
                return attn.last_launch_count()

            def dkdv(i):  # shared dK/dV: one call after another
                nonlocal prev
                if prev is not None:
                    st.wait_event(prev)
                launched = call(i, "dkdv")
                prev = torch.cuda.Event()
                prev.record(st)
                return launched

            late = []
            for i in range(len(pcs)):  # independent: every call has its own rows
                n += call(i, "preprocess")
                if self.order[r][i][0] == "dkdv":  # dS path: its dq stage reads the blocks
                    n += dkdv(i)
                    n += call(i, "dq")
                else:
                    n += call(i, "dq")
                    late.append(i)
            for i in late:
                n += dkdv(i)
        self.streams.join()
        self.launches += n
        return self.dq, self.dk, self.dv


class CPA2A:
    """One-GPU emulation of the all-to-all (head-parallel) CP variant
    (TransformerEngine PR #3527 review notes on a2a: after the all-to-all each
    rank holds the full sequence for a subset of heads, so there is no ring
    and no LSE correction, and a window applies unchanged).

    The ranks' inputs are the dual-chunk-swap sequence shards, stacked
    [cp, 2*chunk, H, d].  ``attn_cp_relayout`` moves them to head shards
    [cp, S, H/cp, d] (the all-to-all of cp ranks held on one GPU), every rank
    runs attn_fwd / attn_bwd over the whole sequence for its heads, and O, LSE
    and the gradients move back to the sequence shards.  Query and key/value
    head counts must both divide by cp."""

    def __init__(self, q, k, v, dout, cp=8, scale=None, window=(-1, 0)):
        assert q.shape[0] == 1, "the emulation runs batch 1"
        s, hq, dqk = q.shape[1:]
        hkv, dv = k.shape[2], v.shape[3]
        assert hq % cp == 0 and hkv % cp == 0, "head counts must divide by cp"
        self.cp, self.scale, self.window = cp, scale, (window[0], 0)
        self.chunk = s // (2 * cp)
        stack = lambda x: torch.stack([t[0] for t in shard(x, cp)])  # noqa: E731
        self.q_seq, self.k_seq, self.v_seq, self.do_seq = (stack(t) for t in (q, k, v, dout))
        dev, dt = q.device, q.dtype
        e = lambda *shape, dtype=dt: torch.empty(shape, dtype=dtype, device=dev)  # noqa: E731
        self.q_h, self.k_h, self.v_h = e(cp, s, hq // cp, dqk), e(cp, s, hkv // cp, dqk), \
            e(cp, s, hkv // cp, dv)
        self.do_h, self.o_h = e(cp, s, hq // cp, dv), e(cp, s, hq // cp, dv)
        self.lse_h = e(cp, hq // cp, s, dtype=torch.float32)
        self.dq_h, self.dk_h, self.dv_h = (torch.empty_like(t) for t in (self.q_h, self.k_h, self.v_h))
        self.o_seq = e(cp, 2 * self.chunk, hq, dv)
        self.lse_seq = e(cp, hq, 2 * self.chunk, dtype=torch.float32)
        self.dq_seq, self.dk_seq, self.dv_seq = (torch.empty_like(t) for t in
                                                 (self.q_seq, self.k_seq, self.v_seq))
        self.fwd_ws = torch.empty(256, dtype=torch.uint8, device=dev)
        need = attn.workspace_size("bwd", self.q_h[:1], self.k_h[:1], self.v_h[:1],
                                   causal=True, window=self.window)
        self.bwd_ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        self.launches = 0

    def _kw(self):
        return dict(causal=True, window=self.window, scale=self.scale)

    def forward(self):
        n = 0
        for src, dst in ((self.q_seq, self.q_h), (self.k_seq, self.k_h), (self.v_seq, self.v_h)):
            attn.cp_relayout(src, dst, to_heads=True, cp=self.cp)
            n += 1
        for r in range(self.cp):
            sl = slice(r, r + 1)
            attn.fwd(self.q_h[sl], self.k_h[sl], self.v_h[sl], out=self.o_h[sl],
                     lse=self.lse_h[sl], workspace=self.fwd_ws, **self._kw())
            n += attn.last_launch_count()
        attn.cp_relayout(self.o_h, self.o_seq, to_heads=False, cp=self.cp)
        attn.cp_relayout(self.lse_h, self.lse_seq, to_heads=False, cp=self.cp)
        self.launches = n + 2
        return self.o_seq, self.lse_seq

    def backward(self):
        attn.cp_relayout(self.do_seq, self.do_h, to_heads=True, cp=self.cp)
        n = 1
        for r in range(self.cp):
            sl = slice(r, r + 1)
            attn.bwd(self.q_h[sl], self.k_h[sl], self.v_h[sl], self.o_h[sl], self.do_h[sl],
                     self.lse_h[sl], dq=self.dq_h[sl], dk=self.dk_h[sl], dv=self.dv_h[sl],
                     workspace=self.bwd_ws, **self._kw())
            n += attn.last_launch_count()
        for src, dst in ((self.dq_h, self.dq_seq), (self.dk_h, self.dk_seq), (self.dv_h, self.dv_seq)):
            attn.cp_relayout(src, dst, to_heads=False, cp=self.cp)
            n += 1
        self.launches += n
        return self.dq_seq, self.dk_seq, self.dv_seq
