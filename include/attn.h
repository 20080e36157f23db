/*
 * attn.h -- C ABI of libattn.so: fused causal scaled-dot-product attention
 * (forward, backward, LSE merge) for NVIDIA GB300 (sm_103a).
 *
 * Sources for the operations (web pages on Blackwell attention backends):
 *  - TransformerEngine PR #3527, "cuDNN FROST attention backend for head_dim in
 *    (256, 512], with context parallelism": forward with a natural-log FP32
 *    log-sum-exp; graphs built from each tensor's actual strides; output
 *    buffers owned by the caller; unsupported configurations refused rather
 *    than approximated; k/v stride agreement and GQA divisibility checks;
 *    sliding window (left, right) with -1 unbounded and a causal mask pinning
 *    the right bound to the diagonal; top-left / bottom-right causal alignment;
 *    the stream bound per call; a context-parallel ring merging partial
 *    results through LSE differences.
 *  - TransformerEngine PR #3699, "cuDNN FROST D128/D256 backward dispatch":
 *    the backward helper chain (the D = rowsum(dO * O) preprocess, gradient
 *    reductions over GQA groups), per-execution device checks of cu_seqlens,
 *    pointers / stream / workspace bound per call, exactly zero dQ on rows
 *    that see no key.
 *  - TransformerEngine PR #3149, "FA4 for context parallelism": packed THD
 *    tensors addressed through cu_seqlens.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no memory and keeps no state between calls (except a
 *    thread-local error string and a cached driver entry point).
 *  - Work is enqueued on `stream`; calls return once it is enqueued.
 *  - A problem the host can see (bad shape, stride, alignment, dtype, head
 *    dim, workspace) is returned at once and nothing is launched.
 *  - A problem only the device can see (inconsistent cu_seqlens, a wait that
 *    exceeded its time limit) is written to the status word at the start of
 *    the workspace; the kernels then stop early and leave the outputs
 *    undefined.  attn_query_status() reads it.  No kernel ever traps.
 *  - Element strides are given as {batch, token, head}; the head-dim axis is
 *    contiguous.  Q/K/V/O/dO/dQ/dK/dV may each have their own strides.
 *  - Dense layout (cu_seqlens NULL): tensors are [batch][seqlen][heads][d].
 *    Varlen THD layout (cu_seqlens set): tensors are [total][heads][d] and
 *    sequence b owns rows [cu_seqlens[b], cu_seqlens[b+1]); the batch stride
 *    is ignored.
 *  - LSE is FP32 natural log.  Default layout [batch][heads_q][seqlen_q]
 *    (dense) or [heads_q][total_q] (THD); stride_lse overrides it.
 *  - A query row that sees no key gets O = 0, LSE = -inf and dQ = 0.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* null pointer, negative size, inconsistent shape */
  ATTN_ERR_UNSUPPORTED = 2,  /* valid request this library refuses (head dim, dtype mix) */
  ATTN_ERR_ALIGNMENT = 3,    /* pointer or stride not 16-byte aligned as required */
  ATTN_ERR_WORKSPACE = 4,    /* workspace missing or smaller than *_workspace_size() */
  ATTN_ERR_BAD_METADATA = 5, /* device check: cu_seqlens inconsistent (status word) */
  ATTN_ERR_TIMEOUT = 6,      /* device wait exceeded its time limit (status word) */
  ATTN_ERR_CUDA = 7          /* a CUDA runtime call failed; see attn_last_error() */
} attn_status_t;

typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1, ATTN_FP32 = 2 } attn_dtype_t;

typedef struct {
  attn_dtype_t dtype;      /* Q, K, V, dO: ATTN_BF16 or ATTN_FP16 */
  attn_dtype_t o_dtype;    /* O: == dtype, or ATTN_FP32 (partials for attn_lse_merge) */
  attn_dtype_t grad_dtype; /* dQ, dK, dV: == dtype, or ATTN_FP32 */
  int batch;               /* dense: batch size; THD: number of sequences */
  int seqlen_q, seqlen_k;  /* dense: sequence lengths; THD: maximum lengths */
  const int32_t* cu_seqlens_q; /* device [batch+1] prefix sums, or NULL for dense */
  const int32_t* cu_seqlens_k; /* device [batch+1]; must be set iff cu_seqlens_q is */
  int total_q, total_k;    /* THD: rows of the packed tensors (== cu_seqlens[batch]) */
  int heads_q, heads_kv;   /* heads_q % heads_kv == 0; query head h uses kv head h/(hq/hkv) */
  int d_qk, d_v;           /* (64,64) (128,128) (192,128) (256,256) (512,512) */
  int64_t stride_q[3], stride_k[3], stride_v[3], stride_o[3]; /* {batch, token, head} */
  int64_t stride_do[3], stride_dq[3], stride_dk[3], stride_dv[3];
  int64_t stride_lse[2];   /* {batch, head} in elements; {0, 0} = default layout */
  int causal;              /* 1: key j visible only if j <= i + off */
  int bottom_right;        /* off = seqlen_k - seqlen_q (per sequence) if 1, else 0 */
  int window_left;         /* visible only if j >= i + off - window_left; -1 unbounded */
  int window_right;        /* visible only if j <= i + off + window_right; -1 unbounded */
  float softmax_scale;     /* > 0, typically 1/sqrt(d_qk) */
  int accumulate;          /* attn_bwd with grad_dtype FP32 only: 1 adds the gradients
                              into dq/dk/dv instead of overwriting them (used to sum
                              the partial gradients of a context-parallel ring) */
  const int32_t* seqused_q; /* THD only, device [batch] or NULL: padded layout (PR #3149:
                               physical padded offsets plus visible lengths).  Sequence b
                               then uses rows [cu_seqlens_q[b], cu_seqlens_q[b] +
                               seqused_q[b]); the rows up to cu_seqlens_q[b+1] are a gap
                               that no kernel reads or writes. */
  const int32_t* seqused_k; /* the same for keys/values; set both or neither */
  int bwd_ds;              /* backward at head dims (128,128) and (192,128): 0 = auto
                              (keep dS in the workspace when its blocks take at most
                              64 GiB), 1 = keep dS, -1 = never (recompute the scores
                              for dQ: the smallest workspace).  See attn_bwd_path. */
} attn_params_t;

/* Bytes of workspace attn_fwd / attn_bwd need for `p` (always >= 256: the
 * status word lives at offset 0).  The workspace must be 256-byte aligned.
 * On the ATTN_BWD_PDS path the backward also keeps P and dS of every visible
 * 128-query x 128-key tile (64 KiB each, all query heads) in the workspace,
 * on the ATTN_BWD_DS path dS alone (32 KiB each): the count is exact for
 * dense inputs, and for THD it is a bound that takes every document's keys
 * as max_seqlen_k long (P and dS: about 8.7 GB for batch 1, 16 query heads,
 * 16384 causal tokens; dS: about 34.5 GB for batch 1, 32 query heads, 32768
 * causal tokens). */
size_t attn_fwd_workspace_size(const attn_params_t* p);
size_t attn_bwd_workspace_size(const attn_params_t* p);

/* The backward that attn_bwd runs for `p` (a pure function of `p`):
 *   ATTN_BWD_RECOMPUTE  a query-stationary dQ kernel and a key-stationary
 *                       dK/dV kernel that both compute S and dP;
 *   ATTN_BWD_DS         head dims (128,128) and (192,128) as bwd_ds allows:
 *                       the dK/dV kernel also writes dS (16-bit)
 *                       into the workspace and dQ = scale dS K is a GEMM over
 *                       it, so S and dP are computed once per query-key pair;
 *   ATTN_BWD_PDS        head dim 512, and 256 while its blocks take at most
 *                       16 GiB: P and dS are written to the workspace and the
 *                       five contractions run once each.
 * All three give results within the same bound of the exact gradients, each
 * bitwise reproducible; they differ in rounding order.  Returns -1 for
 * invalid params. */
typedef enum {
  ATTN_BWD_RECOMPUTE = 0,
  ATTN_BWD_DS = 1,
  ATTN_BWD_PDS = 2
} attn_bwd_path_t;
int attn_bwd_path(const attn_params_t* p);

/*
 * Forward (PR #3527): O = softmax(scale * Q K^T + mask) V per (sequence, query
 * head) with an online softmax over 128-key tiles, and LSE = ln sum_j exp(s_ij)
 * over visible keys.  q, k, v: dtype; o: o_dtype; lse: FP32.  The result is
 * bitwise reproducible (no atomics, fixed reduction order).
 * Alignment: every base pointer 16-byte aligned; every token/head/batch stride
 * a multiple of 8 elements (16-bit tensors) or 4 (FP32 O).
 */
attn_status_t attn_fwd(const attn_params_t* p, const void* q, const void* k, const void* v,
                       void* o, float* lse, void* workspace, size_t workspace_bytes,
                       attn_stream_t stream);

/*
 * Backward (PR #3510 head-parallel backward, PR #3699 helper chain): from Q,
 * K, V, O, dO and the forward's LSE computes D = rowsum(dO * O) (FP32, kept in
 * the workspace beside each row's LSE in base 2, the pair the later kernels
 * read), then per visible tile P = exp(scale QK^T - LSE),
 * dP = dO V^T, dS = P (dP - D), dV = P^T dO, dK = scale dS^T Q,
 * dQ = scale dS K; dK/dV are summed over the query heads of a GQA group
 * inside the kernel.  dq/dk/dv are fully overwritten (grad_dtype).  The
 * reduction order is fixed, so the backward is bitwise reproducible.
 * attn_bwd_path tells which kernels run.  On the ATTN_BWD_PDS path (head dim
 * 512, PR #3527: the d512 backward; head dim 256 up to 16 GiB of blocks) P and
 * dS are written once to the workspace (16-bit, as the fused kernels round
 * them too) and the five contractions run in three kernels; on the
 * ATTN_BWD_DS path the dK/dV kernel writes dS and a GEMM forms dQ from it.  A
 * workspace whose block table does not fit sets ATTN_ERR_WORKSPACE in the
 * status word.
 */
attn_status_t attn_bwd(const attn_params_t* p, const void* q, const void* k, const void* v,
                       const void* o, const void* dout, const float* lse, void* dq, void* dk,
                       void* dv, void* workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * The three stages of attn_bwd, callable one by one with the same arguments
 * (attn_bwd == preprocess, then dq, then dkdv, on one stream; on the
 * ATTN_BWD_DS path preprocess, then dkdv, then dq):
 *   attn_bwd_preprocess: D = rowsum(dO * O) and LSE * log2 e per query row
 *                        into the workspace; resets the status word (PR #3699
 *                        "backward helper chain");
 *   attn_bwd_dq:         dQ (reads D and LSE from the workspace);
 *   attn_bwd_dkdv:       dK and dV, reduced over each GQA group (reads D and
 *                        LSE from the workspace).
 * The dq and dkdv stages require a preprocess earlier on the stream, on the
 * same workspace, for a problem with the same query rows, query heads, dtype,
 * batch/cu_seqlens_q layout and LSE: D and LSE depend only on each query row,
 * so one preprocess serves several calls that differ only in their keys, mask
 * or window (a context-parallel ring does this; its LSE is the merged one).
 * The dq and dkdv stages ignore their `lse` argument.  Where the backward
 * materialises P and dS (head dim 512; head dim 256 up to 16 GiB of blocks)
 * the dq stage also writes them, with their block plan, into the workspace
 * and the dkdv stage reads them: it then requires the dq stage of the same
 * problem earlier on the stream as well.  On the ATTN_BWD_DS path it is the
 * other way round: the dkdv stage writes dS and its block plan, and the dq
 * stage requires the dkdv stage of the same problem earlier on the stream.
 * Arguments a stage does not use may be NULL.
 */
attn_status_t attn_bwd_preprocess(const attn_params_t* p, const void* q, const void* k,
                                  const void* v, const void* o, const void* dout,
                                  const float* lse, void* dq, void* dk, void* dv,
                                  void* workspace, size_t workspace_bytes, attn_stream_t stream);
attn_status_t attn_bwd_dq(const attn_params_t* p, const void* q, const void* k, const void* v,
                          const void* o, const void* dout, const float* lse, void* dq, void* dk,
                          void* dv, void* workspace, size_t workspace_bytes,
                          attn_stream_t stream);
attn_status_t attn_bwd_dkdv(const attn_params_t* p, const void* q, const void* k, const void* v,
                            const void* o, const void* dout, const float* lse, void* dq,
                            void* dk, void* dv, void* workspace, size_t workspace_bytes,
                            attn_stream_t stream);

/*
 * attn_bwd for callers that cannot allocate device memory (this entry point
 * has no counterpart on the attention pages; it is a deployment aid).
 *
 * Some callers are not allowed to call cudaMalloc while they run: cudaMalloc
 * may synchronise the whole device and takes an unbounded time, so serving
 * loops with latency budgets, plugin hosts that plan every byte of device
 * memory up front, and code running inside another runtime's callbacks
 * forbid it -- and such callers often have no allocator of their own from
 * which to hand attn_bwd a workspace.  attn_bwd_noalloc takes the same
 * arguments as attn_bwd minus the workspace and uses instead a scratch area
 * that the library reserves statically: 8 MiB of device memory per GPU that
 * loads the library, held until the process exits.  That covers problems
 * whose attn_bwd_workspace_size() is at most 8 MiB (about one million
 * query rows x query heads); larger ones return ATTN_ERR_WORKSPACE and
 * nothing is launched.  With bwd_ds = 0 it takes the ATTN_BWD_RECOMPUTE
 * path (the ATTN_BWD_DS path's blocks rarely fit).  It calls no allocating
 * routine.
 *
 * The first call on each device looks up the scratch area's device address
 * (with that device current) and caches it; make that first call before any
 * stream capture.  Every call on a device shares the one scratch area and
 * the status word in it, so calls whose work overlaps on the GPU (different
 * streams, or host threads) race with each other: serialise them.  The
 * status word is cleared at the start of each call; as the caller holds no
 * pointer to it, device-detected problems (inconsistent cu_seqlens, a wait
 * past its limit) are not reported to it -- use attn_bwd where that matters.
 * Results are identical to attn_bwd's.
 */
attn_status_t attn_bwd_noalloc(const attn_params_t* p, const void* q, const void* k,
                               const void* v, const void* o, const void* dout, const float* lse,
                               void* dq, void* dk, void* dv, attn_stream_t stream);

/*
 * One forward + backward step from HOST buffers (a deployment aid with no
 * counterpart on the attention pages: the end-to-end path of a caller whose
 * tensors live in host memory).
 *
 * q, k, v, dout (inputs) and o, lse, dq, dk, dv (outputs) are HOST pointers,
 * laid out with the strides, dtypes and LSE layout that `p` gives, exactly as
 * attn_fwd / attn_bwd would take them on the device; for THD inputs
 * p->cu_seqlens_q/k (and seqused_q/k) are HOST arrays here too.  On `stream`,
 * in order: every input is copied into `arena` (one cudaMemcpyAsync per
 * tensor, the span from its base to its last element), attn_fwd and attn_bwd
 * run there, and O, LSE, dQ, dK, dV are copied back.  With p->accumulate the
 * host dq/dk/dv are uploaded first and the gradients are added to them.
 *
 * arena: caller-owned DEVICE memory, 256-byte aligned, at least
 * attn_host_arena_size(p) bytes: the forward's workspace (its first 256 bytes),
 * then the backward's, then the device copies of all nine tensors.  So
 * attn_query_status(arena) reports device-detected problems of the forward and
 * attn_query_status((char*)arena + 256) those of the backward.  The call
 * returns once the work is enqueued.  Host buffers, and for THD the host
 * cu_seqlens / seqused arrays, should be pinned (cudaHostAlloc /
 * cudaHostRegister) for the copies to be asynchronous: a copy from pageable
 * memory holds the calling thread until the stream has drained, which
 * serialises a pipeline of steps on several streams.  The inputs must not change and the
 * outputs must not be read until the stream has passed the call.  Two calls on
 * two streams with two arenas overlap one step's copies with the other's
 * kernels.  A device pointer among the buffers is refused with
 * ATTN_ERR_INVALID_ARG.  Results are identical to attn_fwd + attn_bwd on the
 * device copies.  attn_host_arena_size returns 0 for parameters that
 * attn_fwd / attn_bwd would refuse.
 */
size_t attn_host_arena_size(const attn_params_t* p);
attn_status_t attn_fwd_bwd_host(const attn_params_t* p, const void* q, const void* k,
                                const void* v, const void* dout, void* o, float* lse, void* dq,
                                void* dk, void* dv, void* arena, size_t arena_bytes,
                                attn_stream_t stream);

/*
 * attn_fwd_bwd_host in stages, for callers that pipeline consecutive steps:
 * `stages` is a mask of ATTN_HOST_UPLOAD (the host inputs, metadata and, with
 * accumulate, the host gradients into the arena), ATTN_HOST_COMPUTE (attn_fwd
 * and attn_bwd on the arena's copies) and ATTN_HOST_DOWNLOAD (O, LSE, dQ, dK,
 * dV back to host memory); ATTN_HOST_ALL is attn_fwd_bwd_host.  Each stage
 * enqueues on `stream`, so a caller can upload step s+1 on one stream while
 * step s computes on another and step s-1 downloads on a third, ordering
 * them with its own events; one arena must not be uploaded into while its
 * previous step still computes or downloads.  The same parameters (shape,
 * strides, flags) must be passed to every stage of one step; the buffers a
 * stage does not touch may be NULL.
 */
enum { ATTN_HOST_UPLOAD = 1, ATTN_HOST_COMPUTE = 2, ATTN_HOST_DOWNLOAD = 4, ATTN_HOST_ALL = 7 };
attn_status_t attn_fwd_bwd_host_stages(const attn_params_t* p, const void* q, const void* k,
                                       const void* v, const void* dout, void* o, float* lse,
                                       void* dq, void* dk, void* dv, void* arena,
                                       size_t arena_bytes, unsigned stages, attn_stream_t stream);

/*
 * LSE-weighted merge of partial attention results over disjoint key sets
 * (PR #3527: the context-parallel ring correction exponentiates LSE
 * differences):  LSE = ln sum_p exp(LSE_p),  O = sum_p exp(LSE_p - LSE) O_p,
 * with the maximum subtracted first; a part whose LSE is -inf has weight 0 and
 * a row with no finite part gets O = 0, LSE = -inf.
 *   o_parts[p]:   device FP32 [part_rows[p]][heads][d_v], contiguous
 *   lse_parts[p]: device FP32 [heads][part_rows[p]], contiguous
 *   part part p covers output rows [part_row0[p], part_row0[p] + part_rows[p])
 *   o_out: [rows][heads][d_v] of o_dtype (BF16, FP16 or FP32), contiguous
 *   lse_out: [heads][rows] FP32.
 * The pointer and range arrays are HOST arrays of n_parts entries
 * (1 <= n_parts <= 64); d_v % 4 == 0.
 */
attn_status_t attn_lse_merge(int n_parts, const float* const* o_parts,
                             const float* const* lse_parts, const int64_t* part_row0,
                             const int64_t* part_rows, int64_t rows, int heads, int d_v,
                             void* o_out, attn_dtype_t o_dtype, float* lse_out,
                             attn_stream_t stream);

/*
 * Local data movement of the all-to-all context-parallel path (PR #3527: after
 * the all-to-all each rank holds the full sequence for a subset of heads), for
 * the cp ranks of a dual-chunk-swap layout held in device memory:
 *   sequence side: rank r holds global chunks r and 2cp-1-r (chunk =
 *     seqlen / (2 cp)) as its local tokens [0, chunk) and [chunk, 2 chunk),
 *     all `heads` heads;
 *   head side:     rank r holds heads [r*heads/cp, (r+1)*heads/cp) of every
 *     token, in sequence order.
 * to_heads = 1 copies sequence side -> head side (src is the sequence side),
 * 0 the reverse.  Each side is described by element strides {rank, token,
 * head}; the d elements of one (token, head) are contiguous and elem_bytes
 * wide (2 for BF16/FP16 tensors, 4 for FP32 such as LSE, which is d = 1 with
 * head-major strides).  A bit-preserving copy; src and dst must not overlap.
 * Requirements: cp >= 1, seqlen a positive multiple of 2 cp, heads % cp == 0,
 * elem_bytes 2 or 4, pointers aligned to elem_bytes.
 */
attn_status_t attn_cp_relayout(int to_heads, int cp, int64_t seqlen, int heads, int d,
                               int elem_bytes, const void* src, const int64_t src_strides[3],
                               void* dst, const int64_t dst_strides[3], attn_stream_t stream);

/* Synchronises `stream` and returns the status word in `workspace`
 * (ATTN_OK, ATTN_ERR_BAD_METADATA, ATTN_ERR_TIMEOUT or, for the head-dim-512
 * backward, ATTN_ERR_WORKSPACE). */
attn_status_t attn_query_status(const void* workspace, attn_stream_t stream);

/* Message of the last error returned on this thread ("" if none). */
const char* attn_last_error(void);

/* Number of kernels the last successful attn_fwd / attn_bwd / attn_lse_merge
 * call on this thread enqueued. */
int attn_last_launch_count(void);

/*
 * TEST ONLY: fault injection for the bounded-wait unwind path.  Every wait of
 * the attention kernels on an mbarrier phase has a wall-clock limit (2 s by
 * default); when one runs out the CTA raises ATTN_ERR_TIMEOUT in the status
 * word, lets its in-flight copies land, drains its MMAs, frees its TMEM and
 * returns -- no kernel traps or hangs (PR #3699's bot review found a
 * "missing wait" on a reused barrier phase; this is the guard against that
 * class of bug).  This call arms the NEXT attn_fwd / attn_bwd* call on the
 * calling thread, then clears itself: in every kernel selected by
 * `kernel_mask` (ATTN_DEBUG_* bits), one CTA leaves out load number
 * `drop_load` (-1: none) and, if `wait_limit_ns` is non-zero, waits at most
 * that long instead of 2 s.  In the dQ kernel, which runs work items from a
 * queue, it is the CTA that runs the first work item (the heaviest query
 * tile of the first head), the load is the K tile number `drop_load` of that
 * item, and every CTA of the launch uses the shorter limit (a healthy wait
 * lasts microseconds); in the other
 * kernels it is the first CTA (block 0,0,0), the load number counts its
 * stage/ring loads, and only that CTA uses the shorter limit.  No other call
 * is affected.  A dropped load makes a wait run out, so the call reports
 * ATTN_ERR_TIMEOUT through attn_query_status and leaves its outputs
 * undefined; the device stays usable and later calls are unaffected.
 */
enum {
  ATTN_DEBUG_FWD = 1,    /* forward kernel */
  ATTN_DEBUG_DQ = 2,     /* dQ kernel, or the dQ GEMM of the materialising backward */
  ATTN_DEBUG_DKDV = 4,   /* dK/dV kernel, or the dK/dV GEMMs of the materialising backward */
  ATTN_DEBUG_SCORES = 8  /* P/dS scores kernel of the materialising backward */
};
void attn_debug_inject(unsigned kernel_mask, int drop_load, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif
#endif /* ATTN_H_ */
