// api.cu -- the C ABI declared in include/attn.h: host-side validation,
// tensor-map construction and kernel dispatch.  No call allocates memory; the
// only state is a thread-local error string, cached device attributes and
// (for attn_bwd_noalloc) a static scratch area and its per-device address.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/attn.h"
#include "bwd.h"
#include "kcommon.cuh"

#include "small_params.h"

namespace attn {
cudaError_t launch_fwd(const FwdParams& p, int dqk, int dv, bool bf16, bool o_f32,
                       cudaStream_t st);
}  // namespace attn

namespace {

thread_local char g_err[512] = "";
thread_local int g_launches = 0;

// Test-only fault injection armed by attn_debug_inject for the next call on
// this thread (then cleared).
struct Inject {
  unsigned mask;
  int drop_load;
  unsigned long long wait_ns;
};
thread_local Inject g_inject = {0u, -1, 0ull};

Inject take_inject() {
  const Inject r = g_inject;
  g_inject = Inject{0u, -1, 0ull};
  return r;
}

attn::DebugInject inject_for(const Inject& in, unsigned kernel_bit) {
  attn::DebugInject d;
  d.wait_ns = (in.mask & kernel_bit) ? in.wait_ns : 0ull;
  d.drop_load = (in.mask & kernel_bit) ? in.drop_load : -1;
  return d;
}

attn_status_t fail(attn_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

attn_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

constexpr size_t kStatusBytes = 256;

bool is_16(attn_dtype_t t) { return t == ATTN_BF16 || t == ATTN_FP16; }
size_t esize(attn_dtype_t t) { return t == ATTN_FP32 ? 4 : 2; }

bool supported_dims(int dqk, int dv) {
  return (dqk == 64 && dv == 64) || (dqk == 128 && dv == 128) || (dqk == 192 && dv == 128) ||
         (dqk == 256 && dv == 256) || (dqk == 512 && dv == 512);
}

bool thd(const attn_params_t* p) { return p->cu_seqlens_q != nullptr; }
int64_t rows_q(const attn_params_t* p) {
  return thd(p) ? (int64_t)p->total_q : (int64_t)p->batch * p->seqlen_q;
}
int64_t rows_k(const attn_params_t* p) {
  return thd(p) ? (int64_t)p->total_k : (int64_t)p->batch * p->seqlen_k;
}

struct Span {
  uintptr_t lo, hi;  // [lo, hi) bytes; hi == lo means empty
};

Span span_of(const void* base, const int64_t s[3], const attn_params_t* p, bool is_q, int heads,
             int d, size_t es) {
  Span r{(uintptr_t)base, (uintptr_t)base};
  const int64_t nrow = is_q ? (thd(p) ? p->total_q : p->seqlen_q) : (thd(p) ? p->total_k : p->seqlen_k);
  const int64_t nb = thd(p) ? 1 : p->batch;
  if (nrow <= 0 || nb <= 0 || heads <= 0) return r;
  const int64_t last = (nb - 1) * (thd(p) ? 0 : s[0]) + (nrow - 1) * s[1] + (int64_t)(heads - 1) * s[2] + d;
  r.hi = r.lo + (uintptr_t)(last * (int64_t)es);
  return r;
}

bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

attn_status_t check_tensor(const char* name, const void* ptr, const int64_t s[3],
                           const attn_params_t* p, size_t es, bool nonempty) {
  if (!nonempty) return ATTN_OK;
  if (!ptr) return fail(ATTN_ERR_INVALID_ARG, "%s is NULL", name);
  if ((uintptr_t)ptr % 16) return fail(ATTN_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
  const int64_t align_el = 16 / (int64_t)es;
  for (int i = 0; i < 3; ++i) {
    if (i == 0 && thd(p)) continue;
    if (s[i] < 0) return fail(ATTN_ERR_INVALID_ARG, "%s stride[%d] is negative", name, i);
    if (s[i] % align_el)
      return fail(ATTN_ERR_ALIGNMENT, "%s stride[%d]=%lld is not a multiple of %lld elements",
                  name, i, (long long)s[i], (long long)align_el);
  }
  return ATTN_OK;
}

attn_status_t check_params(const attn_params_t* p) {
  if (!p) return fail(ATTN_ERR_INVALID_ARG, "params is NULL");
  if (!is_16(p->dtype)) return fail(ATTN_ERR_UNSUPPORTED, "dtype must be BF16 or FP16");
  if (p->o_dtype != p->dtype && p->o_dtype != ATTN_FP32)
    return fail(ATTN_ERR_UNSUPPORTED, "o_dtype must equal dtype or be FP32");
  if (p->grad_dtype != p->dtype && p->grad_dtype != ATTN_FP32)
    return fail(ATTN_ERR_UNSUPPORTED, "grad_dtype must equal dtype or be FP32");
  if (p->batch < 0) return fail(ATTN_ERR_INVALID_ARG, "batch < 0");
  if (p->heads_q <= 0 || p->heads_kv <= 0)
    return fail(ATTN_ERR_INVALID_ARG, "heads must be positive");
  if (p->heads_q % p->heads_kv)
    return fail(ATTN_ERR_INVALID_ARG, "heads_q (%d) is not divisible by heads_kv (%d)",
                p->heads_q, p->heads_kv);
  if (p->d_qk % 8 || p->d_v % 8)
    return fail(ATTN_ERR_INVALID_ARG, "head dims must be multiples of 8");
  if (!supported_dims(p->d_qk, p->d_v))
    return fail(ATTN_ERR_UNSUPPORTED,
                "head dims (%d,%d) not supported: use (64,64) (128,128) (192,128) (256,256) "
                "(512,512)",
                p->d_qk, p->d_v);
  if (p->seqlen_q < 0 || p->seqlen_k < 0) return fail(ATTN_ERR_INVALID_ARG, "seqlen < 0");
  if ((p->cu_seqlens_q == nullptr) != (p->cu_seqlens_k == nullptr))
    return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must both be set or NULL");
  if (thd(p)) {
    if (p->total_q < 0 || p->total_k < 0) return fail(ATTN_ERR_INVALID_ARG, "total < 0");
    if ((uintptr_t)p->cu_seqlens_q % 4 || (uintptr_t)p->cu_seqlens_k % 4)
      return fail(ATTN_ERR_ALIGNMENT, "cu_seqlens must be 4-byte aligned");
  }
  if (p->seqused_q || p->seqused_k) {
    if (!thd(p)) return fail(ATTN_ERR_INVALID_ARG, "seqused needs the packed (THD) layout");
    if (!p->seqused_q || !p->seqused_k)
      return fail(ATTN_ERR_INVALID_ARG, "seqused_q and seqused_k must both be set or NULL");
    if ((uintptr_t)p->seqused_q % 4 || (uintptr_t)p->seqused_k % 4)
      return fail(ATTN_ERR_ALIGNMENT, "seqused must be 4-byte aligned");
  }
  if (p->window_left < -1 || p->window_right < -1)
    return fail(ATTN_ERR_INVALID_ARG, "window bounds must be >= -1");
  if (!(p->softmax_scale > 0.0f) || !std::isfinite(p->softmax_scale))
    return fail(ATTN_ERR_INVALID_ARG, "softmax_scale must be positive and finite");
  if (p->stride_lse[0] < 0 || p->stride_lse[1] < 0)
    return fail(ATTN_ERR_INVALID_ARG, "stride_lse must be >= 0");
  if (p->bwd_ds < -1 || p->bwd_ds > 1) return fail(ATTN_ERR_INVALID_ARG, "bwd_ds must be -1, 0 or 1");
  return ATTN_OK;
}

// LSE/D layout {batch stride, head stride}
void lse_strides(const attn_params_t* p, int64_t& sb, int64_t& sh) {
  if (p->stride_lse[0] || p->stride_lse[1]) {
    sb = p->stride_lse[0];
    sh = p->stride_lse[1];
  } else if (thd(p)) {
    sb = 0;
    sh = p->total_q;
  } else {
    sb = (int64_t)p->heads_q * p->seqlen_q;
    sh = p->seqlen_q;
  }
}
void default_d_strides(const attn_params_t* p, int64_t& sb, int64_t& sh) {
  if (thd(p)) {
    sb = 0;
    sh = p->total_q;
  } else {
    sb = (int64_t)p->heads_q * p->seqlen_q;
    sh = p->seqlen_q;
  }
}

attn::Geometry geometry(const attn_params_t* p) {
  attn::Geometry g;
  g.cu_q = p->cu_seqlens_q;
  g.cu_k = p->cu_seqlens_k;
  g.used_q = p->seqused_q;
  g.used_k = p->seqused_k;
  g.seqlen_q = p->seqlen_q;
  g.seqlen_k = p->seqlen_k;
  g.causal = p->causal ? 1 : 0;
  g.bottom_right = p->bottom_right ? 1 : 0;
  g.wl = p->window_left;
  g.wr = p->window_right;
  return g;
}

int map_rows(attn::MapOrder* o, CUtensorMap* m, const void* base, const attn_params_t* p,
             const int64_t s[3], bool is_q, int heads, int d, int box_rows) {
  const bool bf16 = p->dtype == ATTN_BF16;
  if (thd(p)) {
    const int64_t T = is_q ? p->total_q : p->total_k;
    return attn::make_row_map(m, o, base, bf16, d, heads, T > 0 ? T : 1, 1, s[2], s[1],
                              s[1] * (T > 0 ? T : 1), box_rows);
  }
  const int64_t S = is_q ? p->seqlen_q : p->seqlen_k;
  return attn::make_row_map(m, o, base, bf16, d, heads, S > 0 ? S : 1, p->batch, s[2], s[1],
                            s[0], box_rows);
}

attn_status_t launch_check_if_thd(const attn_params_t* p, int* status, cudaStream_t st) {
  if (!thd(p)) return ATTN_OK;
  attn::CheckParams c;
  c.cu_q = p->cu_seqlens_q;
  c.cu_k = p->cu_seqlens_k;
  c.used_q = p->seqused_q;
  c.used_k = p->seqused_k;
  c.batch = p->batch;
  c.max_q = p->seqlen_q;
  c.max_k = p->seqlen_k;
  c.total_q = p->total_q;
  c.total_k = p->total_k;
  c.status = status;
  cudaError_t e = attn::launch_check(c, st);
  if (e != cudaSuccess) return cuda_fail(e, "check kernel launch");
  ++g_launches;
  return ATTN_OK;
}

// Backward workspace: [status][row statistics: rows x heads_q x {LSE * log2 e,
// D} fp32] and, on the PDS and
// DS paths, [per-sequence block prefix][64 KiB P/dS or 32 KiB dS blocks].
struct BwdLayout {
  size_t d_off, plan_off, blk_off, total;
  long long cap;  // blocks
};

long long wide_block_count(const attn_params_t* p);
bool wide(const attn_params_t* p) {
  if (p->d_qk < 256 || p->d_v < 256) return false;
  return attn::wide_backward(p->d_qk, p->d_v, wide_block_count(p) * (long long)attn::kWideBlock);
}
bool ds_path(const attn_params_t* p) {
  if (p->d_qk > 192) return false;
  const long long n = wide_block_count(p);  // the kernels index blocks in 32 bits
  return n <= INT_MAX && attn::ds_backward(p->d_qk, p->d_v, n * (long long)attn::kDsBlock, p->bwd_ds);
}

// Score blocks of the wide backward over all query heads: exact for dense
// inputs; for packed (THD) inputs a bound that takes every document's keys
// as max_seqlen_k long.
long long wide_block_count(const attn_params_t* p) {
  const long long hq = p->heads_q > 0 ? p->heads_q : 0;
  if (p->batch <= 0 || hq == 0) return 0;
  if (thd(p)) {
    const long long nq = (p->total_q > 0 ? p->total_q : 0) / 128 + p->batch;
    const long long nk = (p->seqlen_k > 0 ? (long long)p->seqlen_k + 127 : 0) / 128;
    return hq * nq * nk;
  }
  if (p->seqlen_q <= 0 || p->seqlen_k <= 0) return 0;
  attn::Seq s;
  s.q_start = s.k_start = 0;
  s.lq = p->seqlen_q;
  s.lk = p->seqlen_k;
  s.off = p->bottom_right ? (long long)(s.lk - s.lq) : 0ll;
  s.L = p->window_left < 0 ? attn::kInfBound : (long long)p->window_left;
  s.R = p->causal ? 0ll : (p->window_right < 0 ? attn::kInfBound : (long long)p->window_right);
  long long t = 0;
  int kb0;
  for (int qt = 0; qt < (s.lq + 127) / 128; ++qt) t += attn::wide_blocks_of_qtile(s, qt, kb0);
  return (long long)p->batch * hq * t;
}

BwdLayout bwd_layout(const attn_params_t* p) {
  BwdLayout l;
  memset(&l, 0, sizeof(l));
  const int64_t rq = rows_q(p);
  // per row (token, query head) {LSE * log2 e, D}: two floats
  const size_t d_bytes = (size_t)(rq > 0 ? rq : 0) * (size_t)(p->heads_q > 0 ? p->heads_q : 0) * 8;
  l.d_off = kStatusBytes;
  l.total = l.d_off + ((d_bytes + 255) / 256) * 256;
  const bool w = wide(p);
  if (w || ds_path(p)) {
    l.plan_off = l.total;
    const size_t plan_bytes = (size_t)(p->batch > 0 ? p->batch + 1 : 1) * 8;
    l.blk_off = ((l.plan_off + plan_bytes + 1023) / 1024) * 1024;
    l.cap = wide_block_count(p);
    l.total = l.blk_off + (size_t)l.cap * (w ? attn::kWideBlock : attn::kDsBlock);
  }
  return l;
}

}  // namespace

extern "C" {

size_t attn_fwd_workspace_size(const attn_params_t* p) {
  (void)p;
  return kStatusBytes;
}

size_t attn_bwd_workspace_size(const attn_params_t* p) {
  if (!p) return kStatusBytes;
  return bwd_layout(p).total;
}

int attn_bwd_path(const attn_params_t* p) {
  if (check_params(p)) return -1;
  if (wide(p)) return ATTN_BWD_PDS;
  return ds_path(p) ? ATTN_BWD_DS : ATTN_BWD_RECOMPUTE;
}

attn_status_t attn_fwd(const attn_params_t* p, const void* q, const void* k, const void* v,
                       void* o, float* lse, void* ws, size_t ws_bytes, attn_stream_t stream) {
  g_err[0] = 0;
  g_launches = 0;
  const Inject inj = take_inject();
  attn_status_t s = check_params(p);
  if (s) return s;
  cudaStream_t st = (cudaStream_t)stream;
  const bool has_q = rows_q(p) > 0, has_k = rows_k(p) > 0;
  if ((s = check_tensor("q", q, p->stride_q, p, 2, has_q))) return s;
  if ((s = check_tensor("k", k, p->stride_k, p, 2, has_k))) return s;
  if ((s = check_tensor("v", v, p->stride_v, p, 2, has_k))) return s;
  if ((s = check_tensor("o", o, p->stride_o, p, esize(p->o_dtype), has_q))) return s;
  if (has_q && !lse) return fail(ATTN_ERR_INVALID_ARG, "lse is NULL");
  if (!ws) return fail(ATTN_ERR_WORKSPACE, "workspace is NULL");
  if ((uintptr_t)ws % 256) return fail(ATTN_ERR_ALIGNMENT, "workspace is not 256-byte aligned");
  if (ws_bytes < attn_fwd_workspace_size(p))
    return fail(ATTN_ERR_WORKSPACE, "workspace too small (%zu < %zu)", ws_bytes,
                attn_fwd_workspace_size(p));
  const Span so = span_of(o, p->stride_o, p, true, p->heads_q, p->d_v, esize(p->o_dtype));
  if (overlap(so, span_of(q, p->stride_q, p, true, p->heads_q, p->d_qk, 2)) ||
      overlap(so, span_of(k, p->stride_k, p, false, p->heads_kv, p->d_qk, 2)) ||
      overlap(so, span_of(v, p->stride_v, p, false, p->heads_kv, p->d_v, 2)))
    return fail(ATTN_ERR_INVALID_ARG, "o overlaps an input");
  int* status = (int*)ws;
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), st);
  if (e != cudaSuccess) return cuda_fail(e, "status reset");
  if (!has_q || p->batch == 0) return ATTN_OK;
  if ((s = launch_check_if_thd(p, status, st))) return s;

  attn::FwdParams fp;
  memset(&fp, 0, sizeof(fp));
  const int kb = has_k ? 1 : 0;
  if (map_rows(&fp.oq, &fp.tm_q, q, p, p->stride_q, true, p->heads_q, p->d_qk, 128))
    return fail(ATTN_ERR_INVALID_ARG, "cannot build the tensor map of q");
  if (kb && map_rows(&fp.ok, &fp.tm_k, k, p, p->stride_k, false, p->heads_kv, p->d_qk, 128))
    return fail(ATTN_ERR_INVALID_ARG, "cannot build the tensor map of k");
  if (kb && map_rows(&fp.ov, &fp.tm_v, v, p, p->stride_v, false, p->heads_kv, p->d_v, 128))
    return fail(ATTN_ERR_INVALID_ARG, "cannot build the tensor map of v");
  if (!kb) {  // no keys at all: maps are never used, point them at q
    fp.tm_k = fp.tm_q;
    fp.tm_v = fp.tm_q;
    fp.ok = fp.oq;
    fp.ov = fp.oq;
  }
  fp.geo = geometry(p);
  fp.o = o;
  fp.lse = lse;
  fp.so_b = thd(p) ? 0 : p->stride_o[0];
  fp.so_t = p->stride_o[1];
  fp.so_h = p->stride_o[2];
  lse_strides(p, fp.lse_sb, fp.lse_sh);
  fp.batch = p->batch;
  fp.hq = p->heads_q;
  fp.hkv = p->heads_kv;
  fp.n_qtiles = (p->seqlen_q + 127) / 128;
  fp.n_split = p->d_v > 256 ? p->d_v / 256 : 1;
  fp.scale_log2 = p->softmax_scale * 1.4426950408889634f;
  fp.status = status;
  fp.dbg = inject_for(inj, ATTN_DEBUG_FWD);
  if (fp.n_qtiles == 0) return ATTN_OK;
  if (fp.n_qtiles > 65535 || p->batch > 65535)
    return fail(ATTN_ERR_UNSUPPORTED, "sequence or batch too large for the grid");
  e = attn::launch_fwd(fp, p->d_qk, p->d_v, p->dtype == ATTN_BF16, p->o_dtype == ATTN_FP32, st);
  if (e == cudaErrorNotSupported) return fail(ATTN_ERR_UNSUPPORTED, "no forward kernel");
  if (e != cudaSuccess) return cuda_fail(e, "forward kernel launch");
  ++g_launches;
  return ATTN_OK;
}

}  // extern "C"

namespace {

enum : int { kStagePre = 1, kStageDq = 2, kStageDkv = 4, kStageAll = 7 };

attn_status_t bwd_impl(const attn_params_t* p, const void* q, const void* k, const void* v,
                       const void* o, const void* dout, const float* lse, void* dq, void* dk,
                       void* dv, void* ws, size_t ws_bytes, attn_stream_t stream, int stages) {
  g_err[0] = 0;
  g_launches = 0;
  const Inject inj = take_inject();
  attn_status_t s = check_params(p);
  if (s) return s;
  if (p->o_dtype != p->dtype)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_bwd reads O in the input dtype (o_dtype == dtype)");
  if (p->accumulate && p->grad_dtype != ATTN_FP32)
    return fail(ATTN_ERR_UNSUPPORTED, "accumulate requires grad_dtype FP32");
  cudaStream_t st = (cudaStream_t)stream;
  const bool has_q = rows_q(p) > 0, has_k = rows_k(p) > 0;
  const size_t ge = esize(p->grad_dtype);
  const bool pre = stages & kStagePre, sdq = stages & kStageDq, skv = stages & kStageDkv;
  const bool need_qkv = sdq || skv;
  if (need_qkv) {
    if ((s = check_tensor("q", q, p->stride_q, p, 2, has_q))) return s;
    if ((s = check_tensor("k", k, p->stride_k, p, 2, has_k))) return s;
    if ((s = check_tensor("v", v, p->stride_v, p, 2, has_k))) return s;
  }
  // the preprocess stores each row's LSE beside D; the later stages read them there
  if (pre && has_q && !lse) return fail(ATTN_ERR_INVALID_ARG, "lse is NULL");
  if (pre && (s = check_tensor("o", o, p->stride_o, p, 2, has_q))) return s;
  if ((s = check_tensor("dout", dout, p->stride_do, p, 2, has_q))) return s;
  if (sdq && (s = check_tensor("dq", dq, p->stride_dq, p, ge, has_q))) return s;
  if (skv && (s = check_tensor("dk", dk, p->stride_dk, p, ge, has_k))) return s;
  if (skv && (s = check_tensor("dv", dv, p->stride_dv, p, ge, has_k))) return s;
  if (!ws) return fail(ATTN_ERR_WORKSPACE, "workspace is NULL");
  if ((uintptr_t)ws % 256) return fail(ATTN_ERR_ALIGNMENT, "workspace is not 256-byte aligned");
  if (ws_bytes < attn_bwd_workspace_size(p))
    return fail(ATTN_ERR_WORKSPACE, "workspace too small (%zu < %zu)", ws_bytes,
                attn_bwd_workspace_size(p));
  {
    const Span in[5] = {span_of(q, p->stride_q, p, true, p->heads_q, p->d_qk, 2),
                        span_of(k, p->stride_k, p, false, p->heads_kv, p->d_qk, 2),
                        span_of(v, p->stride_v, p, false, p->heads_kv, p->d_v, 2),
                        span_of(o, p->stride_o, p, true, p->heads_q, p->d_v, 2),
                        span_of(dout, p->stride_do, p, true, p->heads_q, p->d_v, 2)};
    const Span none{0, 0};
    const Span out[3] = {sdq ? span_of(dq, p->stride_dq, p, true, p->heads_q, p->d_qk, ge) : none,
                         skv ? span_of(dk, p->stride_dk, p, false, p->heads_kv, p->d_qk, ge) : none,
                         skv ? span_of(dv, p->stride_dv, p, false, p->heads_kv, p->d_v, ge) : none};
    const Span wsp{(uintptr_t)ws, (uintptr_t)ws + attn_bwd_workspace_size(p)};
    for (int a = 0; a < 3; ++a) {
      for (int b = 0; b < 5; ++b)
        if (overlap(out[a], in[b])) return fail(ATTN_ERR_INVALID_ARG, "a gradient overlaps an input");
      for (int b = a + 1; b < 3; ++b)
        if (overlap(out[a], out[b])) return fail(ATTN_ERR_INVALID_ARG, "gradients overlap");
      if (overlap(out[a], wsp)) return fail(ATTN_ERR_INVALID_ARG, "a gradient overlaps the workspace");
    }
  }
  int* status = (int*)ws;
  const BwdLayout lay = bwd_layout(p);
  float2* dbuf = (float2*)((char*)ws + lay.d_off);
  cudaError_t e;
  if (pre) {
    e = cudaMemsetAsync(status, 0, sizeof(int), st);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
  }
  if (p->batch == 0 || (!has_q && !has_k)) return ATTN_OK;
  if (pre && (s = launch_check_if_thd(p, status, st))) return s;

  attn::BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.geo = geometry(p);
  a.batch = p->batch;
  a.hq = p->heads_q;
  a.hkv = p->heads_kv;
  a.dqk = p->d_qk;
  a.dv = p->d_v;
  a.bf16 = p->dtype == ATTN_BF16;
  a.g_f32 = p->grad_dtype == ATTN_FP32;
  a.accum = p->accumulate ? 1 : 0;
  a.scale = p->softmax_scale;
  a.scale_log2 = p->softmax_scale * 1.4426950408889634f;
  a.status = status;
  a.dbg_dq = inject_for(inj, ATTN_DEBUG_DQ);
  a.dbg_dkdv = inject_for(inj, ATTN_DEBUG_DKDV);
  a.dbg_scores = inject_for(inj, ATTN_DEBUG_SCORES);
  a.num_sms = num_sms();
  a.queue_counter = (int*)((char*)ws + attn::kQueueCounterOffset);
  a.seqlen_q = p->seqlen_q;
  a.seqlen_k = p->seqlen_k;
  a.total_q = p->total_q;
  a.total_k = p->total_k;
  a.thd = thd(p);
  a.lse = lse;
  lse_strides(p, a.lse_sb, a.lse_sh);
  a.d = dbuf;
  default_d_strides(p, a.d_sb, a.d_sh);
  if (wide(p)) {
    a.wide = 1;
    a.wide_plan = (long long*)((char*)ws + lay.plan_off);
    a.wide_blocks = (uint8_t*)ws + lay.blk_off;
    a.wide_cap = lay.cap;
  } else if (ds_path(p)) {
    a.ds = 1;
    a.ds_plan = (long long*)((char*)ws + lay.plan_off);
    a.ds_blocks = (uint8_t*)ws + lay.blk_off;
    a.ds_cap = lay.cap;
  }
  a.q = q; a.k = k; a.v = v; a.o = o; a.dout = dout;
  a.dq = dq; a.dk = dk; a.dvp = dv;
  memcpy(a.sq, p->stride_q, sizeof(a.sq));
  memcpy(a.sk, p->stride_k, sizeof(a.sk));
  memcpy(a.sv, p->stride_v, sizeof(a.sv));
  memcpy(a.so, p->stride_o, sizeof(a.so));
  memcpy(a.sdo, p->stride_do, sizeof(a.sdo));
  memcpy(a.sdq, p->stride_dq, sizeof(a.sdq));
  memcpy(a.sdk, p->stride_dk, sizeof(a.sdk));
  memcpy(a.sdv, p->stride_dv, sizeof(a.sdv));
  if (thd(p)) a.sq[0] = a.sk[0] = a.sv[0] = a.so[0] = a.sdo[0] = a.sdq[0] = a.sdk[0] = a.sdv[0] = 0;
  // tensor maps: 128-row boxes for stationary tiles, 64- or 128-row boxes for streamed ones
  bool ok = true;
  if (need_qkv && has_q) {
    ok &= !map_rows(&a.oq, &a.tm_q128, q, p, p->stride_q, true, p->heads_q, p->d_qk, 128);
    ok &= !map_rows(&a.oq, &a.tm_q64, q, p, p->stride_q, true, p->heads_q, p->d_qk, 64);
    ok &= !map_rows(&a.odo, &a.tm_do128, dout, p, p->stride_do, true, p->heads_q, p->d_v, 128);
    ok &= !map_rows(&a.odo, &a.tm_do64, dout, p, p->stride_do, true, p->heads_q, p->d_v, 64);
  }
  if (need_qkv && has_k) {
    ok &= !map_rows(&a.ok, &a.tm_k128, k, p, p->stride_k, false, p->heads_kv, p->d_qk, 128);
    ok &= !map_rows(&a.ok, &a.tm_k64, k, p, p->stride_k, false, p->heads_kv, p->d_qk, 64);
    ok &= !map_rows(&a.ov, &a.tm_v128, v, p, p->stride_v, false, p->heads_kv, p->d_v, 128);
    ok &= !map_rows(&a.ov, &a.tm_v64, v, p, p->stride_v, false, p->heads_kv, p->d_v, 64);
  }
  if (!ok) return fail(ATTN_ERR_INVALID_ARG, "cannot build a tensor map");
  int n = 0;
  e = attn::launch_bwd(a, st, stages, &n);
  g_launches += n;
  if (e == cudaErrorNotSupported) return fail(ATTN_ERR_UNSUPPORTED, "no backward kernel");
  if (e != cudaSuccess) return cuda_fail(e, "backward kernel launch");
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status_t attn_bwd(const attn_params_t* p, const void* q, const void* k, const void* v,
                       const void* o, const void* dout, const float* lse, void* dq, void* dk,
                       void* dv, void* ws, size_t ws_bytes, attn_stream_t stream) {
  return bwd_impl(p, q, k, v, o, dout, lse, dq, dk, dv, ws, ws_bytes, stream, kStageAll);
}

attn_status_t attn_bwd_preprocess(const attn_params_t* p, const void* q, const void* k,
                                  const void* v, const void* o, const void* dout,
                                  const float* lse, void* dq, void* dk, void* dv, void* ws,
                                  size_t ws_bytes, attn_stream_t stream) {
  return bwd_impl(p, q, k, v, o, dout, lse, dq, dk, dv, ws, ws_bytes, stream, kStagePre);
}

attn_status_t attn_bwd_dq(const attn_params_t* p, const void* q, const void* k, const void* v,
                          const void* o, const void* dout, const float* lse, void* dq, void* dk,
                          void* dv, void* ws, size_t ws_bytes, attn_stream_t stream) {
  return bwd_impl(p, q, k, v, o, dout, lse, dq, dk, dv, ws, ws_bytes, stream, kStageDq);
}

attn_status_t attn_bwd_dkdv(const attn_params_t* p, const void* q, const void* k, const void* v,
                            const void* o, const void* dout, const float* lse, void* dq,
                            void* dk, void* dv, void* ws, size_t ws_bytes,
                            attn_stream_t stream) {
  return bwd_impl(p, q, k, v, o, dout, lse, dq, dk, dv, ws, ws_bytes, stream, kStageDkv);
}

}  // extern "C"

// ----------------------------------------------------------------- attn_bwd_noalloc
// Scratch for callers that cannot allocate: reserved in this library's image,
// so every GPU that loads the library holds it until the process exits.  In
// host code the symbol is only a host-side stand-in; kernels get its device
// address, looked up once per device with that device current.
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_noalloc_addr[kMaxDevices];

attn_status_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device index %d", dev);
  void* ptr = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_noalloc_addr[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return ATTN_OK;
}
}  // namespace

extern "C" {

attn_status_t attn_bwd_noalloc(const attn_params_t* p, const void* q, const void* k,
                               const void* v, const void* o, const void* dout, const float* lse,
                               void* dq, void* dk, void* dv, attn_stream_t stream) {
  g_err[0] = 0;
  g_launches = 0;
  if (attn_status_t s0 = check_params(p)) return s0;
  attn_params_t pr = *p;  // auto: the recompute path, whose workspace is small
  if (pr.bwd_ds == 0) pr.bwd_ds = -1;
  p = &pr;
  const size_t need = attn_bwd_workspace_size(p);
  if (need > kNoAllocScratchBytes)
    return fail(ATTN_ERR_WORKSPACE,
                "problem needs %zu bytes of scratch; attn_bwd_noalloc has a fixed %zu-byte "
                "area (use attn_bwd with a caller workspace)",
                need, kNoAllocScratchBytes);
  void* ws = nullptr;
  attn_status_t s = noalloc_scratch(&ws);
  if (s) return s;
  return bwd_impl(p, q, k, v, o, dout, lse, dq, dk, dv, ws, kNoAllocScratchBytes, stream,
                  kStageAll);
}

}  // extern "C"

// ----------------------------------------------------------------- attn_fwd_bwd_host
// One step from host buffers: every tensor is copied into the caller's device
// arena, the forward and backward run there, and the results are copied back,
// all in order on the caller's stream.  The arena holds each tensor with the
// layout (strides) the caller gave for its host copy.
namespace {

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Bytes from a tensor's base to the end of its last element.
size_t tensor_bytes(const int64_t s[3], const attn_params_t* p, bool is_q, int heads, int d,
                    size_t es) {
  return (size_t)span_of(nullptr, s, p, is_q, heads, d, es).hi;
}

size_t lse_bytes(const attn_params_t* p) {
  int64_t sb = 0, sh = 0;
  lse_strides(p, sb, sh);
  const int64_t rows = thd(p) ? p->total_q : p->seqlen_q;
  const int64_t nb = thd(p) ? 1 : p->batch;
  if (rows <= 0 || nb <= 0 || p->heads_q <= 0) return 0;
  return (size_t)(((nb - 1) * sb + (int64_t)(p->heads_q - 1) * sh + rows) * 4);
}

struct HostArena {
  // byte offsets into the arena, and the bytes each tensor spans
  size_t fws, bws, off[9], bytes[9], cu_q, cu_k, used_q, used_k, total;
};
enum { kQ, kK, kV, kDo, kO, kLse, kDq, kDk, kDv };

HostArena host_arena(const attn_params_t* p) {
  HostArena a;
  memset(&a, 0, sizeof(a));
  const size_t g = esize(p->grad_dtype);
  a.bytes[kQ] = tensor_bytes(p->stride_q, p, true, p->heads_q, p->d_qk, 2);
  a.bytes[kK] = tensor_bytes(p->stride_k, p, false, p->heads_kv, p->d_qk, 2);
  a.bytes[kV] = tensor_bytes(p->stride_v, p, false, p->heads_kv, p->d_v, 2);
  a.bytes[kDo] = tensor_bytes(p->stride_do, p, true, p->heads_q, p->d_v, 2);
  a.bytes[kO] = tensor_bytes(p->stride_o, p, true, p->heads_q, p->d_v, esize(p->o_dtype));
  a.bytes[kLse] = lse_bytes(p);
  a.bytes[kDq] = tensor_bytes(p->stride_dq, p, true, p->heads_q, p->d_qk, g);
  a.bytes[kDk] = tensor_bytes(p->stride_dk, p, false, p->heads_kv, p->d_qk, g);
  a.bytes[kDv] = tensor_bytes(p->stride_dv, p, false, p->heads_kv, p->d_v, g);
  size_t at = 0;
  a.fws = at;
  at += up256(attn_fwd_workspace_size(p));
  a.bws = at;
  at += up256(attn_bwd_workspace_size(p));
  for (int i = 0; i < 9; ++i) {
    a.off[i] = at;
    at += up256(a.bytes[i]);
  }
  if (thd(p)) {
    const size_t cu = (size_t)(p->batch + 1) * 4, used = (size_t)p->batch * 4;
    a.cu_q = at;
    at += up256(cu);
    a.cu_k = at;
    at += up256(cu);
    if (p->seqused_q) {
      a.used_q = at;
      at += up256(used);
      a.used_k = at;
      at += up256(used);
    }
  }
  a.total = at;
  return a;
}

// The caller's buffers must be host memory: a device pointer here is a mix-up.
attn_status_t check_host(const char* name, const void* ptr) {
  if (!ptr) return ATTN_OK;
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();  // older drivers flag unregistered host memory; it is fine here
    return ATTN_OK;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged)
    return fail(ATTN_ERR_INVALID_ARG, "%s is device memory; attn_fwd_bwd_host takes host buffers",
                name);
  return ATTN_OK;
}

attn_status_t copy(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind,
                   cudaStream_t st, const char* what) {
  if (!bytes) return ATTN_OK;
  const cudaError_t e = cudaMemcpyAsync(dst, src, bytes, kind, st);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, what);
}

}  // namespace

extern "C" {

size_t attn_host_arena_size(const attn_params_t* p) {
  if (!p || check_params(p)) return 0;
  return host_arena(p).total;
}

attn_status_t attn_fwd_bwd_host_stages(const attn_params_t* p, const void* q, const void* k,
                                       const void* v, const void* dout, void* o, float* lse,
                                       void* dq, void* dk, void* dv, void* arena,
                                       size_t arena_bytes, unsigned stages, attn_stream_t stream) {
  g_err[0] = 0;
  g_launches = 0;
  attn_status_t s = check_params(p);
  if (s) return s;
  if (!stages || (stages & ~7u)) return fail(ATTN_ERR_INVALID_ARG, "stages must be a mask of 1, 2, 4");
  const HostArena a = host_arena(p);
  if (!arena) return fail(ATTN_ERR_WORKSPACE, "arena is NULL");
  if ((uintptr_t)arena % 256) return fail(ATTN_ERR_ALIGNMENT, "arena is not 256-byte aligned");
  if (arena_bytes < a.total)
    return fail(ATTN_ERR_WORKSPACE, "arena too small (%zu < %zu)", arena_bytes, a.total);
  const bool up = stages & ATTN_HOST_UPLOAD, run = stages & ATTN_HOST_COMPUTE,
             down = stages & ATTN_HOST_DOWNLOAD;
  const void* host_in[4] = {q, k, v, dout};
  void* host_out[5] = {o, lse, dq, dk, dv};
  static const char* const names[9] = {"q", "k", "v", "dout", "o", "lse", "dq", "dk", "dv"};
  for (int i = 0; i < 9; ++i) {
    // inputs are read by the upload; outputs written by the download (and the
    // gradients read by the upload when they are accumulated)
    const bool used = i < 4 ? up : (down || (up && p->accumulate && i >= kDq));
    if (!used) continue;
    const void* h = i < 4 ? host_in[i] : host_out[i - 4];
    if (a.bytes[i] && !h) return fail(ATTN_ERR_INVALID_ARG, "%s is NULL", names[i]);
    if ((s = check_host(names[i], h))) return s;
  }
  if (up) {
    if ((s = check_host("cu_seqlens_q", p->cu_seqlens_q))) return s;
    if ((s = check_host("seqused_q", p->seqused_q))) return s;
  }
  cudaStream_t st = (cudaStream_t)stream;
  char* base = (char*)arena;
  if (up) {
    if (thd(p)) {
      const size_t cu = (size_t)(p->batch + 1) * 4, used = (size_t)p->batch * 4;
      if ((s = copy(base + a.cu_q, p->cu_seqlens_q, cu, cudaMemcpyHostToDevice, st, "cu_seqlens_q")) ||
          (s = copy(base + a.cu_k, p->cu_seqlens_k, cu, cudaMemcpyHostToDevice, st, "cu_seqlens_k")))
        return s;
      if (p->seqused_q &&
          ((s = copy(base + a.used_q, p->seqused_q, used, cudaMemcpyHostToDevice, st, "seqused_q")) ||
           (s = copy(base + a.used_k, p->seqused_k, used, cudaMemcpyHostToDevice, st, "seqused_k"))))
        return s;
    }
    for (int i = 0; i < 4; ++i)
      if ((s = copy(base + a.off[i], host_in[i], a.bytes[i], cudaMemcpyHostToDevice, st, names[i])))
        return s;
    if (p->accumulate)  // the gradients are summed into the caller's values
      for (int i = kDq; i <= kDv; ++i)
        if ((s = copy(base + a.off[i], host_out[i - 4], a.bytes[i], cudaMemcpyHostToDevice, st,
                      names[i])))
          return s;
  }
  if (run) {
    // the device copy of the parameters: same shape and strides, the
    // metadata arrays in the arena
    attn_params_t pd = *p;
    if (thd(p)) {
      pd.cu_seqlens_q = (const int32_t*)(base + a.cu_q);
      pd.cu_seqlens_k = (const int32_t*)(base + a.cu_k);
      if (p->seqused_q) {
        pd.seqused_q = (const int32_t*)(base + a.used_q);
        pd.seqused_k = (const int32_t*)(base + a.used_k);
      }
    }
    s = attn_fwd(&pd, base + a.off[kQ], base + a.off[kK], base + a.off[kV], base + a.off[kO],
                 (float*)(base + a.off[kLse]), base + a.fws, a.bws - a.fws, stream);
    if (s) return s;
    const int fwd_launches = g_launches;
    s = attn_bwd(&pd, base + a.off[kQ], base + a.off[kK], base + a.off[kV], base + a.off[kO],
                 base + a.off[kDo], (const float*)(base + a.off[kLse]), base + a.off[kDq],
                 base + a.off[kDk], base + a.off[kDv], base + a.bws, a.off[0] - a.bws, stream);
    g_launches += fwd_launches;
    if (s) return s;
  }
  if (down)
    for (int i = kO; i <= kDv; ++i)
      if ((s = copy(host_out[i - 4], base + a.off[i], a.bytes[i], cudaMemcpyDeviceToHost, st,
                    names[i])))
        return s;
  return ATTN_OK;
}

attn_status_t attn_fwd_bwd_host(const attn_params_t* p, const void* q, const void* k,
                                const void* v, const void* dout, void* o, float* lse, void* dq,
                                void* dk, void* dv, void* arena, size_t arena_bytes,
                                attn_stream_t stream) {
  return attn_fwd_bwd_host_stages(p, q, k, v, dout, o, lse, dq, dk, dv, arena, arena_bytes,
                                  ATTN_HOST_ALL, stream);
}

attn_status_t attn_lse_merge(int n_parts, const float* const* o_parts,
                             const float* const* lse_parts, const int64_t* part_row0,
                             const int64_t* part_rows, int64_t rows, int heads, int d_v,
                             void* o_out, attn_dtype_t o_dtype, float* lse_out,
                             attn_stream_t stream) {
  g_err[0] = 0;
  g_launches = 0;
  if (n_parts < 1 || n_parts > attn::kMaxParts)
    return fail(ATTN_ERR_INVALID_ARG, "n_parts must be in [1, %d]", attn::kMaxParts);
  if (!o_parts || !lse_parts || !part_row0 || !part_rows)
    return fail(ATTN_ERR_INVALID_ARG, "part arrays must not be NULL");
  if (rows < 0 || heads <= 0 || d_v <= 0) return fail(ATTN_ERR_INVALID_ARG, "bad shape");
  if (d_v % 4) return fail(ATTN_ERR_UNSUPPORTED, "d_v must be a multiple of 4");
  if (o_dtype != ATTN_BF16 && o_dtype != ATTN_FP16 && o_dtype != ATTN_FP32)
    return fail(ATTN_ERR_INVALID_ARG, "bad o_dtype");
  if (rows == 0) return ATTN_OK;
  if (!o_out || !lse_out) return fail(ATTN_ERR_INVALID_ARG, "outputs must not be NULL");
  const size_t oe = esize(o_dtype);
  if ((uintptr_t)o_out % (oe * 4) != 0)
    return fail(ATTN_ERR_ALIGNMENT, "o_out must be aligned to 4 elements");
  attn::MergeParams mp;
  memset(&mp, 0, sizeof(mp));
  const Span out_o{(uintptr_t)o_out, (uintptr_t)o_out + (uintptr_t)(rows * heads * (int64_t)d_v * oe)};
  const Span out_l{(uintptr_t)lse_out, (uintptr_t)lse_out + (uintptr_t)(rows * heads * 4)};
  for (int i = 0; i < n_parts; ++i) {
    if (part_rows[i] < 0 || part_row0[i] < 0 || part_row0[i] + part_rows[i] > rows)
      return fail(ATTN_ERR_INVALID_ARG, "part %d row range outside [0, rows)", i);
    if (part_rows[i] > 0) {
      if (!o_parts[i] || !lse_parts[i])
        return fail(ATTN_ERR_INVALID_ARG, "part %d pointer is NULL", i);
      if ((uintptr_t)o_parts[i] % 16)
        return fail(ATTN_ERR_ALIGNMENT, "part %d O is not 16-byte aligned", i);
      const Span po{(uintptr_t)o_parts[i],
                    (uintptr_t)o_parts[i] + (uintptr_t)(part_rows[i] * heads * (int64_t)d_v * 4)};
      const Span pl{(uintptr_t)lse_parts[i],
                    (uintptr_t)lse_parts[i] + (uintptr_t)(part_rows[i] * heads * 4)};
      if (overlap(po, out_o) || overlap(po, out_l) || overlap(pl, out_o) || overlap(pl, out_l))
        return fail(ATTN_ERR_INVALID_ARG, "part %d overlaps an output", i);
    }
    mp.o[i] = o_parts[i];
    mp.lse[i] = lse_parts[i];
    mp.row0[i] = part_row0[i];
    mp.nrows[i] = part_rows[i];
  }
  mp.n = n_parts;
  mp.rows = rows;
  mp.heads = heads;
  mp.dv = d_v;
  mp.o_out = o_out;
  mp.lse_out = lse_out;
  mp.out_kind = o_dtype == ATTN_BF16 ? 0 : (o_dtype == ATTN_FP16 ? 1 : 2);
  cudaError_t e = attn::launch_merge(mp, num_sms(), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  g_launches = 1;
  return ATTN_OK;
}

attn_status_t attn_cp_relayout(int to_heads, int cp, int64_t seqlen, int heads, int d,
                               int elem_bytes, const void* src, const int64_t src_strides[3],
                               void* dst, const int64_t dst_strides[3], attn_stream_t stream) {
  g_err[0] = 0;
  g_launches = 0;
  if (cp < 1 || heads < 1 || d < 1 || seqlen < 1)
    return fail(ATTN_ERR_INVALID_ARG, "cp, heads, d and seqlen must be positive");
  if (seqlen % (2 * (int64_t)cp)) return fail(ATTN_ERR_INVALID_ARG, "seqlen must split into 2*cp chunks");
  if (heads % cp) return fail(ATTN_ERR_INVALID_ARG, "heads must divide by cp");
  if (elem_bytes != 2 && elem_bytes != 4) return fail(ATTN_ERR_INVALID_ARG, "elem_bytes must be 2 or 4");
  if (!src || !dst || !src_strides || !dst_strides) return fail(ATTN_ERR_INVALID_ARG, "NULL argument");
  if ((uintptr_t)src % elem_bytes || (uintptr_t)dst % elem_bytes)
    return fail(ATTN_ERR_ALIGNMENT, "pointers must be aligned to elem_bytes");
  for (int i = 0; i < 3; ++i)
    if (src_strides[i] < 0 || dst_strides[i] < 0) return fail(ATTN_ERR_INVALID_ARG, "negative stride");
  // extents of both sides (elements), for the overlap check
  const int64_t chunk = seqlen / (2 * cp);
  const int64_t* ss = to_heads ? src_strides : dst_strides;  // sequence side
  const int64_t* hs = to_heads ? dst_strides : src_strides;  // head side
  const int64_t seq_last = (cp - 1) * ss[0] + (2 * chunk - 1) * ss[1] + (int64_t)(heads - 1) * ss[2] + d;
  const int64_t head_last = (cp - 1) * hs[0] + (seqlen - 1) * hs[1] + (int64_t)(heads / cp - 1) * hs[2] + d;
  const Span s_src{(uintptr_t)src, (uintptr_t)src + (uintptr_t)((to_heads ? seq_last : head_last) * elem_bytes)};
  const Span s_dst{(uintptr_t)dst, (uintptr_t)dst + (uintptr_t)((to_heads ? head_last : seq_last) * elem_bytes)};
  if (overlap(s_src, s_dst)) return fail(ATTN_ERR_INVALID_ARG, "src and dst overlap");
  attn::RelayoutParams rp;
  memset(&rp, 0, sizeof(rp));
  rp.src = (const uint8_t*)src;
  rp.dst = (uint8_t*)dst;
  memcpy(rp.seq_s, ss, sizeof(rp.seq_s));
  memcpy(rp.head_s, hs, sizeof(rp.head_s));
  rp.seqlen = seqlen;
  rp.cp = cp;
  rp.heads = heads;
  rp.d = d;
  rp.elem_bytes = elem_bytes;
  rp.to_heads = to_heads ? 1 : 0;
  cudaError_t e = attn::launch_relayout(rp, num_sms(), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "relayout kernel launch");
  g_launches = 1;
  return ATTN_OK;
}

attn_status_t attn_query_status(const void* ws, attn_stream_t stream) {
  if (!ws) return fail(ATTN_ERR_INVALID_ARG, "workspace is NULL");
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (v == attn::DEV_OK) return ATTN_OK;
  if (v == attn::DEV_BAD_SEQLENS)
    return fail(ATTN_ERR_BAD_METADATA, "device check: cu_seqlens inconsistent");
  if (v == attn::DEV_TIMEOUT) return fail(ATTN_ERR_TIMEOUT, "device wait exceeded its limit");
  if (v == attn::DEV_WORKSPACE)
    return fail(ATTN_ERR_WORKSPACE, "device check: score tiles exceed the workspace");
  return fail(ATTN_ERR_CUDA, "device status %d", v);
}

const char* attn_last_error(void) { return g_err; }

void attn_debug_inject(unsigned kernel_mask, int drop_load, uint64_t wait_limit_ns) {
  g_inject = Inject{kernel_mask, drop_load, (unsigned long long)wait_limit_ns};
}

int attn_last_launch_count(void) { return g_launches; }

}  // extern "C"
