// kcommon.cuh -- sequence geometry, visibility bounds and kernel parameter
// blocks shared by the attention kernels.
//
// Visibility (TransformerEngine PR #3527 review notes on sliding windows and
// causal alignment): with off = Lk - Lq for bottom-right alignment (0 for
// top-left), key j is visible from query i iff
//     i + off - L <= j <= i + off + R,   0 <= j < Lk,
// where L = window_left (unbounded if < 0) and R = 0 when causal, else
// window_right (unbounded if < 0).  A causal mask pins the right bound to the
// diagonal; the left bound counts visible tokens including the diagonal.
#pragma once
#include <stdint.h>

#include "tc.cuh"
#include "tmap.h"

namespace attn {

constexpr int kBlockM = 128;  // stationary rows per CTA (TMEM lanes)
constexpr int kBlockN = 128;  // streamed rows per tile
constexpr int kSlotBytes = 128 * 64 * 2;
constexpr int kMaxSlots = 14;  // 14 x 16 KiB + alignment pad fits in 227 KiB
constexpr long long kInfBound = (1ll << 40);

// Grid order.  With many tiles per head, x walks the tiles of one head so the
// CTAs resident at one time stream the same head's operands from L2; with
// few, x walks the heads so the heaviest tiles of every head start first.
constexpr int kTileMajorMin = 64;
__host__ __device__ inline bool tile_major(int n_tiles) { return n_tiles >= kTileMajorMin; }

struct Geometry {
  const int32_t* cu_q;  // null: dense
  const int32_t* cu_k;
  const int32_t* used_q;  // padded THD: visible length of each sequence (else null)
  const int32_t* used_k;
  int seqlen_q, seqlen_k;  // dense lengths (ignored for varlen)
  int causal, bottom_right, wl, wr;
};

struct Seq {
  int q_start, k_start;  // first token of the sequence (THD) or 0
  int lq, lk;
  long long off, L, R;
};

__device__ __forceinline__ Seq load_seq(const Geometry& g, int b) {
  Seq s;
  if (g.cu_q) {
    s.q_start = g.cu_q[b];
    s.lq = g.used_q ? g.used_q[b] : g.cu_q[b + 1] - s.q_start;
    s.k_start = g.cu_k[b];
    s.lk = g.used_k ? g.used_k[b] : g.cu_k[b + 1] - s.k_start;
  } else {
    s.q_start = 0;
    s.k_start = 0;
    s.lq = g.seqlen_q;
    s.lk = g.seqlen_k;
  }
  s.off = g.bottom_right ? (long long)(s.lk - s.lq) : 0ll;
  s.L = g.wl < 0 ? kInfBound : (long long)g.wl;
  s.R = g.causal ? 0ll : (g.wr < 0 ? kInfBound : (long long)g.wr);
  return s;
}

// Keys visible from any query in [i0, i1] (inclusive) -> [j0, j1]; empty if j1 < j0.
__host__ __device__ inline void key_range(const Seq& s, long long i0, long long i1, long long& j0,
                                          long long& j1) {
  j0 = i0 + s.off - s.L;
  j1 = i1 + s.off + s.R;
  if (j0 < 0) j0 = 0;
  if (j1 > s.lk - 1) j1 = s.lk - 1;
}

// Queries that see any key in [j0, j1] -> [i0, i1]; empty if i1 < i0.
__host__ __device__ inline void query_range(const Seq& s, long long j0, long long j1,
                                            long long& i0, long long& i1) {
  i0 = j0 - s.off - s.R;
  i1 = j1 - s.off + s.L;
  if (i0 < 0) i0 = 0;
  if (i1 > s.lq - 1) i1 = s.lq - 1;
}

// ----------------------------------------------------------------- fault injection
// Test-only (attn_debug_inject): the first CTA of a launch may run with a
// shorter wait limit and leave out one of its loads, so that a wait is certain
// to run out and the unwind path (abort flag, status word, in-flight copies
// landed, MMAs drained, TMEM freed) runs.  Every other CTA, and every launch
// without an injection, uses kWaitLimitNs and leaves out nothing.
struct DebugInject {
  unsigned long long wait_ns;  // 0: kWaitLimitNs
  int drop_load;               // index of the load the first CTA leaves out; -1: none
};

__device__ __forceinline__ bool first_cta() {
  return (blockIdx.x | blockIdx.y | blockIdx.z) == 0;
}
__device__ __forceinline__ unsigned long long wait_limit(const DebugInject& d) {
  return (d.wait_ns && first_cta()) ? d.wait_ns : kWaitLimitNs;
}
__device__ __forceinline__ int dropped_load(const DebugInject& d) {
  return first_cta() ? d.drop_load : -1;
}

// ----------------------------------------------------------------- params
struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;
  MapOrder oq, ok, ov;
  Geometry geo;
  void* o;            // [B,S,Hq,dv] (dense) or [T,Hq,dv]; element strides below
  float* lse;         // natural-log LSE
  int64_t so_b, so_t, so_h;
  int64_t lse_sb, lse_sh;  // LSE index = b*lse_sb + h*lse_sh + token
  int batch, hq, hkv, n_qtiles, n_split;
  float scale_log2;
  int* status;
  DebugInject dbg;
};

}  // namespace attn
