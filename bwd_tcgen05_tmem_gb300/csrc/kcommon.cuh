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
// The persistent kernel (CTAs take work items from a queue): every CTA uses
// the injected wait limit, and the CTA that runs work item 0 leaves out load
// `drop_load` of that item (a healthy wait lasts microseconds, so the short
// limit only runs out where the load is missing).
__device__ __forceinline__ unsigned long long wait_limit_all(const DebugInject& d) {
  return d.wait_ns ? d.wait_ns : kWaitLimitNs;
}

// ----------------------------------------------------------------- work queue
// A persistent kernel (one CTA per SM) takes its work items from a global
// counter, in the order a one-CTA-per-item grid would run them, so the SMs
// stay balanced the way the hardware's block scheduler balances blocks.  One
// lane of the producer warp takes the next index (atomicAdd) and publishes it
// in a small shared ring; every other role pops the indices in the same
// order.  -1 marks the end.  The counter (in the caller's workspace) is zeroed
// before each launch.
template <int N>
struct ItemRing {
  int idx[N];
  uint64_t full[N], empty[N];
};

template <int N>
__device__ __forceinline__ void item_ring_init(ItemRing<N>& r, uint32_t consumers) {
  for (int i = 0; i < N; ++i) {
    mbar_init(&r.full[i], 1);
    mbar_init(&r.empty[i], consumers);
  }
}

// Producer warp (all lanes): the q-th item index, or -1 past the last item.
template <int N>
__device__ __forceinline__ int item_ring_push(ItemRing<N>& r, int q, int* counter, int n_items,
                                              const Abort& ab, bool& ok) {
  const int slot = q % N;
  if (q >= N && !mbar_wait_warp(&r.empty[slot], ((q / N) - 1) & 1u, ab)) {
    ok = false;
    return -1;
  }
  int v = -1;
  if ((threadIdx.x & 31) == 0) {
    v = atomicAdd(counter, 1);
    if (v >= n_items) v = -1;
    r.idx[slot] = v;
    mbar_arrive(&r.full[slot]);
  }
  return __shfl_sync(0xffffffffu, v, 0);
}

// Consumer warp (all lanes): the q-th item index, or -1 past the last item.
template <int N>
__device__ __forceinline__ int item_ring_pop(ItemRing<N>& r, int q, const Abort& ab, bool& ok) {
  const int slot = q % N;
  if (!mbar_wait_warp(&r.full[slot], (q / N) & 1u, ab)) {
    ok = false;
    return -1;
  }
  const int v = *(volatile int*)&r.idx[slot];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&r.empty[slot]);
  return v;
}

// Byte offset of the work-queue counter in a workspace (after the status word).
constexpr int kQueueCounterOffset = 128;

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
