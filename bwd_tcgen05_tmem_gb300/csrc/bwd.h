// bwd.h -- argument block of the backward pass and its kernel parameter
// blocks (definitions in bwd_dq.cu, bwd_dkdv.cu, bwd_dq_ds.cu, bwd_wide.cu,
// bwd.cu).
#pragma once
#include "kcommon.cuh"

namespace attn {

// Everything attn_bwd resolved on the host.
struct BwdArgs {
  Geometry geo;
  int batch, hq, hkv, dqk, dv, seqlen_q, seqlen_k, total_q, total_k, thd;
  bool bf16, g_f32;
  int accum;  // FP32 gradients: add into the outputs
  float scale, scale_log2;
  int* status;
  int num_sms;
  int* queue_counter;  // work-queue counter in the workspace (persistent kernels)
  const float* lse;
  int64_t lse_sb, lse_sh;
  // per row {LSE * log2 e (+inf for a row without keys), D}: written by the
  // preprocess, the only row statistics the backward kernels read (one array
  // read in lockstep, wherever the caller's LSE lives)
  float2* d;
  int64_t d_sb, d_sh;
  const void *q, *k, *v, *o, *dout;
  void *dq, *dk, *dvp;
  int64_t sq[3], sk[3], sv[3], so[3], sdo[3], sdq[3], sdk[3], sdv[3];
  CUtensorMap tm_q128, tm_q64, tm_do128, tm_do64, tm_k128, tm_k64, tm_v128, tm_v64;
  MapOrder oq, odo, ok, ov;
  // the materialising backward (see wide_backward): per-sequence block
  // prefix and the score tiles
  int wide;
  long long* wide_plan;
  uint8_t* wide_blocks;
  long long wide_cap;
  // the dS backward (see ds_backward): the dK/dV kernel also writes dS, the
  // dQ GEMM reads it; per-sequence block prefix and the dS blocks
  int ds;
  long long* ds_plan;
  uint8_t* ds_blocks;
  long long ds_cap;
  // test-only fault injection (attn_debug_inject), per kernel: dQ / dK-dV
  // kernels, or the scores kernel and the dQ / dK-dV GEMMs of the wide path
  DebugInject dbg_dq, dbg_dkdv, dbg_scores;
};

// ---------------------------------------------------------------- wide path
// Head dims above 256 materialise P and dS: one 64 KiB block per (sequence,
// query head, 128-row query tile, visible 128-key block), holding four
// 128 x 64 16-bit tiles in their 128-byte-swizzled shared-memory image:
// P keys 0-63, P keys 64-127, dS keys 0-63, dS keys 64-127.
constexpr int kWideTile = 128 * 64 * 2;
constexpr int kWideBlock = 4 * kWideTile;

// The backward materialises P and dS for head dims above 256 (the fused
// kernels cannot hold them), and at head dim 256 whenever the P/dS blocks fit
// in kWideD256Cap bytes: there the fused path needs a dV-only and a dK-only
// launch that both recompute the scores, while this path runs each
// contraction once (20-25 % faster, bit-identical results on GB300).
constexpr long long kWideD256Cap = 16ll << 30;
inline bool wide_backward(int dqk, int dv, long long block_bytes) {
  return dqk > 256 || dv > 256 || (dqk == 256 && dv == 256 && block_bytes <= kWideD256Cap);
}

// Visible 128-key blocks of query tile qt: returns their count, first in kb0.
__host__ __device__ inline int wide_blocks_of_qtile(const Seq& s, int qt, int& kb0) {
  const long long i0 = (long long)qt * 128;
  kb0 = 0;
  if (i0 > (long long)s.lq - 1) return 0;
  const long long i1 = i0 + 127 < (long long)s.lq - 1 ? i0 + 127 : (long long)s.lq - 1;
  long long j0, j1;
  key_range(s, i0, i1, j0, j1);
  if (j1 < j0) return 0;
  kb0 = (int)(j0 / 128);
  return (int)(j1 / 128) - kb0 + 1;
}

// Blocks of query tiles [0, qt) of one sequence; called by a whole warp.
__device__ inline long long blocks_row_prefix(const Seq& s, int qt) {
  long long acc = 0;
  int kb0;
  for (int t = (int)(threadIdx.x & 31); t < qt; t += 32) acc += wide_blocks_of_qtile(s, t, kb0);
#pragma unroll
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

__device__ __forceinline__ bool status_set(const int* status) {
  return status && *(volatile const int*)status;
}

__device__ __forceinline__ void raise_status(int* status, int code) {
  if (status) atomicCAS(status, DEV_OK, code);
}

// ---------------------------------------------------------------- dS path
// At head dims up to 192 the backward can keep dS instead of recomputing the
// scores for dQ: the key-stationary dK/dV kernel, which computes every dS
// element anyway, writes it once to the workspace, and dQ = scale dS K is a
// GEMM over those blocks (S and dP are then computed once per query-key pair
// instead of twice).  One 32 KiB block per (sequence, query head, 128-row
// query tile, visible 128-key block), indexed like the wide path's blocks
// (hq*plan[b] + h*T_b + rowprefix_b(qt) + kb - kb0(qt)), holding dS as the
// MN-major A operand of the dQ MMA in the unswizzled layout: the 16 bytes of
// queries 8c .. 8c+7 of key row r sit at c*2048 + r*16.  Then the 32 key rows
// a warp of the dK/dV kernel holds land in 512 contiguous bytes per store.
constexpr int kDsChunk = 128 * 16;  // one 8-query column of all 128 key rows
constexpr int kDsBlock = 16 * kDsChunk;

// The dS path serves head dims 128/128 and 192/128 (single-launch dK/dV
// kernels) while its blocks take at most kDsCap bytes; ds_mode (the params'
// bwd_ds field) forces it off (-1) or on (1).  The trade, measured on GB300:
// the dK/dV kernel slows by about a fifth with 32 KiB of dS stores per tile,
// the dQ GEMM streams them at the copy bandwidth, and dQ no longer
// recomputes S and dP per pair: B1 H32 S32K 192/128 fwd+bwd 33.0 -> 28.9 ms,
// THD 65K tokens 128/128 9.39 -> 8.99 ms.  At 64/64 recomputing is cheaper
// than streaming 32 KiB per 128 x 128 tile.
constexpr long long kDsCap = 64ll << 30;
inline bool ds_backward(int dqk, int dv, long long block_bytes, int ds_mode) {
  const bool shape = (dqk == 128 && dv == 128) || (dqk == 192 && dv == 128);
  if (!shape || ds_mode < 0) return false;
  return ds_mode > 0 || block_bytes <= kDsCap;
}

struct WidePlanParams {
  Geometry geo;
  long long* plan;  // [batch + 1] exclusive prefix of per-sequence block counts
  long long cap;    // blocks the workspace holds
  int batch, hq;
  int* status;
};

struct WideScoresParams {
  CUtensorMap tm_q, tm_k, tm_v;  // 128-row boxes
  MapOrder oq, ok, ov;
  Geometry geo;
  const float2* d;  // per row {LSE * log2 e, D} (the preprocess writes it)
  int64_t d_sb, d_sh;
  const void* dout;
  int64_t sdo_b, sdo_t, sdo_h;
  const long long* plan;
  uint8_t* blocks;
  long long cap;
  int batch, hq, hkv, n_qtiles;
  float scale_log2;
  int* status;
  DebugInject dbg;
};

// dQ (kind 0: per query tile) and dV / dK (kind 1: per key tile) GEMMs over
// the materialised tiles.
struct WideAccParams {
  CUtensorMap tm_b0, tm_b1;  // B operand (64-row boxes): dQ: K, -;  dK/dV: dO, Q
  MapOrder ob0, ob1;
  Geometry geo;
  const long long* plan;
  const uint8_t* blocks;
  long long cap;
  void* out0;  // dQ, or dV
  int64_t so0_b, so0_t, so0_h;
  void* out1;  // dK
  int64_t so1_b, so1_t, so1_h;
  int accum;
  int batch, hq, hkv, n_tiles;
  float scale;
  int* status;
  DebugInject dbg;
};

// q-stationary kernel: dQ = scale * sum_j dS_ij k_j
struct DqParams {
  CUtensorMap tm_q, tm_do, tm_k, tm_v;  // q/do: 128-row boxes, k/v: BKV-row boxes
  MapOrder oq, odo, ok, ov;
  Geometry geo;
  const float2* d;  // per row {LSE * log2 e, D} (the preprocess writes it)
  int64_t d_sb, d_sh;
  void* dq;
  int64_t sdq_b, sdq_t, sdq_h;
  int accum;
  int batch, hq, hkv, n_qtiles;
  int* counter;  // work-queue counter (zeroed before the launch)
  float scale, scale_log2;
  int* status;
  DebugInject dbg;
};

// kv-stationary kernel: dV = sum P^T dO, dK = scale * sum dS^T Q over the group
struct DkvParams {
  CUtensorMap tm_k, tm_v, tm_q, tm_do;  // k/v: 128-row boxes, q/do: BQ-row boxes
  MapOrder ok, ov, oq, odo;
  Geometry geo;
  const float2* d;  // per row {LSE * log2 e, D} (the preprocess writes it)
  int64_t d_sb, d_sh;
  void *dk, *dv;
  int64_t sdk_b, sdk_t, sdk_h, sdv_b, sdv_t, sdv_h;
  int accum;
  int batch, hq, hkv, n_ktiles;
  float scale, scale_log2;
  int* status;
  DebugInject dbg;
  // dS path: write dS of every visited tile into its block (null: do not)
  uint8_t* ds;
  const long long* plan;
  long long cap;
};

// dQ GEMM of the dS path: dQ = scale * sum_kb dS_kb K_kb per query tile
struct DqDsParams {
  CUtensorMap tm_k;  // 128-row boxes
  MapOrder ok;
  Geometry geo;
  const long long* plan;
  const uint8_t* blocks;
  long long cap;
  void* dq;
  int64_t sdq_b, sdq_t, sdq_h;
  int accum;
  int batch, hq, hkv, n_qtiles;
  int* counter;  // work-queue counter (zeroed before the launch)
  float scale;
  int* status;
  DebugInject dbg;
};

cudaError_t launch_wide_plan(const WidePlanParams& p, cudaStream_t st);
cudaError_t launch_dq_ds(const DqDsParams& p, int dqk, bool bf16, bool gf32, int num_sms,
                         cudaStream_t st);

cudaError_t launch_bwd_wide(const BwdArgs& a, cudaStream_t st, int stages, int* n_launches);

// stages: bit 0 D preprocess, bit 1 dQ, bit 2 dK/dV
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t st, int stages, int* n_launches);

}  // namespace attn
