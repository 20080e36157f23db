// bwd.h -- argument block of the backward pass and its kernel parameter
// blocks (definitions in bwd_dq.cu, bwd_dkdv.cu, bwd.cu).
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
  const float* lse;
  int64_t lse_sb, lse_sh;
  float* d;
  int64_t d_sb, d_sh;
  const void *q, *k, *v, *o, *dout;
  void *dq, *dk, *dvp;
  int64_t sq[3], sk[3], sv[3], so[3], sdo[3], sdq[3], sdk[3], sdv[3];
  CUtensorMap tm_q128, tm_q64, tm_do128, tm_do64, tm_k128, tm_k64, tm_v128, tm_v64;
  MapOrder oq, odo, ok, ov;
};

// q-stationary kernel: dQ = scale * sum_j dS_ij k_j
struct DqParams {
  CUtensorMap tm_q, tm_do, tm_k, tm_v;  // q/do: 128-row boxes, k/v: BKV-row boxes
  MapOrder oq, odo, ok, ov;
  Geometry geo;
  const float* lse;
  int64_t lse_sb, lse_sh;
  const float* d;
  int64_t d_sb, d_sh;
  void* dq;
  int64_t sdq_b, sdq_t, sdq_h;
  int accum;
  int batch, hq, hkv, n_qtiles;
  float scale, scale_log2;
  int* status;
};

// kv-stationary kernel: dV = sum P^T dO, dK = scale * sum dS^T Q over the group
struct DkvParams {
  CUtensorMap tm_k, tm_v, tm_q, tm_do;  // k/v: 128-row boxes, q/do: BQ-row boxes
  MapOrder ok, ov, oq, odo;
  Geometry geo;
  const float* lse;
  int64_t lse_sb, lse_sh;
  const float* d;
  int64_t d_sb, d_sh;
  void *dk, *dv;
  int64_t sdk_b, sdk_t, sdk_h, sdv_b, sdv_t, sdv_h;
  int accum;
  int batch, hq, hkv, n_ktiles;
  float scale, scale_log2;
  int* status;
};

// stages: bit 0 D preprocess, bit 1 dQ, bit 2 dK/dV
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t st, int stages, int* n_launches);

}  // namespace attn
