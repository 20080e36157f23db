// small_params.h -- parameter blocks and launchers of the memory-bound kernels
// (D preprocess, LSE merge, cu_seqlens check) defined in small.cu.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

struct PreParams {
  const void* o;
  const void* dout;
  // per row (token, query head), in the LSE layout: {LSE * log2 e (+inf
  // for a row without keys), D}, what the backward kernels read together
  float2* d;
  const float* lse;
  int64_t lse_sb, lse_sh;  // LSE index = b*lse_sb + h*lse_sh + token
  const int32_t* cu_q;  // null: dense
  const int32_t* used_q;  // padded THD: rows past used_q[b] are a gap (skipped)
  int64_t so_b, so_t, so_h, sdo_b, sdo_t, sdo_h;
  int64_t d_sb, d_sh;   // row statistics index = b*d_sb + h*d_sh + token
  int batch, seqlen_q, total_q, hq, dv;
  int* status;
};

constexpr int kMaxParts = 64;
struct MergeParams {
  const float* o[kMaxParts];
  const float* lse[kMaxParts];
  int64_t row0[kMaxParts], nrows[kMaxParts];
  int n;
  int64_t rows;
  int heads, dv;
  void* o_out;
  float* lse_out;
  int out_kind;  // 0 bf16, 1 fp16, 2 fp32
};

struct CheckParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* used_q;  // optional visible lengths (padded THD)
  const int32_t* used_k;
  int batch, max_q, max_k, total_q, total_k;
  int* status;
};

// Context-parallel all-to-all relayout: sequence shards <-> head shards.
// Sequence side: rank r holds chunks r and 2cp-1-r (chunk = seqlen / 2cp) as
// its local tokens [0, 2*chunk); head side: rank r holds heads
// [r*heads/cp, (r+1)*heads/cp) of every token in sequence order.  Strides are
// in elements {rank, token, head}; the d elements of one (token, head) are
// contiguous.
struct RelayoutParams {
  const uint8_t* src;
  uint8_t* dst;
  int64_t seq_s[3], head_s[3];  // strides of the sequence-side / head-side tensors
  int64_t seqlen;
  int cp, heads, d, elem_bytes;
  int to_heads;  // 1: sequence side -> head side, 0: head side -> sequence side
};

cudaError_t launch_pre(const PreParams& p, bool bf16, int num_sms, cudaStream_t st);
cudaError_t launch_relayout(const RelayoutParams& p, int num_sms, cudaStream_t st);
cudaError_t launch_merge(const MergeParams& p, int num_sms, cudaStream_t st);
cudaError_t launch_check(const CheckParams& p, cudaStream_t st);

}  // namespace attn
