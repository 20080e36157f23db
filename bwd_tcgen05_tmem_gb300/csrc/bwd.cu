// bwd.cu -- backward dispatch: D preprocess, then the query-stationary dQ
// kernel and the key/value-stationary dK/dV kernel(s), all on one stream.
// On the dS path (ds_backward) the dK/dV kernel also writes dS and the dQ
// stage is the GEMM of bwd_dq_ds.cu over it, so dK/dV runs first.  Head dims
// above 256 go to the materialising path of bwd_wide.cu.
#include "bwd.h"
#include "small_params.h"

namespace attn {

cudaError_t launch_dq(const DqParams& p, int dqk, int dv, bool bf16, bool gf32, int num_sms,
                      cudaStream_t st);
int dq_block_kv(int dqk, int dv);
int dkv_plan(int dqk, int dv, int* bq, int* mode);
cudaError_t launch_dkv(const DkvParams& p, int dqk, int dv, int mode, bool bf16, bool gf32,
                       cudaStream_t st);

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t st, int stages, int* n_launches) {
  *n_launches = 0;
  if (a.wide) return launch_bwd_wide(a, st, stages, n_launches);
  const bool has_q = (a.thd ? a.total_q : a.batch * a.seqlen_q) > 0;
  const bool has_k = (a.thd ? a.total_k : a.batch * a.seqlen_k) > 0;
  int bq[2], mode[2];
  const int nplan = dkv_plan(a.dqk, a.dv, bq, mode);
  if (nplan == 0) return cudaErrorNotSupported;
  cudaError_t e;
  if (has_q && (stages & 1)) {
    PreParams pp;
    pp.o = a.o;
    pp.dout = a.dout;
    pp.d = a.d;
    pp.lse = a.lse;
    pp.lse_sb = a.lse_sb;
    pp.lse_sh = a.lse_sh;
    pp.cu_q = a.thd ? a.geo.cu_q : nullptr;
    pp.used_q = a.thd ? a.geo.used_q : nullptr;
    pp.so_b = a.so[0]; pp.so_t = a.so[1]; pp.so_h = a.so[2];
    pp.sdo_b = a.sdo[0]; pp.sdo_t = a.sdo[1]; pp.sdo_h = a.sdo[2];
    pp.d_sb = a.d_sb;
    pp.d_sh = a.d_sh;
    pp.batch = a.batch;
    pp.seqlen_q = a.seqlen_q;
    pp.total_q = a.total_q;
    pp.hq = a.hq;
    pp.dv = a.dv;
    pp.status = a.status;
    if ((e = launch_pre(pp, a.bf16, a.num_sms, st)) != cudaSuccess) return e;
    ++*n_launches;
  }
  auto run_dq = [&]() -> cudaError_t {
    if (a.ds && has_q && (stages & 2)) {
      // dS path: dQ is a GEMM over the dS blocks the dK/dV stage wrote
      DqDsParams qp;
      memset(&qp, 0, sizeof(qp));
      qp.tm_k = has_k ? a.tm_k128 : a.tm_q128;
      qp.ok = has_k ? a.ok : a.oq;
      qp.geo = a.geo;
      qp.plan = a.ds_plan;
      qp.blocks = a.ds_blocks;
      qp.cap = a.ds_cap;
      qp.dq = a.dq;
      qp.sdq_b = a.sdq[0]; qp.sdq_t = a.sdq[1]; qp.sdq_h = a.sdq[2];
      qp.accum = a.accum;
      qp.batch = a.batch;
      qp.hq = a.hq;
      qp.hkv = a.hkv;
      qp.n_qtiles = (a.seqlen_q + 127) / 128;
      qp.scale = a.scale;
      qp.status = a.status;
      qp.dbg = a.dbg_dq;
      qp.counter = a.queue_counter;
      if (qp.n_qtiles > 65535 || a.batch > 65535 || a.hq > 65535) return cudaErrorInvalidValue;
      // the work-queue counter starts at zero for every launch
      if ((e = cudaMemsetAsync(qp.counter, 0, sizeof(int), st)) != cudaSuccess) return e;
      if ((e = launch_dq_ds(qp, a.dqk, a.bf16, a.g_f32, a.num_sms, st)) != cudaSuccess) return e;
      ++*n_launches;
    } else if (has_q && (stages & 2)) {
      DqParams dq;
      const int bkv = dq_block_kv(a.dqk, a.dv);
      dq.tm_q = a.tm_q128;
      dq.tm_do = a.tm_do128;
      dq.tm_k = has_k ? (bkv == 128 ? a.tm_k128 : a.tm_k64) : a.tm_q128;
      dq.tm_v = has_k ? (bkv == 128 ? a.tm_v128 : a.tm_v64) : a.tm_q128;
      dq.oq = a.oq;
      dq.odo = a.odo;
      dq.ok = has_k ? a.ok : a.oq;
      dq.ov = has_k ? a.ov : a.oq;
      dq.geo = a.geo;
      dq.d = a.d;
      dq.d_sb = a.d_sb;
      dq.d_sh = a.d_sh;
      dq.dq = a.dq;
      dq.sdq_b = a.sdq[0]; dq.sdq_t = a.sdq[1]; dq.sdq_h = a.sdq[2];
      dq.accum = a.accum;
      dq.batch = a.batch;
      dq.hq = a.hq;
      dq.hkv = a.hkv;
      dq.n_qtiles = (a.seqlen_q + 127) / 128;
      dq.scale = a.scale;
      dq.scale_log2 = a.scale_log2;
      dq.status = a.status;
      dq.dbg = a.dbg_dq;
      dq.counter = a.queue_counter;
      if (dq.n_qtiles > 65535 || a.batch > 65535 || a.hq > 65535) return cudaErrorInvalidValue;
      // the work-queue counter starts at zero for every launch
      if ((e = cudaMemsetAsync(dq.counter, 0, sizeof(int), st)) != cudaSuccess) return e;
      if ((e = launch_dq(dq, a.dqk, a.dv, a.bf16, a.g_f32, a.num_sms, st)) != cudaSuccess) return e;
      ++*n_launches;
    }
    return cudaSuccess;
  };
  auto run_dkv = [&]() -> cudaError_t {
    if (a.ds && (stages & 4)) {
      // the block plan belongs to the stage that writes the blocks (it depends
      // on the key side and the mask); the dq stage reads it
      WidePlanParams pl;
      pl.geo = a.geo;
      pl.plan = a.ds_plan;
      pl.cap = a.ds_cap;
      pl.batch = a.batch;
      pl.hq = a.hq;
      pl.status = a.status;
      if ((e = launch_wide_plan(pl, st)) != cudaSuccess) return e;
      ++*n_launches;
    }
    if (has_k && (stages & 4)) {
      for (int i = 0; i < nplan; ++i) {
        DkvParams kp;
        kp.tm_k = a.tm_k128;
        kp.tm_v = a.tm_v128;
        kp.tm_q = has_q ? (bq[i] == 128 ? a.tm_q128 : a.tm_q64) : a.tm_k128;
        kp.tm_do = has_q ? (bq[i] == 128 ? a.tm_do128 : a.tm_do64) : a.tm_k128;
        kp.ok = a.ok;
        kp.ov = a.ov;
        kp.oq = has_q ? a.oq : a.ok;
        kp.odo = has_q ? a.odo : a.ok;
        kp.geo = a.geo;
        kp.d = a.d;
        kp.d_sb = a.d_sb;
        kp.d_sh = a.d_sh;
        kp.dk = a.dk;
        kp.dv = a.dvp;
        kp.sdk_b = a.sdk[0]; kp.sdk_t = a.sdk[1]; kp.sdk_h = a.sdk[2];
        kp.sdv_b = a.sdv[0]; kp.sdv_t = a.sdv[1]; kp.sdv_h = a.sdv[2];
        kp.accum = a.accum;
        kp.batch = a.batch;
        kp.hq = a.hq;
        kp.hkv = a.hkv;
        kp.n_ktiles = (a.seqlen_k + 127) / 128;
        kp.scale = a.scale;
        kp.scale_log2 = a.scale_log2;
        kp.status = a.status;
        kp.dbg = a.dbg_dkdv;
        kp.ds = (a.ds && (mode[i] & 2)) ? a.ds_blocks : nullptr;
        kp.plan = a.ds_plan;
        kp.cap = a.ds_cap;
        if (kp.n_ktiles > 65535 || a.batch > 65535) return cudaErrorInvalidValue;
        if ((e = launch_dkv(kp, a.dqk, a.dv, mode[i], a.bf16, a.g_f32, st)) != cudaSuccess) return e;
        ++*n_launches;
      }
    }
    return cudaSuccess;
  };
  // dS path: the dK/dV stage writes the dS blocks that the dQ GEMM reads
  if (a.ds) {
    if ((e = run_dkv()) != cudaSuccess) return e;
    return run_dq();
  }
  if ((e = run_dq()) != cudaSuccess) return e;
  return run_dkv();
}

}  // namespace attn
