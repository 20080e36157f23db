// small.cu -- the memory-bound kernels of the attention path:
//   * attn_pre_kernel:   D[b,h,i] = sum_c dO[i,h,c] * O[i,h,c] in FP32, stored
//                        with the row's LSE in base 2 as the pair the backward
//                        kernels read (TransformerEngine PR #3699: the backward
//                        helper chain);
//   * attn_merge_kernel: LSE-weighted merge of partial results
//                        (PR #3527: the context-parallel ring correction);
//   * attn_check_kernel: device validation of cu_seqlens (PR #3699: every
//                        execution checks the packed-layout metadata on device);
//   * attn_relayout_kernel: the local data movement of the all-to-all
//                        context-parallel path (PR #3527: after the all-to-all
//                        each rank holds the full sequence for a subset of
//                        heads), sequence shards <-> head shards, bit-preserving.
#include "kcommon.cuh"
#include "small_params.h"

namespace attn {

// ----------------------------------------------------------------- D = rowsum(dO * O)
// Rows are (token, head) pairs.  LPR lanes share a row (each reads 16-byte
// vectors of O and dO, NCH of them), so a warp covers 32/LPR rows per pass
// with every lane busy, and kU passes are unrolled to keep 2*kU*NCH loads in
// flight per lane: the kernel is a pure HBM stream.
template <bool BF16, int LPR, int NCH>
__global__ void __launch_bounds__(256) attn_pre_kernel(const PreParams p) {
  constexpr int kRowsPerPass = 32 / LPR;
  constexpr int kU = 4;
  if (p.status && *(volatile int*)p.status) return;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, l = lane % LPR;
  const int64_t rows = (int64_t)(p.cu_q ? p.total_q : (int64_t)p.batch * p.seqlen_q) * p.hq;
  const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t base = warp_id * (kRowsPerPass * kU); base < rows;
       base += nwarps * (kRowsPerPass * kU)) {
    uint4 ov[kU][NCH], dv[kU][NCH];
    int64_t didx[kU];
    float lsev[kU];  // the row's LSE, loaded with its O / dO vectors
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t r = base + u * kRowsPerPass + sub;
      didx[u] = -1;
      lsev[u] = 0.0f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) ov[u][c] = dv[u][c] = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) {
        // rows < 2^32 (checked at launch): 32-bit division
        const uint32_t r32 = (uint32_t)r;
        const int h = (int)(r32 % (uint32_t)p.hq);
        const uint32_t t = r32 / (uint32_t)p.hq;  // token (dense: b*S + i)
        int b = 0;
        int64_t tok;
        if (p.cu_q) {
          // packed rows are addressed by token alone (D has no batch stride);
          // only a padded layout needs the sequence that owns token t, to
          // leave its gap rows alone
          tok = t;
          if (p.used_q) {
            int lo = 0, hi = p.batch;
            while (hi - lo > 1) {
              const int mid = (lo + hi) >> 1;
              if ((uint32_t)p.cu_q[mid] <= t) lo = mid; else hi = mid;
            }
            b = lo;
            if ((int64_t)t - p.cu_q[b] >= p.used_q[b]) continue;  // a gap row: no D
          }
        } else {
          b = (int)(t / (uint32_t)p.seqlen_q);
          tok = t - (uint32_t)b * (uint32_t)p.seqlen_q;
        }
        const int64_t bb = p.cu_q ? 0 : b;
        const uint4* orow = reinterpret_cast<const uint4*>(
            (const uint16_t*)p.o + bb * p.so_b + tok * p.so_t + (int64_t)h * p.so_h);
        const uint4* drow = reinterpret_cast<const uint4*>(
            (const uint16_t*)p.dout + bb * p.sdo_b + tok * p.sdo_t + (int64_t)h * p.sdo_h);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          ov[u][c] = orow[c * LPR + l];
          dv[u][c] = drow[c * LPR + l];
        }
        didx[u] = (int64_t)b * p.d_sb + (int64_t)h * p.d_sh + tok;
        if (l == 0) lsev[u] = p.lse[(int64_t)b * p.lse_sb + (int64_t)h * p.lse_sh + tok];
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      float acc = 0.0f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const uint16_t* oe = reinterpret_cast<const uint16_t*>(&ov[u][c]);
        const uint16_t* de = reinterpret_cast<const uint16_t*>(&dv[u][c]);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(Pack<BF16>::to_f(oe[e]), Pack<BF16>::to_f(de[e]), acc);
      }
#pragma unroll
      for (int s = LPR / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
      if (l == 0 && didx[u] >= 0) {
        float l2 = lsev[u] * 1.4426950408889634f;
        if (l2 == -INFINITY) l2 = INFINITY;  // keyless row: every key is masked anyway
        p.d[didx[u]] = make_float2(l2, acc);
      }
    }
  }
}

template <bool BF16>
static cudaError_t launch_pre_t(const PreParams& p, unsigned blocks, cudaStream_t st) {
  switch (p.dv) {
    case 64: attn_pre_kernel<BF16, 8, 1><<<blocks, 256, 0, st>>>(p); break;
    case 128: attn_pre_kernel<BF16, 16, 1><<<blocks, 256, 0, st>>>(p); break;
    case 256: attn_pre_kernel<BF16, 32, 1><<<blocks, 256, 0, st>>>(p); break;
    case 512: attn_pre_kernel<BF16, 32, 2><<<blocks, 256, 0, st>>>(p); break;
    default: return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

cudaError_t launch_pre(const PreParams& p, bool bf16, int num_sms, cudaStream_t st) {
  const int64_t rows = (int64_t)(p.cu_q ? p.total_q : (int64_t)p.batch * p.seqlen_q) * p.hq;
  if (rows >= (int64_t(1) << 32)) return cudaErrorNotSupported;
  const int lpr = p.dv >= 256 ? 32 : p.dv / 8;
  const int64_t per_block = 8 * (32 / lpr) * 4;  // 8 warps x rows per pass x unroll
  int64_t blocks = (rows + per_block - 1) / per_block;
  const int64_t cap = (int64_t)num_sms * 8;  // 8 resident blocks per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return bf16 ? launch_pre_t<true>(p, (unsigned)blocks, st) : launch_pre_t<false>(p, (unsigned)blocks, st);
}

// ----------------------------------------------------------------- LSE merge
// One warp per (row, head).  Lane q fetches the LSE of parts q and q + 32 at
// this row (-inf where a part does not cover it); the maximum and the sum of
// exp(LSE_p - max) are warp reductions.  The O rows of the covering parts are
// loaded (16-byte loads, lane = 4 value columns) together with the LSE, eight
// parts at a time, so a row costs one round trip to memory rather than two;
// each part's weight exp(LSE_p - LSE) is broadcast by a shuffle, and a part
// whose weight is 0 (LSE = -inf, or not covering the row) is left out of the
// sum, so a NaN in its O never reaches the result.
constexpr int kMergeGroup = 8;

__global__ void __launch_bounds__(256, 4) attn_merge_kernel(const __grid_constant__ MergeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t total = p.rows * p.heads;
  const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t w = warp_id; w < total; w += nwarps) {
    const int64_t r = w / p.heads;
    const int h = (int)(w % p.heads);
    float l[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int q = lane + 32 * u;
      if (q < p.n) {
        const int64_t x = r - p.row0[q];
        if (x >= 0 && x < p.nrows[q]) l[u] = p.lse[q][(int64_t)h * p.nrows[q] + x];
      }
    }
    float lse = -INFINITY, a0 = 0.0f, a1 = 0.0f;  // a0/a1: weights of parts lane, lane + 32
    bool have_lse = false;
    for (int c0 = 0; c0 < p.dv; c0 += 128) {
      const int c = c0 + lane * 4;
      const bool act = c < p.dv;
      // O of every covering part, issued before the LSE values are used
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int g0 = 0; g0 < p.n; g0 += kMergeGroup) {
        float4 v[kMergeGroup];
#pragma unroll
        for (int t = 0; t < kMergeGroup; ++t) {
          const int q = g0 + t;
          v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (q < p.n && act) {
            const int64_t x = r - p.row0[q];
            if (x >= 0 && x < p.nrows[q])
              v[t] = *reinterpret_cast<const float4*>(p.o[q] + (x * p.heads + h) * (int64_t)p.dv + c);
          }
        }
        if (!have_lse) {  // the weights, once per row (the LSE loads are in flight too)
          float m = fmaxf(l[0], l[1]);
#pragma unroll
          for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          float sum = (l[0] == -INFINITY ? 0.0f : __expf(l[0] - m)) +
                      (l[1] == -INFINITY ? 0.0f : __expf(l[1] - m));
#pragma unroll
          for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
          lse = (m == -INFINITY) ? -INFINITY : m + __logf(sum);
          a0 = l[0] == -INFINITY ? 0.0f : __expf(l[0] - lse);
          a1 = l[1] == -INFINITY ? 0.0f : __expf(l[1] - lse);
          have_lse = true;
        }
#pragma unroll
        for (int t = 0; t < kMergeGroup; ++t) {
          const int q = g0 + t;
          const float aq = __shfl_sync(0xffffffffu, q < 32 ? a0 : a1, q & 31);
          if (aq != 0.0f) {  // warp-uniform; -inf parts (and non-covering ones) skipped
            acc.x = fmaf(aq, v[t].x, acc.x);
            acc.y = fmaf(aq, v[t].y, acc.y);
            acc.z = fmaf(aq, v[t].z, acc.z);
            acc.w = fmaf(aq, v[t].w, acc.w);
          }
        }
      }
      if (c0 == 0 && lane == 0) p.lse_out[(int64_t)h * p.rows + r] = lse;
      if (!act) continue;
      const int64_t off = (r * p.heads + h) * (int64_t)p.dv + c;
      if (p.out_kind == 2) {
        *reinterpret_cast<float4*>((float*)p.o_out + off) = acc;
      } else {
        uint2 pk;
        if (p.out_kind == 0) {
          pk.x = Pack<true>::two(acc.x, acc.y);
          pk.y = Pack<true>::two(acc.z, acc.w);
        } else {
          pk.x = Pack<false>::two(acc.x, acc.y);
          pk.y = Pack<false>::two(acc.z, acc.w);
        }
        *reinterpret_cast<uint2*>((uint16_t*)p.o_out + off) = pk;
      }
    }
  }
}

cudaError_t launch_merge(const MergeParams& p, int num_sms, cudaStream_t st) {
  const int64_t total = p.rows * p.heads;
  int64_t blocks = (total + 7) / 8;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  attn_merge_kernel<<<(unsigned)blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

// ----------------------------------------------------------------- cu_seqlens check
// Single block.  Sets *status = DEV_BAD_SEQLENS unless, for both q and k:
// cu[0] == 0, cu non-decreasing, every length <= the declared maximum and
// cu[batch] == the declared total.
__global__ void __launch_bounds__(256) attn_check_kernel(const CheckParams p) {
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  int local = 0;
  for (int b = threadIdx.x; b < p.batch; b += blockDim.x) {
    const int lq = p.cu_q[b + 1] - p.cu_q[b];
    const int lk = p.cu_k[b + 1] - p.cu_k[b];
    if (lq < 0 || lq > p.max_q || lk < 0 || lk > p.max_k) local = 1;
    // padded layout: the visible length fits in the sequence's padded extent
    if (p.used_q && (p.used_q[b] < 0 || p.used_q[b] > lq)) local = 1;
    if (p.used_k && (p.used_k[b] < 0 || p.used_k[b] > lk)) local = 1;
  }
  if (threadIdx.x == 0) {
    if (p.cu_q[0] != 0 || p.cu_k[0] != 0) local = 1;
    if (p.cu_q[p.batch] != p.total_q || p.cu_k[p.batch] != p.total_k) local = 1;
  }
  if (local) atomicOr(&bad, 1);
  __syncthreads();
  if (threadIdx.x == 0 && bad) atomicExch(p.status, DEV_BAD_SEQLENS);
}

cudaError_t launch_check(const CheckParams& p, cudaStream_t st) {
  attn_check_kernel<<<1, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace attn

namespace attn {

// ----------------------------------------------------------------- CP relayout
// Rows are (token, head) pairs of d elements.  VEC: 16-byte vectors (d *
// elem_bytes a multiple of 16 and 16-byte-aligned rows): a warp treats its
// rows' vectors as one flat list, so every lane is busy whatever d is, and
// keeps kU vectors in flight per lane; otherwise single elements of
// elem_bytes.  Pure copy: every bit is preserved.
// IDX: the index type of the row arithmetic (32-bit when every index fits).
template <typename IDX>
__device__ __forceinline__ void relayout_row_addr(const RelayoutParams& p, IDX r,
                                                  const uint8_t*& src, uint8_t*& dst) {
  const IDX chunk = (IDX)(p.seqlen / (2 * p.cp));
  const int hpr = p.heads / p.cp;  // heads per rank on the head side
  const IDX t = r / (IDX)p.heads;  // global token
  const int h = (int)(r - t * (IDX)p.heads);
  const IDX ch = t / chunk, u = t - ch * chunk;
  // sequence side: owner rank and local token of global token t
  const int64_t srank = (int64_t)ch < p.cp ? (int64_t)ch : 2 * p.cp - 1 - (int64_t)ch;
  const int64_t stok = (int64_t)ch < p.cp ? (int64_t)u : (int64_t)(chunk + u);
  const int64_t seq_off = srank * p.seq_s[0] + stok * p.seq_s[1] + (int64_t)h * p.seq_s[2];
  const int64_t head_off = (int64_t)(h / hpr) * p.head_s[0] + (int64_t)t * p.head_s[1] +
                           (int64_t)(h % hpr) * p.head_s[2];
  src = p.src + (p.to_heads ? seq_off : head_off) * p.elem_bytes;
  dst = p.dst + (p.to_heads ? head_off : seq_off) * p.elem_bytes;
}

// VEC requires rows * (d * elem_bytes / 16) < 2^32 (checked at launch): its
// index arithmetic is 32-bit.
template <bool VEC>
__global__ void __launch_bounds__(256) attn_relayout_kernel(const RelayoutParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = p.seqlen * p.heads;
  const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int row_bytes = p.d * p.elem_bytes;
  if (VEC) {
    constexpr int kU = 4;
    const uint32_t vpr = (uint32_t)row_bytes / 16;  // vectors per row
    const uint32_t nvec = (uint32_t)rows * vpr;      // all vectors, row-major
    const uint32_t per_warp = 32 * kU;
    for (int64_t base = warp_id * per_warp; base < nvec; base += nwarps * per_warp) {
      uint4 val[kU];
      uint8_t* dsts[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t vi64 = base + u * 32 + lane;
        dsts[u] = nullptr;
        if (vi64 < nvec) {
          const uint32_t vi = (uint32_t)vi64;
          const uint32_t r = vi / vpr;
          const int c = (int)(vi - r * vpr) * 16;
          const uint8_t* src;
          uint8_t* dst;
          relayout_row_addr<uint32_t>(p, r, src, dst);
          val[u] = *reinterpret_cast<const uint4*>(src + c);
          dsts[u] = dst + c;
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (dsts[u]) *reinterpret_cast<uint4*>(dsts[u]) = val[u];
    }
  } else {
    for (int64_t r = warp_id; r < rows; r += nwarps) {
      const uint8_t* src;
      uint8_t* dst;
      relayout_row_addr<int64_t>(p, r, src, dst);
      for (int c = lane * p.elem_bytes; c < row_bytes; c += 32 * p.elem_bytes) {
        if (p.elem_bytes == 4)
          *reinterpret_cast<uint32_t*>(dst + c) = *reinterpret_cast<const uint32_t*>(src + c);
        else
          *reinterpret_cast<uint16_t*>(dst + c) = *reinterpret_cast<const uint16_t*>(src + c);
      }
    }
  }
}

cudaError_t launch_relayout(const RelayoutParams& p, int num_sms, cudaStream_t st) {
  const int64_t rows = p.seqlen * p.heads;
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = (int64_t)num_sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  bool vec = (p.d * p.elem_bytes) % 16 == 0 && ((uintptr_t)p.src % 16) == 0 &&
             ((uintptr_t)p.dst % 16) == 0;
  for (int i = 0; i < 3; ++i)
    vec = vec && (p.seq_s[i] * p.elem_bytes) % 16 == 0 && (p.head_s[i] * p.elem_bytes) % 16 == 0;
  vec = vec && rows * (p.d * p.elem_bytes / 16) < (int64_t(1) << 32);
  if (vec)
    attn_relayout_kernel<true><<<(unsigned)blocks, 256, 0, st>>>(p);
  else
    attn_relayout_kernel<false><<<(unsigned)blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
