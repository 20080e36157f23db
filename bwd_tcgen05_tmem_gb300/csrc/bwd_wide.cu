// bwd_wide.cu -- backward for head dims above 256, and for head dim 256 when
// its score tiles fit the cap of wide_backward() (tcgen05 / TMEM / TMA).
//
// At head dim 512 one SM cannot hold what the fused kernels keep on chip:
// the dK and dV accumulators of a 128-key tile need 2 x 512 TMEM columns
// (the SM has 512), and K and V of that tile need 256 KiB of shared memory
// (it has 227 KiB).  So this path materialises P and dS in HBM, as 16-bit
// tiles already laid out in their 128-byte-swizzled shared-memory image, and
// splits the chain of the backward (TransformerEngine PR #3527: the d512
// backward; PR #3510 backward chain) into three kernels:
//
//   scores  query-stationary, per 128-row query tile and visible 128-key
//           block:
//             S  = Q K^T      (SS MMA, Q resident in shared memory)
//             dP = dO V^T     (TS MMA, dO resident in TMEM as operand A)
//             P  = exp(scale S - LSE),  dS = P (dP - D)   (softmax warps)
//           and stores P and dS (16-bit) into the block;
//   dQ      query-stationary GEMM:  dQ = scale sum_kb dS_kb K_kb;
//   dK/dV   key-stationary GEMMs:   dV = sum P^T dO,  dK = scale sum dS^T Q,
//           over every visible query tile and every query head of the group.
//
// Each of the five contractions runs once (no recompute), on tcgen05 with an
// FP32 TMEM accumulator; every element of dQ/dK/dV is written by one CTA, in a
// fixed order, so the result is bitwise reproducible.  P and dS are rounded
// to the input type before their contractions, as in the fused kernels.
//
// Workspace blocks: a per-sequence prefix (the planning kernel) gives block
// (b, h, qt, kb) the index  hq*plan[b] + h*T_b + rowprefix_b(qt) + kb - kb0(qt),
// T_b = plan[b+1] - plan[b], rowprefix_b(qt) = blocks of the query tiles
// before qt.  Every kernel checks the index range against the capacity.
#include "bwd.h"
#include "small_params.h"

namespace attn {

// ------------------------------------------------------------------ planning
// One CTA: per-sequence block counts, their exclusive prefix, capacity check.
__global__ void __launch_bounds__(256) attn_wide_plan_kernel(const WidePlanParams p) {
  __shared__ long long part[256];
  __shared__ int skip;
  if (threadIdx.x == 0) skip = status_set(p.status) ? 1 : 0;
  __syncthreads();
  if (skip) return;
  long long carry = 0;
  for (int b0 = 0; b0 < p.batch; b0 += 256) {
    const int b = b0 + (int)threadIdx.x;
    long long t = 0;
    if (b < p.batch) {
      const Seq s = load_seq(p.geo, b);
      const int nqt = s.lq > 0 ? (s.lq + 127) / 128 : 0;
      int kb0;
      for (int qt = 0; qt < nqt; ++qt) t += wide_blocks_of_qtile(s, qt, kb0);
    }
    part[threadIdx.x] = t;
    __syncthreads();
    for (int o = 1; o < 256; o <<= 1) {  // inclusive scan
      const long long v = threadIdx.x >= (unsigned)o ? part[threadIdx.x - o] : 0ll;
      __syncthreads();
      part[threadIdx.x] += v;
      __syncthreads();
    }
    if (b < p.batch) p.plan[b] = carry + part[threadIdx.x] - t;
    carry += part[255];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.plan[p.batch] = carry;
    if (carry * (long long)p.hq > p.cap) raise_status(p.status, DEV_WORKSPACE);
  }
}

cudaError_t launch_wide_plan(const WidePlanParams& p, cudaStream_t st) {
  attn_wide_plan_kernel<<<1, 256, 0, st>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ scores
// Per visible 128-key block: S (N = 128, SS) and dP (N = 128, TS).  Each score
// MMA covers the whole block: one thread needs about 60 cycles to issue a
// tcgen05.mma, so an M = 128 MMA with N = 64 (32 cycles of tensor work) would
// leave the pipe idle half the time.  TMEM holds one S, one dP and dO; S and
// dP have their own full / free barriers, so S of block n+1 runs while the
// softmax waits for dP of block n, and dP of block n+1 while it computes P.
// Warp roles (384 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer, warps 4..11 softmax (one query row per TMEM lane, the two
// warpgroups take the two 64-key halves of a block).
template <int DQK, int DV>
struct WideScoresCfg {
  static constexpr int kQCh = DQK / 64;
  static constexpr int kVCh = DV / 64;
  static constexpr int kChunk = kSlotBytes;  // 128 key rows x 64 columns
  static constexpr int kQBytes = kQCh * kSlotBytes;
  static constexpr int kRingRaw = (232448 - 2048 - kQBytes) / kChunk;
  static constexpr int kRing = kRingRaw > 12 ? 12 : kRingRaw;
  static constexpr int kSmem = kQBytes + kRing * kChunk + 1024;
  static constexpr int kTS = 0, kTdP = 128, kTdO = 256;  // TMEM columns
  static_assert(kTdO + DV / 2 <= 512, "TMEM budget");
  static_assert(kRing >= 4, "ring");
};

template <int DQK, int DV, bool BF16>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_wide_scores_kernel(const __grid_constant__ WideScoresParams p) {
  using C = WideScoresCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + C::kQBytes;

  __shared__ uint64_t rfull[C::kRing], rempty[C::kRing];
  __shared__ uint64_t q_bar, do_ready, s_full, dp_full, s_free, dp_free, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag, skip_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool tmaj = tile_major(p.n_qtiles);  // grid order, heaviest tiles first
  const int h = tmaj ? blockIdx.y : blockIdx.x;
  const int qt = p.n_qtiles - 1 - (int)(tmaj ? blockIdx.x : blockIdx.y);
  const int b = blockIdx.z;
  const int tb = p.geo.cu_q ? 0 : b;
  const int g = h / (p.hq / p.hkv);

  const Seq sq = load_seq(p.geo, b);
  const int q0 = qt * 128;
  if (q0 >= sq.lq) return;
  int kb0 = 0;
  const int n_kb = wide_blocks_of_qtile(sq, qt, kb0);
  if (n_kb == 0) return;  // nothing visible: no block (the dQ kernel writes zeros)
  if (threadIdx.x == 0) skip_sh = status_set(p.status) ? 1 : 0;
  __syncthreads();
  if (skip_sh) return;

  const unsigned long long lim = wait_limit(p.dbg);
  const int drop = dropped_load(p.dbg);
  Abort ab{&abort_flag, p.status, lim};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < C::kRing; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], 1);
    }
    mbar_init(&q_bar, 1);
    mbar_init(&do_ready, 256);
    mbar_init(&s_full, 1);
    mbar_init(&dp_full, 1);
    mbar_init(&s_free, 256);
    mbar_init(&dp_free, 256);
    mbar_init(&drain_bar, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Q once; then per block its K chunks and V chunks (ring)
    int c1, c2, c3;
    map_coords(p.oq, 0, h, sq.q_start + q0, tb, c1, c2, c3);
    if (elect_sync()) {
      mbar_arrive_tx(&q_bar, C::kQBytes);
      for (int c = 0; c < C::kQCh; ++c)
        tma_load_4d(sQ + c * kSlotBytes, &p.tm_q, &q_bar, c * 64, c1, c2, c3);
    }
    __syncwarp();
    uint32_t cnt = 0;
    bool ok = true;
    for (int n = 0; n < n_kb && ok; ++n) {
      const int krow = sq.k_start + (kb0 + n) * 128;
      int k1, k2, k3, v1, v2, v3;
      map_coords(p.ok, 0, g, krow, tb, k1, k2, k3);
      map_coords(p.ov, 0, g, krow, tb, v1, v2, v3);
#pragma unroll
      for (int c = 0; c < C::kQCh + C::kVCh; ++c) {
        const uint32_t slot = cnt % C::kRing;
        if (!mbar_wait_warp(&rempty[slot], ((cnt / C::kRing) & 1u) ^ 1u, ab)) {
          ok = false;
          break;
        }
        if ((int)cnt != drop && elect_sync()) {  // drop: test-only injected missing load
          mbar_arrive_tx(&rfull[slot], C::kChunk);
          if (c < C::kQCh)
            tma_load_4d(sRing + slot * C::kChunk, &p.tm_k, &rfull[slot], c * 64, k1, k2, k3);
          else
            tma_load_4d(sRing + slot * C::kChunk, &p.tm_v, &rfull[slot], (c - C::kQCh) * 64, v1,
                        v2, v3);
        }
        __syncwarp();
        ++cnt;
      }
    }
    // let the copies in flight land before the CTA exits
    mbar_wait_quiet(&q_bar, 0, lim);
    const uint32_t first = cnt > (uint32_t)C::kRing ? cnt - C::kRing : 0u;
    for (uint32_t c = first; c < cnt; ++c)
      mbar_wait_quiet(&rfull[c % C::kRing], (c / C::kRing) & 1u, lim);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = make_idesc(128, 128, BF16, false, false);
    const uint64_t qdesc = make_sdesc(smem_u32(sQ), 16, 1024);
    const uint64_t rdesc = make_sdesc(smem_u32(sRing), 16, 1024);
    uint32_t cnt = 0;
    bool ok = mbar_wait_warp(&q_bar, 0, ab) && mbar_wait_warp(&do_ready, 0, ab);
    tc_fence_after();
    // next ring chunk (K or V rows of the block), in load order
    auto chunk = [&]() -> uint64_t {
      const uint32_t slot = cnt % C::kRing;
      if (!mbar_wait_warp(&rfull[slot], (cnt / C::kRing) & 1u, ab)) {
        ok = false;
        return 0ull;
      }
      tc_fence_after();
      return rdesc + (uint64_t)((slot * C::kChunk) >> 4);
    };
    for (int n = 0; n < n_kb && ok; ++n) {
      // S of block n-1 must be in the softmax's registers before S is overwritten
      if (n > 0 && !mbar_wait_warp(&s_free, (n - 1) & 1u, ab)) break;
      tc_fence_after();
      for (int c = 0; c < C::kQCh && ok; ++c) {  // S += Q_c K_c^T
        const uint64_t kd = chunk();
        if (!ok) break;
        const uint64_t qa = qdesc + (uint64_t)(c * (kSlotBytes >> 4));
        if (elect_sync()) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + C::kTS, qa + 2 * k, kd + 2 * k, idesc, (c | k) ? 1u : 0u);
          mma_commit(&rempty[cnt % C::kRing]);
          if (c == C::kQCh - 1) mma_commit(&s_full);
        }
        __syncwarp();
        ++cnt;
      }
      if (!ok) break;
      if (n > 0 && !mbar_wait_warp(&dp_free, (n - 1) & 1u, ab)) break;
      tc_fence_after();
      for (int c = 0; c < C::kVCh && ok; ++c) {  // dP += dO_c V_c^T, dO from TMEM
        const uint64_t vd = chunk();
        if (!ok) break;
        if (elect_sync()) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + C::kTdP, tmem + C::kTdO + c * 32 + k * 8, vd + 2 * k, idesc,
                   (c | k) ? 1u : 0u);
          mma_commit(&rempty[cnt % C::kRing]);
          if (c == C::kVCh - 1) mma_commit(&dp_full);
        }
        __syncwarp();
        ++cnt;
      }
    }
    if (elect_sync()) {
      mma_commit(&drain_bar);
      mbar_wait_quiet(&drain_bar, 0, lim);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / dS
    const int wq = (warp - 4) & 3;  // TMEM lane quadrant
    const int wg = (warp - 4) >> 2;  // 64-key half of a block = its P/dS sub-tile
    const int r = wq * 32 + lane;
    const int i = q0 + r;
    const bool valid = i < sq.lq;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int64_t tok = (int64_t)sq.q_start + i;
    float l2 = INFINITY, dd = 0.0f;  // rows past the end: P = dS = 0
    if (valid) {  // LSE * log2 e (+inf for a keyless row) and D
      const float2 st = p.d[(int64_t)b * p.d_sb + (int64_t)h * p.d_sh + tok];
      l2 = st.x;
      dd = st.y;
    }
    // dO row (this warpgroup's half of the columns) into TMEM
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          (const char*)p.dout +
          ((int64_t)tb * p.sdo_b + tok * p.sdo_t + (int64_t)h * p.sdo_h + wg * (DV / 2)) * 2);
#pragma unroll
      for (int c = 0; c < DV / 64; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint4 v = valid ? src[c * 4 + t] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * t + 0] = v.x;
          w[4 * t + 1] = v.y;
          w[4 * t + 2] = v.z;
          w[4 * t + 3] = v.w;
        }
        tmem_st16(tmem + lane_off + C::kTdO + wg * (DV / 4) + c * 16, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&do_ready);
    }
    // keys visible from row i
    long long vlo = (long long)i + sq.off - sq.L;
    if (vlo < 0) vlo = 0;
    long long vhi = (long long)i + sq.off + sq.R;
    if (vhi > sq.lk - 1) vhi = sq.lk - 1;
    const long long T_b = p.plan[b + 1] - p.plan[b];
    const long long first = (long long)p.hq * p.plan[b] + (long long)h * T_b + blocks_row_prefix(sq, qt);
    bool ok = first >= 0 && first + n_kb <= p.cap;
    if (!ok) {  // inconsistent plan: stop every role of the CTA
      if (r == 0 && wg == 0) raise_status(p.status, DEV_WORKSPACE);
      *(volatile int*)&abort_flag = 1;
    }
    uint8_t* blk0 = p.blocks + (size_t)(ok ? first : 0) * kWideBlock;
    const float sl2 = p.scale_log2;
    const int sw = r & 7;  // 128-byte swizzle phase of row r
    for (int n = 0; n < n_kb && ok; ++n) {
      if (!mbar_wait_warp(&s_full, n & 1u, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float e[64];
      {
        uint32_t sa[32], sb[32];  // S columns 0..31 and 32..63 of this half
        tmem_ld32(tmem + lane_off + C::kTS + 64 * wg, sa);
        tmem_ld32(tmem + lane_off + C::kTS + 64 * wg + 32, sb);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&s_free);
        const long long k0 = (long long)(kb0 + n) * 128 + 64 * wg;
        const long long lo = vlo - k0, hi = vhi - k0;
        const bool full = lo <= 0 && hi >= 63;
#pragma unroll
        for (int t = 0; t < 64; ++t) {
          float x = ex2(fmaf(__uint_as_float(t < 32 ? sa[t] : sb[t - 32]), sl2, -l2));
          if (!full && (t < lo || t > hi)) x = 0.0f;
          e[t] = x;
        }
      }
      uint8_t* prow = blk0 + (size_t)n * kWideBlock + wg * kWideTile + r * 128;
      uint8_t* drow = prow + 2 * kWideTile;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const int pc = (cc ^ sw) * 16;
        const float* x = e + 8 * cc;
        *reinterpret_cast<uint4*>(prow + pc) =
            make_uint4(Pack<BF16>::two(x[0], x[1]), Pack<BF16>::two(x[2], x[3]),
                       Pack<BF16>::two(x[4], x[5]), Pack<BF16>::two(x[6], x[7]));
      }
      if (!mbar_wait_warp(&dp_full, n & 1u, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t pa[32], pb[32];  // dP columns 0..31 and 32..63 of this half
      tmem_ld32(tmem + lane_off + C::kTdP + 64 * wg, pa);
      tmem_ld32(tmem + lane_off + C::kTdP + 64 * wg + 32, pb);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&dp_free);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const int pc = (cc ^ sw) * 16;
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int c = 8 * cc + 2 * t;
          const float d0 = __uint_as_float(c < 32 ? pa[c] : pb[c - 32]);
          const float d1 = __uint_as_float(c + 1 < 32 ? pa[c + 1] : pb[c - 31]);
          w[t] = Pack<BF16>::two(e[c] * (d0 - dd), e[c + 1] * (d1 - dd));
        }
        *reinterpret_cast<uint4*>(drow + pc) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ GEMMs
// acc[128 x D] = sum over steps of A_s[128 x 64] B_s[64 x D]
//   KIND 0 (dQ, per query tile):  A = dS sub-tile (K-major: rows = queries),
//                                 B = 64 key rows of K (MN-major)
//   KIND 1 (dV / dK, per key tile): A = P^T / dS^T: 64 query rows of both
//                                 sub-tiles (MN-major: keys contiguous),
//                                 B = 64 query rows of dO / Q (MN-major)
// B arrives as quads of four 64-column chunks (N = 256 per MMA).
template <int D>
struct WideAccCfg {
  static constexpr int kNH = D / 256;     // MMAs per K-step (N = 256 each)
  static constexpr int kChunk = 64 * 128;  // 64 rows x 64 columns
  static constexpr int kQuad = 4 * kChunk;
  static constexpr int kA = kWideTile;     // A of one step
  static constexpr int kNA = 3;
  static constexpr int kNB = 5;
  static constexpr int kSmem = kNA * kA + kNB * kQuad + 1024;
  static_assert(D % 256 == 0 && D <= 512, "accumulator width");
  static_assert(kSmem <= 232448 - 1024, "shared memory");
};

template <int D, int KIND, bool BF16, bool G_F32>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_wide_acc_kernel(const __grid_constant__ WideAccParams p) {
  using C = WideAccCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::kNA * C::kA;

  __shared__ uint64_t afull[C::kNA], aempty[C::kNA], bfull[C::kNB], bempty[C::kNB];
  __shared__ uint64_t acc_done, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag, skip_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = p.hq / p.hkv;
  // (tile, head) in the grid order of tile_major(), heaviest tiles first:
  // KIND 0 query tile and query head, KIND 1 key tile and kv head with
  // z = 2 * sequence + (0: dV, 1: dK)
  const bool tmaj = tile_major(p.n_tiles);
  const int hx = tmaj ? blockIdx.y : blockIdx.x;
  const int tx = tmaj ? blockIdx.x : blockIdx.y;
  const int tile = KIND == 0 ? p.n_tiles - 1 - tx : tx;
  const int b = KIND == 0 ? (int)blockIdx.z : (int)(blockIdx.z >> 1);
  const int which = KIND == 0 ? 0 : (int)(blockIdx.z & 1);
  const int tb = p.geo.cu_q ? 0 : b;

  const Seq sq = load_seq(p.geo, b);
  const int r0 = tile * 128;
  if (r0 >= (KIND == 0 ? sq.lq : sq.lk)) return;
  // steps
  int kb0 = 0, n_kb = 0, qt0 = 0, n_qt = 0;
  if (KIND == 0) {
    n_kb = wide_blocks_of_qtile(sq, tile, kb0);
  } else {
    long long i0, i1;
    query_range(sq, r0, min(r0 + 128, sq.lk) - 1, i0, i1);
    if (i1 >= i0) {
      qt0 = (int)(i0 / 128);
      n_qt = (int)(i1 / 128) - qt0 + 1;
    }
  }
  const int n_steps = KIND == 0 ? 2 * n_kb : 2 * n_qt * grp;
  if (threadIdx.x == 0) skip_sh = status_set(p.status) ? 1 : 0;
  __syncthreads();
  if (skip_sh) return;

  const unsigned long long lim = wait_limit(p.dbg);
  const int drop = dropped_load(p.dbg);
  Abort ab{&abort_flag, p.status, lim};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < C::kNA; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&aempty[i], 1);
    }
    for (int i = 0; i < C::kNB; ++i) {
      mbar_init(&bfull[i], 1);
      mbar_init(&bempty[i], 1);
    }
    mbar_init(&acc_done, 1);
    mbar_init(&drain_bar, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const long long T_b = p.plan[b + 1] - p.plan[b];
    const long long pre0 = blocks_row_prefix(sq, KIND == 0 ? tile : qt0);  // whole warp
    // the whole warp runs the loop (its values stay warp-uniform); one elected
    // lane issues the copies
    if (n_steps > 0) {
      const CUtensorMap* bmap = (KIND == 1 && which == 1) ? &p.tm_b1 : &p.tm_b0;
      const MapOrder bord = (KIND == 1 && which == 1) ? p.ob1 : p.ob0;
      uint32_t bcnt = 0;
      int s = 0;
      bool ok = true;
      // KIND 1 walk state: head hh of the group, query tile qt, its row prefix
      int hh = 0, qt = qt0;
      long long pre = pre0;
      for (; s < n_steps && ok; ++s) {
        const int half = s & 1;
        long long blk;
        int brow, bhead;
        if (KIND == 0) {
          blk = (long long)p.hq * p.plan[b] + (long long)hx * T_b + pre0 + (s >> 1);
          brow = sq.k_start + (kb0 + (s >> 1)) * 128 + half * 64;
          bhead = hx / grp;
        } else {
          int kbq;
          wide_blocks_of_qtile(sq, qt, kbq);
          const int h = hx * grp + hh;
          blk = (long long)p.hq * p.plan[b] + (long long)h * T_b + pre + (tile - kbq);
          brow = sq.q_start + qt * 128 + half * 64;
          bhead = h;
        }
        if (blk < 0 || blk >= p.cap) {
          if (elect_sync()) {
            raise_status(p.status, DEV_WORKSPACE);
            *(volatile int*)&abort_flag = 1;
          }
          __syncwarp();
          ok = false;
          break;
        }
        const uint8_t* src = p.blocks + (size_t)blk * kWideBlock;
        const int as = s % C::kNA;
        if (!mbar_wait_warp(&aempty[as], ((s / C::kNA) & 1) ^ 1, ab)) {
          ok = false;
          break;
        }
        uint8_t* adst = sA + as * C::kA;
        if (s != drop && elect_sync()) {  // drop: test-only injected missing load
          mbar_arrive_tx(&afull[as], C::kA);
          if (KIND == 0) {  // dS sub-tile `half`: 128 query rows x 64 keys
            bulk_load(adst, src + 2 * kWideTile + half * kWideTile, kWideTile, &afull[as]);
          } else {  // query rows [64 half, 64 half + 64) of both 64-key sub-tiles
            const uint8_t* t0 = src + (which ? 2 * kWideTile : 0) + half * (kWideTile / 2);
            bulk_load(adst, t0, kWideTile / 2, &afull[as]);
            bulk_load(adst + kWideTile / 2, t0 + kWideTile, kWideTile / 2, &afull[as]);
          }
        }
        __syncwarp();
        int c1, c2, c3;
        map_coords(bord, 0, bhead, brow, tb, c1, c2, c3);
#pragma unroll
        for (int nh = 0; nh < C::kNH; ++nh, ++bcnt) {
          const uint32_t q = bcnt % C::kNB;
          if (!mbar_wait_warp(&bempty[q], ((bcnt / C::kNB) & 1u) ^ 1u, ab)) {
            ok = false;
            break;
          }
          if (elect_sync()) {
            mbar_arrive_tx(&bfull[q], C::kQuad);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              tma_load_4d(sB + q * C::kQuad + c * C::kChunk, bmap, &bfull[q], (4 * nh + c) * 64,
                          c1, c2, c3);
          }
          __syncwarp();
        }
        if (KIND == 1 && half == 1) {  // next query tile (then next head)
          int kbq;
          pre += wide_blocks_of_qtile(sq, qt, kbq);
          if (++qt == qt0 + n_qt) {
            qt = qt0;
            pre = pre0;
            ++hh;
          }
        }
      }
      // let the copies in flight land
      for (int v = s > C::kNA ? s - C::kNA : 0; v < s; ++v)
        mbar_wait_quiet(&afull[v % C::kNA], (v / C::kNA) & 1, lim);
      const uint32_t first = bcnt > (uint32_t)C::kNB ? bcnt - C::kNB : 0u;
      for (uint32_t c = first; c < bcnt; ++c)
        mbar_wait_quiet(&bfull[c % C::kNB], (c / C::kNB) & 1u, lim);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs the loop; the elected lane issues every MMA and commit
    if (n_steps > 0) {
      constexpr uint32_t idesc = make_idesc(128, 256, BF16, KIND == 1, true);
      const uint64_t adesc = KIND == 0 ? make_sdesc(smem_u32(sA), 16, 1024)
                                       : make_sdesc(smem_u32(sA), kWideTile / 2, 1024);
      const uint64_t bdesc = make_sdesc(smem_u32(sB), C::kChunk, 1024);
      uint32_t bcnt = 0;
      bool ok = true;
      for (int s = 0; s < n_steps && ok; ++s) {
        const int as = s % C::kNA;
        if (!mbar_wait_warp(&afull[as], (s / C::kNA) & 1, ab)) break;
        tc_fence_after();
        const uint64_t ad = adesc + (uint64_t)((as * C::kA) >> 4);
#pragma unroll
        for (int nh = 0; nh < C::kNH; ++nh, ++bcnt) {
          const uint32_t q = bcnt % C::kNB;
          if (!mbar_wait_warp(&bfull[q], (bcnt / C::kNB) & 1u, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = bdesc + (uint64_t)((q * C::kQuad) >> 4);
          if (elect_sync()) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(tmem + 256 * nh, ad + (KIND == 0 ? 2 * k : 128 * k), bd + 128 * k, idesc,
                     (s | k) ? 1u : 0u);
            mma_commit(&bempty[q]);
          }
          __syncwarp();
        }
        if (elect_sync()) mma_commit(&aempty[as]);
        __syncwarp();
      }
      if (elect_sync()) {
        mma_commit(&acc_done);
        mma_commit(&drain_bar);
        mbar_wait_quiet(&drain_bar, 0, lim);
      }
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int wq = (warp - 4) & 3;
    const int wg = (warp - 4) >> 2;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    bool ok = n_steps == 0 || mbar_wait_warp(&acc_done, 0, ab);
    if (ok && *(volatile int*)&abort_flag) ok = false;  // partial sums: leave the output
    if (ok) {
      tc_fence_after();
      const int row = r0 + r;
      const bool valid = row < (KIND == 0 ? sq.lq : sq.lk);
      const int64_t tok = (int64_t)(KIND == 0 ? sq.q_start : sq.k_start) + row;
      void* base = (KIND == 1 && which == 1) ? p.out1 : p.out0;
      const int64_t sb = (KIND == 1 && which == 1) ? p.so1_b : p.so0_b;
      const int64_t st = (KIND == 1 && which == 1) ? p.so1_t : p.so0_t;
      const int64_t sh = (KIND == 1 && which == 1) ? p.so1_h : p.so0_h;
      const float mul = (KIND == 1 && which == 0) ? 1.0f : p.scale;  // dV unscaled
      char* orow = (char*)base + ((int64_t)tb * sb + tok * st + (int64_t)hx * sh) * (G_F32 ? 4 : 2);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        const int col = wg * (D / 2) + c * 32;
        uint32_t rr[32];
        if (n_steps > 0) {
          tmem_ld32(tmem + lane_off + col, rr);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) rr[t] = 0u;
        }
        if (!valid) continue;
        if (G_F32) {
          float4* dst = reinterpret_cast<float4*>(orow + col * 4);
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            float4 w = make_float4(__uint_as_float(rr[4 * t]) * mul, __uint_as_float(rr[4 * t + 1]) * mul,
                                   __uint_as_float(rr[4 * t + 2]) * mul,
                                   __uint_as_float(rr[4 * t + 3]) * mul);
            if (p.accum) {  // sum into the caller's FP32 gradient
              const float4 old = dst[t];
              w.x += old.x;
              w.y += old.y;
              w.z += old.z;
              w.w += old.w;
            }
            dst[t] = w;
          }
        } else {
          uint4* dst = reinterpret_cast<uint4*>(orow + col * 2);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 v;
            v.x = Pack<BF16>::two(__uint_as_float(rr[8 * t + 0]) * mul, __uint_as_float(rr[8 * t + 1]) * mul);
            v.y = Pack<BF16>::two(__uint_as_float(rr[8 * t + 2]) * mul, __uint_as_float(rr[8 * t + 3]) * mul);
            v.z = Pack<BF16>::two(__uint_as_float(rr[8 * t + 4]) * mul, __uint_as_float(rr[8 * t + 5]) * mul);
            v.w = Pack<BF16>::two(__uint_as_float(rr[8 * t + 6]) * mul, __uint_as_float(rr[8 * t + 7]) * mul);
            dst[t] = v;
          }
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host side
namespace {

template <int D, bool BF16>
cudaError_t launch_scores_t(const WideScoresParams& p, cudaStream_t st) {
  using C = WideScoresCfg<D, D>;
  auto k = attn_bwd_wide_scores_kernel<D, D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid = tile_major(p.n_qtiles) ? dim3((unsigned)p.n_qtiles, (unsigned)p.hq, (unsigned)p.batch)
                                            : dim3((unsigned)p.hq, (unsigned)p.n_qtiles, (unsigned)p.batch);
  k<<<grid, 384, C::kSmem, st>>>(p);
  return cudaGetLastError();
}

template <int D, int KIND, bool BF16, bool G_F32>
cudaError_t launch_acc_t(const WideAccParams& p, cudaStream_t st) {
  using C = WideAccCfg<D>;
  auto k = attn_bwd_wide_acc_kernel<D, KIND, BF16, G_F32>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const unsigned nh = (unsigned)(KIND == 0 ? p.hq : p.hkv);
  const unsigned nz = (unsigned)(KIND == 0 ? p.batch : 2 * p.batch);
  const dim3 grid = tile_major(p.n_tiles) ? dim3((unsigned)p.n_tiles, nh, nz)
                                          : dim3(nh, (unsigned)p.n_tiles, nz);
  k<<<grid, 384, C::kSmem, st>>>(p);
  return cudaGetLastError();
}

template <int D, int KIND>
cudaError_t launch_acc_d(const WideAccParams& p, bool bf16, bool gf32, cudaStream_t st) {
  if (bf16) return gf32 ? launch_acc_t<D, KIND, true, true>(p, st) : launch_acc_t<D, KIND, true, false>(p, st);
  return gf32 ? launch_acc_t<D, KIND, false, true>(p, st) : launch_acc_t<D, KIND, false, false>(p, st);
}

template <int KIND>
cudaError_t launch_acc(const WideAccParams& p, int d, bool bf16, bool gf32, cudaStream_t st) {
  return d == 512 ? launch_acc_d<512, KIND>(p, bf16, gf32, st) : launch_acc_d<256, KIND>(p, bf16, gf32, st);
}

template <bool BF16>
cudaError_t launch_scores(const WideScoresParams& p, int d, cudaStream_t st) {
  return d == 512 ? launch_scores_t<512, BF16>(p, st) : launch_scores_t<256, BF16>(p, st);
}

}  // namespace

cudaError_t launch_bwd_wide(const BwdArgs& a, cudaStream_t st, int stages, int* n_launches) {
  *n_launches = 0;
  if (a.dqk != a.dv || (a.dqk != 512 && a.dqk != 256)) return cudaErrorNotSupported;
  const bool has_q = (a.thd ? a.total_q : a.batch * a.seqlen_q) > 0;
  const bool has_k = (a.thd ? a.total_k : a.batch * a.seqlen_k) > 0;
  const int nqt = (a.seqlen_q + 127) / 128, nkt = (a.seqlen_k + 127) / 128;
  if (nqt > 65535 || nkt > 65535 || a.batch > 32767 || a.hq > 65535) return cudaErrorInvalidValue;
  cudaError_t e;
  if (stages & 1) {
    if (has_q) {
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
  }
  // the block plan belongs to the dq stage (it depends on the key side and the
  // mask), so a D preprocess is valid for every problem with the same query rows
  if (stages & 2) {
    WidePlanParams pl;
    pl.geo = a.geo;
    pl.plan = a.wide_plan;
    pl.cap = a.wide_cap;
    pl.batch = a.batch;
    pl.hq = a.hq;
    pl.status = a.status;
    if ((e = launch_wide_plan(pl, st)) != cudaSuccess) return e;
    ++*n_launches;
  }
  if ((stages & 2) && has_q) {
    if (has_k) {
      WideScoresParams sp;
      sp.tm_q = a.tm_q128;
      sp.tm_k = a.tm_k128;
      sp.tm_v = a.tm_v128;
      sp.oq = a.oq;
      sp.ok = a.ok;
      sp.ov = a.ov;
      sp.geo = a.geo;
      sp.d = a.d;
      sp.d_sb = a.d_sb;
      sp.d_sh = a.d_sh;
      sp.dout = a.dout;
      sp.sdo_b = a.sdo[0]; sp.sdo_t = a.sdo[1]; sp.sdo_h = a.sdo[2];
      sp.plan = a.wide_plan;
      sp.blocks = a.wide_blocks;
      sp.cap = a.wide_cap;
      sp.batch = a.batch;
      sp.hq = a.hq;
      sp.hkv = a.hkv;
      sp.n_qtiles = nqt;
      sp.scale_log2 = a.scale_log2;
      sp.status = a.status;
      sp.dbg = a.dbg_scores;
      if ((e = a.bf16 ? launch_scores<true>(sp, a.dqk, st) : launch_scores<false>(sp, a.dqk, st)) !=
          cudaSuccess)
        return e;
      ++*n_launches;
    }
    WideAccParams qp;
    memset(&qp, 0, sizeof(qp));
    qp.tm_b0 = has_k ? a.tm_k64 : a.tm_q64;
    qp.tm_b1 = qp.tm_b0;
    qp.ob0 = has_k ? a.ok : a.oq;
    qp.ob1 = qp.ob0;
    qp.geo = a.geo;
    qp.plan = a.wide_plan;
    qp.blocks = a.wide_blocks;
    qp.cap = a.wide_cap;
    qp.out0 = a.dq;
    qp.so0_b = a.sdq[0]; qp.so0_t = a.sdq[1]; qp.so0_h = a.sdq[2];
    qp.out1 = a.dq;
    qp.so1_b = a.sdq[0]; qp.so1_t = a.sdq[1]; qp.so1_h = a.sdq[2];
    qp.accum = a.accum;
    qp.batch = a.batch;
    qp.hq = a.hq;
    qp.hkv = a.hkv;
    qp.n_tiles = nqt;
    qp.scale = a.scale;
    qp.status = a.status;
    qp.dbg = a.dbg_dq;
    if ((e = launch_acc<0>(qp, a.dqk, a.bf16, a.g_f32, st)) != cudaSuccess) return e;
    ++*n_launches;
  }
  if ((stages & 4) && has_k) {
    WideAccParams kp;
    memset(&kp, 0, sizeof(kp));
    kp.tm_b0 = has_q ? a.tm_do64 : a.tm_k64;
    kp.tm_b1 = has_q ? a.tm_q64 : a.tm_k64;
    kp.ob0 = has_q ? a.odo : a.ok;
    kp.ob1 = has_q ? a.oq : a.ok;
    kp.geo = a.geo;
    kp.plan = a.wide_plan;
    kp.blocks = a.wide_blocks;
    kp.cap = a.wide_cap;
    kp.out0 = a.dvp;
    kp.so0_b = a.sdv[0]; kp.so0_t = a.sdv[1]; kp.so0_h = a.sdv[2];
    kp.out1 = a.dk;
    kp.so1_b = a.sdk[0]; kp.so1_t = a.sdk[1]; kp.so1_h = a.sdk[2];
    kp.accum = a.accum;
    kp.batch = a.batch;
    kp.hq = a.hq;
    kp.hkv = a.hkv;
    kp.n_tiles = nkt;
    kp.scale = a.scale;
    kp.status = a.status;
    kp.dbg = a.dbg_dkdv;
    if ((e = launch_acc<1>(kp, a.dqk, a.bf16, a.g_f32, st)) != cudaSuccess) return e;
    ++*n_launches;
  }
  return cudaSuccess;
}

}  // namespace attn
