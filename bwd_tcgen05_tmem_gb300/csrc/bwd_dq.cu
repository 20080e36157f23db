// bwd_dq.cu -- query-stationary backward kernel: dQ (tcgen05 / TMEM / TMA).
//
// For 128 query rows of one (sequence, query head) and every visible key tile
// j (TransformerEngine PR #3510 / PR #3699 backward chain):
//   S  = Q K_j^T          (SS MMA, Q resident in shared memory)
//   dP = dO V_j^T         (SS MMA, dO resident)
//   P  = exp(scale S - LSE),  dS = P (dP - D)      (softmax warps, FP32)
//   dQ += dS K_j          (TS MMA: dS from TMEM, K_j chunk MN-major)
// and finally dQ *= scale.  No atomics: every dQ element is written once, so
// the result is bitwise reproducible.
//
// Warp roles (352 threads): warp 0 TMA producer, warp 1 TMEM allocator and
// S/dP issuer, warp 2 dQ issuer, warps 3..10 two softmax warpgroups; warpgroup w owns key
// columns [w*BKV/2, (w+1)*BKV/2) of every tile (the backward needs no row
// reduction, so splitting columns is free).  The softmax signals "scores
// consumed" right after loading S/dP so the next tile's S/dP MMAs overlap the
// exponentials.  The producer and issuer warps run their loops on all 32
// lanes and issue each copy, MMA and commit from an elect.sync lane.
// TMEM: S [0,BKV)  dP [BKV,2BKV)  dS [2BKV, 2.5BKV) (16-bit, 2 per column)
//       dQ [kTdQ, kTdQ + DQK).
#include "bwd.h"

namespace attn {

template <int DQK, int DV, int BKV>
struct DqCfg {
  static constexpr int kQSlots = DQK / 64;
  static constexpr int kDoSlots = DV / 64;
  static constexpr int kChunk = BKV * 128;  // one 64-column chunk of a key/value tile
  static constexpr int kKCh = DQK / 64;
  static constexpr int kVCh = DV / 64;
  static constexpr int kResident = (kQSlots + kDoSlots) * kSlotBytes;
  static constexpr int kBudget = kMaxSlots * kSlotBytes;  // dynamic bytes beyond the pad
  // K tiles live in whole stages (the dQ MMA reads K MN-major across its
  // chunks); V chunks go through a ring (the dP MMA reads them one by one).
  static constexpr int kKStage = kKCh * kChunk;
  static constexpr int kKStages = (kBudget - kResident - 3 * kKStage >= kVCh * kChunk) ? 3 : 2;
  static constexpr int kVRingRaw = (kBudget - kResident - kKStages * kKStage) / kChunk;
  static constexpr int kVRing = kVRingRaw > 12 ? 12 : kVRingRaw;
  static constexpr int kSmem = kResident + kKStages * kKStage + kVRing * kChunk + 1024;
  static constexpr int kTdP = BKV;
  static constexpr int kTdS = 2 * BKV;
  static constexpr int kTdQ = ((5 * BKV / 2) + 31) / 32 * 32;
  static constexpr int kHalf = BKV / 2;  // columns per softmax warpgroup
  // exponent arguments as packed pairs too: fewer instructions, but at QK head
  // dim 192 the register pairs cost more than they save (measured 11.91 vs
  // 12.01 ms at 32K; at head dim 128 packing them is the faster, 3.29 vs 3.34 ms)
  static constexpr bool kPackArg = DQK != 192;
  static_assert(kTdQ + DQK <= 512, "TMEM budget");
  static_assert(kVRing >= kVCh, "V ring must hold one tile");
  static_assert(BKV == 64 || BKV == 128, "BKV");
  static_assert(DQK <= 256, "one MMA covers the dQ columns");
};

// Eleven warps: no idle fourth warp, so each thread may hold 184 registers
// (65536 / 352) instead of 168, which the softmax's 64 scores, 64 dP values and
// packed dS need to keep several exponentials in flight.
constexpr int kDqThreads = 352;

template <int DQK, int DV, int BKV, bool BF16, bool G_F32>
__global__ void __launch_bounds__(kDqThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ DqParams p) {
  using C = DqCfg<DQK, DV, BKV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem;
  uint8_t* sDo = smem + C::kQSlots * kSlotBytes;
  uint8_t* sK = smem + C::kResident;
  uint8_t* sV = sK + C::kKStages * C::kKStage;

  __shared__ uint64_t kfull[C::kKStages], kempty[C::kKStages], vfull[C::kVRing], vempty[C::kVRing];
  __shared__ uint64_t q_bar, q_free, sdp_full, sc_free, ds_full, dq_done, drain_bar, drain_bar2;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag, skip_sh;

  const int warp = threadIdx.x >> 5;
  // Persistent: one CTA per SM takes work items (query tile, head, batch)
  // from the work queue, in the order the one-CTA-per-item grid had (heaviest
  // query tiles first: with tile_major(), x walks the query tiles of a head, y
  // the heads, z the batch; otherwise x walks the heads).  Every role decodes
  // the same items, and the barrier phases run on across items, so the next
  // item's Q/dO loads and first S/dP MMAs overlap this item's last tiles and
  // epilogue.
  const bool tmaj = tile_major(p.n_qtiles);
  const int gx = tmaj ? p.n_qtiles : p.hq, gy = tmaj ? p.hq : p.n_qtiles;
  const int n_items = gx * gy * p.batch;  // the launch checks that it fits
  __shared__ ItemRing<4> iring;
  struct Item {
    Seq sq;
    int h, g, b, tb, q0, kt0, n_kv;
    bool live;  // the query tile lies inside its sequence
  };
  auto item = [&](int L) {
    Item it;
    const int x = L % gx;
    const int rest = L / gx;
    const int y = rest % gy;
    it.b = rest / gy;
    it.h = tmaj ? y : x;
    it.g = it.h / (p.hq / p.hkv);
    it.tb = p.geo.cu_q ? 0 : it.b;  // TMA batch coordinate (packed THD tensors have one)
    it.sq = load_seq(p.geo, it.b);
    it.q0 = (p.n_qtiles - 1 - (tmaj ? x : y)) * kBlockM;
    it.live = it.q0 < it.sq.lq;
    it.kt0 = 0;
    it.n_kv = 0;
    if (it.live) {
      long long j0, j1;
      key_range(it.sq, it.q0, min(it.q0 + kBlockM, it.sq.lq) - 1, j0, j1);
      it.kt0 = (j1 >= j0) ? (int)(j0 / BKV) : 0;
      it.n_kv = (j1 >= j0) ? (int)(j1 / BKV) - it.kt0 + 1 : 0;
    }
    return it;
  };

  const unsigned long long lim = wait_limit_all(p.dbg);
  Abort ab{&abort_flag, p.status, lim};
  if (threadIdx.x == 0) {
    // a failed device check or an earlier abort stops every CTA
    const int status = p.status ? *(volatile int*)p.status : 0;
    abort_flag = 0;
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < C::kVRing; ++i) {
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
    }
    mbar_init(&q_bar, 1);
    mbar_init(&q_free, 1);
    item_ring_init(iring, 10);  // consumers: the two MMA issuers, eight softmax warps
    mbar_init(&sdp_full, 1);
    mbar_init(&sc_free, 256);
    mbar_init(&ds_full, 256);
    mbar_init(&dq_done, 1);
    mbar_init(&drain_bar, 1);
    mbar_init(&drain_bar2, 1);
    fence_barrier_init();
    skip_sh = status != 0;
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (skip_sh) {
    if (warp == 1) tmem_dealloc(tmem, 512);
    return;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // per item: Q and dO once their buffers are free (the previous item's
    // S/dP MMAs have run), then per key tile the V chunks (ring) and the K
    // stage.  The whole warp runs the loop (indices stay warp-uniform); one
    // elected lane issues the copies.
    uint32_t vcnt = 0;
    int gk = 0, ni = 0;  // K stages and items issued
    bool ok = true;
    for (int q = 0; ok; ++q) {
      const int L = item_ring_push(iring, q, p.counter, n_items, ab, ok);
      if (L < 0) break;
      const Item it = item(L);
      if (!it.live || it.n_kv == 0) continue;
      if (ni > 0 && !mbar_wait_warp(&q_free, (ni - 1) & 1u, ab)) {
        ok = false;
        break;
      }
      int c1, c2, c3, o1, o2, o3;
      map_coords(p.oq, 0, it.h, it.sq.q_start + it.q0, it.tb, c1, c2, c3);
      map_coords(p.odo, 0, it.h, it.sq.q_start + it.q0, it.tb, o1, o2, o3);
      if (elect_sync()) {
        mbar_arrive_tx(&q_bar, (C::kQSlots + C::kDoSlots) * kSlotBytes);
        for (int c = 0; c < C::kQSlots; ++c)
          tma_load_4d(sQ + c * kSlotBytes, &p.tm_q, &q_bar, c * 64, c1, c2, c3);
        for (int c = 0; c < C::kDoSlots; ++c)
          tma_load_4d(sDo + c * kSlotBytes, &p.tm_do, &q_bar, c * 64, o1, o2, o3);
      }
      __syncwarp();
      ++ni;
      for (int jt = 0; jt < it.n_kv && ok; ++jt) {
        const int krow = it.sq.k_start + (it.kt0 + jt) * BKV;
        int d1, d2, d3;
        map_coords(p.ov, 0, it.g, krow, it.tb, d1, d2, d3);
#pragma unroll
        for (int c = 0; c < C::kVCh; ++c, ++vcnt) {
          const uint32_t slot = vcnt % C::kVRing;
          if (!mbar_wait_warp(&vempty[slot], ((vcnt / C::kVRing) & 1u) ^ 1u, ab)) {
            ok = false;
            break;
          }
          if (elect_sync()) {
            mbar_arrive_tx(&vfull[slot], C::kChunk);
            tma_load_4d(sV + slot * C::kChunk, &p.tm_v, &vfull[slot], c * 64, d1, d2, d3);
          }
          __syncwarp();
        }
        if (!ok) break;
        const int st = gk % C::kKStages;
        if (!mbar_wait_warp(&kempty[st], ((gk / C::kKStages) & 1) ^ 1, ab)) {
          ok = false;
          break;
        }
        map_coords(p.ok, 0, it.g, krow, it.tb, d1, d2, d3);
        // test-only injected missing load: K of tile `drop_load` of work item 0
        if (!(L == 0 && jt == p.dbg.drop_load) && elect_sync()) {
          mbar_arrive_tx(&kfull[st], C::kKStage);
#pragma unroll
          for (int c = 0; c < C::kKCh; ++c)
            tma_load_4d(sK + st * C::kKStage + c * C::kChunk, &p.tm_k, &kfull[st], c * 64, d1, d2,
                        d3);
        }
        __syncwarp();
        ++gk;
      }
    }
    // let every copy still in flight land before the CTA can exit
    if (ni > 0) mbar_wait_quiet(&q_bar, (ni - 1) & 1u, lim);
    const uint32_t first = vcnt > (uint32_t)C::kVRing ? vcnt - C::kVRing : 0u;
    for (uint32_t c = first; c < vcnt; ++c)
      mbar_wait_quiet(&vfull[c % C::kVRing], (c / C::kVRing) & 1u, lim);
    for (int v = gk > C::kKStages ? gk - C::kKStages : 0; v < gk; ++v)
      mbar_wait_quiet(&kfull[v % C::kKStages], (v / C::kKStages) & 1, lim);
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // warp 1 issues S and dP, warp 2 issues dQ += dS K: one thread issues a
    // tcgen05.mma about every 60 cycles, so each product gets its own issuer.
    // Each warp runs its loop on all lanes; the elected lane issues the MMAs
    // and commits.  gt counts the key tiles of all items of this CTA.
    const bool sc_role = warp == 1;
    constexpr uint32_t idesc_s = make_idesc(128, BKV, BF16, false, false);
    constexpr uint32_t idesc_q = make_idesc(128, DQK, BF16, false, true);
    const uint64_t qdesc = make_sdesc(smem_u32(sQ), 16, 1024);
    const uint64_t ddesc = make_sdesc(smem_u32(sDo), 16, 1024);
    const uint64_t kdesc = make_sdesc(smem_u32(sK), 16, 1024);
    const uint64_t kdesc_mn = make_sdesc(smem_u32(sK), C::kChunk, 1024);
    const uint64_t vdesc = make_sdesc(smem_u32(sV), 16, 1024);
    uint32_t vcnt = 0;
    int gt = 0, ni = 0;
    bool ok = true;
    auto issue_scores = [&]() {
#pragma unroll
      for (int c = 0; c < C::kVCh; ++c, ++vcnt) {  // dP = dO V^T
        const uint32_t slot = vcnt % C::kVRing;
        if (!mbar_wait_warp(&vfull[slot], (vcnt / C::kVRing) & 1u, ab)) {
          ok = false;
          return;
        }
        tc_fence_after();
        const uint64_t da = ddesc + (uint64_t)(c * (kSlotBytes >> 4));
        const uint64_t vb = vdesc + (uint64_t)(slot * (C::kChunk >> 4));
        if (elect_sync()) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + C::kTdP, da + 2 * k, vb + 2 * k, idesc_s, (c | k) ? 1u : 0u);
          mma_commit(&vempty[slot]);
        }
        __syncwarp();
      }
      const int st = gt % C::kKStages;  // S = Q K^T
      if (!mbar_wait_warp(&kfull[st], (gt / C::kKStages) & 1, ab)) {
        ok = false;
        return;
      }
      tc_fence_after();
      if (elect_sync()) {
#pragma unroll
        for (int c = 0; c < C::kKCh; ++c) {
          const uint64_t qa = qdesc + (uint64_t)(c * (kSlotBytes >> 4));
          const uint64_t kb = kdesc + (uint64_t)((st * C::kKStage + c * C::kChunk) >> 4);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem, qa + 2 * k, kb + 2 * k, idesc_s, (c | k) ? 1u : 0u);
        }
        mma_commit(&sdp_full);
      }
      __syncwarp();
    };
    auto issue_dq = [&](bool accumulate) {  // dQ += dS K  (K stage read MN-major, N = DQK)
      const int st = gt % C::kKStages;
      const uint64_t kb = kdesc_mn + (uint64_t)((st * C::kKStage) >> 4);
      if (elect_sync()) {
        mma_ts(tmem + C::kTdQ, tmem + C::kTdS, kb, idesc_q, accumulate ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < BKV / 16; ++k)
          mma_ts(tmem + C::kTdQ, tmem + C::kTdS + k * 8, kb + k * 128, idesc_q, 1u);
        mma_commit(&kempty[st]);
        mma_commit(&dq_done);
      }
      __syncwarp();
    };
    for (int q = 0; ok; ++q) {
      const int L = item_ring_pop(iring, q, ab, ok);
      if (L < 0) break;
      const Item it = item(L);
      if (!it.live || it.n_kv == 0) continue;
      if (sc_role) {
        if (!mbar_wait_warp(&q_bar, ni & 1u, ab)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int jt = 0; jt < it.n_kv && ok; ++jt, ++gt) {
          // S/dP of this tile overwrite the previous tile's: the softmax must hold them
          if (gt > 0 && !mbar_wait_warp(&sc_free, (gt - 1) & 1u, ab)) {
            ok = false;
            break;
          }
          issue_scores();
        }
        if (!ok) break;
        if (elect_sync()) mma_commit(&q_free);  // Q and dO are read once these have run
        __syncwarp();
        ++ni;
      } else {
        // the first dQ MMA of an item overwrites the accumulator: the softmax
        // warps have read the previous item's dQ before they hand over its dS
        for (int jt = 0; jt < it.n_kv && ok; ++jt, ++gt) {
          if (!mbar_wait_warp(&ds_full, gt & 1u, ab)) {
            ok = false;
            break;
          }
          // the K stage of this tile: loaded (its S MMAs ran), released below
          if (!mbar_wait_warp(&kfull[gt % C::kKStages], (gt / C::kKStages) & 1, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_dq(jt > 0);
        }
      }
    }
    uint64_t* drain = sc_role ? &drain_bar : &drain_bar2;
    if (elect_sync()) {
      mma_commit(drain);
      mbar_wait_quiet(drain, 0, lim);
    }
    __syncwarp();
  } else if (warp >= 3) {
    // ------------------------------------------------------------ softmax / dS
    // warps 3..10; a warp reads and writes the TMEM lanes of its sub-partition
    const int wq = warp & 3;
    const int wg = (warp - 3) >> 2;
    const int r = wq * 32 + (threadIdx.x & 31);
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int col0 = wg * C::kHalf;
    const float sl2 = p.scale_log2;
    int gt = 0;
    bool ok = true;
    for (int q = 0; ok; ++q) {
      const int L = item_ring_pop(iring, q, ab, ok);
      if (L < 0) break;
      const Item it = item(L);
      if (!it.live) continue;
      const Seq& sq = it.sq;
      const int q0 = it.q0;
      const int i = q0 + r;
      const int64_t tok = (int64_t)sq.q_start + i;
      float lse2 = INFINITY, Dr = 0.0f;
      if (i < sq.lq) {  // LSE * log2 e (+inf for a keyless row: every key is masked) and D
        const float2 st = p.d[(int64_t)it.b * p.d_sb + (int64_t)it.h * p.d_sh + tok];
        lse2 = st.x;
        Dr = st.y;
      }
      const long long vis_lo = (long long)i + sq.off - sq.L;
      long long vis_hi = (long long)i + sq.off + sq.R;
      if (vis_hi > sq.lk - 1) vis_hi = sq.lk - 1;
      const long long rows_last = min(q0 + kBlockM, sq.lq) - 1;
      for (int jt = 0; jt < it.n_kv; ++jt, ++gt) {
        const int k0 = (it.kt0 + jt) * BKV;
        if (!mbar_wait_warp(&sdp_full, gt & 1u, ab)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[C::kHalf], dp[C::kHalf];
#pragma unroll
        for (int c = 0; c < C::kHalf / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_off + col0 + c * 32, rr);
#pragma unroll
          for (int t = 0; t < 32; ++t) s[c * 32 + t] = __uint_as_float(rr[t]);
          tmem_ld32(tmem + lane_off + C::kTdP + col0 + c * 32, rr);
#pragma unroll
          for (int t = 0; t < 32; ++t) dp[c * 32 + t] = __uint_as_float(rr[t]);
        }
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&sc_free);
        const int c0 = k0 + col0;  // first key of this warpgroup's columns
        const bool full_tile = (c0 + C::kHalf - 1 <= sq.lk - 1) &&
                               ((long long)c0 >= rows_last + sq.off - sq.L) &&
                               ((long long)(c0 + C::kHalf - 1) <= (long long)q0 + sq.off + sq.R);
        uint32_t pk[C::kHalf / 2];
        const long long lo = vis_lo - c0, hi = vis_hi - c0;
        // P = exp2(s * scale * log2 e - LSE log2 e), dS = P (dP - D), two
        // columns per packed FP32 operation (the softmax warps are bound by
        // instruction issue; a - b is a + (-b) exactly, so the results are
        // unchanged)
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2 = f2_pack(-lse2, -lse2);
        const uint64_t nd2 = f2_pack(-Dr, -Dr);
#pragma unroll
        for (int t = 0; t < C::kHalf; t += 2) {
          float x0, x1;
          if constexpr (C::kPackArg) {
            f2_unpack(f2_fma(f2_pack(s[t], s[t + 1]), sl2x2, nl2), x0, x1);
          } else {
            x0 = fmaf(s[t], sl2, -lse2);
            x1 = fmaf(s[t + 1], sl2, -lse2);
          }
          float e0 = ex2(x0);
          float e1 = ex2(x1);
          if (!full_tile) {
            if (t < lo || t > hi) e0 = 0.0f;
            if (t + 1 < lo || t + 1 > hi) e1 = 0.0f;
          }
          float g0, g1;
          f2_unpack(f2_mul(f2_pack(e0, e1), f2_add(f2_pack(dp[t], dp[t + 1]), nd2)), g0, g1);
          pk[t / 2] = Pack<BF16>::two(g0, g1);
        }
        // the dS columns were last read by the previous tile's dQ MMAs
        if (gt > 0 && !mbar_wait_warp(&dq_done, (gt - 1) & 1u, ab)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < C::kHalf / 32; ++c) {
          uint32_t w16[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) w16[t] = pk[c * 16 + t];
          tmem_st16(tmem + lane_off + C::kTdS + col0 / 2 + c * 16, w16);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ds_full);
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (it.n_kv > 0 && !mbar_wait_warp(&dq_done, (gt - 1) & 1u, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool valid = i < sq.lq;
      char* row = (char*)p.dq + ((int64_t)it.b * p.sdq_b + tok * p.sdq_t + (int64_t)it.h * p.sdq_h) *
                                    (G_F32 ? 4 : 2);
      constexpr int kCols = DQK / 2;  // dQ columns stored by this warpgroup
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c) {
        const int col = wg * kCols + c * 32;
        uint32_t rr[32];
        if (it.n_kv > 0) {
          tmem_ld32(tmem + lane_off + C::kTdQ + col, rr);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) rr[t] = 0u;
        }
        if (valid) {
          if (G_F32) {
            float4* dst = reinterpret_cast<float4*>(row + col * 4);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              float4 w = make_float4(__uint_as_float(rr[4 * t]) * p.scale,
                                     __uint_as_float(rr[4 * t + 1]) * p.scale,
                                     __uint_as_float(rr[4 * t + 2]) * p.scale,
                                     __uint_as_float(rr[4 * t + 3]) * p.scale);
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
            uint4* dst = reinterpret_cast<uint4*>(row + col * 2);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              uint4 v;
              v.x = Pack<BF16>::two(__uint_as_float(rr[8 * t + 0]) * p.scale,
                                    __uint_as_float(rr[8 * t + 1]) * p.scale);
              v.y = Pack<BF16>::two(__uint_as_float(rr[8 * t + 2]) * p.scale,
                                    __uint_as_float(rr[8 * t + 3]) * p.scale);
              v.z = Pack<BF16>::two(__uint_as_float(rr[8 * t + 4]) * p.scale,
                                    __uint_as_float(rr[8 * t + 5]) * p.scale);
              v.w = Pack<BF16>::two(__uint_as_float(rr[8 * t + 6]) * p.scale,
                                    __uint_as_float(rr[8 * t + 7]) * p.scale);
              dst[t] = v;
            }
          }
        }
      }
      // the epilogue's TMEM reads are complete (tcgen05.wait::ld) before this
      // thread hands over the next item's first dS, which the dQ issuer
      // waits for before its first MMA of that item overwrites the accumulator
      tc_fence_before();
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK, int DV, int BKV, bool BF16, bool G_F32>
static cudaError_t launch_dq_t(const DqParams& p, int num_sms, cudaStream_t st) {
  using C = DqCfg<DQK, DV, BKV>;
  auto k = attn_bwd_dq_kernel<DQK, DV, BKV, BF16, G_F32>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  // persistent: at most one CTA per SM, each taking items from the work queue
  const long long items = (long long)p.n_qtiles * p.hq * p.batch;
  if (items > 0x7fffffffll || !p.counter) return cudaErrorInvalidValue;
  const long long ctas = items < num_sms ? items : num_sms;
  if (ctas <= 0) return cudaSuccess;
  k<<<(unsigned)ctas, kDqThreads, C::kSmem, st>>>(p);
  return cudaGetLastError();
}

template <int DQK, int DV, int BKV>
static cudaError_t launch_dq_d(const DqParams& p, bool bf16, bool gf32, int num_sms,
                               cudaStream_t st) {
  if (bf16)
    return gf32 ? launch_dq_t<DQK, DV, BKV, true, true>(p, num_sms, st)
                : launch_dq_t<DQK, DV, BKV, true, false>(p, num_sms, st);
  return gf32 ? launch_dq_t<DQK, DV, BKV, false, true>(p, num_sms, st)
              : launch_dq_t<DQK, DV, BKV, false, false>(p, num_sms, st);
}

// Rows of the key/value tile streamed by the dQ kernel for a head-dim pair.
int dq_block_kv(int dqk, int dv) { return (dqk >= 256 || dv >= 256) ? 64 : 128; }

cudaError_t launch_dq(const DqParams& p, int dqk, int dv, bool bf16, bool gf32, int num_sms,
                      cudaStream_t st) {
  if (dqk == 64 && dv == 64) return launch_dq_d<64, 64, 128>(p, bf16, gf32, num_sms, st);
  if (dqk == 128 && dv == 128) return launch_dq_d<128, 128, 128>(p, bf16, gf32, num_sms, st);
  if (dqk == 192 && dv == 128) return launch_dq_d<192, 128, 128>(p, bf16, gf32, num_sms, st);
  if (dqk == 256 && dv == 256) return launch_dq_d<256, 256, 64>(p, bf16, gf32, num_sms, st);
  return cudaErrorNotSupported;
}

}  // namespace attn
