// bwd_dkdv.cu -- key/value-stationary backward kernel: dK and dV
// (tcgen05 / TMEM / TMA).
//
// One CTA owns 128 key rows of one (sequence, key/value head) and walks every
// query head of its GQA group and every visible query tile i of BQ rows
// (TransformerEngine PR #3699: gradients reduced over the GQA group; PR #3510
// backward chain):
//   S^T  = K Q_i^T            (SS MMA, K resident)
//   dP^T = V dO_i^T           (SS MMA, V resident)            [dK]
//   P^T  = exp(scale S^T - LSE_i),  dS^T = P^T (dP^T - D_i)   (softmax warps)
//   dV  += P^T dO_i           (TS MMA: P^T from TMEM)         [dV]
//   dK  += dS^T Q_i           (TS MMA: dS^T from TMEM)        [dK]
// then dK *= scale.  The group reduction happens in TMEM, in a fixed order:
// no atomics, bitwise reproducible.
//
// With a dS workspace (the dS path of the backward) the softmax warps also
// store each dS^T tile, as the MN-major A operand image of the dQ GEMM's
// 32 KiB blocks (bwd.h), so that dQ needs no second pass over the scores.
//
// MODE selects the accumulators: 3 = dK and dV, 1 = dV only, 2 = dK only
// (head dim 256 runs one launch of each: both accumulators do not fit in the
// 512 TMEM columns next to the score tiles).
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 TMEM allocator and
// score-MMA issuer, warp 2 loads LSE_i / D_i into shared memory, warp 3
// accumulate-MMA issuer, warps 4..11 two
// softmax warpgroups splitting the BQ query columns.  The producer and issuer
// warps run their loops on all 32 lanes and issue each copy, MMA and commit
// from an elect.sync lane.
#include "bwd.h"

namespace attn {

template <int DQK, int DV, int BQ, int MODE>
struct DkvCfg {
  static constexpr bool kDV = (MODE & 1) != 0;
  static constexpr bool kDK = (MODE & 2) != 0;
  static constexpr int kKSlots = DQK / 64;
  static constexpr int kVSlots = kDK ? DV / 64 : 0;
  static constexpr int kResident = (kKSlots + kVSlots) * kSlotBytes;
  static constexpr int kChunk = BQ * 128;  // one 64-column chunk of a query tile
  static constexpr int kQCh = DQK / 64;
  static constexpr int kDoCh = DV / 64;
  // A streamed operand that an accumulate MMA reads MN-major (Q for dK, dO
  // for dV) is staged: a whole tile, contiguous, held until that MMA.  The
  // other operand goes through a chunk ring released after the score MMA.
  static constexpr bool kQStaged = kDK;
  static constexpr bool kDStaged = kDV;
  static constexpr int kStageBytes = (kQStaged ? kQCh : 0) * kChunk + (kDStaged ? kDoCh : 0) * kChunk;
  static constexpr int kRingTile = (kQStaged ? 0 : kQCh) + (kDStaged ? 0 : kDoCh);  // ring chunks per tile
  static constexpr int kStatic = 2 * BQ * 4 * (kDK ? 2 : 1) + 512;  // LSE/D staging + barriers
  static constexpr int kBudget = 232448 - 1024 - kStatic;
  static constexpr int kStages = (kBudget - kResident - 3 * kStageBytes >= 2 * kRingTile * kChunk) ? 3 : 2;
  static constexpr int kRingRaw = kRingTile ? (kBudget - kResident - kStages * kStageBytes) / kChunk : 1;
  static constexpr int kRing = kRingRaw > 12 ? 12 : kRingRaw;
  static constexpr int kRingAlloc = kRingTile ? kRing : 0;  // ring slots in shared memory
  static constexpr int kSmem = kResident + kStages * kStageBytes + kRingAlloc * kChunk + 1024;
  static constexpr int kHalf = BQ / 2;
  // the dS path runs at these shapes (ds_backward)
  static constexpr bool kCanDs = kDK && kDV && (DQK == 128 || DQK == 192);
  // TMEM columns
  static constexpr int kTS = 0;
  static constexpr int kTdP = BQ;
  static constexpr int kTP = kDK ? 2 * BQ : BQ;
  static constexpr int kTdS = kTP + (kDV ? BQ / 2 : 0);
  static constexpr int kTAcc = ((kTdS + (kDK ? BQ / 2 : 0)) + 31) / 32 * 32;
  static constexpr int kTdV = kTAcc;
  static constexpr int kTdK = kTAcc + (kDV ? DV : 0);
  static constexpr int kTEnd = kTdK + (kDK ? DQK : 0);
  static_assert(kTEnd <= 512, "TMEM budget");
  static_assert(BQ == 64 || BQ == 128, "BQ");
  static_assert(MODE >= 1 && MODE <= 3, "MODE");
  static_assert(kRingTile == 0 || kRing >= 2, "ring");
  static_assert(DQK <= 256 && DV <= 256, "one MMA covers the accumulator columns");
};

template <int DQK, int DV, int BQ, int MODE, bool BF16, bool G_F32, bool WDS>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ DkvParams p) {
  using C = DkvCfg<DQK, DV, BQ, MODE>;
  static_assert(!WDS || (C::kCanDs && BQ == 64), "dS stores");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kKSlots * kSlotBytes;
  uint8_t* sStage = smem + C::kResident;          // [kStages][Q chunks | dO chunks]
  uint8_t* sRing = sStage + C::kStages * C::kStageBytes;
  constexpr int kQOff = 0;                                     // inside a stage
  constexpr int kDOff = C::kQStaged ? C::kQCh * C::kChunk : 0;

  __shared__ uint64_t sfull[C::kStages], sempty[C::kStages], rfull[C::kRing], rempty[C::kRing];
  __shared__ uint64_t kv_bar, sdp_full, sc_free, pds_full, acc_done, drain_bar, drain_bar2;
  __shared__ uint64_t ld_full[2], ld_empty[2];
  __shared__ __align__(16) float s_lse2[2][BQ];
  __shared__ __align__(16) float s_d[2][C::kDK ? BQ : 4];
  __shared__ int s_dsblk[2];  // dS path: block of the tile whose LSE / D are staged
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag, skip_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // (key tile, kv head) in the grid order of tile_major(); under a causal mask
  // the lowest key tiles are the heaviest and start first
  const bool tmaj = tile_major(p.n_ktiles);
  const int g = tmaj ? blockIdx.y : blockIdx.x;
  const int ktile = tmaj ? blockIdx.x : blockIdx.y;
  const int b = blockIdx.z;
  const int tb = p.geo.cu_q ? 0 : b;  // TMA batch coordinate (packed THD tensors have one)
  const int grp = p.hq / p.hkv;

  const Seq sq = load_seq(p.geo, b);
  const int k0 = ktile * kBlockM;
  if (k0 >= sq.lk) return;
  long long i0, i1;
  query_range(sq, k0, min(k0 + kBlockM, sq.lk) - 1, i0, i1);
  const int qt0 = (i1 >= i0) ? (int)(i0 / BQ) : 0;
  const int n_qt = (i1 >= i0) ? (int)(i1 / BQ) - qt0 + 1 : 0;
  const int n_it = n_qt * grp;  // iterations: head-major over the group, then query tiles

  const unsigned long long lim = wait_limit(p.dbg);
  const int drop = dropped_load(p.dbg);
  Abort ab{&abort_flag, p.status, lim};
  if (threadIdx.x == 0) {
    // a failed device check or an earlier abort stops every CTA; the status
    // word is tested only once the barriers are set up and the resident K and
    // V copies are under way (tensor-map copies stay in bounds regardless)
    const int status = p.status ? *(volatile int*)p.status : 0;
    abort_flag = 0;
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], 1);
    }
    for (int i = 0; i < C::kRing; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], 1);
    }
    mbar_init(&kv_bar, 1);
    mbar_init(&sdp_full, 1);
    mbar_init(&sc_free, 256);
    mbar_init(&pds_full, 256);
    mbar_init(&acc_done, 1);
    mbar_init(&drain_bar, 1);
    mbar_init(&drain_bar2, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ld_full[s], 32);
      mbar_init(&ld_empty[s], 256);
    }
    fence_barrier_init();
    if (n_it > 0) {
      int c1, c2, c3, v1, v2, v3;
      map_coords(p.ok, 0, g, sq.k_start + k0, tb, c1, c2, c3);
      map_coords(p.ov, 0, g, sq.k_start + k0, tb, v1, v2, v3);
      mbar_arrive_tx(&kv_bar, (C::kKSlots + C::kVSlots) * kSlotBytes);
      for (int c = 0; c < C::kKSlots; ++c)
        tma_load_4d(sK + c * kSlotBytes, &p.tm_k, &kv_bar, c * 64, c1, c2, c3);
      if (C::kDK) {
        for (int c = 0; c < C::kVSlots; ++c)
          tma_load_4d(sV + c * kSlotBytes, &p.tm_v, &kv_bar, c * 64, v1, v2, v3);
      }
    }
    skip_sh = status != 0;
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (skip_sh) {  // let the resident copies land, free TMEM, leave
    if (threadIdx.x == 0 && n_it > 0) mbar_wait_quiet(&kv_bar, 0, lim);
    if (warp == 1) tmem_dealloc(tmem, 512);
    return;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // per query tile: the ring chunks (score-only operand), then the stage
    // (K and V were issued with the barrier set-up); the whole warp runs the
    // loop (indices stay warp-uniform); one elected lane issues the copies
    if (n_it > 0) {
      uint32_t rcnt = 0;
      int it = 0, hh = 0, tq = 0;  // iteration it = head hh of the group, query tile tq
      bool ok = true;
      for (; it < n_it && ok; ++it, (++tq == n_qt) ? (tq = 0, ++hh) : 0) {
        const int h = g * grp + hh;
        const int qrow = sq.q_start + (qt0 + tq) * BQ;
        int qc1, qc2, qc3, dc1, dc2, dc3;
        map_coords(p.oq, 0, h, qrow, tb, qc1, qc2, qc3);
        map_coords(p.odo, 0, h, qrow, tb, dc1, dc2, dc3);
        if constexpr (C::kRingTile > 0) {
          constexpr int nch = C::kQStaged ? C::kDoCh : C::kQCh;
          const CUtensorMap* m = C::kQStaged ? &p.tm_do : &p.tm_q;
#pragma unroll
          for (int c = 0; c < nch; ++c, ++rcnt) {
            const uint32_t slot = rcnt % C::kRing;
            if (!mbar_wait_warp(&rempty[slot], ((rcnt / C::kRing) & 1u) ^ 1u, ab)) {
              ok = false;
              break;
            }
            if (elect_sync()) {
              mbar_arrive_tx(&rfull[slot], C::kChunk);
              if (C::kQStaged)
                tma_load_4d(sRing + slot * C::kChunk, m, &rfull[slot], c * 64, dc1, dc2, dc3);
              else
                tma_load_4d(sRing + slot * C::kChunk, m, &rfull[slot], c * 64, qc1, qc2, qc3);
            }
            __syncwarp();
          }
          if (!ok) break;
        }
        const int st = it % C::kStages;
        if (!mbar_wait_warp(&sempty[st], ((it / C::kStages) & 1) ^ 1, ab)) {
          ok = false;
          break;
        }
        if (it != drop && elect_sync()) {  // drop: test-only injected missing load
          mbar_arrive_tx(&sfull[st], C::kStageBytes);
          uint8_t* dst = sStage + st * C::kStageBytes;
          if constexpr (C::kQStaged) {
#pragma unroll
            for (int c = 0; c < C::kQCh; ++c)
              tma_load_4d(dst + kQOff + c * C::kChunk, &p.tm_q, &sfull[st], c * 64, qc1, qc2, qc3);
          }
          if constexpr (C::kDStaged) {
#pragma unroll
            for (int c = 0; c < C::kDoCh; ++c)
              tma_load_4d(dst + kDOff + c * C::kChunk, &p.tm_do, &sfull[st], c * 64, dc1, dc2, dc3);
          }
        }
        __syncwarp();
      }
      mbar_wait_quiet(&kv_bar, 0, lim);
      const uint32_t first = rcnt > (uint32_t)C::kRing ? rcnt - C::kRing : 0u;
      for (uint32_t c = first; c < rcnt; ++c)
        mbar_wait_quiet(&rfull[c % C::kRing], (c / C::kRing) & 1u, lim);
      const int ns = ok ? n_it : it;  // stages issued
      for (int v = ns > C::kStages ? ns - C::kStages : 0; v < ns; ++v)
        mbar_wait_quiet(&sfull[v % C::kStages], (v / C::kStages) & 1, lim);
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // warp 1 issues the score MMAs (S^T, dP^T), warp 3 the accumulate MMAs
    // (dV, dK): one thread issues a tcgen05.mma about every 60 cycles, so each
    // gets its own issuer.  Each warp runs its loop on all lanes; the elected
    // lane issues the MMAs and commits.
    if (n_it > 0) {
      const bool sc_role = warp == 1;
      constexpr uint32_t idesc_s = make_idesc(128, BQ, BF16, false, false);
      constexpr uint32_t idesc_v = make_idesc(128, DV, BF16, false, true);
      constexpr uint32_t idesc_k = make_idesc(128, DQK, BF16, false, true);
      const uint64_t kdesc = make_sdesc(smem_u32(sK), 16, 1024);
      const uint64_t vdesc = make_sdesc(smem_u32(sV), 16, 1024);
      const uint64_t stdesc = make_sdesc(smem_u32(sStage), 16, 1024);           // K-major view
      const uint64_t stdesc_mn = make_sdesc(smem_u32(sStage), C::kChunk, 1024);  // MN-major view
      const uint64_t rdesc = make_sdesc(smem_u32(sRing), 16, 1024);
      uint32_t rcnt = 0;
      bool ok = sc_role ? mbar_wait_warp(&kv_bar, 0, ab) : true;
      tc_fence_after();
      // ring chunks are consumed one by one in load order and released as soon
      // as their score MMAs complete; the stage is held until issue_acc
      auto ring_chunk = [&]() -> uint64_t {
        const uint32_t slot = rcnt % C::kRing;
        if (!mbar_wait_warp(&rfull[slot], (rcnt / C::kRing) & 1u, ab)) {
          ok = false;
          return 0ull;
        }
        tc_fence_after();
        return rdesc + (uint64_t)((slot * C::kChunk) >> 4);
      };
      auto ring_release = [&]() {  // called by the elected lane
        mma_commit(&rempty[rcnt % C::kRing]);
      };
      // The stage of tile `it` is awaited only right before its first use:
      // the producer loads a tile's ring chunks before its stage, so waiting
      // for the stage first would deadlock once the ring is full.
      auto wait_stage = [&](int it) {
        if (!mbar_wait_warp(&sfull[it % C::kStages], (it / C::kStages) & 1, ab)) ok = false;
        tc_fence_after();
      };
      auto issue_scores = [&](int it) {
        const int st = it % C::kStages;
        const uint32_t st_off = (uint32_t)((st * C::kStageBytes) >> 4);
        if constexpr (C::kQStaged) {
          wait_stage(it);
          if (!ok) return;
        }
        // S^T = K Q^T
#pragma unroll
        for (int c = 0; c < C::kQCh; ++c) {
          const uint64_t ka = kdesc + (uint64_t)(c * (kSlotBytes >> 4));
          uint64_t qb;
          if constexpr (C::kQStaged) {
            qb = stdesc + st_off + (uint64_t)((kQOff + c * C::kChunk) >> 4);
          } else {
            qb = ring_chunk();
            if (!ok) return;
          }
          if (elect_sync()) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(tmem + C::kTS, ka + 2 * k, qb + 2 * k, idesc_s, (c | k) ? 1u : 0u);
            if constexpr (!C::kQStaged) ring_release();
          }
          __syncwarp();
          if constexpr (!C::kQStaged) ++rcnt;
        }
        // dP^T = V dO^T
        if constexpr (C::kDK) {
          if constexpr (C::kDStaged && !C::kQStaged) {
            wait_stage(it);
            if (!ok) return;
          }
#pragma unroll
          for (int c = 0; c < C::kDoCh; ++c) {
            const uint64_t va = vdesc + (uint64_t)(c * (kSlotBytes >> 4));
            uint64_t db;
            if constexpr (C::kDStaged) {
              db = stdesc + st_off + (uint64_t)((kDOff + c * C::kChunk) >> 4);
            } else {
              db = ring_chunk();
              if (!ok) return;
            }
            if (elect_sync()) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_ss(tmem + C::kTdP, va + 2 * k, db + 2 * k, idesc_s, (c | k) ? 1u : 0u);
              if constexpr (!C::kDStaged) ring_release();
            }
            __syncwarp();
            if constexpr (!C::kDStaged) ++rcnt;
          }
        }
        if (elect_sync()) mma_commit(&sdp_full);
        __syncwarp();
      };
      auto issue_acc = [&](int it) {
        const int st = it % C::kStages;
        wait_stage(it);  // completes at once if the score MMAs already waited
        if (!ok) return;
        const uint32_t st_off = (uint32_t)((st * C::kStageBytes) >> 4);
        const uint32_t first = it > 0 ? 1u : 0u;
        if (elect_sync()) {
          if constexpr (C::kDV) {  // dV += P^T dO   (dO stage MN-major, N = DV)
            const uint64_t db = stdesc_mn + st_off + (uint64_t)(kDOff >> 4);
            mma_ts(tmem + C::kTdV, tmem + C::kTP, db, idesc_v, first);
#pragma unroll
            for (int k = 1; k < BQ / 16; ++k)
              mma_ts(tmem + C::kTdV, tmem + C::kTP + k * 8, db + k * 128, idesc_v, 1u);
          }
          if constexpr (C::kDK) {  // dK += dS^T Q   (Q stage MN-major, N = DQK)
            const uint64_t qb = stdesc_mn + st_off + (uint64_t)(kQOff >> 4);
            mma_ts(tmem + C::kTdK, tmem + C::kTdS, qb, idesc_k, first);
#pragma unroll
            for (int k = 1; k < BQ / 16; ++k)
              mma_ts(tmem + C::kTdK, tmem + C::kTdS + k * 8, qb + k * 128, idesc_k, 1u);
          }
          mma_commit(&sempty[st]);
          mma_commit(&acc_done);
        }
        __syncwarp();
      };
      if (sc_role) {
        for (int it = 0; it < n_it && ok; ++it) {
          // S^T/dP^T of tile it overwrite those of it-1: the softmax must hold them
          if (it > 0 && !mbar_wait_warp(&sc_free, (it - 1) & 1u, ab)) break;
          issue_scores(it);
        }
      } else {
        for (int it = 0; it < n_it && ok; ++it) {
          if (!mbar_wait_warp(&pds_full, it & 1u, ab)) break;
          tc_fence_after();
          issue_acc(it);
        }
      }
      uint64_t* drain = sc_role ? &drain_bar : &drain_bar2;
      if (elect_sync()) {
        mma_commit(drain);
        mbar_wait_quiet(drain, 0, lim);
      }
      __syncwarp();
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ LSE / D loader
    // On the dS path this warp also walks the block table (block indexes fit
    // in 32 bits, the host checks): ds_row is the first block of the current
    // 128-row query tile ds_q128 of the current head, ds_kb0 / ds_nkb its
    // first visible key block and their count, ds_head0 the first block of
    // head g * grp, ds_tb the blocks of one head of this sequence.  With each
    // tile's LSE and D it stages the index of the tile's dS block.
    const bool wds = WDS && n_it > 0;
    int ds_head0 = 0, ds_tb = 0, ds_row = 0, ds_q128 = 0, ds_kb0 = 0, ds_nkb = 0;
    if (wds) {
      ds_tb = (int)(p.plan[b + 1] - p.plan[b]);
      ds_head0 = (int)((long long)p.hq * p.plan[b] + (long long)g * grp * ds_tb) +
                 (int)blocks_row_prefix(sq, (qt0 * BQ) >> 7);  // whole warp
      if constexpr (BQ == 64) {
        // A visible block whose other 64-row half this CTA never visits (no
        // query of that half sees a key of this tile) gets zeros there: the
        // first tile's lower half, the last tile's upper half if it holds rows.
        const int ql = qt0 + n_qt - 1;
        const bool lo_gap = (qt0 & 1) != 0;
        const bool hi_gap = (ql & 1) == 0 && (long long)(ql + 1) * 64 < sq.lq;
        const int hi_off = hi_gap ? (int)(blocks_row_prefix(sq, ql >> 1) -
                                          blocks_row_prefix(sq, qt0 >> 1))
                                  : 0;  // whole warp
        const uint64_t pol = l2_evict_first();
        for (int half = 0; half < 2; ++half) {
          if (!(half == 0 ? lo_gap : hi_gap)) continue;
          int kb0;
          const int nkb = wide_blocks_of_qtile(sq, half == 0 ? qt0 >> 1 : ql >> 1, kb0);
          for (int hh = 0; hh < grp; ++hh) {
            const int blk = ds_head0 + hh * ds_tb + (half ? hi_off : 0) + (ktile - kb0);
            if (!(blk >= 0 && blk < p.cap && ktile >= kb0 && ktile < kb0 + nkb)) {
              if (lane == 0) raise_status(p.status, DEV_WORKSPACE);  // inconsistent plan
              continue;
            }
            uint4* dst = reinterpret_cast<uint4*>(p.ds + (size_t)blk * kDsBlock + half * (kDsBlock / 2));
            for (int t = lane; t < kDsBlock / 32; t += 32) st_global_hint(dst + t, make_uint4(0u, 0u, 0u, 0u), pol);
          }
        }
      }
    }
    bool ok = true;
    int hh = 0, tq = 0;  // iteration it = head hh of the group, query tile tq
    for (int it = 0; it < n_it && ok; ++it, (++tq == n_qt) ? (tq = 0, ++hh) : 0) {
      const int st = it & 1;
      if (!mbar_wait_warp(&ld_empty[st], ((it >> 1) & 1u) ^ 1u, ab)) break;
      const int h = g * grp + hh;
      const int q0 = (qt0 + tq) * BQ;
      if constexpr (WDS) {
        int blk = -1;
        if (wds) {
          if (tq == 0) {  // first tile of a head
            ds_row = ds_head0 + hh * ds_tb;
            ds_q128 = q0 >> 7;
            ds_nkb = wide_blocks_of_qtile(sq, ds_q128, ds_kb0);
          } else if ((q0 >> 7) != ds_q128) {
            ds_row += ds_nkb;
            ds_q128 = q0 >> 7;
            ds_nkb = wide_blocks_of_qtile(sq, ds_q128, ds_kb0);
          }
          blk = ds_row + (ktile - ds_kb0);
          if (!(blk >= 0 && blk < p.cap && ktile >= ds_kb0 && ktile < ds_kb0 + ds_nkb)) {
            if (lane == 0) raise_status(p.status, DEV_WORKSPACE);  // inconsistent plan: no store
            blk = -1;
          }
        }
        if (lane == 0) s_dsblk[st] = blk;
      }
      for (int t = lane; t < BQ; t += 32) {
        const int i = q0 + t;
        float l2 = INFINITY, dd = 0.0f;
        if (i < sq.lq) {  // LSE * log2 e (+inf for a keyless row: masked anyway) and D
          const int64_t tok = (int64_t)sq.q_start + i;
          const float2 st = p.d[(int64_t)b * p.d_sb + (int64_t)h * p.d_sh + tok];
          l2 = st.x;
          dd = st.y;
        }
        s_lse2[st][t] = -l2;  // negated: the softmax adds them
        s_d[st][t] = -dd;
      }
      mbar_arrive(&ld_full[st]);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / dS
    const int wq = (warp - 4) & 3;
    const int wg = (warp - 4) >> 2;
    const int r = wq * 32 + lane;
    const int j = k0 + r;  // key row within the sequence
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int col0 = wg * C::kHalf;
    const float sl2 = p.scale_log2;
    // query rows that see key j: [vis_lo, vis_hi]
    const long long vis_lo = (long long)j - sq.off - sq.R;
    long long vis_hi = (long long)j - sq.off + sq.L;
    if (vis_hi > sq.lq - 1) vis_hi = sq.lq - 1;
    // dS path: a key row past the sequence sees no query, so its dS row is
    // zero in the block (the dQ GEMM reads whole blocks, and the K rows it
    // multiplies there may belong to the next packed sequence); such a tile
    // takes the masked path
    if (WDS && j >= sq.lk) vis_hi = -1;
    const bool part_tile = WDS && k0 + kBlockM > sq.lk;
    const long long krow_last = min(k0 + kBlockM, sq.lk) - 1;
    bool ok = true;
    int tq = 0;  // query tile of iteration it
    for (int it = 0; it < n_it; ++it, tq = (tq + 1 == n_qt) ? 0 : tq + 1) {
      const int st = it & 1;
      const int q0 = (qt0 + tq) * BQ;
      if (!mbar_wait_warp(&sdp_full, it & 1u, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[C::kHalf], dp[C::kHalf];
#pragma unroll
      for (int c = 0; c < C::kHalf / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_off + C::kTS + col0 + c * 32, rr);
#pragma unroll
        for (int t = 0; t < 32; ++t) s[c * 32 + t] = __uint_as_float(rr[t]);
        if constexpr (C::kDK) {
          tmem_ld32(tmem + lane_off + C::kTdP + col0 + c * 32, rr);
#pragma unroll
          for (int t = 0; t < 32; ++t) dp[c * 32 + t] = __uint_as_float(rr[t]);
        }
      }
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&sc_free);
      if (!mbar_wait_warp(&ld_full[st], (it >> 1) & 1u, ab)) {
        ok = false;
        break;
      }
      const int c0 = q0 + col0;  // first query row of this warpgroup's columns
      const bool full_tile = !part_tile && ((long long)(c0 + C::kHalf - 1) <= sq.lq - 1) &&
                             ((long long)c0 >= krow_last - sq.off - sq.R) &&
                             ((long long)(c0 + C::kHalf - 1) <= (long long)k0 - sq.off + sq.L);
      const long long lo = vis_lo - c0, hi = vis_hi - c0;
      // this warpgroup's LSE / D columns, read as 16-byte shared loads
      const float4* l4 = reinterpret_cast<const float4*>(&s_lse2[st][col0]);
      const float4* d4 = reinterpret_cast<const float4*>(&s_d[st][col0]);
      uint32_t pp[C::kHalf / 2], pd[C::kHalf / 2];
      // P = exp2(s * scale * log2 e - LSE log2 e), dS = P (dP - D), two columns
      // per packed FP32 operation (shared memory holds -LSE log2 e and -D; the
      // softmax warps are bound by instruction issue)
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      // dS path: this thread's key row of dS^T goes into the block as 16-byte
      // chunks of 8 queries, each stored as soon as it is computed so that the
      // stores drain while the warp computes; a warp's 32 rows of one chunk
      // are 512 contiguous bytes.  Written once and read once by the dQ GEMM:
      // L2 evict-first, so the reused Q / dO tiles stay.
      bool ds_on = false;
      uint4* ds_dst = nullptr;
      uint64_t ds_pol = 0;
      if constexpr (WDS) {
        const int dsb = s_dsblk[st];
        ds_on = dsb >= 0;
        ds_pol = l2_evict_first();
        ds_dst = reinterpret_cast<uint4*>(p.ds + (size_t)(ds_on ? dsb : 0) * kDsBlock) + r +
                 (((q0 + col0) & 127) >> 3) * (kDsChunk / 16);
      }
#pragma unroll
      for (int t4 = 0; t4 < C::kHalf / 4; ++t4) {
        const float4 la = l4[t4];
        const uint64_t nl[2] = {f2_pack(la.x, la.y), f2_pack(la.z, la.w)};
        uint64_t nd[2] = {0ull, 0ull};
        if constexpr (C::kDK) {
          const float4 da = d4[t4];
          nd[0] = f2_pack(da.x, da.y);
          nd[1] = f2_pack(da.z, da.w);
        }
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
          const int t = 4 * t4 + u;
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(s[t], s[t + 1]), sl2x2, nl[u / 2]), x0, x1);
          float e0 = ex2(x0);
          float e1 = ex2(x1);
          if (!full_tile) {
            if (t < lo || t > hi) e0 = 0.0f;
            if (t + 1 < lo || t + 1 > hi) e1 = 0.0f;
          }
          if constexpr (C::kDV) pp[t / 2] = Pack<BF16>::two(e0, e1);
          if constexpr (C::kDK) {
            float g0, g1;
            f2_unpack(f2_mul(f2_pack(e0, e1), f2_add(f2_pack(dp[t], dp[t + 1]), nd[u / 2])), g0, g1);
            pd[t / 2] = Pack<BF16>::two(g0, g1);
          }
        }
        if constexpr (WDS) {
          if ((t4 & 1) && ds_on) {
            const int k = t4 >> 1;
            st_global_hint(ds_dst + k * (kDsChunk / 16),
                           make_uint4(pd[4 * k], pd[4 * k + 1], pd[4 * k + 2], pd[4 * k + 3]), ds_pol);
          }
        }
      }
      mbar_arrive(&ld_empty[st]);
      if (it > 0 && !mbar_wait_warp(&acc_done, (it - 1) & 1u, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < C::kHalf / 32; ++c) {
        uint32_t w16[16];
        if constexpr (C::kDV) {
#pragma unroll
          for (int t = 0; t < 16; ++t) w16[t] = pp[c * 16 + t];
          tmem_st16(tmem + lane_off + C::kTP + col0 / 2 + c * 16, w16);
        }
        if constexpr (C::kDK) {
#pragma unroll
          for (int t = 0; t < 16; ++t) w16[t] = pd[c * 16 + t];
          tmem_st16(tmem + lane_off + C::kTdS + col0 / 2 + c * 16, w16);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&pds_full);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n_it > 0) ok = mbar_wait_warp(&acc_done, (n_it - 1) & 1u, ab);
    if (ok) {
      tc_fence_after();
      const bool valid = j < sq.lk;
      const int64_t tok = (int64_t)sq.k_start + j;
      auto store = [&](void* base, int64_t sb, int64_t st_, int64_t sh, int tcol, int D,
                       float mul) {
        char* row = (char*)base + ((int64_t)b * sb + tok * st_ + (int64_t)g * sh) * (G_F32 ? 4 : 2);
        const int half = D / 2;
        for (int c = 0; c < half / 32; ++c) {
          const int col = wg * half + c * 32;
          uint32_t rr[32];
          if (n_it > 0) {
            tmem_ld32(tmem + lane_off + tcol + col, rr);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) rr[t] = 0u;
          }
          if (!valid) continue;
          if (G_F32) {
            float4* dst = reinterpret_cast<float4*>(row + col * 4);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              float4 w = make_float4(__uint_as_float(rr[4 * t]) * mul,
                                     __uint_as_float(rr[4 * t + 1]) * mul,
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
            uint4* dst = reinterpret_cast<uint4*>(row + col * 2);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              uint4 v;
              v.x = Pack<BF16>::two(__uint_as_float(rr[8 * t + 0]) * mul,
                                    __uint_as_float(rr[8 * t + 1]) * mul);
              v.y = Pack<BF16>::two(__uint_as_float(rr[8 * t + 2]) * mul,
                                    __uint_as_float(rr[8 * t + 3]) * mul);
              v.z = Pack<BF16>::two(__uint_as_float(rr[8 * t + 4]) * mul,
                                    __uint_as_float(rr[8 * t + 5]) * mul);
              v.w = Pack<BF16>::two(__uint_as_float(rr[8 * t + 6]) * mul,
                                    __uint_as_float(rr[8 * t + 7]) * mul);
              dst[t] = v;
            }
          }
        }
      };
      if (C::kDV) store(p.dv, p.sdv_b, p.sdv_t, p.sdv_h, C::kTdV, DV, 1.0f);
      if (C::kDK) store(p.dk, p.sdk_b, p.sdk_t, p.sdk_h, C::kTdK, DQK, p.scale);
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK, int DV, int BQ, int MODE, bool BF16, bool G_F32, bool WDS>
static cudaError_t launch_dkv_w(const DkvParams& p, cudaStream_t st) {
  using C = DkvCfg<DQK, DV, BQ, MODE>;
  auto k = attn_bwd_dkdv_kernel<DQK, DV, BQ, MODE, BF16, G_F32, WDS>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid = tile_major(p.n_ktiles) ? dim3((unsigned)p.n_ktiles, (unsigned)p.hkv, (unsigned)p.batch)
                                      : dim3((unsigned)p.hkv, (unsigned)p.n_ktiles, (unsigned)p.batch);
  k<<<grid, 384, C::kSmem, st>>>(p);
  return cudaGetLastError();
}

// the dS-writing variant where the dS path runs (p.ds set), else without it
template <int DQK, int DV, int BQ, int MODE, bool BF16, bool G_F32>
static cudaError_t launch_dkv_t(const DkvParams& p, cudaStream_t st) {
  if constexpr (DkvCfg<DQK, DV, BQ, MODE>::kCanDs) {
    if (p.ds) return launch_dkv_w<DQK, DV, BQ, MODE, BF16, G_F32, true>(p, st);
  } else {
    if (p.ds) return cudaErrorInvalidValue;
  }
  return launch_dkv_w<DQK, DV, BQ, MODE, BF16, G_F32, false>(p, st);
}

template <int DQK, int DV, int BQ, int MODE>
static cudaError_t launch_dkv_d(const DkvParams& p, bool bf16, bool gf32, cudaStream_t st) {
  if (bf16)
    return gf32 ? launch_dkv_t<DQK, DV, BQ, MODE, true, true>(p, st)
                : launch_dkv_t<DQK, DV, BQ, MODE, true, false>(p, st);
  return gf32 ? launch_dkv_t<DQK, DV, BQ, MODE, false, true>(p, st)
              : launch_dkv_t<DQK, DV, BQ, MODE, false, false>(p, st);
}

// Query-tile rows streamed by the dK/dV kernel(s) and the launches needed.
// Returns the number of launches (0 if unsupported); bq[i] / mode[i] describe each.
int dkv_plan(int dqk, int dv, int* bq, int* mode) {
  if (dqk == 64 && dv == 64) { bq[0] = 128; mode[0] = 3; return 1; }
  if (dqk == 128 && dv == 128) { bq[0] = 64; mode[0] = 3; return 1; }
  if (dqk == 192 && dv == 128) { bq[0] = 64; mode[0] = 3; return 1; }
  if (dqk == 256 && dv == 256) { bq[0] = 128; mode[0] = 1; bq[1] = 64; mode[1] = 2; return 2; }
  return 0;
}

cudaError_t launch_dkv(const DkvParams& p, int dqk, int dv, int mode, bool bf16, bool gf32,
                       cudaStream_t st) {
  if (dqk == 64 && dv == 64 && mode == 3) return launch_dkv_d<64, 64, 128, 3>(p, bf16, gf32, st);
  if (dqk == 128 && dv == 128 && mode == 3) return launch_dkv_d<128, 128, 64, 3>(p, bf16, gf32, st);
  if (dqk == 192 && dv == 128 && mode == 3) return launch_dkv_d<192, 128, 64, 3>(p, bf16, gf32, st);
  if (dqk == 256 && dv == 256 && mode == 1) return launch_dkv_d<256, 256, 128, 1>(p, bf16, gf32, st);
  if (dqk == 256 && dv == 256 && mode == 2) return launch_dkv_d<256, 256, 64, 2>(p, bf16, gf32, st);
  return cudaErrorNotSupported;
}

}  // namespace attn
