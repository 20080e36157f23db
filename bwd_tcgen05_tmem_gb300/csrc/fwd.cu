// fwd.cu -- fused attention forward on tcgen05 / TMEM / TMA (sm_103a).
//
// Computes O = softmax(scale * Q K^T + mask) V and the natural-log LSE per
// query row with an online (running-maximum) softmax over key tiles
// (TransformerEngine PR #3527: the forward saves a natural-log logsumexp in
// FP32; PR #3510: causal FP16/BF16 attention on Blackwell).
//
// One CTA owns 128 query rows of one (sequence, query head) and, for head dim
// 512, one half of the value columns.  Warp roles (256 threads):
//   warp 0      TMA producer: Q once, then K chunks (ring) and V tiles (stages)
//   warp 1      TMEM allocator and S-MMA issuer
//   warp 2      PV-MMA issuer
//   (warps 0-2 run their loops on all 32 lanes and issue each copy, MMA and
//   commit from an elect.sync lane)
//   warps 4..7  softmax: one TMEM lane (= query row) per thread; rescales O
//               in TMEM when the running maximum grows, writes P (16-bit)
//               into TMEM, and runs the epilogue.
// TMEM columns: kSB S buffers of 128 columns (P overwrites the first 64
// columns of its S buffer), then the O accumulator.  Three S buffers when O
// is at most 128 columns wide: S(j+2) can then start before PV(j) finishes.
// MMAs: S = Q K^T   SS, both K-major (128 x 128 x DQK)
//       O += P V    TS, A = P from TMEM, B = V chunk (MN-major), N = 64 each.
#include "kcommon.cuh"

namespace attn {

template <int DQK, int DV_CTA, bool BF16, bool O_F32>
struct FwdCfg {
  static constexpr int kQSlots = DQK / 64;
  static constexpr int kKCh = DQK / 64;    // K tile = kKCh 64-column chunks (K-major)
  static constexpr int kVCh = DV_CTA / 64;  // V tile = kVCh chunks, kept contiguous
  // V tiles live in whole stages so that one MMA covers all DV_CTA columns
  // (the B operand is MN-major and spans the chunks through LBO); K chunks go
  // through their own ring since the S MMA consumes them one chunk at a time.
  static constexpr int kVStages = (kQSlots + 2 * kVCh + 2 <= kMaxSlots) ? 2 : 1;
  static constexpr int kKRingRaw = kMaxSlots - kQSlots - kVStages * kVCh;
  static constexpr int kKRing = kKRingRaw > 16 ? 16 : kKRingRaw;
  // Where Q leaves too little room for a K ring of two tiles next to the V
  // stages (head dims 256 and 512: a K tile is 64-128 KB), K and V stream
  // through one ring of slot pairs instead (32 KB each, two 64-column chunks):
  // every slot beyond Q serves whichever operand the MMAs need next.  A K pair
  // feeds 8 S MMAs, a V pair one N = 128 half of the PV product.
  static constexpr bool kPR = kKRingRaw < 2 * kKCh;
  static constexpr int kPairs = (kMaxSlots - kQSlots) / 2;
  static constexpr int kKP = kKCh / 2;  // K pairs per key tile
  static constexpr int kVP = kVCh / 2;  // V pairs per key tile
  static constexpr int kSmem =
      (kPR ? kQSlots + 2 * kPairs : kQSlots + kVStages * kVCh + kKRing) * kSlotBytes + 1024;
  static_assert(!kPR || (kKCh % 2 == 0 && kVCh % 2 == 0 && kPairs >= 2), "pair ring");
  static constexpr int kSB = DV_CTA <= 128 ? 3 : 2;  // S buffers
  static constexpr int kTmemO = 128 * kSB;
  static_assert(kTmemO + DV_CTA <= 512, "TMEM budget");
  static_assert(DQK % 64 == 0 && DV_CTA % 64 == 0 && DV_CTA <= 256, "head dim");
  static_assert(kKRing >= 2, "ring");
};

template <int DQK, int DV_CTA, bool BF16, bool O_F32>
__global__ void __launch_bounds__(256, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<DQK, DV_CTA, BF16, O_F32>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem;
  uint8_t* sV = smem + C::kQSlots * kSlotBytes;
  uint8_t* sK = sV + C::kVStages * C::kVCh * kSlotBytes;

  __shared__ uint64_t kfull[C::kKRing], kempty[C::kKRing], vfull[C::kVStages], vempty[C::kVStages];
  // pair ring (kPR): one empty barrier per pair, and a full barrier per pair
  // and consumer -- each issuer waits only on loads meant for it, so its parity
  // wait can never match an older, still pending load of the other issuer
  constexpr int kNP = C::kPR ? C::kPairs : 1;
  __shared__ uint64_t pempty[kNP], pfull_k[kNP], pfull_v[kNP];
  uint8_t* sRing = smem + C::kQSlots * kSlotBytes;  // kPR: pair s at sRing + s * 2 slots
  // o_done[b]: PV of the key tiles that used S buffer b (one phase per use)
  __shared__ uint64_t q_bar, s_full[C::kSB], p_full[C::kSB], o_done[C::kSB], drain_bar, drain_bar2;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag, skip_sh;

  const int warp = threadIdx.x >> 5;
  // (query tile, head x column split) in the grid order of tile_major()
  const bool tmaj = tile_major(p.n_qtiles);
  const int hs = tmaj ? blockIdx.y : blockIdx.x;
  const int split = hs % p.n_split;
  const int h = hs / p.n_split;
  const int tile = p.n_qtiles - 1 - (tmaj ? blockIdx.x : blockIdx.y);
  const int b = blockIdx.z;
  const int tb = p.geo.cu_q ? 0 : b;  // TMA batch coordinate (packed THD tensors have one)
  const int g = h / (p.hq / p.hkv);

  const Seq sq = load_seq(p.geo, b);
  const int q0 = tile * kBlockM;
  if (q0 >= sq.lq) return;  // tile past the end of this sequence (uniform)
  long long j0, j1;
  key_range(sq, q0, min(q0 + kBlockM, sq.lq) - 1, j0, j1);
  const int kt0 = (j1 >= j0) ? (int)(j0 / kBlockN) : 0;
  const int n_kv = (j1 >= j0) ? (int)(j1 / kBlockN) - kt0 + 1 : 0;

  const unsigned long long lim = wait_limit(p.dbg);
  const int drop = dropped_load(p.dbg);
  Abort ab{&abort_flag, p.status, lim};
  if (threadIdx.x == 0) {
    // A failed device check (cu_seqlens) or an earlier abort stops every CTA.
    // The status word is loaded first and tested only after the barriers are
    // set up and Q's copy is under way: Q heads the critical path, and a
    // tensor-map copy stays in bounds whatever the sequence metadata says.
    const int status = p.status ? *(volatile int*)p.status : 0;
    abort_flag = 0;
    for (int i = 0; i < C::kKRing; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
    }
    for (int i = 0; i < kNP; ++i) {
      mbar_init(&pempty[i], 1);
      mbar_init(&pfull_k[i], 1);
      mbar_init(&pfull_v[i], 1);
    }
    mbar_init(&q_bar, 1);
    for (int i = 0; i < C::kSB; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(&drain_bar, 1);
    mbar_init(&drain_bar2, 1);
    fence_barrier_init();
    if (n_kv > 0) {
      int c1, c2, c3;
      map_coords(p.oq, 0, h, sq.q_start + q0, tb, c1, c2, c3);
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_tx(&q_bar, C::kQSlots * kSlotBytes);
      for (int c = 0; c < C::kQSlots; ++c)
        tma_load_4d(sQ + c * kSlotBytes, &p.tm_q, &q_bar, c * 64, c1, c2, c3);
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
  if (skip_sh) {  // let Q's copy land, free TMEM, leave
    if (threadIdx.x == 0 && n_kv > 0) mbar_wait_quiet(&q_bar, 0, lim);
    if (warp == 1) tmem_dealloc(tmem, 512);
    return;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // load order = MMA order: K0, K1, V0, K2, V1, ..., K(n-1), V(n-2), V(n-1)
    // (Q was issued with the barrier set-up); the whole warp runs the loop
    // (indices stay warp-uniform); one elected lane issues the copies
    if (n_kv > 0) {
      uint32_t kcnt = 0;
      int vcnt = 0;
      bool ok = true;
      auto load_k = [&](int jt) {
        int d1, d2, d3;
        map_coords(p.ok, 0, g, sq.k_start + (kt0 + jt) * kBlockN, tb, d1, d2, d3);
#pragma unroll
        for (int c = 0; c < C::kKCh; ++c, ++kcnt) {
          const uint32_t slot = kcnt % C::kKRing;
          if (!mbar_wait_warp(&kempty[slot], ((kcnt / C::kKRing) & 1u) ^ 1u, ab)) {
            ok = false;
            return;
          }
          if (elect_sync()) {
            mbar_arrive_tx(&kfull[slot], kSlotBytes);
            tma_load_4d(sK + slot * kSlotBytes, &p.tm_k, &kfull[slot], c * 64, d1, d2, d3);
          }
          __syncwarp();
        }
      };
      auto load_v = [&](int jt) {
        int d1, d2, d3;
        map_coords(p.ov, 0, g, sq.k_start + (kt0 + jt) * kBlockN, tb, d1, d2, d3);
        const int st = vcnt % C::kVStages;
        if (!mbar_wait_warp(&vempty[st], ((vcnt / C::kVStages) & 1) ^ 1, ab)) {
          ok = false;
          return;
        }
        if (vcnt != drop && elect_sync()) {  // drop: test-only injected missing load
          mbar_arrive_tx(&vfull[st], C::kVCh * kSlotBytes);
#pragma unroll
          for (int c = 0; c < C::kVCh; ++c)
            tma_load_4d(sV + (st * C::kVCh + c) * kSlotBytes, &p.tm_v, &vfull[st],
                        split * DV_CTA + c * 64, d1, d2, d3);
        }
        __syncwarp();
        ++vcnt;
      };
      if constexpr (!C::kPR) {
        load_k(0);
        for (int jt = 0; jt < n_kv && ok; ++jt) {
          if (jt + 1 < n_kv) load_k(jt + 1);
          if (ok) load_v(jt);
        }
      } else {
        // pair ring: the same order (K0, K1, V0, K2, V1, ...) at pair granularity.
        // Per slot: which consumer the last load was for and the parity it
        // completes, to let copies in flight land before the CTA exits.
        uint32_t L = 0, kpar = 0, vpar = 0, lastk = 0, lastpar = 0, used = 0;
        auto load_pair = [&](bool is_k, int jt, int pp) {
          const uint32_t slot = L % C::kPairs;
          if (!mbar_wait_warp(&pempty[slot], ((L / C::kPairs) & 1u) ^ 1u, ab)) {
            ok = false;
            return;
          }
          const uint32_t bit = 1u << slot;
          const uint32_t par = ((is_k ? kpar : vpar) & bit) ? 1u : 0u;
          if (is_k) kpar ^= bit; else vpar ^= bit;
          lastk = is_k ? (lastk | bit) : (lastk & ~bit);
          lastpar = par ? (lastpar | bit) : (lastpar & ~bit);
          used |= bit;
          uint64_t* full = is_k ? &pfull_k[slot] : &pfull_v[slot];
          int d1, d2, d3;
          map_coords(is_k ? p.ok : p.ov, 0, g, sq.k_start + (kt0 + jt) * kBlockN, tb, d1, d2, d3);
          uint8_t* dst = sRing + slot * 2 * kSlotBytes;
          // drop: test-only injected missing load (the first V pair of tile `drop`)
          if (!(!is_k && pp == 0 && jt == drop) && elect_sync()) {
            mbar_arrive_tx(full, 2 * kSlotBytes);
            for (int c = 0; c < 2; ++c) {
              if (is_k)
                tma_load_4d(dst + c * kSlotBytes, &p.tm_k, full, (2 * pp + c) * 64, d1, d2, d3);
              else
                tma_load_4d(dst + c * kSlotBytes, &p.tm_v, full,
                            split * DV_CTA + (2 * pp + c) * 64, d1, d2, d3);
            }
          }
          __syncwarp();
          ++L;
        };
        for (int pp = 0; pp < C::kKP && ok; ++pp) load_pair(true, 0, pp);
        for (int jt = 0; jt < n_kv && ok; ++jt) {
          if (jt + 1 < n_kv)
            for (int pp = 0; pp < C::kKP && ok; ++pp) load_pair(true, jt + 1, pp);
          for (int pp = 0; pp < C::kVP && ok; ++pp) load_pair(false, jt, pp);
        }
        for (int sl = 0; sl < C::kPairs; ++sl)
          if (used & (1u << sl))
            mbar_wait_quiet((lastk >> sl) & 1u ? &pfull_k[sl] : &pfull_v[sl],
                            (lastpar >> sl) & 1u, lim);
      }
      // let every copy still in flight land before the CTA can exit
      mbar_wait_quiet(&q_bar, 0, lim);
      if constexpr (!C::kPR) {
        const uint32_t first = kcnt > (uint32_t)C::kKRing ? kcnt - C::kKRing : 0u;
        for (uint32_t c = first; c < kcnt; ++c)
          mbar_wait_quiet(&kfull[c % C::kKRing], (c / C::kKRing) & 1u, lim);
        for (int v = vcnt > C::kVStages ? vcnt - C::kVStages : 0; v < vcnt; ++v)
          mbar_wait_quiet(&vfull[v % C::kVStages], (v / C::kVStages) & 1, lim);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // warp 1 issues S = Q K^T, warp 2 issues O += P V: each blocks on its own
    // barriers while the other keeps the tensor pipe fed.  Descriptors are
    // built once; per MMA only small constant offsets are added (the
    // start-address field counts 16-byte units).  The whole warp runs the
    // loop; the elected lane issues every MMA and commit.
    if (n_kv > 0) {
      const bool s_role = warp == 1;
      constexpr uint32_t idesc_s = make_idesc(128, 128, BF16, false, false);
      constexpr uint32_t idesc_o = make_idesc(128, DV_CTA, BF16, false, true);
      const uint64_t qdesc = make_sdesc(smem_u32(sQ), 16, 1024);
      const uint64_t kdesc = make_sdesc(smem_u32(sK), 16, 1024);
      const uint64_t vdesc = make_sdesc(smem_u32(sV), kSlotBytes, 1024);
      uint32_t kcnt = 0;
      bool ok = s_role ? mbar_wait_warp(&q_bar, 0, ab) : true;
      tc_fence_after();
      auto issue_s = [&](int jt) {
        const uint32_t d = tmem + (uint32_t)((jt % C::kSB) * 128);
#pragma unroll
        for (int c = 0; c < C::kKCh; ++c, ++kcnt) {
          const uint32_t slot = kcnt % C::kKRing;
          if (!mbar_wait_warp(&kfull[slot], (kcnt / C::kKRing) & 1u, ab)) {
            ok = false;
            return;
          }
          tc_fence_after();
          const uint64_t qa = qdesc + (uint64_t)(c * (kSlotBytes >> 4));
          const uint64_t kb = kdesc + (uint64_t)(slot * (kSlotBytes >> 4));
          if (elect_sync()) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(d, qa + 2 * k, kb + 2 * k, idesc_s, (c | k) ? 1u : 0u);
            mma_commit(&kempty[slot]);
            if (c == C::kKCh - 1) mma_commit(&s_full[jt % C::kSB]);
          }
          __syncwarp();
        }
      };
      auto issue_pv = [&](int jt) {
        if (!mbar_wait_warp(&p_full[jt % C::kSB], (jt / C::kSB) & 1u, ab)) {
          ok = false;
          return;
        }
        const int st = jt % C::kVStages;
        if (!mbar_wait_warp(&vfull[st], (jt / C::kVStages) & 1, ab)) {
          ok = false;
          return;
        }
        tc_fence_after();
        const uint32_t pa = tmem + (uint32_t)((jt % C::kSB) * 128);
        const uint64_t vb = vdesc + (uint64_t)(st * C::kVCh * (kSlotBytes >> 4));
        if (elect_sync()) {
          mma_ts(tmem + C::kTmemO, pa, vb, idesc_o, jt > 0 ? 1u : 0u);
#pragma unroll
          for (int k = 1; k < 8; ++k)
            mma_ts(tmem + C::kTmemO, pa + k * 8, vb + k * 128, idesc_o, 1u);
          mma_commit(&vempty[st]);
          mma_commit(&o_done[jt % C::kSB]);
        }
        __syncwarp();
      };
      // pair ring: a load's position in the producer's sequence fixes its slot
      //   K(j) pair p: j == 0 ? p : kKP + (j - 1)(kKP + kVP) + p
      //   V(j) pair p: kKP + j (kKP + kVP) + (j + 1 < n_kv ? kKP : 0) + p
      const uint64_t rdesc = make_sdesc(smem_u32(sRing), 16, 1024);              // K-major
      const uint64_t rdesc_mn = make_sdesc(smem_u32(sRing), kSlotBytes, 1024);   // MN-major
      constexpr uint32_t idesc_o2 = make_idesc(128, 128, BF16, false, true);
      uint32_t rpar = 0;  // per slot: parity of this issuer's next wait on it
      auto issue_s_pr = [&](int jt) {
        const uint32_t d = tmem + (uint32_t)((jt % C::kSB) * 128);
        for (int pp = 0; pp < C::kKP; ++pp) {
          const uint32_t L = jt == 0 ? (uint32_t)pp
                                     : (uint32_t)(C::kKP + (jt - 1) * (C::kKP + C::kVP) + pp);
          const uint32_t slot = L % C::kPairs;
          if (!mbar_wait_warp(&pfull_k[slot], (rpar >> slot) & 1u, ab)) {
            ok = false;
            return;
          }
          rpar ^= 1u << slot;
          tc_fence_after();
          const uint64_t kb = rdesc + (uint64_t)((slot * 2 * kSlotBytes) >> 4);
          if (elect_sync()) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint64_t qa = qdesc + (uint64_t)((2 * pp + c) * (kSlotBytes >> 4));
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_ss(d, qa + 2 * k, kb + (uint64_t)(c * (kSlotBytes >> 4)) + 2 * k, idesc_s,
                       (pp | c | k) ? 1u : 0u);
            }
            mma_commit(&pempty[slot]);
            if (pp == C::kKP - 1) mma_commit(&s_full[jt % C::kSB]);
          }
          __syncwarp();
        }
      };
      auto issue_pv_pr = [&](int jt) {
        if (!mbar_wait_warp(&p_full[jt % C::kSB], (jt / C::kSB) & 1u, ab)) {
          ok = false;
          return;
        }
        const uint32_t pa = tmem + (uint32_t)((jt % C::kSB) * 128);
        for (int pp = 0; pp < C::kVP; ++pp) {
          const uint32_t L = (uint32_t)(C::kKP + jt * (C::kKP + C::kVP) +
                                        (jt + 1 < n_kv ? C::kKP : 0) + pp);
          const uint32_t slot = L % C::kPairs;
          if (!mbar_wait_warp(&pfull_v[slot], (rpar >> slot) & 1u, ab)) {
            ok = false;
            return;
          }
          rpar ^= 1u << slot;
          tc_fence_after();
          const uint64_t vb = rdesc_mn + (uint64_t)((slot * 2 * kSlotBytes) >> 4);
          if (elect_sync()) {  // O columns [128 pp, 128 pp + 128) += P V_pair
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ts(tmem + C::kTmemO + pp * 128, pa + k * 8, vb + k * 128, idesc_o2,
                     (jt > 0 || k > 0) ? 1u : 0u);
            mma_commit(&pempty[slot]);
            if (pp == C::kVP - 1) mma_commit(&o_done[jt % C::kSB]);
          }
          __syncwarp();
        }
      };
      if (s_role) {
        for (int jt = 0; jt < n_kv && ok; ++jt) {
          // S buffer jt%kSB last held P(jt-kSB): wait until PV(jt-kSB) has read it
          if (jt >= C::kSB &&
              !mbar_wait_warp(&o_done[jt % C::kSB], ((jt - C::kSB) / C::kSB) & 1u, ab))
            break;
          if constexpr (C::kPR) issue_s_pr(jt); else issue_s(jt);
        }
      } else {
        for (int jt = 0; jt < n_kv && ok; ++jt) {
          if constexpr (C::kPR) issue_pv_pr(jt); else issue_pv(jt);
        }
      }
      uint64_t* drain = s_role ? &drain_bar : &drain_bar2;
      if (elect_sync()) {
        mma_commit(drain);
        mbar_wait_quiet(drain, 0, lim);
      }
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int wq = warp - 4;
    const int r = wq * 32 + (threadIdx.x & 31);
    const int i = q0 + r;  // query row within the sequence
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.0f;
    const long long vis_lo = (long long)i + sq.off - sq.L;  // first visible key
    long long vis_hi = (long long)i + sq.off + sq.R;        // last visible key
    if (vis_hi > sq.lk - 1) vis_hi = sq.lk - 1;
    // rows that see every key of a tile need no per-element mask; decide per tile
    const long long rows_last = min(q0 + kBlockM, sq.lq) - 1;
    bool ok = true;
    for (int jt = 0; jt < n_kv; ++jt) {
      const int k0 = (kt0 + jt) * kBlockN;
      if (!mbar_wait_warp(&s_full[jt % C::kSB], (jt / C::kSB) & 1u, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sb = tmem + lane_off + (uint32_t)((jt % C::kSB) * 128);
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t rr[32];
        tmem_ld32(sb + c * 32, rr);
#pragma unroll
        for (int t = 0; t < 32; ++t) s[c * 32 + t] = __uint_as_float(rr[t]);
      }
      tmem_ld_wait();
      const bool full_tile = (k0 + kBlockN - 1 <= sq.lk - 1) &&
                             ((long long)k0 >= rows_last + sq.off - sq.L) &&
                             ((long long)(k0 + kBlockN - 1) <= (long long)q0 + sq.off + sq.R);
      if (!full_tile) {
        const long long lo = vis_lo - k0, hi = vis_hi - k0;
#pragma unroll
        for (int t = 0; t < 128; ++t)
          if (t < lo || t > hi) s[t] = -INFINITY;
      }
      // exp2(s * scale * log2 e - m) and the row sum in packed pairs (eight
      // sum chains, element t into chain t % 8, as four pairs); P is stored
      // into the first half of the S buffer
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      auto exps = [&](float neg_m) -> float {
        const uint64_t negm2 = f2_pack(neg_m, neg_m);
        uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[c * 32 + 2 * t], s[c * 32 + 2 * t + 1]), sl2x2, negm2),
                      x0, x1);
            const float e0 = ex2(x0), e1 = ex2(x1);
            acc2[t & 3] = f2_add(acc2[t & 3], f2_pack(e0, e1));
            pk[t] = Pack<BF16>::two(e0, e1);
          }
          tmem_st16(sb + c * 16, pk);
        }
        float rsv[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) f2_unpack(acc2[u], rsv[2 * u], rsv[2 * u + 1]);
        return ((rsv[0] + rsv[1]) + (rsv[2] + rsv[3])) + ((rsv[4] + rsv[5]) + (rsv[6] + rsv[7]));
      };
      // The softmax warps are bound by instruction issue, so the tile's row
      // maximum is computed only when needed: against the running maximum a
      // row sum of at most 2^7 bounds every exponential by 2^7, so the maximum
      // has not grown by the 2^8 that triggers a rescale, and P and the sum
      // are exactly what the full computation gives.  Otherwise (a row's
      // first keys, or a larger sum in any row of the warp) the warp computes
      // the maximum and the exponentials again.
      float rs = 0.0f, alpha = 1.0f;
      bool grow = false;
      bool need_max = __any_sync(0xffffffffu, m_run == -INFINITY);
      if (!need_max) {
        rs = exps(-m_run);
        need_max = __any_sync(0xffffffffu, !(rs <= 128.0f));
      }
      if (need_max) {
        // row maximum as 8 independent chains (one warp per sub-partition has
        // no other warp to hide a 128-long dependency chain), two elements per
        // three-input max
        float mxv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mxv[u] = s[u];
#pragma unroll
        for (int t = 8; t < 120; t += 16)
#pragma unroll
          for (int u = 0; u < 8; ++u) mxv[u] = fmax3(mxv[u], s[t + u], s[t + 8 + u]);
#pragma unroll
        for (int u = 0; u < 8; ++u) mxv[u] = fmaxf(mxv[u], s[120 + u]);
        const float mx = fmaxf(fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3])),
                               fmaxf(fmaxf(mxv[4], mxv[5]), fmaxf(mxv[6], mxv[7])));
        const float m_tile = mx * sl2;
        grow = m_tile > m_run + 8.0f;
        const float m_new = grow ? m_tile : m_run;
        alpha = grow ? ex2(m_run - m_new) : 1.0f;
        m_run = m_new;
        rs = exps((m_run == -INFINITY) ? 0.0f : -m_run);
      }
      l_run = l_run * alpha + rs;
      // rescale O rows whose maximum grew (after PV(jt-1) has finished)
      if (__any_sync(0xffffffffu, grow && jt > 0)) {
        if (!mbar_wait_warp(&o_done[(jt - 1) % C::kSB], ((jt - 1) / C::kSB) & 1u, ab)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < DV_CTA / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_off + C::kTmemO + c * 32, rr);
          tmem_ld_wait();
          uint32_t lo16[16], hi16[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            lo16[t] = __float_as_uint(__uint_as_float(rr[t]) * alpha);
            hi16[t] = __float_as_uint(__uint_as_float(rr[16 + t]) * alpha);
          }
          tmem_st16(tmem + lane_off + C::kTmemO + c * 32, lo16);
          tmem_st16(tmem + lane_off + C::kTmemO + c * 32 + 16, hi16);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[jt % C::kSB]);
    }
    // ------------------------------------------------------------ epilogue
    // the last PV of every S buffer, in order (each barrier is at most one
    // phase behind: S(n-1) already waited for PV(n-1-kSB))
    for (int t = n_kv > C::kSB ? n_kv - C::kSB : 0; t < n_kv && ok; ++t)
      ok = mbar_wait_warp(&o_done[t % C::kSB], (t / C::kSB) & 1u, ab);
    if (ok) {
      tc_fence_after();
      const bool valid = i < sq.lq;
      const bool keyless = !(l_run > 0.0f);
      const float inv_l = keyless ? 0.0f : 1.0f / l_run;
      const int64_t tok = (int64_t)sq.q_start + i;
      if (valid && split == 0)
        p.lse[(int64_t)b * p.lse_sb + (int64_t)h * p.lse_sh + tok] =
            keyless ? -INFINITY : (m_run + __log2f(l_run)) * 0.69314718055994530942f;
      char* orow = (char*)p.o +
                   ((int64_t)b * p.so_b + tok * p.so_t + (int64_t)h * p.so_h +
                    (int64_t)split * DV_CTA) *
                       (O_F32 ? 4 : 2);
#pragma unroll
      for (int c = 0; c < DV_CTA / 32; ++c) {
        uint32_t rr[32];
        if (n_kv > 0) {
          tmem_ld32(tmem + lane_off + C::kTmemO + c * 32, rr);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) rr[t] = 0u;
        }
        if (valid) {
          if (O_F32) {
            float4* dst = reinterpret_cast<float4*>(orow + c * 32 * 4);
#pragma unroll
            for (int t = 0; t < 8; ++t)
              dst[t] = make_float4(__uint_as_float(rr[4 * t]) * inv_l,
                                   __uint_as_float(rr[4 * t + 1]) * inv_l,
                                   __uint_as_float(rr[4 * t + 2]) * inv_l,
                                   __uint_as_float(rr[4 * t + 3]) * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32 * 2);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              uint4 v;
              v.x = Pack<BF16>::two(__uint_as_float(rr[8 * t + 0]) * inv_l,
                                    __uint_as_float(rr[8 * t + 1]) * inv_l);
              v.y = Pack<BF16>::two(__uint_as_float(rr[8 * t + 2]) * inv_l,
                                    __uint_as_float(rr[8 * t + 3]) * inv_l);
              v.z = Pack<BF16>::two(__uint_as_float(rr[8 * t + 4]) * inv_l,
                                    __uint_as_float(rr[8 * t + 5]) * inv_l);
              v.w = Pack<BF16>::two(__uint_as_float(rr[8 * t + 6]) * inv_l,
                                    __uint_as_float(rr[8 * t + 7]) * inv_l);
              dst[t] = v;
            }
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

// ----------------------------------------------------------------- launch
template <int DQK, int DV_CTA, bool BF16, bool O_F32>
static cudaError_t launch_fwd_t(const FwdParams& p, dim3 grid, cudaStream_t st) {
  using C = FwdCfg<DQK, DV_CTA, BF16, O_F32>;
  auto k = attn_fwd_kernel<DQK, DV_CTA, BF16, O_F32>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  k<<<grid, 256, C::kSmem, st>>>(p);
  return cudaGetLastError();
}

template <int DQK, int DV_CTA>
static cudaError_t launch_fwd_d(const FwdParams& p, dim3 grid, bool bf16, bool of32,
                                cudaStream_t st) {
  if (bf16)
    return of32 ? launch_fwd_t<DQK, DV_CTA, true, true>(p, grid, st)
                : launch_fwd_t<DQK, DV_CTA, true, false>(p, grid, st);
  return of32 ? launch_fwd_t<DQK, DV_CTA, false, true>(p, grid, st)
              : launch_fwd_t<DQK, DV_CTA, false, false>(p, grid, st);
}

// Returns cudaErrorNotSupported for head dims without an instantiation.
cudaError_t launch_fwd(const FwdParams& p, int dqk, int dv, bool bf16, bool o_f32,
                       cudaStream_t st) {
  const int nsplit = dv > 256 ? dv / 256 : 1;
  if (p.n_split != nsplit) return cudaErrorInvalidValue;
  dim3 grid = tile_major(p.n_qtiles)
                  ? dim3((unsigned)p.n_qtiles, (unsigned)(p.hq * nsplit), (unsigned)p.batch)
                  : dim3((unsigned)(p.hq * nsplit), (unsigned)p.n_qtiles, (unsigned)p.batch);
  if (dqk == 64 && dv == 64) return launch_fwd_d<64, 64>(p, grid, bf16, o_f32, st);
  if (dqk == 128 && dv == 128) return launch_fwd_d<128, 128>(p, grid, bf16, o_f32, st);
  if (dqk == 192 && dv == 128) return launch_fwd_d<192, 128>(p, grid, bf16, o_f32, st);
  if (dqk == 256 && dv == 256) return launch_fwd_d<256, 256>(p, grid, bf16, o_f32, st);
  if (dqk == 512 && dv == 512) return launch_fwd_d<512, 256>(p, grid, bf16, o_f32, st);
  return cudaErrorNotSupported;
}

}  // namespace attn
