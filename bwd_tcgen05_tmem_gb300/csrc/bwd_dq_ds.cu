// bwd_dq_ds.cu -- dQ GEMM of the dS backward path (tcgen05 / TMEM / TMA).
//
// dQ_i = scale * sum_kb dS_{i,kb} K_kb  for the 128-row query tiles i of one
// (sequence, query head), over their visible 128-key blocks kb, with the dS
// blocks the key-stationary dK/dV kernel wrote (layout in bwd.h) and K from
// the caller's tensor (TransformerEngine PR #3510 backward chain: dQ = dS K;
// PR #3699: the helper chain around it).  Every dQ element is produced by one
// CTA, accumulated in TMEM in key-block order, so the result is bitwise
// reproducible.
//
// A work item is a pair of adjacent query tiles (2t, 2t+1) of one (sequence,
// query head): per key block the CTA copies the K tile in once and multiplies
// it into the accumulators of both tiles.  What bounds the GEMM is what each
// SM takes in rather than HBM: per key block 32 KiB of dS from HBM and, at
// DQK = 192, 48 KiB of K from L2.  Timing-only copies of a one-tile-per-item
// form of this kernel on GB300 at 32K took 6.45 ms in full, 5.61 ms without
// the MMAs and 4.92 ms without the K copies as well (the bare dS stream at
// 7.1 TB/s); a pair takes in 112 KiB per two blocks instead of 160, and took
// that GEMM to 5.56 ms (same GPU, bit-identical dQ).
//
// Four dS stages keep up to 128 KiB in flight per SM; the kernel is
// persistent, so the stream does not pause between items.  dS and K have
// producers of their own (three 32 KiB K stages at DQK = 128, two 48 KiB ones
// at 192), so the dS copies run up to four blocks ahead of the MMAs (with one
// producer issuing each block's dS and then its K copy the 32K GEMM took
// 5.54 instead of 5.41 ms, same GPU).  TMEM holds two accumulator pairs at
// DQK = 128 (an item's epilogue overlaps the next item's MMAs) and one at
// DQK = 192 (two 192-column accumulators in the 512 columns).
//
// Warp roles (224 threads): warp 0 dS producer (it also takes the items from
// the work queue), warp 1 TMEM owner and MMA issuer, warps 2..5 epilogue (TMEM
// lane quarter warp & 3), warp 6 K producer.  MMA per K-step of 16 keys: M = 128 queries, N = DQK, A = dS
// (MN-major, unswizzled: 8-query groups SBO = 2 KiB apart, 8-key groups LBO =
// 128 bytes apart), B = K (MN-major: head-dim contiguous, 128-byte swizzle,
// 64-column chunks LBO apart).
#include "bwd.h"

namespace attn {

template <int DQK>
struct DqDsCfg {
  static constexpr int kKCh = DQK / 64;
  static constexpr int kKTile = kKCh * kSlotBytes;  // 128 keys x DQK
  static constexpr int kDsStages = 4;
  static constexpr int kBudget = 232448 - 1024 - 512;
  static constexpr int kKStagesRaw = (kBudget - kDsStages * kDsBlock) / kKTile;
  static constexpr int kKStages = kKStagesRaw > 4 ? 4 : kKStagesRaw;
  static constexpr int kSmem = kDsStages * kDsBlock + kKStages * kKTile + 1024;
  static constexpr int kTileCols = DQK <= 128 ? 128 : 256;  // TMEM columns of one tile's dQ
  static constexpr int kTmemCols = 512;
  static constexpr int kAccBufs = 4 * kTileCols <= kTmemCols ? 2 : 1;  // accumulator pairs
  static constexpr int kThreads = 224;
  static_assert(DQK % 64 == 0 && DQK <= 256, "head dim");
  static_assert(kKStages >= 2, "K stages");
};

template <int DQK, bool BF16, bool G_F32>
__global__ void __launch_bounds__(DqDsCfg<DQK>::kThreads, 1) attn_bwd_dq_ds_kernel(const __grid_constant__ DqDsParams p) {
  using C = DqDsCfg<DQK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sDs = smem;
  uint8_t* sK = smem + C::kDsStages * kDsBlock;

  __shared__ uint64_t ds_full[C::kDsStages], ds_empty[C::kDsStages];
  __shared__ uint64_t k_full[C::kKStages], k_empty[C::kKStages];
  // accumulator pair b: acc_full[b] when an item's MMAs into it are done,
  // acc_free[b] when the epilogue has read it (one phase per use)
  __shared__ uint64_t acc_full[C::kAccBufs], acc_free[C::kAccBufs], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag, skip_sh;

  const int warp = threadIdx.x >> 5;
  // Persistent: one CTA per SM takes work items (pair of query tiles, query
  // head, sequence) from the work queue, in the order a one-CTA-per-item grid
  // had (tile_major(): the tile pairs of a head, heaviest first, then the
  // next head; otherwise the heads of a tile pair).
  const bool tmaj = tile_major(p.n_qtiles);
  const int n_pairs = (p.n_qtiles + 1) / 2;
  const int gx = tmaj ? n_pairs : p.hq, gy = tmaj ? p.hq : n_pairs;
  const int n_items = gx * gy * p.batch;  // the launch checks that it fits
  __shared__ ItemRing<4> iring;
  struct Item {
    Seq sq;
    int h, b, q0;        // q0: first query row of the pair's first tile
    int kb0[2], nkb[2];  // visible key blocks of each tile (none past the sequence)
    bool live[2];        // the tile lies inside its sequence
    int lo, hi;          // key blocks [lo, hi) that either tile sees
  };
  auto item = [&](int L) {
    Item it;
    const int x = L % gx;
    const int rest = L / gx;
    const int y = rest % gy;
    it.b = rest / gy;
    it.h = tmaj ? y : x;
    it.sq = load_seq(p.geo, it.b);
    const int qt = 2 * (n_pairs - 1 - (tmaj ? x : y));
    it.q0 = qt * kBlockM;
    it.lo = 0x7fffffff;
    it.hi = 0;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      it.live[u] = it.q0 + u * kBlockM < it.sq.lq;
      it.kb0[u] = 0;
      it.nkb[u] = it.live[u] ? wide_blocks_of_qtile(it.sq, qt + u, it.kb0[u]) : 0;
      if (it.nkb[u] > 0) {
        it.lo = min(it.lo, it.kb0[u]);
        it.hi = max(it.hi, it.kb0[u] + it.nkb[u]);
      }
    }
    if (it.hi == 0) it.lo = 0;  // no keys: an empty range
    return it;
  };
  // tile u of the item reads key block kb
  auto active = [](const Item& it, int u, int kb) {
    return kb >= it.kb0[u] && kb < it.kb0[u] + it.nkb[u];
  };

  const unsigned long long lim = wait_limit_all(p.dbg);
  Abort ab{&abort_flag, p.status, lim};
  if (threadIdx.x == 0) {
    const int status = p.status ? *(volatile int*)p.status : 0;
    abort_flag = 0;
    for (int i = 0; i < C::kDsStages; ++i) {
      mbar_init(&ds_full[i], 1);
      mbar_init(&ds_empty[i], 1);
    }
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < C::kAccBufs; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_free[i], 4);  // one arrival per epilogue warp
    }
    mbar_init(&drain_bar, 1);
    item_ring_init(iring, 6);  // consumers: MMA, four epilogue warps, K producer
    fence_barrier_init();
    tma_prefetch_desc(&p.tm_k);
    skip_sh = status != 0;
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (skip_sh) {
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
    return;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ dS producer
    // per key block the dS block of each tile that sees it (one 32 KiB bulk
    // copy each, read once: L2 evict-first); the whole warp runs the loop, one
    // elected lane issues the copies; the count runs over all items
    const uint64_t pol = l2_evict_first();
    bool ok = true;
    int nd = 0;  // dS copies issued
    for (int q = 0; ok; ++q) {
      const int li = item_ring_push(iring, q, p.counter, n_items, ab, ok);
      if (li < 0) break;
      const Item it = item(li);
      if (it.hi <= it.lo) continue;
      const int drop = li == 0 ? p.dbg.drop_load : -1;  // test-only injected missing dS copy
      const long long T_b = p.plan[it.b + 1] - p.plan[it.b];
      long long first[2];
      first[0] = (long long)p.hq * p.plan[it.b] + (long long)it.h * T_b +
                 blocks_row_prefix(it.sq, it.q0 / kBlockM);  // whole warp
      first[1] = first[0] + it.nkb[0];  // the next tile's blocks follow
      if (!(first[0] >= 0 && first[1] + it.nkb[1] <= p.cap)) {  // inconsistent plan
        if (elect_sync()) {
          raise_status(p.status, DEV_WORKSPACE);
          *(volatile int*)&abort_flag = 1;
        }
        __syncwarp();
        ok = false;
        break;
      }
      int jc = 0;  // dS copies of this item
      for (int kb = it.lo; kb < it.hi && ok; ++kb) {
        for (int u = 0; u < 2; ++u) {
          if (!active(it, u, kb)) continue;
          const int s = nd % C::kDsStages;
          if (!mbar_wait_warp(&ds_empty[s], ((nd / C::kDsStages) & 1) ^ 1, ab)) {
            ok = false;
            break;
          }
          if (jc != drop && elect_sync()) {
            mbar_arrive_tx(&ds_full[s], kDsBlock);
            bulk_load_hint(sDs + s * kDsBlock,
                           p.blocks + (size_t)(first[u] + (kb - it.kb0[u])) * kDsBlock, kDsBlock,
                           &ds_full[s], pol);
          }
          __syncwarp();
          ++nd;
          ++jc;
        }
      }
    }
    // let the copies in flight land before the CTA can exit
    for (int v = nd > C::kDsStages ? nd - C::kDsStages : 0; v < nd; ++v)
      mbar_wait_quiet(&ds_full[v % C::kDsStages], (v / C::kDsStages) & 1, lim);
  } else if (warp == 6) {
    // ------------------------------------------------------------ K producer
    // the K tile of every key block either tile sees, in the dS producer's
    // order
    bool ok = true;
    int nk = 0;  // K copies issued
    for (int q = 0; ok; ++q) {
      const int li = item_ring_pop(iring, q, ab, ok);
      if (li < 0) break;
      const Item it = item(li);
      if (it.hi <= it.lo) continue;
      const int g = it.h / (p.hq / p.hkv);
      const int tb = p.geo.cu_q ? 0 : it.b;
      for (int kb = it.lo; kb < it.hi && ok; ++kb) {
        if (!active(it, 0, kb) && !active(it, 1, kb)) continue;
        const int ks = nk % C::kKStages;
        if (!mbar_wait_warp(&k_empty[ks], ((nk / C::kKStages) & 1) ^ 1, ab)) {
          ok = false;
          break;
        }
        int c1, c2, c3;
        map_coords(p.ok, 0, g, it.sq.k_start + kb * kBlockN, tb, c1, c2, c3);
        if (elect_sync()) {
          mbar_arrive_tx(&k_full[ks], C::kKTile);
#pragma unroll
          for (int c = 0; c < C::kKCh; ++c)
            tma_load_4d(sK + ks * C::kKTile + c * kSlotBytes, &p.tm_k, &k_full[ks], c * 64, c1, c2, c3);
        }
        __syncwarp();
        ++nk;
      }
    }
    for (int v = nk > C::kKStages ? nk - C::kKStages : 0; v < nk; ++v)
      mbar_wait_quiet(&k_full[v % C::kKStages], (v / C::kKStages) & 1, lim);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // na counts the items with keys: accumulator pair na % kAccBufs, used for
    // the (na / kAccBufs)-th time; per key block the MMAs of each tile that
    // sees it share the block's K tile
    constexpr uint32_t idesc = make_idesc(128, DQK, BF16, true, true);
    const uint64_t adesc = make_sdesc_noswz(smem_u32(sDs), 128, kDsChunk);
    const uint64_t bdesc = make_sdesc(smem_u32(sK), kSlotBytes, 1024);
    bool ok = true;
    int nd = 0, nk = 0, na = 0;
    for (int q = 0; ok; ++q) {
      const int li = item_ring_pop(iring, q, ab, ok);
      if (li < 0) break;
      const Item it = item(li);
      if (it.hi <= it.lo) continue;
      const int buf = na % C::kAccBufs, use = na / C::kAccBufs;
      if (use > 0 && !mbar_wait_warp(&acc_free[buf], (use - 1) & 1u, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc0 = tmem + (uint32_t)(buf * 2 * C::kTileCols);
      bool started0 = false, started1 = false;
      for (int kb = it.lo; kb < it.hi && ok; ++kb) {
        int sd[2] = {-1, -1};  // dS stage of each tile's block, -1: the tile does not see kb
        for (int u = 0; u < 2; ++u) {
          if (!active(it, u, kb)) continue;
          const int s = nd % C::kDsStages;
          if (!mbar_wait_warp(&ds_full[s], (nd / C::kDsStages) & 1, ab)) {
            ok = false;
            break;
          }
          sd[u] = s;
          ++nd;
        }
        if (!ok) break;
        if (sd[0] < 0 && sd[1] < 0) continue;
        const int ks = nk % C::kKStages;
        if (!mbar_wait_warp(&k_full[ks], (nk / C::kKStages) & 1, ab)) {
          ok = false;
          break;
        }
        ++nk;
        tc_fence_after();
        const uint64_t bd = bdesc + (uint64_t)((ks * C::kKTile) >> 4);
        if (elect_sync()) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (sd[u] < 0) continue;
            const uint64_t ad = adesc + (uint64_t)((sd[u] * kDsBlock) >> 4);
            const uint32_t acc = acc0 + (uint32_t)(u * C::kTileCols);
            const bool started = u ? started1 : started0;
#pragma unroll
            for (int k = 0; k < 8; ++k)  // 16 keys: dS advances 256 bytes, K two 1024-byte groups
              mma_ss(acc, ad + 16 * k, bd + 128 * k, idesc, (started || k) ? 1u : 0u);
            mma_commit(&ds_empty[sd[u]]);
          }
          mma_commit(&k_empty[ks]);
        }
        __syncwarp();
        started0 = started0 || sd[0] >= 0;
        started1 = started1 || sd[1] >= 0;
      }
      if (!ok) break;
      if (elect_sync()) mma_commit(&acc_full[buf]);
      __syncwarp();
      ++na;
    }
    if (elect_sync()) {
      mma_commit(&drain_bar);
      mbar_wait_quiet(&drain_bar, 0, lim);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int r = wq * 32 + (threadIdx.x & 31);
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float mul = p.scale;
    bool ok = true;
    int na = 0;
    for (int q = 0; ok; ++q) {
      const int li = item_ring_pop(iring, q, ab, ok);
      if (li < 0) break;
      const Item it = item(li);
      if (!it.live[0]) continue;  // the pair lies past its sequence
      const bool keys = it.hi > it.lo;
      const int buf = na % C::kAccBufs, use = na / C::kAccBufs;
      if (keys) {
        if (!mbar_wait_warp(&acc_full[buf], use & 1u, ab)) {
          ok = false;
          break;
        }
        if (*(volatile int*)&abort_flag) {  // partial sums: leave the output
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const int tb = p.geo.cu_q ? 0 : it.b;
      for (int u = 0; u < 2; ++u) {
        if (!it.live[u]) continue;
        const bool tkeys = it.nkb[u] > 0;  // else the tile's dQ is zero
        const int i = it.q0 + u * kBlockM + r;
        const bool valid = i < it.sq.lq;
        const int64_t tok = (int64_t)it.sq.q_start + i;
        char* orow = (char*)p.dq + ((int64_t)tb * p.sdq_b + tok * p.sdq_t + (int64_t)it.h * p.sdq_h) *
                                       (G_F32 ? 4 : 2);
        const uint32_t acc = tmem + lane_off + (uint32_t)((buf * 2 + u) * C::kTileCols);
#pragma unroll 1
        for (int c = 0; c < DQK / 32; ++c) {
          uint32_t rr[32];
          if (tkeys) {
            tmem_ld32(acc + c * 32, rr);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) rr[t] = 0u;
          }
          if (!valid) continue;
          if (G_F32) {
            float4* dst = reinterpret_cast<float4*>(orow + c * 32 * 4);
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
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32 * 2);
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
      if (keys) {
        // the TMEM reads are complete (tcgen05.wait::ld) before the pair is
        // handed back to the MMA warp
        tc_fence_before();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&acc_free[buf]);
        ++na;
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

namespace {

template <int DQK, bool BF16, bool G_F32>
cudaError_t launch_dq_ds_t(const DqDsParams& p, unsigned ctas, cudaStream_t st) {
  using C = DqDsCfg<DQK>;
  auto k = attn_bwd_dq_ds_kernel<DQK, BF16, G_F32>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  k<<<ctas, C::kThreads, C::kSmem, st>>>(p);
  return cudaGetLastError();
}

template <int DQK>
cudaError_t launch_dq_ds_d(const DqDsParams& p, bool bf16, bool gf32, unsigned ctas, cudaStream_t st) {
  if (bf16)
    return gf32 ? launch_dq_ds_t<DQK, true, true>(p, ctas, st) : launch_dq_ds_t<DQK, true, false>(p, ctas, st);
  return gf32 ? launch_dq_ds_t<DQK, false, true>(p, ctas, st) : launch_dq_ds_t<DQK, false, false>(p, ctas, st);
}

}  // namespace

// Persistent: at most one CTA per SM (the dS and K stages take the shared
// memory), each taking items (query tile pairs) from the work queue
// (p.counter, zeroed by the caller before the launch).
cudaError_t launch_dq_ds(const DqDsParams& p, int dqk, bool bf16, bool gf32, int num_sms,
                         cudaStream_t st) {
  const long long items = (long long)((p.n_qtiles + 1) / 2) * p.hq * p.batch;
  if (items > 0x7fffffffll || !p.counter || num_sms <= 0) return cudaErrorInvalidValue;
  if (items == 0) return cudaSuccess;
  const unsigned ctas = (unsigned)(items < num_sms ? items : num_sms);
  if (dqk == 128) return launch_dq_ds_d<128>(p, bf16, gf32, ctas, st);
  if (dqk == 192) return launch_dq_ds_d<192>(p, bf16, gf32, ctas, st);
  return cudaErrorNotSupported;
}

}  // namespace attn
