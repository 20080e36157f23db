// bwd_dq_ds.cu -- dQ GEMM of the dS backward path (tcgen05 / TMEM / TMA).
//
// dQ_i = scale * sum_kb dS_{i,kb} K_kb  for one 128-row query tile i of one
// (sequence, query head), over its visible 128-key blocks kb, with the dS
// blocks the key-stationary dK/dV kernel wrote (layout in bwd.h) and K from
// the caller's tensor (TransformerEngine PR #3510 backward chain: dQ = dS K;
// PR #3699: the helper chain around it).  Every dQ element is produced by one
// CTA, accumulated in TMEM in key-block order, so the result is bitwise
// reproducible.
//
// The kernel streams 32 KiB of dS per 128-key block from HBM and multiplies
// it by a K tile that the CTAs working on the same head share through L2:
// per block, 128 x DQK x 128 MACs against 32 KiB, so it is bound by HBM
// bandwidth (at DQK = 192, about 1.3 PFLOP/s at the measured copy bandwidth).
// Four dS stages keep up to 128 KiB in flight per SM; the kernel is
// persistent, so the stream does not pause between query tiles.  At DQK = 128
// (three 32 KiB K stages) dS and K have producers of their own and the dS
// stream runs four blocks ahead of the MMAs; at DQK = 192 (two 48 KiB K
// stages) one producer issues each block's dS and K in turn, which keeps the
// K copies, which gate the MMAs, behind at most one dS copy (measured on one
// GB300, same results bit for bit: a separate K producer took the 32K
// DQK = 192 GEMM from 6.37 to 6.41 ms, and at DQK = 128 the 65K-token packed
// one from 1.75 to 1.70 ms).
//
// Warp roles: warp 0 dS producer (it also takes the items from the work
// queue, and issues the K copies too at DQK = 192), warp 1 TMEM owner and MMA
// issuer, warps 2..5 epilogue (TMEM lane quarter warp & 3), warp 6 K producer
// (DQK = 128 only).  MMA per K-step of 16 keys: M = 128 queries, N = DQK, A = dS
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
  static constexpr int kAccCols = DQK <= 128 ? 128 : 256;  // one accumulator buffer
  static constexpr bool kSplitK = kKStages >= 3;  // a K producer warp of its own
  static constexpr int kThreads = kSplitK ? 224 : 192;
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
  // two TMEM accumulators: acc_full[b] when the MMAs of an item in buffer b
  // are done, acc_free[b] when the epilogue has read it (one phase per use)
  __shared__ uint64_t acc_full[2], acc_free[2], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag, skip_sh;

  const int warp = threadIdx.x >> 5;
  // Persistent: one CTA per SM takes work items (query tile, query head,
  // sequence) from the work queue, in the order a one-CTA-per-item grid had
  // (tile_major(): the query tiles of a head, heaviest first, then the next
  // head; otherwise the heads of a query tile).  The dS stream runs on across
  // items, and an item's epilogue overlaps the next item's MMAs (the other
  // TMEM accumulator).
  const bool tmaj = tile_major(p.n_qtiles);
  const int gx = tmaj ? p.n_qtiles : p.hq, gy = tmaj ? p.hq : p.n_qtiles;
  const int n_items = gx * gy * p.batch;  // the launch checks that it fits
  __shared__ ItemRing<4> iring;
  struct Item {
    Seq sq;
    int h, b, q0, kb0, n_kb;
    bool live;  // the query tile lies inside its sequence
  };
  auto item = [&](int L) {
    Item it;
    const int x = L % gx;
    const int rest = L / gx;
    const int y = rest % gy;
    it.b = rest / gy;
    it.h = tmaj ? y : x;
    it.sq = load_seq(p.geo, it.b);
    const int qt = p.n_qtiles - 1 - (tmaj ? x : y);
    it.q0 = qt * kBlockM;
    it.live = it.q0 < it.sq.lq;
    it.kb0 = 0;
    it.n_kb = it.live ? wide_blocks_of_qtile(it.sq, qt, it.kb0) : 0;
    return it;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_free[i], 4);  // one arrival per epilogue warp
    }
    mbar_init(&drain_bar, 1);
    item_ring_init(iring, C::kSplitK ? 6 : 5);  // MMA, four epilogue warps (, K producer)
    fence_barrier_init();
    tma_prefetch_desc(&p.tm_k);
    skip_sh = status != 0;
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 2 * C::kAccCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (skip_sh) {
    if (warp == 1) tmem_dealloc(tmem, 2 * C::kAccCols);
    return;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ dS producer
    // per key block its dS block (one 32 KiB bulk copy, read once: L2
    // evict-first), then (DQK = 192) its K tile; the whole warp runs the
    // loop, one elected lane issues the copies; n counts the blocks of all items
    const uint64_t pol = l2_evict_first();
    bool ok = true;
    int n = 0, nk = 0;  // dS and K copies issued
    for (int q = 0; ok; ++q) {
      const int li = item_ring_push(iring, q, p.counter, n_items, ab, ok);
      if (li < 0) break;
      const Item it = item(li);
      if (it.n_kb == 0) continue;
      const int drop = li == 0 ? p.dbg.drop_load : -1;  // test-only injected missing load
      const long long T_b = p.plan[it.b + 1] - p.plan[it.b];
      const long long first = (long long)p.hq * p.plan[it.b] + (long long)it.h * T_b +
                              blocks_row_prefix(it.sq, it.q0 / kBlockM);  // whole warp
      if (!(first >= 0 && first + it.n_kb <= p.cap)) {  // inconsistent plan
        if (elect_sync()) {
          raise_status(p.status, DEV_WORKSPACE);
          *(volatile int*)&abort_flag = 1;
        }
        __syncwarp();
        ok = false;
        break;
      }
      for (int j = 0; j < it.n_kb && ok; ++j, ++n) {
        const int s = n % C::kDsStages;
        if (!mbar_wait_warp(&ds_empty[s], ((n / C::kDsStages) & 1) ^ 1, ab)) {
          ok = false;
          break;
        }
        if (j != drop && elect_sync()) {
          mbar_arrive_tx(&ds_full[s], kDsBlock);
          bulk_load_hint(sDs + s * kDsBlock, p.blocks + (size_t)(first + j) * kDsBlock, kDsBlock,
                         &ds_full[s], pol);
        }
        __syncwarp();
        if constexpr (!C::kSplitK) {
          const int ks = n % C::kKStages;
          if (!mbar_wait_warp(&k_empty[ks], ((n / C::kKStages) & 1) ^ 1, ab)) {
            ok = false;
            ++n;  // its dS copy is in flight
            break;
          }
          int c1, c2, c3;
          map_coords(p.ok, 0, it.h / (p.hq / p.hkv), it.sq.k_start + (it.kb0 + j) * kBlockN,
                     p.geo.cu_q ? 0 : it.b, c1, c2, c3);
          if (elect_sync()) {
            mbar_arrive_tx(&k_full[ks], C::kKTile);
#pragma unroll
            for (int c = 0; c < C::kKCh; ++c)
              tma_load_4d(sK + ks * C::kKTile + c * kSlotBytes, &p.tm_k, &k_full[ks], c * 64, c1, c2,
                          c3);
          }
          __syncwarp();
          nk = n + 1;
        }
      }
    }
    // let the copies in flight land before the CTA can exit
    for (int v = n > C::kDsStages ? n - C::kDsStages : 0; v < n; ++v)
      mbar_wait_quiet(&ds_full[v % C::kDsStages], (v / C::kDsStages) & 1, lim);
    for (int v = nk > C::kKStages ? nk - C::kKStages : 0; v < nk; ++v)
      mbar_wait_quiet(&k_full[v % C::kKStages], (v / C::kKStages) & 1, lim);
  } else if (C::kSplitK && warp == 6) {
    // ------------------------------------------------------------ K producer
    // (DQK = 128) the K tile of every block, in the dS producer's order
    bool ok = true;
    int n = 0;  // K copies issued
    for (int q = 0; ok; ++q) {
      const int li = item_ring_pop(iring, q, ab, ok);
      if (li < 0) break;
      const Item it = item(li);
      if (it.n_kb == 0) continue;
      const int g = it.h / (p.hq / p.hkv);
      const int tb = p.geo.cu_q ? 0 : it.b;
      for (int j = 0; j < it.n_kb && ok; ++j, ++n) {
        const int ks = n % C::kKStages;
        if (!mbar_wait_warp(&k_empty[ks], ((n / C::kKStages) & 1) ^ 1, ab)) {
          ok = false;
          break;
        }
        int c1, c2, c3;
        map_coords(p.ok, 0, g, it.sq.k_start + (it.kb0 + j) * kBlockN, tb, c1, c2, c3);
        if (elect_sync()) {
          mbar_arrive_tx(&k_full[ks], C::kKTile);
#pragma unroll
          for (int c = 0; c < C::kKCh; ++c)
            tma_load_4d(sK + ks * C::kKTile + c * kSlotBytes, &p.tm_k, &k_full[ks], c * 64, c1, c2, c3);
        }
        __syncwarp();
      }
    }
    for (int v = n > C::kKStages ? n - C::kKStages : 0; v < n; ++v)
      mbar_wait_quiet(&k_full[v % C::kKStages], (v / C::kKStages) & 1, lim);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // na counts the items with keys: accumulator na & 1, used for the
    // (na >> 1)-th time
    constexpr uint32_t idesc = make_idesc(128, DQK, BF16, true, true);
    const uint64_t adesc = make_sdesc_noswz(smem_u32(sDs), 128, kDsChunk);
    const uint64_t bdesc = make_sdesc(smem_u32(sK), kSlotBytes, 1024);
    bool ok = true;
    int n = 0, na = 0;
    for (int q = 0; ok; ++q) {
      const int li = item_ring_pop(iring, q, ab, ok);
      if (li < 0) break;
      const Item it = item(li);
      if (it.n_kb == 0) continue;
      const int buf = na & 1;
      if (na >= 2 && !mbar_wait_warp(&acc_free[buf], ((na >> 1) - 1) & 1u, ab)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(buf * C::kAccCols);
      for (int j = 0; j < it.n_kb && ok; ++j, ++n) {
        const int s = n % C::kDsStages, ks = n % C::kKStages;
        if (!mbar_wait_warp(&ds_full[s], (n / C::kDsStages) & 1, ab) ||
            !mbar_wait_warp(&k_full[ks], (n / C::kKStages) & 1, ab)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = adesc + (uint64_t)((s * kDsBlock) >> 4);
        const uint64_t bd = bdesc + (uint64_t)((ks * C::kKTile) >> 4);
        if (elect_sync()) {
#pragma unroll
          for (int k = 0; k < 8; ++k)  // 16 keys: dS advances 256 bytes, K two 1024-byte groups
            mma_ss(acc, ad + 16 * k, bd + 128 * k, idesc, (j | k) ? 1u : 0u);
          mma_commit(&ds_empty[s]);
          mma_commit(&k_empty[ks]);
        }
        __syncwarp();
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
      if (!it.live) continue;
      const int buf = na & 1;
      const bool keys = it.n_kb > 0;
      if (keys) {
        if (!mbar_wait_warp(&acc_full[buf], (na >> 1) & 1u, ab)) {
          ok = false;
          break;
        }
        if (*(volatile int*)&abort_flag) {  // partial sums: leave the output
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const int i = it.q0 + r;
      const bool valid = i < it.sq.lq;
      const int64_t tok = (int64_t)it.sq.q_start + i;
      const int tb = p.geo.cu_q ? 0 : it.b;
      char* orow = (char*)p.dq + ((int64_t)tb * p.sdq_b + tok * p.sdq_t + (int64_t)it.h * p.sdq_h) *
                                     (G_F32 ? 4 : 2);
      const uint32_t acc = tmem + lane_off + (uint32_t)(buf * C::kAccCols);
#pragma unroll 1
      for (int c = 0; c < DQK / 32; ++c) {
        uint32_t rr[32];
        if (keys) {
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
      if (keys) {
        // the TMEM reads are complete (tcgen05.wait::ld) before the buffer
        // is handed back to the MMA warp
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
    tmem_dealloc(tmem, 2 * C::kAccCols);
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
// memory), each taking items from the work queue (p.counter, zeroed by the
// caller before the launch).
cudaError_t launch_dq_ds(const DqDsParams& p, int dqk, bool bf16, bool gf32, int num_sms,
                         cudaStream_t st) {
  const long long items = (long long)p.n_qtiles * p.hq * p.batch;
  if (items > 0x7fffffffll || !p.counter || num_sms <= 0) return cudaErrorInvalidValue;
  if (items == 0) return cudaSuccess;
  const unsigned ctas = (unsigned)(items < num_sms ? items : num_sms);
  if (dqk == 128) return launch_dq_ds_d<128>(p, bf16, gf32, ctas, st);
  if (dqk == 192) return launch_dq_ds_d<192>(p, bf16, gf32, ctas, st);
  return cudaErrorNotSupported;
}

}  // namespace attn
