// CTA-pair kernel (cta_group::2): 256-row query tiles on two SMs.
#include "ffpa_common.cuh"

namespace ffpa {

// =====================================================================
// CTA-pair kernel (cta_group::2): two CTAs on two SMs share every K/V tile.
//
// A cluster of two CTAs owns a 256-row query tile: CTA c holds query rows
// 128c .. 128c+127 (Q resident in its shared memory, S/O/P in its TMEM) and
// loads only its half of each key tile (64 keys x 4 D-chunks) and of each V
// stage (half of the slice's output columns).  The leader CTA (rank 0)
// issues M = 256 MMAs that combine both halves, so each SM moves half the
// K/V bytes and each MMA instruction drives both tensor cores.  The peer's
// warps 5/6 relay its "stage landed" events to the leader's full barriers;
// the leader's commits arrive in both CTAs (multicast).  Used when every
// output slice is a multiple of 128 columns and Q fits in shared memory.
// =====================================================================

__device__ __forceinline__ bool decode_item_pair(const Params& p, bool varlen, int L, uint32_t rank,
                                                 Item& it) {
  it.slice = L % p.n_slices;
  L /= p.n_slices;
  const int heads = p.B * p.Hq;
  int qt;
  if (p.causal) {
    const int bh = L % heads;
    qt = p.n_qt - 1 - L / heads;
    it.hq = bh % p.Hq;
    it.b = bh / p.Hq;
  } else {
    qt = L % p.n_qt;
    const int bh = L / p.n_qt;
    it.hq = bh % p.Hq;
    it.b = bh / p.Hq;
  }
  it.hkv = it.hq / p.group;
  if (varlen) {
    it.q_row0 = p.cu_q[it.b];
    it.q_len = p.cu_q[it.b + 1] - it.q_row0;
    it.kv_row0 = p.cu_k[it.b];
    it.kv_len = p.cu_k[it.b + 1] - it.kv_row0;
  } else {
    it.q_row0 = 0;
    it.q_len = p.Nq;
    it.kv_row0 = 0;
    it.kv_len = p.Nkv;
  }
  const int q0_pair = qt * BM_PAIR;
  if (q0_pair >= it.q_len) return false;           // same answer in both CTAs
  it.q0 = q0_pair + BM * (int)rank;                // this CTA's rows
  const int last_row = min(q0_pair + BM_PAIR, it.q_len) - 1;
  long long kv_end = it.kv_len;
  if (p.causal) kv_end = min(kv_end, (long long)last_row + (it.kv_len - it.q_len) + 1);
  it.ntiles = kv_end > 0 ? (int)((kv_end + BN - 1) / BN) : 0;
  // As decode_item: dense causal items start at key tile 0.
  it.rot = (it.ntiles > 0 && !(p.causal && !varlen))
               ? (int)(((unsigned)qt * 37u + (unsigned)it.slice * 17u + (unsigned)it.hq * 13u) %
                       (unsigned)it.ntiles)
               : 0;
  const int c_lo = it.slice * p.nchunks / p.n_slices;
  const int c_hi = (it.slice + 1) * p.nchunks / p.n_slices;
  it.col_lo = c_lo * DK;
  it.dv = (c_hi - c_lo) * DK;
  return true;
}

// NCH = D / 64 as a template parameter: the MMA issue loops unroll.
template <bool VARLEN, int NCH, bool UMASK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    ffpa_fwd_pair_kernel(const __grid_constant__ Params p) {
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  Item it;
  if (!decode_item_pair(p, VARLEN, blockIdx.x >> 1, rank, it)) return;   // uniform across the pair

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int nchunks = NCH, vk = BN;
  const int inject = p.inject;
  const bool fp16 = p.fp16 != 0;
  constexpr int qpairs = (nchunks + 1) >> 1;
  constexpr int KC = nchunks < 4 ? nchunks : 4;
  constexpr int nkst = nchunks / KC;               // K stages per key tile
  const uint32_t kslot = (uint32_t)p.kslot, vslot = (uint32_t)p.vslot;
  const int NS = p.nslot, NSV = p.nslot_v;
  const uint32_t qreg_u32 = smem_u32(smem);
  const uint32_t kring_u32 = qreg_u32 + qpairs * SLOT_BYTES;
  const uint32_t vring_u32 = kring_u32 + NS * kslot;
  __shared__ __align__(8) uint64_t bar_full[NSLOT_MAX], bar_empty[NSLOT_MAX];
  __shared__ __align__(8) uint64_t bar_vfull[NSLOT_V_MAX], bar_vempty[NSLOT_V_MAX];
  __shared__ __align__(8) uint64_t bar_s_full, bar_s_free, bar_p_full[2], bar_pv_done[2], bar_q;
  __shared__ __align__(8) uint64_t bar_drain[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // Leader full barriers also count the peer's relayed arrival.
    const uint32_t nfull = leader ? 2 : 1;
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bar_full[i]), nfull);
      mbar_init(smem_u32(&bar_empty[i]), 1);
    }
    for (int i = 0; i < NSV; ++i) {
      mbar_init(smem_u32(&bar_vfull[i]), nfull);
      mbar_init(smem_u32(&bar_vempty[i]), 1);
    }
    mbar_init(smem_u32(&bar_q), nfull);
    mbar_init(smem_u32(&bar_s_full), 1);
    mbar_init(smem_u32(&bar_s_free), 8);        // 4 softmax warps in each CTA
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bar_p_full[b]), 8);
      mbar_init(smem_u32(&bar_pv_done[b]), 1);
      mbar_init(smem_u32(&bar_drain[b]), 1);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc_pair(smem_u32(&tmem_base_sh), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();      // the peer's barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int T = it.ntiles;
  const unsigned long long tmo = p.timeout_ns;
  int* const err = p.err;

  if (warp == PRODUCER_WARP || warp == V_PRODUCER_WARP) {
    // ------------------------------------------------------------ producers
    if (lane == 0 && T > 0) {
      const bool k_role = warp == PRODUCER_WARP;
      const int nslots = k_role ? NS : NSV;
      const uint32_t base = k_role ? kring_u32 : vring_u32;
      const uint32_t stride = k_role ? kslot : vslot;
      uint64_t* full = k_role ? bar_full : bar_vfull;
      uint64_t* empty = k_role ? bar_empty : bar_vempty;
      if (k_role) {
        prefetch_tmap(&p.tm_q);
        prefetch_tmap(&p.tm_k);
      } else {
        prefetch_tmap(&p.tm_v);
      }
      int slot = 0;
      uint32_t lap = 0;
      int issued = 0;
      bool ok = true;
      bool drop = k_role && leader && inject != 0;   // test hook (see ffpa_test_drop_first_copy)
      auto acquire = [&](uint32_t bytes, uint32_t& fb) -> uint32_t {
        const uint32_t eb = smem_u32(&empty[slot]);
        if (!mbar_try_wait(eb, lap ^ 1u) && !wait_bounded(eb, lap ^ 1u, &abort_flag, tmo, err))
          return ~0u;
        fb = smem_u32(&full[slot]);
        const uint32_t dst = base + slot * stride;
        ++issued;
        if (++slot == nslots) { slot = 0; lap ^= 1u; }
        if (drop) {
          drop = false;
          return 0u;
        }
        mbar_arrive_expect_tx(fb, bytes);
        return dst;
      };
      if (k_role) {
        const uint32_t qb = smem_u32(&bar_q);
        mbar_arrive_expect_tx(qb, (uint32_t)nchunks * CHUNK_BYTES);
        for (int pr = 0; pr < qpairs; ++pr) {
          if (VARLEN)
            tma_load_4d(qreg_u32 + pr * SLOT_BYTES, &p.tm_q, qb, 0, it.q_row0 + it.q0, 2 * pr, it.hq);
          else
            tma_load_5d(qreg_u32 + pr * SLOT_BYTES, &p.tm_q, qb, 0, it.q0, 2 * pr, it.hq, it.b);
        }
        const int myk = KEYS_PER_CTA * (int)rank;
        for (int j = 0; j < T && ok; ++j) {
          const int key0 = kv_tile(it, j) * BN + myk;
          for (int g = 0; g < nkst && ok; ++g) {
            uint32_t fb = 0;
            const uint32_t dst = acquire(kslot, fb);
            if (dst == ~0u) { ok = false; break; }
            if (dst) {
              if (VARLEN)
                tma_load_4d(dst, &p.tm_k, fb, 0, it.kv_row0 + key0, KC * g, it.hkv);
              else
                tma_load_5d(dst, &p.tm_k, fb, 0, key0, KC * g, it.hkv, it.b);
            }
          }
        }
        wait_drain(qb, 0, tmo, err);
      } else {
        const int mycol = (it.col_lo + (it.dv / 2) * (int)rank) / DK;
        for (int j = 0; j < T && ok; ++j) {
          for (int h = 0; h < BN / vk && ok; ++h) {
            uint32_t fb = 0;
            const uint32_t dst = acquire(vslot, fb);
            if (dst == ~0u) { ok = false; break; }
            const int key = kv_tile(it, j) * BN + h * vk;
            if (VARLEN)
              tma_load_4d(dst, &p.tm_v, fb, 0, it.kv_row0 + key, mycol, it.hkv);
            else
              tma_load_5d(dst, &p.tm_v, fb, 0, key, mycol, it.hkv, it.b);
          }
        }
      }
      const int n = issued < nslots ? issued : nslots;
      int s = slot;
      uint32_t lp = lap;
      for (int i = 0; i < n; ++i) {
        if (--s < 0) { s = nslots - 1; lp ^= 1u; }
        if (k_role && leader && inject != 0 && issued - 1 - i == 0) continue;
        wait_drain(smem_u32(&full[s]), lp, tmo, err);
      }
    }
  } else if ((warp == MMA_WARP || warp == PV_WARP) && !leader) {
    // ------------------------------------------------------------ relays
    // Forward each landed stage of this CTA to the leader's full barrier.
    if (lane == 0 && T > 0) {
      const bool k_role = warp == MMA_WARP;
      const int nslots = k_role ? NS : NSV;
      uint64_t* full = k_role ? bar_full : bar_vfull;
      const int per_tile = k_role ? nkst : BN / vk;
      if (k_role) {
        const uint32_t qb = smem_u32(&bar_q);
        if (!(mbar_try_wait(qb, 0) || wait_bounded(qb, 0, &abort_flag, tmo, err))) goto relay_done;
        mbar_arrive_cluster(mapa_shared(qb, 0));
      }
      {
        int slot = 0;
        uint32_t lap = 0;
        for (int i = 0; i < T * per_tile; ++i) {
          const uint32_t fb = smem_u32(&full[slot]);
          if (!(mbar_try_wait(fb, lap) || wait_bounded(fb, lap, &abort_flag, tmo, err))) break;
          mbar_arrive_cluster(mapa_shared(fb, 0));
          if (++slot == nslots) { slot = 0; lap ^= 1u; }
        }
      }
    relay_done:;
    }
  } else if (warp == MMA_WARP || warp == PV_WARP) {
    // ------------------------------------------------------------ MMA issuers (leader)
    if (lane == 0) {
      const bool qk_role = warp == MMA_WARP;
      const int nslots = qk_role ? NS : NSV;
      uint64_t* full = qk_role ? bar_full : bar_vfull;
      int slot = 0;
      uint32_t lap = 0;
      bool ok = true;
      auto take = [&]() -> int {
        const uint32_t fb = smem_u32(&full[slot]);
        if (!mbar_try_wait(fb, lap) && !wait_bounded(fb, lap, &abort_flag, tmo, err)) return -1;
        const int s = slot;
        if (++slot == nslots) { slot = 0; lap ^= 1u; }
        return s;
      };
      auto wait_on = [&](uint32_t bar, uint32_t par) -> bool {
        if (!mbar_try_wait(bar, par) && !wait_bounded(bar, par, &abort_flag, tmo, err)) return false;
        tc_fence_after();
        return true;
      };
      if (qk_role) {
        const uint32_t idesc_qk = idesc_f16(!fp16, BM_PAIR, BN, false, false);
        const uint64_t k_desc = sdesc_sw128(kring_u32, 16, 1024);
        const uint64_t q_desc = sdesc_sw128(qreg_u32, 16, 1024);
        const uint32_t s_col = tmem + S_COL;
        const uint32_t kchunk_step = (KEYS_PER_CTA * 128) >> 4;   // one 64-key chunk
        if (T > 0) ok = wait_on(smem_u32(&bar_q), 0);
        for (int j = 0; j < T && ok; ++j) {
          if (j >= 1 && !(ok = wait_on(smem_u32(&bar_s_free), (j - 1) & 1))) break;
#pragma unroll
          for (int g = 0; g < nkst; ++g) {
            const int sk = take();
            if (sk < 0) { ok = false; break; }
            const uint64_t bd0 = k_desc + ((sk * kslot) >> 4);
#pragma unroll
            for (int cc = 0; cc < KC; ++cc) {
              const uint64_t ad = q_desc + (((KC * g + cc) * CHUNK_BYTES) >> 4);
              const uint64_t bd = bd0 + cc * kchunk_step;
              umma_ss_pair(s_col, ad, bd, idesc_qk, (g > 0 || cc > 0) ? 1u : 0u);
#pragma unroll
              for (int k = 1; k < 4; ++k) umma_ss_pair(s_col, ad + 2 * k, bd + 2 * k, idesc_qk, 1u);
            }
            umma_commit_pair(smem_u32(&bar_empty[sk]));
          }
          if (!ok) break;
          umma_commit_pair(smem_u32(&bar_s_full));
        }
      } else {
        const uint32_t idesc_pv = idesc_f16(!fp16, BM_PAIR, it.dv, false, true);
        const uint64_t v_desc = sdesc_sw128(vring_u32, vk * 128, 1024);
        for (int j = 0; j < T && ok; ++j) {
          const int b = j & 1;
          if (!(ok = wait_on(smem_u32(&bar_p_full[b]), (j >> 1) & 1))) break;
          const uint32_t p_col = tmem + P_COL0 + 64 * b;
          for (int h = 0; h < BN / vk; ++h) {
            const int s = take();
            if (s < 0) { ok = false; break; }
            const uint64_t vd = v_desc + ((s * vslot) >> 4);
            const uint32_t pc = p_col + ((h * vk) >> 1);
#pragma unroll
            for (int kk = 0; kk < vk / 16; ++kk)
              umma_ts_pair(tmem, pc + 8 * kk, vd + 128 * kk, idesc_pv, (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
            umma_commit_pair(smem_u32(&bar_vempty[s]));
          }
          if (!ok) break;
          umma_commit_pair(smem_u32(&bar_pv_done[b]));
        }
      }
      const uint32_t db = smem_u32(&bar_drain[qk_role ? 0 : 1]);
      umma_commit_pair(db);
      wait_drain(db, 0, tmo, err);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    SoftmaxBars bars;
    bars.s_full = smem_u32(&bar_s_full);
    bars.s_free_arrive = mapa_shared(smem_u32(&bar_s_free), 0);
    bars.p_full_arrive = mapa_shared(smem_u32(&bar_p_full[0]), 0);
    bars.pv_done = smem_u32(&bar_pv_done[0]);
    softmax_role<VARLEN, true, UMASK>(p, it, T, tmem, warp, lane, bars, &abort_flag, tmo, err);
  }

  // The leader's last commits also arrive in the peer: wait for them before
  // the pair may exit, then free TMEM in both CTAs together.
  if (!leader && threadIdx.x == 0) {
    wait_drain(smem_u32(&bar_drain[0]), 0, tmo, err);
    wait_drain(smem_u32(&bar_drain[1]), 0, tmo, err);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

template <bool VARLEN, bool UMASK>
static ffpa_status launch_pair_t(const Params& P, int items, size_t smem, cudaStream_t stream) {
  auto kern = P.nchunks == 8   ? ffpa_fwd_pair_kernel<VARLEN, 8, UMASK>
              : P.nchunks == 4 ? ffpa_fwd_pair_kernel<VARLEN, 4, UMASK>
                               : ffpa_fwd_pair_kernel<VARLEN, 2, UMASK>;
  const ffpa_status st =
      set_smem_attr_once(reinterpret_cast<const void*>(kern), P.device, static_cast<int>(SMEM_LIMIT - SMEM_STATIC_RESERVE));
  if (st != FFPA_OK) return st;
  kern<<<2 * items, NTHREADS, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}

ffpa_status launch_pair(bool varlen, bool umask, const Params& P, int items, size_t smem,
                        cudaStream_t stream) {
  return varlen  ? launch_pair_t<true, false>(P, items, smem, stream)
         : umask ? launch_pair_t<false, true>(P, items, smem, stream)
                 : launch_pair_t<false, false>(P, items, smem, stream);
}


}  // namespace ffpa
