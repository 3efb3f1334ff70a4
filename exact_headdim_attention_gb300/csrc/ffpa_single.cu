// Single-CTA kernel: one CTA per 128-row query tile and output slice.
#include "ffpa_common.cuh"

namespace ffpa {

// UMASK: launched with a caller's mask (mask-loading code present).
template <bool VARLEN, bool UMASK>
__global__ void __launch_bounds__(NTHREADS, 1) ffpa_fwd_kernel(const __grid_constant__ Params p) {
  Item it;
  if (!decode_item(p, VARLEN, blockIdx.x, it)) return;   // uniform across the CTA

  // Scalars copied out of the parameter block once: the hot loops below run
  // between asm statements with memory clobbers, which would otherwise force
  // the parameter loads to be repeated.
  const int nchunks = p.nchunks, q_res = p.q_res, vk = p.vk;
  const int kchunks = p.kchunks, inject = p.inject;
  const bool fp16 = p.fp16 != 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int qpairs = (nchunks + 1) >> 1;
  const uint32_t q_region = q_res ? qpairs * SLOT_BYTES : 0u;
  const uint32_t qreg_u32 = smem_u32(smem);
  const uint32_t ring_u32 = qreg_u32 + q_region;
  const int NS = p.nslot;
  const int NSV = p.nslot_v;
  const uint32_t vslot = (uint32_t)p.vslot;
  const uint32_t vring_u32 = ring_u32 + NS * SLOT_BYTES;
  __shared__ __align__(8) uint64_t bar_full[NSLOT_MAX], bar_empty[NSLOT_MAX];
  __shared__ __align__(8) uint64_t bar_vfull[NSLOT_V_MAX], bar_vempty[NSLOT_V_MAX];
  __shared__ __align__(8) uint64_t bar_s_full, bar_s_free, bar_p_full[2], bar_pv_done[2], bar_q;
  __shared__ __align__(8) uint64_t bar_drain[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bar_full[i]), 1);
      mbar_init(smem_u32(&bar_empty[i]), 1);
    }
    for (int i = 0; i < NSV; ++i) {
      mbar_init(smem_u32(&bar_vfull[i]), 1);
      mbar_init(smem_u32(&bar_vempty[i]), 1);
    }
    mbar_init(smem_u32(&bar_s_full), 1);
    mbar_init(smem_u32(&bar_s_free), 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bar_p_full[b]), 4);
      mbar_init(smem_u32(&bar_pv_done[b]), 1);
    }
    mbar_init(smem_u32(&bar_drain[0]), 1);
    mbar_init(smem_u32(&bar_drain[1]), 1);
    mbar_init(smem_u32(&bar_q), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(&tmem_base_sh), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int T = it.ntiles;
  const unsigned long long tmo = p.timeout_ns;
  int* const err = p.err;

  if (warp == PRODUCER_WARP || warp == V_PRODUCER_WARP) {
    // ------------------------------------------------------------ producers
    // Two single-thread producers, each filling its own ring in the order
    // its MMA warp consumes it: warp 4 the K ring (Q pairs when Q is not
    // resident, then K pairs, per key tile), warp 7 the V ring (V stages per
    // key tile).  Separate rings keep every mbarrier phase observed by its
    // only consumer, which parity-based waits require.
    if (lane == 0 && T > 0) {
      const bool k_role = warp == PRODUCER_WARP;
      const int nslots = k_role ? NS : NSV;
      const uint32_t base = k_role ? ring_u32 : vring_u32;
      const uint32_t stride = k_role ? SLOT_BYTES : vslot;
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
      // Test hook: the very first K-ring stage of the CTA is acquired but
      // never armed or copied, so the MMA warp's wait on it runs out.
      bool drop = k_role && inject != 0;
      const uint32_t k_bytes = (uint32_t)kchunks * CHUNK_BYTES;
      // Returns the smem address of an armed slot, 0 when dropped, ~0u on abort.
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
      // Fine head dims: one 4-D box per 64-column chunk (x = 64 c), chunks
      // `stride` bytes apart; columns >= D are zero-filled.
      const bool fine = !VARLEN && p.dfine != 0;
      auto load_fine = [&](uint32_t dst, const CUtensorMap* m, uint32_t fb, int chunk0, int nch,
                           uint32_t stride, int row, int head) {
        for (int c = 0; c < nch; ++c)
          tma_load_4d(dst + c * stride, m, fb, DK * (chunk0 + c), row, head, it.b);
      };
      auto load_q_pair = [&](uint32_t dst, uint32_t fb, int pr) {
        if (VARLEN)
          tma_load_4d(dst, &p.tm_q, fb, 0, it.q_row0 + it.q0, 2 * pr, it.hq);
        else if (fine)
          load_fine(dst, &p.tm_q, fb, 2 * pr, kchunks, CHUNK_BYTES, it.q0, it.hq);
        else
          tma_load_5d(dst, &p.tm_q, fb, 0, it.q0, 2 * pr, it.hq, it.b);
      };
      if (k_role) {
        if (q_res) {
          const uint32_t qb = smem_u32(&bar_q);
          mbar_arrive_expect_tx(qb, qpairs * k_bytes);
          for (int pr = 0; pr < qpairs; ++pr) load_q_pair(qreg_u32 + pr * SLOT_BYTES, qb, pr);
        }
        for (int j = 0; j < T && ok; ++j) {
          const int key0 = kv_tile(it, j) * BN;
          for (int pr = 0; pr < qpairs && ok; ++pr) {
            uint32_t fb = 0, dst;
            if (!q_res) {
              dst = acquire(k_bytes, fb);
              if (dst == ~0u) { ok = false; break; }
              if (dst) load_q_pair(dst, fb, pr);
            }
            dst = acquire(k_bytes, fb);
            if (dst == ~0u) { ok = false; break; }
            if (dst) {
              if (VARLEN)
                tma_load_4d(dst, &p.tm_k, fb, 0, it.kv_row0 + key0, 2 * pr, it.hkv);
              else if (fine)
                load_fine(dst, &p.tm_k, fb, 2 * pr, kchunks, CHUNK_BYTES, key0, it.hkv);
              else
                tma_load_5d(dst, &p.tm_k, fb, 0, key0, 2 * pr, it.hkv, it.b);
            }
          }
        }
        if (q_res) wait_drain(smem_u32(&bar_q), 0, tmo, err);
      } else {
        for (int j = 0; j < T && ok; ++j) {
          for (int h = 0; h < BN / vk && ok; ++h) {
            uint32_t fb = 0;
            const uint32_t dst = acquire(vslot, fb);
            if (dst == ~0u) { ok = false; break; }
            const int key = kv_tile(it, j) * BN + h * vk;
            if (VARLEN)
              tma_load_4d(dst, &p.tm_v, fb, 0, it.kv_row0 + key, it.col_lo / DK, it.hkv);
            else if (fine)
              load_fine(dst, &p.tm_v, fb, it.col_lo / DK, p.vchunks, (uint32_t)vk * 128u, key, it.hkv);
            else
              tma_load_5d(dst, &p.tm_v, fb, 0, key, it.col_lo / DK, it.hkv, it.b);
          }
        }
      }
      // Drain: every copy this thread started has landed before the CTA exits
      // (the dropped test stage, the first K stage, was never armed).
      const int n = issued < nslots ? issued : nslots;
      int s = slot;
      uint32_t lp = lap;
      for (int i = 0; i < n; ++i) {
        if (--s < 0) { s = nslots - 1; lp ^= 1u; }
        if (k_role && inject != 0 && issued - 1 - i == 0) continue;
        wait_drain(smem_u32(&full[s]), lp, tmo, err);
      }
    }
  } else if (warp == MMA_WARP || warp == PV_WARP) {
    // ------------------------------------------------------------ MMA issuers
    // Two warps issue tensor-core work, one thread each: warp 5 the QK^T MMAs
    // (into S), warp 6 the PV MMAs (into O).  Every mbarrier test costs an
    // issuing thread ~100 cycles, longer than the one MMA the tensor queue
    // holds; with two issuers the waits of one are covered by the MMAs of the
    // other.  Each consumes its own ring (K ring / V ring) in order.
    if (lane == 0) {
      const bool qk_role = warp == MMA_WARP;
      const int nV = BN / vk;                       // V stages per key tile
      const int nslots = qk_role ? NS : NSV;
      uint64_t* full = qk_role ? bar_full : bar_vfull;
      uint64_t* empty = qk_role ? bar_empty : bar_vempty;
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
      auto release = [&](int s) { umma_commit(smem_u32(&empty[s])); };
      auto wait_on = [&](uint32_t bar, uint32_t par) -> bool {
        if (!mbar_try_wait(bar, par) && !wait_bounded(bar, par, &abort_flag, tmo, err)) return false;
        tc_fence_after();
        return true;
      };
      if (qk_role) {
        const uint32_t idesc_qk = idesc_f16(!fp16, BM, BN, false, false);
        // Descriptors advance by (byte offset >> 4) in their start-address field.
        const uint64_t ring_desc = sdesc_sw128(ring_u32, 16, 1024);
        const uint64_t q_desc = sdesc_sw128(qreg_u32, 16, 1024);
        const uint32_t s_col = tmem + S_COL;
        if (T > 0 && q_res) ok = wait_on(smem_u32(&bar_q), 0);
        for (int j = 0; j < T && ok; ++j) {
          // S is free once the softmax warps have read S_{j-1}.
          if (j >= 1 && !(ok = wait_on(smem_u32(&bar_s_free), (j - 1) & 1))) break;
          for (int pr = 0; pr < qpairs && ok; ++pr) {
            int sq = -1;
            if (!q_res) {
              sq = take();
              if (sq < 0) { ok = false; break; }
            }
            const int sk = take();
            if (sk < 0) { ok = false; break; }
            const uint64_t ad = q_res ? q_desc + (((2 * pr) * CHUNK_BYTES) >> 4)
                                      : ring_desc + ((sq * SLOT_BYTES) >> 4);
            const uint64_t bd = ring_desc + ((sk * SLOT_BYTES) >> 4);
            // 16 D-elements per MMA: +32 bytes (>>4 = 2) within a 128-byte row;
            // the second chunk of the pair sits 16 KB (>>4 = 1024) further.
            umma_ss(s_col, ad, bd, idesc_qk, pr > 0 ? 1u : 0u);
#pragma unroll
            for (int k = 1; k < 4; ++k) umma_ss(s_col, ad + 2 * k, bd + 2 * k, idesc_qk, 1u);
            if (2 * pr + 1 < nchunks) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_ss(s_col, ad + 1024 + 2 * k, bd + 1024 + 2 * k, idesc_qk, 1u);
            }
            if (sq >= 0) release(sq);
            release(sk);
          }
          if (!ok) break;
          umma_commit(smem_u32(&bar_s_full));
        }
      } else {
        const uint32_t idesc_pv = idesc_f16(!fp16, BM, it.dv, false, true);
        const uint64_t v_desc = sdesc_sw128(vring_u32, vk * 128, 1024);
        for (int j = 0; j < T && ok; ++j) {
          const int b = j & 1;
          if (!(ok = wait_on(smem_u32(&bar_p_full[b]), (j >> 1) & 1))) break;
          const uint32_t p_col = tmem + P_COL0 + 64 * b;
          for (int h = 0; h < nV; ++h) {
            const int s = take();
            if (s < 0) { ok = false; break; }
            const uint64_t vd = v_desc + ((s * vslot) >> 4);
            const uint32_t pc = p_col + ((h * vk) >> 1);
            // 16 keys per MMA: +8 TMEM columns of P, +2048 bytes (>>4 = 128) of V.
            umma_ts(tmem, pc, vd, idesc_pv, (j > 0 || h > 0) ? 1u : 0u);
            umma_ts(tmem, pc + 8, vd + 128, idesc_pv, 1u);
            if (vk >= 64) {
              umma_ts(tmem, pc + 16, vd + 256, idesc_pv, 1u);
              umma_ts(tmem, pc + 24, vd + 384, idesc_pv, 1u);
            }
            if (vk == 128) {
#pragma unroll
              for (int kk = 4; kk < 8; ++kk) umma_ts(tmem, pc + 8 * kk, vd + 128 * kk, idesc_pv, 1u);
            }
            release(s);
          }
          if (!ok) break;
          umma_commit(smem_u32(&bar_pv_done[b]));
        }
      }
      // Drain: all MMAs issued by this thread complete before TMEM is freed.
      const uint32_t db = smem_u32(&bar_drain[qk_role ? 0 : 1]);
      umma_commit(db);
      wait_drain(db, 0, tmo, err);
    }
  } else {
    // ------------------------------------------------------------ softmax
    SoftmaxBars bars;
    bars.s_full = smem_u32(&bar_s_full);
    bars.s_free_arrive = smem_u32(&bar_s_free);
    bars.p_full_arrive = smem_u32(&bar_p_full[0]);
    bars.pv_done = smem_u32(&bar_pv_done[0]);
    softmax_role<VARLEN, false, UMASK>(p, it, T, tmem, warp, lane, bars, &abort_flag, tmo, err);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

ffpa_status launch_single(bool varlen, bool umask, const Params& P, int items, size_t smem,
                          cudaStream_t stream) {
  auto kern = varlen  ? ffpa_fwd_kernel<true, false>
              : umask ? ffpa_fwd_kernel<false, true>
                      : ffpa_fwd_kernel<false, false>;
  const ffpa_status st =
      set_smem_attr_once(reinterpret_cast<const void*>(kern), P.device, static_cast<int>(SMEM_LIMIT - SMEM_STATIC_RESERVE));
  if (st != FFPA_OK) return st;
  kern<<<items, NTHREADS, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}


}  // namespace ffpa
