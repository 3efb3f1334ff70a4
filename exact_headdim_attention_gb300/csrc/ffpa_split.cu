// Column-split kernel: two SMs share a 128-row query tile, each owning half of the output columns.
#include "ffpa_common.cuh"

namespace ffpa {

// =====================================================================
// Column-split pair kernel: no recomputation of S for D up to 512 (the
// clusters of 3 and 4 CTAs for D = 768 and 1024 are in ffpa_cluster.cu).
//
// A cluster of two CTAs owns one 128-row query tile; CTA c owns the output
// columns [c D/2, (c+1) D/2), so each CTA's O accumulator (D/2 <= 256 fp32
// columns) fits in TMEM next to S and a part of Q.  Key tiles alternate
// between the CTAs: in round i, CTA c computes S = Q K^T for tile 2i + c over
// the full head dimension, the two CTAs agree on the running row maximum
// (each stores its tile maximum into the other's shared memory), and each
// CTA writes its P tile into its own shared memory and bulk-copies it into
// the peer's.  Both CTAs then accumulate both P tiles against their half of
// V.  Per CTA and round: one QK^T (full D), two PV products (D/2 columns),
// one softmax tile; the multiply-adds are exactly those of the attention.
//
// Q chunks 0..3 are the MMA's A operand in TMEM; further chunks stay in
// shared memory.  TMEM columns: O [0, D/2), S [256, 384), Q [384, 512).
// Shared memory: Q chunks 4.. | P (own) | P (peer) | ring of 32 KB stages.
// At start the P area holds Q chunks 0..3 on their way into TMEM.
// Warps: 0-3 softmax (thread r owns row r = TMEM lane r), 4 TMA producer,
// 5 MMA issuer.  Every wait is bounded; waits on phases that the peer CTA
// completes use cluster-scope acquire.
// =====================================================================

// NCH = D / 64 is a template parameter so that every MMA issue loop has a
// compile-time trip count and is fully unrolled: the tensor pipe's
// instruction queue is shallow, and loop overhead between MMAs leaves it
// idle (measured: a runtime-count loop of 8 MMAs runs at about half rate).
template <bool VARLEN, int NCH, bool UMASK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(SPLIT_THREADS, 1)
    ffpa_fwd_split_kernel(const __grid_constant__ Params p) {
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  Item it;
  if (!decode_item(p, VARLEN, blockIdx.x >> 1, it)) return;   // same answer in both CTAs
  it.dv = NCH * DK / 2;                                        // padded D: see split_chunks
  it.col_lo = it.dv * (int)rank;
  it.slice = (int)rank;                                        // rank 0 writes the LSE

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int nchunks = NCH;
  constexpr int qt = NCH < Q_TMEM_MAX_CHUNKS ? NCH : Q_TMEM_MAX_CHUNKS;   // Q chunks held in TMEM
  constexpr int VCH = NCH / 2;                                           // V chunks per CTA
  constexpr int vk = VCH * 128 * 128 <= (int)SLOT_BYTES ? 128 : 64;      // keys per V stage
  const int inject = p.inject;
  const bool fp16 = p.fp16 != 0;
  const uint32_t vslot = (uint32_t)p.vslot;
  const int NS = p.nslot;
  const uint32_t qs_u32 = smem_u32(smem);
  const uint32_t pown_u32 = qs_u32 + (uint32_t)(nchunks - qt) * CHUNK_BYTES;
  const uint32_t ppeer_u32 = pown_u32 + P_TILE_BYTES;
  const uint32_t ring_u32 = ppeer_u32 + P_TILE_BYTES;
  __shared__ __align__(8) uint64_t bar_full[NSLOT_MAX], bar_empty[NSLOT_MAX];
  __shared__ __align__(8) uint64_t bar_q, bar_qt, bar_s_full, bar_s_free;
  __shared__ __align__(8) uint64_t bar_pown_full, bar_pown_free, bar_ppeer_full, bar_peer_free;
  __shared__ __align__(8) uint64_t bar_pv_done, bar_x[2], bar_l, bar_drain;
  __shared__ __align__(16) float xbuf[2][BM];
  __shared__ __align__(16) float lbuf[BM];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bar_full[i]), 1);
      mbar_init(smem_u32(&bar_empty[i]), 1);
    }
    mbar_init(smem_u32(&bar_q), 1);           // TMA bytes of Q
    mbar_init(smem_u32(&bar_qt), 4);          // softmax warps: Q chunks 0..3 in TMEM
    mbar_init(smem_u32(&bar_s_full), 1);      // QK commit
    mbar_init(smem_u32(&bar_s_free), 4);      // softmax warps: S read
    mbar_init(smem_u32(&bar_pown_full), 4);   // softmax warps: P written / O rescaled
    mbar_init(smem_u32(&bar_pown_free), 1);   // PV commit: own P tile read
    mbar_init(smem_u32(&bar_ppeer_full), 1);  // bulk-copy bytes of the peer's P tile
    mbar_init(smem_u32(&bar_peer_free), 1);   // the peer read this CTA's P tile
    mbar_init(smem_u32(&bar_pv_done), 1);     // PV commit per round
    mbar_init(smem_u32(&bar_x[0]), 1);        // the peer's tile maxima
    mbar_init(smem_u32(&bar_x[1]), 1);
    mbar_init(smem_u32(&bar_l), 1);           // the peer's row sums
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(&tmem_base_sh), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();      // the peer's barriers exist before any remote operation
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int T = it.ntiles;
  const int R = (T + 1) >> 1;                  // rounds of two key tiles
  const int own0 = (int)rank, peer0 = (int)peer;   // tile of round i: 2 i + own0 / 2 i + peer0
  const unsigned long long tmo = p.timeout_ns;
  int* const err = p.err;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    // One ring, filled in the MMA thread's order: K of the first own tile,
    // then per round i: K of the own tile of round i+1, V (this CTA's
    // columns) of the own tile, V of the peer's tile.
    if (lane == 0 && T > 0) {
      prefetch_tmap(&p.tm_q);
      prefetch_tmap(&p.tm_k);
      prefetch_tmap(&p.tm_v);
      int slot = 0;
      uint32_t lap = 0;
      int issued = 0;
      bool ok = true;
      bool drop = inject != 0 && rank == 0;   // test hook (see ffpa_test_drop_first_copy)
      auto acquire = [&](uint32_t bytes, uint32_t& fb) -> uint32_t {
        const uint32_t eb = smem_u32(&bar_empty[slot]);
        if (!mbar_try_wait(eb, lap ^ 1u) && !wait_bounded(eb, lap ^ 1u, &abort_flag, tmo, err))
          return ~0u;
        fb = smem_u32(&bar_full[slot]);
        const uint32_t dst = ring_u32 + slot * SLOT_BYTES;
        ++issued;
        if (++slot == NS) { slot = 0; lap ^= 1u; }
        if (drop) {
          drop = false;
          return 0u;
        }
        mbar_arrive_expect_tx(fb, bytes);
        return dst;
      };
      const uint32_t qb = smem_u32(&bar_q);
      mbar_arrive_expect_tx(qb, (uint32_t)nchunks * CHUNK_BYTES);
      for (int c = 0; c < nchunks; c += 2) {
        const uint32_t dst = c < qt ? pown_u32 + c * CHUNK_BYTES : qs_u32 + (c - qt) * CHUNK_BYTES;
        if (VARLEN)
          tma_load_4d(dst, &p.tm_q, qb, 0, it.q_row0 + it.q0, c, it.hq);
        else
          tma_load_5d(dst, &p.tm_q, qb, 0, it.q0, c, it.hq, it.b);
      }
      auto load_k = [&](int j) -> bool {
        const int key0 = kv_tile(it, j) * BN;
        for (int c = 0; c < nchunks; c += 2) {
          uint32_t fb = 0;
          const uint32_t dst = acquire(2 * CHUNK_BYTES, fb);
          if (dst == ~0u) return false;
          if (dst) {
            if (VARLEN)
              tma_load_4d(dst, &p.tm_k, fb, 0, it.kv_row0 + key0, c, it.hkv);
            else
              tma_load_5d(dst, &p.tm_k, fb, 0, key0, c, it.hkv, it.b);
          }
        }
        return true;
      };
      auto load_v = [&](int j) -> bool {
        for (int h = 0; h < BN / vk; ++h) {
          uint32_t fb = 0;
          const uint32_t dst = acquire(vslot, fb);
          if (dst == ~0u) return false;
          const int key = kv_tile(it, j) * BN + h * vk;
          if (VARLEN)
            tma_load_4d(dst, &p.tm_v, fb, 0, it.kv_row0 + key, it.col_lo / DK, it.hkv);
          else
            tma_load_5d(dst, &p.tm_v, fb, 0, key, it.col_lo / DK, it.hkv, it.b);
        }
        return true;
      };
      if (own0 < T) ok = load_k(own0);
      for (int i = 0; i < R && ok; ++i) {
        if (2 * i + 2 + own0 < T && !(ok = load_k(2 * i + 2 + own0))) break;
        if (2 * i + own0 < T && !(ok = load_v(2 * i + own0))) break;
        if (2 * i + peer0 < T && !(ok = load_v(2 * i + peer0))) break;
      }
      wait_drain(qb, 0, tmo, err);
      const int n = issued < NS ? issued : NS;
      int s = slot;
      uint32_t lp = lap;
      for (int i = 0; i < n; ++i) {
        if (--s < 0) { s = NS - 1; lp ^= 1u; }
        if (inject != 0 && rank == 0 && issued - 1 - i == 0) continue;   // never armed
        wait_drain(smem_u32(&bar_full[s]), lp, tmo, err);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // Program order: QK(own tile of round 0); per round i: QK(own tile of
    // round i+1), PV(own P tile), PV(peer's P tile).
    if (lane == 0 && T > 0) {
      int slot = 0;
      uint32_t lap = 0;
      bool ok = true;
      auto take = [&]() -> int {
        const uint32_t fb = smem_u32(&bar_full[slot]);
        if (!mbar_try_wait(fb, lap) && !wait_bounded(fb, lap, &abort_flag, tmo, err)) return -1;
        const int s = slot;
        if (++slot == NS) { slot = 0; lap ^= 1u; }
        return s;
      };
      auto wait_on = [&](uint32_t bar, uint32_t par) -> bool {
        if (!mbar_try_wait(bar, par) && !wait_bounded(bar, par, &abort_flag, tmo, err)) return false;
        tc_fence_after();
        return true;
      };
      const uint32_t idesc_qk = idesc_f16(!fp16, BM, BN, false, false);
      const uint32_t idesc_pv = idesc_f16(!fp16, BM, it.dv, false, true);
      const uint64_t ring_desc = sdesc_sw128(ring_u32, 16, 1024);
      const uint64_t qs_desc = sdesc_sw128(qs_u32, 16, 1024);
      const uint64_t pown_desc = sdesc_sw128(pown_u32, 16, 1024);
      const uint64_t ppeer_desc = sdesc_sw128(ppeer_u32, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(ring_u32, vk * 128, 1024);
      const uint32_t s_col = tmem + S_COL;
      const uint32_t q_col = tmem + Q_TMEM_COL;
      ok = wait_on(smem_u32(&bar_q), 0) && wait_on(smem_u32(&bar_qt), 0);
      int nq = 0;
      auto qk = [&](int j) -> bool {
        (void)j;   // the producer loads tile j's stages in this order
        if (nq >= 1 && !wait_on(smem_u32(&bar_s_free), (nq - 1) & 1)) return false;
#pragma unroll
        for (int c = 0; c < nchunks; c += 2) {
          const int sk = take();
          if (sk < 0) return false;
          const uint64_t bd0 = ring_desc + ((sk * SLOT_BYTES) >> 4);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int ch = c + cc;
            const uint64_t bd = bd0 + cc * (CHUNK_BYTES >> 4);
            if (ch < qt) {
              // A from TMEM: 16 D-elements = 8 packed columns per MMA.
              const uint32_t a = q_col + 32 * ch;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_ts(s_col, a + 8 * k, bd + 2 * k, idesc_qk, (ch > 0 || k > 0) ? 1u : 0u);
            } else {
              const uint64_t ad = qs_desc + (((ch - qt) * CHUNK_BYTES) >> 4);
#pragma unroll
              for (int k = 0; k < 4; ++k) umma_ss(s_col, ad + 2 * k, bd + 2 * k, idesc_qk, 1u);
            }
          }
          umma_commit(smem_u32(&bar_empty[sk]));
        }
        umma_commit(smem_u32(&bar_s_full));
        ++nq;
        return true;
      };
      bool o_acc = false;
      auto pv = [&](uint64_t a_desc) -> bool {
#pragma unroll
        for (int h = 0; h < BN / vk; ++h) {
          const int s = take();
          if (s < 0) return false;
          const uint64_t vd = v_desc + ((s * SLOT_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < vk / 16; ++kk) {
            // 16 keys per MMA: P (K-major, 64-key chunks of 16 KB, +32 bytes
            // per 16 keys), V (MN-major, +2048 bytes per 16 keys).
            const int key = h * vk + 16 * kk;
            const uint64_t ad = a_desc + (((key >> 6) * CHUNK_BYTES) >> 4) + 2 * ((key & 63) >> 4);
            umma_ss(tmem, ad, vd + 128 * kk, idesc_pv, o_acc ? 1u : 0u);
            o_acc = true;
          }
          umma_commit(smem_u32(&bar_empty[s]));
        }
        return true;
      };
      if (ok && own0 < T) ok = qk(own0);
      int np = 0;
      for (int i = 0; i < R && ok; ++i) {
        if (2 * i + 2 + own0 < T && !(ok = qk(2 * i + 2 + own0))) break;
        // Softmax round i is done: own P written (if any) and O rescaled.
        if (!(ok = wait_on(smem_u32(&bar_pown_full), i & 1))) break;
        if (2 * i + own0 < T) {
          if (!(ok = pv(pown_desc))) break;
          umma_commit(smem_u32(&bar_pown_free));
        }
        if (2 * i + peer0 < T) {
          const uint32_t pb = smem_u32(&bar_ppeer_full);
          mbar_arrive_expect_tx(pb, P_TILE_BYTES);
          if (!(ok = wait_on(pb, np & 1))) break;
          if (!(ok = pv(ppeer_desc))) break;
          // The peer may overwrite its P tile and copy the next one here.
          umma_commit_mc(smem_u32(&bar_peer_free), (uint16_t)(1u << peer));
          ++np;
        }
        umma_commit(smem_u32(&bar_pv_done));
      }
      const uint32_t db = smem_u32(&bar_drain);
      umma_commit(db);
      wait_drain(db, 0, tmo, err);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int mask_kind = p.mask_kind;
    const bool causal = p.causal != 0;
    const float scale_log2 = p.scale_log2;
    const int r = warp * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int row = it.q0 + r;
    const bool row_valid = row < it.q_len;
    const long long row_limit = (long long)row + (it.kv_len - it.q_len);
    const long long first_limit = (long long)it.q0 + (it.kv_len - it.q_len);
    const uint8_t* mrow = nullptr;
    if (UMASK && mask_kind != FFPA_MASK_NONE && row_valid) {
      const size_t esz = mask_kind == FFPA_MASK_BOOL ? 1 : mask_kind == FFPA_MASK_ADD_F32 ? 4 : 2;
      const long long off = (long long)it.b * p.m_str[0] + (long long)it.hq * p.m_str[1] +
                            (long long)row * p.m_str[2];
      mrow = static_cast<const uint8_t*>(p.mask) + off * (long long)esz;
    }
    const long long mk = p.m_str[3];
    const bool prescale = mask_kind == FFPA_MASK_ADD_F32 || mask_kind == FFPA_MASK_ADD_QTYPE ||
                          !(scale_log2 > 0.f);
    const float xs = prescale ? 1.f : scale_log2;
    const float ld_scale = prescale ? scale_log2 : 1.f;
    bool ok = true;
    if (T > 0) {
      // Q chunks 0..qt-1: staging area -> TMEM (row r = lane r; the 32-bit
      // words of a row in memory order are the packed A-operand columns).
      bool w = wait_bounded(smem_u32(&bar_q), 0, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (ok) {
        const uint32_t sw = (uint32_t)(r & 7);
        for (int c = 0; c < qt; ++c) {
          uint32_t words[32];
          const uint32_t rowaddr = pown_u32 + c * CHUNK_BYTES + r * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 v = ld_shared_v4(rowaddr + (((uint32_t)u ^ sw) << 4));
            words[4 * u] = v.x;
            words[4 * u + 1] = v.y;
            words[4 * u + 2] = v.z;
            words[4 * u + 3] = v.w;
          }
          tmem_st32(lane_base + Q_TMEM_COL + 32 * c, words);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_qt));
        if (r == 0) {
          // All four warps have read the staging area: the peer may copy its
          // first P tile into this CTA's P (peer) area.
          w = wait_bounded(smem_u32(&bar_qt), 0, &abort_flag, tmo, err);
          if (w) mbar_arrive_cluster(mapa_shared(smem_u32(&bar_peer_free), peer));
        }
        ok = __all_sync(0xffffffffu, w);
      }
    }
    float m_ref = -INFINITY;
    float l_sum = 0.f;
    int k_own = 0;
    const uint32_t x_remote = mapa_shared(smem_u32(&xbuf[0][r]), peer);
    const uint32_t xbar_remote = mapa_shared(smem_u32(&bar_x[0]), peer);
    for (int i = 0; i < R && ok; ++i) {
      const bool own = 2 * i + own0 < T;
      float x[BN];
      float t = -INFINITY;
      if (own) {
        bool w = wait_bounded(smem_u32(&bar_s_full), k_own & 1, &abort_flag, tmo, err);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_addr = lane_base + S_COL;
        const int kbase = kv_tile(it, 2 * i + own0) * BN;
        const bool need_mask = (kbase + BN > it.kv_len) ||
                               (causal && (long long)kbase + BN - 1 > first_limit) ||
                               mask_kind != FFPA_MASK_NONE;
        {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32(s_addr, r0);
          tmem_ld32(s_addr + 32, r1);
          tmem_ld32(s_addr + 64, r2);
          tmem_ld32(s_addr + 96, r3);
          tmem_wait_ld();
          reg_fence(r0);
          reg_fence(r1);
          reg_fence(r2);
          reg_fence(r3);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bar_s_free));
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            x[c] = __uint_as_float(r0[c]);
            x[32 + c] = __uint_as_float(r1[c]);
            x[64 + c] = __uint_as_float(r2[c]);
            x[96 + c] = __uint_as_float(r3[c]);
          }
          if (prescale) {
#pragma unroll
            for (int c = 0; c < BN; ++c) x[c] *= ld_scale;
          }
        }
        if (need_mask) {
#pragma unroll
          for (int q4 = 0; q4 < BN / 32; ++q4) {
            apply_mask32<UMASK>(x + 32 * q4, kbase + 32 * q4, it.kv_len, causal, row_limit, mrow,
                                mk, mask_kind, fp16);
            if (UMASK) asm volatile("" ::: "memory");
          }
        }
        t = row_max<BN>(x) * xs;
      }
      // Exchange the tile maxima: both CTAs then take the same decision.
      const int xb = i & 1;
      const uint32_t xbar = smem_u32(&bar_x[xb]);
      if (r == 0) mbar_arrive_expect_tx(xbar, BM * 4);
      st_async_b32(x_remote + xb * BM * 4, __float_as_uint(t), xbar_remote + 8u * xb);
      {
        const bool w = wait_bounded(xbar, (i >> 1) & 1, &abort_flag, tmo, err, true);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
      }
      const float mx = fmaxf(t, ld_shared_f32(smem_u32(&xbuf[xb][r])));
      bool resc = false;
      float alpha = 1.f;
      if (mx > m_ref + RESCALE_LOG2) {
        if (m_ref != -INFINITY) {
          resc = true;
          alpha = ex2_approx(m_ref - mx);
        }
        m_ref = mx;
      }
      // P of the own tile (registers only: no dependence on the PV of the
      // previous round, so this overlaps it).
      l_sum *= alpha;
      uint32_t pk[BN / 2];
      if (own) {
        const float base = m_ref == -INFINITY ? 0.f : m_ref;
        // One branch per tile, not per element: the unrolled loop then holds
        // a single conversion per pair.
        l_sum += fp16 ? form_p<true, BN>(x, xs, base, pk) : form_p<false, BN>(x, xs, base, pk);
      }
      if (own) {
        // The own P area is free once the own PV of the previous own tile is
        // done and the peer has read the previous copy (which also frees the
        // peer's P area for this one).
        bool w = true;
        if (k_own >= 1)
          w = wait_bounded(smem_u32(&bar_pown_free), (k_own - 1) & 1, &abort_flag, tmo, err);
        if (w) w = wait_bounded(smem_u32(&bar_peer_free), k_own & 1, &abort_flag, tmo, err, true);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        // Row r of the P tile: 16 units of 8 keys, 128-byte swizzle.
        const uint32_t prow = pown_u32 + r * 128;
        const uint32_t sw = (uint32_t)(r & 7);
#pragma unroll
        for (int g = 0; g < BN / 8; ++g)
          st_shared_v4(prow + (g >> 3) * CHUNK_BYTES + ((((uint32_t)g & 7u) ^ sw) << 4), pk[4 * g],
                       pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        fence_proxy_async_smem();
      }
      if (i >= 1) {
        // PV of round i-1 done.  Waited every round (not only before a
        // rescale) so that each phase of this barrier is observed: a parity
        // wait cannot tell phase n from phase n-2.
        const bool w = wait_bounded(smem_u32(&bar_pv_done), (i - 1) & 1, &abort_flag, tmo, err);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
      }
      const bool resc_warp = __any_sync(0xffffffffu, resc);
      if (resc_warp) {
        // O holds the products of rounds < i: rescale this warp's rows.
        for (int c0 = 0; c0 < it.dv; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + c0, o);
          tmem_wait_ld();
          reg_fence(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st32(lane_base + c0, o);
        }
      }
      if (resc_warp) tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_pown_full));
      if (own) {
        // This warp's 32 rows of both 64-key chunks (2 x 4 KB, each
        // contiguous) to the peer, as soon as they are written.
        if (lane == 0) {
          const uint32_t pb = mapa_shared(smem_u32(&bar_ppeer_full), peer);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint32_t off = c * CHUNK_BYTES + warp * 32 * 128;
            bulk_copy_to_cta(mapa_shared(ppeer_u32 + off, peer), pown_u32 + off, 32 * 128, pb);
          }
        }
        ++k_own;
      }
    }
    // ------------------------------------------------------------ epilogue
    if (ok && R > 0) {
      bool w = wait_bounded(smem_u32(&bar_pv_done), (R - 1) & 1, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (ok) {
        tc_fence_after();
        // Row sums: each CTA summed the P of its own tiles.
        const uint32_t lbar = smem_u32(&bar_l);
        if (r == 0) mbar_arrive_expect_tx(lbar, BM * 4);
        st_async_b32(mapa_shared(smem_u32(&lbuf[r]), peer), __float_as_uint(l_sum),
                     mapa_shared(lbar, peer));
        w = wait_bounded(lbar, 0, &abort_flag, tmo, err, true);
        ok = __all_sync(0xffffffffu, w);
        if (ok) l_sum += ld_shared_f32(smem_u32(&lbuf[r]));
      }
    }
    if (ok || T == 0) {
      // The ring is idle once the last products are done; 16 KB per warp of
      // it stage the output boxes for tensor stores.  Varlen: only a tile
      // whose 128 rows all lie in its sequence (a box must not reach into
      // the next sequence's rows).
      if (p.o_tma && (!VARLEN || it.q0 + BM <= it.q_len))
        store_output_boxes<VARLEN>(p, it, T > 0, lane_base, warp, lane, row, row_valid, l_sum, m_ref,
                                   ring_u32 + (uint32_t)warp * 16384u);
      else
        store_output<VARLEN>(p, it, T > 0, lane_base, row, row_valid, l_sum, m_ref);
    }
    if (r == 0 && ok && T > 0) {
      // Before this CTA may exit: the peer has read every P tile copied to it.
      const int n_own = (T - own0 + 1) >> 1;
      wait_drain(smem_u32(&bar_peer_free), n_own & 1, tmo, err);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <bool VARLEN, bool UMASK>
static ffpa_status launch_split_t(const Params& P, int items, size_t smem, cudaStream_t stream) {
  if (P.split_c != 2 || (P.nchunks != 2 && P.nchunks != 4 && P.nchunks != 6 && P.nchunks != 8))
    return FFPA_ERR_UNSUPPORTED;   // only the instantiated shapes
  auto kern = P.nchunks == 8   ? ffpa_fwd_split_kernel<VARLEN, 8, UMASK>
              : P.nchunks == 6 ? ffpa_fwd_split_kernel<VARLEN, 6, UMASK>
              : P.nchunks == 4 ? ffpa_fwd_split_kernel<VARLEN, 4, UMASK>
                               : ffpa_fwd_split_kernel<VARLEN, 2, UMASK>;
  const ffpa_status st =
      set_smem_attr_once(reinterpret_cast<const void*>(kern), P.device, static_cast<int>(SMEM_LIMIT - SPLIT_STATIC_RESERVE));
  if (st != FFPA_OK) return st;
  kern<<<2 * items, SPLIT_THREADS, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}

ffpa_status launch_split(bool varlen, bool umask, const Params& P, int items, size_t smem,
                         cudaStream_t stream) {
  return varlen  ? launch_split_t<true, false>(P, items, smem, stream)
         : umask ? launch_split_t<false, true>(P, items, smem, stream)
                 : launch_split_t<false, false>(P, items, smem, stream);
}


}  // namespace ffpa
