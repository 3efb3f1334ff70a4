// FP8 (e4m3) column-split kernel: two SMs share a 128-row query tile, each owning half of
// the output columns, on the tensor cores' kind::f8f6f4 MMA.
#include "ffpa_common.cuh"

namespace ffpa {

// =====================================================================
// The column-split protocol of the 16-bit pair kernel (ffpa_split.cu) with
// the FP8 forward's operands and scales (ffpa_fp8.cu): block-quantised Q,
// K and transposed V from the caller's workspace, s_q s_k folded into each
// tile's softmax scale, the V block scale folded into P, and P in e4m3.
//
// A cluster of two CTAs owns one 128-row query tile; CTA c owns the output
// columns [c D/2, (c+1) D/2).  In round i CTA c computes S = Q K^T for key
// tile 2i + c over the full D, the two CTAs exchange their tile maxima (so
// that both take the same running maximum), and each CTA writes its P tile
// (e4m3, 16 KB) into its own shared memory and bulk-copies it into the
// peer's.  Both accumulate both P tiles against their half of V^T.  S is
// computed once per key tile, and at one byte per element Q stays resident
// in shared memory while the ring keeps four or more 32 KB stages.
//
// TMEM: O [0, D/2), S [256, 384).  Shared memory: Q (D/128 chunks of 16 KB,
// in 32 KB pairs) | P own (16 KB) | P peer (16 KB) | ring of 32 KB stages
// (K chunk pairs, V^T stages of D/2 rows x 128 keys).
// Warps: 0-3 softmax (thread r owns row r = TMEM lane r), 4 TMA producer,
// 5 MMA issuer.  Every wait is bounded; waits on phases that the peer CTA
// completes use cluster-scope acquire.
// =====================================================================

constexpr uint32_t F8S_P_BYTES = BM * BN;      // one e4m3 P tile: 128 rows x 128 keys
constexpr float F8S_RESCALE_LOG2 = 0.75f;      // as the single-CTA FP8 kernel: P <= 431 < 448

// P * c_t = exp2(x - base) for 32 scores as e4m3 (four per word, the first
// key in the lowest byte); returns the sum of the unrounded values.
__device__ __forceinline__ float form_p8s(const float* x, float base, uint32_t* w) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int c = 0; c < 32; c += 4) {
    float a0, a1, a2, a3;
    ffma2_bc(x[c], x[c + 1], 1.f, -base, a0, a1);
    ffma2_bc(x[c + 2], x[c + 3], 1.f, -base, a2, a3);
    const float e0 = ex2_approx(a0), e1 = ex2_approx(a1), e2 = ex2_approx(a2), e3 = ex2_approx(a3);
    fadd2_acc(s0, s1, e0, e1);
    fadd2_acc(s2, s3, e2, e3);
    w[c / 4] = pack_e4m3x4(e0, e1, e2, e3);
  }
  return (s0 + s1) + (s2 + s3);
}

// NCH8 = D / 128 (template: every MMA issue loop unrolls).
template <int NCH8, bool UMASK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(SPLIT_THREADS, 1)
    ffpa_fwd_fp8_split_kernel(const __grid_constant__ Params p) {
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  Item it;
  if (!decode_item(p, false, blockIdx.x >> 1, it)) return;   // same answer in both CTAs
  constexpr int DV = NCH8 * 128 / 2;                          // output columns per CTA
  it.dv = DV;
  it.col_lo = DV * (int)rank;
  it.slice = (int)rank;                                       // rank 0 writes the LSE
  constexpr int QPAIRS = (NCH8 + 1) / 2;                      // 32 KB boxes of two 128-byte chunks

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int inject = p.inject;
  const int NS = p.nslot;
  const uint32_t q_u32 = smem_u32(smem);
  const uint32_t pown_u32 = q_u32 + QPAIRS * SLOT_BYTES;
  const uint32_t ppeer_u32 = pown_u32 + F8S_P_BYTES;
  const uint32_t ring_u32 = ppeer_u32 + F8S_P_BYTES;
  __shared__ __align__(8) uint64_t bar_full[NSLOT_MAX], bar_empty[NSLOT_MAX];
  __shared__ __align__(8) uint64_t bar_q, bar_s_full, bar_s_free;
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
    // Q once; then one ring in the MMA thread's order: K of the first own
    // tile, then per round i: K of the own tile of round i+1, V^T (this
    // CTA's columns) of the own tile, V^T of the peer's tile.
    if (lane == 0 && T > 0) {
      prefetch_tmap(&p.tm_q);
      prefetch_tmap(&p.tm_k);
      prefetch_tmap(&p.tm_v);
      int slot = 0;
      uint32_t lap = 0;
      int issued = 0;
      bool ok = true;
      bool drop = inject != 0 && rank == 0;   // test hook (ffpa_options.test_drop_first_copy)
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
      // Boxes of two 128-byte chunks (the second one past D/128 reads zeros).
      const uint32_t qb = smem_u32(&bar_q);
      mbar_arrive_expect_tx(qb, QPAIRS * SLOT_BYTES);
      for (int pr = 0; pr < QPAIRS; ++pr)
        tma_load_5d(q_u32 + pr * SLOT_BYTES, &p.tm_q, qb, 0, it.q0, 2 * pr, it.hq, it.b);
      auto load_k = [&](int j) -> bool {
        const int key0 = kv_tile(it, j) * BN;
        for (int pr = 0; pr < QPAIRS; ++pr) {
          uint32_t fb = 0;
          const uint32_t dst = acquire(SLOT_BYTES, fb);
          if (dst == ~0u) return false;
          if (dst) tma_load_5d(dst, &p.tm_k, fb, 0, key0, 2 * pr, it.hkv, it.b);
        }
        return true;
      };
      auto load_v = [&](int j) -> bool {
        uint32_t fb = 0;
        const uint32_t dst = acquire((uint32_t)DV * 128u, fb);
        if (dst == ~0u) return false;
        tma_load_4d(dst, &p.tm_v, fb, kv_tile(it, j) * BN, it.col_lo, it.hkv, it.b);
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
      const uint32_t idesc_qk = idesc_e4m3(BM, BN);
      const uint32_t idesc_pv = idesc_e4m3(BM, DV);
      const uint64_t ring_desc = sdesc_sw128(ring_u32, 16, 1024);
      const uint64_t q_desc = sdesc_sw128(q_u32, 16, 1024);
      const uint64_t pown_desc = sdesc_sw128(pown_u32, 16, 1024);
      const uint64_t ppeer_desc = sdesc_sw128(ppeer_u32, 16, 1024);
      const uint32_t s_col = tmem + S_COL;
      ok = wait_on(smem_u32(&bar_q), 0);
      int nq = 0;
      auto qk = [&]() -> bool {
        if (nq >= 1 && !wait_on(smem_u32(&bar_s_free), (nq - 1) & 1)) return false;
#pragma unroll
        for (int pr = 0; pr < QPAIRS; ++pr) {
          const int sk = take();
          if (sk < 0) return false;
          const uint64_t ad = q_desc + (((uint32_t)pr * SLOT_BYTES) >> 4);
          const uint64_t bd = ring_desc + ((sk * SLOT_BYTES) >> 4);
          // 32 e4m3 per MMA: +32 bytes (>>4 = 2) within a 128-byte row; the
          // second chunk of the pair sits 16 KB (>>4 = 1024) further.
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_ss_f8(s_col, ad + 2 * k, bd + 2 * k, idesc_qk, (pr > 0 || k > 0) ? 1u : 0u);
          if (2 * pr + 1 < NCH8) {
#pragma unroll
            for (int k = 0; k < 4; ++k) umma_ss_f8(s_col, ad + 1024 + 2 * k, bd + 1024 + 2 * k, idesc_qk, 1u);
          }
          umma_commit(smem_u32(&bar_empty[sk]));
        }
        umma_commit(smem_u32(&bar_s_full));
        ++nq;
        return true;
      };
      bool o_acc = false;
      auto pv = [&](uint64_t a_desc) -> bool {
        const int s = take();
        if (s < 0) return false;
        const uint64_t vd = ring_desc + ((s * SLOT_BYTES) >> 4);
        // 32 keys per MMA: +32 bytes of P (K-major) and of V^T (K-major).
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          umma_ss_f8(tmem, a_desc + 2 * k, vd + 2 * k, idesc_pv, o_acc ? 1u : 0u);
          o_acc = true;
        }
        umma_commit(smem_u32(&bar_empty[s]));
        return true;
      };
      if (ok && own0 < T) ok = qk();
      int np = 0;
      for (int i = 0; i < R && ok; ++i) {
        if (2 * i + 2 + own0 < T && !(ok = qk())) break;
        // Softmax round i is done: own P written (if any) and O rescaled.
        if (!(ok = wait_on(smem_u32(&bar_pown_full), i & 1))) break;
        if (2 * i + own0 < T) {
          if (!(ok = pv(pown_desc))) break;
          umma_commit(smem_u32(&bar_pown_free));
        }
        if (2 * i + peer0 < T) {
          const uint32_t pb = smem_u32(&bar_ppeer_full);
          mbar_arrive_expect_tx(pb, F8S_P_BYTES);
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
    const bool fp16 = p.fp16 != 0, causal = p.causal != 0;
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
    // Block scales: this tile's Q block, and the head's K and V blocks; G is
    // the head's largest V scale (the same in both CTAs).
    const int Hkv = p.Hq / p.group;
    const float s_q = p.sq[((long long)it.b * p.Hq + it.hq) * p.n_qt + it.q0 / BM];
    const float* s_k = p.sk + ((long long)it.b * Hkv + it.hkv) * p.n_kb;
    const float* s_v = p.sv + ((long long)it.b * Hkv + it.hkv) * p.n_kb;
    float G = 0.f;
    for (int t = 0; t < p.n_kb; ++t) G = fmaxf(G, __ldg(s_v + t));
    const float inv_g256 = 256.f / G;
    float m_ref = -INFINITY;
    float l_sum = 0.f;
    int k_own = 0;
    bool ok = true;
    if (T > 0 && r == 0) {
      // The P (peer) area holds nothing at the start: the peer may copy its
      // first P tile at once.
      mbar_arrive_cluster(mapa_shared(smem_u32(&bar_peer_free), peer));
    }
    const uint32_t x_remote = mapa_shared(smem_u32(&xbuf[0][r]), peer);
    const uint32_t xbar_remote = mapa_shared(smem_u32(&bar_x[0]), peer);
    for (int i = 0; i < R && ok; ++i) {
      const bool own = 2 * i + own0 < T;
      const int tile = own ? kv_tile(it, 2 * i + own0) : 0;
      float x[BN];
      float t = -INFINITY;
      if (own) {
        bool w = wait_bounded(smem_u32(&bar_s_full), k_own & 1, &abort_flag, tmo, err);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        const int kbase = tile * BN;
        const bool need_mask = (kbase + BN > it.kv_len) ||
                               (causal && (long long)kbase + BN - 1 > first_limit) ||
                               mask_kind != FFPA_MASK_NONE;
        // Scores in the log2 domain: the tile's scale folds s_q s_k.
        const float f = p.scale_log2 * s_q * __ldg(s_k + tile);
        {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          const uint32_t s_addr = lane_base + S_COL;
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
            x[c] = __uint_as_float(r0[c]) * f;
            x[32 + c] = __uint_as_float(r1[c]) * f;
            x[64 + c] = __uint_as_float(r2[c]) * f;
            x[96 + c] = __uint_as_float(r3[c]) * f;
          }
        }
        if (need_mask) {
#pragma unroll
          for (int q4 = 0; q4 < BN / 32; ++q4) {
            apply_mask32<UMASK>(x + 32 * q4, kbase + 32 * q4, it.kv_len, causal, row_limit, mrow, mk,
                                mask_kind, fp16);
            if (UMASK) asm volatile("" ::: "memory");
          }
        }
        t = row_max<BN>(x);
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
      if (mx > m_ref + F8S_RESCALE_LOG2) {
        if (m_ref != -INFINITY) {
          resc = true;
          alpha = ex2_approx(m_ref - mx);
        }
        m_ref = mx;
      }
      l_sum *= alpha;
      // P * c_t in e4m3 (c_t = 256 s_v(t) / G): exp2(x - m_ref + log2 c_t);
      // the row sum keeps p.
      uint32_t pw[BN / 4];
      if (own) {
        const float c_t = __ldg(s_v + tile) * inv_g256;
        const float base = (m_ref == -INFINITY ? 0.f : m_ref) - __log2f(c_t);
        float psum = 0.f;
#pragma unroll
        for (int q4 = 0; q4 < BN / 32; ++q4) psum += form_p8s(x + 32 * q4, base, pw + 8 * q4);
        l_sum += psum / c_t;
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
        // Row r of the P tile: 128 keys = one 128-byte swizzle row (8 units
        // of 16 keys).
        const uint32_t prow = pown_u32 + r * 128;
        const uint32_t sw = (uint32_t)(r & 7);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(prow + ((((uint32_t)u) ^ sw) << 4), pw[4 * u], pw[4 * u + 1], pw[4 * u + 2],
                       pw[4 * u + 3]);
        fence_proxy_async_smem();
      }
      if (i >= 1) {
        // PV of round i-1 done (waited every round, so that each phase of
        // this barrier is observed).
        const bool w = wait_bounded(smem_u32(&bar_pv_done), (i - 1) & 1, &abort_flag, tmo, err);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
      }
      const bool resc_warp = __any_sync(0xffffffffu, resc);
      if (resc_warp) {
        // O holds the products of rounds < i: rescale this warp's rows.
        for (int c0 = 0; c0 < DV; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + c0, o);
          tmem_wait_ld();
          reg_fence(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st32(lane_base + c0, o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_pown_full));
      if (own) {
        // This warp's 32 rows (4 KB, contiguous) to the peer.
        if (lane == 0) {
          const uint32_t pb = mapa_shared(smem_u32(&bar_ppeer_full), peer);
          const uint32_t off = warp * 32 * 128;
          bulk_copy_to_cta(mapa_shared(ppeer_u32 + off, peer), pown_u32 + off, 32 * 128, pb);
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
        // Row sums: each CTA summed the p of its own tiles.
        const uint32_t lbar = smem_u32(&bar_l);
        if (r == 0) mbar_arrive_expect_tx(lbar, BM * 4);
        st_async_b32(mapa_shared(smem_u32(&lbuf[r]), peer), __float_as_uint(l_sum),
                     mapa_shared(lbar, peer));
        w = wait_bounded(lbar, 0, &abort_flag, tmo, err, true);
        ok = __all_sync(0xffffffffu, w);
        if (ok) l_sum += ld_shared_f32(smem_u32(&lbuf[r]));
      }
    }
    if (ok || T == 0)
      store_output<false>(p, it, T > 0, lane_base, row, row_valid, l_sum, m_ref, G / 256.f);
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

template <int NCH8>
static ffpa_status launch_fp8_split_t(bool umask, const Params& P, int items, size_t smem, cudaStream_t stream) {
  auto kern = umask ? ffpa_fwd_fp8_split_kernel<NCH8, true> : ffpa_fwd_fp8_split_kernel<NCH8, false>;
  const ffpa_status st = set_smem_attr_once(reinterpret_cast<const void*>(kern), P.device,
                                            static_cast<int>(SMEM_LIMIT - SPLIT_STATIC_RESERVE));
  if (st != FFPA_OK) return st;
  kern<<<2 * items, SPLIT_THREADS, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}

// The attention part of the FP8 forward on the column split (D = 256, 384,
// 512); the quantisation kernel has run on the same stream before.
ffpa_status launch_fp8_split(const Params& P, int items, size_t smem, cudaStream_t stream) {
  const bool umask = P.mask != nullptr;
  switch (P.D / 128) {
    case 2: return launch_fp8_split_t<2>(umask, P, items, smem, stream);
    case 3: return launch_fp8_split_t<3>(umask, P, items, smem, stream);
    case 4: return launch_fp8_split_t<4>(umask, P, items, smem, stream);
    default: return FFPA_ERR_UNSUPPORTED;
  }
}

}  // namespace ffpa
