// Dual-tile kernel: one CTA per 256 query rows (two 128-row tiles) sharing every K/V tile.
#include "ffpa_common.cuh"

namespace ffpa {

// =====================================================================
// Small head dimensions (D = 64, 128; dense batches).  There the MMA work
// of a key tile is small next to its softmax (128 exp2 per row whatever D
// is) and next to its K/V bytes, so the single-CTA kernel waits on both.
// Here one CTA owns two query tiles A (rows q0..q0+127) and B (rows
// q0+128..q0+255) of one head:
//  * each K and V tile is loaded once for both, halving the bytes per MMA
//    cycle;
//  * each tile has its own four softmax warps (warps 0-3 for A, 4-7 for B),
//    so while one group runs its exp2 work the tensor pipe computes the
//    other group's products: per key tile j the MMA thread issues
//    QK_A(j+1), QK_B(j+1), PV_A(j), PV_B(j), and a group has the whole
//    span of the other group's products to produce its P tile.
// TMEM columns: O_A [0, D), O_B [128, 128 + D), S_A [256, 384), S_B
// [384, 512).  P tiles (16-bit, K-major, 128-byte swizzle) go to shared
// memory and the PV products read them from there.
// Shared memory: Q_A | Q_B (D/64 chunks of 16 KB each) | P_A | P_B (32 KB
// each) | ring of one-tile slots (K_{j+1} then V_j per key tile).
// Warps: 0-7 softmax + epilogue, 8 TMA producer, 9 MMA issuer (and the
// TMEM allocation), 10-11 idle.  The third warpgroup exists so that
// registers can move by warpgroup: launched at 168 per thread (three warps
// on some SM sub-partitions), warpgroup 2 drops to DUAL_REGS_LOW and the two
// softmax warpgroups rise to DUAL_REGS_HIGH, whose sum fits the launch's
// 384 x 168 registers exactly.  Every wait is bounded.
// =====================================================================

constexpr int DUAL_THREADS = 384;
constexpr int DUAL_REGS_LAUNCH = 168;   // 65536 / 384, a multiple of 8
constexpr int DUAL_REGS_LOW = 88;       // warpgroup 2 (producer, MMA, idle)
constexpr int DUAL_REGS_HIGH = 208;     // warpgroups 0 and 1 (softmax)
static_assert(2 * 128 * DUAL_REGS_HIGH + 128 * DUAL_REGS_LOW <= DUAL_THREADS * DUAL_REGS_LAUNCH,
              "register split exceeds the launch's registers");
constexpr int DUAL_PRODUCER_WARP = 8;
constexpr int DUAL_MMA_WARP = 9;
constexpr int DUAL_NSLOT_MAX = 8;
constexpr uint32_t DUAL_S_COL = 256;     // S_A at 256, S_B at 384
constexpr uint32_t DUAL_O_STRIDE = 128;  // O_A at 0, O_B at 128

// Work item L: (batch, head, 256-row block).  Causal blocks longest first;
// otherwise the blocks of one head are adjacent (K/V reuse in L2).
__device__ __forceinline__ bool decode_dual(const Params& p, int L, Item& it) {
  const int heads = p.B * p.Hq;
  int blk;
  if (p.causal) {
    const int bh = L % heads;
    blk = p.n_qt - 1 - L / heads;
    it.hq = bh % p.Hq;
    it.b = bh / p.Hq;
  } else {
    blk = L % p.n_qt;
    const int bh = L / p.n_qt;
    it.hq = bh % p.Hq;
    it.b = bh / p.Hq;
  }
  it.hkv = it.hq / p.group;
  it.slice = 0;
  it.q_row0 = 0;
  it.kv_row0 = 0;
  it.q_len = p.Nq;
  it.kv_len = p.Nkv;
  it.q0 = blk * 2 * BM;
  if (it.q0 >= it.q_len) return false;
  const int rows = min(2 * BM, it.q_len - it.q0);
  long long kv_end = it.kv_len;
  if (p.causal) kv_end = min(kv_end, (long long)it.q0 + rows + (it.kv_len - it.q_len));
  it.ntiles = kv_end > 0 ? (int)((kv_end + BN - 1) / BN) : 0;
  it.rot = (it.ntiles > 0 && !p.causal)
               ? (int)(((unsigned)blk * 37u + (unsigned)it.hq * 13u) % (unsigned)it.ntiles)
               : 0;
  it.col_lo = 0;
  it.dv = p.D;
  return true;
}

// No caller's mask here (its loads need more registers than the softmax
// warps have); masked calls at these head dims run on the single-CTA kernel.
template <int NCH>
__global__ void __launch_bounds__(DUAL_THREADS, 1) ffpa_fwd_dual_kernel(const __grid_constant__ Params p) {
  Item it;
  if (!decode_dual(p, blockIdx.x, it)) return;   // uniform across the CTA

  constexpr uint32_t TILE_BYTES = NCH * CHUNK_BYTES;   // one Q, K or V tile
  const int inject = p.inject;
  const bool fp16 = p.fp16 != 0;
  const int NS = p.nslot;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t q_u32 = smem_u32(smem);                   // Q_A, then Q_B
  const uint32_t p_u32 = q_u32 + 2 * TILE_BYTES;           // P_A, then P_B
  const uint32_t ring_u32 = p_u32 + 2 * P_TILE_BYTES;
  __shared__ __align__(8) uint64_t bar_full[DUAL_NSLOT_MAX], bar_empty[DUAL_NSLOT_MAX];
  __shared__ __align__(8) uint64_t bar_q, bar_s_full[2], bar_s_free, bar_p_full, bar_pv_done[2];
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bar_full[i]), 1);
      mbar_init(smem_u32(&bar_empty[i]), 1);
    }
    mbar_init(smem_u32(&bar_q), 1);            // TMA bytes of Q_A and Q_B
    mbar_init(smem_u32(&bar_s_full[0]), 1);    // QK_A commit
    mbar_init(smem_u32(&bar_s_full[1]), 1);    // QK_B commit
    mbar_init(smem_u32(&bar_s_free), 8);       // softmax warps of both groups: S read
    mbar_init(smem_u32(&bar_p_full), 8);       // softmax warps of both groups: P written, O rescaled
    mbar_init(smem_u32(&bar_pv_done[0]), 1);   // PV_A commit
    mbar_init(smem_u32(&bar_pv_done[1]), 1);   // PV_B commit
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == DUAL_MMA_WARP) {
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

  if (warp >= 8) {
    // Each role branch starts with its warpgroup's register change, so that
    // the compiler allocates the branch under that budget.
    regs_lower<DUAL_REGS_LOW>();
    if (warp == DUAL_PRODUCER_WARP) {
      // ------------------------------------------------------------ producer
      // Q_A and Q_B once, then the ring in the MMA thread's order: K_0; per
      // key tile j: K_{j+1}, V_j.
      if (lane == 0 && T > 0) {
        prefetch_tmap(&p.tm_q);
        prefetch_tmap(&p.tm_k);
        prefetch_tmap(&p.tm_v);
        int slot = 0;
        uint32_t lap = 0;
        int issued = 0;
        bool ok = true;
        bool drop = inject != 0;   // test hook: the first K stage never lands
        auto acquire = [&](uint32_t& fb) -> uint32_t {
          const uint32_t eb = smem_u32(&bar_empty[slot]);
          if (!mbar_try_wait(eb, lap ^ 1u) && !wait_bounded_inl(eb, lap ^ 1u, &abort_flag, tmo, err))
            return ~0u;
          fb = smem_u32(&bar_full[slot]);
          const uint32_t dst = ring_u32 + slot * TILE_BYTES;
          ++issued;
          if (++slot == NS) { slot = 0; lap ^= 1u; }
          if (drop) {
            drop = false;
            return 0u;
          }
          mbar_arrive_expect_tx(fb, TILE_BYTES);
          return dst;
        };
        const uint32_t qb = smem_u32(&bar_q);
        mbar_arrive_expect_tx(qb, 2 * TILE_BYTES);
        // Rows of Q_B past Nq (a last block of 129..255 rows, or of <= 128
        // rows) arrive as zeros; their results are never stored.
        tma_load_5d(q_u32, &p.tm_q, qb, 0, it.q0, 0, it.hq, it.b);
        tma_load_5d(q_u32 + TILE_BYTES, &p.tm_q, qb, 0, it.q0 + BM, 0, it.hq, it.b);
        auto load = [&](const CUtensorMap* m, int j) -> bool {
          uint32_t fb = 0;
          const uint32_t dst = acquire(fb);
          if (dst == ~0u) return false;
          if (dst) tma_load_5d(dst, m, fb, 0, kv_tile(it, j) * BN, 0, it.hkv, it.b);
          return true;
        };
        ok = load(&p.tm_k, 0);
        for (int j = 0; j < T && ok; ++j) {
          if (j + 1 < T && !(ok = load(&p.tm_k, j + 1))) break;
          ok = load(&p.tm_v, j);
        }
        wait_drain_inl(qb, 0, tmo, err);
        const int n = issued < NS ? issued : NS;
        int s = slot;
        uint32_t lp = lap;
        for (int i = 0; i < n; ++i) {
          if (--s < 0) { s = NS - 1; lp ^= 1u; }
          if (inject != 0 && issued - 1 - i == 0) continue;   // never armed
          wait_drain_inl(smem_u32(&bar_full[s]), lp, tmo, err);
        }
      }
    } else if (warp == DUAL_MMA_WARP) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0 && T > 0) {
        int slot = 0;
        uint32_t lap = 0;
        bool ok = true;
        auto take = [&]() -> int {
          const uint32_t fb = smem_u32(&bar_full[slot]);
          if (!mbar_try_wait(fb, lap) && !wait_bounded_inl(fb, lap, &abort_flag, tmo, err)) return -1;
          const int s = slot;
          if (++slot == NS) { slot = 0; lap ^= 1u; }
          return s;
        };
        auto wait_on = [&](uint32_t bar, uint32_t par) -> bool {
          if (!mbar_try_wait(bar, par) && !wait_bounded_inl(bar, par, &abort_flag, tmo, err)) return false;
          tc_fence_after();
          return true;
        };
        const uint32_t idesc_qk = idesc_f16(!fp16, BM, BN, false, false);
        const uint32_t idesc_pv = idesc_f16(!fp16, BM, NCH * DK, false, true);
        const uint64_t ring_desc = sdesc_sw128(ring_u32, 16, 1024);
        const uint64_t q_desc = sdesc_sw128(q_u32, 16, 1024);
        const uint64_t p_desc = sdesc_sw128(p_u32, 16, 1024);
        const uint64_t v_desc = sdesc_sw128(ring_u32, CHUNK_BYTES, 1024);
        // S_g = Q_g K^T over D: 4 MMAs of 16 D-elements per 64-column chunk
        // (+32 bytes each, >>4 = 2), chunks 16 KB apart.
        auto qk = [&](int g, int sk) {
          const uint32_t s_col = tmem + DUAL_S_COL + 128u * g;
          const uint64_t ad = q_desc + (((uint32_t)g * TILE_BYTES) >> 4);
          const uint64_t bd = ring_desc + ((sk * TILE_BYTES) >> 4);
#pragma unroll
          for (int c = 0; c < NCH; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_ss(s_col, ad + c * (CHUNK_BYTES >> 4) + 2 * k, bd + c * (CHUNK_BYTES >> 4) + 2 * k,
                      idesc_qk, (c > 0 || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&bar_s_full[g]));
        };
        // O_g += P_g V: 8 MMAs of 16 keys; P K-major (64-key chunks of 16 KB,
        // +32 bytes per 16 keys), V MN-major (+2048 bytes per 16 keys).
        auto pv = [&](int g, int sv, bool acc) {
          const uint32_t o_col = tmem + DUAL_O_STRIDE * g;
          const uint64_t ad0 = p_desc + (((uint32_t)g * P_TILE_BYTES) >> 4);
          const uint64_t vd = v_desc + ((sv * TILE_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const int key = 16 * kk;
            const uint64_t ad = ad0 + (((key >> 6) * CHUNK_BYTES) >> 4) + 2 * ((key & 63) >> 4);
            umma_ss(o_col, ad, vd + 128 * kk, idesc_pv, (acc || kk > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&bar_pv_done[g]));
        };
        ok = wait_on(smem_u32(&bar_q), 0);
        int sk = ok ? take() : -1;
        if (sk < 0) ok = false;
        if (ok) {
          qk(0, sk);
          qk(1, sk);
          umma_commit(smem_u32(&bar_empty[sk]));
        }
        for (int j = 0; j < T && ok; ++j) {
          if (j + 1 < T) {
            if ((sk = take()) < 0) { ok = false; break; }
            // Both groups have read S(j) into registers.
            if (!(ok = wait_on(smem_u32(&bar_s_free), j & 1))) break;
            qk(0, sk);
            qk(1, sk);
            umma_commit(smem_u32(&bar_empty[sk]));
          }
          const int sv = take();
          if (sv < 0) { ok = false; break; }
          // Both groups have written P(j) and rescaled their O where needed.
          if (!(ok = wait_on(smem_u32(&bar_p_full), j & 1))) break;
          pv(0, sv, j > 0);
          pv(1, sv, j > 0);
          umma_commit(smem_u32(&bar_empty[sv]));
        }
        const uint32_t db = smem_u32(&bar_drain);
        umma_commit(db);
        wait_drain_inl(db, 0, tmo, err);
      }
    }
  } else {
    regs_raise<DUAL_REGS_HIGH>();
    // ------------------------------------------------------------ softmax
    // Group g (0: warps 0-3, tile A; 1: warps 4-7, tile B); thread r owns
    // row q0 + 128 g + r of the block, TMEM lane r.
    const int g = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const bool causal = p.causal != 0;
    const float scale_log2 = p.scale_log2;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t s_addr = lane_base + DUAL_S_COL + 128u * g;
    const uint32_t o_base = lane_base + DUAL_O_STRIDE * g;
    const int row = it.q0 + BM * g + r;
    const bool row_valid = row < it.q_len;
    const long long row_limit = (long long)row + (it.kv_len - it.q_len);
    const long long first_limit = (long long)it.q0 + BM * g + (it.kv_len - it.q_len);
    // Scores stay unscaled (x = q.k) so that the exponent is one FFMA, unless
    // the scale is <= 0 (which reverses the maximum).
    const bool prescale = !(scale_log2 > 0.f);
    const float xs = prescale ? 1.f : scale_log2;
    const float ld_scale = prescale ? scale_log2 : 1.f;
    const uint32_t prow = p_u32 + (uint32_t)g * P_TILE_BYTES + r * 128;
    const uint32_t sw = (uint32_t)(r & 7);
    const uint32_t pvb = smem_u32(&bar_pv_done[g]);
    float m_ref = -INFINITY;
    float l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < T && ok; ++j) {
      // Each wait tests the barrier once before entering the bounded loop.
      bool w = mbar_try_wait(smem_u32(&bar_s_full[g]), j & 1) ||
               wait_bounded_inl(smem_u32(&bar_s_full[g]), j & 1, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      tc_fence_after();
      const int kbase = kv_tile(it, j) * BN;
      const bool need_mask = (kbase + BN > it.kv_len) ||
                             (causal && (long long)kbase + BN - 1 > first_limit);
      float x[BN];
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
          apply_mask32<false>(x + 32 * q4, kbase + 32 * q4, it.kv_len, causal, row_limit, nullptr, 0,
                              FFPA_MASK_NONE, fp16);
        }
      }
      const float mx = row_max<BN>(x) * xs;   // log2 domain
      bool resc = false;
      float alpha = 1.f;
      if (mx > m_ref + RESCALE_LOG2) {
        if (m_ref != -INFINITY) {
          resc = true;
          alpha = ex2_approx(m_ref - mx);
        }
        m_ref = mx;
      }
      if (j >= 1) {
        // PV_g(j-1) done: P_g may be overwritten and O_g holds tiles < j.
        // Waited every tile, so that each phase of the barrier is observed;
        // waiting before the exponentials lets P go to shared memory 32 keys
        // at a time (no 64-register P row).
        w = mbar_try_wait(pvb, (j - 1) & 1) || wait_bounded_inl(pvb, (j - 1) & 1, &abort_flag, tmo, err);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, resc)) {
        for (int c0 = 0; c0 < NCH * DK; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(o_base + c0, o);
          tmem_wait_ld();
          reg_fence(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st32(o_base + c0, o);
        }
        tmem_wait_st();
      }
      // P = exp2(x - m) in 16-bit; row r of P_g: 16 units of 8 keys,
      // 128-byte swizzle, 64-key chunks.
      const float base = m_ref == -INFINITY ? 0.f : m_ref;
      float psum = 0.f;
#pragma unroll
      for (int q4 = 0; q4 < BN / 32; ++q4) {
        uint32_t pk[16];
        psum += fp16 ? form_p<true, 32>(x + 32 * q4, xs, base, pk)
                     : form_p<false, 32>(x + 32 * q4, xs, base, pk);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t u = (uint32_t)(4 * q4 + v);
          st_shared_v4(prow + (u >> 3) * CHUNK_BYTES + (((u & 7u) ^ sw) << 4), pk[4 * v],
                       pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_p_full));
      l_sum = l_sum * alpha + psum;
    }
    // ------------------------------------------------------------ epilogue
    if (ok && T > 0) {
      const bool w = wait_bounded_inl(pvb, (T - 1) & 1, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (ok) tc_fence_after();
    }
    if (ok || T == 0) store_output<false>(p, it, T > 0, o_base, row, row_valid, l_sum, m_ref);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == DUAL_MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

ffpa_status launch_dual(bool umask, const Params& P, int items, size_t smem, cudaStream_t stream) {
  if (umask) return FFPA_ERR_UNSUPPORTED;                              // see the kernel
  if (P.nchunks != 1 && P.nchunks != 2) return FFPA_ERR_UNSUPPORTED;   // only the instantiated shapes
  if (P.nslot < 2 || P.nslot > DUAL_NSLOT_MAX) return FFPA_ERR_UNSUPPORTED;
  auto kern = P.nchunks == 2 ? ffpa_fwd_dual_kernel<2> : ffpa_fwd_dual_kernel<1>;
  const ffpa_status st = set_smem_attr_once(reinterpret_cast<const void*>(kern), P.device,
                                            static_cast<int>(SMEM_LIMIT - SMEM_STATIC_RESERVE));
  if (st != FFPA_OK) return st;
  // The register split assumes the launch allocates DUAL_REGS_LAUNCH per
  // thread; with fewer, the softmax warpgroups' increase could never be
  // granted.  The compiled counts are looked up once per process.
  static const bool regs_ok = [] {
    cudaFuncAttributes a1{}, a2{};
    const bool ok =
        cudaFuncGetAttributes(&a1, reinterpret_cast<const void*>(ffpa_fwd_dual_kernel<1>)) == cudaSuccess &&
        cudaFuncGetAttributes(&a2, reinterpret_cast<const void*>(ffpa_fwd_dual_kernel<2>)) == cudaSuccess &&
        a1.numRegs == DUAL_REGS_LAUNCH && a2.numRegs == DUAL_REGS_LAUNCH;
    cudaGetLastError();
    return ok;
  }();
  if (!regs_ok) return FFPA_ERR_UNSUPPORTED;
  kern<<<items, DUAL_THREADS, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}

}  // namespace ffpa
