// Stored-tile backward: P and dS formed once per (query tile, key tile), then dQ, dV and dK
// as plain contractions over the stored tiles.
#include "ffpa_bwd_common.cuh"

namespace ffpa {

using namespace bwd;

// =====================================================================
// Backward by stored score tiles (dense layout, D = 256, 384, 512).
//
// The gradients (backward of FFPAAttnFunc, FFPA API reference,
// "ffpa_attn.ffpa_attn_func") need, per query row i and key j,
//   P  = exp(scale q_i . k_j + mask - LSE_i)   and
//   dS = P (dO_i . v_j - delta_i),
// and then dQ = scale dS K, dV = P^T dO, dK = scale dS^T Q.  The sliced
// kernels of ffpa_bwd.cu keep every output tile in TMEM and recompute S and
// dP for each 256-column output slice: at D = 512 that executes 13 D
// multiply-adds per score against the 5 D of the definition.  Here the
// scores kernel forms P and dS (times scale) once per 128 x 128 tile and
// writes them as 16-bit values to a workspace; the contraction kernel then
// computes the three products, each multiply-add once.  The workspace
// (2 x B Hq Nq Nkv 16-bit values, padded to whole tiles) is written once and
// read three times (P once, dS twice); at D = 512 that is a few percent of
// the time the multiply-adds take.
//
// Scores kernel: one CTA per (batch, query head, 128-row query tile, range
// of its visible key tiles).
//   TMEM     Q in columns [0, D/2) (A operand of S = Q K^T), S [256, 384),
//            dP [384, 512).
//   smem     dO, resident (A operand of dP = dO V^T; at start the staging
//            area of Q on its way into TMEM), then a ring of 32 KB stages:
//            per key tile, K then V in pairs of 64-column chunks.
//   warps    0-7 elementwise: warp w owns TMEM lanes 32 (w % 4) .. +31
//            (query rows) and key columns 64 (w / 4) .. +63 of every tile;
//            8 TMA producer (the ring); 9 MMA issuer (also loads Q and dO).
//   Per key tile the MMA thread issues S, then dP.  The elementwise warps
//   read S, form P (kept in registers) and hand S's columns back while dP is
//   still on the tensor core, so the next tile's S follows without a gap;
//   then they read dP and form dS.  Rows go to the workspace with 16-byte
//   stores.
//
// Contraction kernel: one CTA per output tile of 128 rows x D columns (the
// whole row in TMEM, up to 512 fp32 columns):
//   dQ tile   one query tile of one query head, summed over its visible key
//             tiles: A = stored dS tile (K-major), B = K (MN-major);
//   dV tile   one key tile of one KV head, summed over the group's query
//             heads and the query tiles that see it: A = stored P tile read
//             as P^T (the same bytes, MN-major), B = dO (MN-major);
//   dK tile   as dV with dS and Q.
//   Warps 0-3 epilogue (TMEM -> 16-bit rows), 4 TMA producer, 5 MMA issuer.
//   The three kinds of items are interleaved in one launch (each kind's own
//   order puts its longest items first under causal masking).
// Every wait is bounded (FFPA_ERR_DEVICE_TIMEOUT on expiry, as elsewhere).
// =====================================================================

namespace {

constexpr uint32_t TS_S_COL = 256;
constexpr uint32_t TS_DP_COL = 384;
constexpr int TS_PRODUCER_WARP = 8;
constexpr int TS_MMA_WARP = 9;
constexpr int TC_PRODUCER_WARP = 4;
constexpr int TC_MMA_WARP = 5;

}  // namespace

// NCH = D / 64 (4, 6 or 8): every MMA issue loop has a compile-time trip count.
template <int NCH, bool UMASK>
__global__ void __launch_bounds__(TS_THREADS, 1) ffpa_bwd_scores_kernel(const __grid_constant__ BwdParams p) {
  constexpr int NPR = NCH / 2;   // 32 KB stages per K (or V) tile
  const int part = blockIdx.x % p.kv_parts;
  BwdItem it;
  if (!bwd_decode<true>(p, blockIdx.x / p.kv_parts, it)) return;   // uniform across the CTA
  const int j0 = (int)((long long)it.n_iter * part / p.kv_parts);
  const int j1 = (int)((long long)it.n_iter * (part + 1) / p.kv_parts);
  const int T = j1 - j0;
  if (T <= 0) return;

  const bool fp16 = p.fp16 != 0, causal = p.causal != 0;
  const int NS = p.ts_nslot;
  const unsigned long long tmo = p.timeout_ns;
  int* const err = p.err;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t do_u32 = smem_u32(smem);                      // NCH chunks: Q staging, then dO
  const uint32_t ring_u32 = do_u32 + NCH * CHUNK_BYTES;
  __shared__ __align__(8) uint64_t bar_full[TS_NSLOT_MAX], bar_empty[TS_NSLOT_MAX];
  __shared__ __align__(8) uint64_t bar_q, bar_qt, bar_do, bar_s_full, bar_s_free, bar_dp_full, bar_dp_free;
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
    mbar_init(smem_u32(&bar_q), 1);         // TMA bytes of Q
    mbar_init(smem_u32(&bar_qt), 8);        // elementwise warps: Q in TMEM, staging area read
    mbar_init(smem_u32(&bar_do), 1);        // TMA bytes of dO
    mbar_init(smem_u32(&bar_s_full), 1);    // S commit
    mbar_init(smem_u32(&bar_s_free), 8);    // elementwise warps: S read
    mbar_init(smem_u32(&bar_dp_full), 1);   // dP commit
    mbar_init(smem_u32(&bar_dp_free), 8);   // elementwise warps: dP read
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == TS_MMA_WARP) {
    tmem_alloc(smem_u32(&tmem_base_sh), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t qb = smem_u32(&bar_q);

  if (warp == TS_PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    // Per key tile: K chunk pairs, then V chunk pairs (the MMA thread's order).
    if (lane == 0) {
      prefetch_tmap(&p.tm_k);
      prefetch_tmap(&p.tm_v);
      int slot = 0, issued = 0;
      uint32_t lap = 0;
      // Test hook: the CTA's first ring stage is acquired but never armed or
      // copied, so the MMA thread's wait on it runs out.
      bool drop = p.inject != 0;
      auto load = [&](const CUtensorMap* m, int row, int chunk) -> bool {
        const uint32_t eb = smem_u32(&bar_empty[slot]);
        if (!mbar_try_wait(eb, lap ^ 1u) && !wait_bounded(eb, lap ^ 1u, &abort_flag, tmo, err)) return false;
        const uint32_t fb = smem_u32(&bar_full[slot]);
        if (drop) {
          drop = false;
        } else {
          mbar_arrive_expect_tx(fb, SLOT_BYTES);
          tma_load_5d(ring_u32 + slot * SLOT_BYTES, m, fb, 0, row, chunk, it.hkv, it.b);
        }
        ++issued;
        if (++slot == NS) { slot = 0; lap ^= 1u; }
        return true;
      };
      bool ok = true;
      for (int j = j0; j < j1 && ok; ++j) {
        for (int pr = 0; pr < NPR && ok; ++pr) ok = load(&p.tm_k, j * BN, 2 * pr);
        for (int pr = 0; pr < NPR && ok; ++pr) ok = load(&p.tm_v, j * BN, 2 * pr);
      }
      // Drain: every copy started here has landed before the CTA exits.
      const int n = issued < NS ? issued : NS;
      int s = slot;
      uint32_t lp = lap;
      for (int i = 0; i < n; ++i) {
        if (--s < 0) { s = NS - 1; lp ^= 1u; }
        if (p.inject != 0 && issued - 1 - i == 0) continue;   // the dropped stage was never armed
        wait_drain(smem_u32(&bar_full[s]), lp, tmo, err);
      }
    }
  } else if (warp == TS_MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      prefetch_tmap(&p.tm_q);
      prefetch_tmap(&p.tm_do);
      const uint32_t db = smem_u32(&bar_do);
      mbar_arrive_expect_tx(qb, (uint32_t)NCH * CHUNK_BYTES);
      for (int pr = 0; pr < NPR; ++pr)
        tma_load_5d(do_u32 + pr * SLOT_BYTES, &p.tm_q, qb, 0, it.row0, 2 * pr, it.hq, it.b);
      int slot = 0;
      uint32_t lap = 0;
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
      // Q is in TMEM and the staging area has been read: dO takes its place.
      bool ok = wait_on(smem_u32(&bar_qt), 0);
      const bool do_issued = ok;
      if (ok) {
        mbar_arrive_expect_tx(db, (uint32_t)NCH * CHUNK_BYTES);
        for (int pr = 0; pr < NPR; ++pr)
          tma_load_5d(do_u32 + pr * SLOT_BYTES, &p.tm_do, db, 0, it.row0, 2 * pr, it.hq, it.b);
      }
      const uint32_t idesc = idesc_f16(!fp16, BM, BN, false, false);
      // K-major operands: +32 bytes per 16 D-elements, +16 KB per chunk.
      const uint64_t ring_k = sdesc_sw128(ring_u32, 16, 1024);
      const uint64_t do_desc = sdesc_sw128(do_u32, 16, 1024);
      for (int j = 0; j < T && ok; ++j) {
        // S = Q K^T, A from TMEM (16 D-elements = 8 packed columns per MMA).
        if (j >= 1 && !(ok = wait_on(smem_u32(&bar_s_free), (j - 1) & 1))) break;
#pragma unroll
        for (int pr = 0; pr < NPR; ++pr) {
          const int sk = take();
          if (sk < 0) { ok = false; break; }
          const uint64_t bd0 = ring_k + ((sk * SLOT_BYTES) >> 4);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int ch = 2 * pr + cc;
            const uint32_t a = tmem + 32 * ch;
            const uint64_t bd = bd0 + cc * (CHUNK_BYTES >> 4);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_ts(tmem + TS_S_COL, a + 8 * k, bd + 2 * k, idesc, (ch > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&bar_empty[sk]));
        }
        if (!ok) break;
        umma_commit(smem_u32(&bar_s_full));
        // dP = dO V^T, both operands from shared memory.
        if (j == 0 && !(ok = wait_on(db, 0))) break;
        if (j >= 1 && !(ok = wait_on(smem_u32(&bar_dp_free), (j - 1) & 1))) break;
#pragma unroll
        for (int pr = 0; pr < NPR; ++pr) {
          const int sv = take();
          if (sv < 0) { ok = false; break; }
          const uint64_t bd0 = ring_k + ((sv * SLOT_BYTES) >> 4);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int ch = 2 * pr + cc;
            const uint64_t ad = do_desc + ((ch * CHUNK_BYTES) >> 4);
            const uint64_t bd = bd0 + cc * (CHUNK_BYTES >> 4);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_ss(tmem + TS_DP_COL, ad + 2 * k, bd + 2 * k, idesc, (ch > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&bar_empty[sv]));
        }
        if (!ok) break;
        umma_commit(smem_u32(&bar_dp_full));
      }
      const uint32_t drb = smem_u32(&bar_drain);
      umma_commit(drb);
      wait_drain(drb, 0, tmo, err);
      wait_drain(qb, 0, tmo, err);
      if (do_issued) wait_drain(db, 0, tmo, err);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    const int quad = warp & 3, half = warp >> 2;
    const int r = 32 * quad + lane;                 // TMEM lane = query row of the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * quad) << 16);
    // Q chunks (this warp: chunks of parity `half`) from the staging area
    // into TMEM: row r = lane r, the 32-bit words of a row in memory order
    // are the packed A-operand columns.
    bool w = wait_bounded(qb, 0, &abort_flag, tmo, err);
    bool ok = __all_sync(0xffffffffu, w);
    if (ok) {
      const uint32_t sw = (uint32_t)(r & 7);
      for (int c = half; c < NCH; c += 2) {
        uint32_t words[32];
        const uint32_t rowaddr = do_u32 + c * CHUNK_BYTES + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = ld_shared_v4(rowaddr + (((uint32_t)u ^ sw) << 4));
          words[4 * u] = v.x;
          words[4 * u + 1] = v.y;
          words[4 * u + 2] = v.z;
          words[4 * u + 3] = v.w;
        }
        tmem_st32(lane_base + 32 * c, words);
      }
      tmem_wait_st();
      fence_proxy_async_smem();   // the staging area is rewritten by the dO copy next
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_qt));
    }
    const int my_row = it.row0 + r;
    float lse_r = INFINITY, delta_r = 0.f;
    if (my_row < it.q_len) {
      const long long li = bwd_stat_index(p, it, it.hq, my_row);
      const float l = p.lse[li];
      lse_r = l > -INFINITY ? l * LOG2E_F : INFINITY;   // a row with no softmax has P = 0
      delta_r = p.delta[li];
    }
    const float sl2 = p.scale_log2, sc = p.scale;
    const long long off = (long long)it.kv_len - it.q_len;   // tail alignment of the causal limit
    const int mkind = p.mask_kind;
    const uint8_t* mbase = static_cast<const uint8_t*>(p.mask);
    long long mrow = 0;
    if (UMASK)
      mrow = (long long)it.b * p.m_str[0] + (long long)it.hq * p.m_str[1] + (long long)my_row * p.m_str[2];
    const long long mstep = UMASK ? p.m_str[3] : 0;
    // This thread's row of the stored P and dS (every row of the tile is
    // written, zeros where the row or key is out of range).
    const long long ws_off =
        ((long long)(it.b * p.Hq + it.hq) * (p.n_qt * BM) + my_row) * p.ws_ld + 64 * half;
    uint8_t* const prow = static_cast<uint8_t*>(p.ws_p) + ws_off * 2;
    uint8_t* const dsrow = static_cast<uint8_t*>(p.ws_ds) + ws_off * 2;
    const int c_lo = 64 * half;
    for (int jj = 0; jj < T && ok; ++jj) {
      const int rs = (j0 + jj) * BN;   // first key of the tile
      w = wait_bounded(smem_u32(&bar_s_full), jj & 1, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      tc_fence_after();
      const bool need_mask = (long long)rs + BN > it.kv_len ||
                             (causal && (long long)rs + BN - 1 > (long long)it.row0 + off);
      const long long lim = (long long)my_row + off - rs;   // last visible column
      const int kv_cols = it.kv_len - rs;                   // key columns in range
      const int mcols = (UMASK && my_row < it.q_len) ? kv_cols : 0;
      const long long moff = mrow + (long long)rs * mstep;
      float pv[64];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t sr[16];
        tmem_ld16(lane_base + TS_S_COL + c_lo + 16 * g, sr);
        tmem_wait_ld();
        reg_fence(sr);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = c_lo + 16 * g + e;
          float arg = fmaf(__uint_as_float(sr[e]), sl2, -lse_r);
          if (UMASK && col < mcols) arg = add_mask_term(arg, mbase, moff + col * mstep, mkind, fp16);
          float v = ex2_approx(arg);
          if (need_mask) {
            const bool vis = col < kv_cols && (!causal || (long long)col <= lim);
            v = vis ? v : 0.f;
          }
          pv[16 * g + e] = v;
        }
      }
      // S is in registers: the next tile's S may overwrite it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_s_free));
      {
        uint4* dst = reinterpret_cast<uint4*>(prow + (long long)rs * 2);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float* x = pv + 8 * q;
          dst[q] = fp16 ? make_uint4(pack_f16(x[0], x[1]), pack_f16(x[2], x[3]), pack_f16(x[4], x[5]),
                                     pack_f16(x[6], x[7]))
                        : make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                                     pack_bf16(x[6], x[7]));
        }
      }
      w = wait_bounded(smem_u32(&bar_dp_full), jj & 1, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      tc_fence_after();
      uint4* dst = reinterpret_cast<uint4*>(dsrow + (long long)rs * 2);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t dr[16];
        tmem_ld16(lane_base + TS_DP_COL + c_lo + 16 * g, dr);
        tmem_wait_ld();
        reg_fence(dr);
        if (g == 3) {
          // dP is in registers: the next tile's dP may overwrite it.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bar_dp_free));
        }
        float x[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = pv[16 * g + e] * sc * (__uint_as_float(dr[e]) - delta_r);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float* y = x + 8 * q;
          dst[2 * g + q] = fp16 ? make_uint4(pack_f16(y[0], y[1]), pack_f16(y[2], y[3]),
                                             pack_f16(y[4], y[5]), pack_f16(y[6], y[7]))
                                : make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]),
                                             pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == TS_MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Role and rank of contraction item L: dQ, dV and dK items interleaved
// (rank r of each kind at 3 r, 3 r + 1, 3 r + 2), then the remaining items
// of the more numerous kind.
__device__ __forceinline__ void contract_role(const BwdParams& p, int L, int& role, int& rank) {
  const int m = min(p.n_dq_items, p.n_kv_items);
  if (L < 3 * m) {
    role = L % 3;   // BWD_ROLE_DQ, BWD_ROLE_DV, BWD_ROLE_DK
    rank = L / 3;
  } else if (p.n_dq_items > p.n_kv_items) {
    role = BWD_ROLE_DQ;
    rank = m + (L - 3 * m);
  } else {
    role = 1 + (L - 3 * m) % 2;
    rank = m + (L - 3 * m) / 2;
  }
}

template <int NCH>
__global__ void __launch_bounds__(TC_THREADS, 1) ffpa_bwd_contract_kernel(const __grid_constant__ BwdParams p) {
  constexpr int NPR = NCH / 2;   // 32 KB B-operand stages per contraction step (128 output columns each)
  int role, rank;
  contract_role(p, blockIdx.x, role, rank);
  const bool dq_role = role == BWD_ROLE_DQ;
  BwdItem it;
  const bool have = dq_role ? bwd_decode<true>(p, rank, it) : bwd_decode<false>(p, rank, it);
  if (!have) return;   // uniform across the CTA
  const int T = it.n_iter;
  const bool fp16 = p.fp16 != 0;
  const int NS = p.tc_nslot;
  const unsigned long long tmo = p.timeout_ns;
  int* const err = p.err;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t ring_u32 = smem_u32(smem);
  __shared__ __align__(8) uint64_t bar_full[TC_NSLOT_MAX], bar_empty[TC_NSLOT_MAX];
  __shared__ __align__(8) uint64_t bar_acc, bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bar_full[i]), 1);
      mbar_init(smem_u32(&bar_empty[i]), 1);
    }
    mbar_init(smem_u32(&bar_acc), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == TC_MMA_WARP) {
    tmem_alloc(smem_u32(&tmem_base_sh), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int nqp = p.n_qt * BM;

  if (warp == TC_PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    // Per contraction step: the stored tile (A), then the B operand's chunk pairs.
    if (lane == 0 && T > 0) {
      const CUtensorMap* amap = role == BWD_ROLE_DV ? &p.tm_ws_p : &p.tm_ws_ds;
      const CUtensorMap* bmap = dq_role ? &p.tm_k : role == BWD_ROLE_DV ? &p.tm_do : &p.tm_q;
      prefetch_tmap(amap);
      prefetch_tmap(bmap);
      int slot = 0, issued = 0;
      uint32_t lap = 0;
      bool drop = p.inject != 0;   // test hook, as in the scores kernel
      auto acquire = [&](uint32_t& fb) -> uint32_t {
        const uint32_t eb = smem_u32(&bar_empty[slot]);
        if (!mbar_try_wait(eb, lap ^ 1u) && !wait_bounded(eb, lap ^ 1u, &abort_flag, tmo, err)) return ~0u;
        fb = smem_u32(&bar_full[slot]);
        const uint32_t dst = ring_u32 + slot * SLOT_BYTES;
        ++issued;
        if (++slot == NS) { slot = 0; lap ^= 1u; }
        if (drop) {
          drop = false;
          return 0u;
        }
        mbar_arrive_expect_tx(fb, SLOT_BYTES);
        return dst;
      };
      bool ok = true;
      for (int i = 0; i < T && ok; ++i) {
        int ws_row, ws_kc, b_row, b_head;
        if (dq_role) {
          ws_row = (it.b * p.Hq + it.hq) * nqp + it.row0;
          ws_kc = i * (BN / DK);
          b_row = i * BN;
          b_head = it.hkv;
        } else {
          const int hs = it.hq + i / it.nq;
          const int qrow = (it.qt_first + i % it.nq) * BM;
          ws_row = (it.b * p.Hq + hs) * nqp + qrow;
          ws_kc = it.row0 / DK;
          b_row = qrow;
          b_head = hs;
        }
        uint32_t fb = 0;
        uint32_t dst = acquire(fb);
        if (dst == ~0u) { ok = false; break; }
        if (dst) tma_load_3d(dst, amap, fb, 0, ws_row, ws_kc);
        for (int pr = 0; pr < NPR; ++pr) {
          dst = acquire(fb);
          if (dst == ~0u) { ok = false; break; }
          if (dst) tma_load_5d(dst, bmap, fb, 0, b_row, 2 * pr, b_head, it.b);
        }
      }
      const int n = issued < NS ? issued : NS;
      int s = slot;
      uint32_t lp = lap;
      for (int i = 0; i < n; ++i) {
        if (--s < 0) { s = NS - 1; lp ^= 1u; }
        if (p.inject != 0 && issued - 1 - i == 0) continue;   // the dropped stage was never armed
        wait_drain(smem_u32(&bar_full[s]), lp, tmo, err);
      }
    }
  } else if (warp == TC_MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      int slot = 0;
      uint32_t lap = 0;
      auto take = [&]() -> int {
        const uint32_t fb = smem_u32(&bar_full[slot]);
        if (!mbar_try_wait(fb, lap) && !wait_bounded(fb, lap, &abort_flag, tmo, err)) return -1;
        const int s = slot;
        if (++slot == NS) { slot = 0; lap ^= 1u; }
        return s;
      };
      // dQ: A = dS (rows = queries, K-major over keys).  dV / dK: A = P^T or
      // dS^T, the stored tile read MN-major (M = keys in two 64-key chunks
      // 16 KB apart, +2048 bytes per 16 queries).  B always MN-major.
      const uint32_t idesc = idesc_f16(!fp16, BM, 128, !dq_role, true);
      bool ok = true;
      for (int i = 0; i < T && ok; ++i) {
        const int sa = take();
        if (sa < 0) { ok = false; break; }
        const uint32_t a_u32 = ring_u32 + sa * SLOT_BYTES;
        const uint64_t a_desc = dq_role ? sdesc_sw128(a_u32, 16, 1024) : sdesc_sw128(a_u32, CHUNK_BYTES, 1024);
#pragma unroll
        for (int pr = 0; pr < NPR; ++pr) {
          const int sb = take();
          if (sb < 0) { ok = false; break; }
          const uint64_t bd = sdesc_sw128(ring_u32 + sb * SLOT_BYTES, CHUNK_BYTES, 1024);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t ad = dq_role ? a_desc + (((kk >> 2) * CHUNK_BYTES) >> 4) + 2 * (kk & 3)
                                        : a_desc + 128 * kk;
            umma_ss(tmem + 128 * pr, ad, bd + 128 * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&bar_empty[sb]));
        }
        if (!ok) break;
        umma_commit(smem_u32(&bar_empty[sa]));
      }
      if (ok) umma_commit(smem_u32(&bar_acc));
      const uint32_t drb = smem_u32(&bar_drain);
      umma_commit(drb);
      wait_drain(drb, 0, tmo, err);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    const int r = warp * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int my_row = it.row0 + r;
    bool ok = true;
    if (T > 0) {
      const bool w = wait_bounded(smem_u32(&bar_acc), 0, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (ok) tc_fence_after();
    }
    if (ok) {
      uint8_t* dst = nullptr;
      if (dq_role) {
        if (my_row < it.q_len)
          dst = static_cast<uint8_t*>(p.dq) + bwd_row_offset(p, it, p.dq_str, it.q_row0, my_row, it.hq) * 2;
      } else if (my_row < it.kv_len) {
        const bool dv_role = role == BWD_ROLE_DV;
        dst = static_cast<uint8_t*>(dv_role ? p.dv : p.dk) +
              bwd_row_offset(p, it, dv_role ? p.dv_str : p.dk_str, it.kv_row0, my_row, it.hkv) * 2;
      }
      bwd_store_row(lane_base, p.D, 1.f, dst, fp16, T > 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == TC_MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int NCH>
static ffpa_status launch_tiles_t(const BwdParams& P, int score_items, int contract_items, size_t smem_s,
                                  size_t smem_c, cudaStream_t stream) {
  if (score_items > 0) {
    auto ks = P.mask != nullptr ? ffpa_bwd_scores_kernel<NCH, true> : ffpa_bwd_scores_kernel<NCH, false>;
    const ffpa_status st = set_smem_attr_once(reinterpret_cast<const void*>(ks), P.device, static_cast<int>(smem_s));
    if (st != FFPA_OK) return st;
    ks<<<score_items, TS_THREADS, smem_s, stream>>>(P);
    if (cudaGetLastError() != cudaSuccess) return FFPA_ERR_CUDA;
  }
  if (contract_items > 0) {
    auto kc = ffpa_bwd_contract_kernel<NCH>;
    const ffpa_status st = set_smem_attr_once(reinterpret_cast<const void*>(kc), P.device, static_cast<int>(smem_c));
    if (st != FFPA_OK) return st;
    kc<<<contract_items, TC_THREADS, smem_c, stream>>>(P);
    if (cudaGetLastError() != cudaSuccess) return FFPA_ERR_CUDA;
  }
  return FFPA_OK;
}

ffpa_status launch_bwd_tiles(const BwdParams& P, int score_items, int contract_items, size_t smem_scores,
                             size_t smem_contract, cudaStream_t stream) {
  if (launch_bwd_delta(P, stream) != FFPA_OK) return FFPA_ERR_CUDA;
  switch (P.nchunks) {
    case 4: return launch_tiles_t<4>(P, score_items, contract_items, smem_scores, smem_contract, stream);
    case 6: return launch_tiles_t<6>(P, score_items, contract_items, smem_scores, smem_contract, stream);
    case 8: return launch_tiles_t<8>(P, score_items, contract_items, smem_scores, smem_contract, stream);
    default: return FFPA_ERR_UNSUPPORTED;
  }
}

}  // namespace ffpa
