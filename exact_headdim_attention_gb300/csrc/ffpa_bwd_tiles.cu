// Stored-tile backward: P and dS formed once per (query tile, key tile), then dQ, dV and dK
// as plain contractions over the stored tiles.
#include "ffpa_bwd_common.cuh"

namespace ffpa {

using namespace bwd;

// =====================================================================
// Backward by stored score tiles (dense and varlen layouts, D = 128, 256, 384, 512).
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
// Contraction kernel: CTA pairs (cta_group::2), each CTA one output tile of
// 128 rows x D columns (the whole row in TMEM, up to 512 fp32 columns):
//   dQ tiles  two adjacent query tiles of one query head, summed over the
//             visible key tiles: A = stored dS tile (K-major), B = K;
//   dV tiles  two adjacent key tiles of one KV head, summed over the group's
//             query heads and the query tiles that see them: A = stored P
//             tile read as P^T (the same bytes, MN-major), B = dO;
//   dK tiles  as dV with dS and Q.
//   B is read MN-major, each CTA loading its 128 of every 256 output columns.
//   Warps 0-3 epilogue (TMEM -> 16-bit rows), 4 TMA producer, 5 MMA issuer
//   (leader) or relay (peer).  The three kinds of items are interleaved in
//   one launch (each kind's own order puts its longest items first under
//   causal masking).
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

// Block of the stored P (or dS) for (batch or sequence b, query head h, query
// tile qt, key tile kt) of a problem with q_len queries and kv_len keys.
template <bool VARLEN>
__device__ __forceinline__ long long stored_block(const BwdParams& p, int b, int h, int q_len, int kv_len, int qt,
                                                  int kt) {
  if constexpr (VARLEN) {
    const long long per_head = bwd_stored_before((q_len + BM - 1) / BM, q_len, kv_len, p.causal);
    return p.ws_base[b] + (long long)h * per_head + bwd_stored_before(qt, q_len, kv_len, p.causal) + kt;
  }
  return (long long)(b * p.Hq + h) * p.ws_head + bwd_stored_before(qt, p.Nq, p.Nkv, p.causal) + kt;
}

// A block index past the caller's workspace: recorded as an invalid
// argument in the call's status word (a varlen workspace smaller than the
// sequences need); the block is then neither written nor read.  The dense
// workspace is sized by the library itself: no check.
template <bool VARLEN>
__device__ __forceinline__ bool block_in_workspace(const BwdParams& p, long long blk) {
  if constexpr (!VARLEN) {
    return true;
  } else {
    if (blk < p.ws_blocks) return true;
    atomicExch(p.err, (int)FFPA_ERR_INVALID);
    return false;
  }
}

// Varlen: the first stored block of every sequence (an exclusive scan of
// Hq x blocks per head over the sequences), and the total at index nseq.
__global__ void __launch_bounds__(1024) ffpa_bwd_bases_kernel(const __grid_constant__ BwdParams p) {
  __shared__ long long part[1024];
  const int n = p.B, t = threadIdx.x;
  const int per = (n + 1023) / 1024;
  const int s0 = min(n, t * per), s1 = min(n, s0 + per);
  auto blocks = [&](int s) -> long long {
    const int lq = p.cu_q[s + 1] - p.cu_q[s], lk = p.cu_k[s + 1] - p.cu_k[s];
    return (long long)p.Hq * bwd_stored_before((lq + BM - 1) / BM, lq, lk, p.causal);
  };
  long long sum = 0;
  for (int s = s0; s < s1; ++s) sum += blocks(s);
  part[t] = sum;
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {
    const long long v = t >= d ? part[t - d] : 0;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  long long base = part[t] - sum;
  long long* out = const_cast<long long*>(p.ws_base);
  for (int s = s0; s < s1; ++s) {
    out[s] = base;
    base += blocks(s);
  }
  if (t == 1023) out[n] = part[1023];
}

// NCH = D / 64 (2, 4, 6 or 8): every MMA issue loop has a compile-time trip count.
template <int NCH, bool UMASK, bool VARLEN>
__global__ void __launch_bounds__(TS_THREADS, 1) ffpa_bwd_scores_kernel(const __grid_constant__ BwdParams p) {
  constexpr int NPR = NCH / 2;   // 32 KB stages per K (or V) tile
  if (blockIdx.x == 0) {
    // The block of zeros the contraction kernel reads for tiles outside a
    // CTA's range.
    uint4* z = static_cast<uint4*>(p.ws_zero);
    for (int i = threadIdx.x; i < (int)(P_TILE_BYTES / 16); i += TS_THREADS) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
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
          if constexpr (VARLEN)
            tma_load_4d(ring_u32 + slot * SLOT_BYTES, m, fb, 0, it.kv_row0 + row, chunk, it.hkv);
          else
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
      auto qload = [&](const CUtensorMap* m, uint32_t bar) {
        for (int pr = 0; pr < NPR; ++pr) {
          if constexpr (VARLEN)
            tma_load_4d(do_u32 + pr * SLOT_BYTES, m, bar, 0, it.q_row0 + it.row0, 2 * pr, it.hq);
          else
            tma_load_5d(do_u32 + pr * SLOT_BYTES, m, bar, 0, it.row0, 2 * pr, it.hq, it.b);
        }
      };
      qload(&p.tm_q, qb);
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
        qload(&p.tm_do, db);
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
    // This thread's 16-byte units (keys 64 half + 8 q .. +7, q = 0..7) of row
    // r in the stored blocks: every row of a block is written, zeros where
    // the row or key is out of range.  A warp's store covers 32 consecutive
    // rows of one unit: 512 contiguous bytes.
    const long long blk0 = stored_block<VARLEN>(p, it.b, it.hq, it.q_len, it.kv_len, it.row0 / BM, 0);
    const long long uoff = (blk0 << 15) + (long long)(8 * half) * 2048 + r * 16;
    uint8_t* const pbase = static_cast<uint8_t*>(p.ws_p) + uoff;
    uint8_t* const dsbase = static_cast<uint8_t*>(p.ws_ds) + uoff;
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
      // This warp's 64 columns of S in one round trip; once they are in
      // registers the next tile's S may overwrite them.
      float pv[64];
      {
        uint32_t sa[32], sb[32];
        tmem_ld32(lane_base + TS_S_COL + c_lo, sa);
        tmem_ld32(lane_base + TS_S_COL + c_lo + 32, sb);
        tmem_wait_ld();
        reg_fence(sa);
        reg_fence(sb);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_s_free));
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const int col = c_lo + e;
          float arg = fmaf(__uint_as_float(e < 32 ? sa[e] : sb[e - 32]), sl2, -lse_r);
          if (UMASK && col < mcols) arg = add_mask_term(arg, mbase, moff + col * mstep, mkind, fp16);
          float v = ex2_approx(arg);
          if (need_mask) {
            const bool vis = col < kv_cols && (!causal || (long long)col <= lim);
            v = vis ? v : 0.f;
          }
          pv[e] = v;
        }
      }
      const bool in_ws = block_in_workspace<VARLEN>(p, blk0 + j0 + jj);
      if (in_ws) {
        uint8_t* const dst = pbase + ((long long)(j0 + jj) << 15);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float* x = pv + 8 * q;
          *reinterpret_cast<uint4*>(dst + q * 2048) = fp16 ? make_uint4(pack_f16(x[0], x[1]), pack_f16(x[2], x[3]), pack_f16(x[4], x[5]),
                                     pack_f16(x[6], x[7]))
                        : make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                                     pack_bf16(x[6], x[7]));
        }
      }
      w = wait_bounded(smem_u32(&bar_dp_full), jj & 1, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      tc_fence_after();
      uint8_t* const dst = dsbase + ((long long)(j0 + jj) << 15);
      // dP likewise: one round trip, then the next tile's dP may overwrite it.
      uint32_t da[32], db[32];
      tmem_ld32(lane_base + TS_DP_COL + c_lo, da);
      tmem_ld32(lane_base + TS_DP_COL + c_lo + 32, db);
      tmem_wait_ld();
      reg_fence(da);
      reg_fence(db);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_dp_free));
#pragma unroll
      for (int g = 0; g < 4 && in_ws; ++g) {
        float x[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = 16 * g + e;
          x[e] = pv[c] * sc * (__uint_as_float(c < 32 ? da[c] : db[c - 32]) - delta_r);
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float* y = x + 8 * q;
          *reinterpret_cast<uint4*>(dst + (2 * g + q) * 2048) = fp16 ? make_uint4(pack_f16(y[0], y[1]), pack_f16(y[2], y[3]),
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

// Role and rank of contraction pair item L: dQ, dV and dK items interleaved
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

// One output tile pair of the contraction kernel: two adjacent query tiles
// (dQ) or key tiles (dV, dK) of one head, rank r of the pair owning tile
// tile0 + r.  Both CTAs walk the same contraction steps (the union of their
// ranges; a step outside a CTA's own range contributes a zero tile).
struct PairItem {
  int role, b, hq, hkv;
  int q_len, kv_len;       // this problem's (sequence's) lengths
  int q_row0, kv_row0;     // varlen: first packed row of the sequence (dense: 0)
  int n_qt, n_kt;          // its query and key tiles
  int tile0, my_tile;
  int n_iter;       // contraction steps
  int qt_first;     // dV / dK: first query tile of the range
  int nq;           // dV / dK: query tiles per head in the range
};

// False for a pair past the end of its sequence (varlen; same answer in
// both CTAs).
template <bool VARLEN>
__device__ __forceinline__ bool decode_pair_item(const BwdParams& p, int L, uint32_t rank, PairItem& it) {
  int r;
  contract_role(p, L, it.role, r);
  const bool dq = it.role == BWD_ROLE_DQ;
  const int heads = p.B * (dq ? p.Hq : p.Hkv);
  const int npairs = dq ? (p.n_qt + 1) >> 1 : (p.n_kt + 1) >> 1;
  int pi, bh;
  if (p.causal) {            // dQ: longest query tiles first; dV / dK: key tile 0 (seen by all) first
    bh = r % heads;
    pi = dq ? npairs - 1 - r / heads : r / heads;
  } else {
    pi = r % npairs;
    bh = r / npairs;
  }
  if (dq) {
    it.hq = bh % p.Hq;
    it.b = bh / p.Hq;
    it.hkv = it.hq / p.group;
  } else {
    it.hkv = bh % p.Hkv;
    it.b = bh / p.Hkv;
    it.hq = it.hkv * p.group;
  }
  if constexpr (VARLEN) {
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
  it.n_qt = (it.q_len + BM - 1) / BM;
  it.n_kt = (it.kv_len + BN - 1) / BN;
  it.tile0 = 2 * pi;
  it.my_tile = it.tile0 + (int)rank;
  if (dq) {
    if (it.tile0 >= it.n_qt) return false;
    it.n_iter = bwd_stored_tiles(min(it.tile0 + 1, it.n_qt - 1), it.q_len, it.kv_len, p.causal);
    it.qt_first = 0;
    it.nq = 0;
  } else {
    if (it.tile0 >= it.n_kt) return false;
    // Query row i sees key k when k <= i + (Nkv - Nq): the first query tile
    // with a row that sees the pair's first key.
    const int first_row = p.causal ? max(0, it.tile0 * BN - (it.kv_len - it.q_len)) : 0;
    it.qt_first = first_row / BM;
    it.nq = max(0, it.n_qt - it.qt_first);
    it.n_iter = p.group * it.nq;
  }
  return true;
}

// Contraction kernel on CTA pairs (cta_group::2): one M = 256 MMA per
// 16-row step covers both CTAs' output tiles, and each CTA loads only half
// of the shared B operand (its 128 of every 256 output columns), so per SM
// the bytes per multiply-add are about 60 % of a single CTA's.  The peer's
// warp 5 relays its "stage landed" events to the leader's full barriers; the
// leader's commits arrive in both CTAs.
template <int NCH, bool VARLEN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TC_THREADS, 1)
    ffpa_bwd_contract_kernel(const __grid_constant__ BwdParams p) {
  constexpr int NG = (NCH + 3) / 4;   // 256-column groups (the last may have 128)
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  PairItem it;
  if (!decode_pair_item<VARLEN>(p, blockIdx.x >> 1, rank, it)) return;   // same answer in both CTAs
  const bool dq_role = it.role == BWD_ROLE_DQ;
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
    // Leader full barriers also count the peer's relayed arrival.
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bar_full[i]), leader ? 2 : 1);
      mbar_init(smem_u32(&bar_empty[i]), 1);
    }
    mbar_init(smem_u32(&bar_acc), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == TC_MMA_WARP) {
    tmem_alloc_pair(smem_u32(&tmem_base_sh), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();      // the peer's barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == TC_PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    // Per contraction step: this CTA's stored tile (A), then its half of
    // each 256-column group of the B operand.
    if (lane == 0 && T > 0) {
      const uint8_t* abase = static_cast<const uint8_t*>(it.role == BWD_ROLE_DV ? p.ws_p : p.ws_ds);
      const CUtensorMap* bmap = dq_role ? &p.tm_k : it.role == BWD_ROLE_DV ? &p.tm_do : &p.tm_q;
      prefetch_tmap(bmap);
      int slot = 0, issued = 0;
      uint32_t lap = 0;
      bool drop = leader && p.inject != 0;   // test hook, as in the scores kernel
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
      // Step i's stored block (the zero block outside this CTA's range) and
      // the B operand's rows and head.
      auto step = [&](int i, int& b_row, int& head) -> const void* {
        int qt, kt;
        if (dq_role) {
          qt = it.my_tile;
          kt = i;
          head = it.hq;
          b_row = i * BN;
        } else {
          head = it.hq + i / it.nq;
          qt = it.qt_first + i % it.nq;
          kt = it.my_tile;
          b_row = qt * BM;
        }
        const bool real = qt < it.n_qt && kt < bwd_stored_tiles(qt, it.q_len, it.kv_len, p.causal);
        if (!real) return p.ws_zero;
        const long long blk = stored_block<VARLEN>(p, it.b, head, it.q_len, it.kv_len, qt, kt);
        return block_in_workspace<VARLEN>(p, blk) ? static_cast<const void*>(abase + (blk << 15)) : p.ws_zero;
      };
      // The stored blocks come from DRAM: each is requested into L2 this many
      // steps before its copy into the ring.  Measured on GB300 (TFLOPS of the
      // whole backward, B1 N4096; same-box A/B, two rounds): D = 512 1047 with
      // 6 steps, 1052 with 2 (3: 1052, 4: 1051, 5: 1050, 8: 1046), causal GQA
      // Hq16 Hkv4 949 -> 980; D = 384 893 -> 895; D = 128 416 -> 433 (3: 431,
      // 6: 423); D = 256 831 without, 807 with 2 steps, 809 with 1: none there.
      constexpr int PF = NCH == 4 ? 0 : 2;
      for (int i = 0; i < PF && i < T; ++i) {
        int br, hd;
        prefetch_l2_bulk(step(i, br, hd), P_TILE_BYTES);
      }
      bool ok = true;
      for (int i = 0; i < T && ok; ++i) {
        int b_row, head;
        const void* src = step(i, b_row, head);
        if (PF > 0 && i + PF < T) {
          int br, hd;
          prefetch_l2_bulk(step(i + PF, br, hd), P_TILE_BYTES);
        }
        uint32_t fb = 0;
        uint32_t dst = acquire(fb);
        if (dst == ~0u) { ok = false; break; }
        if (dst) bulk_load_g2s(dst, src, P_TILE_BYTES, fb);
        const int b_head = dq_role ? it.hkv : head;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          dst = acquire(fb);
          if (dst == ~0u) { ok = false; break; }
          // 256-column group: chunks 4g + 2 rank, +1; a 128-column tail: chunk 4g + rank.
          const int c0 = (4 * g + 4 <= NCH) ? 4 * g + 2 * (int)rank : 4 * g + (int)rank;
          if (dst) {
            if constexpr (VARLEN)
              tma_load_4d(dst, bmap, fb, 0, (dq_role ? it.kv_row0 : it.q_row0) + b_row, c0, b_head);
            else
              tma_load_5d(dst, bmap, fb, 0, b_row, c0, b_head, it.b);
          }
        }
      }
      const int n = issued < NS ? issued : NS;
      int s = slot;
      uint32_t lp = lap;
      for (int i = 0; i < n; ++i) {
        if (--s < 0) { s = NS - 1; lp ^= 1u; }
        if (leader && p.inject != 0 && issued - 1 - i == 0) continue;   // the dropped stage was never armed
        wait_drain(smem_u32(&bar_full[s]), lp, tmo, err);
      }
    }
  } else if (warp == TC_MMA_WARP && !leader) {
    // ------------------------------------------------------------ relay (peer)
    if (lane == 0 && T > 0) {
      int slot = 0;
      uint32_t lap = 0;
      for (int i = 0; i < T * (1 + NG); ++i) {
        const uint32_t fb = smem_u32(&bar_full[slot]);
        if (!(mbar_try_wait(fb, lap) || wait_bounded(fb, lap, &abort_flag, tmo, err))) break;
        mbar_arrive_cluster(mapa_shared(fb, 0));
        if (++slot == NS) { slot = 0; lap ^= 1u; }
      }
    }
  } else if (warp == TC_MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer (leader)
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
      // The stored block without swizzle: core matrices of 8 rows x 8 keys
      // (128 bytes), 2048 bytes apart along the keys and 128 along the rows.
      // Without swizzle the descriptor's stride fields are: along K (leading
      // byte offset) and along M (stride byte offset), for either major.
      // dQ: A = dS K-major (M = queries, K = keys; +4096 bytes per 16 keys).
      // dV / dK: A = P^T or dS^T, the same bytes MN-major (M = keys, K =
      // queries; +256 bytes per 16 queries).  B always MN-major.
      bool ok = true;
      for (int i = 0; i < T && ok; ++i) {
        const int sa = take();
        if (sa < 0) { ok = false; break; }
        const uint32_t a_u32 = ring_u32 + sa * SLOT_BYTES;
        const uint64_t a_desc = dq_role ? sdesc_noswz(a_u32, 2048, 128) : sdesc_noswz(a_u32, 128, 2048);
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const int sb = take();
          if (sb < 0) { ok = false; break; }
          const int ng = (4 * g + 4 <= NCH) ? 256 : 128;
          const uint32_t idesc = idesc_f16(!fp16, 2 * BM, ng, !dq_role, true);
          const uint64_t bd = sdesc_sw128(ring_u32 + sb * SLOT_BYTES, CHUNK_BYTES, 1024);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t ad = dq_role ? a_desc + 256 * kk : a_desc + 16 * kk;
            umma_ss_pair(tmem + 256 * g, ad, bd + 128 * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit_pair(smem_u32(&bar_empty[sb]));
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&bar_empty[sa]));
      }
      if (ok) umma_commit_pair(smem_u32(&bar_acc));
      const uint32_t drb = smem_u32(&bar_drain);
      umma_commit_pair(drb);
      wait_drain(drb, 0, tmo, err);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    // Warp w's 32 rows go through ring slot w (idle once the accumulator is
    // complete).  Dense: tensor stores of 32-row boxes.  Varlen (a box could
    // reach into the next sequence's rows): thread t writes its row's 16-bit
    // values there (16-byte unit x of row t at unit x ^ (t & 7),
    // conflict-free), then the warp stores the rows one by one, each warp
    // store covering 512 contiguous bytes.
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bool ok = true;
    if (T > 0) {
      const bool w = wait_bounded(smem_u32(&bar_acc), 0, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (ok) tc_fence_after();
    }
    if (ok && !VARLEN) {
      // Dense: per 64-column chunk a 32-row x 128-byte box of the slot
      // (4 KB, 128-byte swizzle: unit u of row t at u ^ (t & 7)), written out
      // by tensor stores; the rows past the tensor's end are not written.
      const uint32_t stage = ring_u32 + warp * SLOT_BYTES;
      const uint32_t sw = (uint32_t)(lane & 7);
#pragma unroll 1
      for (int c0 = 0; c0 < NCH * DK; c0 += 64) {
        uint32_t va[32], vb[32];
        if (T > 0) {
          tmem_ld32(lane_base + c0, va);
          tmem_ld32(lane_base + c0 + 32, vb);
          tmem_wait_ld();
          reg_fence(va);
          reg_fence(vb);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) va[c] = vb[c] = 0u;
        }
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int e = 2 * c;
          const float a0 = __uint_as_float(e < 32 ? va[e] : vb[e - 32]);
          const float a1 = __uint_as_float(e + 1 < 32 ? va[e + 1] : vb[e + 1 - 32]);
          pk[c] = fp16 ? pack_f16(a0, a1) : pack_bf16(a0, a1);
        }
        const uint32_t box = stage + (uint32_t)(c0 / 64) * 4096u + lane * 128u;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          st_shared_v4(box + (((uint32_t)q ^ sw) << 4), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int row0 = it.my_tile * BM + warp * 32;
      if (lane == 0 && row0 < (dq_role ? it.q_len : it.kv_len)) {
        const CUtensorMap* om = dq_role ? &p.tm_dq : it.role == BWD_ROLE_DV ? &p.tm_dv : &p.tm_dk;
        const int head = dq_role ? it.hq : it.hkv;
#pragma unroll 1
        for (int c = 0; c < NCH; ++c) tma_store_5d(om, stage + (uint32_t)c * 4096u, 0, row0, c, head, it.b);
        bulk_commit_group();
        bulk_wait_read_all();   // the slot is read before the CTA may exit
      }
      __syncwarp();
    } else if (ok) {
      constexpr int ROWB = NCH * DK * 2;   // bytes of one output row
      constexpr int UNITS = ROWB / 16;
      const uint32_t stage = ring_u32 + warp * SLOT_BYTES;
      const uint32_t sw = (uint32_t)(lane & 7);
#pragma unroll 1
      for (int c0 = 0; c0 < NCH * DK; c0 += 64) {   // 64 columns per TMEM round trip
        uint32_t va[32], vb[32];
        if (T > 0) {
          tmem_ld32(lane_base + c0, va);
          tmem_ld32(lane_base + c0 + 32, vb);
          tmem_wait_ld();
          reg_fence(va);
          reg_fence(vb);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) va[c] = vb[c] = 0u;
        }
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int e = 2 * c;
          const float a0 = __uint_as_float(e < 32 ? va[e] : vb[e - 32]);
          const float a1 = __uint_as_float(e + 1 < 32 ? va[e + 1] : vb[e + 1 - 32]);
          pk[c] = fp16 ? pack_f16(a0, a1) : pack_bf16(a0, a1);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t x = (uint32_t)(c0 / 8 + q);
          st_shared_v4(stage + lane * ROWB + ((x ^ sw) << 4), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      __syncwarp();
      BwdItem bi;
      bi.b = it.b;
      bi.q_row0 = it.q_row0;
      bi.kv_row0 = it.kv_row0;
      const bool dv_role = it.role == BWD_ROLE_DV;
      uint8_t* const obase = static_cast<uint8_t*>(dq_role ? p.dq : dv_role ? p.dv : p.dk);
      const int64_t* ostr = dq_role ? p.dq_str : dv_role ? p.dv_str : p.dk_str;
      const int head = dq_role ? it.hq : it.hkv;
      const int rows = dq_role ? it.q_len : it.kv_len;
      const int seq_row0 = dq_role ? it.q_row0 : it.kv_row0;
      const int row0 = it.my_tile * BM + warp * 32;
#pragma unroll 1
      for (int rr = 0; rr < 32 && row0 + rr < rows; ++rr) {
        uint8_t* const orow = obase + bwd_row_offset(p, bi, ostr, seq_row0, row0 + rr, head) * 2;
        const uint32_t srow = stage + rr * ROWB;
        const uint32_t rsw = (uint32_t)(rr & 7);
#pragma unroll
        for (int x = lane; x < UNITS; x += 32) {
          const uint4 val = ld_shared_v4(srow + (((uint32_t)x ^ rsw) << 4));
          *reinterpret_cast<uint4*>(orow + x * 16) = val;
        }
      }
    }
  }

  // The leader's last commits also arrive in the peer: wait for them before
  // the pair may exit, then free TMEM in both CTAs together.
  if (!leader && threadIdx.x == 0 && T > 0) wait_drain(smem_u32(&bar_drain), 0, tmo, err);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == TC_MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

template <int NCH>
static ffpa_status launch_tiles_t(const BwdParams& P, int score_items, int contract_items, size_t smem_s,
                                  size_t smem_c, cudaStream_t stream) {
  if (score_items > 0) {
    auto ks = P.varlen           ? ffpa_bwd_scores_kernel<NCH, false, true>
              : P.mask != nullptr ? ffpa_bwd_scores_kernel<NCH, true, false>
                                  : ffpa_bwd_scores_kernel<NCH, false, false>;
    const ffpa_status st = set_smem_attr_once(reinterpret_cast<const void*>(ks), P.device, static_cast<int>(smem_s));
    if (st != FFPA_OK) return st;
    ks<<<score_items, TS_THREADS, smem_s, stream>>>(P);
    if (cudaGetLastError() != cudaSuccess) return FFPA_ERR_CUDA;
  }
  if (contract_items > 0) {
    auto kc = P.varlen ? ffpa_bwd_contract_kernel<NCH, true> : ffpa_bwd_contract_kernel<NCH, false>;
    const ffpa_status st = set_smem_attr_once(reinterpret_cast<const void*>(kc), P.device, static_cast<int>(smem_c));
    if (st != FFPA_OK) return st;
    kc<<<2 * contract_items, TC_THREADS, smem_c, stream>>>(P);
    if (cudaGetLastError() != cudaSuccess) return FFPA_ERR_CUDA;
  }
  return FFPA_OK;
}

ffpa_status launch_bwd_tiles_bases(const BwdParams& P, cudaStream_t stream) {
  ffpa_bwd_bases_kernel<<<1, 1024, 0, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}

ffpa_status launch_bwd_tiles(const BwdParams& P, int score_items, int contract_items, size_t smem_scores,
                             size_t smem_contract, cudaStream_t stream) {
  if (launch_bwd_delta(P, stream) != FFPA_OK) return FFPA_ERR_CUDA;
  if (P.varlen && launch_bwd_tiles_bases(P, stream) != FFPA_OK) return FFPA_ERR_CUDA;
  switch (P.nchunks) {
    case 2: return launch_tiles_t<2>(P, score_items, contract_items, smem_scores, smem_contract, stream);
    case 4: return launch_tiles_t<4>(P, score_items, contract_items, smem_scores, smem_contract, stream);
    case 6: return launch_tiles_t<6>(P, score_items, contract_items, smem_scores, smem_contract, stream);
    case 8: return launch_tiles_t<8>(P, score_items, contract_items, smem_scores, smem_contract, stream);
    default: return FFPA_ERR_UNSUPPORTED;
  }
}

}  // namespace ffpa
