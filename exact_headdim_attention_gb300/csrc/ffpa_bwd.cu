// Backward of exact attention: dQ, dK and dV from Q, K, V, O, dO and the
// forward's natural-log LSE (FFPA API reference, "ffpa_attn.ffpa_attn_func":
// backward through FFPAAttnFunc; the Triton backend's `split_launch` option
// launches the dK/dV and the dQ parts separately, which is the split used
// here).
//
// With P = exp(scale * Q K^T - LSE) (the forward's softmax, recomputed),
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - delta),  delta = rowsum(dO * O),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Four launches on the caller's stream:
//   delta   one warp per query row, 16-byte loads of O and dO.
//   dQ      one CTA per (batch, query head, 128-row query tile, <= 256 dQ
//           columns); loops over the visible key tiles.
//   dV, dK  one CTA per (batch, key/value head, 128-key tile, <= 256
//           columns); loops over every query head of the group and the
//           query tiles that see the key tile, so grouped heads add up in
//           TMEM and no atomics are needed.
// The three tensor-core kernels share one body (ROLE selects).  Per
// iteration the MMA thread computes the full-D contractions into TMEM
// (S = A1 B1^T, and for dQ and dK also dP = A2 B2^T: for dQ A = Q, dO and
// B = K, V; for dV and dK A = K, V and B = Q, dO, i.e. S^T and dP^T), the
// elementwise warps turn them into a 16-bit tile in shared memory (128-byte
// swizzle, K-major): dS for dQ, P^T for dV, dS^T for dK; and the MMA thread
// accumulates the output slice from it (dQ += dS K; dV += P^T dO;
// dK += dS^T Q) with the B operand read MN-major from 64-column boxes of the
// same tensors.  For D > 128, dV and dK are separate kernels so that each
// holds one tile and a deeper ring, and dV needs neither dP nor delta; for
// D <= 128 one dK/dV kernel forms both from a single S, dP (both tiles,
// dV and dK in TMEM columns [0, 128) and [128, 256)).  TMEM holds the output
// accumulators in columns [0, 256) and S, dP in [256, 384), [384, 512).
// The contractions of iteration i+1 are issued before the slice MMAs of
// iteration i, so the tensor core works while the elementwise warps run.
// When D exceeds the output columns of one CTA, the CTAs of the other
// column slices recompute S and dP.
#include "ffpa_bwd_common.cuh"

namespace ffpa {

using namespace bwd;

__global__ void __launch_bounds__(256) ffpa_bwd_delta_kernel(const __grid_constant__ BwdParams p) {
  // Dense: row = (b Hq + h) Nq + i.  Varlen: row = h Tq + t (the [Hq, Tq]
  // layout of LSE and delta).
  const long long rows = p.varlen ? (long long)p.Hq * p.Tq : (long long)p.B * p.Hq * p.Nq;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  long long oo, od;
  if (p.varlen) {
    const long long t = row % p.Tq, h = row / p.Tq;
    oo = t * p.o_str[0] + h * p.o_str[1];
    od = t * p.do_str[0] + h * p.do_str[1];
  } else {
    const long long i = row % p.Nq;
    const long long bh = row / p.Nq;
    const long long h = bh % p.Hq, b = bh / p.Hq;
    oo = b * p.o_str[0] + h * p.o_str[1] + i * p.o_str[2];
    od = b * p.do_str[0] + h * p.do_str[1] + i * p.do_str[2];
  }
  const uint16_t* orow = static_cast<const uint16_t*>(p.o) + oo;
  const uint16_t* drow = static_cast<const uint16_t*>(p.dout) + od;
  const bool fp16 = p.fp16 != 0;
  float acc = 0.f;
  for (int d0 = lane * 8; d0 < p.D; d0 += 256)
    acc += dot8(__ldg(reinterpret_cast<const uint4*>(orow + d0)),
                __ldg(reinterpret_cast<const uint4*>(drow + d0)), fp16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) p.delta[row] = acc;
}

// ROLE: BWD_ROLE_DQ / DV / DK.  UMASK: launched with a caller's mask
// (mask-loading code present).
template <int ROLE, bool UMASK>
__global__ void __launch_bounds__(BWD_THREADS, 1) ffpa_bwd_kernel(const __grid_constant__ BwdParams p) {
  constexpr bool DQ = ROLE == BWD_ROLE_DQ;         // rows are queries (else keys)
  constexpr bool NEED_DP = ROLE != BWD_ROLE_DV;    // dS needs dP and delta; dV needs only P
  constexpr bool TWO = ROLE == BWD_ROLE_DKDV;      // two tiles (P^T, dS^T) and two outputs
  BwdItem it;
  if (!bwd_decode<DQ>(p, blockIdx.x, it)) return;   // uniform across the CTA

  const int npairs = p.npairs, nchunks = p.nchunks;
  const bool fp16 = p.fp16 != 0, causal = p.causal != 0;
  const int NS = TWO ? p.nslot_two : p.nslot;
  const int T = it.n_iter;
  const unsigned long long tmo = p.timeout_ns;
  int* const err = p.err;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // [tile: dS (dQ), P^T (dV, dK/dV) or dS^T (dK)] [dS^T (dK/dV)] [ring: NS x 32 KB]
  const uint32_t t1_u32 = smem_u32(smem);
  const uint32_t t2_u32 = t1_u32 + P_TILE_BYTES;
  const uint32_t ring_u32 = t1_u32 + (TWO ? 2u : 1u) * P_TILE_BYTES;
  __shared__ __align__(8) uint64_t bar_full[BWD_NSLOT_MAX], bar_empty[BWD_NSLOT_MAX];
  __shared__ __align__(8) uint64_t bar_sd_full, bar_s_free, bar_p_full, bar_pd_done, bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  // dV, dK: per-warp copies of the current query tile's log2-domain LSE and
  // delta (each warp loads and reads its own, so no cross-warp barrier).
  __shared__ __align__(16) float stat_sh[DQ ? 4 : 4 * 2 * BM];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bar_full[i]), 1);
      mbar_init(smem_u32(&bar_empty[i]), 1);
    }
    mbar_init(smem_u32(&bar_sd_full), 1);
    mbar_init(smem_u32(&bar_s_free), 4);
    mbar_init(smem_u32(&bar_p_full), 4);
    mbar_init(smem_u32(&bar_pd_done), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == BWD_MMA_WARP) {
    tmem_alloc(smem_u32(&tmem_base_sh), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  // Streaming-side head and first row of iteration i (key-row roles: query head and
  // query tile; dQ: the key tile).
  auto stream_coords = [&](int i, int& head, int& row) {
    if (DQ) {
      head = it.hkv;
      row = i * BN;
    } else {
      head = it.hq + i / it.nq;
      row = (it.qt_first + i % it.nq) * BM;
    }
  };
  const int nbox = (it.dv + 127) / 128;   // 64..128-column boxes of the output slice

  if (warp == BWD_PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && T > 0) {
      prefetch_tmap(&p.tm_q);
      prefetch_tmap(&p.tm_k);
      prefetch_tmap(&p.tm_v);
      prefetch_tmap(&p.tm_do);
      const uint32_t box_bytes = (uint32_t)p.kchunks * CHUNK_BYTES;
      int slot = 0, issued = 0;
      uint32_t lap = 0;
      // Test hook: the CTA's first ring stage is acquired but never armed or
      // copied, so the MMA thread's wait on it runs out.
      bool drop = p.inject != 0;
      // row: within the item's problem; qside: a query-side tensor (Q, dO).
      auto load = [&](const CUtensorMap* m, int row, int chunk, int head, bool qside) -> bool {
        const uint32_t eb = smem_u32(&bar_empty[slot]);
        if (!mbar_try_wait(eb, lap ^ 1u) && !wait_bounded(eb, lap ^ 1u, &abort_flag, tmo, err)) return false;
        const uint32_t fb = smem_u32(&bar_full[slot]);
        if (drop) {
          drop = false;
        } else {
          mbar_arrive_expect_tx(fb, box_bytes);
          if (p.varlen)
            tma_load_4d(ring_u32 + slot * SLOT_BYTES, m, fb, 0, (qside ? it.q_row0 : it.kv_row0) + row, chunk,
                        head);
          else
            tma_load_5d(ring_u32 + slot * SLOT_BYTES, m, fb, 0, row, chunk, head, it.b);
        }
        ++issued;
        if (++slot == NS) { slot = 0; lap ^= 1u; }
        return true;
      };
      const CUtensorMap* a1 = DQ ? &p.tm_q : &p.tm_k;
      const CUtensorMap* b1 = DQ ? &p.tm_k : &p.tm_q;
      const CUtensorMap* a2 = DQ ? &p.tm_do : &p.tm_v;
      const CUtensorMap* b2 = DQ ? &p.tm_v : &p.tm_do;
      const int ha = DQ ? it.hq : it.hkv;
      auto contraction_loads = [&](int i) -> bool {
        int hs, rs;
        stream_coords(i, hs, rs);
        // dQ: A = Q, dO (query side), B = K, V; the key-row roles the other way round.
        for (int pr = 0; pr < npairs; ++pr)
          if (!load(a1, it.row0, 2 * pr, ha, DQ) || !load(b1, rs, 2 * pr, hs, !DQ)) return false;
        if (NEED_DP)
          for (int pr = 0; pr < npairs; ++pr)
            if (!load(a2, it.row0, 2 * pr, ha, DQ) || !load(b2, rs, 2 * pr, hs, !DQ)) return false;
        return true;
      };
      auto slice_loads = [&](int i) -> bool {
        int hs, rs;
        stream_coords(i, hs, rs);
        // The B operand of the slice product: K (dQ), dO (dV) or Q (dK); the
        // dK/dV role takes dO then Q.
        const int c0 = it.col_lo / DK;
        if (TWO) return load(&p.tm_do, rs, c0, hs, true) && load(&p.tm_q, rs, c0, hs, true);
        const CUtensorMap* m = DQ ? &p.tm_k : ROLE == BWD_ROLE_DV ? &p.tm_do : &p.tm_q;
        for (int bx = 0; bx < nbox; ++bx)
          if (!load(m, rs, c0 + 2 * bx, hs, !DQ)) return false;
        return true;
      };
      // Same order as the MMA thread consumes: contractions of iteration 0,
      // then per iteration i the contractions of i+1 and the slices of i.
      bool ok = contraction_loads(0);
      for (int i = 0; i < T && ok; ++i) {
        if (i + 1 < T) ok = contraction_loads(i + 1);
        if (ok) ok = slice_loads(i);
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
  } else if (warp == BWD_MMA_WARP) {
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
      auto release = [&](int s) { umma_commit(smem_u32(&bar_empty[s])); };
      auto wait_on = [&](uint32_t bar, uint32_t par) -> bool {
        if (!mbar_try_wait(bar, par) && !wait_bounded(bar, par, &abort_flag, tmo, err)) return false;
        tc_fence_after();
        return true;
      };
      const uint32_t idesc_s = idesc_f16(!fp16, BM, BN, false, false);
      // Both operands K-major: +32 bytes per 16 D-elements, +16 KB per chunk.
      const uint64_t ring_k = sdesc_sw128(ring_u32, 16, 1024);
      // MN-major B (rows = contraction index): 64-column chunks 16 KB apart,
      // +2048 bytes per 16 rows.
      const uint64_t ring_mn = sdesc_sw128(ring_u32, BM * 128, 1024);
      const uint64_t t1_desc = sdesc_sw128(t1_u32, 16, 1024);
      const uint64_t t2_desc = sdesc_sw128(t2_u32, 16, 1024);
      auto contract = [&](uint32_t dcol) -> bool {
        for (int pr = 0; pr < npairs; ++pr) {
          const int sa = take();
          if (sa < 0) return false;
          const int sb = take();
          if (sb < 0) return false;
          const uint64_t ad = ring_k + ((sa * SLOT_BYTES) >> 4);
          const uint64_t bd = ring_k + ((sb * SLOT_BYTES) >> 4);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_ss(tmem + dcol, ad + 2 * k, bd + 2 * k, idesc_s, (pr > 0 || k > 0) ? 1u : 0u);
          if (2 * pr + 1 < nchunks) {
#pragma unroll
            for (int k = 0; k < 4; ++k) umma_ss(tmem + dcol, ad + 1024 + 2 * k, bd + 1024 + 2 * k, idesc_s, 1u);
          }
          release(sa);
          release(sb);
        }
        return true;
      };
      auto contractions = [&]() -> bool {
        if (!contract(BWD_S_COL) || (NEED_DP && !contract(BWD_DP_COL))) return false;
        umma_commit(smem_u32(&bar_sd_full));
        return true;
      };
      // D[dcol, +n) (+)= A (128 x 128 tile, K-major) * B (box, MN-major).
      auto slice_mma = [&](uint32_t dcol, uint64_t a_desc, int n, bool acc) -> bool {
        const int s = take();
        if (s < 0) return false;
        const uint64_t bd = ring_mn + ((s * SLOT_BYTES) >> 4);
        const uint32_t idesc = idesc_f16(!fp16, BM, n, false, true);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_ss(tmem + dcol, a_desc + (((kk >> 2) * CHUNK_BYTES) >> 4) + 2 * (kk & 3), bd + 128 * kk,
                  idesc, (acc || kk > 0) ? 1u : 0u);
        release(s);
        return true;
      };
      bool ok = contractions();
      for (int i = 0; i < T && ok; ++i) {
        // S and dP of iteration i are in registers of the elementwise warps.
        if (!(ok = wait_on(smem_u32(&bar_s_free), i & 1))) break;
        if (i + 1 < T && !(ok = contractions())) break;
        if (!(ok = wait_on(smem_u32(&bar_p_full), i & 1))) break;
        if (TWO) {
          ok = slice_mma(0, t1_desc, it.dv, i > 0) && slice_mma(128, t2_desc, it.dv, i > 0);
        } else {
          for (int bx = 0; bx < nbox && ok; ++bx)
            ok = slice_mma(128 * bx, t1_desc, min(128, it.dv - 128 * bx), i > 0);
        }
        if (!ok) break;
        umma_commit(smem_u32(&bar_pd_done));
      }
      const uint32_t db = smem_u32(&bar_drain);
      umma_commit(db);
      wait_drain(db, 0, tmo, err);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    // Thread r owns TMEM lane r: query row row0 + r (dQ) or key row row0 + r
    // (key-row roles).  Columns are keys (dQ) or queries (key-row roles).
    const int r = warp * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl2 = p.scale_log2;
    const long long off = (long long)it.kv_len - it.q_len;   // tail alignment of the causal limit
    const int my_row = it.row0 + r;
    float lse_r = INFINITY, delta_r = 0.f;           // dQ: this row's statistics
    if (DQ && my_row < it.q_len) {
      const long long li = bwd_stat_index(p, it, it.hq, my_row);
      const float l = p.lse[li];
      lse_r = l > -INFINITY ? l * LOG2E_F : INFINITY;   // a row with no softmax has P = 0
      delta_r = p.delta[li];
    }
    float* st = stat_sh + (DQ ? 0 : warp * 2 * BM);   // [lse(128) | delta(128)] of this warp
    // Caller's mask: element (query, key) at b m0 + hq m1 + query m2 + key m3.
    const int mkind = p.mask_kind;
    const uint8_t* mbase = static_cast<const uint8_t*>(p.mask);
    const bool mrow_ok = DQ ? my_row < it.q_len : my_row < it.kv_len;
    const uint32_t st_u32 = smem_u32(st);
    bool ok = true;
    for (int i = 0; i < T; ++i) {
      int hs, rs;
      stream_coords(i, hs, rs);
      if (!DQ) {
        // Query-tile statistics: lane l loads queries l, l+32, l+64, l+96.
        __syncwarp();
        const long long lbase = bwd_stat_index(p, it, hs, 0);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int qi = rs + 32 * q4 + lane;
          float l2 = INFINITY, dl = 0.f;
          if (qi < it.q_len) {
            const float l = p.lse[lbase + qi];
            l2 = l > -INFINITY ? l * LOG2E_F : INFINITY;
            dl = p.delta[lbase + qi];
          }
          st[32 * q4 + lane] = l2;
          st[BM + 32 * q4 + lane] = dl;
        }
        __syncwarp();
      }
      bool w = wait_bounded(smem_u32(&bar_sd_full), i & 1, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      tc_fence_after();
      // Causal limits: dQ row i sees key k <= i + off; key row k is
      // seen by query q >= k - off.
      const bool need_mask = DQ ? ((long long)rs + BN > it.kv_len ||
                                   (causal && (long long)rs + BN - 1 > (long long)it.row0 + off))
                                : (causal && (long long)it.row0 + BM - 1 - off > (long long)rs);
      const long long lim = DQ ? (long long)my_row + off - rs      // last visible column
                               : (long long)my_row - off - rs;     // first visible column
      const int kv_cols = it.kv_len - rs;                          // dQ: key columns in range
      // Mask offset of this row at column 0 of the tile, step per column, and
      // the columns in range (dQ: keys; key-row roles: queries of head hs).
      long long moff = 0, mstep = 0;
      int mcols = 0;
      if (UMASK) {
        if (DQ) {
          moff = (long long)it.b * p.m_str[0] + (long long)it.hq * p.m_str[1] +
                 (long long)my_row * p.m_str[2] + (long long)rs * p.m_str[3];
          mstep = p.m_str[3];
          mcols = mrow_ok ? it.kv_len - rs : 0;
        } else {
          moff = (long long)it.b * p.m_str[0] + (long long)hs * p.m_str[1] +
                 (long long)rs * p.m_str[2] + (long long)my_row * p.m_str[3];
          mstep = p.m_str[2];
          mcols = mrow_ok ? it.q_len - rs : 0;
        }
      }
      uint32_t tpk[BN / 2];              // the 16-bit tile row: P (dV, dK/dV) or dS (dQ, dK)
      uint32_t tpk2[TWO ? BN / 2 : 1];   // dK/dV: the dS^T row
#pragma unroll
      for (int g = 0; g < BN / 16; ++g) {
        uint32_t sr[16], dr[16];
        tmem_ld16(lane_base + BWD_S_COL + 16 * g, sr);
        if (NEED_DP) tmem_ld16(lane_base + BWD_DP_COL + 16 * g, dr);
        tmem_wait_ld();
        reg_fence(sr);
        if (NEED_DP) reg_fence(dr);
        float l16[16], d16[16];
        if (DQ) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            l16[e] = lse_r;
            d16[e] = delta_r;
          }
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 a = ld_shared_v4(st_u32 + (uint32_t)(16 * g + 4 * q) * 4u);
            const uint4 b = ld_shared_v4(st_u32 + (uint32_t)(BM + 16 * g + 4 * q) * 4u);
            l16[4 * q] = __uint_as_float(a.x);
            l16[4 * q + 1] = __uint_as_float(a.y);
            l16[4 * q + 2] = __uint_as_float(a.z);
            l16[4 * q + 3] = __uint_as_float(a.w);
            d16[4 * q] = __uint_as_float(b.x);
            d16[4 * q + 1] = __uint_as_float(b.y);
            d16[4 * q + 2] = __uint_as_float(b.z);
            d16[4 * q + 3] = __uint_as_float(b.w);
          }
        }
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
          float pe[2], ds[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int col = 16 * g + c + e;
            float arg = fmaf(__uint_as_float(sr[c + e]), sl2, -l16[c + e]);
            if (UMASK && col < mcols) arg = add_mask_term(arg, mbase, moff + col * mstep, mkind, fp16);
            float v = ex2_approx(arg);
            if (need_mask) {
              const bool vis = DQ ? (col < kv_cols && (!causal || (long long)col <= lim))
                                  : ((long long)col >= lim);
              v = vis ? v : 0.f;
            }
            pe[e] = v;
            ds[e] = NEED_DP ? v * (__uint_as_float(dr[c + e]) - d16[c + e]) : 0.f;
          }
          const bool use_p = TWO || !NEED_DP;
          const float t0 = use_p ? pe[0] : ds[0], t1 = use_p ? pe[1] : ds[1];
          tpk[8 * g + c / 2] = fp16 ? pack_f16(t0, t1) : pack_bf16(t0, t1);
          if (TWO) tpk2[8 * g + c / 2] = fp16 ? pack_f16(ds[0], ds[1]) : pack_bf16(ds[0], ds[1]);
        }
      }
      // S and dP are in registers: the next contractions may overwrite them.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_s_free));
      // The tile is free once the slice MMAs of iteration i-1 are done.
      if (i >= 1) {
        w = wait_bounded(smem_u32(&bar_pd_done), (i - 1) & 1, &abort_flag, tmo, err);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
      }
      bwd_write_tile_row(t1_u32, r, tpk);
      if (TWO) bwd_write_tile_row(t2_u32, r, tpk2);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_p_full));
    }
    // ------------------------------------------------------------ epilogue
    if (ok && T > 0) {
      const bool w = wait_bounded(smem_u32(&bar_pd_done), (T - 1) & 1, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (ok) tc_fence_after();
    }
    if (ok) {
      if (DQ) {
        uint8_t* dst = nullptr;
        if (my_row < it.q_len)
          dst = static_cast<uint8_t*>(p.dq) +
                (bwd_row_offset(p, it, p.dq_str, it.q_row0, my_row, it.hq) + it.col_lo) * 2;
        bwd_store_row(lane_base, it.dv, p.scale, dst, fp16, T > 0);
      } else {
        // dV (no scale) and/or dK (times scale): TMEM column 0, or 0 and 128
        // for the dK/dV role.
        const bool row_in = my_row < it.kv_len;
        if (ROLE == BWD_ROLE_DV || TWO) {
          uint8_t* dst = row_in ? static_cast<uint8_t*>(p.dv) +
                                      (bwd_row_offset(p, it, p.dv_str, it.kv_row0, my_row, it.hkv) +
                                       it.col_lo) * 2
                                : nullptr;
          bwd_store_row(lane_base, it.dv, 1.f, dst, fp16, T > 0);
        }
        if (ROLE == BWD_ROLE_DK || TWO) {
          uint8_t* dst = row_in ? static_cast<uint8_t*>(p.dk) +
                                      (bwd_row_offset(p, it, p.dk_str, it.kv_row0, my_row, it.hkv) +
                                       it.col_lo) * 2
                                : nullptr;
          bwd_store_row(lane_base + (TWO ? 128u : 0u), it.dv, p.scale, dst, fp16, T > 0);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == BWD_MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int ROLE>
static ffpa_status launch_role(const BwdParams& P, int items, size_t smem, cudaStream_t stream) {
  auto kern = P.mask != nullptr ? ffpa_bwd_kernel<ROLE, true> : ffpa_bwd_kernel<ROLE, false>;
  const ffpa_status st =
      set_smem_attr_once(reinterpret_cast<const void*>(kern), P.device, static_cast<int>(smem));
  if (st != FFPA_OK) return st;
  kern<<<items, BWD_THREADS, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}

ffpa_status launch_bwd_delta(const BwdParams& P, cudaStream_t stream) {
  const long long rows = P.varlen ? (long long)P.Hq * P.Tq : (long long)P.B * P.Hq * P.Nq;
  if (rows > 0) {
    ffpa_bwd_delta_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(P);
    if (cudaGetLastError() != cudaSuccess) return FFPA_ERR_CUDA;
  }
  return FFPA_OK;
}

ffpa_status launch_bwd(const BwdParams& P, int dq_items, int kv_items, size_t smem, size_t smem_two,
                       cudaStream_t stream) {
  if (launch_bwd_delta(P, stream) != FFPA_OK) return FFPA_ERR_CUDA;
  if (dq_items > 0 && launch_role<BWD_ROLE_DQ>(P, dq_items, smem, stream) != FFPA_OK) return FFPA_ERR_CUDA;
  if (kv_items > 0) {
    if (P.kv_together) {
      if (launch_role<BWD_ROLE_DKDV>(P, kv_items, smem_two, stream) != FFPA_OK) return FFPA_ERR_CUDA;
    } else {
      if (launch_role<BWD_ROLE_DV>(P, kv_items, smem, stream) != FFPA_OK) return FFPA_ERR_CUDA;
      if (launch_role<BWD_ROLE_DK>(P, kv_items, smem, stream) != FFPA_OK) return FFPA_ERR_CUDA;
    }
  }
  return FFPA_OK;
}


}  // namespace ffpa
