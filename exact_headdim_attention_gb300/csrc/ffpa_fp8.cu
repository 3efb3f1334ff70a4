// FP8 (e4m3) forward: block quantisation of Q, K, V, then attention on the
// tensor cores' kind::f8f6f4 MMA.
#include "ffpa_common.cuh"

namespace ffpa {

// =====================================================================
// FP8 forward (FFPA README, "Backends" / "Latest News": FP8 attention
// kernels that take bf16/fp16 tensors and return the input type, with the
// quantisation scales folded into the computation).  The quantisation is
// this library's reading, since the pages give no formula:
//
//   Q, K and V are quantised per (batch, head, block of 128 rows) to e4m3:
//   amax = max |x| over the block, inv = 448 / amax, s = amax / 448
//   (inv = 0, s = 1 for a zero block); code = e4m3(x * inv), nearest-even,
//   saturated.  A query tile and a key tile are each one block, so
//     S_tile = s_q * s_k * (Q8 K8^T)        (s_q s_k folded into the
//                                            tile's softmax scale)
//   and the V block scale is folded into P: P8 = e4m3(p * c_t) with
//   c_t = 256 s_v(t) / G, G = the largest V block scale of the head, so
//     sum_t P8_t V8_t ~= (256 / G) sum_t p_t v_t,
//   and O = acc * (G / 256) / l, with l the sum of the unrounded p.
//
// The kernel is the single-CTA kernel's structure (one CTA per 128-row
// query tile and output slice of at most 256 columns) with e4m3 operands:
// one 128-byte swizzle row holds 128 elements, so QK^T takes D/128 chunks of
// four K=32 MMAs; P (4 e4m3 per TMEM column) is the A operand of PV from
// TMEM; V is quantised transposed ([B, H, D, N]), so that both operands of
// PV are K-major.  Dense layout only; D a multiple of 128.
// =====================================================================

constexpr int F8_BLOCK = 128;                  // rows per quantisation block = tile
constexpr uint32_t F8_P_COL0 = 384;            // P buffer b at [384 + 32 b, +32)
// The running maximum is raised once a tile's maximum exceeds it by more
// than 2^0.75, so p <= 1.69 and p * c_t <= 431 < 448 (c_t <= 256): P never
// saturates e4m3 (the 16-bit kernels allow 2^8).
constexpr float F8_RESCALE_LOG2 = 0.75f;

__device__ __forceinline__ float widen16(uint32_t h, bool fp16) {
  return fp16 ? __half2float(__ushort_as_half((uint16_t)h)) : __bfloat162float(__ushort_as_bfloat16((uint16_t)h));
}

// One CTA per (tensor, batch, head, block of 128 rows): the block's amax,
// its scale, and its codes (Q, K row-major; V transposed through shared
// memory, 128 columns at a time).  HBM-bound: reads the block twice (the
// second time from L2) and writes one byte per element.
__global__ void __launch_bounds__(256) ffpa_fp8_quant_kernel(const __grid_constant__ Fp8Quant z) {
  __shared__ __align__(16) uint8_t tile[128][144];
  __shared__ float red[8];
  const long long cta = blockIdx.x;
  const int t = cta < z.cta_end[0] ? 0 : cta < z.cta_end[1] ? 1 : 2;
  long long local = cta - (t ? z.cta_end[t - 1] : 0);
  const int blk = (int)(local % z.nblk[t]);
  local /= z.nblk[t];
  const int H = z.H[t];
  const int h = (int)(local % H);
  const int b = (int)(local / H);
  const int D = z.D, r0 = blk * F8_BLOCK;
  const int rows = min(F8_BLOCK, z.N[t] - r0);
  const bool fp16 = z.fp16 != 0;
  const uint16_t* base = static_cast<const uint16_t*>(z.src[t]) + b * z.str[t][0] + h * z.str[t][1];
  const long long rs = z.str[t][2];
  // ---- amax over the block's rows
  float amax = 0.f;
  const int v8 = D / 8;
  for (int i = threadIdx.x; i < rows * v8; i += blockDim.x) {
    const int r = i / v8, c = (i % v8) * 8;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(base + (r0 + r) * rs + c));
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax = fmaxf(amax, fabsf(widen16(wd[j] & 0xffffu, fp16)));
      amax = fmaxf(amax, fabsf(widen16(wd[j] >> 16, fp16)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, red[w]);
  float inv = 0.f, s = 1.f;
  if (amax > 0.f) {
    const float t_inv = __fdiv_rn(448.f, amax);
    if (isfinite(t_inv)) {
      inv = t_inv;
      s = __fdiv_rn(amax, 448.f);
    }
  }
  if (threadIdx.x == 0) z.scales[t][((long long)b * H + h) * z.nblk[t] + blk] = s;
  auto q8 = [&](uint32_t w, float* y) {
    y[0] = fminf(fmaxf(__fmul_rn(widen16(w & 0xffffu, fp16), inv), -448.f), 448.f);
    y[1] = fminf(fmaxf(__fmul_rn(widen16(w >> 16, fp16), inv), -448.f), 448.f);
  };
  const long long npad = z.npad[t];
  if (t < 2) {
    // ---- Q, K: row-major codes, 16 per thread and step (one 16-byte store)
    uint8_t* out = z.codes[t] + (((long long)b * H + h) * npad + r0) * D;
    const int v16 = D / 16;
    for (int i = threadIdx.x; i < F8_BLOCK * v16; i += blockDim.x) {
      const int r = i / v16, c = (i % v16) * 16;
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
      if (r < rows) {
        const uint4* src = reinterpret_cast<const uint4*>(base + (r0 + r) * rs + c);
        const uint4 a = __ldg(src), bq = __ldg(src + 1);
        const uint32_t wd[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
        float y[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) q8(wd[j], y + 2 * j);
        o.x = pack_e4m3x4(y[0], y[1], y[2], y[3]);
        o.y = pack_e4m3x4(y[4], y[5], y[6], y[7]);
        o.z = pack_e4m3x4(y[8], y[9], y[10], y[11]);
        o.w = pack_e4m3x4(y[12], y[13], y[14], y[15]);
      }
      *reinterpret_cast<uint4*>(out + (long long)r * D + c) = o;
    }
  } else {
    // ---- V: transposed, V8T[b][h][col][r0 + r], 128 columns at a time
    uint8_t* out = z.codes[2] + ((long long)b * H + h) * D * npad + r0;
    for (int c0 = 0; c0 < D; c0 += 128) {
      for (int i = threadIdx.x; i < F8_BLOCK * 16; i += blockDim.x) {
        const int r = i / 16, c = (i % 16) * 8;
        uint32_t lo = 0u, hi = 0u;
        if (r < rows) {
          const uint4 a = __ldg(reinterpret_cast<const uint4*>(base + (r0 + r) * rs + c0 + c));
          float y[8];
          q8(a.x, y);
          q8(a.y, y + 2);
          q8(a.z, y + 4);
          q8(a.w, y + 6);
          lo = pack_e4m3x4(y[0], y[1], y[2], y[3]);
          hi = pack_e4m3x4(y[4], y[5], y[6], y[7]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          tile[c + j][r] = (uint8_t)(lo >> (8 * j));
          tile[c + 4 + j][r] = (uint8_t)(hi >> (8 * j));
        }
      }
      __syncthreads();
      for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
        const int c = i / 8, k = (i % 8) * 16;
        *reinterpret_cast<uint4*>(out + (long long)(c0 + c) * npad + k) =
            *reinterpret_cast<const uint4*>(&tile[c][k]);
      }
      __syncthreads();
    }
  }
}

// P = exp2(x - base) for 32 scores, as e4m3 (four per word, the first key
// in the lowest byte); returns the sum of the unrounded values.
__device__ __forceinline__ float form_p8(const float* x, float base, uint32_t* w) {
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
__global__ void __launch_bounds__(NTHREADS, 1) ffpa_fwd_fp8_kernel(const __grid_constant__ Params p) {
  Item it;
  if (!decode_item(p, false, blockIdx.x, it)) return;   // uniform across the CTA
  constexpr bool QRES = NCH8 <= 4;                       // Q (128 x D bytes) resident up to D = 512
  constexpr int QPAIRS = (NCH8 + 1) / 2;                 // 32 KB slots of two 128-byte chunks
  const int inject = p.inject;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t qreg_u32 = smem_u32(smem);
  const uint32_t ring_u32 = qreg_u32 + (QRES ? QPAIRS * SLOT_BYTES : 0u);
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
      mbar_init(smem_u32(&bar_drain[b]), 1);
    }
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
  constexpr uint32_t PAIR_BYTES = (NCH8 >= 2 ? 2 : 1) * CHUNK_BYTES;   // one box: 1 or 2 chunks

  if (warp == PRODUCER_WARP || warp == V_PRODUCER_WARP) {
    // ------------------------------------------------------------ producers
    // Warp 4 fills the K ring (Q pairs too when Q is not resident), warp 7
    // the V ring (one stage per key tile: it.dv rows of 128 keys).
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
      bool drop = k_role && inject != 0;   // test hook (ffpa_options.test_drop_first_copy)
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
        if (QRES) {
          const uint32_t qb = smem_u32(&bar_q);
          mbar_arrive_expect_tx(qb, QPAIRS * PAIR_BYTES);
          for (int pr = 0; pr < QPAIRS; ++pr)
            tma_load_5d(qreg_u32 + pr * SLOT_BYTES, &p.tm_q, qb, 0, it.q0, 2 * pr, it.hq, it.b);
        }
        for (int j = 0; j < T && ok; ++j) {
          const int key0 = kv_tile(it, j) * BN;
          for (int pr = 0; pr < QPAIRS && ok; ++pr) {
            uint32_t fb = 0, dst;
            if (!QRES) {
              dst = acquire(PAIR_BYTES, fb);
              if (dst == ~0u) { ok = false; break; }
              if (dst) tma_load_5d(dst, &p.tm_q, fb, 0, it.q0, 2 * pr, it.hq, it.b);
            }
            dst = acquire(PAIR_BYTES, fb);
            if (dst == ~0u) { ok = false; break; }
            if (dst) tma_load_5d(dst, &p.tm_k, fb, 0, key0, 2 * pr, it.hkv, it.b);
          }
        }
        if (QRES) wait_drain(smem_u32(&bar_q), 0, tmo, err);
      } else {
        for (int j = 0; j < T && ok; ++j) {
          uint32_t fb = 0;
          const uint32_t dst = acquire(vslot, fb);
          if (dst == ~0u) { ok = false; break; }
          tma_load_4d(dst, &p.tm_v, fb, kv_tile(it, j) * BN, it.col_lo, it.hkv, it.b);
        }
      }
      const int n = issued < nslots ? issued : nslots;
      int s = slot;
      uint32_t lp = lap;
      for (int i = 0; i < n; ++i) {
        if (--s < 0) { s = nslots - 1; lp ^= 1u; }
        if (k_role && inject != 0 && issued - 1 - i == 0) continue;   // never armed
        wait_drain(smem_u32(&full[s]), lp, tmo, err);
      }
    }
  } else if (warp == MMA_WARP || warp == PV_WARP) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      const bool qk_role = warp == MMA_WARP;
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
      auto wait_on = [&](uint32_t bar, uint32_t par) -> bool {
        if (!mbar_try_wait(bar, par) && !wait_bounded(bar, par, &abort_flag, tmo, err)) return false;
        tc_fence_after();
        return true;
      };
      if (qk_role) {
        const uint32_t idesc_qk = idesc_e4m3(BM, BN);
        const uint64_t ring_desc = sdesc_sw128(ring_u32, 16, 1024);
        const uint64_t q_desc = sdesc_sw128(qreg_u32, 16, 1024);
        const uint32_t s_col = tmem + S_COL;
        if (T > 0 && QRES) ok = wait_on(smem_u32(&bar_q), 0);
        for (int j = 0; j < T && ok; ++j) {
          if (j >= 1 && !(ok = wait_on(smem_u32(&bar_s_free), (j - 1) & 1))) break;
#pragma unroll
          for (int pr = 0; pr < QPAIRS; ++pr) {
            int sq = -1;
            if (!QRES) {
              sq = take();
              if (sq < 0) { ok = false; break; }
            }
            const int sk = take();
            if (sk < 0) { ok = false; break; }
            const uint64_t ad = QRES ? q_desc + (((2 * pr) * CHUNK_BYTES) >> 4)
                                     : ring_desc + ((sq * SLOT_BYTES) >> 4);
            const uint64_t bd = ring_desc + ((sk * SLOT_BYTES) >> 4);
            // 32 e4m3 per MMA: +32 bytes (>>4 = 2) within a 128-byte row; the
            // second chunk of the pair sits 16 KB (>>4 = 1024) further.
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_ss_f8(s_col, ad + 2 * k, bd + 2 * k, idesc_qk, (pr > 0 || k > 0) ? 1u : 0u);
            if (2 * pr + 1 < NCH8) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_ss_f8(s_col, ad + 1024 + 2 * k, bd + 1024 + 2 * k, idesc_qk, 1u);
            }
            if (sq >= 0) umma_commit(smem_u32(&empty[sq]));
            umma_commit(smem_u32(&empty[sk]));
          }
          if (!ok) break;
          umma_commit(smem_u32(&bar_s_full));
        }
      } else {
        const uint32_t idesc_pv = idesc_e4m3(BM, it.dv);
        const uint64_t v_desc = sdesc_sw128(vring_u32, 16, 1024);
        for (int j = 0; j < T && ok; ++j) {
          const int b = j & 1;
          if (!(ok = wait_on(smem_u32(&bar_p_full[b]), (j >> 1) & 1))) break;
          const int s = take();
          if (s < 0) { ok = false; break; }
          const uint64_t vd = v_desc + ((s * vslot) >> 4);
          const uint32_t p_col = tmem + F8_P_COL0 + 32 * b;
          // 32 keys per MMA: +8 TMEM columns of P (4 keys each), +32 bytes of V.
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_ts_f8(tmem, p_col + 8 * k, vd + 2 * k, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&empty[s]));
          umma_commit(smem_u32(&bar_pv_done[b]));
        }
      }
      const uint32_t db = smem_u32(&bar_drain[qk_role ? 0 : 1]);
      umma_commit(db);
      wait_drain(db, 0, tmo, err);
    }
  } else {
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
    // Block scales: this tile's Q block, and the head's K and V blocks.
    const int Hkv = p.Hq / p.group;
    const float s_q = p.sq[((long long)it.b * p.Hq + it.hq) * p.n_qt + it.q0 / F8_BLOCK];
    const float* s_k = p.sk + ((long long)it.b * Hkv + it.hkv) * p.n_kb;
    const float* s_v = p.sv + ((long long)it.b * Hkv + it.hkv) * p.n_kb;
    float G = 0.f;
    for (int t = 0; t < p.n_kb; ++t) G = fmaxf(G, __ldg(s_v + t));
    float m_ref = -INFINITY;
    float l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int b = j & 1;
      bool w = wait_bounded(smem_u32(&bar_s_full), j & 1, &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      tc_fence_after();
      const int tile = kv_tile(it, j);
      const int kbase = tile * BN;
      const bool need_mask = (kbase + BN > it.kv_len) ||
                             (causal && (long long)kbase + BN - 1 > first_limit) ||
                             mask_kind != FFPA_MASK_NONE;
      // Scores in the log2 domain: the tile's scale folds s_q s_k.
      const float f = p.scale_log2 * s_q * __ldg(s_k + tile);
      const float c_t = 256.f * __ldg(s_v + tile) / G;
      float x[BN];
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
      const float mx = row_max<BN>(x);
      bool resc = false;
      float alpha = 1.f;
      if (mx > m_ref + F8_RESCALE_LOG2) {
        if (m_ref != -INFINITY) {
          resc = true;
          alpha = ex2_approx(m_ref - mx);
        }
        m_ref = mx;
      }
      if (__any_sync(0xffffffffu, resc)) {
        w = wait_bounded(smem_u32(&bar_pv_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, &abort_flag, tmo, err);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
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
      if (j >= 2) {   // P buffer b was read by PV_{j-2}
        w = wait_bounded(smem_u32(&bar_pv_done[b]), ((j - 2) >> 1) & 1, &abort_flag, tmo, err);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
      }
      // P * c_t in e4m3: exp2(x - m_ref + log2 c_t); the row sum keeps p.
      const float base = (m_ref == -INFINITY ? 0.f : m_ref) - __log2f(c_t);
      uint32_t pw[32];
      float psum = 0.f;
#pragma unroll
      for (int g = 0; g < 4; ++g) psum += form_p8(x + 32 * g, base, pw + 8 * g);
      l_sum = l_sum * alpha + psum / c_t;
      tmem_st32(lane_base + F8_P_COL0 + 32 * b, pw);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_p_full[b]));
    }
    if (ok && T > 0) {
      const bool w = wait_bounded(smem_u32(&bar_pv_done[(T - 1) & 1]), ((T - 1) >> 1) & 1,
                                  &abort_flag, tmo, err);
      ok = __all_sync(0xffffffffu, w);
      if (ok) tc_fence_after();
    }
    if (ok || T == 0)
      store_output<false>(p, it, T > 0, lane_base, row, row_valid, l_sum, m_ref, G / 256.f);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int NCH8>
static ffpa_status launch_fp8_t(bool umask, const Params& P, int items, size_t smem, cudaStream_t stream) {
  auto kern = umask ? ffpa_fwd_fp8_kernel<NCH8, true> : ffpa_fwd_fp8_kernel<NCH8, false>;
  const ffpa_status st = set_smem_attr_once(reinterpret_cast<const void*>(kern), P.device,
                                            static_cast<int>(SMEM_LIMIT - SMEM_STATIC_RESERVE));
  if (st != FFPA_OK) return st;
  kern<<<items, NTHREADS, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}

ffpa_status launch_fp8(const Fp8Quant& Qz, const Params& P, int items, size_t smem, bool split,
                       cudaStream_t stream) {
  const long long ctas = Qz.cta_end[2];
  if (ctas > 0) {
    ffpa_fp8_quant_kernel<<<(unsigned)ctas, 256, 0, stream>>>(Qz);
    if (cudaGetLastError() != cudaSuccess) return FFPA_ERR_CUDA;
  }
  if (split) return launch_fp8_split(P, items, smem, stream);
  const bool umask = P.mask != nullptr;
  switch (P.D / 128) {
    case 1: return launch_fp8_t<1>(umask, P, items, smem, stream);
    case 2: return launch_fp8_t<2>(umask, P, items, smem, stream);
    case 3: return launch_fp8_t<3>(umask, P, items, smem, stream);
    case 4: return launch_fp8_t<4>(umask, P, items, smem, stream);
    case 5: return launch_fp8_t<5>(umask, P, items, smem, stream);
    case 6: return launch_fp8_t<6>(umask, P, items, smem, stream);
    case 7: return launch_fp8_t<7>(umask, P, items, smem, stream);
    case 8: return launch_fp8_t<8>(umask, P, items, smem, stream);
    default: return FFPA_ERR_UNSUPPORTED;
  }
}

}  // namespace ffpa
