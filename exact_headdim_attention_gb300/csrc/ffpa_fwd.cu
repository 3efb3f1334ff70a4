// Exact attention forward for large head dimensions on GB300 (sm_103a).
//
// Method (FFPA README, "Split-D and TiledMMA"; FFPA API reference,
// "ffpa_attn.ffpa_attn_func" / "ffpa_attn_varlen_func"): a FlashAttention
// style online softmax over key tiles, with the head dimension D split into
// 64-wide chunks so that the on-chip staging of Q, K and V does not grow
// with D ("Split-D").  On Blackwell the accumulators live in Tensor Memory
// (TMEM, 128 lanes x 512 fp32 columns per SM) instead of registers, so the
// pages' register-pressure problem becomes a TMEM-capacity problem: a CTA
// owns at most 256 output columns ("output-D slice") next to one 128-column
// S buffer and two 64-column P buffers.  When D > 256 the output columns are
// split across CTAs and each CTA recomputes S for its slice.
//
// Per CTA (one work item = batch b, query head h, 128-row query tile,
// output-D slice) the warps specialise:
//   warps 0-3  softmax: row r = 32*warp + lane; read S from TMEM, mask,
//              online max / exp2 / sum, write P (16-bit) to a P buffer, rescale
//              O when the running max moved by more than 2^8, epilogue.
//   warp 4     TMA producer: Q/K D-chunk pairs and V stages into a ring of
//              32 KB shared-memory slots (128-byte swizzle), in the exact
//              order the MMA warp consumes them.
//   warp 5     MMA issuer (one thread): S_j = sum_c Q_c K_{j,c}^T into TMEM
//              (tcgen05.mma, smem x smem), O += P_j V_j (P from TMEM).
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the
// kernel records FFPA_ERR_DEVICE_TIMEOUT, drains its own copies and MMAs,
// frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "ffpa.h"
#include "ptx.cuh"

namespace ffpa {

constexpr int BM = 128;              // query rows per tile = TMEM lanes
constexpr int BN = 128;              // keys per S tile
constexpr int DK = 64;               // D chunk: one 128-byte swizzle row of 16-bit values
constexpr int DV_MAX = 256;          // output columns per CTA
constexpr int NSLOT_MAX = 6;         // K-ring slots (fewer when Q is resident)
constexpr int NSLOT_V_MAX = 2;       // V-ring slots
constexpr uint32_t SLOT_BYTES = 32768;         // one TMA box of 2 D-chunks (32 KB)
constexpr uint32_t CHUNK_BYTES = BM * DK * 2;  // 16 KB: one 128x64 tile
constexpr int Q_RESIDENT_MAX_CHUNKS = 8;       // Q stays in smem for D <= 512
constexpr size_t SMEM_LIMIT = 232448;          // opt-in dynamic smem per block (sm_103)
constexpr size_t SMEM_STATIC_RESERVE = 1024;
constexpr int NTHREADS = 256;
constexpr int PRODUCER_WARP = 4;     // TMA for Q and the K ring
constexpr int MMA_WARP = 5;          // issues S = Q K^T; owns the TMEM allocation
constexpr int PV_WARP = 6;           // issues O += P V
constexpr int V_PRODUCER_WARP = 7;   // TMA for the V ring
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 256;      // S (fp32, 128 keys) occupies columns [256, 384)
constexpr uint32_t P_COL0 = 384;     // P buffer b (16-bit pairs, 128 keys) at [384 + 64 b, +64)
constexpr float RESCALE_LOG2 = 8.0f; // rescale O only when the max grows by > 2^8

__device__ int g_err_word;

struct Params {
  // Views with D split as (64, D/64): dense (64, N, D/64, H, B); varlen
  // (64, T, D/64, H).  Q and K boxes: 64 x 128 rows x min(2, D/64) chunks;
  // V box: 64 x vk rows x vchunks chunks.
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  void* o;
  float* lse;
  const void* mask;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int64_t o_str[4];    // dense (b, h, n, d); varlen (t, h, d)
  int64_t m_str[4];
  int mask_kind;
  int B;               // batches (dense) or sequences (varlen)
  int Hq, group, Nq, Nkv, D, Tq;
  int n_qt, n_slices, nchunks, vk, vchunks, kchunks;
  int q_res, nslot;    // Q resident in smem (1) or streamed through the K ring (0); K-ring depth
  int nslot_v, vslot;  // V-ring depth and slot bytes (vk keys x vchunks 64-column chunks)
  int kslot, kc;       // pair kernel: K-ring slot bytes and D-chunks per K stage
  int qt_chunks;       // column-split kernel: Q chunks held in TMEM
  float scale_log2;
  int causal, fp16, inject;
  unsigned long long timeout_ns;
};

struct Item {
  int b, hq, hkv, slice;
  int q0, q_len, kv_len, q_row0, kv_row0;
  int col_lo, dv, ntiles;
  int rot;   // first key tile visited; tiles are visited rot, rot+1, ... (mod ntiles)
};

// Key tile visited at step j.  Work items of one head start at different
// tiles so that they do not all miss in L2 on the same tile at the same time;
// the online softmax gives the same result for any visiting order.
__device__ __forceinline__ int kv_tile(const Item& it, int j) {
  const int t = j + it.rot;
  return t >= it.ntiles ? t - it.ntiles : t;
}

__device__ __forceinline__ bool decode_item(const Params& p, bool varlen, int L, Item& it) {
  it.slice = L % p.n_slices;
  L /= p.n_slices;
  const int heads = p.B * p.Hq;
  int qt;
  if (p.causal) {                    // longest query tiles first
    const int bh = L % heads;
    qt = p.n_qt - 1 - L / heads;
    it.hq = bh % p.Hq;
    it.b = bh / p.Hq;
  } else {                           // tiles of one head adjacent: K/V reuse in L2
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
  it.q0 = qt * BM;
  if (it.q0 >= it.q_len) return false;
  const int rows = min(BM, it.q_len - it.q0);
  long long kv_end = it.kv_len;
  if (p.causal) {
    const long long last_visible = (long long)it.q0 + rows - 1 + (it.kv_len - it.q_len);
    kv_end = min(kv_end, last_visible + 1);
  }
  it.ntiles = kv_end > 0 ? (int)((kv_end + BN - 1) / BN) : 0;
  it.rot = it.ntiles > 0 ? (int)(((unsigned)qt * 37u + (unsigned)it.slice * 17u + (unsigned)it.hq * 13u) %
                                 (unsigned)it.ntiles)
                         : 0;
  const int c_lo = it.slice * p.nchunks / p.n_slices;
  const int c_hi = (it.slice + 1) * p.nchunks / p.n_slices;
  it.col_lo = c_lo * DK;
  it.dv = (c_hi - c_lo) * DK;
  return true;
}

// Bounded wait on an mbarrier phase.  Returns false when this CTA has been
// told to abort or when the limit expires (then the error word is set).
// `cluster` selects cluster-scope acquire, for phases that another CTA of
// the cluster completes.
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long timeout_ns, bool cluster = false) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    // Suspended waiting keeps idle warps from taking issue slots away from
    // the MMA and TMA threads that share their SM sub-partition.
    if (cluster ? mbar_try_wait_sleep_cluster(bar, parity, 20000u)
                : mbar_try_wait_sleep(bar, parity, 20000u))
      return true;
    if ((it & 7u) == 7u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        atomicExch(&g_err_word, (int)FFPA_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

// Drain wait used on the way out: ignores the abort flag.
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, unsigned long long timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) {
      atomicExch(&g_err_word, (int)FFPA_ERR_DEVICE_TIMEOUT);
      return;
    }
  }
}

// Masks 32 consecutive scores (log2 domain) of one row: keys past the end,
// keys beyond the causal limit, and the caller's bool/additive mask.
__device__ __forceinline__ void apply_mask32(float* x, int key0, int kv_len, bool causal,
                                             long long row_limit, const uint8_t* mrow,
                                             long long mk, int mask_kind, bool fp16) {
  const float LOG2E = 1.4426950408889634f;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const int key = key0 + c;
    bool vis = key < kv_len && (!causal || (long long)key <= row_limit);
    float add = 0.f;
    if (vis && mrow != nullptr) {
      const long long e = (long long)key * mk;
      if (mask_kind == FFPA_MASK_BOOL) {
        vis = mrow[e] != 0;
      } else if (mask_kind == FFPA_MASK_ADD_F32) {
        add = reinterpret_cast<const float*>(mrow)[e] * LOG2E;
      } else {
        const uint16_t hbits = reinterpret_cast<const uint16_t*>(mrow)[e];
        const float hv = fp16 ? __half2float(__ushort_as_half(hbits))
                              : __bfloat162float(__ushort_as_bfloat16(hbits));
        add = hv * LOG2E;
      }
    }
    x[c] = vis ? x[c] + add : -INFINITY;
  }
}

// Epilogue of one row: O (TMEM columns [0, it.dv), or zeros when no key
// tile was visited) scaled by 1/l, written as 16-bit values to the output
// columns [it.col_lo, it.col_lo + it.dv); the LSE by the CTA of slice 0.
template <bool VARLEN>
__device__ __forceinline__ void store_output(const Params& p, const Item& it, bool have_o,
                                             uint32_t lane_base, int row, bool row_valid,
                                             float l_sum, float m_ref) {
  const bool fp16 = p.fp16 != 0;
  const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
  uint8_t* obase = nullptr;
  if (row_valid) {
    long long off;
    if (VARLEN)
      off = (long long)(it.q_row0 + row) * p.o_str[0] + (long long)it.hq * p.o_str[1];
    else
      off = (long long)it.b * p.o_str[0] + (long long)it.hq * p.o_str[1] +
            (long long)row * p.o_str[2];
    obase = static_cast<uint8_t*>(p.o) + (off + it.col_lo) * 2;
  }
  for (int c0 = 0; c0 < it.dv; c0 += 32) {
    uint32_t o[32];
    if (have_o) {
      tmem_ld32(lane_base + c0, o);
      tmem_wait_ld();
      reg_fence(o);
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) o[c] = 0u;
    }
    uint32_t pkd[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float a0 = __uint_as_float(o[2 * c]) * inv_l;
      const float a1 = __uint_as_float(o[2 * c + 1]) * inv_l;
      pkd[c] = fp16 ? pack_f16(a0, a1) : pack_bf16(a0, a1);
    }
    if (row_valid) {
      uint4* dst = reinterpret_cast<uint4*>(obase + c0 * 2);
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4)
        dst[v4] = make_uint4(pkd[4 * v4], pkd[4 * v4 + 1], pkd[4 * v4 + 2], pkd[4 * v4 + 3]);
    }
  }
  if (row_valid && p.lse != nullptr && it.slice == 0) {
    const float lse = l_sum > 0.f ? (m_ref + log2f(l_sum)) * 0.6931471805599453f : -INFINITY;
    long long li;
    if (VARLEN)
      li = (long long)it.hq * p.Tq + it.q_row0 + row;
    else
      li = ((long long)it.b * p.Hq + it.hq) * p.Nq + row;
    p.lse[li] = lse;
  }
}

// P = exp2(x * xs - base) for n scores, packed to 16-bit pairs; returns the
// sum of the (unrounded) values.
template <bool F16, int N>
__device__ __forceinline__ float form_p(const float* x, float xs, float base, uint32_t* pk) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int c = 0; c < N; c += 4) {
    const float e0 = ex2_approx(fmaf(x[c], xs, -base));
    const float e1 = ex2_approx(fmaf(x[c + 1], xs, -base));
    const float e2 = ex2_approx(fmaf(x[c + 2], xs, -base));
    const float e3 = ex2_approx(fmaf(x[c + 3], xs, -base));
    s0 += e0; s1 += e1; s2 += e2; s3 += e3;
    pk[c / 2] = F16 ? pack_f16(e0, e1) : pack_bf16(e0, e1);
    pk[c / 2 + 1] = F16 ? pack_f16(e2, e3) : pack_bf16(e2, e3);
  }
  return (s0 + s1) + (s2 + s3);
}

// Barrier addresses seen by the softmax warps.  The arrive addresses are
// shared::cluster addresses (the leader CTA's barriers) in pair mode and
// plain shared-memory addresses of this CTA otherwise.
// The two-entry barrier arrays are consecutive 8-byte objects, so entry b
// sits at base + 8 b.
struct SoftmaxBars {
  uint32_t s_full;
  uint32_t s_free_arrive;
  uint32_t p_full_arrive;   // entry 0 of p_full[2]
  uint32_t pv_done;         // entry 0 of pv_done[2]
};

// The softmax arrivals follow tcgen05.wait::ld (S read into registers) or
// tcgen05.wait::st + tcgen05.fence (P written to TMEM); no generic-memory
// write has to become visible, so the pair form is a relaxed arrive (a
// cluster-scope release costs ~1000 cycles on this critical path).
template <bool PAIR>
__device__ __forceinline__ void arrive_to(uint32_t addr) {
  if (PAIR)
    mbar_arrive_cluster_relaxed(addr);
  else
    mbar_arrive(addr);
}

// Softmax warps 0-3 and the epilogue: thread r owns query row it.q0 + r,
// which is TMEM lane r of this CTA.
template <bool VARLEN, bool PAIR>
__device__ __forceinline__ void softmax_role(const Params& p, const Item& it, int T, uint32_t tmem,
                                             int warp, int lane, const SoftmaxBars bars,
                                             volatile int* abort_flag, unsigned long long tmo) {
  const int mask_kind = p.mask_kind;
  const bool fp16 = p.fp16 != 0, causal = p.causal != 0;
  const float scale_log2 = p.scale_log2;
    // ------------------------------------------------------------ softmax
  const int r = warp * 32 + lane;                 // row within the tile = TMEM lane
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const int row = it.q0 + r;                      // row within the sequence
  const bool row_valid = row < it.q_len;
  const long long row_limit = (long long)row + (it.kv_len - it.q_len);   // causal
  const long long first_limit = (long long)it.q0 + (it.kv_len - it.q_len);
  const uint8_t* mrow = nullptr;
  if (mask_kind != FFPA_MASK_NONE && row_valid) {
    const size_t esz = mask_kind == FFPA_MASK_BOOL ? 1 : mask_kind == FFPA_MASK_ADD_F32 ? 4 : 2;
    const long long off = (long long)it.b * p.m_str[0] + (long long)it.hq * p.m_str[1] +
                          (long long)row * p.m_str[2];
    mrow = static_cast<const uint8_t*>(p.mask) + off * (long long)esz;
  }
  const long long mk = p.m_str[3];
  // Scores stay unscaled (x = q.k) when possible, so that the exponent
  // x*scale*log2(e) - m is one FFMA; additive masks (or a scale <= 0, which
  // reverses the max) need x pre-scaled into the log2 domain.
  const bool prescale = mask_kind == FFPA_MASK_ADD_F32 || mask_kind == FFPA_MASK_ADD_QTYPE ||
                        !(scale_log2 > 0.f);
  const float xs = prescale ? 1.f : scale_log2;
  const float ld_scale = prescale ? scale_log2 : 1.f;
  float m_ref = -INFINITY;
  float l_sum = 0.f;
  bool ok = true;
  for (int j = 0; j < T; ++j) {
    const int b = j & 1;
    bool w = wait_bounded(bars.s_full, j & 1, abort_flag, tmo);
    ok = __all_sync(0xffffffffu, w);
    if (!ok) break;
    tc_fence_after();
    const uint32_t s_addr = lane_base + S_COL;
    const uint32_t p_addr = lane_base + P_COL0 + 64 * b;
    const int kbase = kv_tile(it, j) * BN;
    const bool need_mask = (kbase + BN > it.kv_len) ||
                           (causal && (long long)kbase + BN - 1 > first_limit) ||
                           mask_kind != FFPA_MASK_NONE;
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
      // S has been read into registers: the next QK may overwrite it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_to<PAIR>(bars.s_free_arrive);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        x[c] = __uint_as_float(r0[c]) * ld_scale;
        x[32 + c] = __uint_as_float(r1[c]) * ld_scale;
        x[64 + c] = __uint_as_float(r2[c]) * ld_scale;
        x[96 + c] = __uint_as_float(r3[c]) * ld_scale;
      }
    }
    if (need_mask) {
#pragma unroll
      for (int q4 = 0; q4 < BN / 32; ++q4)
        apply_mask32(x + 32 * q4, kbase + 32 * q4, it.kv_len, causal, row_limit, mrow, mk,
                     mask_kind, fp16);
    }
    float mx;
    {   // tree maximum: eight independent chains, then combine
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = x[i];
#pragma unroll
      for (int c = 8; c < BN; c += 8)
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], x[c + i]);
      mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                 fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      mx *= xs;   // into the log2 domain (-inf stays -inf: xs > 0)
    }
    bool resc = false;
    float alpha = 1.f;
    if (mx > m_ref + RESCALE_LOG2) {
      if (m_ref != -INFINITY) {
        resc = true;
        alpha = ex2_approx(m_ref - mx);
      }
      m_ref = mx;
    }
    if (__any_sync(0xffffffffu, resc)) {
      // O holds PV up to tile j-1: wait for it, then scale this warp's rows.
      w = wait_bounded(bars.pv_done + 8u * ((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag, tmo);
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
      w = wait_bounded(bars.pv_done + 8u * b, ((j - 2) >> 1) & 1, abort_flag, tmo);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      tc_fence_after();
    }
    // P = exp2(x - m_ref) in 16-bit, into P buffer b.
    const float base = m_ref == -INFINITY ? 0.f : m_ref;
    float psum = 0.f;
#pragma unroll
    for (int g = 0; g < BN / 32; ++g) {
      uint32_t pk[16];
      psum += fp16 ? form_p<true, 32>(x + 32 * g, xs, base, pk)
                   : form_p<false, 32>(x + 32 * g, xs, base, pk);
      tmem_st16(p_addr + 16 * g, pk);
    }
    l_sum = l_sum * alpha + psum;
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) arrive_to<PAIR>(bars.p_full_arrive + 8u * b);
  }
  // ------------------------------------------------------------ epilogue
  if (ok && T > 0) {
    const bool w = wait_bounded(bars.pv_done + 8u * ((T - 1) & 1), ((T - 1) >> 1) & 1,
                                abort_flag, tmo);
    ok = __all_sync(0xffffffffu, w);
    if (ok) tc_fence_after();
  }
  if (ok || T == 0) store_output<VARLEN>(p, it, T > 0, lane_base, row, row_valid, l_sum, m_ref);
}

template <bool VARLEN>
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
        if (!mbar_try_wait(eb, lap ^ 1u) && !wait_bounded(eb, lap ^ 1u, &abort_flag, tmo))
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
      auto load_q_pair = [&](uint32_t dst, uint32_t fb, int pr) {
        if (VARLEN)
          tma_load_4d(dst, &p.tm_q, fb, 0, it.q_row0 + it.q0, 2 * pr, it.hq);
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
              else
                tma_load_5d(dst, &p.tm_k, fb, 0, key0, 2 * pr, it.hkv, it.b);
            }
          }
        }
        if (q_res) wait_drain(smem_u32(&bar_q), 0, tmo);
      } else {
        for (int j = 0; j < T && ok; ++j) {
          for (int h = 0; h < BN / vk && ok; ++h) {
            uint32_t fb = 0;
            const uint32_t dst = acquire(vslot, fb);
            if (dst == ~0u) { ok = false; break; }
            const int key = kv_tile(it, j) * BN + h * vk;
            if (VARLEN)
              tma_load_4d(dst, &p.tm_v, fb, 0, it.kv_row0 + key, it.col_lo / DK, it.hkv);
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
        wait_drain(smem_u32(&full[s]), lp, tmo);
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
        if (!mbar_try_wait(fb, lap) && !wait_bounded(fb, lap, &abort_flag, tmo)) return -1;
        const int s = slot;
        if (++slot == nslots) { slot = 0; lap ^= 1u; }
        return s;
      };
      auto release = [&](int s) { umma_commit(smem_u32(&empty[s])); };
      auto wait_on = [&](uint32_t bar, uint32_t par) -> bool {
        if (!mbar_try_wait(bar, par) && !wait_bounded(bar, par, &abort_flag, tmo)) return false;
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
      wait_drain(db, 0, tmo);
    }
  } else {
    // ------------------------------------------------------------ softmax
    SoftmaxBars bars;
    bars.s_full = smem_u32(&bar_s_full);
    bars.s_free_arrive = smem_u32(&bar_s_free);
    bars.p_full_arrive = smem_u32(&bar_p_full[0]);
    bars.pv_done = smem_u32(&bar_pv_done[0]);
    softmax_role<VARLEN, false>(p, it, T, tmem, warp, lane, bars, &abort_flag, tmo);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}


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
constexpr int BM_PAIR = 256;
constexpr int KEYS_PER_CTA = BN / 2;

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
  it.rot = it.ntiles > 0 ? (int)(((unsigned)qt * 37u + (unsigned)it.slice * 17u + (unsigned)it.hq * 13u) %
                                 (unsigned)it.ntiles)
                         : 0;
  const int c_lo = it.slice * p.nchunks / p.n_slices;
  const int c_hi = (it.slice + 1) * p.nchunks / p.n_slices;
  it.col_lo = c_lo * DK;
  it.dv = (c_hi - c_lo) * DK;
  return true;
}

// NCH = D / 64 as a template parameter: the MMA issue loops unroll.
template <bool VARLEN, int NCH>
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
        if (!mbar_try_wait(eb, lap ^ 1u) && !wait_bounded(eb, lap ^ 1u, &abort_flag, tmo))
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
        wait_drain(qb, 0, tmo);
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
        wait_drain(smem_u32(&full[s]), lp, tmo);
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
        if (!(mbar_try_wait(qb, 0) || wait_bounded(qb, 0, &abort_flag, tmo))) goto relay_done;
        mbar_arrive_cluster(mapa_shared(qb, 0));
      }
      {
        int slot = 0;
        uint32_t lap = 0;
        for (int i = 0; i < T * per_tile; ++i) {
          const uint32_t fb = smem_u32(&full[slot]);
          if (!(mbar_try_wait(fb, lap) || wait_bounded(fb, lap, &abort_flag, tmo))) break;
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
        if (!mbar_try_wait(fb, lap) && !wait_bounded(fb, lap, &abort_flag, tmo)) return -1;
        const int s = slot;
        if (++slot == nslots) { slot = 0; lap ^= 1u; }
        return s;
      };
      auto wait_on = [&](uint32_t bar, uint32_t par) -> bool {
        if (!mbar_try_wait(bar, par) && !wait_bounded(bar, par, &abort_flag, tmo)) return false;
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
      wait_drain(db, 0, tmo);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    SoftmaxBars bars;
    bars.s_full = smem_u32(&bar_s_full);
    bars.s_free_arrive = mapa_shared(smem_u32(&bar_s_free), 0);
    bars.p_full_arrive = mapa_shared(smem_u32(&bar_p_full[0]), 0);
    bars.pv_done = smem_u32(&bar_pv_done[0]);
    softmax_role<VARLEN, true>(p, it, T, tmem, warp, lane, bars, &abort_flag, tmo);
  }

  // The leader's last commits also arrive in the peer: wait for them before
  // the pair may exit, then free TMEM in both CTAs together.
  if (!leader && threadIdx.x == 0) {
    wait_drain(smem_u32(&bar_drain[0]), 0, tmo);
    wait_drain(smem_u32(&bar_drain[1]), 0, tmo);
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


// =====================================================================
// Column-split pair kernel: no recomputation of S for D up to 512.
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
constexpr int SPLIT_THREADS = 192;
constexpr uint32_t Q_TMEM_COL = 384;
constexpr int Q_TMEM_MAX_CHUNKS = 4;
constexpr uint32_t P_TILE_BYTES = BM * BN * 2;   // 2 x (128 rows x 64 keys), 16-bit
constexpr size_t SPLIT_STATIC_RESERVE = 2048;

// NCH = D / 64 is a template parameter so that every MMA issue loop has a
// compile-time trip count and is fully unrolled: the tensor pipe's
// instruction queue is shallow, and loop overhead between MMAs leaves it
// idle (measured: a runtime-count loop of 8 MMAs runs at about half rate).
template <bool VARLEN, int NCH>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(SPLIT_THREADS, 1)
    ffpa_fwd_split_kernel(const __grid_constant__ Params p) {
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  Item it;
  if (!decode_item(p, VARLEN, blockIdx.x >> 1, it)) return;   // same answer in both CTAs
  it.dv = p.D / 2;
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
        if (!mbar_try_wait(eb, lap ^ 1u) && !wait_bounded(eb, lap ^ 1u, &abort_flag, tmo))
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
      wait_drain(qb, 0, tmo);
      const int n = issued < NS ? issued : NS;
      int s = slot;
      uint32_t lp = lap;
      for (int i = 0; i < n; ++i) {
        if (--s < 0) { s = NS - 1; lp ^= 1u; }
        if (inject != 0 && rank == 0 && issued - 1 - i == 0) continue;   // never armed
        wait_drain(smem_u32(&bar_full[s]), lp, tmo);
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
        if (!mbar_try_wait(fb, lap) && !wait_bounded(fb, lap, &abort_flag, tmo)) return -1;
        const int s = slot;
        if (++slot == NS) { slot = 0; lap ^= 1u; }
        return s;
      };
      auto wait_on = [&](uint32_t bar, uint32_t par) -> bool {
        if (!mbar_try_wait(bar, par) && !wait_bounded(bar, par, &abort_flag, tmo)) return false;
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
      wait_drain(db, 0, tmo);
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
    if (mask_kind != FFPA_MASK_NONE && row_valid) {
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
      bool w = wait_bounded(smem_u32(&bar_q), 0, &abort_flag, tmo);
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
          w = wait_bounded(smem_u32(&bar_qt), 0, &abort_flag, tmo);
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
        bool w = wait_bounded(smem_u32(&bar_s_full), k_own & 1, &abort_flag, tmo);
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
            x[c] = __uint_as_float(r0[c]) * ld_scale;
            x[32 + c] = __uint_as_float(r1[c]) * ld_scale;
            x[64 + c] = __uint_as_float(r2[c]) * ld_scale;
            x[96 + c] = __uint_as_float(r3[c]) * ld_scale;
          }
        }
        if (need_mask) {
#pragma unroll
          for (int q4 = 0; q4 < BN / 32; ++q4)
            apply_mask32(x + 32 * q4, kbase + 32 * q4, it.kv_len, causal, row_limit, mrow, mk,
                         mask_kind, fp16);
        }
        float m8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) m8[u] = x[u];
#pragma unroll
        for (int c = 8; c < BN; c += 8)
#pragma unroll
          for (int u = 0; u < 8; ++u) m8[u] = fmaxf(m8[u], x[c + u]);
        t = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                  fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        t *= xs;
      }
      // Exchange the tile maxima: both CTAs then take the same decision.
      const int xb = i & 1;
      const uint32_t xbar = smem_u32(&bar_x[xb]);
      if (r == 0) mbar_arrive_expect_tx(xbar, BM * 4);
      st_async_b32(x_remote + xb * BM * 4, __float_as_uint(t), xbar_remote + 8u * xb);
      {
        const bool w = wait_bounded(xbar, (i >> 1) & 1, &abort_flag, tmo, true);
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
          w = wait_bounded(smem_u32(&bar_pown_free), (k_own - 1) & 1, &abort_flag, tmo);
        if (w) w = wait_bounded(smem_u32(&bar_peer_free), k_own & 1, &abort_flag, tmo, true);
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
        const bool w = wait_bounded(smem_u32(&bar_pv_done), (i - 1) & 1, &abort_flag, tmo);
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
      bool w = wait_bounded(smem_u32(&bar_pv_done), (R - 1) & 1, &abort_flag, tmo);
      ok = __all_sync(0xffffffffu, w);
      if (ok) {
        tc_fence_after();
        // Row sums: each CTA summed the P of its own tiles.
        const uint32_t lbar = smem_u32(&bar_l);
        if (r == 0) mbar_arrive_expect_tx(lbar, BM * 4);
        st_async_b32(mapa_shared(smem_u32(&lbuf[r]), peer), __float_as_uint(l_sum),
                     mapa_shared(lbar, peer));
        w = wait_bounded(lbar, 0, &abort_flag, tmo, true);
        ok = __all_sync(0xffffffffu, w);
        if (ok) l_sum += ld_shared_f32(smem_u32(&lbuf[r]));
      }
    }
    if (ok || T == 0) store_output<VARLEN>(p, it, T > 0, lane_base, row, row_valid, l_sum, m_ref);
    if (r == 0 && ok && T > 0) {
      // Before this CTA may exit: the peer has read every P tile copied to it.
      const int n_own = (T - own0 + 1) >> 1;
      wait_drain(smem_u32(&bar_peer_free), n_own & 1, tmo);
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

}  // namespace ffpa

// =====================================================================
// Host side: validation, planning, tensor maps, launch.
// =====================================================================
namespace {

using namespace ffpa;

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<int> g_variant{FFPA_VARIANT_AUTO};
std::atomic<int> g_drop_first_copy{0};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Element strides of every non-unit dimension but the last must be a
// multiple of 8 elements (16 bytes for 16-bit types); the last must be 1.
bool strides_ok(const int64_t* str, const int64_t* size, int rank) {
  if (str[rank - 1] != 1) return false;
  for (int i = 0; i < rank - 1; ++i) {
    if (size[i] <= 1) continue;
    if (str[i] <= 0 || (str[i] % 8) != 0) return false;
  }
  return true;
}

// Tiled tensor map with 128-byte swizzle.  dims[0] is always 64 (one
// 128-byte row of 16-bit values); byte strides are given for dims 1..rank-1.
// A size-1 dimension gets a harmless stride so its (never used) value cannot
// fail the encoder's alignment checks.
ffpa_status encode_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* stride_bytes, const uint32_t* box) {
  auto enc = encode_fn();
  if (!enc) return FFPA_ERR_CUDA;
  cuuint64_t gdim[5];
  cuuint64_t gstr[4];
  cuuint32_t bx[5];
  cuuint32_t es[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 1; i < rank; ++i) {
    uint64_t st = stride_bytes[i - 1];
    if (dims[i] <= 1 && (st == 0 || st % 16 != 0)) st = 128;
    gstr[i - 1] = st;
  }
  CUresult r = enc(m, dt, rank, const_cast<void*>(base), gdim, gstr, bx, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FFPA_OK : FFPA_ERR_INVALID;
}

// Makes the device that owns `ptr` current for this library's runtime (the
// runtime is linked statically, so its current device is not the caller's),
// then requires compute capability 10.3 (sm_103).
ffpa_status check_device(const void* ptr, int* dev_out) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();
    return FFPA_ERR_CUDA;
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return FFPA_ERR_INVALID;
  const int dev = attr.device;
  if (cudaSetDevice(dev) != cudaSuccess) return FFPA_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FFPA_ERR_CUDA;
  if (major != 10 || minor != 3) return FFPA_ERR_UNSUPPORTED;
  *dev_out = dev;
  return FFPA_OK;
}

// Splits D into at most 256-column output slices, sizes the V stage, and
// decides whether Q stays resident in shared memory (D <= 512) and how many
// 32 KB ring slots fit beside it.  Returns the dynamic shared memory bytes.
size_t plan(int D, Params* P) {
  P->nchunks = D / DK;
  P->n_slices = (D + DV_MAX - 1) / DV_MAX;
  const int max_dv = ((P->nchunks + P->n_slices - 1) / P->n_slices) * DK;
  P->vchunks = max_dv / DK;
  P->kchunks = P->nchunks < 2 ? P->nchunks : 2;
  P->q_res = P->nchunks <= Q_RESIDENT_MAX_CHUNKS;
  const size_t q_region = P->q_res ? ((P->nchunks + 1) / 2) * (size_t)SLOT_BYTES : 0;
  const size_t budget = SMEM_LIMIT - SMEM_STATIC_RESERVE - 1024 - q_region;
  // V stages: up to 32 KB (vk keys x vchunks chunks of 128-byte rows), two
  // slots; halve vk while that leaves fewer than two K-ring slots.
  int vk = 128;
  while (vk > 16 && (size_t)vk * P->vchunks * 128 > SLOT_BYTES) vk >>= 1;
  P->nslot_v = NSLOT_V_MAX;
  while (vk > 32 && budget < 2 * (size_t)SLOT_BYTES + (size_t)NSLOT_V_MAX * vk * P->vchunks * 128)
    vk >>= 1;
  P->vk = vk;
  P->vslot = vk * P->vchunks * 128;
  size_t ns = (budget - (size_t)P->nslot_v * P->vslot) / SLOT_BYTES;
  if (ns > (size_t)NSLOT_MAX) ns = NSLOT_MAX;
  P->nslot = static_cast<int>(ns);
  return 1024 + q_region + ns * SLOT_BYTES + (size_t)P->nslot_v * P->vslot;
}

// The CTA-pair kernel needs every output slice to split into two halves of
// whole 64-column chunks, Q resident, and K stages of equal chunk count.
bool pair_eligible(int D) {
  const int nchunks = D / DK;
  if (nchunks > Q_RESIDENT_MAX_CHUNKS) return false;
  const int n_slices = (D + DV_MAX - 1) / DV_MAX;
  for (int sl = 0; sl < n_slices; ++sl) {
    const int w = (sl + 1) * nchunks / n_slices - sl * nchunks / n_slices;
    if (w % 2 != 0) return false;
  }
  const int kc = nchunks < 4 ? nchunks : 4;
  return nchunks % kc == 0;
}

enum class Kern { SINGLE, PAIR, SPLIT };

// The column-split kernel needs each CTA's half of the output columns to be
// whole 64-column chunks of at most 256 columns.
bool split_eligible(int D) { return D >= 128 && D % 128 == 0 && D / 2 <= DV_MAX; }

// Kernel choice, from measurements on GB300 (bf16): at D=512 the column-split
// kernel wins on dense, causal and varlen batches (it does not recompute S);
// at D=256 (no recompute anyway) the pair kernel wins on dense batches; at
// D=128 the single-CTA kernel's shorter per-tile chain wins, and on packed
// varlen batches of mixed lengths the 256-row pair tiles waste more rows on
// short sequences than they save.
Kern choose_kernel(int D, bool varlen) {
  const int v = g_variant.load();
  if (v == FFPA_VARIANT_SINGLE) return Kern::SINGLE;
  if (v == FFPA_VARIANT_PAIR) return pair_eligible(D) ? Kern::PAIR : Kern::SINGLE;
  if (v == FFPA_VARIANT_SPLIT) return split_eligible(D) ? Kern::SPLIT : Kern::SINGLE;
  if (D == 512) return Kern::SPLIT;
  if (!varlen && D == 256) return Kern::PAIR;
  return Kern::SINGLE;
}

// Column-split plan: Q chunks 0..3 in TMEM, the rest resident in shared
// memory, two P tiles, V stages of vk keys x D/2 columns, 32 KB ring slots.
size_t plan_split(int D, Params* P) {
  P->nchunks = D / DK;
  P->n_slices = 1;
  P->qt_chunks = P->nchunks < Q_TMEM_MAX_CHUNKS ? P->nchunks : Q_TMEM_MAX_CHUNKS;
  P->kchunks = 2;
  P->kc = 2;
  P->q_res = 1;
  P->vchunks = D / 2 / DK;
  int vk = 128;
  while (vk > 16 && (size_t)vk * P->vchunks * 128 > SLOT_BYTES) vk >>= 1;
  P->vk = vk;
  P->vslot = vk * P->vchunks * 128;
  P->nslot_v = 0;
  const size_t fixed = (size_t)(P->nchunks - P->qt_chunks) * CHUNK_BYTES + 2 * (size_t)P_TILE_BYTES;
  size_t ns = (SMEM_LIMIT - SPLIT_STATIC_RESERVE - 1024 - fixed) / SLOT_BYTES;
  if (ns > (size_t)NSLOT_MAX) ns = NSLOT_MAX;
  P->nslot = static_cast<int>(ns);
  return 1024 + fixed + ns * SLOT_BYTES;
}

// Pair-kernel plan: K stages of 64 keys x kc chunks, V stages of 128 keys x
// half the slice's columns, Q resident; returns the dynamic smem bytes.
size_t plan_pair(int D, Params* P) {
  plan(D, P);
  P->q_res = 1;
  P->kc = P->nchunks < 4 ? P->nchunks : 4;
  P->kslot = (BN / 2) * P->kc * 128;
  const int max_dv = P->vchunks * DK;
  P->vchunks = max_dv / 2 / DK;
  P->vk = BN;
  P->vslot = P->vk * P->vchunks * 128;
  const size_t q_region = ((P->nchunks + 1) / 2) * (size_t)SLOT_BYTES;
  const size_t budget = SMEM_LIMIT - SMEM_STATIC_RESERVE - 1024 - q_region;
  int nsv = NSLOT_V_MAX;
  if (budget < (size_t)nsv * P->vslot + 2 * (size_t)P->kslot) nsv = 1;
  size_t ns = (budget - (size_t)nsv * P->vslot) / P->kslot;
  if (ns > (size_t)NSLOT_MAX) ns = NSLOT_MAX;
  P->nslot = static_cast<int>(ns);
  P->nslot_v = nsv;
  return 1024 + q_region + ns * P->kslot + (size_t)nsv * P->vslot;
}

template <bool VARLEN>
ffpa_status launch_pair(const Params& P, int items, size_t smem, cudaStream_t stream) {
  auto kern = P.nchunks == 8   ? ffpa_fwd_pair_kernel<VARLEN, 8>
              : P.nchunks == 4 ? ffpa_fwd_pair_kernel<VARLEN, 4>
                               : ffpa_fwd_pair_kernel<VARLEN, 2>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(SMEM_LIMIT - SMEM_STATIC_RESERVE)) != cudaSuccess)
    return FFPA_ERR_CUDA;
  kern<<<2 * items, NTHREADS, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}

template <bool VARLEN>
ffpa_status launch_split(const Params& P, int items, size_t smem, cudaStream_t stream) {
  auto kern = P.nchunks == 8   ? ffpa_fwd_split_kernel<VARLEN, 8>
              : P.nchunks == 6 ? ffpa_fwd_split_kernel<VARLEN, 6>
              : P.nchunks == 4 ? ffpa_fwd_split_kernel<VARLEN, 4>
                               : ffpa_fwd_split_kernel<VARLEN, 2>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(SMEM_LIMIT - SPLIT_STATIC_RESERVE)) != cudaSuccess)
    return FFPA_ERR_CUDA;
  kern<<<2 * items, SPLIT_THREADS, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}

template <bool VARLEN>
ffpa_status launch_kernel(Kern kn, const Params& P, int items, size_t smem, cudaStream_t stream);

template <bool VARLEN>
ffpa_status launch(const Params& P, int items, size_t smem, cudaStream_t stream) {
  auto kern = ffpa_fwd_kernel<VARLEN>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(SMEM_LIMIT - SMEM_STATIC_RESERVE)) != cudaSuccess)
    return FFPA_ERR_CUDA;
  kern<<<items, NTHREADS, smem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}

template <bool VARLEN>
ffpa_status launch_kernel(Kern kn, const Params& P, int items, size_t smem, cudaStream_t stream) {
  if (kn == Kern::PAIR) return launch_pair<VARLEN>(P, items, smem, stream);
  if (kn == Kern::SPLIT) return launch_split<VARLEN>(P, items, smem, stream);
  return launch<VARLEN>(P, items, smem, stream);
}

size_t plan_for(Kern kn, int D, Params* P) {
  if (kn == Kern::PAIR) return plan_pair(D, P);
  if (kn == Kern::SPLIT) return plan_split(D, P);
  return plan(D, P);
}

}  // namespace

extern "C" {

const char* ffpa_status_string(ffpa_status s) {
  switch (s) {
    case FFPA_OK: return "FFPA_OK";
    case FFPA_ERR_DTYPE: return "FFPA_ERR_DTYPE: inputs must be bf16 or fp16";
    case FFPA_ERR_INVALID: return "FFPA_ERR_INVALID: invalid shape, stride, pointer or option";
    case FFPA_ERR_UNSUPPORTED: return "FFPA_ERR_UNSUPPORTED: head dim or device not supported";
    case FFPA_ERR_CUDA: return "FFPA_ERR_CUDA: a CUDA runtime call failed";
    case FFPA_ERR_DEVICE_TIMEOUT: return "FFPA_ERR_DEVICE_TIMEOUT: a kernel wait ran out of time";
  }
  return "FFPA: unknown status";
}

void ffpa_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 2000000000ull); }

void ffpa_test_drop_first_copy(int enable) { g_drop_first_copy.store(enable ? 1 : 0); }

void ffpa_set_kernel_variant(int variant) {
  if (variant >= FFPA_VARIANT_AUTO && variant <= FFPA_VARIANT_SPLIT) g_variant.store(variant);
}

int ffpa_selected_kernel(int D, int varlen) {
  if (D < 64 || D > 1024 || D % 64 != 0) return -1;
  const Kern kn = choose_kernel(D, varlen != 0);
  return kn == Kern::PAIR ? FFPA_VARIANT_PAIR : kn == Kern::SPLIT ? FFPA_VARIANT_SPLIT : FFPA_VARIANT_SINGLE;
}

ffpa_status ffpa_last_device_error(ffpa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FFPA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, ffpa::g_err_word, sizeof(int)) != cudaSuccess) return FFPA_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(ffpa::g_err_word, &zero, sizeof(int)) != cudaSuccess) return FFPA_ERR_CUDA;
    return static_cast<ffpa_status>(word);
  }
  return FFPA_OK;
}

ffpa_status ffpa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                     const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                     const int64_t o_str[4], const void* mask, ffpa_mask_kind mask_kind,
                     const int64_t mask_str[4], const float* scale, int is_causal, int enable_gqa,
                     ffpa_stream_t stream) {
  if (dt != FFPA_BF16 && dt != FFPA_FP16) return FFPA_ERR_DTYPE;
  if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nkv < 0) return FFPA_ERR_INVALID;
  if (D < 64 || D > 1024 || D % 64 != 0) return FFPA_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return FFPA_ERR_INVALID;
  if (Hq != Hkv && !enable_gqa) return FFPA_ERR_INVALID;
  if (is_causal && Nkv < Nq) return FFPA_ERR_INVALID;
  if (mask_kind < FFPA_MASK_NONE || mask_kind > FFPA_MASK_ADD_QTYPE) return FFPA_ERR_INVALID;
  const float sc = scale ? *scale : 1.0f / std::sqrt(static_cast<float>(D));
  if (!std::isfinite(sc)) return FFPA_ERR_INVALID;
  if (B == 0 || Nq == 0) return FFPA_OK;          // nothing to read or write
  if (!q || !o || !q_str || !k_str || !v_str || !o_str) return FFPA_ERR_INVALID;
  if (Nkv > 0 && (!k || !v)) return FFPA_ERR_INVALID;
  if (mask_kind != FFPA_MASK_NONE && Nkv > 0) {
    if (!mask || !mask_str) return FFPA_ERR_INVALID;
    for (int i = 0; i < 4; ++i)
      if (mask_str[i] < 0) return FFPA_ERR_INVALID;
  }
  const int64_t qsz[4] = {B, Hq, Nq, D}, ksz[4] = {B, Hkv, Nkv, D};
  if (!strides_ok(q_str, qsz, 4) || !strides_ok(o_str, qsz, 4)) return FFPA_ERR_INVALID;
  if (Nkv > 0 && (!strides_ok(k_str, ksz, 4) || !strides_ok(v_str, ksz, 4))) return FFPA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(o) || (Nkv > 0 && (!aligned16(k) || !aligned16(v))))
    return FFPA_ERR_INVALID;
  int dev = 0;
  ffpa_status st = check_device(q, &dev);
  if (st != FFPA_OK) return st;

  Params P{};
  const CUtensorMapDataType tdt =
      dt == FFPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const Kern kn = choose_kernel(D, false);
  const bool pair = kn == Kern::PAIR;
  const size_t smem = plan_for(kn, D, &P);
  const uint32_t k_rows = pair ? BN / 2 : BN;
  const uint32_t k_box_chunks = pair ? (uint32_t)P.kc : (uint32_t)P.kchunks;
  const uint64_t nch = (uint64_t)P.nchunks;
  {
    const uint64_t dq[5] = {64, (uint64_t)Nq, nch, (uint64_t)Hq, (uint64_t)B};
    const uint64_t sq[4] = {(uint64_t)q_str[2] * 2, 128, (uint64_t)q_str[1] * 2, (uint64_t)q_str[0] * 2};
    const uint32_t bq[5] = {64, BM, (uint32_t)P.kchunks, 1, 1};
    if ((st = encode_map(&P.tm_q, tdt, 5, q, dq, sq, bq)) != FFPA_OK) return st;
  }
  if (Nkv > 0) {   // with no keys no work item issues a copy; the maps stay unused
    const uint64_t dk[5] = {64, (uint64_t)Nkv, nch, (uint64_t)Hkv, (uint64_t)B};
    const uint64_t sk[4] = {(uint64_t)k_str[2] * 2, 128, (uint64_t)k_str[1] * 2, (uint64_t)k_str[0] * 2};
    const uint32_t bk[5] = {64, k_rows, k_box_chunks, 1, 1};
    if ((st = encode_map(&P.tm_k, tdt, 5, k, dk, sk, bk)) != FFPA_OK) return st;
    const uint64_t sv[4] = {(uint64_t)v_str[2] * 2, 128, (uint64_t)v_str[1] * 2, (uint64_t)v_str[0] * 2};
    const uint32_t bv[5] = {64, (uint32_t)P.vk, (uint32_t)P.vchunks, 1, 1};
    if ((st = encode_map(&P.tm_v, tdt, 5, v, dk, sv, bv)) != FFPA_OK) return st;
  }
  P.o = o;
  P.lse = lse;
  P.mask = mask_kind != FFPA_MASK_NONE ? mask : nullptr;
  P.mask_kind = mask_kind;
  for (int i = 0; i < 4; ++i) {
    P.o_str[i] = o_str[i];
    P.m_str[i] = mask_kind != FFPA_MASK_NONE ? mask_str[i] : 0;
  }
  P.B = B;
  P.Hq = Hq;
  P.group = Hq / Hkv;
  P.Nq = Nq;
  P.Nkv = Nkv;
  P.D = D;
  P.Tq = 0;
  const int q_tile = pair ? BM_PAIR : BM;
  P.n_qt = (Nq + q_tile - 1) / q_tile;
  P.scale_log2 = sc * 1.4426950408889634f;
  P.causal = is_causal ? 1 : 0;
  P.fp16 = dt == FFPA_FP16;
  P.inject = g_drop_first_copy.load();
  P.timeout_ns = g_timeout_ns.load();
  const long long items = (long long)B * Hq * P.n_qt * P.n_slices;
  if (items > 0x7fffffffLL) return FFPA_ERR_INVALID;
  return launch_kernel<false>(kn, P, static_cast<int>(items), smem,
                              reinterpret_cast<cudaStream_t>(stream));
}

ffpa_status ffpa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                            const int64_t q_str[3], const int64_t k_str[3],
                            const int64_t v_str[3], const int64_t o_str[3],
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                            int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                            int enable_gqa, ffpa_stream_t stream) {
  if (dt != FFPA_BF16 && dt != FFPA_FP16) return FFPA_ERR_DTYPE;
  if (Tq < 0 || Tk < 0 || Hq < 1 || Hkv < 1) return FFPA_ERR_INVALID;
  if (D < 64 || D > 1024 || D % 64 != 0) return FFPA_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return FFPA_ERR_INVALID;
  if (Hq != Hkv && !enable_gqa) return FFPA_ERR_INVALID;
  if (nseq < 1 || max_seqlen_q < 0 || max_seqlen_k < 0) return FFPA_ERR_INVALID;
  if (!cu_seqlens_q) return FFPA_ERR_INVALID;
  const float sc = scale ? *scale : 1.0f / std::sqrt(static_cast<float>(D));
  if (!std::isfinite(sc)) return FFPA_ERR_INVALID;
  if (Tq == 0 || max_seqlen_q == 0) return FFPA_OK;   // nothing to read or write
  if (!q || !o || !q_str || !k_str || !v_str || !o_str) return FFPA_ERR_INVALID;
  if (Tk > 0 && (!k || !v)) return FFPA_ERR_INVALID;
  const int64_t qsz[3] = {Tq, Hq, D}, ksz[3] = {Tk, Hkv, D};
  if (!strides_ok(q_str, qsz, 3) || !strides_ok(o_str, qsz, 3)) return FFPA_ERR_INVALID;
  if (Tk > 0 && (!strides_ok(k_str, ksz, 3) || !strides_ok(v_str, ksz, 3))) return FFPA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(o) || (Tk > 0 && (!aligned16(k) || !aligned16(v))))
    return FFPA_ERR_INVALID;
  int dev = 0;
  ffpa_status st = check_device(q, &dev);
  if (st != FFPA_OK) return st;

  Params P{};
  const CUtensorMapDataType tdt =
      dt == FFPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const Kern kn = choose_kernel(D, true);
  const bool pair = kn == Kern::PAIR;
  const size_t smem = plan_for(kn, D, &P);
  const uint32_t k_rows = pair ? BN / 2 : BN;
  const uint32_t k_box_chunks = pair ? (uint32_t)P.kc : (uint32_t)P.kchunks;
  const uint64_t nch = (uint64_t)P.nchunks;
  {
    const uint64_t dq[4] = {64, (uint64_t)Tq, nch, (uint64_t)Hq};
    const uint64_t sq[3] = {(uint64_t)q_str[0] * 2, 128, (uint64_t)q_str[1] * 2};
    const uint32_t bq[4] = {64, BM, (uint32_t)P.kchunks, 1};
    if ((st = encode_map(&P.tm_q, tdt, 4, q, dq, sq, bq)) != FFPA_OK) return st;
  }
  if (Tk > 0) {
    const uint64_t dk[4] = {64, (uint64_t)Tk, nch, (uint64_t)Hkv};
    const uint64_t sk[3] = {(uint64_t)k_str[0] * 2, 128, (uint64_t)k_str[1] * 2};
    const uint32_t bk[4] = {64, k_rows, k_box_chunks, 1};
    if ((st = encode_map(&P.tm_k, tdt, 4, k, dk, sk, bk)) != FFPA_OK) return st;
    const uint64_t sv[3] = {(uint64_t)v_str[0] * 2, 128, (uint64_t)v_str[1] * 2};
    const uint32_t bv[4] = {64, (uint32_t)P.vk, (uint32_t)P.vchunks, 1};
    if ((st = encode_map(&P.tm_v, tdt, 4, v, dk, sv, bv)) != FFPA_OK) return st;
  }
  P.o = o;
  P.lse = lse;
  P.mask = nullptr;
  P.mask_kind = FFPA_MASK_NONE;
  P.o_str[0] = o_str[0];
  P.o_str[1] = o_str[1];
  P.o_str[2] = o_str[2];
  P.cu_q = cu_seqlens_q;
  P.cu_k = cu_seqlens_k ? cu_seqlens_k : cu_seqlens_q;
  P.B = nseq;
  P.Hq = Hq;
  P.group = Hq / Hkv;
  P.Nq = 0;
  P.Nkv = 0;
  P.D = D;
  P.Tq = Tq;
  const int q_tile = pair ? BM_PAIR : BM;
  P.n_qt = (max_seqlen_q + q_tile - 1) / q_tile;
  P.scale_log2 = sc * 1.4426950408889634f;
  P.causal = causal ? 1 : 0;
  P.fp16 = dt == FFPA_FP16;
  P.inject = g_drop_first_copy.load();
  P.timeout_ns = g_timeout_ns.load();
  (void)max_seqlen_k;
  const long long items = (long long)nseq * Hq * P.n_qt * P.n_slices;
  if (items > 0x7fffffffLL) return FFPA_ERR_INVALID;
  return launch_kernel<true>(kn, P, static_cast<int>(items), smem,
                              reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
