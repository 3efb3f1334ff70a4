#pragma once
// Device helpers shared by the two backward translation units: the sliced
// kernels (ffpa_bwd.cu) and the stored-tile kernels (ffpa_bwd_tiles.cu).
#include "ffpa_common.cuh"

namespace ffpa {
namespace bwd {

constexpr int BWD_ROLE_DQ = 0;   // rows = queries: dQ
constexpr int BWD_ROLE_DV = 1;   // rows = keys: dV (P only)
constexpr int BWD_ROLE_DK = 2;   // rows = keys: dK
constexpr int BWD_ROLE_DKDV = 3; // rows = keys: dV and dK together (D <= 128)
constexpr uint32_t BWD_S_COL = 256;
constexpr uint32_t BWD_DP_COL = 384;
constexpr int BWD_PRODUCER_WARP = 4;
constexpr int BWD_MMA_WARP = 5;
constexpr float LOG2E_F = 1.4426950408889634f;

// Dot product of 8 16-bit pairs held in two uint4.
__device__ __forceinline__ float dot8(uint4 a, uint4 b, bool fp16) {
  const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
  const uint32_t wb[4] = {b.x, b.y, b.z, b.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a0, a1, b0, b1;
    if (fp16) {
      const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&wa[i]));
      const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&wb[i]));
      a0 = fa.x; a1 = fa.y; b0 = fb.x; b1 = fb.y;
    } else {
      a0 = __uint_as_float(wa[i] << 16);
      a1 = __uint_as_float(wa[i] & 0xffff0000u);
      b0 = __uint_as_float(wb[i] << 16);
      b1 = __uint_as_float(wb[i] & 0xffff0000u);
    }
    s = fmaf(a0, b0, s);
    s = fmaf(a1, b1, s);
  }
  return s;
}

struct BwdItem {
  int b, hq, hkv, slice;
  int q_len, kv_len;       // this problem's (sequence's) lengths
  int q_row0, kv_row0;     // varlen: first packed row of the sequence (dense: 0)
  int row0;       // first row of this CTA's tile: query row (dQ) or key row (key-row roles)
  int n_iter;     // dQ: key tiles; key-row roles (dV, dK, dK/dV): group heads x visible query tiles
  int qt_first;   // key-row roles: first query tile that sees the key tile
  int nq;         // key-row roles: query tiles per head
  int col_lo, dv; // output columns [col_lo, col_lo + dv)
};

// Lengths and packed row offsets of item it's problem (sequence it.b when
// varlen).
__device__ __forceinline__ void bwd_lengths(const BwdParams& p, BwdItem& it) {
  if (p.varlen) {
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
}

// Index of (query head h, query row i of the item's problem) in the LSE and
// delta arrays: dense [B, Hq, Nq], varlen [Hq, Tq].
__device__ __forceinline__ long long bwd_stat_index(const BwdParams& p, const BwdItem& it, int h, int i) {
  return p.varlen ? (long long)h * p.Tq + it.q_row0 + i : ((long long)it.b * p.Hq + h) * p.Nq + i;
}

// Element offset of row `row` of head h in an output tensor with strides
// str: dense (b, h, n, d), varlen (t, h, d).
__device__ __forceinline__ long long bwd_row_offset(const BwdParams& p, const BwdItem& it, const int64_t* str,
                                                    int row0, int row, int h) {
  return p.varlen ? (long long)(row0 + row) * str[0] + (long long)h * str[1]
                  : (long long)it.b * str[0] + (long long)h * str[1] + (long long)row * str[2];
}

template <bool DQ>
__device__ __forceinline__ bool bwd_decode(const BwdParams& p, int L, BwdItem& it) {
  if (DQ) {
    it.slice = L % p.n_sl;
    L /= p.n_sl;
    const int heads = p.B * p.Hq;
    int qt, bh;
    if (p.causal) {            // longest query tiles (most visible keys) first
      bh = L % heads;
      qt = p.n_qt - 1 - L / heads;
    } else {
      qt = L % p.n_qt;
      bh = L / p.n_qt;
    }
    it.hq = bh % p.Hq;
    it.b = bh / p.Hq;
    it.hkv = it.hq / p.group;
    bwd_lengths(p, it);
    it.row0 = qt * BM;
    if (it.row0 >= it.q_len) return false;
    long long kv_end = it.kv_len;
    if (p.causal) {
      const int rows = min(BM, it.q_len - it.row0);
      kv_end = min(kv_end, (long long)it.row0 + rows + (it.kv_len - it.q_len));
    }
    it.n_iter = kv_end > 0 ? (int)((kv_end + BN - 1) / BN) : 0;
    it.qt_first = 0;
    it.nq = 0;
    it.col_lo = it.slice * BWD_OUT_COLS;
    it.dv = min(BWD_OUT_COLS, p.D - it.col_lo);
  } else {
    it.slice = L % p.n_sl;
    L /= p.n_sl;
    const int heads = p.B * p.Hkv;
    int kt, bh;
    if (p.causal) {            // key tile 0 is seen by every query tile: first
      bh = L % heads;
      kt = L / heads;
    } else {
      kt = L % p.n_kt;
      bh = L / p.n_kt;
    }
    it.hkv = bh % p.Hkv;
    it.b = bh / p.Hkv;
    it.hq = it.hkv * p.group;
    bwd_lengths(p, it);
    it.row0 = kt * BN;
    if (it.row0 >= it.kv_len) return false;
    // Query row i sees key k when k <= i + (Nkv - Nq): the first query
    // tile with a row that sees this tile's first key.
    const int first_row = p.causal ? max(0, it.row0 - (it.kv_len - it.q_len)) : 0;
    it.qt_first = first_row / BM;
    it.nq = max(0, (it.q_len + BM - 1) / BM - it.qt_first);
    it.n_iter = p.group * it.nq;
    it.col_lo = it.slice * BWD_OUT_COLS;
    it.dv = min(BWD_OUT_COLS, p.D - it.col_lo);
  }
  return true;
}

// Rows of a TMEM accumulator (columns [tcol, tcol + ncols) of this thread's
// lane) times `mul`, rounded to 16 bits and stored at dst (nullptr: row out
// of range).  have == false stores zeros.
__device__ __forceinline__ void bwd_store_row(uint32_t taddr, int ncols, float mul, uint8_t* dst,
                                              bool fp16, bool have) {
  for (int c0 = 0; c0 < ncols; c0 += 32) {
    uint32_t v[32];
    if (have) {
      tmem_ld32(taddr + c0, v);
      tmem_wait_ld();
      reg_fence(v);
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) v[c] = 0u;
    }
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float a0 = __uint_as_float(v[2 * c]) * mul;
      const float a1 = __uint_as_float(v[2 * c + 1]) * mul;
      pk[c] = fp16 ? pack_f16(a0, a1) : pack_bf16(a0, a1);
    }
    if (dst != nullptr) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + c0 * 2);
#pragma unroll
      for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
  }
}

// Writes 128 16-bit values (64 packed pairs) of row r into a 128 x 128
// K-major tile with 128-byte swizzle: two 16 KB chunks of 64 columns, 16-byte
// unit u of row r at unit u ^ (r & 7).
__device__ __forceinline__ void bwd_write_tile_row(uint32_t tile, int r, const uint32_t* pk) {
  const uint32_t row = tile + (uint32_t)r * 128u;
  const uint32_t sw = (uint32_t)(r & 7);
#pragma unroll
  for (int g = 0; g < BN / 8; ++g)
    st_shared_v4(row + (g >> 3) * CHUNK_BYTES + ((((uint32_t)g & 7u) ^ sw) << 4), pk[4 * g],
                 pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
}

// The caller's mask term for one score, in the log2 domain: the bool mask
// turns the exponent argument into -inf where false; an additive mask adds
// its value times log2(e).  off is the element offset from base.
__device__ __forceinline__ float add_mask_term(float arg, const uint8_t* base, long long off, int kind,
                                               bool fp16) {
  if (kind == FFPA_MASK_BOOL) return base[off] != 0 ? arg : -INFINITY;
  if (kind == FFPA_MASK_ADD_F32) return arg + __ldg(reinterpret_cast<const float*>(base) + off) * LOG2E_F;
  const uint16_t h = __ldg(reinterpret_cast<const unsigned short*>(base) + off);
  const float hv = fp16 ? __half2float(__ushort_as_half(h)) : __bfloat162float(__ushort_as_bfloat16(h));
  return arg + hv * LOG2E_F;
}

}  // namespace bwd
}  // namespace ffpa
