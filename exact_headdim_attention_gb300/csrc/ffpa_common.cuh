#pragma once
// Exact attention forward for large head dimensions on GB300 (sm_103a):
// device code shared by the three kernels (single-CTA, CTA pair, column
// split), one translation unit each.
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

#include <cmath>
#include <cstdint>

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

// CTA-pair kernel: a 256-row query tile per pair, 64 keys of each K tile per CTA.
constexpr int BM_PAIR = 256;
constexpr int KEYS_PER_CTA = BN / 2;

// Column-split kernel (see ffpa_split.cu).
constexpr int SPLIT_THREADS = 192;
constexpr uint32_t Q_TMEM_COL = 384;
constexpr int Q_TMEM_MAX_CHUNKS = 4;
constexpr uint32_t P_TILE_BYTES = BM * BN * 2;   // 2 x (128 rows x 64 keys), 16-bit
constexpr size_t SPLIT_STATIC_RESERVE = 2048;    // static shared memory of the column-split kernel

// ------------------------------------------------------------------ host
// Launches of the forward kernels (one translation unit each; the column
// split has a pair kernel and a kernel for clusters of 3 or 4 CTAs).
struct Params;
ffpa_status launch_single(bool varlen, bool umask, const Params& P, int items, size_t smem, cudaStream_t stream);
ffpa_status launch_pair(bool varlen, bool umask, const Params& P, int items, size_t smem, cudaStream_t stream);
ffpa_status launch_split(bool varlen, bool umask, const Params& P, int items, size_t smem, cudaStream_t stream);
ffpa_status launch_cluster(bool varlen, bool umask, const Params& P, int items, size_t smem, cudaStream_t stream);
// Two 128-row query tiles per CTA sharing every K/V tile (ffpa_dual.cu; dense, D = 64, 128).
ffpa_status launch_dual(bool umask, const Params& P, int items, size_t smem, cudaStream_t stream);
// FP8 forward: the quantisation of Q, K, V into the workspace, then the
// e4m3 attention kernel (ffpa_fp8.cu).
struct Fp8Quant {
  const void* src[3];                          // q, k, v (16-bit)
  int64_t str[3][4];                           // element strides (b, h, n, d)
  uint8_t* codes[3];                           // q8, k8 [B,H,Npad,D]; v8t [B,H,D,Npad]
  float* scales[3];                            // [B, H, Npad / 128]
  int H[3], N[3], npad[3], nblk[3];
  long long cta_end[3];                        // cumulative CTA counts of q, k, v
  int B, D, fp16;
};
ffpa_status launch_fp8(const Fp8Quant& Qz, const Params& P, int items, size_t smem, bool split,
                       cudaStream_t stream);
// The FP8 attention on the column split (ffpa_fp8_split.cu; D = 256, 384, 512).
ffpa_status launch_fp8_split(const Params& P, int items, size_t smem, cudaStream_t stream);
// Raises kernel `fn`'s dynamic shared-memory limit to `bytes` on `device`,
// once per (kernel, device) pair; later calls only look the pair up.
ffpa_status set_smem_attr_once(const void* fn, int device, int bytes);

// Binds the primary context of `dev` to the calling thread for the lifetime
// of the object (tensor-map encoding, symbol lookups and launches need a
// current context; a framework's worker thread may have none), and puts the
// thread's previous driver context back afterwards (none, if it had none),
// so that a call leaves the caller's thread as it found it.
class DeviceScope {
 public:
  explicit DeviceScope(int dev);
  ~DeviceScope();
  bool ok() const { return ok_; }
  DeviceScope(const DeviceScope&) = delete;
  DeviceScope& operator=(const DeviceScope&) = delete;

 private:
  CUcontext saved_ = nullptr;
  bool restore_ = false;
  bool ok_ = false;
};

// Backward (ffpa_bwd.cu): a delta pass, then one kernel for dQ (rows =
// queries) and one each for dV and dK (rows = keys; one for both when
// D <= 128).
struct BwdParams;
ffpa_status launch_bwd(const BwdParams& P, int dq_items, int kv_items, size_t smem, size_t smem_two,
                       cudaStream_t stream);
// The delta pass alone (rowsum(dO * O) into P.delta).
ffpa_status launch_bwd_delta(const BwdParams& P, cudaStream_t stream);
// Stored-tile backward (ffpa_bwd_tiles.cu): the delta pass, the scores
// kernel (P and dS once per query tile x key tile into the caller's
// workspace) and the contraction kernel (dQ, dV and dK from the stored
// tiles).  D / 64 in {2, 4, 6, 8}.
ffpa_status launch_bwd_tiles(const BwdParams& P, int score_items, int contract_items, size_t smem_scores,
                             size_t smem_contract, cudaStream_t stream);
// Varlen: the first stored block of every sequence (P.ws_base), from
// cu_seqlens on the device.
ffpa_status launch_bwd_tiles_bases(const BwdParams& P, cudaStream_t stream);
constexpr int TS_THREADS = 320;            // scores: warps 0-7 elementwise, 8 TMA, 9 MMA
constexpr int TC_THREADS = 192;            // contraction: warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr int TS_NSLOT_MAX = 6;
constexpr int TC_NSLOT_MAX = 7;
constexpr size_t TS_STATIC_RESERVE = 1024;
constexpr size_t TC_STATIC_RESERVE = 1024;
constexpr int BWD_THREADS = 192;           // warps 0-3 elementwise, 4 TMA, 5 MMA
constexpr int BWD_NSLOT_MAX = 6;
constexpr size_t BWD_STATIC_RESERVE = 6144;
constexpr int BWD_OUT_COLS = 256;          // dQ, dV or dK columns per CTA

// Stored-tile backward: key tiles kept for query tile qt (those its rows
// see: every key tile, or under causal masking, lower right, the tiles up to
// its last row's limit), and the blocks of query tiles 0 .. qt-1 of one head
// in closed form: a full query tile t keeps clamp(t + 1 + c, 0, n_kt) tiles
// with c = ceil((Nkv - Nq) / 128), the last one its own count.
__host__ __device__ inline int bwd_stored_tiles(int qt, int Nq, int Nkv, int causal) {
  if (Nq <= 0 || Nkv <= 0) return 0;
  const int n_kt = (Nkv + BN - 1) / BN;
  if (!causal) return n_kt;
  const int rows_end = (qt + 1) * BM < Nq ? (qt + 1) * BM : Nq;
  const long long kv_end0 = (long long)rows_end + (Nkv - Nq);
  const long long kv_end = kv_end0 < Nkv ? kv_end0 : Nkv;
  return kv_end > 0 ? (int)((kv_end + BN - 1) / BN) : 0;
}
__host__ __device__ inline long long bwd_stored_before(int qt, int Nq, int Nkv, int causal) {
  if (Nq <= 0 || Nkv <= 0) return 0;
  const long long n_kt = (Nkv + BN - 1) / BN, n_qt = (Nq + BM - 1) / BM;
  if (!causal) return (long long)qt * n_kt;
  if (n_qt == 0) return 0;
  const long long off = (long long)Nkv - Nq;
  const long long c = off >= 0 ? (off + BN - 1) / BN : -((-off) / BN);
  const long long full = (long long)qt < n_qt - 1 ? qt : n_qt - 1;   // full query tiles below qt
  const long long lo = c < 0 ? -c : 0;                              // first t keeping a tile
  const long long hi = n_kt - c;                                    // t < hi: below the cap
  const long long a0 = full < lo ? full : lo;
  const long long lin_end = full < hi ? full : hi;
  const long long a1 = lin_end > lo ? lin_end - lo : 0;
  const long long a2 = full - a0 - a1;
  long long s = a1 * (lo + 1 + c) + a1 * (a1 - 1) / 2 + a2 * n_kt;
  if ((long long)qt > n_qt - 1) s += bwd_stored_tiles((int)(n_qt - 1), Nq, Nkv, causal);
  return s;
}

struct BwdParams {
  // Views (64, N, D/64, H, B) of Q, K, V and dO; box 64 x 128 rows x kchunks.
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  // dQ, dK, dV with box 64 x 32 rows (the stored-tile contraction's output
  // stores, dense layout).
  CUtensorMap tm_dq;
  CUtensorMap tm_dk;
  CUtensorMap tm_dv;
  const void* o;
  const void* dout;
  const float* lse;
  float* delta;
  void* dq;
  void* dk;
  void* dv;
  int64_t o_str[4], do_str[4], dq_str[4], dk_str[4], dv_str[4];
  const void* mask;     // broadcast to [B, Hq, Nq, Nkv] by m_str (0 on broadcast dims)
  int64_t m_str[4];
  int mask_kind;
  // Packed variable-length input (varlen = 1): B sequences, rows of sequence
  // s at cu_q[s].. / cu_k[s].. of [T, H, D] tensors; LSE and delta [Hq, Tq];
  // Nq / Nkv are then the maximum sequence lengths.
  int varlen, Tq;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int B, Hq, Hkv, group, Nq, Nkv, D;
  int nchunks, npairs, kchunks;
  int n_qt, n_kt, n_sl;   // query tiles, key tiles, 256-column output slices
  int nslot;              // ring depth (one tile)
  int kv_together;        // D <= 128: one dK/dV kernel (two tiles, ring depth nslot_two)
  int nslot_two;
  float scale, scale_log2;
  int causal, fp16, inject;
  unsigned long long timeout_ns;
  int* err;     // device status word of this call (set to FFPA_ERR_DEVICE_TIMEOUT on expiry)
  int device;   // host only: the device the launch goes to
  // Stored-tile backward: P and dS (dS times the softmax scale), 16-bit, one
  // 32 KB block per (b, hq, query tile, stored key tile) in the caller's
  // workspace: block (b Hq + hq) ws_head + bwd_stored_before(qt) + kt; inside
  // a block the 16-byte unit of 8 keys (8u .. 8u+7) of row r sits at byte
  // 2048 u + 16 r (the tensor core's layout without swizzle).  ws_zero: one
  // block of zeros.
  void* ws_zero;
  void* ws_p;
  void* ws_ds;
  long long ws_head;          // dense: stored blocks per head
  const long long* ws_base;   // varlen: first block of sequence s (device, nseq + 1 entries)
  long long ws_blocks;        // blocks the workspace holds for P (and for dS)
  int kv_parts;      // scores kernel: key-tile ranges per query tile
  int ts_nslot;      // scores kernel: ring depth
  int tc_nslot;      // contraction kernel: ring depth
  int n_dq_items, n_kv_items;   // contraction kernel: dQ items, and dV (= dK) items
};

struct Params {
  // Views with D split as (64, D/64): dense (64, N, D/64, H, B); varlen
  // (64, T, D/64, H).  Q and K boxes: 64 x 128 rows x min(2, D/64) chunks;
  // V box: 64 x vk rows x vchunks chunks.
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  // O with box 64 x 32 rows: the column-split kernel's output stores (dense
  // layout; o_tma = 1 when encoded).
  CUtensorMap tm_o;
  int o_tma;
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
  int split_c;         // column-split kernel: CTAs per cluster (output columns D / split_c each)
  float scale_log2;
  int causal, fp16, inject;
  // Dense head dims that are not a multiple of 64 (D % 8 == 0): the maps
  // are 4-D (D, N, H, B) with one 64-column box per chunk, so columns >= D
  // arrive as zeros (single-CTA kernel only).
  int dfine;
  unsigned long long timeout_ns;
  int* err;     // device status word of this call (set to FFPA_ERR_DEVICE_TIMEOUT on expiry)
  int device;   // host only: the device the launch goes to
  // FP8 forward: e4m3 block scales (per batch, head, 128-row block) of Q, K
  // and V in the caller's workspace; n_kb key blocks per head.
  const float* sq;
  const float* sk;
  const float* sv;
  int n_kb;
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
  // Dense causal items all start at key tile 0 (measured on GB300, causal
  // GQA D=512: 1032 vs 921 TFLOPS); otherwise the start is spread (non-causal
  // D=512: 1164 vs 1132; varlen: 676 vs 650).
  it.rot = (it.ntiles > 0 && !(p.causal && !varlen))
               ? (int)(((unsigned)qt * 37u + (unsigned)it.slice * 17u + (unsigned)it.hq * 13u) %
                       (unsigned)it.ntiles)
               : 0;
  const int c_lo = it.slice * p.nchunks / p.n_slices;
  const int c_hi = (it.slice + 1) * p.nchunks / p.n_slices;
  it.col_lo = c_lo * DK;
  it.dv = (c_hi - c_lo) * DK;
  return true;
}

// Bounded wait on an mbarrier phase.  Returns false when this CTA has been
// told to abort or when the limit expires (then the call's status word *err
// is set).  `cluster` selects cluster-scope acquire, for phases that another
// CTA of the cluster completes.  The inline body serves kernels that change
// their register budget per warpgroup (an out-of-line function cannot be
// compiled for two budgets); the others call the out-of-line copy.
static __device__ __forceinline__ bool wait_bounded_inl(uint32_t bar, uint32_t parity,
                                                        volatile int* abort_flag,
                                                        unsigned long long timeout_ns, int* err,
                                                        bool cluster = false) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    // try_wait without a suspend-time hint (the instruction still waits a
    // hardware-chosen while before it reports an incomplete phase): the
    // waiting warp resumes sooner after the phase completes than a suspended
    // one (measured on GB300: D=512 forward 1173 -> 1204 TFLOPS, causal GQA
    // 1063 -> 1075, backward 1.315 -> 1.309 ms).
    if (cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity))
      return true;
    if ((it & 7u) == 7u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        atomicExch(err, (int)FFPA_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

static __device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                 unsigned long long timeout_ns, int* err,
                                                 bool cluster = false) {
  return wait_bounded_inl(bar, parity, abort_flag, timeout_ns, err, cluster);
}

// Drain wait used on the way out: ignores the abort flag.
static __device__ __forceinline__ void wait_drain_inl(uint32_t bar, uint32_t parity,
                                                      unsigned long long timeout_ns, int* err) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) {
      atomicExch(err, (int)FFPA_ERR_DEVICE_TIMEOUT);
      return;
    }
  }
}

static __device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, unsigned long long timeout_ns,
                                               int* err) {
  wait_drain_inl(bar, parity, timeout_ns, err);
}

// Masks 32 consecutive scores (log2 domain) of one row: keys past the end,
// keys beyond the causal limit, and (UMASK) the caller's bool/additive mask.
// Kernels launched without a mask are instantiated with UMASK = false and
// carry none of the mask-loading code.  With a mask, 32 entries that are
// contiguous, in range and 16-byte aligned are read with 16-byte loads (8
// for fp32, 4 for 16-bit, 2 for bool); otherwise entry by entry, only for
// keys that are still visible.
template <bool UMASK>
__device__ __forceinline__ void apply_mask32(float* x, int key0, int kv_len, bool causal,
                                             long long row_limit, const uint8_t* mrow,
                                             long long mk, int mask_kind, bool fp16) {
  const float LOG2E = 1.4426950408889634f;
  if (UMASK && mrow != nullptr && mk == 1 && key0 + 32 <= kv_len) {
    const int esz = mask_kind == FFPA_MASK_BOOL ? 1 : mask_kind == FFPA_MASK_ADD_F32 ? 4 : 2;
    const uint8_t* mp = mrow + (long long)key0 * esz;
    if ((reinterpret_cast<uintptr_t>(mp) & 15u) == 0) {
      const uint4* m4 = reinterpret_cast<const uint4*>(mp);
      if (mask_kind == FFPA_MASK_ADD_F32) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 w = __ldg(m4 + v);
          x[4 * v] += __uint_as_float(w.x) * LOG2E;
          x[4 * v + 1] += __uint_as_float(w.y) * LOG2E;
          x[4 * v + 2] += __uint_as_float(w.z) * LOG2E;
          x[4 * v + 3] += __uint_as_float(w.w) * LOG2E;
        }
      } else if (mask_kind == FFPA_MASK_BOOL) {
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          const uint4 w = __ldg(m4 + v);
          const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int b = 0; b < 16; ++b)
            if (((wd[b >> 2] >> (8 * (b & 3))) & 0xffu) == 0u) x[16 * v + b] = -INFINITY;
        }
      } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 w = __ldg(m4 + v);
          const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const uint16_t hbits = (uint16_t)(wd[b >> 1] >> (16 * (b & 1)));
            const float hv = fp16 ? __half2float(__ushort_as_half(hbits))
                                  : __bfloat162float(__ushort_as_bfloat16(hbits));
            x[8 * v + b] += hv * LOG2E;
          }
        }
      }
      if (causal) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if ((long long)(key0 + c) > row_limit) x[c] = -INFINITY;
      }
      return;
    }
  }
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const int key = key0 + c;
    bool vis = key < kv_len && (!causal || (long long)key <= row_limit);
    float add = 0.f;
    if (UMASK && vis && mrow != nullptr) {
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
// o_scale multiplies the accumulator on top of 1/l (the FP8 kernel's P
// carries a per-tile factor; 1 elsewhere).
template <bool VARLEN>
__device__ __forceinline__ void store_output(const Params& p, const Item& it, bool have_o,
                                             uint32_t lane_base, int row, bool row_valid,
                                             float l_sum, float m_ref, float o_scale = 1.f) {
  const bool fp16 = p.fp16 != 0;
  const float inv_l = l_sum > 0.f ? o_scale / l_sum : 0.f;
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
  const int dcols = min(it.dv, p.D - it.col_lo);   // columns >= D are zero padding
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
        if (c0 + 8 * v4 < dcols)
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

// store_output for the dense layout through tensor stores: the warp's 32
// rows are staged at `stage` (1 KB aligned, 4 KB per 64 columns) as 32-row
// boxes with the 128-byte swizzle (unit u of row t at u ^ (t & 7)), and one
// thread writes them with p.tm_o (rows past Nq and the zero padding
// columns past D are not written).  The LSE as store_output.
template <bool VARLEN>
__device__ __forceinline__ void store_output_boxes(const Params& p, const Item& it, bool have_o,
                                                   uint32_t lane_base, int warp, int lane, int row,
                                                   bool row_valid, float l_sum, float m_ref, uint32_t stage) {
  const bool fp16 = p.fp16 != 0;
  const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
  const uint32_t sw = (uint32_t)(lane & 7);
  for (int c0 = 0; c0 < it.dv; c0 += 64) {
    uint32_t va[32], vb[32];
    if (have_o) {
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
      const float a0 = __uint_as_float(e < 32 ? va[e] : vb[e - 32]) * inv_l;
      const float a1 = __uint_as_float(e + 1 < 32 ? va[e + 1] : vb[e + 1 - 32]) * inv_l;
      pk[c] = fp16 ? pack_f16(a0, a1) : pack_bf16(a0, a1);
    }
    const uint32_t box = stage + (uint32_t)(c0 / 64) * 4096u + (uint32_t)lane * 128u;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      st_shared_v4(box + (((uint32_t)q ^ sw) << 4), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
  }
  fence_proxy_async_smem();
  __syncwarp();
  const int row0 = it.q0 + 32 * warp;
  if (lane == 0 && row0 < it.q_len) {
    const int nch = (p.D + DK - 1) / DK;
    for (int c = 0; c < it.dv / 64; ++c) {
      const int chunk = it.col_lo / 64 + c;
      if (chunk >= nch) continue;
      if (VARLEN)
        tma_store_4d(&p.tm_o, stage + (uint32_t)c * 4096u, 0, it.q_row0 + row0, chunk, it.hq);
      else
        tma_store_5d(&p.tm_o, stage + (uint32_t)c * 4096u, 0, row0, chunk, it.hq, it.b);
    }
    bulk_commit_group();
    bulk_wait_read_all();   // the staging area is read before the CTA may exit
  }
  __syncwarp();
  if (row_valid && p.lse != nullptr && it.slice == 0) {
    const float lse = l_sum > 0.f ? (m_ref + log2f(l_sum)) * 0.6931471805599453f : -INFINITY;
    const long long li = VARLEN ? (long long)it.hq * p.Tq + it.q_row0 + row
                                : ((long long)it.b * p.Hq + it.hq) * p.Nq + row;
    p.lse[li] = lse;
  }
}

// Maximum of n scores (n a multiple of 16): eight independent chains of
// three-input maxima, then a small tree.
template <int N>
__device__ __forceinline__ float row_max(const float* x) {
  float m8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m8[i] = fmaxf(x[i], x[8 + i]);
#pragma unroll
  for (int c = 16; c < N; c += 16)
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], x[c + i], x[c + 8 + i]);
  return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

// P = exp2(x * xs - base) for n scores, packed to 16-bit pairs; returns the
// sum of the (unrounded) values.  The exponent arguments and the partial
// sums use packed fp32 pair instructions.
template <bool F16, int N>
__device__ __forceinline__ float form_p(const float* x, float xs, float base, uint32_t* pk) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int c = 0; c < N; c += 4) {
    float a0, a1, a2, a3;
    ffma2_bc(x[c], x[c + 1], xs, -base, a0, a1);
    ffma2_bc(x[c + 2], x[c + 3], xs, -base, a2, a3);
    const float e0 = ex2_approx(a0);
    const float e1 = ex2_approx(a1);
    const float e2 = ex2_approx(a2);
    const float e3 = ex2_approx(a3);
    fadd2_acc(s0, s1, e0, e1);
    fadd2_acc(s2, s3, e2, e3);
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
template <bool VARLEN, bool PAIR, bool UMASK>
__device__ __forceinline__ void softmax_role(const Params& p, const Item& it, int T, uint32_t tmem,
                                             int warp, int lane, const SoftmaxBars bars,
                                             volatile int* abort_flag, unsigned long long tmo,
                                             int* err) {
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
  if (UMASK && mask_kind != FFPA_MASK_NONE && row_valid) {
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
    bool w = wait_bounded(bars.s_full, j & 1, abort_flag, tmo, err);
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
        apply_mask32<UMASK>(x + 32 * q4, kbase + 32 * q4, it.kv_len, causal, row_limit, mrow, mk,
                            mask_kind, fp16);
        // One 32-key group at a time: keeps the mask loads of later groups
        // from being hoisted (register pressure).
        if (UMASK) asm volatile("" ::: "memory");
      }
    }
    const float mx = row_max<BN>(x) * xs;   // log2 domain (-inf stays -inf: xs > 0)
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
      w = wait_bounded(bars.pv_done + 8u * ((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag, tmo, err);
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
      w = wait_bounded(bars.pv_done + 8u * b, ((j - 2) >> 1) & 1, abort_flag, tmo, err);
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
                                abort_flag, tmo, err);
    ok = __all_sync(0xffffffffu, w);
    if (ok) tc_fence_after();
  }
  if (ok || T == 0) store_output<VARLEN>(p, it, T > 0, lane_base, row, row_valid, l_sum, m_ref);
}

}  // namespace ffpa
