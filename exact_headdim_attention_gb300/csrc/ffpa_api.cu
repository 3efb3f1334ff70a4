// Host side of libffpa.so: argument validation, kernel choice, planning,
// tensor maps, launch, and the C ABI declared in include/ffpa.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <initializer_list>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "ffpa_common.cuh"

// =====================================================================
// Host side: validation, planning, tensor maps, launch.
// =====================================================================
namespace {

using namespace ffpa;

constexpr unsigned long long DEFAULT_TIMEOUT_NS = 2000000000ull;
constexpr int MAX_DEVICES = 64;

// Status word of calls that pass none (one per device, set by the kernels
// when a wait runs out; read and cleared by ffpa_last_device_error).
__device__ int g_status_fallback;

// What one call asked for (ffpa_options), with the defaults filled in.
struct CallOpts {
  int* status;                   // device word, or NULL for the device's fallback word
  unsigned long long timeout_ns;
  int kernel;                    // FFPA_VARIANT_*
  int drop;                      // test hook
};

ffpa_status read_opts(const ffpa_options* o, CallOpts* c) {
  c->status = o ? o->status : nullptr;
  c->timeout_ns = o && o->wait_timeout_ns ? o->wait_timeout_ns : DEFAULT_TIMEOUT_NS;
  c->kernel = o ? o->kernel : FFPA_VARIANT_AUTO;
  c->drop = o && o->test_drop_first_copy ? 1 : 0;
  if (c->kernel < FFPA_VARIANT_AUTO || c->kernel > FFPA_VARIANT_DUAL) return FFPA_ERR_INVALID;
  return FFPA_OK;
}

// Facts about a device that never change while the process runs, looked up
// once: whether it is an sm_103 part, and the address of its fallback word.
struct DeviceFacts {
  std::once_flag once;
  ffpa_status arch = FFPA_ERR_CUDA;
  int* fallback = nullptr;
  int sms = 0;
};
DeviceFacts g_devices[MAX_DEVICES];

// The device's facts (computed on first use with `dev` current).
const DeviceFacts& device_facts(int dev) {
  DeviceFacts& f = g_devices[dev];
  std::call_once(f.once, [&] {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      f.arch = FFPA_ERR_CUDA;
      return;
    }
    f.arch = (major == 10 && minor == 3) ? FFPA_OK : FFPA_ERR_UNSUPPORTED;
    if (cudaDeviceGetAttribute(&f.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      f.sms = 0;
    }
    void* addr = nullptr;
    if (f.arch == FFPA_OK) {
      if (cudaGetSymbolAddress(&addr, g_status_fallback) != cudaSuccess) {
        cudaGetLastError();
        f.arch = FFPA_ERR_CUDA;
      }
    }
    f.fallback = static_cast<int*>(addr);
  });
  return f;
}

// The device that owns `ptr`: device or managed memory only (host memory,
// even mapped, is rejected: the tensor-memory-accelerator copies and the
// kernels' stores expect memory of the GPU they run on).
ffpa_status pointer_device(const void* ptr, int* dev) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();
    return FFPA_ERR_CUDA;
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return FFPA_ERR_INVALID;
  if (attr.device < 0 || attr.device >= MAX_DEVICES) return FFPA_ERR_UNSUPPORTED;
  *dev = attr.device;
  return FFPA_OK;
}

// Every non-null pointer of the call lives on the device of the first one;
// that device is an sm_103 part.  On success *dev is that device.
ffpa_status check_devices(std::initializer_list<const void*> ptrs, int* dev) {
  int d0 = -1;
  for (const void* p : ptrs) {
    if (!p) continue;
    int d = -1;
    const ffpa_status st = pointer_device(p, &d);
    if (st != FFPA_OK) return st;
    if (d0 < 0)
      d0 = d;
    else if (d != d0)
      return FFPA_ERR_INVALID;
  }
  if (d0 < 0) return FFPA_ERR_INVALID;
  *dev = d0;
  return FFPA_OK;
}

// Device set-up shared by the entry points once the arguments are valid:
// the arch check and the status word the kernels report to.
ffpa_status device_status_word(int dev, const CallOpts& o, int** err) {
  const DeviceFacts& f = device_facts(dev);
  if (f.arch != FFPA_OK) return f.arch;
  if (o.status) {
    int d = -1;
    const ffpa_status st = pointer_device(o.status, &d);
    if (st != FFPA_OK) return st;
    if (d != dev || (reinterpret_cast<uintptr_t>(o.status) & 3u) != 0) return FFPA_ERR_INVALID;
  }
  *err = o.status ? o.status : f.fallback;
  return FFPA_OK;
}

// Element size of a mask kind (bytes).
size_t mask_esz(ffpa_mask_kind mk) {
  return mk == FFPA_MASK_BOOL ? 1 : mk == FFPA_MASK_ADD_F32 ? 4 : 2;
}

bool aligned_to(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

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

// Splits D into at most 256-column output slices, sizes the V stage, and
// decides whether Q stays resident in shared memory (D <= 512) and how many
// 32 KB ring slots fit beside it.  Returns the dynamic shared memory bytes.
size_t plan(int D, Params* P) {
  P->nchunks = (D + DK - 1) / DK;   // a head dim below a multiple of 64 is zero-padded
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
  if (D % DK != 0) return false;
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

enum class Kern { SINGLE, PAIR, SPLIT, DUAL };

// The dual-tile kernel: dense batches, D = 64 or 128 (instantiated shapes).
bool dual_eligible(int D, bool varlen) { return !varlen && (D == 64 || D == 128); }

// Column-split kernels for head dimension D (a multiple of 64, 128..1024):
// the D/64 chunks are rounded up to an instantiated shape (2, 4, 6 or 8
// chunks on clusters of C = 2 CTAs; 12 on C = 3; 16 on C = 4), each CTA
// owning an equal share of whole chunks (at most 256 columns).  The chunks
// past D lie beyond the tensor maps' chunk extent, so the TMA unit reads
// them as zeros: they add nothing to S, and their output columns are not
// stored.  0 = the kernels do not take D.
int split_chunks(int D) {
  if (D % DK != 0) return 0;
  const int n = D / DK;
  if (n < 2) return 0;
  if (n <= 8) return (n + 1) & ~1;
  if (n <= 12) return 12;
  if (n <= 16) return 16;
  return 0;
}

int split_ways(int D) {
  const int n = split_chunks(D);
  return n == 0 ? 0 : n <= 8 ? 2 : n == 12 ? 3 : 4;
}

bool split_eligible(int D) { return split_ways(D) != 0; }

// Kernel choice, from measurements on GB300 (bf16): above D=256 the
// column-split kernels win on dense, causal and varlen batches (they do not
// recompute S; D=384: 1048 vs 732 TFLOPS for the single-CTA kernel, and at
// D=320 the split padded to 384 columns beats the single-CTA kernel's two
// slices); at D=256 (no recompute anyway) the pair kernel wins on dense
// batches; at dense D=64 and D=128 the dual-tile kernel (two query tiles
// per SM sharing K/V) wins; on packed varlen batches of mixed lengths the
// 256-row tiles of the pair and dual kernels waste more rows on short
// sequences than they save, and the single-CTA kernel runs.
Kern choose_kernel(int D, bool varlen, int v) {
  if (D % DK != 0) return Kern::SINGLE;   // only the single-CTA kernel takes zero-padded chunks
  if (v == FFPA_VARIANT_SINGLE) return Kern::SINGLE;
  if (v == FFPA_VARIANT_PAIR) return pair_eligible(D) ? Kern::PAIR : Kern::SINGLE;
  if (v == FFPA_VARIANT_SPLIT) return split_eligible(D) ? Kern::SPLIT : Kern::SINGLE;
  if (v == FFPA_VARIANT_DUAL) return dual_eligible(D, varlen) ? Kern::DUAL : Kern::SINGLE;
  if (D > 256 && split_eligible(D)) return Kern::SPLIT;
  if (!varlen && D == 256) return Kern::PAIR;
  if (dual_eligible(D, varlen)) return Kern::DUAL;
  return Kern::SINGLE;
}

// Dual-tile plan: Q_A and Q_B resident, two P tiles, a ring of one-tile
// slots (K or V: 128 keys x D); boxes of 128 rows x D/64 chunks.
size_t plan_dual(int D, Params* P) {
  P->nchunks = D / DK;
  P->n_slices = 1;
  P->kchunks = P->nchunks;
  P->vchunks = P->nchunks;
  P->vk = BN;
  P->vslot = BN * P->vchunks * 128;
  P->q_res = 1;
  P->nslot_v = 0;
  const size_t tile = (size_t)P->nchunks * CHUNK_BYTES;
  const size_t fixed = 2 * tile + 2 * (size_t)P_TILE_BYTES;
  size_t ns = (SMEM_LIMIT - SMEM_STATIC_RESERVE - 1024 - fixed) / tile;
  if (ns > 8) ns = 8;
  P->nslot = static_cast<int>(ns);
  return 1024 + fixed + ns * tile;
}

// Column-split plan: Q chunks 0..3 in TMEM, the rest resident in shared
// memory when they fit (else streamed through the ring), C P tiles, V
// stages of vk keys x D/C columns, 32 KB ring slots.
size_t plan_split(int D, Params* P) {
  const int C = split_ways(D);
  P->split_c = C;
  P->nchunks = split_chunks(D);
  P->n_slices = 1;
  P->qt_chunks = P->nchunks < Q_TMEM_MAX_CHUNKS ? P->nchunks : Q_TMEM_MAX_CHUNKS;
  P->kchunks = 2;
  P->kc = 2;
  const bool qres = (size_t)(P->nchunks - P->qt_chunks) * CHUNK_BYTES + (size_t)C * P_TILE_BYTES +
                        3 * (size_t)SLOT_BYTES <=
                    SMEM_LIMIT - SPLIT_STATIC_RESERVE - 1024;
  P->q_res = qres ? 1 : 0;
  P->vchunks = P->nchunks / C;
  int vk = 128;
  while (vk > 16 && (size_t)vk * P->vchunks * 128 > SLOT_BYTES) vk >>= 1;
  P->vk = vk;
  P->vslot = vk * P->vchunks * 128;
  P->nslot_v = 0;
  const size_t fixed =
      (qres ? (size_t)(P->nchunks - P->qt_chunks) * CHUNK_BYTES : 0) + (size_t)C * P_TILE_BYTES;
  size_t ns = (SMEM_LIMIT - SPLIT_STATIC_RESERVE - 1024 - fixed) / SLOT_BYTES;
  if (ns > (size_t)NSLOT_MAX) ns = NSLOT_MAX;
  P->nslot = static_cast<int>(ns);
  return 1024 + fixed + ns * SLOT_BYTES;
}

// FP8 workspace: e4m3 Q [B,Hq,Nqp,D], K [B,Hkv,Nkp,D], transposed V
// [B,Hkv,D,Nkp] and the fp32 block scales of each (N rounded up to 128 in
// Nqp / Nkp); every part 256-byte aligned.
struct Fp8Layout {
  size_t off[6];   // q8, k8, v8t, sq, sk, sv
  size_t total;
  int64_t nqp, nkp;
  int nqb, nkb;
};

Fp8Layout fp8_layout(int B, int Hq, int Hkv, int Nq, int Nkv, int D) {
  Fp8Layout L{};
  L.nqb = (Nq + 127) / 128;
  L.nkb = (Nkv + 127) / 128;
  L.nqp = (int64_t)L.nqb * 128;
  L.nkp = (int64_t)L.nkb * 128;
  const size_t sizes[6] = {(size_t)B * Hq * L.nqp * D, (size_t)B * Hkv * L.nkp * D,
                           (size_t)B * Hkv * L.nkp * D, (size_t)B * Hq * L.nqb * 4,
                           (size_t)B * Hkv * L.nkb * 4, (size_t)B * Hkv * L.nkb * 4};
  size_t at = 0;
  for (int i = 0; i < 6; ++i) {
    L.off[i] = at;
    at += (sizes[i] + 255) & ~(size_t)255;
  }
  L.total = at;
  return L;
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

ffpa_status launch_kernel(Kern kn, bool varlen, const Params& P, int items, size_t smem,
                          cudaStream_t stream) {
  const bool umask = P.mask != nullptr;
  if (kn == Kern::PAIR) return launch_pair(varlen, umask, P, items, smem, stream);
  if (kn == Kern::DUAL) return varlen ? FFPA_ERR_UNSUPPORTED : launch_dual(umask, P, items, smem, stream);
  if (kn == Kern::SPLIT)
    return (P.split_c == 2 && P.q_res != 0) ? launch_split(varlen, umask, P, items, smem, stream)
                          : launch_cluster(varlen, umask, P, items, smem, stream);
  return launch_single(varlen, umask, P, items, smem, stream);
}

size_t plan_for(Kern kn, int D, Params* P) {
  if (kn == Kern::PAIR) return plan_pair(D, P);
  if (kn == Kern::SPLIT) return plan_split(D, P);
  if (kn == Kern::DUAL) return plan_dual(D, P);
  return plan(D, P);
}

// Backward: output slices, ring depths, shared memory, work items; then the
// three or four launches.  P's sizes, tiles, maps, pointers, scale, causal and fp16
// are set by the caller.
ffpa_status bwd_launch(BwdParams& P, bool any_q, bool any_k, const CallOpts& o, cudaStream_t stream) {
  P.nchunks = P.D / DK;
  P.n_sl = (P.D + BWD_OUT_COLS - 1) / BWD_OUT_COLS;
  // Shared memory: one 32 KB P/dS tile, then the ring.
  size_t ns = (SMEM_LIMIT - BWD_STATIC_RESERVE - 1024 - P_TILE_BYTES) / SLOT_BYTES;
  if (ns > (size_t)BWD_NSLOT_MAX) ns = BWD_NSLOT_MAX;
  P.nslot = static_cast<int>(ns);
  const size_t smem = 1024 + P_TILE_BYTES + ns * SLOT_BYTES;
  // D <= 128: dV and dK from one S, dP in one kernel (measured on GB300 at
  // D=128: 324 vs 255 TFLOPS for separate dV and dK kernels; at D=512 the
  // separate kernels win, 324 vs 288).
  P.kv_together = P.D <= 128;
  size_t ns2 = (SMEM_LIMIT - BWD_STATIC_RESERVE - 1024 - 2 * (size_t)P_TILE_BYTES) / SLOT_BYTES;
  if (ns2 > (size_t)BWD_NSLOT_MAX) ns2 = BWD_NSLOT_MAX;
  P.nslot_two = static_cast<int>(ns2);
  const size_t smem_two = 1024 + 2 * (size_t)P_TILE_BYTES + ns2 * SLOT_BYTES;
  P.scale_log2 = P.scale * 1.4426950408889634f;
  P.inject = o.drop;
  P.timeout_ns = o.timeout_ns;
  const long long dq_items = any_q ? (long long)P.B * P.Hq * P.n_qt * P.n_sl : 0;
  const long long kv_items = any_k ? (long long)P.B * P.Hkv * P.n_kt * P.n_sl : 0;
  if (dq_items > 0x7fffffffLL || kv_items > 0x7fffffffLL) return FFPA_ERR_INVALID;
  return launch_bwd(P, static_cast<int>(dq_items), static_cast<int>(kv_items), smem, smem_two, stream);
}

// Stored-tile backward: dense, D = 128, 256, 384 or 512, at least one query row
// and one key.  Workspace bytes (0: the path does not apply): a 32 KB block
// of zeros, then P and dS, one 32 KB block (128 x 128 16-bit values) per
// (b, hq, query tile, stored key tile) each (causal: only the key tiles the
// query tile sees).
size_t bwd_tiles_bytes(int B, int Hq, int Nq, int Nkv, int D, int causal) {
  if (!(D == 128 || D == 256 || D == 384 || D == 512) || B < 1 || Hq < 1 || Nq < 1 || Nkv < 1) return 0;
  if (causal && Nkv < Nq) return 0;
  const long long blocks = (long long)B * Hq * bwd_stored_before((Nq + BM - 1) / BM, Nq, Nkv, causal);
  if (blocks > (1LL << 30)) return 0;
  return static_cast<size_t>((2 * blocks + 1) * (long long)P_TILE_BYTES);
}

// Varlen stored-tile workspace: the per-sequence block bases (nseq + 1
// int64, rounded up to 1 KB), a 32 KB block of zeros, then P and dS blocks.
size_t bwd_varlen_header_bytes(int nseq) { return (((size_t)nseq + 1) * 8 + 1023) / 1024 * 1024; }

size_t bwd_varlen_tiles_bytes(const int32_t* cu_q, const int32_t* cu_k, int nseq, int Hq, int D, int causal) {
  if (!(D == 128 || D == 256 || D == 384 || D == 512) || !cu_q || nseq < 1 || Hq < 1) return 0;
  if (!cu_k) cu_k = cu_q;
  long long blocks = 0;
  for (int s = 0; s < nseq; ++s) {
    const int lq = cu_q[s + 1] - cu_q[s], lk = cu_k[s + 1] - cu_k[s];
    if (lq < 0 || lk < 0) return 0;
    blocks += (long long)Hq * bwd_stored_before((lq + BM - 1) / BM, lq, lk, causal);
    if (blocks > (1LL << 30)) return 0;
  }
  if (blocks == 0) return 0;
  return bwd_varlen_header_bytes(nseq) + static_cast<size_t>((2 * blocks + 1) * (long long)P_TILE_BYTES);
}

// Plans and launches the stored-tile path: the caller has set P as for
// bwd_launch and checked the workspace (`ws`, `ws_bytes`: dense, at least
// bwd_tiles_bytes(); varlen, at least the header and three blocks, the
// kernels checking every block index against what it holds).
ffpa_status bwd_tiles_launch(BwdParams& P, void* ws, size_t ws_bytes, int sms, const CallOpts& o,
                             cudaStream_t stream) {
  P.nchunks = P.D / DK;
  P.n_sl = 1;
  long long blocks;
  uint8_t* w = static_cast<uint8_t*>(ws);
  if (P.varlen) {
    const size_t hdr = bwd_varlen_header_bytes(P.B);
    P.ws_head = 0;
    P.ws_base = reinterpret_cast<const long long*>(w);
    w += hdr;
    blocks = (long long)((ws_bytes - hdr - P_TILE_BYTES) / (2 * (size_t)P_TILE_BYTES));
  } else {
    P.ws_head = bwd_stored_before(P.n_qt, P.Nq, P.Nkv, P.causal);
    P.ws_base = nullptr;
    blocks = (long long)P.B * P.Hq * P.ws_head;
  }
  P.ws_blocks = blocks;
  P.ws_zero = w;
  P.ws_p = w + P_TILE_BYTES;
  P.ws_ds = w + (1 + blocks) * (long long)P_TILE_BYTES;
  // Scores kernel: dO (D/64 chunks) resident, then the ring.
  size_t ns = (SMEM_LIMIT - TS_STATIC_RESERVE - 1024 - (size_t)P.nchunks * CHUNK_BYTES) / SLOT_BYTES;
  if (ns > (size_t)TS_NSLOT_MAX) ns = TS_NSLOT_MAX;
  P.ts_nslot = static_cast<int>(ns);
  const size_t smem_s = 1024 + (size_t)P.nchunks * CHUNK_BYTES + ns * SLOT_BYTES;
  size_t nc = (SMEM_LIMIT - TC_STATIC_RESERVE - 1024) / SLOT_BYTES;
  if (nc > (size_t)TC_NSLOT_MAX) nc = TC_NSLOT_MAX;
  P.tc_nslot = static_cast<int>(nc);
  const size_t smem_c = 1024 + nc * SLOT_BYTES;
  // Key-tile ranges per query tile (non-causal only; causal items are
  // ordered longest first instead): the count whose last wave is fullest,
  // keeping at least 8 key tiles per range (each range loads Q and dO once).
  const long long base = (long long)P.B * P.Hq * P.n_qt;
  P.kv_parts = 1;
  if (!P.causal && !P.varlen && sms > 0) {
    double best = -1.0;
    for (int parts = 1; parts <= 4; parts *= 2) {
      if (parts > 1 && P.n_kt / parts < 8) break;
      const double waves = (double)(base * parts) / sms;
      const double eff = waves / std::ceil(waves);
      if (eff > best + 0.03) {
        best = eff;
        P.kv_parts = parts;
      }
    }
  }
  P.scale_log2 = P.scale * 1.4426950408889634f;
  P.inject = o.drop;
  P.timeout_ns = o.timeout_ns;
  const long long score_items = base * P.kv_parts;
  // Contraction: CTA pairs over two adjacent query tiles (dQ) or key tiles (dV, dK).
  const long long n_dq = (long long)P.B * P.Hq * ((P.n_qt + 1) / 2);
  const long long n_kv = (long long)P.B * P.Hkv * ((P.n_kt + 1) / 2);
  const long long contract_items = n_dq + 2 * n_kv;
  if (score_items > 0x7fffffffLL || 2 * contract_items > 0x7fffffffLL) return FFPA_ERR_INVALID;
  P.n_dq_items = static_cast<int>(n_dq);
  P.n_kv_items = static_cast<int>(n_kv);
  return launch_bwd_tiles(P, static_cast<int>(score_items), static_cast<int>(contract_items), smem_s, smem_c,
                          stream);
}

}  // namespace

namespace ffpa {

namespace {
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get = nullptr;
  PFN_cuCtxSetCurrent_v4000 set = nullptr;
};
const CtxFns& ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* g = nullptr;
    void* s = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &g, 4000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxSetCurrent", &s, 4000, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess) {
      f.get = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(g);
      f.set = reinterpret_cast<PFN_cuCtxSetCurrent_v4000>(s);
    } else {
      cudaGetLastError();
    }
  });
  return f;
}
}  // namespace

DeviceScope::DeviceScope(int dev) {
  const CtxFns& f = ctx_fns();
  if (!f.get || !f.set || f.get(&saved_) != CUDA_SUCCESS) return;
  if (cudaSetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  // Since CUDA 12, cudaSetDevice initialises the primary context and makes
  // it current on this thread at once.
  CUcontext now = nullptr;
  if (f.get(&now) != CUDA_SUCCESS || now == nullptr) return;
  restore_ = now != saved_;
  ok_ = true;
}

DeviceScope::~DeviceScope() {
  if (restore_) ctx_fns().set(saved_);
}

// Kernels whose shared-memory limit was raised, per device (set-once facts).
ffpa_status set_smem_attr_once(const void* fn, int device, int bytes) {
  struct Entry {
    const void* fn;
    int device, bytes;
  };
  static std::mutex mu;
  static Entry table[256];
  static int n = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (table[i].fn == fn && table[i].device == device && table[i].bytes >= bytes) return FFPA_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return FFPA_ERR_CUDA;
  }
  for (int i = 0; i < n; ++i)
    if (table[i].fn == fn && table[i].device == device) {
      table[i].bytes = bytes;
      return FFPA_OK;
    }
  if (n < 256) table[n++] = Entry{fn, device, bytes};
  return FFPA_OK;
}

}  // namespace ffpa

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

int ffpa_selected_kernel(int D, int varlen, int kernel) {
  if (D < 64 || D > 1024 || D % (varlen ? 64 : 8) != 0) return -1;
  if (kernel < FFPA_VARIANT_AUTO || kernel > FFPA_VARIANT_DUAL) return -1;
  const Kern kn = choose_kernel(D, varlen != 0, kernel);
  return kn == Kern::PAIR    ? FFPA_VARIANT_PAIR
         : kn == Kern::SPLIT ? FFPA_VARIANT_SPLIT
         : kn == Kern::DUAL  ? FFPA_VARIANT_DUAL
                             : FFPA_VARIANT_SINGLE;
}

ffpa_status ffpa_last_device_error(ffpa_stream_t stream) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = -1;
  if (cudaStreamGetDevice(s, &dev) != cudaSuccess) {
    cudaGetLastError();
    return FFPA_ERR_CUDA;
  }
  if (dev < 0 || dev >= MAX_DEVICES) return FFPA_ERR_CUDA;
  DeviceScope scope(dev);
  if (!scope.ok()) return FFPA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FFPA_ERR_CUDA;
  const DeviceFacts& f = device_facts(dev);
  if (f.arch == FFPA_ERR_UNSUPPORTED) return FFPA_OK;   // no kernel of this library runs there
  if (f.arch != FFPA_OK) return FFPA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, f.fallback, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FFPA_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpy(f.fallback, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return FFPA_ERR_CUDA;
  }
  return static_cast<ffpa_status>(word);
}

ffpa_status ffpa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                        ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                        const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                        const int64_t o_str[4], const void* mask, ffpa_mask_kind mask_kind,
                        const int64_t mask_str[4], const float* scale, int is_causal,
                        int enable_gqa, ffpa_stream_t stream, const ffpa_options* options) {
  if (dt != FFPA_BF16 && dt != FFPA_FP16) return FFPA_ERR_DTYPE;
  if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nkv < 0) return FFPA_ERR_INVALID;
  if (D < 64 || D > 1024 || D % 8 != 0) return FFPA_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return FFPA_ERR_INVALID;
  if (Hq != Hkv && !enable_gqa) return FFPA_ERR_INVALID;
  if (is_causal && Nkv < Nq) return FFPA_ERR_INVALID;
  if (mask_kind < FFPA_MASK_NONE || mask_kind > FFPA_MASK_ADD_QTYPE) return FFPA_ERR_INVALID;
  CallOpts opt;
  if (read_opts(options, &opt) != FFPA_OK) return FFPA_ERR_INVALID;
  const float sc = scale ? *scale : 1.0f / std::sqrt(static_cast<float>(D));
  if (!std::isfinite(sc)) return FFPA_ERR_INVALID;
  if (B == 0 || Nq == 0) return FFPA_OK;          // nothing to read or write
  if (!q || !o || !q_str || !k_str || !v_str || !o_str) return FFPA_ERR_INVALID;
  if (Nkv > 0 && (!k || !v)) return FFPA_ERR_INVALID;
  const bool umask = mask_kind != FFPA_MASK_NONE && Nkv > 0;
  if (umask) {
    if (!mask || !mask_str) return FFPA_ERR_INVALID;
    for (int i = 0; i < 4; ++i)
      if (mask_str[i] < 0) return FFPA_ERR_INVALID;
    if (!aligned_to(mask, mask_esz(mask_kind))) return FFPA_ERR_INVALID;
  }
  const int64_t qsz[4] = {B, Hq, Nq, D}, ksz[4] = {B, Hkv, Nkv, D};
  if (!strides_ok(q_str, qsz, 4) || !strides_ok(o_str, qsz, 4)) return FFPA_ERR_INVALID;
  if (Nkv > 0 && (!strides_ok(k_str, ksz, 4) || !strides_ok(v_str, ksz, 4))) return FFPA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(o) || (Nkv > 0 && (!aligned16(k) || !aligned16(v))))
    return FFPA_ERR_INVALID;
  if (lse && !aligned_to(lse, 4)) return FFPA_ERR_INVALID;
  int dev = 0;
  ffpa_status st = check_devices({q, o, Nkv > 0 ? k : nullptr, Nkv > 0 ? v : nullptr, lse,
                                  umask ? mask : nullptr},
                                 &dev);
  if (st != FFPA_OK) return st;
  DeviceScope scope(dev);
  if (!scope.ok()) return FFPA_ERR_CUDA;
  int* err = nullptr;
  if ((st = device_status_word(dev, opt, &err)) != FFPA_OK) return st;

  Params P{};
  const CUtensorMapDataType tdt =
      dt == FFPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  Kern kn = choose_kernel(D, false, opt.kernel);
  if (kn == Kern::DUAL && umask) kn = Kern::SINGLE;   // the dual-tile kernel takes no mask
  const bool pair = kn == Kern::PAIR;
  size_t smem = plan_for(kn, D, &P);
  if (kn == Kern::SPLIT && is_causal && P.split_c == 2 && P.nchunks == 8) {
    // Dense causal at D = 512: Q streamed through a five-stage ring (the
    // cluster kernel at C = 2) instead of resident beside three stages
    // (measured on causal GQA B2 Hq32 Hkv8 N8192: 1058 vs 1031 TFLOPS; the
    // dense and varlen batches run faster with Q resident).
    P.q_res = 0;
    size_t ns = (SMEM_LIMIT - SPLIT_STATIC_RESERVE - 1024 - 2 * (size_t)P_TILE_BYTES) / SLOT_BYTES;
    if (ns > (size_t)NSLOT_MAX) ns = NSLOT_MAX;
    P.nslot = static_cast<int>(ns);
    smem = 1024 + 2 * (size_t)P_TILE_BYTES + ns * SLOT_BYTES;
  }
  const uint32_t k_rows = pair ? BN / 2 : BN;
  const uint32_t k_box_chunks = pair ? (uint32_t)P.kc : (uint32_t)P.kchunks;
  // The maps span the real D/64 chunks; a column-split plan may run more
  // (padding chunks, read as zeros past this extent).
  const uint64_t nch = (uint64_t)(D / DK);
  P.dfine = D % DK != 0;
  if (P.dfine) {
    // (D, N, H, B) views with one 64-column box per chunk: the TMA unit
    // zero-fills the columns past D of the last chunk.
    const uint64_t dq4[4] = {(uint64_t)D, (uint64_t)Nq, (uint64_t)Hq, (uint64_t)B};
    const uint64_t sq[3] = {(uint64_t)q_str[2] * 2, (uint64_t)q_str[1] * 2, (uint64_t)q_str[0] * 2};
    const uint32_t bq[4] = {64, BM, 1, 1};
    if ((st = encode_map(&P.tm_q, tdt, 4, q, dq4, sq, bq)) != FFPA_OK) return st;
    if (Nkv > 0) {
      const uint64_t dk4[4] = {(uint64_t)D, (uint64_t)Nkv, (uint64_t)Hkv, (uint64_t)B};
      const uint64_t sk[3] = {(uint64_t)k_str[2] * 2, (uint64_t)k_str[1] * 2, (uint64_t)k_str[0] * 2};
      const uint64_t sv[3] = {(uint64_t)v_str[2] * 2, (uint64_t)v_str[1] * 2, (uint64_t)v_str[0] * 2};
      const uint32_t bk[4] = {64, BN, 1, 1};
      const uint32_t bv[4] = {64, (uint32_t)P.vk, 1, 1};
      if ((st = encode_map(&P.tm_k, tdt, 4, k, dk4, sk, bk)) != FFPA_OK) return st;
      if ((st = encode_map(&P.tm_v, tdt, 4, v, dk4, sv, bv)) != FFPA_OK) return st;
    }
  } else {
    const uint64_t dq[5] = {64, (uint64_t)Nq, nch, (uint64_t)Hq, (uint64_t)B};
    const uint64_t sq[4] = {(uint64_t)q_str[2] * 2, 128, (uint64_t)q_str[1] * 2, (uint64_t)q_str[0] * 2};
    const uint32_t bq[5] = {64, BM, (uint32_t)P.kchunks, 1, 1};
    if ((st = encode_map(&P.tm_q, tdt, 5, q, dq, sq, bq)) != FFPA_OK) return st;
    if (Nkv > 0) {   // with no keys no work item issues a copy; the maps stay unused
      const uint64_t dk[5] = {64, (uint64_t)Nkv, nch, (uint64_t)Hkv, (uint64_t)B};
      const uint64_t sk[4] = {(uint64_t)k_str[2] * 2, 128, (uint64_t)k_str[1] * 2, (uint64_t)k_str[0] * 2};
      const uint32_t bk[5] = {64, k_rows, k_box_chunks, 1, 1};
      if ((st = encode_map(&P.tm_k, tdt, 5, k, dk, sk, bk)) != FFPA_OK) return st;
      const uint64_t sv[4] = {(uint64_t)v_str[2] * 2, 128, (uint64_t)v_str[1] * 2, (uint64_t)v_str[0] * 2};
      const uint32_t bv[5] = {64, (uint32_t)P.vk, (uint32_t)P.vchunks, 1, 1};
      if ((st = encode_map(&P.tm_v, tdt, 5, v, dk, sv, bv)) != FFPA_OK) return st;
    }
    if (kn == Kern::SPLIT && P.split_c == 2 && P.q_res && Nq > 0) {
      // The column-split pair kernel stores O through 32-row boxes.
      const uint64_t so[4] = {(uint64_t)o_str[2] * 2, 128, (uint64_t)o_str[1] * 2, (uint64_t)o_str[0] * 2};
      const uint32_t bo[5] = {64, 32, 1, 1, 1};
      if ((st = encode_map(&P.tm_o, tdt, 5, o, dq, so, bo)) != FFPA_OK) return st;
      P.o_tma = 1;
    }
  }
  P.o = o;
  P.lse = lse;
  P.mask = umask ? mask : nullptr;
  P.mask_kind = umask ? mask_kind : FFPA_MASK_NONE;
  for (int i = 0; i < 4; ++i) {
    P.o_str[i] = o_str[i];
    P.m_str[i] = umask ? mask_str[i] : 0;
  }
  P.B = B;
  P.Hq = Hq;
  P.group = Hq / Hkv;
  P.Nq = Nq;
  P.Nkv = Nkv;
  P.D = D;
  P.Tq = 0;
  const int q_tile = (pair || kn == Kern::DUAL) ? 2 * BM : BM;
  P.n_qt = (Nq + q_tile - 1) / q_tile;
  P.scale_log2 = sc * 1.4426950408889634f;
  P.causal = is_causal ? 1 : 0;
  P.fp16 = dt == FFPA_FP16;
  P.inject = opt.drop;
  P.timeout_ns = opt.timeout_ns;
  P.err = err;
  P.device = dev;
  const long long items = (long long)B * Hq * P.n_qt * P.n_slices;
  if (items > 0x7fffffffLL) return FFPA_ERR_INVALID;
  return launch_kernel(kn, false, P, static_cast<int>(items), smem,
                       reinterpret_cast<cudaStream_t>(stream));
}

ffpa_status ffpa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                     const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                     const int64_t o_str[4], const void* mask, ffpa_mask_kind mask_kind,
                     const int64_t mask_str[4], const float* scale, int is_causal, int enable_gqa,
                     ffpa_stream_t stream) {
  return ffpa_fwd_ex(q, k, v, o, lse, dt, B, Hq, Hkv, Nq, Nkv, D, q_str, k_str, v_str, o_str, mask,
                     mask_kind, mask_str, scale, is_causal, enable_gqa, stream, nullptr);
}

ffpa_status ffpa_bwd_ws_ex(const void* q, const void* k, const void* v, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           float* delta, ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                           const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                           const int64_t o_str[4], const int64_t do_str[4], const int64_t dq_str[4],
                           const int64_t dk_str[4], const int64_t dv_str[4], const void* mask,
                           ffpa_mask_kind mask_kind, const int64_t mask_str[4], const float* scale,
                           int is_causal, int enable_gqa, void* workspace, size_t workspace_bytes,
                           ffpa_stream_t stream, const ffpa_options* options) {
  if (dt != FFPA_BF16 && dt != FFPA_FP16) return FFPA_ERR_DTYPE;
  if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nkv < 0) return FFPA_ERR_INVALID;
  if (D < 64 || D > 1024 || D % 64 != 0) return FFPA_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return FFPA_ERR_INVALID;
  if (Hq != Hkv && !enable_gqa) return FFPA_ERR_INVALID;
  if (is_causal && Nkv < Nq) return FFPA_ERR_INVALID;
  if (mask_kind < FFPA_MASK_NONE || mask_kind > FFPA_MASK_ADD_QTYPE) return FFPA_ERR_INVALID;
  CallOpts opt;
  if (read_opts(options, &opt) != FFPA_OK) return FFPA_ERR_INVALID;
  const float sc = scale ? *scale : 1.0f / std::sqrt(static_cast<float>(D));
  if (!std::isfinite(sc)) return FFPA_ERR_INVALID;
  if (B == 0 || (Nq == 0 && Nkv == 0)) return FFPA_OK;   // nothing to write
  const bool umask = mask_kind != FFPA_MASK_NONE && Nq > 0 && Nkv > 0;
  if (umask) {
    if (!mask || !mask_str) return FFPA_ERR_INVALID;
    for (int i = 0; i < 4; ++i)
      if (mask_str[i] < 0) return FFPA_ERR_INVALID;
    if (!aligned_to(mask, mask_esz(mask_kind))) return FFPA_ERR_INVALID;
  }
  if (!q_str || !k_str || !v_str || !o_str || !do_str || !dq_str || !dk_str || !dv_str)
    return FFPA_ERR_INVALID;
  const int64_t qsz[4] = {B, Hq, Nq, D}, ksz[4] = {B, Hkv, Nkv, D};
  if (Nq > 0) {
    if (!q || !o || !dout || !dq || !lse || !delta) return FFPA_ERR_INVALID;
    if (!strides_ok(q_str, qsz, 4) || !strides_ok(o_str, qsz, 4) || !strides_ok(do_str, qsz, 4) ||
        !strides_ok(dq_str, qsz, 4))
      return FFPA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(o) || !aligned16(dout) || !aligned16(dq)) return FFPA_ERR_INVALID;
    if (!aligned_to(lse, 4) || !aligned_to(delta, 4)) return FFPA_ERR_INVALID;
  }
  if (Nkv > 0) {
    if (!k || !v || !dk || !dv) return FFPA_ERR_INVALID;
    if (!strides_ok(k_str, ksz, 4) || !strides_ok(v_str, ksz, 4) || !strides_ok(dk_str, ksz, 4) ||
        !strides_ok(dv_str, ksz, 4))
      return FFPA_ERR_INVALID;
    if (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv)) return FFPA_ERR_INVALID;
  }
  int dev = 0;
  const bool any_q = Nq > 0, any_k = Nkv > 0;
  // The stored-tile path runs when it applies and the workspace holds it;
  // otherwise the sliced kernels run and the workspace is not touched.
  const size_t ws_need = bwd_tiles_bytes(B, Hq, Nq, Nkv, D, is_causal ? 1 : 0);
  const bool tiles = workspace != nullptr && ws_need > 0 && workspace_bytes >= ws_need;
  if (tiles && !aligned16(workspace)) return FFPA_ERR_INVALID;
  ffpa_status st = check_devices({any_q ? q : nullptr, any_q ? o : nullptr, any_q ? dout : nullptr,
                                  any_q ? dq : nullptr, any_q ? lse : nullptr, any_q ? delta : nullptr,
                                  any_k ? k : nullptr, any_k ? v : nullptr, any_k ? dk : nullptr,
                                  any_k ? dv : nullptr, umask ? mask : nullptr,
                                  tiles ? workspace : nullptr},
                                 &dev);
  if (st != FFPA_OK) return st;
  DeviceScope scope(dev);
  if (!scope.ok()) return FFPA_ERR_CUDA;
  int* err = nullptr;
  if ((st = device_status_word(dev, opt, &err)) != FFPA_OK) return st;

  BwdParams P{};
  const CUtensorMapDataType tdt =
      dt == FFPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  P.nchunks = D / DK;
  P.npairs = (P.nchunks + 1) / 2;
  P.kchunks = P.nchunks < 2 ? P.nchunks : 2;
  const uint64_t nch = (uint64_t)P.nchunks;
  const uint32_t box[5] = {64, BM, (uint32_t)P.kchunks, 1, 1};
  // With no query rows (or no keys) no work item copies from those maps.
  if (any_q) {
    const uint64_t dq5[5] = {64, (uint64_t)Nq, nch, (uint64_t)Hq, (uint64_t)B};
    const uint64_t sq[4] = {(uint64_t)q_str[2] * 2, 128, (uint64_t)q_str[1] * 2, (uint64_t)q_str[0] * 2};
    const uint64_t sd[4] = {(uint64_t)do_str[2] * 2, 128, (uint64_t)do_str[1] * 2, (uint64_t)do_str[0] * 2};
    if ((st = encode_map(&P.tm_q, tdt, 5, q, dq5, sq, box)) != FFPA_OK) return st;
    if ((st = encode_map(&P.tm_do, tdt, 5, dout, dq5, sd, box)) != FFPA_OK) return st;
    if (tiles) {   // output stores of the contraction: box 64 x 32 rows
      const uint32_t obox[5] = {64, 32, 1, 1, 1};
      const uint64_t sdq[4] = {(uint64_t)dq_str[2] * 2, 128, (uint64_t)dq_str[1] * 2, (uint64_t)dq_str[0] * 2};
      if ((st = encode_map(&P.tm_dq, tdt, 5, dq, dq5, sdq, obox)) != FFPA_OK) return st;
    }
  }
  if (any_k) {
    const uint64_t dk5[5] = {64, (uint64_t)Nkv, nch, (uint64_t)Hkv, (uint64_t)B};
    const uint64_t sk[4] = {(uint64_t)k_str[2] * 2, 128, (uint64_t)k_str[1] * 2, (uint64_t)k_str[0] * 2};
    const uint64_t sv[4] = {(uint64_t)v_str[2] * 2, 128, (uint64_t)v_str[1] * 2, (uint64_t)v_str[0] * 2};
    if ((st = encode_map(&P.tm_k, tdt, 5, k, dk5, sk, box)) != FFPA_OK) return st;
    if ((st = encode_map(&P.tm_v, tdt, 5, v, dk5, sv, box)) != FFPA_OK) return st;
    if (tiles) {
      const uint32_t obox[5] = {64, 32, 1, 1, 1};
      const uint64_t sdk[4] = {(uint64_t)dk_str[2] * 2, 128, (uint64_t)dk_str[1] * 2, (uint64_t)dk_str[0] * 2};
      const uint64_t sdv[4] = {(uint64_t)dv_str[2] * 2, 128, (uint64_t)dv_str[1] * 2, (uint64_t)dv_str[0] * 2};
      if ((st = encode_map(&P.tm_dk, tdt, 5, dk, dk5, sdk, obox)) != FFPA_OK) return st;
      if ((st = encode_map(&P.tm_dv, tdt, 5, dv, dk5, sdv, obox)) != FFPA_OK) return st;
    }
  }
  P.o = o;
  P.dout = dout;
  P.lse = lse;
  P.mask = umask ? mask : nullptr;
  P.mask_kind = umask ? mask_kind : FFPA_MASK_NONE;
  for (int i = 0; i < 4; ++i) P.m_str[i] = umask ? mask_str[i] : 0;
  P.delta = delta;
  P.dq = dq;
  P.dk = dk;
  P.dv = dv;
  for (int i = 0; i < 4; ++i) {
    P.o_str[i] = o_str[i];
    P.do_str[i] = do_str[i];
    P.dq_str[i] = dq_str[i];
    P.dk_str[i] = dk_str[i];
    P.dv_str[i] = dv_str[i];
  }
  P.B = B;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.group = Hq / Hkv;
  P.Nq = Nq;
  P.Nkv = Nkv;
  P.D = D;
  P.n_qt = (Nq + BM - 1) / BM;
  P.n_kt = (Nkv + BN - 1) / BN;
  P.scale = sc;
  P.causal = is_causal ? 1 : 0;
  P.fp16 = dt == FFPA_FP16;
  P.err = err;
  P.device = dev;
  if (tiles)
    return bwd_tiles_launch(P, workspace, workspace_bytes, device_facts(dev).sms, opt,
                            reinterpret_cast<cudaStream_t>(stream));
  return bwd_launch(P, any_q, any_k, opt, reinterpret_cast<cudaStream_t>(stream));
}

ffpa_status ffpa_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        float* delta, ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                        const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                        const int64_t o_str[4], const int64_t do_str[4], const int64_t dq_str[4],
                        const int64_t dk_str[4], const int64_t dv_str[4], const void* mask,
                        ffpa_mask_kind mask_kind, const int64_t mask_str[4], const float* scale,
                        int is_causal, int enable_gqa, ffpa_stream_t stream,
                        const ffpa_options* options) {
  return ffpa_bwd_ws_ex(q, k, v, o, dout, lse, dq, dk, dv, delta, dt, B, Hq, Hkv, Nq, Nkv, D, q_str,
                        k_str, v_str, o_str, do_str, dq_str, dk_str, dv_str, mask, mask_kind, mask_str,
                        scale, is_causal, enable_gqa, nullptr, 0, stream, options);
}

size_t ffpa_bwd_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nkv, int D, int is_causal) {
  if (Hkv < 1 || Hq % Hkv != 0) return 0;
  return bwd_tiles_bytes(B, Hq, Nq, Nkv, D, is_causal ? 1 : 0);
}

ffpa_status ffpa_bwd_ws(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, float* delta, ffpa_dtype dt,
                        int B, int Hq, int Hkv, int Nq, int Nkv, int D, const int64_t q_str[4],
                        const int64_t k_str[4], const int64_t v_str[4], const int64_t o_str[4],
                        const int64_t do_str[4], const int64_t dq_str[4], const int64_t dk_str[4],
                        const int64_t dv_str[4], const void* mask, ffpa_mask_kind mask_kind,
                        const int64_t mask_str[4], const float* scale, int is_causal, int enable_gqa,
                        void* workspace, size_t workspace_bytes, ffpa_stream_t stream) {
  return ffpa_bwd_ws_ex(q, k, v, o, dout, lse, dq, dk, dv, delta, dt, B, Hq, Hkv, Nq, Nkv, D, q_str,
                        k_str, v_str, o_str, do_str, dq_str, dk_str, dv_str, mask, mask_kind, mask_str,
                        scale, is_causal, enable_gqa, workspace, workspace_bytes, stream, nullptr);
}

ffpa_status ffpa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, float* delta, ffpa_dtype dt,
                     int B, int Hq, int Hkv, int Nq, int Nkv, int D, const int64_t q_str[4],
                     const int64_t k_str[4], const int64_t v_str[4], const int64_t o_str[4],
                     const int64_t do_str[4], const int64_t dq_str[4], const int64_t dk_str[4],
                     const int64_t dv_str[4], const void* mask, ffpa_mask_kind mask_kind,
                     const int64_t mask_str[4], const float* scale, int is_causal, int enable_gqa,
                     ffpa_stream_t stream) {
  return ffpa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, delta, dt, B, Hq, Hkv, Nq, Nkv, D, q_str,
                     k_str, v_str, o_str, do_str, dq_str, dk_str, dv_str, mask, mask_kind, mask_str,
                     scale, is_causal, enable_gqa, stream, nullptr);
}

ffpa_status ffpa_bwd_varlen_ws_ex(const void* q, const void* k, const void* v, const void* o,
                                  const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                  float* delta, ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                                  const int64_t q_str[3], const int64_t k_str[3],
                                  const int64_t v_str[3], const int64_t o_str[3],
                                  const int64_t do_str[3], const int64_t dq_str[3],
                                  const int64_t dk_str[3], const int64_t dv_str[3],
                                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                                  int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                                  int enable_gqa, void* workspace, size_t workspace_bytes,
                                  ffpa_stream_t stream, const ffpa_options* options) {
  if (dt != FFPA_BF16 && dt != FFPA_FP16) return FFPA_ERR_DTYPE;
  if (Tq < 0 || Tk < 0 || Hq < 1 || Hkv < 1) return FFPA_ERR_INVALID;
  if (D < 64 || D > 1024 || D % 64 != 0) return FFPA_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return FFPA_ERR_INVALID;
  if (Hq != Hkv && !enable_gqa) return FFPA_ERR_INVALID;
  if (nseq < 1 || max_seqlen_q < 0 || max_seqlen_k < 0) return FFPA_ERR_INVALID;
  if (!cu_seqlens_q) return FFPA_ERR_INVALID;
  CallOpts opt;
  if (read_opts(options, &opt) != FFPA_OK) return FFPA_ERR_INVALID;
  const float sc = scale ? *scale : 1.0f / std::sqrt(static_cast<float>(D));
  if (!std::isfinite(sc)) return FFPA_ERR_INVALID;
  if ((Tq == 0 || max_seqlen_q == 0) && (Tk == 0 || max_seqlen_k == 0)) return FFPA_OK;
  if (!q_str || !k_str || !v_str || !o_str || !do_str || !dq_str || !dk_str || !dv_str)
    return FFPA_ERR_INVALID;
  if (!aligned_to(cu_seqlens_q, 4) || (cu_seqlens_k && !aligned_to(cu_seqlens_k, 4)))
    return FFPA_ERR_INVALID;
  const int64_t qsz[3] = {Tq, Hq, D}, ksz[3] = {Tk, Hkv, D};
  const bool any_q = Tq > 0 && max_seqlen_q > 0, any_k = Tk > 0 && max_seqlen_k > 0;
  if (any_q) {
    if (!q || !o || !dout || !dq || !lse || !delta) return FFPA_ERR_INVALID;
    if (!strides_ok(q_str, qsz, 3) || !strides_ok(o_str, qsz, 3) || !strides_ok(do_str, qsz, 3) ||
        !strides_ok(dq_str, qsz, 3))
      return FFPA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(o) || !aligned16(dout) || !aligned16(dq)) return FFPA_ERR_INVALID;
    if (!aligned_to(lse, 4) || !aligned_to(delta, 4)) return FFPA_ERR_INVALID;
  }
  if (any_k) {
    if (!k || !v || !dk || !dv) return FFPA_ERR_INVALID;
    if (!strides_ok(k_str, ksz, 3) || !strides_ok(v_str, ksz, 3) || !strides_ok(dk_str, ksz, 3) ||
        !strides_ok(dv_str, ksz, 3))
      return FFPA_ERR_INVALID;
    if (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv)) return FFPA_ERR_INVALID;
  }
  int dev = 0;
  // The stored-tile path: D = 128, 256, 384 or 512, both sides present, and a
  // workspace of at least the header and three blocks (the kernels check
  // every block index against the blocks it holds).
  const bool tiles = workspace != nullptr && (D == 128 || D == 256 || D == 384 || D == 512) && any_q && any_k &&
                     workspace_bytes >= bwd_varlen_header_bytes(nseq) + 3 * (size_t)P_TILE_BYTES;
  if (tiles && !aligned16(workspace)) return FFPA_ERR_INVALID;
  ffpa_status st = check_devices({any_q ? q : nullptr, any_q ? o : nullptr, any_q ? dout : nullptr,
                                  any_q ? dq : nullptr, any_q ? lse : nullptr, any_q ? delta : nullptr,
                                  any_k ? k : nullptr, any_k ? v : nullptr, any_k ? dk : nullptr,
                                  any_k ? dv : nullptr, cu_seqlens_q, cu_seqlens_k,
                                  tiles ? workspace : nullptr},
                                 &dev);
  if (st != FFPA_OK) return st;
  DeviceScope scope(dev);
  if (!scope.ok()) return FFPA_ERR_CUDA;
  int* err = nullptr;
  if ((st = device_status_word(dev, opt, &err)) != FFPA_OK) return st;

  BwdParams P{};
  const CUtensorMapDataType tdt =
      dt == FFPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  P.D = D;
  P.npairs = (D / DK + 1) / 2;
  P.kchunks = D / DK < 2 ? D / DK : 2;
  const uint64_t nch = (uint64_t)(D / DK);
  const uint32_t box[4] = {64, BM, (uint32_t)P.kchunks, 1};
  if (any_q) {
    const uint64_t dq4[4] = {64, (uint64_t)Tq, nch, (uint64_t)Hq};
    const uint64_t sq[3] = {(uint64_t)q_str[0] * 2, 128, (uint64_t)q_str[1] * 2};
    const uint64_t sd[3] = {(uint64_t)do_str[0] * 2, 128, (uint64_t)do_str[1] * 2};
    if ((st = encode_map(&P.tm_q, tdt, 4, q, dq4, sq, box)) != FFPA_OK) return st;
    if ((st = encode_map(&P.tm_do, tdt, 4, dout, dq4, sd, box)) != FFPA_OK) return st;
  }
  if (any_k) {
    const uint64_t dk4[4] = {64, (uint64_t)Tk, nch, (uint64_t)Hkv};
    const uint64_t sk[3] = {(uint64_t)k_str[0] * 2, 128, (uint64_t)k_str[1] * 2};
    const uint64_t sv[3] = {(uint64_t)v_str[0] * 2, 128, (uint64_t)v_str[1] * 2};
    if ((st = encode_map(&P.tm_k, tdt, 4, k, dk4, sk, box)) != FFPA_OK) return st;
    if ((st = encode_map(&P.tm_v, tdt, 4, v, dk4, sv, box)) != FFPA_OK) return st;
  }
  P.o = o;
  P.dout = dout;
  P.lse = lse;
  P.delta = delta;
  P.dq = dq;
  P.dk = dk;
  P.dv = dv;
  for (int i = 0; i < 3; ++i) {
    P.o_str[i] = o_str[i];
    P.do_str[i] = do_str[i];
    P.dq_str[i] = dq_str[i];
    P.dk_str[i] = dk_str[i];
    P.dv_str[i] = dv_str[i];
  }
  P.mask = nullptr;
  P.mask_kind = FFPA_MASK_NONE;
  P.varlen = 1;
  P.Tq = Tq;
  P.cu_q = cu_seqlens_q;
  P.cu_k = cu_seqlens_k ? cu_seqlens_k : cu_seqlens_q;
  P.B = nseq;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.group = Hq / Hkv;
  P.Nq = max_seqlen_q;
  P.Nkv = max_seqlen_k;
  P.n_qt = (max_seqlen_q + BM - 1) / BM;
  P.n_kt = (max_seqlen_k + BN - 1) / BN;
  P.scale = sc;
  P.causal = causal ? 1 : 0;
  P.fp16 = dt == FFPA_FP16;
  P.err = err;
  P.device = dev;
  if (tiles)
    return bwd_tiles_launch(P, workspace, workspace_bytes, device_facts(dev).sms, opt,
                            reinterpret_cast<cudaStream_t>(stream));
  return bwd_launch(P, any_q, any_k, opt, reinterpret_cast<cudaStream_t>(stream));
}

ffpa_status ffpa_bwd_varlen_ex(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               float* delta, ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                               const int64_t q_str[3], const int64_t k_str[3],
                               const int64_t v_str[3], const int64_t o_str[3],
                               const int64_t do_str[3], const int64_t dq_str[3],
                               const int64_t dk_str[3], const int64_t dv_str[3],
                               const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                               int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                               int enable_gqa, ffpa_stream_t stream, const ffpa_options* options) {
  return ffpa_bwd_varlen_ws_ex(q, k, v, o, dout, lse, dq, dk, dv, delta, dt, Tq, Tk, Hq, Hkv, D, q_str, k_str,
                               v_str, o_str, do_str, dq_str, dk_str, dv_str, cu_seqlens_q, cu_seqlens_k, nseq,
                               max_seqlen_q, max_seqlen_k, scale, causal, enable_gqa, nullptr, 0, stream,
                               options);
}

size_t ffpa_bwd_varlen_workspace_bytes(const int32_t* cu_seqlens_q_host, const int32_t* cu_seqlens_k_host,
                                       int nseq, int Hq, int Hkv, int D, int is_causal) {
  if (Hkv < 1 || Hq % Hkv != 0) return 0;
  return bwd_varlen_tiles_bytes(cu_seqlens_q_host, cu_seqlens_k_host, nseq, Hq, D, is_causal ? 1 : 0);
}

ffpa_status ffpa_bwd_varlen_ws(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               float* delta, ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                               const int64_t q_str[3], const int64_t k_str[3],
                               const int64_t v_str[3], const int64_t o_str[3],
                               const int64_t do_str[3], const int64_t dq_str[3],
                               const int64_t dk_str[3], const int64_t dv_str[3],
                               const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                               int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                               int enable_gqa, void* workspace, size_t workspace_bytes,
                               ffpa_stream_t stream) {
  return ffpa_bwd_varlen_ws_ex(q, k, v, o, dout, lse, dq, dk, dv, delta, dt, Tq, Tk, Hq, Hkv, D, q_str, k_str,
                               v_str, o_str, do_str, dq_str, dk_str, dv_str, cu_seqlens_q, cu_seqlens_k, nseq,
                               max_seqlen_q, max_seqlen_k, scale, causal, enable_gqa, workspace,
                               workspace_bytes, stream, nullptr);
}

ffpa_status ffpa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            float* delta, ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                            const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                            const int64_t o_str[3], const int64_t do_str[3], const int64_t dq_str[3],
                            const int64_t dk_str[3], const int64_t dv_str[3],
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                            int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                            int enable_gqa, ffpa_stream_t stream) {
  return ffpa_bwd_varlen_ex(q, k, v, o, dout, lse, dq, dk, dv, delta, dt, Tq, Tk, Hq, Hkv, D, q_str,
                            k_str, v_str, o_str, do_str, dq_str, dk_str, dv_str, cu_seqlens_q,
                            cu_seqlens_k, nseq, max_seqlen_q, max_seqlen_k, scale, causal,
                            enable_gqa, stream, nullptr);
}

ffpa_status ffpa_fwd_varlen_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                               ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                               const int64_t q_str[3], const int64_t k_str[3],
                               const int64_t v_str[3], const int64_t o_str[3],
                               const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                               int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                               int enable_gqa, ffpa_stream_t stream, const ffpa_options* options) {
  if (dt != FFPA_BF16 && dt != FFPA_FP16) return FFPA_ERR_DTYPE;
  if (Tq < 0 || Tk < 0 || Hq < 1 || Hkv < 1) return FFPA_ERR_INVALID;
  if (D < 64 || D > 1024 || D % 64 != 0) return FFPA_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return FFPA_ERR_INVALID;
  if (Hq != Hkv && !enable_gqa) return FFPA_ERR_INVALID;
  if (nseq < 1 || max_seqlen_q < 0 || max_seqlen_k < 0) return FFPA_ERR_INVALID;
  if (!cu_seqlens_q) return FFPA_ERR_INVALID;
  CallOpts opt;
  if (read_opts(options, &opt) != FFPA_OK) return FFPA_ERR_INVALID;
  const float sc = scale ? *scale : 1.0f / std::sqrt(static_cast<float>(D));
  if (!std::isfinite(sc)) return FFPA_ERR_INVALID;
  if (Tq == 0 || max_seqlen_q == 0) return FFPA_OK;   // nothing to read or write
  if (!q || !o || !q_str || !k_str || !v_str || !o_str) return FFPA_ERR_INVALID;
  if (Tk > 0 && (!k || !v)) return FFPA_ERR_INVALID;
  if (!aligned_to(cu_seqlens_q, 4) || (cu_seqlens_k && !aligned_to(cu_seqlens_k, 4)))
    return FFPA_ERR_INVALID;
  const int64_t qsz[3] = {Tq, Hq, D}, ksz[3] = {Tk, Hkv, D};
  if (!strides_ok(q_str, qsz, 3) || !strides_ok(o_str, qsz, 3)) return FFPA_ERR_INVALID;
  if (Tk > 0 && (!strides_ok(k_str, ksz, 3) || !strides_ok(v_str, ksz, 3))) return FFPA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(o) || (Tk > 0 && (!aligned16(k) || !aligned16(v))))
    return FFPA_ERR_INVALID;
  if (lse && !aligned_to(lse, 4)) return FFPA_ERR_INVALID;
  int dev = 0;
  ffpa_status st = check_devices({q, o, Tk > 0 ? k : nullptr, Tk > 0 ? v : nullptr, lse,
                                  cu_seqlens_q, cu_seqlens_k},
                                 &dev);
  if (st != FFPA_OK) return st;
  DeviceScope scope(dev);
  if (!scope.ok()) return FFPA_ERR_CUDA;
  int* err = nullptr;
  if ((st = device_status_word(dev, opt, &err)) != FFPA_OK) return st;

  Params P{};
  const CUtensorMapDataType tdt =
      dt == FFPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const Kern kn = choose_kernel(D, true, opt.kernel);
  const bool pair = kn == Kern::PAIR;
  const size_t smem = plan_for(kn, D, &P);
  const uint32_t k_rows = pair ? BN / 2 : BN;
  const uint32_t k_box_chunks = pair ? (uint32_t)P.kc : (uint32_t)P.kchunks;
  const uint64_t nch = (uint64_t)(D / DK);   // real chunks (see ffpa_fwd_ex)
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
  if (kn == Kern::SPLIT && P.split_c == 2 && P.q_res && Tq > 0) {
    // The column-split pair kernel stores the O tiles that lie inside their
    // sequence through 32-row boxes of the packed rows.
    const uint64_t dq[4] = {64, (uint64_t)Tq, nch, (uint64_t)Hq};
    const uint64_t so[3] = {(uint64_t)o_str[0] * 2, 128, (uint64_t)o_str[1] * 2};
    const uint32_t bo[4] = {64, 32, 1, 1};
    if ((st = encode_map(&P.tm_o, tdt, 4, o, dq, so, bo)) != FFPA_OK) return st;
    P.o_tma = 1;
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
  P.inject = opt.drop;
  P.timeout_ns = opt.timeout_ns;
  P.err = err;
  P.device = dev;
  (void)max_seqlen_k;
  const long long items = (long long)nseq * Hq * P.n_qt * P.n_slices;
  if (items > 0x7fffffffLL) return FFPA_ERR_INVALID;
  return launch_kernel(kn, true, P, static_cast<int>(items), smem,
                       reinterpret_cast<cudaStream_t>(stream));
}

ffpa_status ffpa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            ffpa_dtype dt, int Tq, int Tk, int Hq, int Hkv, int D,
                            const int64_t q_str[3], const int64_t k_str[3],
                            const int64_t v_str[3], const int64_t o_str[3],
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                            int max_seqlen_q, int max_seqlen_k, const float* scale, int causal,
                            int enable_gqa, ffpa_stream_t stream) {
  return ffpa_fwd_varlen_ex(q, k, v, o, lse, dt, Tq, Tk, Hq, Hkv, D, q_str, k_str, v_str, o_str,
                            cu_seqlens_q, cu_seqlens_k, nseq, max_seqlen_q, max_seqlen_k, scale,
                            causal, enable_gqa, stream, nullptr);
}

size_t ffpa_fwd_fp8_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nkv, int D) {
  if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nkv < 0 || D < 128 || D > 1024 || D % 128 != 0)
    return 0;
  return fp8_layout(B, Hq, Hkv, Nq, Nkv, D).total;
}

ffpa_status ffpa_fwd_fp8_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                            ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                            const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                            const int64_t o_str[4], const void* mask, ffpa_mask_kind mask_kind,
                            const int64_t mask_str[4], const float* scale, int is_causal,
                            int enable_gqa, void* workspace, size_t workspace_bytes,
                            ffpa_stream_t stream, const ffpa_options* options) {
  if (dt != FFPA_BF16 && dt != FFPA_FP16) return FFPA_ERR_DTYPE;
  if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nkv < 0) return FFPA_ERR_INVALID;
  if (D < 128 || D > 1024 || D % 128 != 0) return FFPA_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return FFPA_ERR_INVALID;
  if (Hq != Hkv && !enable_gqa) return FFPA_ERR_INVALID;
  if (is_causal && Nkv < Nq) return FFPA_ERR_INVALID;
  if (mask_kind < FFPA_MASK_NONE || mask_kind > FFPA_MASK_ADD_QTYPE) return FFPA_ERR_INVALID;
  CallOpts opt;
  if (read_opts(options, &opt) != FFPA_OK) return FFPA_ERR_INVALID;
  const float sc = scale ? *scale : 1.0f / std::sqrt(static_cast<float>(D));
  if (!std::isfinite(sc)) return FFPA_ERR_INVALID;
  if (B == 0 || Nq == 0) return FFPA_OK;          // nothing to read or write
  if (!q || !o || !q_str || !k_str || !v_str || !o_str) return FFPA_ERR_INVALID;
  if (Nkv > 0 && (!k || !v)) return FFPA_ERR_INVALID;
  const bool umask = mask_kind != FFPA_MASK_NONE && Nkv > 0;
  if (umask) {
    if (!mask || !mask_str) return FFPA_ERR_INVALID;
    for (int i = 0; i < 4; ++i)
      if (mask_str[i] < 0) return FFPA_ERR_INVALID;
    if (!aligned_to(mask, mask_esz(mask_kind))) return FFPA_ERR_INVALID;
  }
  const int64_t qsz[4] = {B, Hq, Nq, D}, ksz[4] = {B, Hkv, Nkv, D};
  if (!strides_ok(q_str, qsz, 4) || !strides_ok(o_str, qsz, 4)) return FFPA_ERR_INVALID;
  if (Nkv > 0 && (!strides_ok(k_str, ksz, 4) || !strides_ok(v_str, ksz, 4))) return FFPA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(o) || (Nkv > 0 && (!aligned16(k) || !aligned16(v))))
    return FFPA_ERR_INVALID;
  if (lse && !aligned_to(lse, 4)) return FFPA_ERR_INVALID;
  const Fp8Layout L = fp8_layout(B, Hq, Hkv, Nq, Nkv, D);
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < L.total) return FFPA_ERR_INVALID;
  int dev = 0;
  ffpa_status st = check_devices({q, o, Nkv > 0 ? k : nullptr, Nkv > 0 ? v : nullptr, lse,
                                  umask ? mask : nullptr, workspace},
                                 &dev);
  if (st != FFPA_OK) return st;
  DeviceScope scope(dev);
  if (!scope.ok()) return FFPA_ERR_CUDA;
  int* err = nullptr;
  if ((st = device_status_word(dev, opt, &err)) != FFPA_OK) return st;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Fp8Quant Z{};
  const void* srcs[3] = {q, k, v};
  const int64_t* strs[3] = {q_str, k_str, v_str};
  const int Hs[3] = {Hq, Hkv, Hkv}, Ns[3] = {Nq, Nkv, Nkv};
  long long ctas = 0;
  for (int t = 0; t < 3; ++t) {
    Z.src[t] = srcs[t];
    for (int i = 0; i < 4; ++i) Z.str[t][i] = strs[t][i];
    Z.codes[t] = ws + L.off[t];
    Z.scales[t] = reinterpret_cast<float*>(ws + L.off[3 + t]);
    Z.H[t] = Hs[t];
    Z.N[t] = Ns[t];
    Z.npad[t] = static_cast<int>(t == 0 ? L.nqp : L.nkp);
    Z.nblk[t] = t == 0 ? L.nqb : L.nkb;
    ctas += (long long)B * Hs[t] * Z.nblk[t];
    Z.cta_end[t] = ctas;
  }
  Z.B = B;
  Z.D = D;
  Z.fp16 = dt == FFPA_FP16;
  if (ctas > 0x7fffffffLL) return FFPA_ERR_INVALID;

  Params P{};
  P.nchunks = D / DK;                        // 64-column units: output slices
  P.n_slices = (D + DV_MAX - 1) / DV_MAX;
  int dv_max = 0;
  for (int sl = 0; sl < P.n_slices; ++sl) {
    const int w = ((sl + 1) * P.nchunks / P.n_slices - sl * P.nchunks / P.n_slices) * DK;
    dv_max = w > dv_max ? w : dv_max;
  }
  const int nch8 = D / 128;
  // Column split (a pair of CTAs per 128-row tile, each owning D/2 output
  // columns; S once per key tile) where D/2 fits beside S in TMEM and the
  // single-CTA FP8 kernel would recompute S (D = 384, 512; measured at
  // D=512: 1024 vs 957 TFLOPS, at D=256, where the single-CTA kernel has
  // one slice: 649 vs 878).  FFPA_VARIANT_SPLIT also takes D = 256;
  // FFPA_VARIANT_SINGLE forces the single-CTA kernel.
  const bool fsplit = opt.kernel == FFPA_VARIANT_SPLIT ? (D == 256 || D == 384 || D == 512)
                      : opt.kernel == FFPA_VARIANT_SINGLE ? false
                                                          : (D == 384 || D == 512);
  size_t smem = 0;
  if (fsplit) {
    // Q resident (32 KB boxes of two 128-byte chunks), two e4m3 P tiles,
    // a ring of 32 KB stages.
    P.n_slices = 1;
    dv_max = D / 2;
    const size_t q_region = (size_t)((nch8 + 1) / 2) * SLOT_BYTES;
    const size_t p_tiles = 2 * (size_t)BM * BN;
    size_t ns = (SMEM_LIMIT - SPLIT_STATIC_RESERVE - 1024 - q_region - p_tiles) / SLOT_BYTES;
    if (ns > (size_t)NSLOT_MAX) ns = NSLOT_MAX;
    if (ns < 3) return FFPA_ERR_UNSUPPORTED;
    P.nslot = static_cast<int>(ns);
    P.split_c = 2;
    smem = 1024 + q_region + p_tiles + ns * SLOT_BYTES;
  } else {
    const bool qres = nch8 <= 4;
    const size_t q_region = qres ? (size_t)((nch8 + 1) / 2) * SLOT_BYTES : 0;
    P.vslot = dv_max * 128;
    P.nslot_v = NSLOT_V_MAX;
    size_t ns = (SMEM_LIMIT - SMEM_STATIC_RESERVE - 1024 - q_region - (size_t)P.nslot_v * P.vslot) / SLOT_BYTES;
    if (ns > (size_t)NSLOT_MAX) ns = NSLOT_MAX;
    if (ns < 2) return FFPA_ERR_UNSUPPORTED;
    P.nslot = static_cast<int>(ns);
    smem = 1024 + q_region + ns * SLOT_BYTES + (size_t)P.nslot_v * P.vslot;
  }
  const uint32_t box_ch = nch8 >= 2 ? 2u : 1u;
  {
    const uint64_t dq[5] = {128, (uint64_t)L.nqp, (uint64_t)nch8, (uint64_t)Hq, (uint64_t)B};
    const uint64_t sq[4] = {(uint64_t)D, 128, (uint64_t)(L.nqp * D), (uint64_t)(Hq * L.nqp * D)};
    const uint32_t bq[5] = {128, BM, box_ch, 1, 1};
    if ((st = encode_map(&P.tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, ws + L.off[0], dq, sq, bq)) != FFPA_OK)
      return st;
  }
  if (Nkv > 0) {
    const uint64_t dk[5] = {128, (uint64_t)L.nkp, (uint64_t)nch8, (uint64_t)Hkv, (uint64_t)B};
    const uint64_t sk[4] = {(uint64_t)D, 128, (uint64_t)(L.nkp * D), (uint64_t)(Hkv * L.nkp * D)};
    const uint32_t bk[5] = {128, BN, box_ch, 1, 1};
    if ((st = encode_map(&P.tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, ws + L.off[1], dk, sk, bk)) != FFPA_OK)
      return st;
    const uint64_t dv4[4] = {(uint64_t)L.nkp, (uint64_t)D, (uint64_t)Hkv, (uint64_t)B};
    const uint64_t sv[3] = {(uint64_t)L.nkp, (uint64_t)(D * L.nkp), (uint64_t)(Hkv * D * L.nkp)};
    const uint32_t bv[4] = {128, (uint32_t)dv_max, 1, 1};
    if ((st = encode_map(&P.tm_v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, ws + L.off[2], dv4, sv, bv)) != FFPA_OK)
      return st;
  }
  P.o = o;
  P.lse = lse;
  P.mask = umask ? mask : nullptr;
  P.mask_kind = umask ? mask_kind : FFPA_MASK_NONE;
  for (int i = 0; i < 4; ++i) {
    P.o_str[i] = o_str[i];
    P.m_str[i] = umask ? mask_str[i] : 0;
  }
  P.B = B;
  P.Hq = Hq;
  P.group = Hq / Hkv;
  P.Nq = Nq;
  P.Nkv = Nkv;
  P.D = D;
  P.n_qt = L.nqb;
  P.n_kb = L.nkb;
  P.sq = reinterpret_cast<const float*>(ws + L.off[3]);
  P.sk = reinterpret_cast<const float*>(ws + L.off[4]);
  P.sv = reinterpret_cast<const float*>(ws + L.off[5]);
  P.scale_log2 = sc * 1.4426950408889634f;
  P.causal = is_causal ? 1 : 0;
  P.fp16 = dt == FFPA_FP16;
  P.inject = opt.drop;
  P.timeout_ns = opt.timeout_ns;
  P.err = err;
  P.device = dev;
  const long long items = (long long)B * Hq * P.n_qt * P.n_slices;
  if (items > 0x7fffffffLL) return FFPA_ERR_INVALID;
  return launch_fp8(Z, P, static_cast<int>(items), smem, fsplit, reinterpret_cast<cudaStream_t>(stream));
}

ffpa_status ffpa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                         ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                         const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                         const int64_t o_str[4], const void* mask, ffpa_mask_kind mask_kind,
                         const int64_t mask_str[4], const float* scale, int is_causal,
                         int enable_gqa, void* workspace, size_t workspace_bytes,
                         ffpa_stream_t stream) {
  return ffpa_fwd_fp8_ex(q, k, v, o, lse, dt, B, Hq, Hkv, Nq, Nkv, D, q_str, k_str, v_str, o_str,
                         mask, mask_kind, mask_str, scale, is_causal, enable_gqa, workspace,
                         workspace_bytes, stream, nullptr);
}

}  // extern "C"
