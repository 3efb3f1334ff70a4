// ffpa_bwd_noalloc: the dense backward for callers that cannot allocate
// device memory.  The backward needs one fp32 value per query row between
// its first kernel and the gradient kernels (delta = rowsum(dO * O)); the
// plain ffpa_bwd takes that buffer from the caller.  Here it lives in a
// fixed array inside the library instead, so the caller passes only the
// inputs and the three gradient outputs.
#include <cuda_runtime.h>

#include <mutex>

#include "ffpa_common.cuh"

namespace {

constexpr int MAX_DEVICES = 64;

// The scratch rows of every call on a device.  Every GPU that loads the
// library holds this array (4 MiB) until the process exits.
static __device__ __align__(256) float g_bwd_delta_scratch[FFPA_BWD_NOALLOC_MAX_ROWS];

struct Scratch {
  std::once_flag once;
  float* ptr = nullptr;   // device address of g_bwd_delta_scratch on this device
};
Scratch g_scratch[MAX_DEVICES];

// Device address of the array on `dev`, looked up once per device with that
// device current (the host-side name of the array is only a stand-in, not
// an address a kernel may use).  NULL if the lookup failed.
float* scratch_on(int dev) {
  Scratch& s = g_scratch[dev];
  std::call_once(s.once, [&] {
    ffpa::DeviceScope scope(dev);
    if (!scope.ok()) return;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_delta_scratch) == cudaSuccess)
      s.ptr = static_cast<float*>(p);
    else
      cudaGetLastError();
  });
  return s.ptr;
}

}  // namespace

extern "C" ffpa_status ffpa_bwd_noalloc(
    const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
    void* dq, void* dk, void* dv, ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
    const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4], const int64_t o_str[4],
    const int64_t do_str[4], const int64_t dq_str[4], const int64_t dk_str[4],
    const int64_t dv_str[4], const void* mask, ffpa_mask_kind mask_kind, const int64_t mask_str[4],
    const float* scale, int is_causal, int enable_gqa, ffpa_stream_t stream) {
  if (B < 0 || Hq < 1 || Nq < 0) return FFPA_ERR_INVALID;
  const long long rows = (long long)B * Hq * Nq;
  if (rows > FFPA_BWD_NOALLOC_MAX_ROWS) return FFPA_ERR_INVALID;   // beyond the fixed scratch
  float* delta = nullptr;
  if (rows > 0) {
    // The scratch of the device that holds q (the plain entry point then
    // checks that every other pointer lives there too).
    cudaPointerAttributes attr;
    if (!q || cudaPointerGetAttributes(&attr, q) != cudaSuccess) {
      cudaGetLastError();
      return q ? FFPA_ERR_CUDA : FFPA_ERR_INVALID;
    }
    if ((attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) ||
        attr.device < 0 || attr.device >= MAX_DEVICES)
      return FFPA_ERR_INVALID;
    delta = scratch_on(attr.device);
    if (!delta) return FFPA_ERR_CUDA;
  }
  return ffpa_bwd(q, k, v, o, dout, lse, dq, dk, dv, delta, dt, B, Hq, Hkv, Nq, Nkv, D, q_str,
                  k_str, v_str, o_str, do_str, dq_str, dk_str, dv_str, mask, mask_kind, mask_str,
                  scale, is_causal, enable_gqa, stream);
}
