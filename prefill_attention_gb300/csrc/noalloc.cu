// noalloc.cu -- a paged-decode entry point that allocates nothing, for callers that cannot
// hand the library a workspace.
//
// Split-KV decode needs scratch memory for its per-split partials (o_part, ml_part).  The
// regular entry point takes that scratch from the caller.  Some callers cannot provide
// it: an operator running inside an inference runtime whose memory planner owns every
// device byte and only forwards inputs and outputs, or a process that must not grow its
// device memory after start-up.  For them this file compiles a fixed scratch array into
// the library (every GPU that loads the library holds it until the process exits) and
// runs the regular decode on it.
//
// Rules of use:
//   * The first call on a device resolves the array's device address with
//     cudaGetSymbolAddress while that device is current; make that first call before any
//     stream capture.
//   * All calls share the one array, so calls that overlap on the GPU (different streams,
//     or different host threads without ordering) race on it; serialise them.
//   * The array keeps the previous call's contents; nothing in it needs to start at zero
//     because every partial the combine reads is written by the same call (a split kernel
//     that gives up writes its partials as NaN, and reports it in the status word).
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "astr_attn.h"
#include "astr_attn_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB of partials per process and device
using astr::kMaxDevices;

__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (resolved once per device).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ASTR_ERR_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return ASTR_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return ASTR_ERR_DEVICE;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ASTR_OK;
}

}  // namespace

extern "C" {

int astr_attn_paged_decode_noalloc(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                                   const int32_t* req_to_token, const int32_t* seq_lens, const int32_t* kv_indptr,
                                   uint16_t* out, const astr_attn_dims* dims, float sm_scale, void* stream) {
  // the argument checks of astr_attn_paged_decode, in its order, come first, so both entry
  // points return the same status for the same arguments (an empty batch included)
  if (!q || !k_pool || !v_pool || !req_to_token || !seq_lens || !kv_indptr || !out) return ASTR_ERR_INVALID_ARG;
  const auto misaligned = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a != 0; };
  if (misaligned(q, 16) || misaligned(k_pool, 16) || misaligned(v_pool, 16) || misaligned(out, 16) ||
      misaligned(req_to_token, 4) || misaligned(seq_lens, 4) || misaligned(kv_indptr, 4))
    return ASTR_ERR_MISALIGNED;
  if (dims == nullptr) return ASTR_ERR_INVALID_ARG;
  size_t o_bytes = 0, ml_bytes = 0;
  int st = astr_attn_decode_workspace_bytes(dims, &o_bytes, &ml_bytes);
  if (st != ASTR_OK) return st;
  const size_t ml_off = (o_bytes + 255) & ~size_t(255);
  if (ml_off + ml_bytes > kScratchBytes) return ASTR_ERR_WORKSPACE_TOO_SMALL;
  void* base = nullptr;
  if ((st = scratch_for_current_device(&base)) != ASTR_OK) return st;
  float* o_part = static_cast<float*>(base);
  float* ml_part = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + ml_off);
  return astr_attn_paged_decode(q, k_pool, v_pool, req_to_token, seq_lens, kv_indptr, o_part, ml_part, out, dims,
                                sm_scale, stream);
}

}  // extern "C"
