// append.cu -- the KV-append step: every new token's K and V rows (all KV heads) are copied
// into the pool slot that the slot table assigns to its position.
//
// Source: AstrAI commit page "astrai/extension/attention_backend.py @47b3ed4",
// write-then-gather helper commit: the backends write the new tokens' K/V into the pool and
// then gather the request's keys from it.  New token i of request b (flat row
// r = qo_indptr[b] + i) is key position c_b + i, c_b = seq_len_b - q_len_b (the same causal
// offset the prefill uses), so it lands in slot req_to_token[b * r2t_stride + c_b + i].
//
// Pure data movement, HBM bound: algorithmic bytes = 4 * total_q * Hkv * d * 2 (read the new
// K and V rows, write them into the pool); every slot row [Hkv, d] is contiguous in both
// arrays, so each token is two contiguous reads and two contiguous writes.  One warp per
// new token.  The warp's 16-byte loads of its K and V rows depend on nothing, so they are
// issued first; the request lookup (a 32-way search of qo_indptr, one ballot per round: one
// round for up to 32 requests, two up to 1024) and the slot-id read run while those loads
// are in flight, then the stores follow.  Rows wider than 32 lanes x kVecPerLane vectors
// (Hkv * d > 1024) continue in further rounds of loads and stores.
#include <cstdint>

#include <cuda_runtime.h>

#include "astr_attn_internal.h"
#include "common.cuh"

namespace astr {
namespace {

constexpr int kAppendWarps = 8;   // new tokens per CTA (one warp each)
constexpr int kVecPerLane = 4;    // 16-byte vectors per lane per tensor per round

// Read-once input rows: no L1 allocation, and first to leave L2 under `policy` (an
// evict-first access policy), so the pool rows written next stay there for the attention
// kernel that reads them.
__device__ __forceinline__ uint4 ld_stream128(const uint4* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void st128(uint4* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// The request that owns flat row r: the largest b in [0, B) with qo_indptr[b] <= r.  Every
// lane returns the same b.  Only qo_indptr[0 .. B-1] is read, whatever its contents.
__device__ __forceinline__ int request_of_row(const int32_t* qo_indptr, int B, int r, int lane) {
  int lo = 0, n = B;
  while (n > 1) {
    const int step = (n + 31) >> 5;
    const int off = lane * step;
    const bool le = off < n && __ldg(qo_indptr + lo + off) <= r;
    const unsigned m = __ballot_sync(kFullMask, le);
    const int k = m ? 31 - __clz(m) : 0;
    lo += k * step;
    n = min(step, n - k * step);
  }
  return lo;
}

__global__ void __launch_bounds__(kAppendWarps * 32) kv_append_kernel(const AppendParams p) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  if (r >= p.total_q) return;  // warp-uniform
  const int nvec = p.row_vecs;
  const uint64_t once = evict_first_policy();
  const uint4* ks = reinterpret_cast<const uint4*>(p.k_new) + (size_t)r * nvec;
  const uint4* vs = reinterpret_cast<const uint4*>(p.v_new) + (size_t)r * nvec;
  uint4 kr[kVecPerLane], vr[kVecPerLane];
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    const int v = lane + 32 * j;
    if (v < nvec) {
      kr[j] = ld_stream128(ks + v, once);
      vr[j] = ld_stream128(vs + v, once);
    }
  }
  const int b = request_of_row(p.qo_indptr, p.batch, r, lane);
  const int q0 = __ldg(p.qo_indptr + b), q1 = __ldg(p.qo_indptr + b + 1);
  const int64_t pos = (int64_t)__ldg(p.seq_lens + b) - ((int64_t)q1 - q0) + ((int64_t)r - q0);
  int64_t slot = -1;
  if (pos >= 0 && pos < p.r2t_stride) slot = __ldg(p.req_to_token + (size_t)b * p.r2t_stride + pos);
  if (slot < 0 || slot >= p.num_slots) {  // warp-uniform: ids outside the pool are skipped and reported
    if (lane == 0 && p.status != nullptr) atomicOr(p.status, kStatusBadInput);
    return;
  }
  uint4* kd = reinterpret_cast<uint4*>(p.k_pool) + (size_t)slot * nvec;
  uint4* vd = reinterpret_cast<uint4*>(p.v_pool) + (size_t)slot * nvec;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    const int v = lane + 32 * j;
    if (v < nvec) {
      st128(kd + v, kr[j]);
      st128(vd + v, vr[j]);
    }
  }
  for (int base = 32 * kVecPerLane; base < nvec; base += 32 * kVecPerLane) {
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
      const int v = base + lane + 32 * j;
      if (v < nvec) {
        kr[j] = ld_stream128(ks + v, once);
        vr[j] = ld_stream128(vs + v, once);
      }
    }
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
      const int v = base + lane + 32 * j;
      if (v < nvec) {
        st128(kd + v, kr[j]);
        st128(vd + v, vr[j]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream) {
  if (p.total_q <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)((p.total_q + kAppendWarps - 1) / kAppendWarps);
  kv_append_kernel<<<grid, kAppendWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace astr
