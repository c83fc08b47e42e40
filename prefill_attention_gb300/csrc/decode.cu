// decode.cu -- split-KV paged decode for sm_103a: split kernel + log-sum-exp combine.
//
// Method (AstrAI commit log, page "astrai/extension @6f67ba8"):
//   * CUDA-backend commit: req_to_token is the page table with one token per page, so
//     every key row is gathered through its own slot id.
//   * kernel-rename commit: decode is split-KV only; each split writes an unnormalised
//     partial plus its (max, sum) pair and a shared combine kernel merges them.
//   * split-partials commit: the partial buffers are not cleared, because every split
//     writes every slot it owns -- so empty splits here write (m=-inf, l=0, o=0).
//   * pipeline commit: several tile loads stay in flight while an older tile is used.
//
// GB300 design (not the pages' sm_89 design):
//   grid (split, kv_head, request); 4 warps per CTA, each warp streams a contiguous share
//   of the split's keys through its own 4-stage cp.async ring (8 keys per stage, K and V
//   rows of 16-byte chunks, zero-filled past the end), so no CTA-wide barrier sits in the
//   key loop.  All G query heads of a KV head are served from each K/V row load.
//   Scores: each lane multiplies its slice of the row with its slice of the G query rows
//   (packed fp32x2 FMAs), then a transpose-reduction across the lanes of a row leaves one
//   finished score per lane.  Online softmax in base 2 (the scale carries log2 e) with a
//   warp vote that skips the accumulator rescale when no running max moved.
//   Warps merge in shared memory at the end and write one partial per (head, split).
#include <cuda_runtime.h>
#include <math_constants.h>

#include "common.cuh"

namespace astr {
namespace {

template <int D, int G>
struct DecodeCfg {
  static constexpr int EPL = (D == 128 && G <= 4) ? 16 : 8;  // elements per lane per row
  static constexpr int CPL = EPL / 8;                          // 16-byte chunks per lane per row
  static constexpr int CPR = D / 8;                            // 16-byte chunks per row
  static constexpr int LPR = D / EPL;                          // lanes sharing one row
  static constexpr int RPI = 32 / LPR;                         // rows a warp covers per load
  static constexpr int TPS = 8;                                // keys per warp stage
  static constexpr int NT = TPS / RPI;                         // keys per lane per stage
  static constexpr int NV = NT * G;                            // partial scores per lane
  static constexpr int NF = NV >= LPR ? NV / LPR : 1;          // finished scores per lane
  static constexpr int NW = 4;                                 // warps per CTA
  static constexpr int STAGES = 4;
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int KV_BYTES = TPS * ROW_BYTES;             // one K (or V) stage tile
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;      // per warp
  static constexpr int PS_BYTES = (TPS * G + G) * 4;           // per warp: p[TPS][G], alpha[G]
  static constexpr int RED_BYTES = NW * RPI * G * D * 4;       // end-of-CTA merge buffer
  static constexpr int MAIN_BYTES = NW * RING_BYTES > RED_BYTES ? NW * RING_BYTES : RED_BYTES;
  static constexpr int SMEM_BYTES = MAIN_BYTES + NW * PS_BYTES + NW * G * 2 * 4;
  static constexpr int LOADS_PER_LANE = 2 * TPS * CPR / 32;    // cp.async per lane per stage
  static_assert(NT >= 1 && NT * RPI == TPS, "stage must cover whole row groups");
  static_assert(LPR * CPL == CPR, "lanes x chunks must cover a row");
  static_assert((2 * TPS * CPR) % 32 == 0, "stage copies must split evenly over the warp");
};

// Transpose-reduction over the LPR lanes of a row group.  Input: v[0..N) partial sums in
// every lane.  Each step pairs the lower and upper halves of the live values; the lane whose
// step bit is set keeps the upper half and receives its partner's copy of it.  After the
// steps the lane holds N/LPR finished sums (or 1, replicated, when N < LPR).
template <int N, int M>
struct TReduce {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (M >= 1) {
      if constexpr (N >= 2) {
        const bool up = (lane & M) != 0;
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
          const float send = up ? v[i] : v[i + N / 2];
          const float keep = up ? v[i + N / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(kFullMask, send, M);
        }
        TReduce<N / 2, M / 2>::run(v, lane);
      } else {
        v[0] += __shfl_xor_sync(kFullMask, v[0], M);
        TReduce<1, M / 2>::run(v, lane);
      }
    }
  }
};

// Which lane bits decide the head of a finished score (the "head mask"), and which mark
// replicas (lanes holding copies of the same score).  Everything else distinguishes keys.
template <int D, int G>
struct LaneRoles {
  using C = DecodeCfg<D, G>;
  static constexpr unsigned compute_head_mask() {
    unsigned mask = 0;
    int n = C::NV;
    for (int m = C::LPR / 2; m >= 1; m /= 2) {
      if (n >= 2) {
        if (n / 2 < G) mask |= (unsigned)m;  // this step chose an index bit below log2(G)
        n /= 2;
      }
    }
    return mask;
  }
  static constexpr unsigned compute_replica_mask() {
    unsigned mask = 0;
    int n = C::NV;
    for (int m = C::LPR / 2; m >= 1; m /= 2) {
      if (n >= 2) n /= 2; else mask |= (unsigned)m;
    }
    return mask;
  }
  static constexpr unsigned kHead = compute_head_mask();
  static constexpr unsigned kReplica = compute_replica_mask();
  static constexpr unsigned kKey = 31u & ~kHead & ~kReplica;  // lane bits that select keys
};

// Butterfly over the lane bits in MASK (compile-time), max or sum.
template <unsigned MASK, bool IS_MAX>
__device__ __forceinline__ float butterfly(float x) {
#pragma unroll
  for (int m = 16; m >= 1; m /= 2) {
    if (MASK & (unsigned)m) {
      const float y = __shfl_xor_sync(kFullMask, x, m);
      x = IS_MAX ? fmaxf(x, y) : x + y;
    }
  }
  return x;
}

// Index of the first finished score a lane holds (position in the [NT][G] score list).
template <int D, int G>
__device__ __forceinline__ int finished_base(int lane) {
  using C = DecodeCfg<D, G>;
  int base = 0, n = C::NV;
#pragma unroll
  for (int m = C::LPR / 2; m >= 1; m /= 2) {
    if (n >= 2) {
      if (lane & m) base += n / 2;
      n /= 2;
    }
  }
  return base;
}

template <int D, int G>
__global__ void __launch_bounds__(128, 3) decode_split_kernel(const DecodeParams p) {
  using C = DecodeCfg<D, G>;
  using R = LaneRoles<D, G>;
  extern __shared__ __align__(128) unsigned char smem[];

  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane / C::LPR, sub = lane % C::LPR;

  // ---- this CTA's key range [lo, hi) of request b, and this warp's share [wlo, whi)
  const int n = __ldg(p.seq_lens + b);
  const int S = p.num_splits;
  const int chunk = (n + S - 1) / S;
  const int lo = min(s * chunk, n), hi = min(lo + chunk, n);
  const int per_warp = (((hi - lo) + C::TPS * C::NW - 1) / (C::TPS * C::NW)) * C::TPS;
  const int wlo = min(lo + warp * per_warp, hi), whi = min(wlo + per_warp, hi);
  const int nst = (whi - wlo + C::TPS - 1) / C::TPS;

  const uint32_t ring = smem_u32(smem) + warp * C::RING_BYTES;
  float* ps = reinterpret_cast<float*>(smem + C::MAIN_BYTES + warp * C::PS_BYTES);  // p[TPS][G], alpha[G]
  const uint32_t ps_addr = smem_u32(ps);

  const int32_t* r2t = p.req_to_token + (int64_t)b * p.r2t_stride;
  const size_t head_stride = (size_t)p.num_kv_heads * D;
  const uint16_t* kbase = p.k_pool + (size_t)kvh * D;
  const uint16_t* vbase = p.v_pool + (size_t)kvh * D;

  // ---- slot ids: lane i holds the slot of key (blk + i); two 32-key blocks kept in registers
  auto load_ids = [&](int first) -> int {
    const int t = first + lane;
    return (t < whi) ? ldg_nc_i32(r2t + t) : 0;
  };
  int ids_cur = load_ids(wlo), ids_nxt = load_ids(wlo + 32);

  // ---- query rows of the G heads sharing kvh, pre-scaled by sm_scale*log2(e)
  float2 q2[G][C::CPL * 4];
  {
    const uint16_t* qrow = p.q + ((size_t)b * p.num_qo_heads + (size_t)kvh * G) * D;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int c = 0; c < C::CPL; ++c) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(qrow + (size_t)g * D + (sub + c * C::LPR) * 8));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = bf16x2_to_float2(ww[j]);
          q2[g][c * 4 + j] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
        }
      }
  }

  // ---- issue stage `st` (keys wlo + st*TPS ...) into ring slot st % STAGES
  auto issue = [&](int st) {
    if (st < nst) {
      const int off = st * C::TPS;                   // keys since wlo
      if ((off & 31) == 0 && off > 0) {              // entering a new 32-key block
        ids_cur = ids_nxt;
        ids_nxt = load_ids(wlo + off + 32);
      }
      const uint32_t dst_stage = ring + (st % C::STAGES) * C::STAGE_BYTES;
#pragma unroll
      for (int it = 0; it < C::LOADS_PER_LANE; ++it) {
        const int flat = it * 32 + lane;
        const int kv = flat / (C::TPS * C::CPR);
        const int rem = flat % (C::TPS * C::CPR);
        const int r = rem / C::CPR, ch = rem % C::CPR;
        const int slot = __shfl_sync(kFullMask, ids_cur, (off & 31) + r);
        const bool valid = wlo + off + r < whi;
        const uint16_t* src = (kv == 0 ? kbase : vbase) + (valid ? (size_t)slot * head_stride : 0) + ch * 8;
        cp_async16(dst_stage + kv * C::KV_BYTES + r * C::ROW_BYTES + ch * 16, src, valid);
      }
    }
    cp_async_commit();  // possibly empty: keeps the group count uniform
  };

  float m_run[C::NF], l_run[C::NF];
#pragma unroll
  for (int k = 0; k < C::NF; ++k) { m_run[k] = -CUDART_INF_F; l_run[k] = 0.f; }
  float2 acc[G][C::CPL * 4];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int j = 0; j < C::CPL * 4; ++j) acc[g][j] = make_float2(0.f, 0.f);

  const int fbase = finished_base<D, G>(lane);

#pragma unroll
  for (int st = 0; st < C::STAGES - 1; ++st) issue(st);

  for (int st = 0; st < nst; ++st) {
    issue(st + C::STAGES - 1);
    cp_async_wait<C::STAGES - 1>();
    __syncwarp();
    const uint32_t kt = ring + (st % C::STAGES) * C::STAGE_BYTES;
    const uint32_t vt = kt + C::KV_BYTES;
    const int t0 = wlo + st * C::TPS;

    // -- scores: partial dot products of this lane's slice, then transpose-reduce
    float sc[C::NV];
#pragma unroll
    for (int t = 0; t < C::NT; ++t) {
      const int row = rg + C::RPI * t;
      float2 part[G];
#pragma unroll
      for (int g = 0; g < G; ++g) part[g] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < C::CPL; ++c) {
        const uint4 kw = lds128(kt + row * C::ROW_BYTES + (sub + c * C::LPR) * 16);
        const float2 k0 = bf16x2_to_float2(kw.x), k1 = bf16x2_to_float2(kw.y);
        const float2 k2 = bf16x2_to_float2(kw.z), k3 = bf16x2_to_float2(kw.w);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          part[g] = __ffma2_rn(q2[g][c * 4 + 0], k0, part[g]);
          part[g] = __ffma2_rn(q2[g][c * 4 + 1], k1, part[g]);
          part[g] = __ffma2_rn(q2[g][c * 4 + 2], k2, part[g]);
          part[g] = __ffma2_rn(q2[g][c * 4 + 3], k3, part[g]);
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) sc[t * G + g] = part[g].x + part[g].y;
    }
    TReduce<C::NV, C::LPR / 2>::run(sc, lane);

    // -- online softmax on the finished scores (base 2)
    bool moved = false;
#pragma unroll
    for (int k = 0; k < C::NF; ++k) {
      const int idx = fbase + k;
      const int tl = idx / G, g = idx % G;
      const int key = rg + C::RPI * tl;
      const float sv = (t0 + key < whi) ? sc[k] : -CUDART_INF_F;
      const float tmax = butterfly<R::kKey, true>(sv);
      const float m_new = fmaxf(m_run[k], tmax);
      const float alpha = exp2f(m_run[k] - m_new);   // 0 on the first stage (m_run = -inf)
      const float pk = exp2f(sv - m_new);
      l_run[k] = l_run[k] * alpha + pk;
      moved |= (m_new != m_run[k]);
      m_run[k] = m_new;
      ps[key * G + g] = pk;
      ps[C::TPS * G + g] = alpha;   // every lane holding head g writes the same value
    }
    const bool any_moved = __any_sync(kFullMask, moved);
    __syncwarp();

    // -- rescale only when some running max moved
    if (any_moved) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float a = ps[C::TPS * G + g];
        const float2 a2 = make_float2(a, a);
#pragma unroll
        for (int j = 0; j < C::CPL * 4; ++j) acc[g][j] = __fmul2_rn(acc[g][j], a2);
      }
    }

    // -- P V
#pragma unroll
    for (int t = 0; t < C::NT; ++t) {
      const int row = rg + C::RPI * t;
      float pg[G];
#pragma unroll
      for (int g = 0; g < G; ++g) pg[g] = ps[row * G + g];
#pragma unroll
      for (int c = 0; c < C::CPL; ++c) {
        const uint4 vw = lds128(vt + row * C::ROW_BYTES + (sub + c * C::LPR) * 16);
        const float2 v0 = bf16x2_to_float2(vw.x), v1 = bf16x2_to_float2(vw.y);
        const float2 v2 = bf16x2_to_float2(vw.z), v3 = bf16x2_to_float2(vw.w);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 pp = make_float2(pg[g], pg[g]);
          acc[g][c * 4 + 0] = __ffma2_rn(pp, v0, acc[g][c * 4 + 0]);
          acc[g][c * 4 + 1] = __ffma2_rn(pp, v1, acc[g][c * 4 + 1]);
          acc[g][c * 4 + 2] = __ffma2_rn(pp, v2, acc[g][c * 4 + 2]);
          acc[g][c * 4 + 3] = __ffma2_rn(pp, v3, acc[g][c * 4 + 3]);
        }
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // ---- per-warp (m, l): sum l over the lanes that hold different keys of the same head
  float* wml = reinterpret_cast<float*>(smem + C::MAIN_BYTES + C::NW * C::PS_BYTES);  // [NW][G][2]
#pragma unroll
  for (int k = 0; k < C::NF; ++k) {
    const float lsum = butterfly<R::kKey, false>(l_run[k]);
    const int g = (fbase + k) % G;
    if ((lane & (R::kKey | R::kReplica)) == 0) {
      wml[(warp * G + g) * 2 + 0] = m_run[k];
      wml[(warp * G + g) * 2 + 1] = lsum;
    }
  }
  if (nst == 0) {  // this warp saw no keys: neutral (m, l)
    if (lane < G) {
      wml[(warp * G + lane) * 2 + 0] = -CUDART_INF_F;
      wml[(warp * G + lane) * 2 + 1] = 0.f;
    }
  }
  __syncthreads();  // every warp is done with its ring: reuse it as the merge buffer

  // ---- accumulators to shared memory: red[warp][rg][g][D]
  float* red = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int c = 0; c < C::CPL; ++c) {
      float* dst = red + (((size_t)warp * C::RPI + rg) * G + g) * D + (sub + c * C::LPR) * 8;
      reinterpret_cast<float4*>(dst)[0] = make_float4(acc[g][c * 4 + 0].x, acc[g][c * 4 + 0].y,
                                                      acc[g][c * 4 + 1].x, acc[g][c * 4 + 1].y);
      reinterpret_cast<float4*>(dst)[1] = make_float4(acc[g][c * 4 + 2].x, acc[g][c * 4 + 2].y,
                                                      acc[g][c * 4 + 3].x, acc[g][c * 4 + 3].y);
    }
  __syncthreads();

  // ---- merge warps (log-sum-exp) and write the split partial
  for (int o = threadIdx.x; o < G * (D / 4); o += blockDim.x) {
    const int g = o / (D / 4), d4 = o % (D / 4);
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) M = fmaxf(M, wml[(w * G + g) * 2]);
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < C::NW; ++w) {
        const float f = exp2f(wml[(w * G + g) * 2] - M);
        L += f * wml[(w * G + g) * 2 + 1];
#pragma unroll
        for (int r = 0; r < C::RPI; ++r) {
          const float4 a = reinterpret_cast<const float4*>(red + (((size_t)w * C::RPI + r) * G + g) * D)[d4];
          O.x += f * a.x; O.y += f * a.y; O.z += f * a.z; O.w += f * a.w;
        }
      }
    }
    const int h = kvh * G + g;
    const size_t row = ((size_t)b * p.num_qo_heads + h) * p.part_pitch + s;
    reinterpret_cast<float4*>(p.o_part + row * D)[d4] = O;
    if (d4 == 0) {
      p.ml_part[row * 2 + 0] = (M == -CUDART_INF_F) ? M : M * kLn2;  // natural-log units
      p.ml_part[row * 2 + 1] = L;
    }
  }
}

// One warp per (request, query head): merge the S partials and write bf16.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeParams p) {
  constexpr int VPL = D / 32;  // output elements per lane
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= p.batch * p.num_qo_heads) return;
  const size_t base = (size_t)wid * p.part_pitch;
  const int S = p.num_splits;
  const float* ml = p.ml_part + base * 2;

  float M = -CUDART_INF_F;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, ml[2 * s]);
  M = butterfly<31u, true>(M);

  float acc[VPL];
#pragma unroll
  for (int e = 0; e < VPL; ++e) acc[e] = 0.f;
  float L = 0.f;
  if (M != -CUDART_INF_F) {
    for (int s = 0; s < S; ++s) {
      const float m = ml[2 * s];
      const float w = (m == -CUDART_INF_F) ? 0.f : exp2f((m - M) * kLog2e);
      L += w * ml[2 * s + 1];
      const float* o = p.o_part + (base + s) * D + lane * VPL;
      if constexpr (VPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(o);
        acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(o);
        acc[0] += w * v.x; acc[1] += w * v.y;
      }
    }
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  uint16_t* dst = p.out + (size_t)wid * D + lane * VPL;
  if constexpr (VPL == 4) {
    uint2 pk;
    pk.x = float2_to_bf16x2_rn(acc[0] * inv, acc[1] * inv);
    pk.y = float2_to_bf16x2_rn(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = float2_to_bf16x2_rn(acc[0] * inv, acc[1] * inv);
  }
}

template <int D, int G>
cudaError_t launch_split_t(const DecodeParams& p, cudaStream_t stream) {
  using C = DecodeCfg<D, G>;
  static bool attr_set = false;  // per process; the attribute is per function and device-agnostic here
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(p.num_splits, p.num_kv_heads, p.batch);
  decode_split_kernel<D, G><<<grid, C::NW * 32, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool decode_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) && (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_decode_split(const DecodeParams& p, cudaStream_t stream) {
  const int G = p.num_qo_heads / p.num_kv_heads;
#define ASTR_DEC_CASE(DD, GG) \
  if (p.head_dim == DD && G == GG) return launch_split_t<DD, GG>(p, stream);
  ASTR_DEC_CASE(128, 4) ASTR_DEC_CASE(128, 1) ASTR_DEC_CASE(128, 2) ASTR_DEC_CASE(128, 8)
  ASTR_DEC_CASE(64, 4) ASTR_DEC_CASE(64, 1) ASTR_DEC_CASE(64, 2) ASTR_DEC_CASE(64, 8)
#undef ASTR_DEC_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream) {
  const int rows = p.batch * p.num_qo_heads;
  const int warps_per_block = 8;
  dim3 grid((rows + warps_per_block - 1) / warps_per_block);
  if (p.head_dim == 128) decode_combine_kernel<128><<<grid, warps_per_block * 32, 0, stream>>>(p);
  else if (p.head_dim == 64) decode_combine_kernel<64><<<grid, warps_per_block * 32, 0, stream>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace astr
