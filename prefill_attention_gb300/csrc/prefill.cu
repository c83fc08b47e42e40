// prefill.cu -- ragged packed prefill/extend attention on the sm_103a tensor core (tcgen05).
//
// Method (AstrAI commit log):
//   * page "astrai/extension/backend/attention.py @c9ceca1", batched-SDPA commit: query
//     rows of all requests are packed flat by qo_indptr; request b uses the causal offset
//     c_b = seq_len_b - q_len_b, so local query row i sees keys j <= c_b + i; masked keys
//     carry exactly zero weight.
//   * page "astrai/extension @6f67ba8", CUDA-backend commit: keys are gathered through
//     req_to_token (one token per page); unified-causal-offset commit: the offset is the
//     absolute position of the first query row.
//
// GB300 design:
//   * One CTA = one (request, query tile, KV head).  The 128-row MMA tile packs BQ = 128/G
//     query positions x the G query heads that share the KV head, so each gathered K/V
//     tile feeds all G heads (row r = position r / G, head r % G).
//   * S = Q K^T and O += P V run as tcgen05.mma (bf16 in, fp32 accumulate) with both
//     accumulators in tensor memory: S in BN = 64 columns, O in D columns.  One thread
//     issues the MMAs; an mbarrier armed by tcgen05.commit reports completion.
//   * K/V rows are gathered slot by slot with 16-byte cp.async into 128-byte-swizzled
//     shared-memory tiles (double buffered: tile j+1 loads while tile j is in softmax).
//     The same tile layout serves K as a K-major operand and V as an MN-major operand.
//   * Softmax: thread t owns TMEM lane t (one row).  Base-2 online softmax with a lazy
//     rescale: O and l are rescaled only when a row's max grows by more than 8 (so
//     unnormalised P stays below 2^8), which keeps the result exact because the same
//     reference max is used for P, l and O.
//   * P never goes through shared memory: each thread stores its row of P into tensor
//     memory as two bf16 planes, hi = bf16(p) and lo = bf16(p - hi), and O accumulates
//     P_hi V + P_lo V (A operand read from TMEM).  p is thus carried to ~2^-17 relative
//     instead of bf16's 2^-9, so the only bf16 rounding left is the final output's.
//   * Two CTAs share an SM (96 KB of tiles each), so one CTA's softmax overlaps the
//     other's MMAs and loads.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace astr {
namespace {

template <int D, int G>
struct PrefillCfg {
  static constexpr int M = 128;                        // tile rows = query positions x heads
  static constexpr int BQ = M / G;                     // query positions per tile
  static constexpr int BN = 64;                        // keys per KV tile
  static constexpr int THREADS = 128;
  static constexpr int CPR = D / 8;                    // 16-byte chunks per row
  static constexpr int Q_BYTES = M * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;          // one K (or V) tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + Q_BYTES;        // 2 stages
  static constexpr int V_OFF = K_OFF + 2 * KV_BYTES;   // 2 stages
  static constexpr int BAR_OFF = V_OFF + 2 * KV_BYTES; // bar_s, bar_o, tmem slot
  static constexpr int SMEM_BYTES = BAR_OFF + 32;
  static constexpr uint32_t TMEM_O = 0;                // O: columns [0, D)
  static constexpr uint32_t TMEM_S = D;                // S: columns [D, D + BN)
  static constexpr uint32_t TMEM_PH = D + BN;          // P high part, bf16 pairs: BN/2 columns
  static constexpr uint32_t TMEM_PL = D + BN + BN / 2; // P low part (p - bf16(p)), BN/2 columns
  static constexpr uint32_t TMEM_COLS = 256;           // D + 2 BN <= 256
  static constexpr int Q_IT = M * CPR / THREADS;       // cp.async per thread for Q
  static constexpr int KV_IT = BN * CPR / THREADS;     // cp.async per thread per K (and per V) tile
  static constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(M, BN, false, false);   // K-major A and B
  static constexpr uint32_t IDESC_PV = tc::idesc_bf16_f32(M, D, false, true);    // B (V) MN-major
  static constexpr float kRescaleThreshold = 8.f;     // log2 units
  static_assert(Q_IT * THREADS == M * CPR && KV_IT * THREADS == BN * CPR, "even copy split");
  static_assert((Q_OFF | K_OFF | V_OFF) % 1024 == 0, "swizzle atoms must be 1024-byte aligned");
  static_assert(D + 2 * BN <= (int)TMEM_COLS, "tensor-memory budget");
};

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile whose
// 64-element column blocks each hold `rows` rows.
__device__ __forceinline__ uint32_t sw128(int r, int c, int rows) {
  return (uint32_t)((c >> 3) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
}


template <int D, int G>
__global__ void __launch_bounds__(128, 2) prefill_kernel(const PrefillParams p) {
  using C = PrefillCfg<D, G>;
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y;

  // ---- (request, query tile) of this CTA from qo_indptr: warp-parallel prefix scan of
  //      per-request tile counts (every warp computes the same answer)
  int b = -1, qt = 0;
  {
    const int x = blockIdx.x;
    int acc = 0;
    for (int base = 0; base < p.batch; base += 32) {
      const int bb = base + lane;
      int nt = 0;
      if (bb < p.batch) {
        const int ql = __ldg(p.qo_indptr + bb + 1) - __ldg(p.qo_indptr + bb);
        nt = (ql + C::BQ - 1) / C::BQ;
      }
      int inc = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFullMask, inc, o);
        if (lane >= o) inc += y;
      }
      const int total = __shfl_sync(kFullMask, inc, 31);
      if (x < acc + total) {
        const unsigned ball = __ballot_sync(kFullMask, x < acc + inc);
        const int first = __ffs(ball) - 1;
        const int excl = __shfl_sync(kFullMask, inc - nt, first);
        b = base + first;
        qt = x - acc - excl;
        break;
      }
      acc += total;
    }
  }
  if (b < 0) return;                  // grid upper bound exceeds the real tile count
  if ((sbase & 1023u) != 0) return;   // swizzle atoms need a 1024-byte aligned window

  const int q0 = __ldg(p.qo_indptr + b);
  const int q_len = __ldg(p.qo_indptr + b + 1) - q0;
  const int cb = __ldg(p.seq_lens + b) - q_len;       // causal offset
  const int qi_first = qt * C::BQ;
  const int qi_last = min(q_len, qi_first + C::BQ) - 1;
  const int kv_end = cb + qi_last + 1;                 // keys any row of the tile sees
  const int n_tiles = (kv_end + C::BN - 1) / C::BN;

  const int qi = qi_first + tid / G;                   // this thread's row (= TMEM lane)
  const int g = tid % G;
  const bool row_valid = qi <= qi_last;
  const int limit = cb + min(qi, qi_last);             // last key this row attends

  const uint32_t bar_s = sbase + C::BAR_OFF, bar_o = bar_s + 8, slot = bar_s + 16;
  if (tid == 0) {
    tc::mbar_init(bar_s, 1);
    tc::mbar_init(bar_o, 1);
    tc::fence_mbarrier_init();
  }
  if (warp == 0) tc::tmem_alloc<C::TMEM_COLS>(slot);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::BAR_OFF + 16);
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  // ---- Q tile: rows (position, head) contiguous in the packed q array
  {
    const uint16_t* qbase = p.q + ((size_t)q0 * p.num_qo_heads + (size_t)kvh * G) * D;
#pragma unroll
    for (int it = 0; it < C::Q_IT; ++it) {
      const int flat = it * C::THREADS + tid;
      const int row = flat / C::CPR, c = flat % C::CPR;
      const int rqi = qi_first + row / G;
      const bool valid = rqi <= qi_last;
      const uint16_t* src = valid ? qbase + ((size_t)rqi * p.num_qo_heads + row % G) * D + c * 8 : p.q;
      cp_async16(sbase + C::Q_OFF + sw128(row, c, C::M), src, valid);
    }
  }

  // ---- K/V gather through the slot table
  const int32_t* r2t = p.req_to_token + (size_t)b * p.r2t_stride;
  const size_t head_stride = (size_t)p.num_kv_heads * D;
  int ids[C::KV_IT];
  auto load_ids = [&](int tile) {
#pragma unroll
    for (int it = 0; it < C::KV_IT; ++it) {
      const int key = (it * C::THREADS + tid) / C::CPR;
      const int j = tile * C::BN + key;
      ids[it] = (tile < n_tiles && j < kv_end) ? ldg_nc_i32(r2t + j) : -1;
    }
  };
  auto issue_kv = [&](int tile) {
    const uint32_t kdst = sbase + C::K_OFF + (tile & 1) * C::KV_BYTES;
    const uint32_t vdst = sbase + C::V_OFF + (tile & 1) * C::KV_BYTES;
#pragma unroll
    for (int it = 0; it < C::KV_IT; ++it) {
      const int flat = it * C::THREADS + tid;
      const int key = flat / C::CPR, c = flat % C::CPR;
      const bool valid = ids[it] >= 0;
      const size_t off = valid ? (size_t)ids[it] * head_stride + (size_t)kvh * D + c * 8 : 0;
      const uint32_t o = sw128(key, c, C::BN);
      cp_async16(kdst + o, p.k_pool + off, valid);
      cp_async16(vdst + o, p.v_pool + off, valid);
    }
    cp_async_commit();
  };

  load_ids(0);
  issue_kv(0);  // group 0 = Q + KV tile 0
  load_ids(1);

  float m_run = -CUDART_INF_F, l_run = 0.f;
  bool ok = true;
  const float scale = p.scale_log2;

  for (int j = 0; j < n_tiles; ++j) {
    const int stage = j & 1;
    // A. tile j is resident and visible to the tensor core; stop early if any wait timed out
    cp_async_wait<0>();
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    tc::fence_after_sync();
    if (!ok) break;

    // B. S = Q K_j^T  (fp32 in TMEM columns [D, D+BN))
    if (tid == 0) {
      const uint32_t qa = sbase + C::Q_OFF, ka = sbase + C::K_OFF + stage * C::KV_BYTES;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t ad = tc::smem_desc_sw128(qa + (kk >> 2) * (C::M * 128) + (kk & 3) * 32, 16, 1024);
        const uint64_t bd = tc::smem_desc_sw128(ka + (kk >> 2) * (C::BN * 128) + (kk & 3) * 32, 16, 1024);
        tc::mma_bf16_ss(tmem + C::TMEM_S, ad, bd, C::IDESC_S, kk > 0 ? 1u : 0u);
      }
      tc::mma_commit(bar_s);
    }

    // C. S_j done (and, in issue order, P V_{j-1}: P buffer, O and stage j+1 are free)
    ok &= tc::mbar_wait(bar_s, (uint32_t)(j & 1));
    tc::fence_after_sync();

    // D. prefetch tile j+1 and the slot ids of tile j+2
    if (j + 1 < n_tiles) {
      issue_kv(j + 1);
      load_ids(j + 2);
    }

    // E. softmax of this thread's row
    float s[C::BN];
    {
      uint32_t raw[32];
#pragma unroll
      for (int half = 0; half < C::BN / 32; ++half) {
        tc::tmem_ld32(tmem + lane_base + C::TMEM_S + half * 32, raw);
        tc::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) s[half * 32 + c] = __uint_as_float(raw[c]);
      }
    }
    const int j0 = j * C::BN;
    float mx = -CUDART_INF_F;
#pragma unroll
    for (int c = 0; c < C::BN; ++c) {
      const float x = (j0 + c <= limit) ? s[c] * scale : -CUDART_INF_F;
      s[c] = x;
      mx = fmaxf(mx, x);
    }
    const float m_new = fmaxf(m_run, mx);
    const bool need = m_new > m_run + C::kRescaleThreshold;   // always true on the first tile
    if (__any_sync(kFullMask, need)) {
      if (j > 0) {
        const float alpha = exp2f(m_run - m_new);
        l_run *= alpha;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tc::tmem_ld32(tmem + lane_base + C::TMEM_O + cc * 32, o);
          tc::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tc::tmem_st32(tmem + lane_base + C::TMEM_O + cc * 32, o);
        }
        tc::tmem_st_wait();
      }
      m_run = m_new;
    }
    // P = exp2(s - m) split into bf16 high and low parts (p = hi + lo to ~2^-17 relative),
    // stored to this row's TMEM lane; P V then runs as two MMAs so P is not rounded to bf16.
    float lsum = 0.f;
    {
      uint32_t ph[C::BN / 2], pl[C::BN / 2];
#pragma unroll
      for (int e = 0; e < C::BN / 2; ++e) {
        const float p0 = exp2f(s[2 * e] - m_run);
        const float p1 = exp2f(s[2 * e + 1] - m_run);
        lsum += p0 + p1;
        ph[e] = float2_to_bf16x2_rn(p0, p1);
        const float2 h = bf16x2_to_float2(ph[e]);
        pl[e] = float2_to_bf16x2_rn(p0 - h.x, p1 - h.y);
      }
      tc::tmem_st32(tmem + lane_base + C::TMEM_PH, ph);
      tc::tmem_st32(tmem + lane_base + C::TMEM_PL, pl);
      tc::tmem_st_wait();
    }
    l_run += lsum;

    // F. P and any O rescale are in tensor memory before the MMA is issued
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // G. O += P V_j  (fp32 in TMEM columns [0, D)); completion is observed through the
    //    next commit (S_{j+1}) or the final one.
    if (tid == 0) {
      const uint32_t va = sbase + C::V_OFF + stage * C::KV_BYTES;
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk) {
        const uint64_t bd = tc::smem_desc_sw128(va + kk * 16 * 128, C::BN * 128, 1024);
        tc::mma_bf16_ts(tmem + C::TMEM_O, tmem + C::TMEM_PH + kk * 8, bd, C::IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        tc::mma_bf16_ts(tmem + C::TMEM_O, tmem + C::TMEM_PL + kk * 8, bd, C::IDESC_PV, 1u);
      }
    }
  }

  // ---- epilogue: O / l -> bf16 rows of out
  cp_async_wait<0>();
  if (tid == 0) tc::mma_commit(bar_o);
  if (ok) ok = tc::mbar_wait(bar_o, 0);
  tc::fence_after_sync();
  const bool all_ok = __syncthreads_and(ok ? 1 : 0) != 0;
  const float inv = all_ok ? 1.f / l_run : CUDART_NAN_F;   // a timed-out wait poisons the tile
  uint16_t* orow = p.out + ((size_t)(q0 + qi) * p.num_qo_heads + (size_t)kvh * G + g) * D;
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t o[32];
    tc::tmem_ld32(tmem + lane_base + C::TMEM_O + cc * 32, o);
    tc::tmem_ld_wait();
    if (row_valid) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4 v;
        v.x = float2_to_bf16x2_rn(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv);
        v.y = float2_to_bf16x2_rn(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv);
        v.z = float2_to_bf16x2_rn(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv);
        v.w = float2_to_bf16x2_rn(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv);
        reinterpret_cast<uint4*>(orow + cc * 32)[q4] = v;
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc<C::TMEM_COLS>(tmem);
  }
}

template <int D, int G>
cudaError_t launch_prefill_t(const PrefillParams& p, cudaStream_t stream) {
  using C = PrefillCfg<D, G>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(p.num_q_tiles, p.num_kv_heads);
  prefill_kernel<D, G><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int prefill_rows_per_tile() { return 128; }

bool prefill_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) && (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream) {
  const int G = p.num_qo_heads / p.num_kv_heads;
#define ASTR_PF_CASE(DD, GG) \
  if (p.head_dim == DD && G == GG) return launch_prefill_t<DD, GG>(p, stream);
  ASTR_PF_CASE(128, 4) ASTR_PF_CASE(128, 1) ASTR_PF_CASE(128, 2) ASTR_PF_CASE(128, 8) ASTR_PF_CASE(128, 16)
  ASTR_PF_CASE(64, 4) ASTR_PF_CASE(64, 1) ASTR_PF_CASE(64, 2) ASTR_PF_CASE(64, 8) ASTR_PF_CASE(64, 16)
#undef ASTR_PF_CASE
  return cudaErrorInvalidValue;
}

}  // namespace astr
