// decode.cu -- split-KV paged decode for sm_103a on the 5th-generation tensor core.
//
// Method (AstrAI commit log, page "astrai/extension @6f67ba8"):
//   * CUDA-backend commit: req_to_token is the page table with one token per page, so
//     every key row is gathered through its own slot id.
//   * kernel-rename commit: decode is split-KV only; each split writes an unnormalised
//     partial plus its (max, sum) pair and a shared combine kernel merges them with a
//     log-sum-exp rescale.
//   * split-partials commit: partial buffers are never cleared -- every partial slot the
//     combine reads is written by exactly one split.
//   * pipeline commit: several tile loads stay in flight while an older tile is used.
//   * kv_indptr commit: kv_indptr (exclusive prefix sum of seq_lens) is built once per
//     step; here it drives the split schedule.
//
// GB300 design:
//   * Token-balanced split schedule.  For each KV head the flat key space [0, T) of the
//     whole batch (T = kv_indptr[B]) is cut into equal chunks of C keys, one CTA per chunk,
//     so every CTA moves the same number of bytes however skewed seq_lens is.  A chunk may
//     hold the tail of one request and the head of the next; each such piece produces one
//     partial, indexed by (chunk - first chunk of the request).  C depends only on T, the
//     grid and a host-supplied floor, so the combine recomputes it identically.
//   * One persistent CTA per SM, warp specialised:
//       warps 4-9 (producers) -- three groups of two warps, group g owning ring stage g
//               (tiles g, g+3, ...): a group gathers the K and V rows of its 128-key tile slot
//               by slot with 16-byte cp.async into the 128-byte-swizzled layout the tensor
//               core reads (XOR of the 16-byte chunk index with the row), waits for its own
//               copies, fences them to the async proxy and arrives on the stage's full
//               barrier.  Three tiles are in flight and each is published as soon as it
//               lands.  (TMA tile::gather4 was measured first: at one
//               128-byte row per gathered row it delivered ~12 GB/s per SM, well below the
//               ~45 GB/s per SM the HBM roofline needs, so the gather stays on the LSU path.)
//       warp 10 (MMA)     -- one thread issues S^T = K Q^T (M = 128 keys, N = 16 padded
//               query heads) into a double-buffered TMEM accumulator, one tile ahead of the
//               softmax, then O^T += V^T P^T (M = head_dim, V read MN-major from the same
//               tile) and releases the stage with tcgen05.commit.
//       warps 0-3 (softmax) -- thread t owns key t of the tile: it reads its S^T row from
//               TMEM, the per-head max goes through warp shuffles and a 4-entry exchange,
//               exp2 runs on the CUDA cores (the scale carries log2 e), and P^T is written
//               as two bf16 planes, hi = bf16(p) and lo = bf16(p - hi), side by side in the
//               N dimension, so O^T accumulates p to ~2^-17 relative precision.  At the end
//               of a request piece the same warps read O^T (thread = head_dim row) and
//               write the partial.
//     All G query heads of a KV head are served by each K/V tile.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace astr {

// Chunk length (keys per CTA) for T keys over n_chunks CTAs; shared by split and combine.
__device__ __forceinline__ int decode_chunk_len(int T, int n_chunks, int min_chunk, int max_splits) {
  if (max_splits <= 1) return T > 0 ? T : 1;
  int c = (T + n_chunks - 1) / n_chunks;
  c = (c + 15) & ~15;
  return c > min_chunk ? c : min_chunk;
}

namespace {

constexpr float kRescaleLog2 = 8.f;  // lazy-rescale threshold (base-2 logit units)

template <int D, int G>
struct DecCfg {
  static constexpr int BK = 128;                   // keys per tile (MMA M for S^T)
  static constexpr int STAGES = 3;
  static constexpr int THREADS = 352;              // 4 softmax warps, 6 producer warps, MMA warp
  static constexpr int NPROD = 64;                 // producer threads per group (one group per stage)
  static constexpr int MMA_WARP = 10;
  static constexpr int NSM = 128;                  // softmax threads
  static constexpr int NS = 16;                    // S^T columns: query heads padded to 16
  static constexpr int NPV = (G <= 8) ? 16 : 32;   // O^T columns: hi heads then lo heads
  static constexpr int HALF = NPV / 2;
  static constexpr int NCB = D / 64;               // 128-byte column blocks per K/V row
  static constexpr int TILE = BK * D * 2;          // one K (or V) tile
  static constexpr int ZERO = (D == 64) ? BK * 128 : 0;   // pads V^T to M = 128 when D = 64
  static constexpr int STAGE_BYTES = 2 * TILE + ZERO;     // K | V | zero block
  static constexpr int QBUFS = 4;
  static constexpr int Q_BYTES = NS * D * 2;
  static constexpr int P_BYTES = NPV * BK * 2;
  static constexpr int Q_OFF = STAGES * STAGE_BYTES;
  static constexpr int P_OFF = Q_OFF + QBUFS * Q_BYTES;   // 2 buffers
  static constexpr int RED_OFF = P_OFF + 2 * P_BYTES;     // [2][4 warps][16] floats (max), [4][16] (sum)
  static constexpr int BAR_OFF = RED_OFF + 3 * 4 * 16 * 4;
  // barriers: full[3], empty[3], s_full[2], p_full[2], pv_done[2], then tmem slot, error flag
  static constexpr int NBAR = 3 + 3 + 2 + 2 + 2;
  static constexpr int SMEM_BYTES = BAR_OFF + NBAR * 8 + 16;
  static constexpr int CPR = D / 8;                      // 16-byte chunks per K/V row
  static constexpr int KV_IT = BK * CPR / NPROD;          // cp.async per producer thread per K tile
  static constexpr uint32_t TMEM_S0 = 0;           // S^T buffers at columns 0 and 16
  static constexpr uint32_t TMEM_O = 32;
  static constexpr uint32_t TMEM_COLS = 64;
  static constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(128, NS, false, false);
  static constexpr uint32_t IDESC_PV = tc::idesc_bf16_f32(128, NPV, true, false);  // A (V^T) MN-major
  static_assert(G <= 16, "at most 16 query heads per KV head");
  static_assert(TMEM_O + NPV <= TMEM_COLS, "tensor-memory budget");
  static_assert(STAGE_BYTES % 1024 == 0 && Q_OFF % 1024 == 0 && P_OFF % 1024 == 0 && Q_BYTES % 1024 == 0 &&
                    P_BYTES % 1024 == 0,
                "swizzle atoms must be 1024-byte aligned");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void sts128_zero(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0) : "memory");
}

// Walks the tiles of one chunk: a tile never crosses a request boundary.
struct TileIter {
  int b, start, end;  // current tile: flat keys [start, end) of request b
  __device__ __forceinline__ void first(const int32_t* ind, int B, int lo, int hi) {
    int l = 0, h = B - 1;  // largest b with ind[b] <= lo
    while (l < h) {
      const int m = (l + h + 1) >> 1;
      if (__ldg(ind + m) <= lo) l = m; else h = m - 1;
    }
    b = l;
    start = lo;
    end = min(start + 128, min(hi, __ldg(ind + b + 1)));
  }
  __device__ __forceinline__ void next(const int32_t* ind, int B, int hi) {
    const int piece_end = min(hi, __ldg(ind + b + 1));
    if (end < piece_end) {
      start = end;
    } else {
      do { ++b; } while (b < B && __ldg(ind + b + 1) <= __ldg(ind + b));  // skip empty requests
      start = (b < B) ? __ldg(ind + b) : hi;
      if (start > hi) start = hi;
    }
    end = (start < hi) ? min(start + 128, min(hi, __ldg(ind + b + 1))) : start;
  }
  __device__ __forceinline__ bool valid(int hi) const { return start < hi; }
  __device__ __forceinline__ bool opens_piece(const int32_t* ind, int lo) const { return start == max(lo, __ldg(ind + b)); }
  __device__ __forceinline__ bool closes_piece(const int32_t* ind, int hi) const { return end == min(hi, __ldg(ind + b + 1)); }
};

// Bounded wait that gives up (and raises the CTA's error flag) on timeout or once the flag is up.
__device__ __forceinline__ bool wait_or_fail(uint32_t bar, uint32_t parity, volatile int* err) {
  if (*err) return false;
  if (tc::mbar_wait(bar, parity)) return true;
  *err = 1;
  return false;
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile whose
// 64-element column blocks each hold `rows` rows.
__device__ __forceinline__ uint32_t sw128(int r, int c, int rows) {
  return (uint32_t)((c >> 3) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D, int G>
__global__ void __launch_bounds__(352, 1) decode_split_tc_kernel(const DecodeParams p) {
  using C = DecCfg<D, G>;
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y, cx = blockIdx.x;
  const int B = p.batch;
  const int32_t* ind = p.kv_indptr;

  const int T = __ldg(ind + B);
  const int CL = decode_chunk_len(T, gridDim.x, p.min_chunk, p.part_pitch);
  const int lo = (int)min((int64_t)cx * CL, (int64_t)T), hi = min(lo + CL, T);
  if (lo >= hi) return;
  if ((sbase & 1023u) != 0) return;  // swizzle atoms need a 1024-byte aligned window

  const uint32_t bars = sbase + C::BAR_OFF;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (3 + s); };
  auto s_full = [&](int i) { return bars + 8u * (6 + i); };
  auto p_full = [&](int i) { return bars + 8u * (8 + i); };
  auto pv_done = [&](int i) { return bars + 8u * (10 + i); };
  const uint32_t slot = bars + 8u * C::NBAR;
  volatile int* err = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 8 * C::NBAR + 4);
  float* red = reinterpret_cast<float*>(smem + C::RED_OFF);

  // ---- set-up: barriers, TMEM, zero padding (P rows of absent heads, V^T pad block)
  if (tid == 0) {
    for (int s = 0; s < 3; ++s) {
      tc::mbar_init(full(s), C::NPROD);
      tc::mbar_init(empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(s_full(i), 1);
      tc::mbar_init(p_full(i), C::NSM);
      tc::mbar_init(pv_done(i), 1);
    }
    *err = 0;
    tc::fence_mbarrier_init();
  }
  if (warp == C::MMA_WARP) tc::tmem_alloc<C::TMEM_COLS>(slot);
  // P^T rows of absent heads and Q rows of absent heads stay zero for the whole kernel
  for (int i = tid; i < 2 * C::P_BYTES / 16; i += C::THREADS) sts128_zero(sbase + C::P_OFF + i * 16);
  for (int i = tid; i < C::QBUFS * C::Q_BYTES / 16; i += C::THREADS) sts128_zero(sbase + C::Q_OFF + i * 16);
  if constexpr (C::ZERO > 0) {
    for (int st = 0; st < C::STAGES; ++st)
      for (int i = tid; i < C::ZERO / 16; i += C::THREADS)
        sts128_zero(sbase + st * C::STAGE_BYTES + 2 * C::TILE + i * 16);
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::BAR_OFF + 8 * C::NBAR);
  // let the combine kernel's CTAs launch now; they wait for this grid's memory to be visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp >= 4 && warp < 10) {
    // ======================= producers: group g fills ring stage g with tiles g, g+3, ...
    const int grp = (warp - 4) >> 1;             // 0..2 = the stage this group owns
    const int pt = tid - C::NSM - grp * C::NPROD;  // 0..63 within the group
    TileIter it;
    it.first(ind, B, lo, hi);
    int piece = 0;
    for (int k = 0; k < grp && it.valid(hi); ++k) {  // advance to tile grp
      if (it.closes_piece(ind, hi)) ++piece;
      it.next(ind, B, hi);
    }
    const size_t head_stride = (size_t)p.num_kv_heads * D;
    // thread pt copies chunk (pt % CPR) of keys (i * NPROD + pt) / CPR, i = 0 .. KV_IT-1
    int ids[C::KV_IT];
    auto load_ids = [&](const TileIter& t) {
#pragma unroll
      for (int i = 0; i < C::KV_IT; ++i) {
        const int key = (i * C::NPROD + pt) / C::CPR;
        const int flat = t.start + key;
        ids[i] = (t.valid(hi) && flat < t.end)
                     ? ldg_nc_i32(p.req_to_token + (int64_t)t.b * p.r2t_stride + (flat - __ldg(ind + t.b)))
                     : -1;
      }
    };
    load_ids(it);
    for (int round = 0; it.valid(hi); ++round) {
      if (round > 0 && !wait_or_fail(empty(grp), (uint32_t)((round - 1) & 1), err)) break;
      const uint32_t kst = sbase + grp * C::STAGE_BYTES, vst = kst + C::TILE;
#pragma unroll
      for (int i = 0; i < C::KV_IT; ++i) {
        const int flat = i * C::NPROD + pt;
        const int key = flat / C::CPR, c = flat % C::CPR;
        const bool valid = ids[i] >= 0;
        const size_t off = valid ? (size_t)ids[i] * head_stride + (size_t)kvh * D + c * 8 : 0;
        const uint32_t o = sw128(key, c, C::BK);
        cp_async16(kst + o, p.k_pool + off, valid);
        cp_async16(vst + o, p.v_pool + off, valid);
      }
      if (it.opens_piece(ind, lo)) {  // first tile of a piece: its G query rows
        const uint32_t qb = sbase + C::Q_OFF + (piece % C::QBUFS) * C::Q_BYTES;
        const uint16_t* qsrc = p.q + ((size_t)it.b * p.num_qo_heads + (size_t)kvh * G) * D;
        for (int i = pt; i < G * C::CPR; i += C::NPROD) {
          const int g = i / C::CPR, c = i % C::CPR;
          cp_async16(qb + sw128(g, c, C::NS), qsrc + (size_t)g * D + c * 8, true);
        }
      }
      cp_async_commit();
      // advance three tiles (this group's next one) and prefetch its slot ids
      for (int k = 0; k < C::STAGES && it.valid(hi); ++k) {
        if (it.closes_piece(ind, hi)) ++piece;
        it.next(ind, B, hi);
      }
      load_ids(it);
      cp_async_wait<0>();
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(full(grp));
    }
  } else if (warp == C::MMA_WARP) {
    // ======================= MMA issuer (one thread)
    // Two streams issued as their inputs become ready, polled without blocking so that
    // neither can hold up the other: S^T of tile k (needs tile k resident and S buffer k&1
    // released by the softmax of tile k-2) and O^T += V^T P^T of tile k (needs P of tile k).
    if (lane == 0) {
      TileIter s_it, v_it;
      s_it.first(ind, B, lo, hi);
      v_it.first(ind, B, lo, hi);
      int s_piece = 0, ns = 0, nv = 0;
      long long idle_since = clock64();
      while (v_it.valid(hi)) {
        bool progress = false;
        if (s_it.valid(hi) && ns <= nv + 1 && tc::mbar_test(full(ns % C::STAGES), (uint32_t)((ns / C::STAGES) & 1))) {
          tc::fence_after_sync();
          const uint32_t kst = sbase + (ns % C::STAGES) * C::STAGE_BYTES;
          const uint32_t qb = sbase + C::Q_OFF + (s_piece % C::QBUFS) * C::Q_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ad = tc::smem_desc_sw128(kst + (kk >> 2) * (C::BK * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = tc::smem_desc_sw128(qb + (kk >> 2) * (C::NS * 128) + (kk & 3) * 32, 16, 1024);
            tc::mma_bf16_ss(tmem + C::TMEM_S0 + (ns & 1) * 16, ad, bd, C::IDESC_S, kk > 0 ? 1u : 0u);
          }
          tc::mma_commit(s_full(ns & 1));
          if (s_it.closes_piece(ind, hi)) ++s_piece;
          s_it.next(ind, B, hi);
          ++ns;
          progress = true;
        }
        if (nv < ns && tc::mbar_test(p_full(nv & 1), (uint32_t)((nv >> 1) & 1))) {
          tc::fence_after_sync();
          const uint32_t vst = sbase + (nv % C::STAGES) * C::STAGE_BYTES + C::TILE;
          const uint32_t pb = sbase + C::P_OFF + (nv & 1) * C::P_BYTES;
          const bool opens = v_it.opens_piece(ind, lo);
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            // A = V^T: M = head_dim (MN-major; second 64-column block at +BK*128 bytes, which
            // is the zero block when head_dim = 64), K = 16 keys per step
            const uint64_t ad = tc::smem_desc_sw128(vst + kk * 16 * 128, C::BK * 128, 1024);
            const uint64_t bd = tc::smem_desc_sw128(pb + (kk >> 2) * (C::NPV * 128) + (kk & 3) * 32, 16, 1024);
            tc::mma_bf16_ss(tmem + C::TMEM_O, ad, bd, C::IDESC_PV, (opens && kk == 0) ? 0u : 1u);
          }
          tc::mma_commit(empty(nv % C::STAGES));
          tc::mma_commit(pv_done(nv & 1));
          v_it.next(ind, B, hi);
          ++nv;
          progress = true;
        }
        if (progress) {
          idle_since = clock64();
        } else if (*err || clock64() - idle_since > (1ll << 31)) {  // ~1 s without progress
          *err = 1;
          break;
        } else {
          __nanosleep(32);
        }
      }
    }
  } else {
    // ======================= softmax warps 0-3 (thread t = key t = TMEM lane t)
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    TileIter it;
    it.first(ind, B, lo, hi);
    float m_run[G], l_thr[G];
#pragma unroll
    for (int g = 0; g < G; ++g) { m_run[g] = -CUDART_INF_F; l_thr[g] = 0.f; }
    const float scale = p.scale_log2;
    for (int j = 0; it.valid(hi); ++j) {
      const bool opens = it.opens_piece(ind, lo), closes = it.closes_piece(ind, hi);
      if (!wait_or_fail(s_full(j & 1), (uint32_t)((j >> 1) & 1), err)) break;
      tc::fence_after_sync();
      const bool kvalid = it.start + tid < it.end;
      float sv[G];
      {
        uint32_t r[16];
        tc::tmem_ld16(tmem + lane_base + C::TMEM_S0 + (j & 1) * 16, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < G; ++g) sv[g] = kvalid ? __uint_as_float(r[g]) * scale : -CUDART_INF_F;
      }
      // Lazy rescale: a head's reference max moves only on the first tile of a piece or
      // when some score exceeds it by more than 2^8, so O^T is rarely rescaled, P stays
      // below 2^8, and the result is exact because P, l and O share one reference max.
      // Common case: one barrier vote that no score is that far above its reference.
      bool over = false;
#pragma unroll
      for (int g = 0; g < G; ++g) over |= sv[g] > m_run[g] + kRescaleLog2;
      const bool exchange = opens || tc::named_bar_or(1, C::NSM, over);
      float alpha[G];
      bool moved = false;
#pragma unroll
      for (int g = 0; g < G; ++g) alpha[g] = 1.f;
      if (exchange) {  // per-head tile max over the 128 keys (exchange buffer alternates with j)
        float* rmax = red + (j & 1) * 64;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float x = sv[g];
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFullMask, x, o));
          if (lane == 0) rmax[warp * 16 + g] = x;
        }
        tc::named_bar_sync(1, C::NSM);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float tmax = fmaxf(fmaxf(rmax[g], rmax[16 + g]), fmaxf(rmax[32 + g], rmax[48 + g]));
          // tmax is finite: the tile has at least one key
          const bool up = opens || tmax > m_run[g] + kRescaleLog2;
          const float m_new = up ? fmaxf(m_run[g], tmax) : m_run[g];
          alpha[g] = fast_exp2(m_run[g] - m_new);  // 0 on the first tile of a piece
          moved |= (up && !opens);
          m_run[g] = m_new;
        }
      }
      // P^T buffer j&1 was last read by O^T += V^T P^T of tile j-2
      if (j >= 2 && !wait_or_fail(pv_done(j & 1), (uint32_t)(((j - 2) >> 1) & 1), err)) break;
      const uint32_t pb = sbase + C::P_OFF + (j & 1) * C::P_BYTES;
      const int col_chunk = (tid & 63) >> 3, blk = tid >> 6, within = (tid & 7) * 2;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pg = fast_exp2(sv[g] - m_run[g]);  // 0 for keys past the piece
        l_thr[g] = l_thr[g] * alpha[g] + pg;
        const uint32_t hi16 = float2_to_bf16x2_rn(pg, 0.f) & 0xffffu;
        const float lo_f = pg - __uint_as_float(hi16 << 16);
        const uint32_t lo16 = float2_to_bf16x2_rn(lo_f, 0.f) & 0xffffu;
        const int gl = C::HALF + g;
        sts16(pb + blk * (C::NPV * 128) + (g >> 3) * 1024 + (g & 7) * 128 + ((col_chunk ^ (g & 7)) << 4) + within,
              (uint16_t)hi16);
        sts16(pb + blk * (C::NPV * 128) + (gl >> 3) * 1024 + (gl & 7) * 128 + ((col_chunk ^ (gl & 7)) << 4) + within,
              (uint16_t)lo16);
      }
      // rescale the live O^T columns when a reference max moved (CTA-uniform decision)
      if (moved) {
        if (!wait_or_fail(pv_done((j - 1) & 1), (uint32_t)(((j - 1) >> 1) & 1), err)) break;
        tc::fence_after_sync();
        if constexpr (C::NPV == 16) {
          uint32_t o[16];
          tc::tmem_ld16(tmem + lane_base + C::TMEM_O, o);
          tc::tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < G; ++g) {
            o[g] = __float_as_uint(__uint_as_float(o[g]) * alpha[g]);
            o[C::HALF + g] = __float_as_uint(__uint_as_float(o[C::HALF + g]) * alpha[g]);
          }
          tc::tmem_st16(tmem + lane_base + C::TMEM_O, o);
        } else {
          uint32_t o[32];
          tc::tmem_ld32(tmem + lane_base + C::TMEM_O, o);
          tc::tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < G; ++g) {
            o[g] = __float_as_uint(__uint_as_float(o[g]) * alpha[g]);
            o[C::HALF + g] = __float_as_uint(__uint_as_float(o[C::HALF + g]) * alpha[g]);
          }
          tc::tmem_st32(tmem + lane_base + C::TMEM_O, o);
        }
        tc::tmem_st_wait();
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(p_full(j & 1));

      if (closes) {
        // piece finished: O^T += V^T P^T of this tile must land, then write the partial
        if (!wait_or_fail(pv_done(j & 1), (uint32_t)((j >> 1) & 1), err)) break;
        tc::fence_after_sync();
        float* rsum = red + 128;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float x = l_thr[g];
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(kFullMask, x, o);
          if (lane == 0) rsum[warp * 16 + g] = x;
        }
        float og[G];
        if constexpr (C::NPV == 16) {
          uint32_t o[16];
          tc::tmem_ld16(tmem + lane_base + C::TMEM_O, o);
          tc::tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < G; ++g) og[g] = __uint_as_float(o[g]) + __uint_as_float(o[C::HALF + g]);
        } else {
          uint32_t o[32];
          tc::tmem_ld32(tmem + lane_base + C::TMEM_O, o);
          tc::tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < G; ++g) og[g] = __uint_as_float(o[g]) + __uint_as_float(o[C::HALF + g]);
        }
        tc::named_bar_sync(1, C::NSM);
        const int b = it.b;
        const int rb = __ldg(ind + b), re = __ldg(ind + b + 1);
        if (p.out != nullptr && rb >= lo && re <= hi) {
          // the whole request lies in this chunk: normalise and write the output directly
          // (the combine skips requests that occupy a single chunk)
          if (tid < D) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float L = rsum[g] + rsum[16 + g] + rsum[32 + g] + rsum[48 + g];
              const float v = og[g] / L;
              const __nv_bfloat16 h = __float2bfloat16_rn(v);
              p.out[((size_t)b * p.num_qo_heads + (size_t)kvh * G + g) * D + tid] =
                  *reinterpret_cast<const uint16_t*>(&h);
            }
          }
        } else {
          const int s = cx - rb / CL;  // partial slot of this piece
          const size_t row0 = ((size_t)b * p.num_qo_heads + (size_t)kvh * G) * p.part_pitch + s;
          if (tid < D) {
#pragma unroll
            for (int g = 0; g < G; ++g) p.o_part[(row0 + (size_t)g * p.part_pitch) * D + tid] = og[g];
          }
#pragma unroll
          for (int g = 0; g < G; ++g) {
            if (tid == g) {
              p.ml_part[(row0 + (size_t)g * p.part_pitch) * 2 + 0] = m_run[g] * kLn2;  // natural-log units
              p.ml_part[(row0 + (size_t)g * p.part_pitch) * 2 + 1] =
                  rsum[g] + rsum[16 + g] + rsum[32 + g] + rsum[48 + g];
            }
          }
        }
        tc::named_bar_sync(1, C::NSM);  // sums read before the next piece reuses the buffer
#pragma unroll
        for (int g = 0; g < G; ++g) { m_run[g] = -CUDART_INF_F; l_thr[g] = 0.f; }
      }
      it.next(ind, B, hi);
    }
  }

  // ---- teardown: every role has finished (all issued MMAs were waited on by the softmax
  //      warps through pv_done of the final tile)
  tc::fence_before_sync();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc::fence_after_sync();
    tc::tmem_dealloc<C::TMEM_COLS>(tmem);
  }
  if (*err && tid < D) {  // a wait timed out: poison what this CTA owns so the call reads as failed
    TileIter it;
    it.first(ind, B, lo, hi);
    for (; it.valid(hi); it.next(ind, B, hi)) {
      if (!it.closes_piece(ind, hi)) continue;
      const int s = cx - __ldg(ind + it.b) / CL;
      const size_t row0 = ((size_t)it.b * p.num_qo_heads + (size_t)kvh * G) * p.part_pitch + s;
      for (int g = 0; g < G; ++g) p.o_part[(row0 + (size_t)g * p.part_pitch) * D + tid] = CUDART_NAN_F;
    }
  }
}

// One warp per (request, query head): merge the request's partials and write bf16.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeParams p) {
  constexpr int VPL = D / 32;  // output elements per lane
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  // launched as a programmatic dependent of the split kernel: wait until its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (wid >= p.batch * p.num_qo_heads) return;
  const int b = wid / p.num_qo_heads;
  int S;
  if (p.kv_indptr != nullptr) {  // token-balanced chunks: the chunks that overlap request b
    const int T = __ldg(p.kv_indptr + p.batch);
    const int CL = decode_chunk_len(T, p.num_splits, p.min_chunk, p.part_pitch);
    const int a = __ldg(p.kv_indptr + b), e = __ldg(p.kv_indptr + b + 1);
    S = (e > a) ? (e - 1) / CL - a / CL + 1 : 0;
    if (S == 1 && !p.combine_all) return;  // written directly by the split kernel
  } else {                       // explicit count (partials supplied by the caller)
    S = p.num_splits;
  }
  const size_t base = (size_t)wid * p.part_pitch;
  const float* ml = p.ml_part + base * 2;

  float M = -CUDART_INF_F;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, ml[2 * s]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, o));

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
  using C = DecCfg<D, G>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_tc_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(p.num_splits, p.num_kv_heads);
  decode_split_tc_kernel<D, G><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool decode_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

cudaError_t launch_decode_split(const DecodeParams& p, cudaStream_t stream) {
  const int G = p.num_qo_heads / p.num_kv_heads;
#define ASTR_DEC_CASE(DD, GG) \
  if (p.head_dim == DD && G == GG) return launch_split_t<DD, GG>(p, stream);
  ASTR_DEC_CASE(128, 4) ASTR_DEC_CASE(128, 1) ASTR_DEC_CASE(128, 2) ASTR_DEC_CASE(128, 8) ASTR_DEC_CASE(128, 16)
  ASTR_DEC_CASE(64, 4) ASTR_DEC_CASE(64, 1) ASTR_DEC_CASE(64, 2) ASTR_DEC_CASE(64, 8) ASTR_DEC_CASE(64, 16)
#undef ASTR_DEC_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream) {
  const int rows = p.batch * p.num_qo_heads;
  const int warps_per_block = 8;
  dim3 grid((rows + warps_per_block - 1) / warps_per_block);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(warps_per_block * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap with the split kernel's tail
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (p.head_dim == 128) e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, p);
  else if (p.head_dim == 64) e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, p);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace astr
