// decode.cu -- split-KV paged decode for sm_103a.
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
//     partial, indexed by (chunk - first chunk of the request), and a request that lies
//     inside one chunk is written to the output directly.  C depends only on T, the grid
//     and a host-supplied floor, so the combine recomputes it identically.
//   * One persistent CTA per SM, warp specialised:
//       warps 4-9 (producers) -- three groups of two warps, group g owning ring stage g
//               (tiles g, g+3, ...): a group gathers the K and V rows of its 128-key tile
//               slot by slot with 16-byte cp.async into a 128-byte-swizzled layout (16-byte
//               chunk c of row r at c ^ (r & 7), so 8 consecutive rows of one chunk hit 8
//               different bank groups), waits for its own copies and arrives on the
//               stage's full barrier.  Three 64 KB tiles are in flight and each is published
//               as soon as it lands.
//       warps 0-3 (consumers) -- warp w owns keys 32w .. 32w+31 of every tile and keeps its
//               own online-softmax state: S = Q K^T and O += P V as warp-level bf16 tensor
//               core MMAs (m16n8k16, fp32 accumulators in registers, operands via ldmatrix
//               from the swizzled tiles).  The 16 MMA rows are the G query heads sharing the
//               KV head (zero-padded), so one K/V load serves all of them.  P is split into
//               hi = bf16(p) and lo = bf16(p - hi) and both halves go through the MMA, which
//               keeps p to ~2^-17 relative precision.  Softmax in base 2 (the scale carries
//               log2 e) with a lazy rescale: a warp moves its reference max only when a
//               score exceeds it by more than 2^8.  The four warps merge once per request
//               piece through shared memory; there is no per-tile CTA synchronisation.
//     Measured alternatives (see the profiles): a CUDA-core version was issue bound
//     (~550 instructions per 4 KB of K/V); a tcgen05 version with S^T / O^T accumulators in
//     tensor memory spent ~150 cycles per M=128 x N=16 x K=16 MMA, ~2400 cycles per 64 KB
//     tile on the critical path; TMA tile::gather4 for the row gather delivered ~12 GB/s
//     per SM.
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
  static constexpr int BK = 128;                   // keys per tile
  static constexpr int STAGES = 3;
  static constexpr int NCONS = 4;                  // consumer warps (32 keys each)
  static constexpr int THREADS = 320;              // 4 consumer warps, 6 producer warps
  static constexpr int NPROD = 64;                 // producer threads per group (one group per stage)
  static constexpr int CPR = D / 8;                // 16-byte chunks per K/V row
  static constexpr int KV_IT = BK * CPR / NPROD;   // cp.async per producer thread per K tile
  static constexpr int TILE = BK * D * 2;          // one K (or V) tile
  static constexpr int STAGE_BYTES = 2 * TILE;     // K | V
  static constexpr int QROWS = 16;                 // MMA rows: query heads, zero padded
  static constexpr int QBUFS = 4;
  static constexpr int Q_BYTES = QROWS * D * 2;
  static constexpr int HG = (D == 128) ? 8 : 16;   // head rows merged per pass at a piece end
  static constexpr int MERGE_BYTES = NCONS * HG * D * 4;
  static constexpr int Q_OFF = STAGES * STAGE_BYTES;
  static constexpr int MERGE_OFF = Q_OFF + QBUFS * Q_BYTES;
  static constexpr int ML_OFF = MERGE_OFF + MERGE_BYTES;   // [NCONS][16] m, then [NCONS][16] l
  static constexpr int BAR_OFF = ML_OFF + 2 * NCONS * 16 * 4;
  static constexpr int NBAR = 2 * STAGES + 1;      // full[3], empty[3], consumer merge barrier
  static constexpr int SMEM_BYTES = BAR_OFF + NBAR * 8 + 16;
  static constexpr int KSTEPS = D / 16;            // MMA k-steps over head_dim
  static constexpr int NT_D = D / 8;               // 8-wide n-tiles over head_dim
  static_assert(G <= 16, "at most 16 query heads per KV head");
  static_assert(STAGE_BYTES % 1024 == 0 && Q_OFF % 1024 == 0 && Q_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void sts128_zero(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A * B for one m16n8k16 bf16 tile with fp32 accumulation.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile whose 64-element
// column blocks each hold `rows` rows.
__device__ __forceinline__ uint32_t sw128(int r, int c, int rows) {
  return (uint32_t)((c >> 3) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
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

template <int D, int G>
__global__ void __launch_bounds__(320, 1) decode_split_kernel(const DecodeParams p) {
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
  auto empty = [&](int s) { return bars + 8u * (C::STAGES + s); };
  const uint32_t cbar = bars + 8u * (2 * C::STAGES);  // the four consumer warps, bounded waits
  volatile int* err = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 8 * C::NBAR);

  // ---- set-up: barriers; Q rows of absent heads stay zero for the whole kernel
  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      tc::mbar_init(full(s), C::NPROD);
      tc::mbar_init(empty(s), C::NCONS * 32);
    }
    tc::mbar_init(cbar, C::NCONS * 32);
    *err = 0;
    tc::fence_mbarrier_init();
  }
  for (int i = tid; i < C::QBUFS * C::Q_BYTES / 16; i += C::THREADS) sts128_zero(sbase + C::Q_OFF + i * 16);
  __syncthreads();
  // let the combine kernel's CTAs launch now; they wait for this grid's memory to be visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp >= C::NCONS) {
    // ======================= producers: group g fills ring stage g with tiles g, g+3, ...
    const int grp = (warp - C::NCONS) >> 1;             // 0..2 = the stage this group owns
    const int pt = tid - C::NCONS * 32 - grp * C::NPROD;  // 0..63 within the group
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
        cp_async16(kst + o, p.k_pool + off, valid);  // rows past the piece are zero-filled
        cp_async16(vst + o, p.v_pool + off, valid);
      }
      if (it.opens_piece(ind, lo)) {  // first tile of a piece: its G query rows
        const uint32_t qb = sbase + C::Q_OFF + (piece % C::QBUFS) * C::Q_BYTES;
        const uint16_t* qsrc = p.q + ((size_t)it.b * p.num_qo_heads + (size_t)kvh * G) * D;
        for (int i = pt; i < G * C::CPR; i += C::NPROD) {
          const int g = i / C::CPR, c = i % C::CPR;
          cp_async16(qb + sw128(g, c, C::QROWS), qsrc + (size_t)g * D + c * 8, true);
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
      tc::mbar_arrive(full(grp));  // release: the copies are visible to the consumers' loads
    }
    cp_async_wait<0>();
  } else {
    // ======================= consumers: warp w owns keys 32w .. 32w+31 of every tile
    const int g4 = lane >> 2, t4 = lane & 3;  // fragment row / column-pair index
    const int lrow = lane & 7, lmat = lane >> 3;  // ldmatrix: row within / index of the 8x8 matrix
    const float scale = p.scale_log2;
    float* mw = reinterpret_cast<float*>(smem + C::ML_OFF);  // [NCONS][16]
    float* lw = mw + C::NCONS * 16;                           // [NCONS][16]
    float* mrg = reinterpret_cast<float*>(smem + C::MERGE_OFF);

    TileIter it;
    it.first(ind, B, lo, hi);
    int piece = 0;
    uint32_t cphase = 0;            // completed phases of the consumer merge barrier
    auto cons_sync = [&]() -> bool {  // barrier over the consumer warps that cannot hang
      tc::mbar_arrive(cbar);
      return wait_or_fail(cbar, (cphase++) & 1u, err);
    };
    uint32_t qa[C::KSTEPS][4];      // Q as the A operand (rows = heads), per k-step
    float acc[C::NT_D][4];          // O rows g4 (c0,c1) and g4+8 (c2,c3) over head_dim
    float m_run[2], l_thr[2];       // rows g4 and g4+8 of this warp
    for (int j = 0; it.valid(hi); ++j) {
      const int st = j % C::STAGES;
      const bool opens = it.opens_piece(ind, lo), closes = it.closes_piece(ind, hi);
      if (!wait_or_fail(full(st), (uint32_t)((j / C::STAGES) & 1), err)) break;
      const uint32_t kst = sbase + st * C::STAGE_BYTES, vst = kst + C::TILE;

      if (opens) {  // new request piece: its query rows, fresh softmax state
        const uint32_t qb = sbase + C::Q_OFF + (piece % C::QBUFS) * C::Q_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
          // matrices: (rows 0-7, chunk 2kk), (rows 8-15, 2kk), (rows 0-7, 2kk+1), (rows 8-15, 2kk+1)
          const int r = lrow + (lmat & 1) * 8, c = 2 * kk + (lmat >> 1);
          ldsm_x4(qb + sw128(r, c, C::QROWS), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
        }
#pragma unroll
        for (int n = 0; n < C::NT_D; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        m_run[0] = m_run[1] = -CUDART_INF_F;
        l_thr[0] = l_thr[1] = 0.f;
      }

      // ---- S = Q K^T for this warp's 32 keys: 4 n-tiles of 8 keys
      const int kbase = warp * 32;
      float s[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < C::KSTEPS; ++kk) {
#pragma unroll
        for (int np = 0; np < 2; ++np) {  // two n-tiles per ldmatrix.x4
          // matrices: (keys n, chunk 2kk), (keys n, 2kk+1), (keys n+8, 2kk), (keys n+8, 2kk+1)
          const int key = kbase + np * 16 + lrow + (lmat >> 1) * 8, c = 2 * kk + (lmat & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kst + sw128(key, c, C::BK), b0, b1, b2, b3);
          mma16816(s[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
          mma16816(s[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
      }

      // ---- online softmax (base 2) on rows g4 (c0,c1) and g4+8 (c2,c3)
      const int nkeys = it.end - it.start;  // valid keys of the tile; the rest are masked
      float rmax[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kbase + n * 8 + 2 * t4 + (e & 1);
          const float x = (key < nkeys) ? s[n][e] * scale : -CUDART_INF_F;
          s[n][e] = x;
          rmax[e >> 1] = fmaxf(rmax[e >> 1], x);
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        rmax[h] = fmaxf(rmax[h], __shfl_xor_sync(kFullMask, rmax[h], 1));
        rmax[h] = fmaxf(rmax[h], __shfl_xor_sync(kFullMask, rmax[h], 2));
      }
      float alpha[2] = {1.f, 1.f};
      bool moved = false;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // a warp whose keys are all masked keeps m = -inf; nothing it adds is nonzero
        if (rmax[h] > m_run[h] + kRescaleLog2) {
          alpha[h] = fast_exp2(m_run[h] - rmax[h]);  // 0 when m_run = -inf
          m_run[h] = rmax[h];
          moved = true;
        }
      }
      if (__any_sync(kFullMask, moved)) {
#pragma unroll
        for (int n = 0; n < C::NT_D; ++n) {
          acc[n][0] *= alpha[0]; acc[n][1] *= alpha[0];
          acc[n][2] *= alpha[1]; acc[n][3] *= alpha[1];
        }
        l_thr[0] *= alpha[0];
        l_thr[1] *= alpha[1];
      }
      // P = exp2(s - m) as hi / lo bf16 A fragments, two k-steps of 16 keys
      uint32_t ph[2][4], pl[2][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mr = m_run[e >> 1];
          pv[e] = (mr == -CUDART_INF_F) ? 0.f : fast_exp2(s[n][e] - mr);
          l_thr[e >> 1] += pv[e];
        }
        const uint32_t h01 = float2_to_bf16x2_rn(pv[0], pv[1]), h23 = float2_to_bf16x2_rn(pv[2], pv[3]);
        const float2 f01 = bf16x2_to_float2(h01), f23 = bf16x2_to_float2(h23);
        const uint32_t l01 = float2_to_bf16x2_rn(pv[0] - f01.x, pv[1] - f01.y);
        const uint32_t l23 = float2_to_bf16x2_rn(pv[2] - f23.x, pv[3] - f23.y);
        // n-tile n covers keys 8n..8n+7 of the warp: k-step n/2, low (a0a1,a2a3) or high (a4a5,a6a7) half
        const int ks = n >> 1, hi8 = (n & 1) * 2;
        ph[ks][hi8 + 0] = h01; ph[ks][hi8 + 1] = h23;
        pl[ks][hi8 + 0] = l01; pl[ks][hi8 + 1] = l23;
      }

      // ---- O += P V over the warp's 32 keys: 2 k-steps x head_dim / 8 n-tiles
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
        for (int np = 0; np < C::NT_D / 2; ++np) {  // two d n-tiles per ldmatrix.x4.trans
          // matrices: (keys 0-7, chunk 2np), (keys 8-15, 2np), (keys 0-7, 2np+1), (keys 8-15, 2np+1)
          const int key = kbase + ks * 16 + lrow + (lmat & 1) * 8, c = 2 * np + (lmat >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vst + sw128(key, c, C::BK), b0, b1, b2, b3);
          mma16816(acc[2 * np], ph[ks][0], ph[ks][1], ph[ks][2], ph[ks][3], b0, b1);
          mma16816(acc[2 * np], pl[ks][0], pl[ks][1], pl[ks][2], pl[ks][3], b0, b1);
          mma16816(acc[2 * np + 1], ph[ks][0], ph[ks][1], ph[ks][2], ph[ks][3], b2, b3);
          mma16816(acc[2 * np + 1], pl[ks][0], pl[ks][1], pl[ks][2], pl[ks][3], b2, b3);
        }
      }
      __syncwarp();
      tc::mbar_arrive(empty(st));  // this warp is done reading stage st

      if (closes) {
        // ---- piece finished: merge the four warps (log-sum-exp) and write it out
        float lsum[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float x = l_thr[h];
          x += __shfl_xor_sync(kFullMask, x, 1);
          x += __shfl_xor_sync(kFullMask, x, 2);
          lsum[h] = x;
        }
        if (t4 == 0) {
          mw[warp * 16 + g4] = m_run[0];
          mw[warp * 16 + g4 + 8] = m_run[1];
          lw[warp * 16 + g4] = lsum[0];
          lw[warp * 16 + g4 + 8] = lsum[1];
        }
        const int b = it.b;
        const int rb = __ldg(ind + b), re = __ldg(ind + b + 1);
        const bool direct = (p.out != nullptr) && rb >= lo && re <= hi;  // whole request in this chunk
        const int slot = cx - rb / CL;
#pragma unroll
        for (int h0 = 0; h0 < G; h0 += C::HG) {
          // this warp's accumulator rows h0 .. h0+HG-1 to shared memory: mrg[warp][row][d]
#pragma unroll
          for (int n = 0; n < C::NT_D; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int row = g4 + (e >> 1) * 8 - h0;
              if (row >= 0 && row < C::HG && row + h0 < G)
                mrg[(warp * C::HG + row) * D + n * 8 + 2 * t4 + (e & 1)] = acc[n][e];
            }
          if (!cons_sync()) break;
          // 128 threads: thread -> (row, d) pairs of this head group
          for (int idx = tid; idx < C::HG * D; idx += C::NCONS * 32) {
            const int row = idx / D, d = idx % D, h = h0 + row;
            if (h >= G) continue;
            float M = -CUDART_INF_F;
#pragma unroll
            for (int w = 0; w < C::NCONS; ++w) M = fmaxf(M, mw[w * 16 + h]);
            float O = 0.f, L = 0.f;
            if (M != -CUDART_INF_F) {
#pragma unroll
              for (int w = 0; w < C::NCONS; ++w) {
                const float f = fast_exp2(mw[w * 16 + h] - M);  // 0 for warps that saw no key
                O += f * mrg[(w * C::HG + row) * D + d];
                L += f * lw[w * 16 + h];
              }
            }
            const size_t qh = (size_t)b * p.num_qo_heads + (size_t)kvh * G + h;
            if (direct) {
              const __nv_bfloat16 v = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
              p.out[qh * D + d] = *reinterpret_cast<const uint16_t*>(&v);
            } else {
              const size_t row0 = qh * p.part_pitch + slot;
              p.o_part[row0 * D + d] = O;
              if (d == 0) {
                p.ml_part[row0 * 2 + 0] = (M == -CUDART_INF_F) ? M : M * kLn2;  // natural-log units
                p.ml_part[row0 * 2 + 1] = L;
              }
            }
          }
          if (!cons_sync()) break;  // merge buffer and m / l free again
        }
        if (*err) break;
        ++piece;
      }
      it.next(ind, B, hi);
    }
  }
  __syncthreads();
  if (*err && tid < C::NCONS * 32) {
    // a wait timed out: poison every partial this CTA owns so the call reads as failed
    TileIter it;
    it.first(ind, B, lo, hi);
    for (; it.valid(hi); it.next(ind, B, hi)) {
      if (!it.closes_piece(ind, hi)) continue;
      const int s = cx - __ldg(ind + it.b) / CL;
      for (int i = tid; i < G * D; i += C::NCONS * 32) {
        const size_t qh = (size_t)it.b * p.num_qo_heads + (size_t)kvh * G + i / D;
        p.o_part[(qh * p.part_pitch + s) * D + i % D] = CUDART_NAN_F;
        if (p.out != nullptr) p.out[qh * D + i % D] = 0x7fc0;
      }
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
    cudaError_t e =
        cudaFuncSetAttribute(decode_split_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(p.num_splits, p.num_kv_heads);
  decode_split_kernel<D, G><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(p);
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
