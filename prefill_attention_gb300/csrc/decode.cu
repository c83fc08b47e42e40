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
//               different bank groups).  Each 32-key quarter of a tile is its own cp.async
//               group with its own full barrier, so a quarter is published as soon as it
//               lands.  Three 64 KB tiles are in flight.
//       warps 0-3 (consumers) -- warp w takes quarter (w + j) mod 4 of tile j and keeps its
//               own online-softmax state.  The products are computed transposed, S^T = K Q^T
//               and O^T += V^T P^T, as warp-level bf16 MMAs (m16n8k16, fp32 accumulators in
//               registers, operands via ldmatrix from the swizzled tiles): the 16-row MMA
//               side is keys or head_dim and the 8-wide side the G query heads of the KV
//               head, so one K/V load serves all of them with little padding.  P goes from
//               the S^T accumulator layout to the B-operand layout with movmatrix.  P is
//               split into hi = bf16(p) and lo = bf16(p - hi) and both halves go through the
//               MMA, which keeps p to ~2^-17 relative precision.  Softmax in base 2 (the
//               scale carries log2 e) with a lazy rescale: a warp moves its reference max
//               only when a score exceeds it by more than 2^8.  A quarter with no valid key
//               (the ragged end of a piece) is skipped; rotating the quarters spreads those
//               savings over the warps.  The four warps merge once per request piece
//               through shared memory; there is no per-tile CTA synchronisation.
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
  static constexpr int NCONS = 4;                  // consumer warps; a tile is 4 quarters of 32 keys
  static constexpr int THREADS = 320;              // 4 consumer warps, 6 producer warps
  static constexpr int NPROD = 64;                 // producer threads per group (one group per stage)
  static constexpr int CPR = D / 8;                // 16-byte chunks per K/V row
  static constexpr int KV_IT = BK * CPR / NPROD;   // cp.async per producer thread per K tile
  static constexpr int KV_IT_Q = KV_IT / NCONS;    // ... per quarter
  static constexpr int TILE = BK * D * 2;          // one K (or V) tile
  static constexpr int STAGE_BYTES = 2 * TILE;     // K | V
  static constexpr int NH = (G + 7) / 8;           // 8-wide MMA n-tiles over the query heads
  static constexpr int QROWS = 8 * NH;             // query rows in shared memory, zero padded
  static constexpr int QBUFS = 4;
  static constexpr int Q_BYTES = QROWS * D * 2;
  static constexpr int HG = (D == 128) ? 8 : 16;   // head rows merged per pass at a piece end
  static constexpr int MERGE_BYTES = NCONS * HG * D * 4;
  static constexpr int Q_OFF = STAGES * STAGE_BYTES;
  static constexpr int MERGE_OFF = Q_OFF + QBUFS * Q_BYTES;
  static constexpr int ML_OFF = MERGE_OFF + MERGE_BYTES;   // [NCONS][16] m, then [NCONS][16] l
  static constexpr int BAR_OFF = ML_OFF + 2 * NCONS * 16 * 4;
  static constexpr int NBAR = STAGES * NCONS + STAGES + 1;  // full[stage][quarter], empty[stage], merge
  static constexpr int SMEM_BYTES = BAR_OFF + NBAR * 8 + 16;
  static constexpr int KSTEPS = D / 16;            // MMA k-steps over head_dim (S^T = K Q^T)
  static constexpr int MT_D = D / 16;              // 16-row m-tiles over head_dim (O^T = V^T P^T)
  static_assert(G <= 16, "at most 16 query heads per KV head");
  static_assert(KV_IT % NCONS == 0, "quarters split the producer loop evenly");
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

// Transpose of one 8x8 b16 matrix held one packed pair per lane (row lane/4, columns 2(lane%4), +1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
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
  constexpr int NH = C::NH;
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y, cx = blockIdx.x;
  const int B = p.batch;
  const int32_t* ind = p.kv_indptr;

  if ((sbase & 1023u) != 0) return;  // swizzle atoms need a 1024-byte aligned window

  const uint32_t bars = sbase + C::BAR_OFF;
  auto full = [&](int s, int q) { return bars + 8u * (s * C::NCONS + q); };
  auto empty = [&](int s) { return bars + 8u * (C::STAGES * C::NCONS + s); };
  const uint32_t cbar = bars + 8u * (C::NBAR - 1);  // the four consumer warps, bounded waits
  volatile int* err = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 8 * C::NBAR);

  // ---- set-up (shared memory only): barriers; Q rows of absent heads stay zero throughout
  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      for (int q = 0; q < C::NCONS; ++q) tc::mbar_init(full(s, q), C::NPROD);
      tc::mbar_init(empty(s), C::NCONS * 32);
    }
    tc::mbar_init(cbar, C::NCONS * 32);
    *err = 0;
    tc::fence_mbarrier_init();
  }
  for (int i = tid; i < C::QBUFS * C::Q_BYTES / 16; i += C::THREADS) sts128_zero(sbase + C::Q_OFF + i * 16);
  __syncthreads();
  // Launched as a programmatic dependent of the previous kernel in the stream: the set-up
  // above overlapped its tail; from here on its writes are visible and its reads are done,
  // so no global memory is touched before this point.  (A no-op for an ordinary launch.)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // let the combine kernel's CTAs launch now; they wait for this grid's memory to be visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int T = __ldg(ind + B);
  const int CL = decode_chunk_len(T, gridDim.x, p.min_chunk, p.part_pitch);
  const int lo = (int)min((int64_t)cx * CL, (int64_t)T), hi = min(lo + CL, T);
  if (lo >= hi) return;  // uniform over the CTA; no barrier follows for it

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
    // thread pt copies chunk (pt % CPR) of keys (i * NPROD + pt) / CPR, i = 0 .. KV_IT-1;
    // iterations [q * KV_IT_Q, (q + 1) * KV_IT_Q) cover exactly the keys of quarter q
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
      if (it.opens_piece(ind, lo)) {  // first tile of a piece: its G query rows (with quarter 0)
        const uint32_t qb = sbase + C::Q_OFF + (piece % C::QBUFS) * C::Q_BYTES;
        const uint16_t* qsrc = p.q + ((size_t)it.b * p.num_qo_heads + (size_t)kvh * G) * D;
        for (int i = pt; i < G * C::CPR; i += C::NPROD) {
          const int g = i / C::CPR, c = i % C::CPR;
          cp_async16(qb + sw128(g, c, C::QROWS), qsrc + (size_t)g * D + c * 8, true);
        }
      }
#pragma unroll
      for (int q = 0; q < C::NCONS; ++q) {  // one cp.async group per quarter
#pragma unroll
        for (int i = q * C::KV_IT_Q; i < (q + 1) * C::KV_IT_Q; ++i) {
          const int flat = i * C::NPROD + pt;
          const int key = flat / C::CPR, c = flat % C::CPR;
          const bool valid = ids[i] >= 0;
          const size_t off = valid ? (size_t)ids[i] * head_stride + (size_t)kvh * D + c * 8 : 0;
          const uint32_t o = sw128(key, c, C::BK);
          cp_async16(kst + o, p.k_pool + off, valid);  // rows past the piece are zero-filled
          cp_async16(vst + o, p.v_pool + off, valid);
        }
        cp_async_commit();
      }
      // advance three tiles (this group's next one) and prefetch its slot ids
      for (int k = 0; k < C::STAGES && it.valid(hi); ++k) {
        if (it.closes_piece(ind, hi)) ++piece;
        it.next(ind, B, hi);
      }
      load_ids(it);
      // publish each quarter as soon as this thread's copies of it have landed
      cp_async_wait<3>();
      tc::mbar_arrive(full(grp, 0));
      cp_async_wait<2>();
      tc::mbar_arrive(full(grp, 1));
      cp_async_wait<1>();
      tc::mbar_arrive(full(grp, 2));
      cp_async_wait<0>();
      tc::mbar_arrive(full(grp, 3));
    }
    cp_async_wait<0>();
  } else {
    // ======================= consumers: warp w takes quarter (w + j) % 4 of tile j
    // Transposed products so the 16-row MMA side is keys / head_dim, not the few heads:
    //   S^T (32 keys x 8 heads) = K Q^T,   O^T (D x 8 heads) += V^T P^T.
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
    uint32_t qb[NH][C::KSTEPS][2];  // Q^T as the B operand (n = heads), per k-step
    float acc[C::MT_D][NH][4];      // O^T: rows d = 16md + g4 (+8), heads 8nh + 2t4 (+1)
    float m_run[NH][2], l_thr[NH][2];  // heads 8nh + 2t4 + e of this warp
    for (int j = 0; it.valid(hi); ++j) {
      const int st = j % C::STAGES;
      const int quarter = (warp + j) & (C::NCONS - 1);
      const bool opens = it.opens_piece(ind, lo), closes = it.closes_piece(ind, hi);
      const int kbase = quarter * 32;
      const int nkeys = it.end - it.start;  // valid keys of the tile; the rest are masked
      const bool work = kbase < nkeys;      // quarters wholly past the piece are skipped
      if (!wait_or_fail(full(st, quarter), (uint32_t)((j / C::STAGES) & 1), err)) break;
      const uint32_t kst = sbase + st * C::STAGE_BYTES, vst = kst + C::TILE;

      if (opens) {  // new request piece: its query rows, fresh softmax state
        const uint32_t qbuf = sbase + C::Q_OFF + (piece % C::QBUFS) * C::Q_BYTES;
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
          for (int kk = 0; kk < C::KSTEPS; kk += 2) {
            // matrices: heads 8nh .. 8nh+7 at chunks 2kk, 2kk+1, 2kk+2, 2kk+3
            ldsm_x4(qbuf + sw128(8 * nh + lrow, 2 * kk + lmat, C::QROWS), qb[nh][kk][0], qb[nh][kk][1],
                    qb[nh][kk + 1][0], qb[nh][kk + 1][1]);
          }
#pragma unroll
        for (int md = 0; md < C::MT_D; ++md)
#pragma unroll
          for (int nh = 0; nh < NH; ++nh) acc[md][nh][0] = acc[md][nh][1] = acc[md][nh][2] = acc[md][nh][3] = 0.f;
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) {
          m_run[nh][0] = m_run[nh][1] = -CUDART_INF_F;
          l_thr[nh][0] = l_thr[nh][1] = 0.f;
        }
      }

      if (work) {
        // ---- S^T = K Q^T: 2 m-tiles of 16 keys; even / odd k-steps in separate accumulators
        float s[2][NH][4], s2[2][NH][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nh = 0; nh < NH; ++nh)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[mt][nh][e] = s2[mt][nh][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            // matrices: (keys 0-7, chunk 2kk), (keys 8-15, 2kk), (keys 0-7, 2kk+1), (keys 8-15, 2kk+1)
            const int key = kbase + mt * 16 + lrow + (lmat & 1) * 8, c = 2 * kk + (lmat >> 1);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kst + sw128(key, c, C::BK), a0, a1, a2, a3);
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) {
              if (kk & 1) mma16816(s2[mt][nh], a0, a1, a2, a3, qb[nh][kk][0], qb[nh][kk][1]);
              else mma16816(s[mt][nh], a0, a1, a2, a3, qb[nh][kk][0], qb[nh][kk][1]);
            }
          }
        }

        // ---- online softmax (base 2) per head; this lane holds keys 16mt + g4 (+8)
        float rmax[NH][2];
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) rmax[nh][0] = rmax[nh][1] = -CUDART_INF_F;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nh = 0; nh < NH; ++nh)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = kbase + mt * 16 + g4 + (e >> 1) * 8;
              const float x = (key < nkeys) ? (s[mt][nh][e] + s2[mt][nh][e]) * scale : -CUDART_INF_F;
              s[mt][nh][e] = x;
              rmax[nh][e & 1] = fmaxf(rmax[nh][e & 1], x);
            }
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float x = rmax[nh][h];
            x = fmaxf(x, __shfl_xor_sync(kFullMask, x, 4));
            x = fmaxf(x, __shfl_xor_sync(kFullMask, x, 8));
            x = fmaxf(x, __shfl_xor_sync(kFullMask, x, 16));
            rmax[nh][h] = x;
          }
        float alpha[NH][2];
        bool moved = false;
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            alpha[nh][h] = 1.f;
            // a warp whose keys are all masked keeps m = -inf; nothing it adds is nonzero
            if (rmax[nh][h] > m_run[nh][h] + kRescaleLog2) {
              alpha[nh][h] = fast_exp2(m_run[nh][h] - rmax[nh][h]);  // 0 when m_run = -inf
              m_run[nh][h] = rmax[nh][h];
              moved = true;
            }
          }
        if (__any_sync(kFullMask, moved)) {
#pragma unroll
          for (int md = 0; md < C::MT_D; ++md)
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) {
              acc[md][nh][0] *= alpha[nh][0]; acc[md][nh][1] *= alpha[nh][1];
              acc[md][nh][2] *= alpha[nh][0]; acc[md][nh][3] *= alpha[nh][1];
            }
#pragma unroll
          for (int nh = 0; nh < NH; ++nh) {
            l_thr[nh][0] *= alpha[nh][0];
            l_thr[nh][1] *= alpha[nh][1];
          }
        }
        // P = exp2(s - m) as hi / lo bf16 pairs, transposed into P^T B fragments
        uint32_t ph[2][NH][2], pl[2][NH][2];  // [k-step = m-tile][nh][keys 0-7 | 8-15]
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nh = 0; nh < NH; ++nh)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float pv[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float mr = m_run[nh][e];
                pv[e] = (mr == -CUDART_INF_F) ? 0.f : fast_exp2(s[mt][nh][2 * half + e] - mr);
                l_thr[nh][e] += pv[e];
              }
              const uint32_t h01 = float2_to_bf16x2_rn(pv[0], pv[1]);
              const float2 f01 = bf16x2_to_float2(h01);
              const uint32_t l01 = float2_to_bf16x2_rn(pv[0] - f01.x, pv[1] - f01.y);
              // (key g4 + 8 half, heads 2t4, 2t4+1) -> (head g4, keys 8 half + 2t4, +1)
              ph[mt][nh][half] = movmatrix_t(h01);
              pl[mt][nh][half] = movmatrix_t(l01);
            }

        // ---- O^T += V^T P^T over the quarter's 32 keys: 2 k-steps x D / 16 m-tiles
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
          for (int md = 0; md < C::MT_D; ++md) {
            // matrices (transposed on load): (d 0-7, keys 0-7), (d 8-15, keys 0-7), (d 0-7, keys 8-15), (d 8-15, keys 8-15)
            const int key = kbase + ks * 16 + lrow + (lmat >> 1) * 8, c = 2 * md + (lmat & 1);
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vst + sw128(key, c, C::BK), a0, a1, a2, a3);
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) {
              mma16816(acc[md][nh], a0, a1, a2, a3, ph[ks][nh][0], ph[ks][nh][1]);
              mma16816(acc[md][nh], a0, a1, a2, a3, pl[ks][nh][0], pl[ks][nh][1]);
            }
          }
        }
      }
      // Quarters land in order, so seeing the last one means all of round j / STAGES is in.
      // The next warp to wait on this stage's barriers may hold another quarter; with this
      // wait, no barrier of the stage can still be a phase behind when it does.
      if (!wait_or_fail(full(st, C::NCONS - 1), (uint32_t)((j / C::STAGES) & 1), err)) break;
      __syncwarp();
      tc::mbar_arrive(empty(st));  // this warp is done reading stage st

      if (closes) {
        // ---- piece finished: merge the four warps (log-sum-exp) and write it out
        float lsum[NH][2];
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float x = l_thr[nh][h];
            x += __shfl_xor_sync(kFullMask, x, 4);
            x += __shfl_xor_sync(kFullMask, x, 8);
            x += __shfl_xor_sync(kFullMask, x, 16);
            lsum[nh][h] = x;
          }
        if (g4 == 0) {
#pragma unroll
          for (int nh = 0; nh < NH; ++nh)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              mw[warp * 16 + 8 * nh + 2 * t4 + h] = m_run[nh][h];
              lw[warp * 16 + 8 * nh + 2 * t4 + h] = lsum[nh][h];
            }
        }
        const int b = it.b;
        const int rb = __ldg(ind + b), re = __ldg(ind + b + 1);
        const bool direct = (p.out != nullptr) && rb >= lo && re <= hi;  // whole request in this chunk
        const int slot = cx - rb / CL;
#pragma unroll
        for (int h0 = 0; h0 < G; h0 += C::HG) {
          // this warp's accumulator rows h0 .. h0+HG-1 to shared memory: mrg[warp][row][d]
#pragma unroll
          for (int md = 0; md < C::MT_D; ++md)
#pragma unroll
            for (int nh = 0; nh < NH; ++nh)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int row = 8 * nh + 2 * t4 + (e & 1) - h0;
                if (row >= 0 && row < C::HG && row + h0 < G)
                  mrg[(warp * C::HG + row) * D + md * 16 + g4 + (e >> 1) * 8] = acc[md][nh][e];
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
  // the next kernel in the stream may start its shared-memory set-up now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits, p.num_kv_heads);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // set-up overlaps the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_split_kernel<D, G>, p);
  if (e != cudaSuccess) return e;
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
