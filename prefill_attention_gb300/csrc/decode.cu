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

#include <type_traits>

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
  static constexpr int NPAIR = kDecodeChunksPerCta;  // independent (producer, consumer) warp pairs
  static constexpr int THREADS = 2 * NPAIR * 32;   // warps 0..3 consume, warps 4..7 produce
  static constexpr int BK = 32;                    // keys per ring slot
  static constexpr int CPR = D / 8;                // 16-byte chunks per K/V row
  static constexpr int KV_IT = BK * CPR / 32;      // cp.async per producer lane per K slot
  static constexpr int NH = (G + 7) / 8;           // 8-wide MMA n-tiles over the query heads
  static constexpr int QROWS = 8 * NH;             // query rows in a slot, zero padded
  static constexpr int KV_BYTES = BK * D * 2;      // K (or V) part of a slot
  static constexpr int Q_BYTES = QROWS * D * 2;
  static constexpr int SLOT = 2 * KV_BYTES + Q_BYTES;   // K | V | Q
  static constexpr int STAGES_FIT = (220 * 1024) / (NPAIR * SLOT);
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;  // ring slots per pair
  static constexpr int RING = STAGES * SLOT;
  static constexpr int BAR_OFF = NPAIR * RING;
  static constexpr int NBAR = NPAIR * 2 * STAGES;  // full[pair][slot], empty[pair][slot]
  static constexpr int SMEM_BYTES = BAR_OFF + NBAR * 8 + 16 * 4;  // + per-pair error flags
  static constexpr int KSTEPS = D / 16;            // MMA k-steps over head_dim (S^T = K Q^T)
  static constexpr int MT_D = D / 16;              // 16-row m-tiles over head_dim (O^T = V^T P^T)
  static constexpr int STG_PITCH = D + 4;          // fp32 staging row pitch (conflict-free writes)
  static_assert(G <= 16, "at most 16 query heads per KV head");
  static_assert(STAGES >= 2, "a ring needs two slots");
  static_assert(SLOT % 1024 == 0 && KV_BYTES % 1024 == 0, "swizzle atoms");
  static_assert((QROWS * STG_PITCH + 2 * QROWS) * 4 <= 2 * KV_BYTES, "piece staging fits in K | V");
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

// Arrive on an mbarrier once every cp.async this thread has issued so far has landed
// (the arrival counts toward the barrier's expected count; it does not add to it).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile whose 64-element
// column blocks each hold `rows` rows.
__device__ __forceinline__ uint32_t sw128(int r, int c, int rows) {
  return (uint32_t)((c >> 3) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Walks the slots of one chunk: BK keys at a time, never across a request boundary.
template <int BK>
struct TileIter {
  int b, start, end;  // current slot: flat keys [start, end) of request b
  __device__ __forceinline__ void first(const int32_t* ind, int B, int lo, int hi) {
    int l = 0, h = B - 1;  // largest b with ind[b] <= lo
    while (l < h) {
      const int m = (l + h + 1) >> 1;
      if (__ldg(ind + m) <= lo) l = m; else h = m - 1;
    }
    b = l;
    start = lo;
    end = min(start + BK, min(hi, __ldg(ind + b + 1)));
  }
  // Same as first() for a chunk whose first request b0 and its end ind[b0 + 1] are known.
  __device__ __forceinline__ void start_at(int b0, int b0_end, int lo, int hi) {
    b = b0;
    start = lo;
    end = min(start + BK, min(hi, b0_end));
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
    end = (start < hi) ? min(start + BK, min(hi, __ldg(ind + b + 1))) : start;
  }
  __device__ __forceinline__ bool valid(int hi) const { return start < hi; }
  __device__ __forceinline__ bool opens_piece(const int32_t* ind, int lo) const { return start == max(lo, __ldg(ind + b)); }
  __device__ __forceinline__ bool closes_piece(const int32_t* ind, int hi) const { return end == min(hi, __ldg(ind + b + 1)); }
};

// Warp-cooperative lookup of the request that holds flat key `lo` (largest b with
// ind[b] <= lo, so empty requests are stepped over), with ind[b] and ind[b + 1].
// Each round samples ind at 128 evenly spaced points of the bracket [l, h) (every point
// once the bracket is that narrow) and keeps the two samples around lo, so a batch of up
// to 128 requests takes one round of loads and 16384 take two.  Needs ind[l] <= lo <
// ind[h] on entry, i.e. l = 0, h = B, ind_h = ind[B] > lo.
__device__ __forceinline__ int pick4(const int (&v)[4], int k) {  // v[k] without local memory
  return k == 0 ? v[0] : k == 1 ? v[1] : k == 2 ? v[2] : v[3];
}
struct ReqBracket {
  int b, start, end;
};
__device__ __forceinline__ ReqBracket locate_request(const int32_t* ind, int B, int lo, int ind_B, int lane) {
  int l = 0, h = B, ind_l = 0, ind_h = ind_B;
  while (h - l > 1) {
    int v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = __ldg(ind + l + (int)((int64_t)(h - l) * (lane * 4 + k) / 128));
    int c = 0;  // samples with ind <= lo; they are samples 0 .. c-1 (ind and positions ascend)
#pragma unroll
    for (int k = 0; k < 4; ++k) c += __popc(__ballot_sync(kFullMask, v[k] <= lo));
    const int i_lo = c - 1;  // >= 0: sample 0 is ind[l] <= lo
    const int vl = __shfl_sync(kFullMask, pick4(v, i_lo & 3), i_lo >> 2);
    const int nl = l + (int)((int64_t)(h - l) * i_lo / 128);
    if (c < 128) {
      const int vh = __shfl_sync(kFullMask, pick4(v, c & 3), c >> 2);
      h = l + (int)((int64_t)(h - l) * c / 128);
      ind_h = vh;
    }
    l = nl;
    ind_l = vl;
  }
  return ReqBracket{l, ind_l, ind_h};
}

// Bounded wait that gives up (and raises the pair's error flag) on timeout or once the flag is up.
__device__ __forceinline__ bool wait_or_fail(uint32_t bar, uint32_t parity, volatile int* err) {
  if (*err) return false;
  if (tc::mbar_wait(bar, parity)) return true;
  *err = 1;
  return false;
}

template <int D, int G>
__global__ void __launch_bounds__(DecCfg<D, G>::THREADS, 1) decode_split_kernel(const DecodeParams p) {
  using C = DecCfg<D, G>;
  constexpr int NH = C::NH;
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = warp & (C::NPAIR - 1);
  const bool is_producer = warp >= C::NPAIR;
  const int kvh = blockIdx.y;
  const int B = p.batch;
  const int32_t* ind = p.kv_indptr;
  if ((sbase & 1023u) != 0) return;  // swizzle atoms need a 1024-byte aligned window

  const uint32_t ring = sbase + pair * C::RING;
  const uint32_t bars = sbase + C::BAR_OFF + 8u * (pair * 2 * C::STAGES);
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (C::STAGES + s); };
  volatile int* err = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 8 * C::NBAR) + pair;

  // ---- set-up (shared memory only): barriers; Q rows of absent heads stay zero throughout
  if (tid == 0) {
    for (int i = 0; i < C::NPAIR * 2 * C::STAGES; ++i) tc::mbar_init(sbase + C::BAR_OFF + 8u * i, 32);
    for (int i = 0; i < C::NPAIR; ++i) reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 8 * C::NBAR)[i] = 0;
    tc::fence_mbarrier_init();
  }
  for (int i = tid; i < C::NPAIR * C::STAGES * (C::Q_BYTES / 16); i += C::THREADS) {
    const int slot = i / (C::Q_BYTES / 16), c = i % (C::Q_BYTES / 16);
    sts128_zero(sbase + slot * C::SLOT + 2 * C::KV_BYTES + c * 16);
  }
  __syncthreads();
  // Launched as a programmatic dependent of the previous kernel in the stream: the set-up
  // above overlapped its tail; from here on its writes are visible and its reads are done,
  // so no global memory is touched before this point.  (A no-op for an ordinary launch.)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // let the combine kernel's CTAs launch now; they wait for this grid's memory to be visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- this pair's chunk (chunk index vc of the KV head) and its first request
  const int vc = blockIdx.x * C::NPAIR + pair;
  const int T = __ldg(ind + B);
  const int CL = decode_chunk_len(T, p.num_splits, p.min_chunk, p.part_pitch);
  const int lo = (vc < p.num_splits) ? (int)min((int64_t)vc * CL, (int64_t)T) : T;
  const int hi = min(lo + CL, T);
  ReqBracket first{0, 0, T};
  if (lo < hi) first = locate_request(ind, B, lo, T, lane);

  if (lo < hi && is_producer) {
    // ======================= producer warp: gathers the chunk's K / V rows slot by slot
    TileIter<C::BK> it;
    it.start_at(first.b, first.end, lo, hi);
    const size_t head_stride = (size_t)p.num_kv_heads * D;
    const unsigned nslots = (unsigned)p.num_slots;
    auto slot_id = [&](const TileIter<C::BK>& t) {  // lane k: slot id of key k of the slot, or -1
      const int flat = t.start + lane;
      return (t.valid(hi) && flat < t.end)
                 ? ldg_nc_i32(p.req_to_token + (int64_t)t.b * p.r2t_stride + (flat - __ldg(ind + t.b)))
                 : -1;
    };
    int my_id = slot_id(it);
    for (int i = 0; it.valid(hi); ++i) {
      const int s = i % C::STAGES;
      if (i >= C::STAGES && !wait_or_fail(empty(s), (uint32_t)((i / C::STAGES - 1) & 1), err)) break;
      const uint32_t kst = ring + s * C::SLOT, vst = kst + C::KV_BYTES, qst = vst + C::KV_BYTES;
      if (it.opens_piece(ind, lo)) {  // first slot of a piece: its G query rows
        const uint16_t* qsrc = p.q + ((size_t)it.b * p.num_qo_heads + (size_t)kvh * G) * D;
        for (int j = lane; j < G * C::CPR; j += 32) {
          const int g = j / C::CPR, c = j % C::CPR;
          cp_async16(qst + sw128(g, c, C::QROWS), qsrc + (size_t)g * D + c * 8, true);
        }
      }
      // lane -> chunk (lane % CPR) of keys (r * 32 + lane) / CPR, r = 0 .. KV_IT-1
#pragma unroll
      for (int r = 0; r < C::KV_IT; ++r) {
        const int flat = r * 32 + lane;
        const int key = flat / C::CPR, c = flat % C::CPR;
        const int id = __shfl_sync(kFullMask, my_id, key);
        const bool valid = (unsigned)id < nslots;  // padding and out-of-range ids read as zeros
        const size_t off = valid ? (size_t)id * head_stride + (size_t)kvh * D + c * 8 : 0;
        const uint32_t o = sw128(key, c, C::BK);
        cp_async16(kst + o, p.k_pool + off, valid);
        cp_async16(vst + o, p.v_pool + off, valid);
      }
      cp_async_arrive_noinc(full(s));  // completes once this lane's copies (and older ones) land
      it.next(ind, B, hi);
      my_id = slot_id(it);
    }
    cp_async_wait<0>();
  } else if (lo < hi) {
    // ======================= consumer warp: online softmax over the chunk's slots
    // Transposed products so the 16-row MMA side is keys / head_dim, not the few heads:
    //   S^T (32 keys x 8 heads) = K Q^T,   O^T (D x 8 heads) += V^T P^T.
    const int g4 = lane >> 2, t4 = lane & 3;  // fragment row / column-pair index
    const int lrow = lane & 7, lmat = lane >> 3;  // ldmatrix: row within / index of the 8x8 matrix
    const float scale = p.scale_log2;
    TileIter<C::BK> it;
    it.start_at(first.b, first.end, lo, hi);
    uint32_t qb[NH][C::KSTEPS][2];  // Q^T as the B operand (n = heads), per k-step
    float acc[C::MT_D][NH][4];      // O^T: rows d = 16md + g4 (+8), heads 8nh + 2t4 (+1)
    float m_run[NH][2], l_thr[NH][2];  // heads 8nh + 2t4 + e: reference max (lazy), sum
    float m_max[NH][2];                // exact running max, for the (max, sum) partial
    for (int i = 0; it.valid(hi); ++i) {
      const int s = i % C::STAGES;
      const bool opens = it.opens_piece(ind, lo), closes = it.closes_piece(ind, hi);
      const int nkeys = it.end - it.start;  // valid keys of the slot; the rest are masked
      if (!wait_or_fail(full(s), (uint32_t)((i / C::STAGES) & 1), err)) break;
      const uint32_t kst = ring + s * C::SLOT, vst = kst + C::KV_BYTES, qst = vst + C::KV_BYTES;

      if (opens) {  // new request piece: its query rows, fresh softmax state
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
          for (int kk = 0; kk < C::KSTEPS; kk += 2) {
            // matrices: heads 8nh .. 8nh+7 at chunks 2kk, 2kk+1, 2kk+2, 2kk+3
            ldsm_x4(qst + sw128(8 * nh + lrow, 2 * kk + lmat, C::QROWS), qb[nh][kk][0], qb[nh][kk][1],
                    qb[nh][kk + 1][0], qb[nh][kk + 1][1]);
          }
#pragma unroll
        for (int md = 0; md < C::MT_D; ++md)
#pragma unroll
          for (int nh = 0; nh < NH; ++nh) acc[md][nh][0] = acc[md][nh][1] = acc[md][nh][2] = acc[md][nh][3] = 0.f;
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) {
          m_run[nh][0] = m_run[nh][1] = -CUDART_INF_F;
          m_max[nh][0] = m_max[nh][1] = -CUDART_INF_F;
          l_thr[nh][0] = l_thr[nh][1] = 0.f;
        }
      }

      // ---- S^T = K Q^T: 2 m-tiles of 16 keys; even / odd k-steps in separate accumulators
      float sc[2][NH][4], s2[2][NH][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[mt][nh][e] = s2[mt][nh][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < C::KSTEPS; ++kk) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          // matrices: (keys 0-7, chunk 2kk), (keys 8-15, 2kk), (keys 0-7, 2kk+1), (keys 8-15, 2kk+1)
          const int key = mt * 16 + lrow + (lmat & 1) * 8, c = 2 * kk + (lmat >> 1);
          uint32_t a0, a1, a2, a3;
          ldsm_x4(kst + sw128(key, c, C::BK), a0, a1, a2, a3);
#pragma unroll
          for (int nh = 0; nh < NH; ++nh) {
            if (kk & 1) mma16816(s2[mt][nh], a0, a1, a2, a3, qb[nh][kk][0], qb[nh][kk][1]);
            else mma16816(sc[mt][nh], a0, a1, a2, a3, qb[nh][kk][0], qb[nh][kk][1]);
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
            const int key = mt * 16 + g4 + (e >> 1) * 8;
            const float x = (key < nkeys) ? (sc[mt][nh][e] + s2[mt][nh][e]) * scale : -CUDART_INF_F;
            sc[mt][nh][e] = x;
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
          m_max[nh][h] = fmaxf(m_max[nh][h], x);
        }
      float alpha[NH][2];
      bool moved = false;
#pragma unroll
      for (int nh = 0; nh < NH; ++nh)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          alpha[nh][h] = 1.f;
          // a slot whose keys are all masked keeps m = -inf; nothing it adds is nonzero
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
              pv[e] = (mr == -CUDART_INF_F) ? 0.f : fast_exp2(sc[mt][nh][2 * half + e] - mr);
              l_thr[nh][e] += pv[e];
            }
            const uint32_t h01 = float2_to_bf16x2_rn(pv[0], pv[1]);
            const float2 f01 = bf16x2_to_float2(h01);
            const uint32_t l01 = float2_to_bf16x2_rn(pv[0] - f01.x, pv[1] - f01.y);
            // (key g4 + 8 half, heads 2t4, 2t4+1) -> (head g4, keys 8 half + 2t4, +1)
            ph[mt][nh][half] = movmatrix_t(h01);
            pl[mt][nh][half] = movmatrix_t(l01);
          }

      // ---- O^T += V^T P^T over the slot's 32 keys: 2 k-steps x D / 16 m-tiles
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
        for (int md = 0; md < C::MT_D; ++md) {
          // matrices (transposed on load): (d 0-7, keys 0-7), (d 8-15, keys 0-7), (d 0-7, keys 8-15), (d 8-15, keys 8-15)
          const int key = ks * 16 + lrow + (lmat >> 1) * 8, c = 2 * md + (lmat & 1);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(vst + sw128(key, c, C::BK), a0, a1, a2, a3);
#pragma unroll
          for (int nh = 0; nh < NH; ++nh) {
            mma16816(acc[md][nh], a0, a1, a2, a3, ph[ks][nh][0], ph[ks][nh][1]);
            mma16816(acc[md][nh], a0, a1, a2, a3, pl[ks][nh][0], pl[ks][nh][1]);
          }
        }
      }

      if (closes) {
        // ---- piece finished: stage O (and m, l) in the slot's K | V area, then write it out
        __syncwarp();  // every lane's ldmatrix reads of K and V are done
        float* stg = reinterpret_cast<float*>(smem + (kst - sbase));   // [QROWS][STG_PITCH]
        float* stg_ml = stg + C::QROWS * C::STG_PITCH;                 // [QROWS][2]
        // move the reference from the lazy max to the exact one: factor 2^(m_run - m_max) in [2^-8, 1]
        float f[NH][2];
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            f[nh][h] = (m_run[nh][h] == -CUDART_INF_F) ? 1.f : fast_exp2(m_run[nh][h] - m_max[nh][h]);
            float x = l_thr[nh][h];
            x += __shfl_xor_sync(kFullMask, x, 4);
            x += __shfl_xor_sync(kFullMask, x, 8);
            x += __shfl_xor_sync(kFullMask, x, 16);
            if (g4 == 0) {
              stg_ml[(8 * nh + 2 * t4 + h) * 2 + 0] = m_max[nh][h];
              stg_ml[(8 * nh + 2 * t4 + h) * 2 + 1] = x * f[nh][h];
            }
          }
#pragma unroll
        for (int md = 0; md < C::MT_D; ++md)
#pragma unroll
          for (int nh = 0; nh < NH; ++nh)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              stg[(8 * nh + 2 * t4 + (e & 1)) * C::STG_PITCH + md * 16 + g4 + (e >> 1) * 8] =
                  acc[md][nh][e] * f[nh][e & 1];
        __syncwarp();
        const int b = it.b;
        const int rb = __ldg(ind + b), re = __ldg(ind + b + 1);
        const bool direct = (p.out != nullptr) && rb >= lo && re <= hi;  // whole request in this chunk
        const size_t qh0 = (size_t)b * p.num_qo_heads + (size_t)kvh * G;
        if (direct) {
          // lane -> 8 consecutive d of one head: bf16(O / l), 16-byte stores
          for (int j = lane; j < G * (D / 8); j += 32) {
            const int h = j / (D / 8), d0 = (j % (D / 8)) * 8;
            const float L = stg_ml[h * 2 + 1];
            const float inv = (L > 0.f) ? 1.f / L : 0.f;
            const float* src = stg + h * C::STG_PITCH + d0;
            uint4 v;
            v.x = float2_to_bf16x2_rn(src[0] * inv, src[1] * inv);
            v.y = float2_to_bf16x2_rn(src[2] * inv, src[3] * inv);
            v.z = float2_to_bf16x2_rn(src[4] * inv, src[5] * inv);
            v.w = float2_to_bf16x2_rn(src[6] * inv, src[7] * inv);
            *reinterpret_cast<uint4*>(p.out + (qh0 + h) * D + d0) = v;
          }
        } else {
          const int slot = vc - rb / CL;
          for (int j = lane; j < G * (D / 4); j += 32) {
            const int h = j / (D / 4), d0 = (j % (D / 4)) * 4;
            const float* src = stg + h * C::STG_PITCH + d0;
            *reinterpret_cast<float4*>(p.o_part + ((qh0 + h) * p.part_pitch + slot) * D + d0) =
                make_float4(src[0], src[1], src[2], src[3]);
          }
          for (int h = lane; h < G; h += 32) {
            const float M = stg_ml[h * 2 + 0];
            float2 ml;
            ml.x = (M == -CUDART_INF_F) ? M : M * kLn2;  // natural-log units
            ml.y = stg_ml[h * 2 + 1];
            *reinterpret_cast<float2*>(p.ml_part + ((qh0 + h) * p.part_pitch + slot) * 2) = ml;
          }
        }
      }
      __syncwarp();
      tc::mbar_arrive(empty(s));  // this slot may be refilled
      it.next(ind, B, hi);
    }
  }
  __syncthreads();
  if (*err && lo < hi && !is_producer) {
    // a wait timed out: poison every output this pair owns so the call reads as failed
    TileIter<C::BK> it;
    it.first(ind, B, lo, hi);
    for (; it.valid(hi); it.next(ind, B, hi)) {
      if (!it.closes_piece(ind, hi)) continue;
      const int s = vc - __ldg(ind + it.b) / CL;
      for (int i = lane; i < G * D; i += 32) {
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
  const bool live = wid < p.batch * p.num_qo_heads;
  const int b = live ? wid / p.num_qo_heads : 0;
  // Split count of request b: the chunks that overlap it (token-balanced schedule), or the
  // caller's explicit count.
  auto split_count = [&]() {
    if (p.kv_indptr == nullptr) return p.num_splits;
    const int T = __ldg(p.kv_indptr + p.batch);
    const int CL = decode_chunk_len(T, p.num_splits, p.min_chunk, p.part_pitch);
    const int a = __ldg(p.kv_indptr + b), e = __ldg(p.kv_indptr + b + 1);
    return (e > a) ? (e - 1) / CL - a / CL + 1 : 0;
  };
  // Right after this call's split kernel, kv_indptr (an input the split kernel does not write)
  // is read before the wait: that kernel has already passed its own wait on the kernels before
  // it.  After any other kernel it is read only once the wait has returned.
  int S = (live && p.indptr_before_wait) ? split_count() : 0;
  // launched as a programmatic dependent of the previous kernel: wait until its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (live && !p.indptr_before_wait) S = split_count();
  // the next kernel in the stream may start its shared-memory set-up now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!live) return;
  if (p.kv_indptr != nullptr && S == 1 && !p.combine_all) return;  // written directly by the split kernel
  const size_t base = (size_t)wid * p.part_pitch;
  const float* ml = p.ml_part + base * 2;
  using VecT = typename std::conditional<VPL == 4, float4, float2>::type;
  const VecT* o = reinterpret_cast<const VecT*>(p.o_part + base * D) + lane;  // slot s at o[s * 32]
  auto fma_vec = [](float (&a)[VPL], float w, const VecT& v) {
    if constexpr (VPL == 4) {
      a[0] += w * v.x; a[1] += w * v.y; a[2] += w * v.z; a[3] += w * v.w;
    } else {
      a[0] += w * v.x; a[1] += w * v.y;
    }
  };
  float acc[VPL];
#pragma unroll
  for (int e = 0; e < VPL; ++e) acc[e] = 0.f;
  float L = 0.f;
  constexpr int kFast = 8;  // up to this many slots: every load of the row in one round
  if (S <= kFast) {
    float2 mlj = make_float2(-CUDART_INF_F, 0.f);
    if (lane < S) mlj = *reinterpret_cast<const float2*>(ml + 2 * lane);
    VecT v[kFast];
#pragma unroll
    for (int k = 0; k < kFast; ++k)
      if (k < S) v[k] = o[k * 32];
    float M = mlj.x;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
    if (M != -CUDART_INF_F) {
      const float wj = (mlj.x == -CUDART_INF_F) ? 0.f : exp2f((mlj.x - M) * kLog2e);
      L = wj * mlj.y;
#pragma unroll
      for (int k = 0; k < kFast; ++k)
        if (k < S) fma_vec(acc, __shfl_sync(kFullMask, wj, k), v[k]);
    }
  } else {
    float M = -CUDART_INF_F;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, ml[2 * s]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
    // O = sum_s w_s o_s, L = sum_s w_s l_s with w_s = e^(m_s - M), 32 slots at a time:
    // lane j computes w of slot s0 + j; the o_s loads of four slots are issued together.
    if (M != -CUDART_INF_F) {
      for (int s0 = 0; s0 < S; s0 += 32) {
        float wj = 0.f;
        if (s0 + lane < S) {
          const float2 mlj = *reinterpret_cast<const float2*>(ml + 2 * (s0 + lane));
          wj = (mlj.x == -CUDART_INF_F) ? 0.f : exp2f((mlj.x - M) * kLog2e);
          L += wj * mlj.y;
        }
        const int n = min(32, S - s0);
        int j = 0;
        for (; j + 4 <= n; j += 4) {
          const VecT v0 = o[(s0 + j) * 32], v1 = o[(s0 + j + 1) * 32];
          const VecT v2 = o[(s0 + j + 2) * 32], v3 = o[(s0 + j + 3) * 32];
          fma_vec(acc, __shfl_sync(kFullMask, wj, j), v0);
          fma_vec(acc, __shfl_sync(kFullMask, wj, j + 1), v1);
          fma_vec(acc, __shfl_sync(kFullMask, wj, j + 2), v2);
          fma_vec(acc, __shfl_sync(kFullMask, wj, j + 3), v3);
        }
        for (; j < n; ++j) fma_vec(acc, __shfl_sync(kFullMask, wj, j), o[(s0 + j) * 32]);
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(kFullMask, L, off);
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
  cfg.gridDim = dim3((p.num_splits + C::NPAIR - 1) / C::NPAIR, p.num_kv_heads);  // NPAIR chunks per CTA
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
