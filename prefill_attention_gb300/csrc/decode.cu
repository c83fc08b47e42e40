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
//   * Slot-balanced split schedule.  Each request's keys are cut into 32-key slots from its
//     first key (the last one possibly short); for each KV head the batch's slots lie end to
//     end (request b starts at slot SP_b) and are cut into equal chunks of C slots, one warp
//     pair per chunk, so every pair runs the same number of ring slots however skewed
//     seq_lens is.  (Slots, not keys: with every pair's slots in flight the memory system is
//     saturated and a pair's pace is its slots in flight per round trip, so a short slot
//     costs as much as a full one.)  A chunk may hold the tail of one request and the head
//     of the next; each such piece produces one partial, indexed by (chunk - SP_b / C), and a
//     request that lies inside one chunk is written to the output directly.  C depends only
//     on kv_indptr, the grid and a host-supplied floor, so the combine recomputes it.
//   * One CTA per SM with four independent (producer, consumer) warp pairs, each with its
//     own chunk and its own ring of 32-key slots (K, V and the piece's query rows):
//       producer -- lane k reads the slot id of key k (one slot ahead) and gathers the K and
//               V rows with 16-byte cp.async into 128-byte-swizzled tiles (chunk c of row r
//               at c ^ (r & 7)); cp.async.mbarrier.arrive publishes a slot when it lands, so
//               the producer never waits for its own copies, only for a free slot.
//       consumer -- S^T = K Q^T and O^T += V^T P^T as warp-level bf16 MMAs (m16n8k16, fp32
//               accumulators in registers, operands by ldmatrix): the 16-row side is keys or
//               head_dim and the 8-wide side the G query heads, so one K/V load serves all
//               of them with little padding.  P goes to the B-operand layout by movmatrix,
//               split into hi = bf16(p) and lo = bf16(p - hi), both through the MMA (p to
//               ~2^-17 relative).  Base-2 softmax with a lazy rescale (the reference max moves
//               only when a score exceeds it by more than 2^8); the exact max is kept for the
//               partial.  At a piece end the result is staged through the slot just used and
//               written with 16-byte stores.
//   * Launched as a programmatic dependent: shared-memory set-up and an L2 warm-up of each
//     pair's first slots (from tables read through L2 only; prefetch hints, nothing kept)
//     run before griddepcontrol.wait, so the first misses overlap the previous kernel.
//   * Variants of the same kernel (template MODE): an explicit mask (page "astrai/extension
//     @6f67ba8", prefill-mask commit) -- the producer copies each slot's 32 mask bytes next to
//     its K/V and the consumer gives masked keys exactly zero weight; and a contiguous K/V
//     cache (stride-addressing and layout commits) -- rows are addressed from the request, the
//     position and the KV head, with no slot-id load.  The plain kernel keeps its own
//     parameter block and code.
//   * Measured alternatives: a CUDA-core version was issue bound (~550 instructions per
//     4 KB of K/V); a tcgen05 version with S^T / O^T accumulators in tensor memory spent
//     ~150 cycles per M=128 x N=16 x K=16 MMA on the critical path; TMA tile::gather4 for
//     the row gather delivered ~12 GB/s per SM.
#include <cuda_runtime.h>
#include <math_constants.h>

#include <type_traits>

#include "common.cuh"
#include "tcgen05.cuh"

namespace astr {

// Split schedule, shared by the split and the combine kernels.  Request b's keys are cut
// into slots of kSlotKeys keys from its first key (the last slot possibly short); the
// batch's slots lie end to end in request order (request b's first slot is SP_b, the sum of
// the slot counts of the requests before it) and are cut into chunks of CS slots.  Every
// chunk thus holds the same number of ring slots, which is what sets a chunk's time: the
// gather pipeline keeps a fixed number of slots in flight, full or not.
constexpr int kSlotKeys = 32;
__device__ __forceinline__ int slots_of(int n) { return n > 0 ? (n + kSlotKeys - 1) / kSlotKeys : 0; }

// Chunk length in slots for S slots over n_chunks chunks.
__device__ __forceinline__ int decode_chunk_slots(int S, int n_chunks, int min_chunk, int max_splits) {
  if (max_splits <= 1) return S > 0 ? S : 1;
  const int c = (S + n_chunks - 1) / n_chunks;
  return c > min_chunk ? c : min_chunk;
}

// Warp-cooperative: the batch's slot count (x) and the slots of requests b < `before` (y).
__device__ __forceinline__ int2 slot_totals(const int32_t* ind, int B, int before, int lane) {
  int tot = 0, pre = 0;
#pragma unroll 4
  for (int base = 0; base < B; base += 32) {
    const int i = base + lane;
    const int x = __ldg(ind + min(i, B));
    const int nx = __ldg(ind + min(base + 32, B));
    int y = __shfl_down_sync(0xffffffffu, x, 1);
    if (lane == 31) y = nx;
    const int sl = (i < B) ? slots_of(y - x) : 0;
    tot += sl;
    if (i < before) pre += sl;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    pre += __shfl_xor_sync(0xffffffffu, pre, o);
  }
  return make_int2(tot, pre);
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
  // rows live in 128-byte-swizzled column blocks of 64 elements; a 32-element row (d = 32)
  // takes the first half of a block's 128-byte row
  static constexpr int NCB = (D + 63) / 64;        // column blocks per row
  static constexpr int KV_BYTES = BK * NCB * 128;  // K (or V) part of a slot
  static constexpr int Q_BYTES = QROWS * NCB * 128;
  static constexpr int SLOT = 2 * KV_BYTES + Q_BYTES;   // K | V | Q
  static constexpr int STAGES_FIT = (220 * 1024) / (NPAIR * SLOT);
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;  // ring slots per pair
  static constexpr int RING = STAGES * SLOT;
  static constexpr int BAR_OFF = NPAIR * RING;
  static constexpr int NBAR = NPAIR * 2 * STAGES;  // full[pair][slot], empty[pair][slot]
  static constexpr int MASK_OFF = BAR_OFF + NBAR * 8 + 16 * 4;  // after the per-pair error flags
  static constexpr int MASK_BYTES = BK;                           // explicit-mask bytes of a ring slot
  static constexpr int SMEM_BYTES = MASK_OFF;                     // without an explicit mask
  static constexpr int SMEM_BYTES_MASKED = MASK_OFF + NPAIR * STAGES * MASK_BYTES;
  static constexpr int KSTEPS = D / 16;            // MMA k-steps over head_dim (S^T = K Q^T)
  static constexpr int MT_D = D / 16;              // 16-row m-tiles over head_dim (O^T = V^T P^T)
  static constexpr int STG_PITCH = D + 4;          // fp32 staging row pitch (conflict-free writes)
  static_assert(G <= 16, "at most 16 query heads per KV head");
  static_assert(D == 32 || D % 64 == 0, "head_dim 32 or a multiple of 64");
  static_assert(STAGES >= 2, "a ring needs two slots");
  static_assert(SLOT % 1024 == 0 && KV_BYTES % 1024 == 0, "swizzle atoms");
  static_assert((QROWS * STG_PITCH + 2 * QROWS) * 4 <= 2 * KV_BYTES, "piece staging fits in K | V");
  static_assert(SMEM_BYTES_MASKED <= 227 * 1024, "shared memory budget");
  static_assert(MASK_OFF % 16 == 0 && MASK_BYTES % 16 == 0, "16-byte cp.async of mask bytes");
};

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

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

// The request that holds slot g of the batch: b, its first slot, its keys [ind_b, ind_b1).
struct SlotBracket {
  int b, spb, ind_b, ind_b1;
};
// Warp-cooperative lookup of the request that holds slot `g` (< the batch's slot count):
// blocks of 32 requests in order, an inclusive scan of their slot counts per block.  A
// batch of up to 32 requests takes one round of loads (already in L1 after slot_totals).
__device__ __forceinline__ SlotBracket locate_slot(const int32_t* ind, int B, int g, int lane) {
  int carry = 0;
  for (int base = 0; base < B; base += 32) {
    const int i = base + lane;
    const int x = __ldg(ind + min(i, B));
    const int nx = __ldg(ind + min(base + 32, B));
    int y = __shfl_down_sync(kFullMask, x, 1);
    if (lane == 31) y = nx;
    const int sl = (i < B) ? slots_of(y - x) : 0;
    int incl = sl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += t;
    }
    const int total = __shfl_sync(kFullMask, incl, 31);
    if (g < carry + total) {  // warp-uniform
      const int f = __ffs(__ballot_sync(kFullMask, carry + incl > g)) - 1;
      SlotBracket r;
      r.b = base + f;
      r.spb = carry + __shfl_sync(kFullMask, incl - sl, f);
      r.ind_b = __shfl_sync(kFullMask, x, f);
      r.ind_b1 = __shfl_sync(kFullMask, y, f);
      return r;
    }
    carry += total;
  }
  return SlotBracket{B, carry, 0, 0};  // g past the last slot (callers never ask)
}

// Walks the ring slots of one chunk (batch slots [ls, hs)): one request slot at a time,
// so a ring slot never spans two requests.
template <int BK>
struct TileIter {
  int b, spb, ind_b, ind_b1;  // current request: first batch slot, keys [ind_b, ind_b1)
  int g;                      // current batch slot
  int start, end;             // its keys [start, end)
  __device__ __forceinline__ int nslots() const { return slots_of(ind_b1 - ind_b); }
  __device__ __forceinline__ void set_keys() {
    start = ind_b + (g - spb) * BK;
    end = min(start + BK, ind_b1);
  }
  __device__ __forceinline__ void start_at(const SlotBracket& f, int ls) {
    b = f.b;
    spb = f.spb;
    ind_b = f.ind_b;
    ind_b1 = f.ind_b1;
    g = ls;
    set_keys();
  }
  __device__ __forceinline__ void next(const int32_t* ind, int B, int hs) {
    if (++g >= hs) return;
    while (g >= spb + nslots() && b < B - 1) {  // on to the next request that has keys
      spb += nslots();
      ++b;
      ind_b = ind_b1;
      ind_b1 = __ldg(ind + b + 1);
    }
    set_keys();
  }
  __device__ __forceinline__ bool valid(int hs) const { return g < hs; }
  __device__ __forceinline__ bool opens_piece(int ls) const { return g == max(ls, spb); }
  __device__ __forceinline__ bool closes_piece(int hs) const { return g + 1 == min(hs, spb + nslots()); }
};

// L2 warm-up of a chunk's first ring slots, run before the dependency wait while the
// previous kernel in the stream may still be writing the tables: kv_indptr and req_to_token
// are read with L2-only loads (so no stale line stays in L1 past the wait), nothing read is
// kept, and only prefetch hints for the first request's K/V rows come out (prefetching its
// query rows as well measured slower).  Every address
// is clamped to its buffer whatever the values read.  kv_indptr is read in R rounds of 32
// requests, one coalesced load and one broadcast per round, all rounds issued together (R is
// picked from the batch size: the unrolled rounds cost latency even when idle); batches of
// more than 256 requests skip the warm-up.
// Prefetch hints into L2 for the K/V rows of the first n_slots slots of a chunk that starts at
// batch slot ls inside request b (first slot spb, keys [ib, ib1) of the flat key range).
template <int D, int G, int BK, bool CONTIG>
__device__ __forceinline__ void warm_slots_from(const DecodeParams& p, const KvStrides& ks, int b, int spb, int ib,
                                                int ib1, int ls, int kvh, int n_slots, int lane) {
  const int k0 = (ls - spb) * BK;  // the chunk's first key within request b
  const size_t head_stride = (size_t)p.num_kv_heads * D;
  for (int k = lane; k < n_slots * BK; k += 32) {
    const int key = k0 + k;
    size_t row;
    if constexpr (CONTIG) {
      if (key < 0 || key >= ib1 - ib || key >= ks.max_len) continue;
      row = (size_t)b * ks.batch + (size_t)key * ks.token + (size_t)kvh * ks.head;
    } else {
      if (key < 0 || key >= ib1 - ib || (int64_t)key >= p.r2t_stride) continue;
      const int id = ldcg_i32(p.req_to_token + (int64_t)b * p.r2t_stride + key);
      if ((uint64_t)(uint32_t)id >= (uint64_t)p.num_slots) continue;  // negative ids wrap past num_slots
      row = (size_t)id * head_stride + (size_t)kvh * D;
    }
    const uint16_t* kr = p.k_pool + row;
    const uint16_t* vr = p.v_pool + row;
#pragma unroll
    for (int off = 0; off < D; off += 64) {  // 128-byte lines
      prefetch_l2(kr + off);
      prefetch_l2(vr + off);
    }
  }
}

template <int D, int G, int BK, int R, bool CONTIG>
__device__ __forceinline__ void warm_first_slots(const DecodeParams& p, const KvStrides& ks, int vc, int kvh,
                                                 int n_slots, int lane) {
  const int B = p.batch;
  const int32_t* ind = p.kv_indptr;
  int x[R], y[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (32 * r < B) {
      x[r] = ldcg_i32(ind + min(32 * r + lane, B));
      y[r] = ldcg_i32(ind + min(32 * r + 32, B));  // the same address in every lane
    }
  }
  int sl[R], incl[R], carry = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    sl[r] = 0;
    incl[r] = carry;
    if (32 * r < B) {
      int nx = __shfl_down_sync(kFullMask, x[r], 1);
      if (lane == 31) nx = y[r];
      y[r] = nx;  // y[r] = ind[32 r + lane + 1]
      sl[r] = (32 * r + lane < B) ? slots_of(y[r] - x[r]) : 0;
      int c = sl[r];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFullMask, c, o);
        if (lane >= o) c += t;
      }
      incl[r] = carry + c;
      carry += __shfl_sync(kFullMask, c, 31);
    }
  }
  const int S_tot = carry;
  const int CS = decode_chunk_slots(S_tot, p.num_splits, p.min_chunk, p.part_pitch);
  const int ls = (vc < p.num_splits) ? (int)min((int64_t)vc * CS, (int64_t)S_tot) : S_tot;
  if (S_tot <= 0 || ls >= S_tot) return;
  int b = -1, spb = 0, ib = 0, ib1 = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (b < 0 && 32 * r < B) {
      const unsigned lanes = __ballot_sync(kFullMask, incl[r] > ls);
      if (lanes != 0u) {
        const int f = __ffs(lanes) - 1;
        b = 32 * r + f;
        spb = __shfl_sync(kFullMask, incl[r] - sl[r], f);
        ib = __shfl_sync(kFullMask, x[r], f);
        ib1 = __shfl_sync(kFullMask, y[r], f);
      }
    }
  }
  if (b < 0 || b >= B) return;
  warm_slots_from<D, G, BK, CONTIG>(p, ks, b, spb, ib, ib1, ls, kvh, n_slots, lane);
}

// Bounded wait, agreed by the whole warp, that gives up (and raises the pair's error flag) on
// timeout or once the flag is up.
__device__ __forceinline__ bool wait_or_fail(uint32_t bar, uint32_t parity, volatile int* err, uint32_t limit) {
  const bool ok = __all_sync(kFullMask, *err == 0 && tc::mbar_wait(bar, parity, limit));
  if (!ok) *err = 1;
  return ok;
}

// Kernel variants: MODE bit 0 = explicit mask, bit 1 = contiguous (stride-addressed) K/V cache
// instead of the slot table, bit 2 = query / output by strides alone (the mask and contiguous
// variants always take strides).  MODE 0 takes DecodeParams alone and the packed query /
// output layout at compile time; the others take the longer block below, so the plain
// kernel's parameter block and code stay as they are (a runtime row pitch there measurably
// slows the split step).
constexpr int kModeMask = 1, kModeContig = 2, kModeStrided = 4;
struct DecodeParamsExt {
  DecodeParams p;
  DecodeMask m;
  KvStrides s;
  QoStrides qo;
};
template <int MODE> struct SplitArg { using type = DecodeParamsExt; };
template <> struct SplitArg<0> { using type = DecodeParams; };
// (host and device: the launcher reads the grid shape through params_of too)
__host__ __device__ __forceinline__ const DecodeParams& params_of(const DecodeParams& a) { return a; }
__host__ __device__ __forceinline__ const DecodeParams& params_of(const DecodeParamsExt& a) { return a.p; }
__host__ __device__ __forceinline__ DecodeMask mask_of(const DecodeParams&) { return DecodeMask{nullptr, 0, 0}; }
__host__ __device__ __forceinline__ DecodeMask mask_of(const DecodeParamsExt& a) { return a.m; }
__host__ __device__ __forceinline__ KvStrides strides_of(const DecodeParams&) { return KvStrides{0, 0, 0, 0}; }
__host__ __device__ __forceinline__ KvStrides strides_of(const DecodeParamsExt& a) { return a.s; }
__host__ __device__ __forceinline__ QoStrides qo_of(const DecodeParams&) { return QoStrides{0, 0, 0, 0}; }
__host__ __device__ __forceinline__ QoStrides qo_of(const DecodeParamsExt& a) { return a.qo; }

template <int D, int G, int MODE>
__global__ void __launch_bounds__(DecCfg<D, G>::THREADS, 1) decode_split_kernel(const typename SplitArg<MODE>::type arg) {
  using C = DecCfg<D, G>;
  constexpr bool MASK = (MODE & kModeMask) != 0, CONTIG = (MODE & kModeContig) != 0, STRIDED = MODE != 0;
  const DecodeParams& p = params_of(arg);
  constexpr int NH = C::NH;
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = warp & (C::NPAIR - 1);
  const bool is_producer = warp >= C::NPAIR;
  const int kvh = blockIdx.y;
  const int B = p.batch;
  const int32_t* ind = p.kv_indptr;
  // swizzle atoms need a 1024-byte aligned window; without one the pairs do no work and
  // poison their outputs (the error flags start raised)
  const bool smem_ok = (sbase & 1023u) == 0;

  const uint32_t ring = sbase + pair * C::RING;
  const uint32_t bars = sbase + C::BAR_OFF + 8u * (pair * 2 * C::STAGES);
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (C::STAGES + s); };
  const uint32_t mask_ring = sbase + C::MASK_OFF + pair * C::STAGES * C::MASK_BYTES;  // explicit-mask bytes
  volatile int* err = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 8 * C::NBAR) + pair;

  // ---- set-up (shared memory only): barriers; Q rows of absent heads stay zero throughout
  if (tid == 0) {
    for (int i = 0; i < C::NPAIR * 2 * C::STAGES; ++i) tc::mbar_init(sbase + C::BAR_OFF + 8u * i, 32);
    for (int i = 0; i < C::NPAIR; ++i) reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 8 * C::NBAR)[i] = smem_ok ? 0 : 1;
    tc::fence_mbarrier_init();
  }
  for (int i = tid; i < C::NPAIR * C::STAGES * (C::Q_BYTES / 16); i += C::THREADS) {
    const int slot = i / (C::Q_BYTES / 16), c = i % (C::Q_BYTES / 16);
    sts128_zero(sbase + slot * C::SLOT + 2 * C::KV_BYTES + c * 16);
  }
  __syncthreads();
  // ---- this pair's chunk (chunk index vc of the KV head): batch slots [ls, hs), and the
  // request that holds slot ls.  Planned after the dependency wait below, or before it when
  // the caller declares the index arrays untouched by the preceding kernel (they are then
  // final already, and the planning overlaps that kernel).
  const int vc = blockIdx.x * C::NPAIR + pair;
  int S_tot = 0, CS = 1, ls = 0, hs = 0;
  SlotBracket first{0, 0, 0, 0};
  auto plan_chunk = [&]() {
    S_tot = slot_totals(ind, B, 0, lane).x;
    CS = decode_chunk_slots(S_tot, p.num_splits, p.min_chunk, p.part_pitch);
    ls = (vc < p.num_splits) ? (int)min((int64_t)vc * CS, (int64_t)S_tot) : S_tot;
    hs = min(ls + CS, S_tot);
    if (ls < hs) first = locate_slot(ind, B, ls, lane);
  };
  if (p.early_index) {
    // the index arrays are final: plan now and warm L2 with the chunk's first slots from the plan
    plan_chunk();
    if (is_producer && ls < hs && B <= 256)
      warm_slots_from<D, G, C::BK, CONTIG>(p, strides_of(arg), first.b, first.spb, first.ind_b, first.ind_b1, ls, kvh,
                                           C::STAGES, lane);
  } else if (is_producer && B <= 32) {
    // before the wait: warm L2 with this pair's first ring slots (prefetch hints only, from
    // tables read through L2 that may still be changing; see warm_first_slots)
    warm_first_slots<D, G, C::BK, 1, CONTIG>(p, strides_of(arg), vc, kvh, C::STAGES, lane);
  } else if (is_producer && B <= 256) {
    warm_first_slots<D, G, C::BK, 8, CONTIG>(p, strides_of(arg), vc, kvh, C::STAGES, lane);
  }
  // Launched as a programmatic dependent of the previous kernel in the stream: the set-up
  // above overlapped its tail; from here on its writes are visible and its reads are done,
  // so nothing read before this point is used (but the index arrays under early_index).
  // (A no-op for an ordinary launch.)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // let the combine kernel's CTAs launch now; they wait for this grid's memory to be visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!p.early_index) plan_chunk();

  if (ls < hs && smem_ok && is_producer) {
    // ======================= producer warp: gathers the chunk's K / V rows slot by slot
    TileIter<C::BK> it;
    it.start_at(first, ls);
    const size_t head_stride = (size_t)p.num_kv_heads * D;
    const unsigned nslots = (unsigned)p.num_slots;
    // lane k: slot id of key k of the slot (-1 past the request's keys); `real` = the key is one
    // of the request's.  A real key whose position is past the table row, or whose id (checked
    // when it is used, one slot later) lies outside the pool, reads as zeros and is reported.
    bool bad_input = false, my_real = false;
    auto slot_id = [&](const TileIter<C::BK>& t, bool& real) {
      if constexpr (CONTIG) {
        real = false;
        return 0;  // contiguous cache: rows are addressed by position, no ids
      } else {
        const int flat = t.start + lane;
        real = t.valid(hs) && flat < t.end;
        if (real && flat - t.ind_b >= p.r2t_stride) {
          bad_input = true;
          real = false;
        }
        return real ? ldg_nc_i32(p.req_to_token + (int64_t)t.b * p.r2t_stride + (flat - t.ind_b)) : -1;
      }
    };
    int my_id = slot_id(it, my_real);
    int i = 0;  // ring slots published so far
    for (; it.valid(hs); ++i) {
      const int s = i % C::STAGES;
      if (i >= C::STAGES && !wait_or_fail(empty(s), (uint32_t)((i / C::STAGES - 1) & 1), err, p.wait_limit)) break;
      const uint32_t kst = ring + s * C::SLOT, vst = kst + C::KV_BYTES, qst = vst + C::KV_BYTES;
      if (it.opens_piece(ls)) {  // first slot of a piece: its G query rows
        const uint16_t* qsrc;
        size_t qpitch;  // elements between the query rows of consecutive heads
        if constexpr (STRIDED) {
          const QoStrides qo = qo_of(arg);
          qsrc = p.q + (size_t)it.b * qo.q_req + (size_t)kvh * G * qo.q_head;
          qpitch = (size_t)qo.q_head;
        } else {
          qsrc = p.q + ((size_t)it.b * p.num_qo_heads + (size_t)kvh * G) * D;
          qpitch = D;
        }
        for (int j = lane; j < G * C::CPR; j += 32) {
          const int g = j / C::CPR, c = j % C::CPR;
          cp_async16(qst + sw128(g, c, C::QROWS), qsrc + (size_t)g * qpitch + c * 8, true);
        }
      }
      // lane -> chunk (lane % CPR) of keys (r * 32 + lane) / CPR, r = 0 .. KV_IT-1
#pragma unroll
      for (int r = 0; r < C::KV_IT; ++r) {
        const int flat = r * 32 + lane;
        const int key = flat / C::CPR, c = flat % C::CPR;
        bool valid;
        size_t off;
        if constexpr (CONTIG) {
          // key `key` of the slot is position (start - ind_b) + key of request b; keys past the
          // request's end read as zeros
          const KvStrides ks = strides_of(arg);
          valid = key < it.end - it.start && it.start - it.ind_b + key < ks.max_len;
          off = valid ? (size_t)it.b * ks.batch + (size_t)(it.start - it.ind_b + key) * ks.token +
                            (size_t)kvh * ks.head + c * 8
                      : 0;
        } else {
          const int id = __shfl_sync(kFullMask, my_id, key);
          valid = (unsigned)id < nslots;  // padding and out-of-range ids read as zeros
          off = valid ? (size_t)id * head_stride + (size_t)kvh * D + c * 8 : 0;
        }
        const uint32_t o = sw128(key, c, C::BK);
        cp_async16(kst + o, p.k_pool + off, valid);
        cp_async16(vst + o, p.v_pool + off, valid);
      }
      if (MASK && lane < C::MASK_BYTES / 16) {
        // the slot's explicit-mask bytes: request-local positions start at a multiple of 32, and
        // a 16-byte chunk that begins inside the row (pitch a multiple of 16) ends inside it;
        // chunks past the row are zero-filled (those keys are past max_seq_len anyway)
        const int pos = it.start - it.ind_b + 16 * lane;
        const DecodeMask mk = mask_of(arg);
        const bool in_row = pos < mk.kv_pitch;
        const uint8_t* src = mk.mask + (in_row ? (int64_t)it.b * mk.req_pitch + pos : 0);
        cp_async16(mask_ring + s * C::MASK_BYTES + 16 * lane, src, in_row);
      }
      cp_async_arrive_noinc(full(s));  // completes once this lane's copies (and older ones) land
      // (checked here, after the copies are issued: a check before them costs the gather ~0.2 us)
      if constexpr (!CONTIG) bad_input |= my_real && (unsigned)my_id >= nslots;
      it.next(ind, B, hs);
      my_id = slot_id(it, my_real);
    }
    cp_async_wait<0>();
    if (*err) {
      // the consumer gave up: let the arrivals of the slots published last land (each slot's
      // newest phase; its 32 arrivals are this warp's) before the CTA's shared memory goes away
      for (int k = max(0, i - C::STAGES); k < i; ++k)
        tc::mbar_wait(full(k % C::STAGES), (uint32_t)((k / C::STAGES) & 1), tc::kWaitLimit);
    }
    if (p.status != nullptr && __any_sync(kFullMask, bad_input) && lane == 0) atomicOr(p.status, kStatusBadInput);
  } else if (ls < hs && smem_ok) {
    // ======================= consumer warp: online softmax over the chunk's slots
    // Transposed products so the 16-row MMA side is keys / head_dim, not the few heads:
    //   S^T (32 keys x 8 heads) = K Q^T,   O^T (D x 8 heads) += V^T P^T.
    const int g4 = lane >> 2, t4 = lane & 3;  // fragment row / column-pair index
    const int lrow = lane & 7, lmat = lane >> 3;  // ldmatrix: row within / index of the 8x8 matrix
    const float scale = p.scale_log2;
    TileIter<C::BK> it;
    it.start_at(first, ls);
    uint32_t qb[NH][C::KSTEPS][2];  // Q^T as the B operand (n = heads), per k-step
    float acc[C::MT_D][NH][4];      // O^T: rows d = 16md + g4 (+8), heads 8nh + 2t4 (+1)
    float m_run[NH][2], l_thr[NH][2];  // heads 8nh + 2t4 + e: reference max (lazy), sum
    float m_max[NH][2];                // exact running max, for the (max, sum) partial
    for (int i = 0; it.valid(hs); ++i) {
      const int s = i % C::STAGES;
      const bool opens = it.opens_piece(ls), closes = it.closes_piece(hs);
      const int nkeys = it.end - it.start;  // valid keys of the slot; the rest are masked
      if (!wait_or_fail(full(s), (uint32_t)((i / C::STAGES) & 1), err, p.wait_limit)) break;
      const uint32_t kst = ring + s * C::SLOT, vst = kst + C::KV_BYTES, qst = vst + C::KV_BYTES;
      // visibility of this lane's keys 16 mt + g4 + 8 hh, bit 2 mt + hh (explicit mask)
      uint32_t kvis = 0u;
      if constexpr (MASK) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          kvis |= (lds_u8(mask_ring + s * C::MASK_BYTES + 16 * (k >> 1) + g4 + 8 * (k & 1)) != 0u ? 1u : 0u) << k;
      }

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
            bool vis = key < nkeys;
            if constexpr (MASK) vis = vis && ((kvis >> (2 * mt + (e >> 1))) & 1u);
            const float x = vis ? (sc[mt][nh][e] + s2[mt][nh][e]) * scale : -CUDART_INF_F;
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
        const bool direct = (p.out != nullptr) && it.spb >= ls && it.spb + it.nslots() <= hs;  // whole request here
        const size_t qh0 = (size_t)b * p.num_qo_heads + (size_t)kvh * G;
        if (direct) {
          uint16_t* orow;  // output row of head kvh * G of request b
          size_t opitch;   // elements between the output rows of consecutive heads
          if constexpr (STRIDED) {
            const QoStrides qo = qo_of(arg);
            orow = p.out + (size_t)b * qo.o_req + (size_t)kvh * G * qo.o_head;
            opitch = (size_t)qo.o_head;
          } else {
            orow = p.out + qh0 * D;
            opitch = D;
          }
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
            *reinterpret_cast<uint4*>(orow + (size_t)h * opitch + d0) = v;
          }
        } else if (vc - it.spb / CS < p.part_pitch) {  // (a request past max_seq_len keys is not written)
          const int slot = vc - it.spb / CS;
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
      it.next(ind, B, hs);
    }
  }
  __syncthreads();
  if (*err && ls < hs && !is_producer) {
    // a wait timed out (or the window was misaligned): report it and poison every output this
    // pair owns so the call reads as failed
    if (p.status != nullptr && lane == 0) atomicOr(p.status, smem_ok ? kStatusTimeout : kStatusSmem);
    TileIter<C::BK> it;
    it.start_at(first, ls);
    for (; it.valid(hs); it.next(ind, B, hs)) {
      if (!it.closes_piece(hs)) continue;
      const int s = vc - it.spb / CS;
      for (int i = lane; i < G * D; i += 32) {
        const size_t qh = (size_t)it.b * p.num_qo_heads + (size_t)kvh * G + i / D;
        if (s < p.part_pitch) p.o_part[(qh * p.part_pitch + s) * D + i % D] = CUDART_NAN_F;
        if (p.out != nullptr) {
          const QoStrides qo = qo_of(arg);
          p.out[STRIDED ? (size_t)it.b * qo.o_req + ((size_t)kvh * G + i / D) * qo.o_head + i % D
                        : qh * D + i % D] = 0x7fc0;
        }
      }
    }
  }
}

// One warp per (request, query head): merge the request's partials and write bf16 (the output
// row at the strides qo when STRIDED, else packed [B, Hq, D]).
template <int D, bool STRIDED>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeParams p, const QoStrides qo) {
  constexpr int VPL = D / 32;  // output elements per lane
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const bool live = wid < p.batch * p.num_qo_heads;
  const int b = live ? wid / p.num_qo_heads : 0;
  // Split count of request b: the chunks that overlap it (slot schedule above, at most
  // max_splits), or the caller's explicit count.  Warp-collective.
  auto split_count = [&]() {
    if (p.kv_indptr == nullptr) return p.num_splits;
    const int2 tp = slot_totals(p.kv_indptr, p.batch, b, lane);
    const int CS = decode_chunk_slots(tp.x, p.num_splits, p.min_chunk, p.part_pitch);
    const int nb = slots_of(__ldg(p.kv_indptr + b + 1) - __ldg(p.kv_indptr + b));
    return nb > 0 ? min((tp.y + nb - 1) / CS - tp.y / CS + 1, p.part_pitch) : 0;
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
  using VecT = typename std::conditional<VPL == 4, float4, typename std::conditional<VPL == 2, float2, float>::type>::type;
  const VecT* o = reinterpret_cast<const VecT*>(p.o_part + base * D) + lane;  // slot s at o[s * 32]
  auto fma_vec = [](float (&a)[VPL], float w, const VecT& v) {
    if constexpr (VPL == 4) {
      a[0] += w * v.x; a[1] += w * v.y; a[2] += w * v.z; a[3] += w * v.w;
    } else if constexpr (VPL == 2) {
      a[0] += w * v.x; a[1] += w * v.y;
    } else {
      a[0] += w * v;
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
  uint16_t* dst = (STRIDED ? p.out + (size_t)b * qo.o_req + (size_t)(wid - b * p.num_qo_heads) * qo.o_head
                           : p.out + (size_t)wid * D) +
                  lane * VPL;
  if constexpr (VPL == 4) {
    uint2 pk;
    pk.x = float2_to_bf16x2_rn(acc[0] * inv, acc[1] * inv);
    pk.y = float2_to_bf16x2_rn(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else if constexpr (VPL == 2) {
    *reinterpret_cast<uint32_t*>(dst) = float2_to_bf16x2_rn(acc[0] * inv, acc[1] * inv);
  } else {
    *dst = (uint16_t)(float2_to_bf16x2_rn(acc[0] * inv, 0.f) & 0xffffu);
  }
}

template <int D, int G, int MODE>
cudaError_t launch_split_t(const typename SplitArg<MODE>::type& arg, cudaStream_t stream) {
  const DecodeParams& p = params_of(arg);
  using C = DecCfg<D, G>;
  constexpr int smem = (MODE & kModeMask) ? C::SMEM_BYTES_MASKED : C::SMEM_BYTES;
  static std::atomic<bool> attr_done[kMaxDevices];
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(decode_split_kernel<D, G, MODE>), smem, attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.num_splits + C::NPAIR - 1) / C::NPAIR, p.num_kv_heads);  // NPAIR chunks per CTA
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // set-up overlaps the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_split_kernel<D, G, MODE>, arg);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool decode_supported(int head_dim, int group) {
  return (head_dim == 32 || head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

cudaError_t launch_decode_split(const DecodeParams& p, const DecodeMask* mask, const KvStrides* strides,
                                const QoStrides* qo, cudaStream_t stream) {
  const int G = p.num_qo_heads / p.num_kv_heads;
  // the kernels with a mask, a contiguous cache or strided query / output rows are separate
  // instantiations with a longer parameter block
  const int64_t row = (int64_t)p.num_qo_heads * p.head_dim;
  const DecodeParamsExt pe{p, mask != nullptr ? *mask : DecodeMask{nullptr, 0, 0},
                           strides != nullptr ? *strides : KvStrides{0, 0, 0, 0},
                           qo != nullptr ? *qo : QoStrides{row, p.head_dim, row, p.head_dim}};
  int mode = (mask != nullptr ? kModeMask : 0) | (strides != nullptr ? kModeContig : 0);
  if (mode == 0 && qo != nullptr) mode = kModeStrided;
#define ASTR_DEC_CASE(DD, GG)                                                     \
  if (p.head_dim == DD && G == GG) {                                              \
    switch (mode) {                                                               \
      case 0: return launch_split_t<DD, GG, 0>(p, stream);                        \
      case kModeStrided: return launch_split_t<DD, GG, kModeStrided>(pe, stream); \
      case kModeMask: return launch_split_t<DD, GG, kModeMask>(pe, stream);       \
      case kModeContig: return launch_split_t<DD, GG, kModeContig>(pe, stream);   \
      default: return launch_split_t<DD, GG, kModeMask | kModeContig>(pe, stream); \
    }                                                                             \
  }
  ASTR_DEC_CASE(128, 4) ASTR_DEC_CASE(128, 1) ASTR_DEC_CASE(128, 2) ASTR_DEC_CASE(128, 8) ASTR_DEC_CASE(128, 16)
  ASTR_DEC_CASE(64, 4) ASTR_DEC_CASE(64, 1) ASTR_DEC_CASE(64, 2) ASTR_DEC_CASE(64, 8) ASTR_DEC_CASE(64, 16)
  ASTR_DEC_CASE(32, 4) ASTR_DEC_CASE(32, 1) ASTR_DEC_CASE(32, 2) ASTR_DEC_CASE(32, 8) ASTR_DEC_CASE(32, 16)
#undef ASTR_DEC_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_combine(const DecodeParams& p, const QoStrides* qo, cudaStream_t stream) {
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
  const QoStrides q = qo != nullptr ? *qo : QoStrides{0, 0, 0, 0};
#define ASTR_COMB_CASE(DD)                                                                         \
  if (p.head_dim == DD)                                                                           \
    e = qo != nullptr ? cudaLaunchKernelEx(&cfg, decode_combine_kernel<DD, true>, p, q)             \
                      : cudaLaunchKernelEx(&cfg, decode_combine_kernel<DD, false>, p, q);
  ASTR_COMB_CASE(128) else ASTR_COMB_CASE(64) else ASTR_COMB_CASE(32) else return cudaErrorInvalidValue;
#undef ASTR_COMB_CASE
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace astr
