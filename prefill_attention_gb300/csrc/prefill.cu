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
//   * Persistent CTAs, one per SM.  A work item is (request, two consecutive query tiles,
//     KV head).  A 128-row MMA tile packs BQ = 128/G query positions x the G query heads
//     that share the KV head (row r = position r / G, head r % G), so each gathered K/V tile
//     feeds 2 x 128 rows.  Every CTA computes the same cost-sorted order of the items in its
//     prologue and takes its share in snake order -- or, when the call carries a work plan
//     made on the host for exactly its batch (checked against a checksum of qo_indptr and
//     seq_lens), reads its own item list from the plan instead.
//   * Warp roles (15 warps): 0-7 softmax and epilogue, four per query tile, thread = row =
//     TMEM lane; 8-9 issue the MMAs, one thread per query tile; 10-13 gather K/V, one warp
//     per ring stage; 14 loads the query tiles by TMA (a box of BQ positions x G heads x one
//     column block is exactly 128 rows of the swizzled operand layout).
//   * S = Q K^T and O += P V run as tcgen05.mma (bf16 in, fp32 accumulate); S is double
//     buffered and O stays in tensor memory.  A K/V ring stage is refilled once the P V that
//     read its V (and so the S that read its K) has completed.
//   * Query tiles go through a ring of three slots, so the next item's first tile loads
//     while the current item runs (its second once the current item's first tile is done).
//     A finished tile's slot then stages its output rows, which leave as 512-byte coalesced
//     stores; O in tensor memory is released as soon as it is read.
//   * Softmax: base-2 online softmax with a lazy reference max (O and l rescaled only when a
//     row's max grows by more than 7), exact because P, l and O share one reference.  The row
//     max is taken only on a row's first visible tile and when the tile's row sum shows that
//     some p may approach the fp16 limit; otherwise a tile costs one packed FMA, two
//     exponentials, one packed add and one fp16 pack per pair of scores.
//   * P V runs in fp16 (P written over S in tensor memory as fp16 pairs; the gather warps turn
//     each V tile into fp16 in shared memory once it lands): fp16 carries p to 2^-11 relative
//     against bf16's 2^-8, which keeps P's rounding well inside the output's (a bf16 P pushed
//     some outputs past a 1e-2 tolerance).  The K/V landing (kv_full) lets S start; the V
//     conversion completes on its own barrier (v_full) that only P V waits for.  V must lie
//     within the fp16 range (|v| <= 65504): a value beyond it makes the rows that read it
//     non-finite, which the epilogue reports in the status word.
//   * Variants of the same template: the causal rule can be switched off (unified-causal-
//     offset commit, offset -1) -- each row's key window then ends at seq_len; MASK adds an
//     explicit 2-D / 3-D mask (prefill-mask commit: causal and mask coexist), read by each
//     softmax thread as 64 bytes per key tile while the tile's scores are computed; CONTIG
//     reads K/V from a contiguous cache by strides (stride-addressing and layout commits)
//     instead of through req_to_token.  The masked and contiguous sets are compiled in
//     prefill_masked.cu and prefill_contig.cu.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace astr {
namespace {

template <int D, int G>
struct PrefillCfg {
  static constexpr int M = 128;                        // rows of one query tile = positions x heads
  static constexpr int BQ = M / G;                     // query positions per tile
  static constexpr int NQ = 2;                         // query tiles per work item (consecutive, same request)
  static constexpr int BN = 64;                        // keys per KV tile
  static constexpr int STAGES = 4;                     // K/V ring; one producer warp per stage
  static constexpr int Q_SLOTS = 3;                    // query-tile ring
  static constexpr int MMA_WARP = 4 * NQ;              // warps 0-3: softmax of tile 0, 4-7: tile 1
  static constexpr int KV_WARP0 = MMA_WARP + NQ;       // one MMA-issuing warp per query tile
  static constexpr int Q_WARP = KV_WARP0 + STAGES;     // query-tile loads
  static constexpr int THREADS = (Q_WARP + 1) * 32;
  static constexpr int CPR = D / 8;                    // 16-byte chunks per row
  // operand tiles are K-major rows in swizzled column blocks: 64 elements (128-byte swizzle)
  // for D >= 64, one block of 32 elements (64-byte swizzle) for D = 32
  static constexpr int SW_BYTES = D * 2 < 128 ? D * 2 : 128;   // bytes of a row in one column block
  static constexpr int CB_ELEMS = SW_BYTES / 2;                 // elements per column block
  static constexpr int NCB = D / CB_ELEMS;                      // column blocks per row
  static constexpr uint32_t ATOM = 8 * SW_BYTES;                // bytes of one 8-row swizzle atom
  static constexpr uint32_t SW_MODE = SW_BYTES == 128 ? 2u : 4u;  // descriptor swizzle field
  static constexpr int KPB = CB_ELEMS / 16;                     // MMA k-steps per column block
  static constexpr int Q_BYTES = M * D * 2;            // one query tile
  static constexpr int KV_BYTES = BN * D * 2;          // one K (or V) tile
  static constexpr int Q_OFF = 0;                      // Q_SLOTS query tiles
  static constexpr int K_OFF = Q_OFF + Q_SLOTS * Q_BYTES;  // STAGES tiles
  static constexpr int V_OFF = K_OFF + STAGES * KV_BYTES;
  static constexpr int BAR_OFF = V_OFF + STAGES * KV_BYTES;
  // barriers: kv_full, kv_empty [STAGES]; q_full, q_free, o_staged [Q_SLOTS]; s_full, p_full
  // [NQ][2]; o_done, o_free [NQ]; fin; v_full [STAGES].  Then the error flag and TMEM address.
  static constexpr int NBAR = 2 * STAGES + 3 * Q_SLOTS + 6 * NQ + 1 + STAGES;  // + v_full [STAGES]
  static constexpr int LIST_OFF = (BAR_OFF + NBAR * 8 + 8 + 15) & ~15;
  // this CTA's items in order, five words each: request | KV head << 16, the request's first
  // query row, query count and key count, the pair's first request-local query position
  static constexpr int MAX_CTA_ITEMS = 128;
  static constexpr int LIST_WORDS = 5;
  static constexpr int SMEM_BYTES = LIST_OFF + MAX_CTA_ITEMS * LIST_WORDS * 4;
  // prologue scratch in the query and K/V rings: copies of qo_indptr and seq_lens, per-request
  // pair offsets, bucket counts, keys, order, the request of each pair
  static constexpr int MAX_SORT_REQS = 1024;
  static constexpr int MAX_SORT_PAIRS = D >= 64 ? 8192 : 4096;  // (the rings are smaller for D = 32)
  static constexpr int SORT_BUCKETS = 1024;              // sort key range (estimated cost, clamped)
  static constexpr int RANK_PAIRS = 256;                 // up to this many pairs: rank count, not counting sort
  static constexpr uint32_t TMEM_TILE = 256;           // tile t: O at 256 t, S buffers at 256 t + D + {0, BN}
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int KV_IT = BN * CPR / 32;          // cp.async per producer lane per K (or V) tile
  static constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(M, BN, false, false);   // K-major A and B
  static constexpr uint32_t IDESC_PV = tc::idesc_f16_f32(M, D, false, true);     // fp16 P and V, V MN-major
  // P = 2^(sm_scale s - m + kPOffset) in fp16: the running reference m moves up when a row's
  // tile max exceeds it by more than kRescaleThreshold, so p <= 2^15 (< 65504) after a max pass;
  // without one, a tile row sum of at most kPSumLimit bounds every p the same way
  static constexpr float kPOffset = 8.f;               // log2 units
  static constexpr float kRescaleThreshold = 7.f;      // log2 units
  static constexpr float kPSumLimit = 32768.f;
  static_assert((Q_OFF | K_OFF | V_OFF | Q_BYTES | KV_BYTES) % 1024 == 0, "swizzle atoms must be 1024-byte aligned");
  static_assert(D + 2 * BN <= (int)TMEM_TILE, "tensor-memory budget per tile");
  static_assert(KV_IT * 32 == BN * CPR && (D == 32 || D % 64 == 0), "whole warp iterations, whole column blocks");
  // scratch offsets in int32 words from the query ring's start (16-byte aligned arrays)
  static constexpr int SCR_RS = MAX_SORT_REQS + 4;                 // seq_lens copy (qo_indptr copy at 0)
  static constexpr int SCR_PST = SCR_RS + MAX_SORT_REQS;           // pair offsets per request
  static constexpr int SCR_CNT = SCR_PST + MAX_SORT_REQS + 4;      // bucket counts / rank words
  static constexpr int SCR_KEY = SCR_CNT + SORT_BUCKETS;           // keys, order, pair -> request (uint16 each)
  static constexpr int SCR_PLAN = SCR_KEY + 3 * MAX_SORT_PAIRS / 2;  // plan header + this CTA's row, 2 words
  static constexpr int SCR_END = SCR_PLAN + kPlanHeader + kPlanRow + 2;
  static_assert(MAX_SORT_REQS % 4 == 0 && MAX_SORT_PAIRS % 8 == 0 && SCR_END * 4 <= Q_SLOTS * Q_BYTES + 2 * STAGES * KV_BYTES,
                "prologue scratch");
  static_assert(MAX_CTA_ITEMS == kPlanMaxItems, "a plan row fits the per-CTA list");
  static_assert(MAX_SORT_REQS <= 65536, "request index and KV head share a list word");
  static_assert(RANK_PAIRS <= SORT_BUCKETS && SORT_BUCKETS * MAX_SORT_PAIRS < (1 << 30), "rank words in the count array");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// Byte offset of 16-byte chunk c of row r in a swizzled K-major tile whose column blocks each
// hold `rows` rows: 128-byte swizzle (SWB = 128: 64-element blocks, chunk c & 7 of a 128-byte
// row at (c ^ r) & 7) or 64-byte swizzle (SWB = 64: one 32-element block, chunk c of a 64-byte
// row at c ^ ((r >> 1) & 3)), the layouts the TMA boxes and the MMA descriptors use.
template <int SWB>
__device__ __forceinline__ uint32_t swz(int r, int c, int rows) {
  if constexpr (SWB == 128) {
    return (uint32_t)((c >> 3) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
  } else {
    static_assert(SWB == 64, "64- or 128-byte swizzle");
    return (uint32_t)((r >> 3) * 512 + (r & 7) * 64 + (((c & 3) ^ ((r >> 1) & 3)) << 4));
  }
}

// Packed fp32 pairs (f32x2 arithmetic on sm_100-family SMs) and three-input max / min.
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// tcgen05.mma with the shared-memory descriptors passed as 32-bit halves.  The start address
// lives in bits 0-13 of the low half, so a descriptor for base + off is (lo + off / 16, hi)
// for the operand offsets used here (all smem addresses are below 256 KB).
__device__ __forceinline__ void mma_ss_h(uint32_t d, uint32_t alo, uint32_t ahi, uint32_t blo, uint32_t bhi,
                                         uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 a, b;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tmov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %4};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, p;\n\t}" ::"r"(d),
      "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts_h(uint32_t d, uint32_t a_tmem, uint32_t blo, uint32_t bhi, uint32_t idesc,
                                         uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 b;\n\t"
      "setp.ne.b32 p, %5, 0;\n\tmov.b64 b, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}
// The same MMAs and the tensor-core commit issued by one elected lane of a converged warp: every
// lane computes the (warp-uniform) descriptors, so they stay in the uniform datapath that the
// tensor-core instructions read, and only the issue itself is single-threaded.  (The leader of
// a fully converged warp is the same lane every time, so the commit tracks its MMAs.)
__device__ __forceinline__ void mma_ss_e(uint32_t d, uint32_t alo, uint32_t ahi, uint32_t blo, uint32_t bhi,
                                         uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 a, b;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tmov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %4};\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, p;\n\t}" ::"r"(d),
      "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts_e(uint32_t d, uint32_t a_tmem, uint32_t blo, uint32_t bhi, uint32_t idesc,
                                         uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 b;\n\t"
      "setp.ne.b32 p, %5, 0;\n\tmov.b64 b, {%2, %3};\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit_e(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// Keeps the values in registers at this point (they are computed before it, not between MMAs).
// 16 mask bytes, read through L1 (the rows of one query position are shared by its G heads).
__device__ __forceinline__ uint4 ldg_nc_v4(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// 64 mask bytes -> 64 bits (bit k = byte k nonzero).  Per 32-bit word: __vcmpne4 turns each
// nonzero byte into 0xff; keeping bit 0 of every byte and multiplying by 0x01020408 moves
// byte k's bit to bit 24 + k (the four partial products land on distinct bits, no carries).
__device__ __forceinline__ uint64_t mask_bits64(const uint4 (&w)[4]) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t v[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t nib = (((__vcmpne4(v[k], 0u) & 0x01010101u) * 0x01020408u) >> 24) & 0xfu;
      const int sh = 16 * c + 4 * k;  // bit position of this word's first byte
      if (sh < 32) lo |= nib << sh;
      else hi |= nib << (sh - 32);
    }
  }
  return ((uint64_t)hi << 32) | lo;
}

template <int N>
__device__ __forceinline__ void keep_regs(uint32_t (&v)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(v[i]));
}

// One work item: KV head kvh, request b, query-tile pair pr (tiles 2 pr and 2 pr + 1 of the
// request, the second possibly absent).  Items are numbered pair-major, KV-head-minor.
// cb is the causal offset seq_len - q_len (with the causal offset off: seq_len - 1, so that
// every row's key window, clipped at kvn = seq_len, is all of the request's keys).
struct PrefillItem {
  int b, kvh, q0, q_len, cb, kvn, first0, nq, n_tiles;
};

// Fills the item's fields from its request's first query row q0, query count q_len and key
// count kvn, and the pair's first request-local query position first0.
template <int BQ2, int BQ, int BN>
__device__ __forceinline__ void fill_item_vals(const PrefillParams& p, int b, int kvh, int q0, int q_len, int kvn,
                                               int first0, PrefillItem& it) {
  it.b = b;
  it.kvh = kvh;
  it.q0 = q0;
  it.q_len = q_len;
  it.kvn = kvn;
  it.cb = p.causal ? kvn - q_len : kvn - 1;
  it.first0 = first0;
  it.nq = min(BQ2 / BQ, (q_len - first0 + BQ - 1) / BQ);
  const int last = min(q_len, first0 + it.nq * BQ) - 1;
  it.n_tiles = (min(it.cb + last + 1, kvn) + BN - 1) / BN;
}

// The same, reading the request's row range and key count from the call's arrays.
template <int BQ2, int BQ, int BN>
__device__ __forceinline__ void fill_item(const PrefillParams& p, int b, int pr, int kvh, PrefillItem& it) {
  const int q0 = __ldg(p.qo_indptr + b);
  fill_item_vals<BQ2, BQ, BN>(p, b, kvh, q0, __ldg(p.qo_indptr + b + 1) - q0, __ldg(p.seq_lens + b), pr * BQ2, it);
}

// Decodes item w of the natural order by a warp-parallel prefix scan of the per-request pair
// counts (all 32 lanes call it and get the same answer).  False once w is past the last item.
template <int BQ2, int BQ, int BN>
__device__ __forceinline__ bool scan_item(const PrefillParams& p, int w, int lane, PrefillItem& it) {
  const int pair_idx = w / p.num_kv_heads;
  int acc = 0;
  for (int base = 0; base < p.batch; base += 32) {
    const int bb = base + lane;
    int np = 0;
    if (bb < p.batch) np = (__ldg(p.qo_indptr + bb + 1) - __ldg(p.qo_indptr + bb) + BQ2 - 1) / BQ2;
    int inc = np;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFullMask, inc, o);
      if (lane >= o) inc += y;
    }
    const int total = __shfl_sync(kFullMask, inc, 31);
    if (pair_idx < acc + total) {
      const unsigned ball = __ballot_sync(kFullMask, pair_idx < acc + inc);
      const int first = __ffs(ball) - 1;
      const int excl = __shfl_sync(kFullMask, inc - np, first);
      fill_item<BQ2, BQ, BN>(p, base + first, pair_idx - acc - excl, w % p.num_kv_heads, it);
      return true;
    }
    acc += total;
  }
  return false;
}

template <int D, int G, bool MASK, bool CONTIG>
__global__ void __launch_bounds__(PrefillCfg<D, G>::THREADS, 1) prefill_kernel(const PrefillParams p,
                                                                                const __grid_constant__ CUtensorMap q_map,
                                                                                const __grid_constant__ CUtensorMap o_map) {
  using C = PrefillCfg<D, G>;
  constexpr int BQ2 = C::NQ * C::BQ;
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((sbase & 1023u) != 0) {  // swizzle atoms need a 1024-byte aligned window: report, do nothing
    if (tid == 0 && p.status != nullptr) atomicOr(p.status, kStatusSmem);
    return;
  }

  // The request tables go to shared memory first (scratch in the query and K/V rings, unused
  // until the work order is known): their one global round trip overlaps the set-up below.
  // A work plan's header and this CTA's row load in the same round trip (the host passes a plan
  // only when it holds a row for every CTA of the launch).
  int* rq = reinterpret_cast<int*>(smem + C::Q_OFF);  // qo_indptr[0 .. B]
  int* rs = rq + C::SCR_RS;                          // seq_lens[0 .. B - 1]
  int* pl = rq + C::SCR_PLAN;                        // plan header, row, then two words of results
  const bool tables = p.batch <= C::MAX_SORT_REQS;
  if (tables && warp > 0) {  // (warp 0 sets up barriers and tensor memory meanwhile)
    for (int i = tid - 32; i <= p.batch; i += C::THREADS - 32) rq[i] = __ldg(p.qo_indptr + i);
    for (int i = tid - 32; i < p.batch; i += C::THREADS - 32) rs[i] = __ldg(p.seq_lens + i);
    if (p.plan != nullptr)
      for (int i = tid - 32; i < kPlanHeader + kPlanRow; i += C::THREADS - 32)
        pl[i] = __ldg(p.plan + (i < kPlanHeader ? i : kPlanHeader + (int64_t)blockIdx.x * kPlanRow + (i - kPlanHeader)));
  }

  const uint32_t bars = sbase + C::BAR_OFF;
  auto kv_full = [&](int s) { return bars + 8u * s; };
  auto kv_empty = [&](int s) { return bars + 8u * (C::STAGES + s); };
  // query tile number u (counted over the CTA's items, in order) lives in slot u % Q_SLOTS
  auto q_full = [&](int u) { return bars + 8u * (2 * C::STAGES + u % C::Q_SLOTS); };
  auto q_free = [&](int u) { return bars + 8u * (2 * C::STAGES + C::Q_SLOTS + u % C::Q_SLOTS); };
  // output rows of tile u staged in its slot (by the tile's softmax warps)
  auto o_staged = [&](int u) { return bars + 8u * (2 * C::STAGES + 2 * C::Q_SLOTS + u % C::Q_SLOTS); };
  auto q_par = [&](int u) { return (uint32_t)((u / C::Q_SLOTS) & 1); };
  auto q_slot = [&](int u) { return sbase + C::Q_OFF + (u % C::Q_SLOTS) * C::Q_BYTES; };
  const uint32_t tb = bars + 8u * (2 * C::STAGES + 3 * C::Q_SLOTS);  // per-tile barriers
  // S / P of the g-th KV tile of query tile t live in buffer g & 1 (g counts over all items);
  // each buffer has its own barriers, so no waiter is ever more than one phase behind.
  auto s_full = [&](int t, int buf) { return tb + 8u * (2 * t + buf); };
  auto p_full = [&](int t, int buf) { return tb + 8u * (2 * C::NQ + 2 * t + buf); };
  auto o_done = [&](int t) { return tb + 8u * (4 * C::NQ + t); };
  auto o_free = [&](int t) { return tb + 8u * (5 * C::NQ + t); };
  const uint32_t fin = tb + 8u * (6 * C::NQ);
  // V of stage s turned into fp16 (the K/V landing itself is kv_full)
  auto v_full = [&](int s) { return fin + 8u + 8u * s; };
  volatile int* err = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 8 * C::NBAR);
  const uint32_t slot = sbase + C::BAR_OFF + 8 * C::NBAR + 4;
  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      tc::mbar_init(kv_full(s), 32);
      tc::mbar_init(kv_empty(s), C::NQ);  // one commit per MMA thread
    }
    for (int u = 0; u < C::Q_SLOTS; ++u) {
      tc::mbar_init(q_full(u), 1);  // arrive + TMA transaction bytes
      tc::mbar_init(q_free(u), C::NQ);  // every MMA thread, once it has seen the tile
      tc::mbar_init(o_staged(u), 4);    // lane 0 of the tile's four softmax warps
    }
    for (int t = 0; t < C::NQ; ++t) {
      for (int buf = 0; buf < 2; ++buf) {
        tc::mbar_init(s_full(t, buf), 1);
        tc::mbar_init(p_full(t, buf), 128);
      }
      tc::mbar_init(o_done(t), 1);
      tc::mbar_init(o_free(t), 128);
    }
    tc::mbar_init(fin, C::NQ);
    for (int s = 0; s < C::STAGES; ++s) tc::mbar_init(v_full(s), 32);
    *err = 0;
    pl[kPlanHeader + kPlanRow] = 0;  // checksum of the request tables (plan check)
    tc::fence_mbarrier_init();
  }
  if (warp == 0) tc::tmem_alloc<C::TMEM_COLS>(slot);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::BAR_OFF + 8 * C::NBAR + 4);

  // ---- work order, computed identically by every CTA (no cross-CTA communication): items
  // sorted by estimated time (descending; ties by index) and dealt out in snake order (CTA c
  // takes sorted positions c, 2G-1-c, 2G+c, ... for G CTAs).  The estimate, in about 10 ns
  // steps, weighs the KV tiles an item streams (the S -> softmax -> P V chain of each query
  // tile sets the pace per KV tile), its (query tile, KV tile) MMA units and a fixed per-item
  // cost (pipeline fill and drain, epilogue): 53 n_tiles + 13 units + 260, coefficients fitted
  // to measured per-CTA busy times (sorted in steps of 16).  The KV heads of one query-tile pair
  // cost the same and have consecutive indices, so the pairs are sorted and then expanded.
  // Each CTA keeps only its own list; problems too large for it use the natural order.  Every
  // step is a short dependent chain on shared memory, so the steps are kept few: a pair -> request
  // map instead of searches, and for up to RANK_PAIRS pairs a rank count (each thread counts the
  // pairs that sort before its own, one compare per pair) instead of the counting sort.
  int* list = reinterpret_cast<int*>(smem + C::LIST_OFF);
  int* pst = rq + C::SCR_PST;
  int* cnt = rq + C::SCR_CNT;  // bucket counts; (key, index) words of the rank count
  uint16_t* key = reinterpret_cast<uint16_t*>(rq + C::SCR_KEY);
  uint16_t* order = key + C::MAX_SORT_PAIRS;
  uint16_t* pmap = order + C::MAX_SORT_PAIRS;  // request of each pair
  const int H = p.num_kv_heads;
  int per_cta = 0;
  bool sorted = tables && H < 32768;
  // A plan is used when its header and the checksum of the request tables match the call (every
  // CTA sees the same tables and header, so all CTAs take the same decision).
  bool planned = false;
  if (sorted && p.plan != nullptr) {
    uint32_t h = 0;
    for (int i = tid; i <= p.batch; i += C::THREADS) h += plan_mix((uint32_t)i, (uint32_t)rq[i]);
    for (int i = tid; i < p.batch; i += C::THREADS) h += plan_mix(kPlanSeqTag + (uint32_t)i, (uint32_t)rs[i]);
    h = __reduce_add_sync(kFullMask, h);
    if (lane == 0) atomicAdd(reinterpret_cast<unsigned*>(pl + kPlanHeader + kPlanRow), h);
    __syncthreads();
    planned = pl[0] == kPlanMagic && pl[1] == kPlanVersion && pl[2] == p.batch && pl[3] == H && pl[4] == BQ2 &&
              pl[5] == (int)gridDim.x && pl[6] == pl[kPlanHeader + kPlanRow] && pl[7] == p.causal;
  }
  if (blockIdx.x == 0 && tid == 0 && p.status != nullptr && (p.plan_rejected || (p.plan != nullptr && !planned)))
    atomicOr(p.status, kStatusPlan);
  if (planned) {
    // this CTA's items, in plan order; an entry that names no item of the call is dropped and
    // reported (the plan's checksum matched, so only a damaged plan buffer has one)
    if (warp == 0) {
      const int n = min(max(pl[kPlanHeader], 0), C::MAX_CTA_ITEMS);
      int kept = 0;
      bool bad = pl[kPlanHeader] != n;
      for (int base = 0; base < n; base += 32) {
        const int k = base + lane;
        int b = -1, kvh = 0, pair = 0;
        bool valid = false;
        if (k < n) {
          b = pl[kPlanHeader + 1 + 2 * k];
          const int pk = pl[kPlanHeader + 2 + 2 * k];
          kvh = pk & 0xffff;
          pair = (int)((uint32_t)pk >> 16);
          valid = b >= 0 && b < p.batch && kvh < H && pair < (rq[b + 1] - rq[b] + BQ2 - 1) / BQ2;
          bad |= !valid;
        }
        const unsigned vm = __ballot_sync(kFullMask, valid);
        if (valid) {
          int* e = list + C::LIST_WORDS * (kept + __popc(vm & ((1u << lane) - 1u)));
          e[0] = b | (kvh << 16);
          e[1] = rq[b];
          e[2] = rq[b + 1] - rq[b];
          e[3] = rs[b];
          e[4] = pair * BQ2;
        }
        kept += __popc(vm);
      }
      if (lane == 0) pl[kPlanHeader + kPlanRow + 1] = kept;
      if (__any_sync(kFullMask, bad) && lane == 0 && p.status != nullptr) atomicOr(p.status, kStatusBadInput);
    }
    __syncthreads();
    per_cta = pl[kPlanHeader + kPlanRow + 1];
  } else if (sorted) {
    if (warp == 0) {  // pst[b] = first pair index of request b, pst[B] = number of pairs
      int acc = 0;
      for (int base = 0; base < p.batch; base += 32) {
        const int bb = base + lane;
        int np = 0;
        if (bb < p.batch) np = (rq[bb + 1] - rq[bb] + BQ2 - 1) / BQ2;
        int inc = np;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(kFullMask, inc, o);
          if (lane >= o) inc += y;
        }
        const int first = acc + inc - np;
        if (bb < p.batch) {
          pst[bb] = first;
          for (int w = first; w < min(first + np, C::MAX_SORT_PAIRS); ++w) pmap[w] = (uint16_t)bb;
        }
        acc += __shfl_sync(kFullMask, inc, 31);
      }
      if (lane == 0) pst[p.batch] = acc;
    }
    __syncthreads();
    const int n_pairs = pst[p.batch];
    sorted = n_pairs <= C::MAX_SORT_PAIRS;
    per_cta = sorted ? (int)(((unsigned)(n_pairs * H) + gridDim.x - 1) / gridDim.x) : 0;
    sorted = sorted && per_cta <= C::MAX_CTA_ITEMS;
  }
  if (sorted && !planned) {
    const int n_pairs = pst[p.batch];
    const bool rank = n_pairs <= C::RANK_PAIRS;
    for (int w = tid; w < n_pairs; w += C::THREADS) {
      const int b = pmap[w];
      PrefillItem it;
      fill_item_vals<BQ2, C::BQ, C::BN>(p, b, 0, rq[b], rq[b + 1] - rq[b], rs[b], (w - pst[b]) * BQ2, it);
      int units = 0;
      for (int t = 0; t < it.nq; ++t)
        units += (min(it.cb + min(it.q_len, it.first0 + (t + 1) * C::BQ), it.kvn) + C::BN - 1) / C::BN;
      const int c = (53 * it.n_tiles + 13 * units + 260) >> 4;  // cost estimate in ~0.16 us steps
      const int k = C::SORT_BUCKETS - 1 - min(max(c, 0), C::SORT_BUCKETS - 1);  // ascending key = descending cost
      if (rank)
        cnt[w] = k * C::MAX_SORT_PAIRS + w;  // (key, index): distinct, ordered like the stable sort
      else
        key[w] = (uint16_t)k;
    }
    if (!rank)
      for (int i = tid; i < C::SORT_BUCKETS; i += C::THREADS) cnt[i] = 0;
    __syncthreads();
    if (rank) {
      for (int w = tid; w < n_pairs; w += C::THREADS) {
        const int mine = cnt[w];
        int r = 0;
        int j = 0;
        for (; j + 4 <= n_pairs; j += 4) {
          const int4 v = *reinterpret_cast<const int4*>(cnt + j);
          r += (v.x < mine) + (v.y < mine) + (v.z < mine) + (v.w < mine);
        }
        for (; j < n_pairs; ++j) r += cnt[j] < mine;
        order[r] = (uint16_t)w;
      }
    } else if (warp == 0) {  // stable counting sort of the pairs, one warp, chunks of 32 in index order
      for (int base = 0; base < n_pairs; base += 32) {
        const int w = base + lane;
        const int k = (w < n_pairs) ? key[w] : -1;
        const unsigned peers = __match_any_sync(kFullMask, k);
        if (w < n_pairs && (peers & ((1u << lane) - 1u)) == 0u) cnt[k] += __popc(peers);
        __syncwarp();
      }
      constexpr int BPL = C::SORT_BUCKETS / 32;  // exclusive scan of the bucket counts, BPL per lane
      int v[BPL];
#pragma unroll
      for (int i = 0; i < BPL; ++i) v[i] = cnt[lane * BPL + i];
      int tot = 0;
#pragma unroll
      for (int i = 0; i < BPL; ++i) tot += v[i];
      int inc = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFullMask, inc, o);
        if (lane >= o) inc += y;
      }
      int run = inc - tot;
#pragma unroll
      for (int i = 0; i < BPL; ++i) {
        cnt[lane * BPL + i] = run;
        run += v[i];
      }
      __syncwarp();
      for (int base = 0; base < n_pairs; base += 32) {
        const int w = base + lane;
        const int k = (w < n_pairs) ? key[w] : -1;
        const unsigned peers = __match_any_sync(kFullMask, k);
        if (w < n_pairs) order[cnt[k] + __popc(peers & ((1u << lane) - 1u))] = (uint16_t)w;
        __syncwarp();
        if (w < n_pairs && (peers & ((1u << lane) - 1u)) == 0u) cnt[k] += __popc(peers);
        __syncwarp();
      }
    }
    __syncthreads();
    for (int k = tid; k < per_cta; k += C::THREADS) {  // this CTA's sorted positions, fields resolved
      const int c = blockIdx.x, nc = gridDim.x;
      const int pos = k * nc + ((k & 1) ? nc - 1 - c : c);
      int* e = list + C::LIST_WORDS * k;
      if (pos < n_pairs * H) {
        const int pair = order[pos / H];
        const int b = pmap[pair];
        e[0] = b | ((pos % H) << 16);
        e[1] = rq[b];
        e[2] = rq[b + 1] - rq[b];
        e[3] = rs[b];
        e[4] = (pair - pst[b]) * BQ2;
      } else {
        e[0] = -1;
      }
    }
    __syncthreads();
  }
  // the k-th item of this CTA (called by all 32 lanes of a warp); false past the last one
  auto get_item = [&](int k, PrefillItem& it) -> bool {
    if (sorted) {
      if (k >= per_cta) return false;
      const int* e = list + C::LIST_WORDS * k;
      if (e[0] < 0) return false;
      fill_item_vals<BQ2, C::BQ, C::BN>(p, e[0] & 0xffff, e[0] >> 16, e[1], e[2], e[3], e[4], it);
      return true;
    }
    const int c = blockIdx.x, nc = gridDim.x;
    return scan_item<BQ2, C::BQ, C::BN>(p, k * nc + ((k & 1) ? nc - 1 - c : c), lane, it);
  };

  // Bounded wait, agreed by the whole warp (so warp-collective tcgen05 ops after it stay
  // converged); a timeout, or an error raised elsewhere, makes every later wait fail.
  auto wait_or_fail = [&](uint32_t bar, uint32_t parity) -> bool {
    bool ok = (*err == 0) && tc::mbar_wait(bar, parity, p.wait_limit);
    ok = __all_sync(kFullMask, ok);
    if (!ok) *err = 1;
    return ok;
  };

  if (warp == C::Q_WARP) {
    // ======================= query tiles in, output tiles out, by TMA, in tile order.  Tile u
    //                         loads into slot u % Q_SLOTS once the tile that used the slot
    //                         before (u - Q_SLOTS) has been written out from it; that tile's
    //                         softmax warps staged its output rows there.  Query rows past the
    //                         request's end hold other requests' queries (never written out)
    //                         or, past the last row, zeros.
    bool ok = true;
    int u = 0;  // query tiles so far
    // query tiles are read and output tiles written once: first out of L2, ahead of the K/V
    // rows that the other query tiles of the same request read again
    const uint64_t once = tc::l2_evict_first_policy();
    // where each slot's tile goes (lane k holds slot k): request, first position (request-local
    // for a padded output, flat for a packed one), first head, rows
    int pend_b = 0, pend_pos = 0, pend_head = 0, pend_rows = 0;
    const bool q_padded = p.q_batch > 0, o_padded = p.o_batch > 0;
    // write tile v's staged rows out: one TMA store per column block when all BQ positions
    // are the request's, else the valid rows with coalesced stores (never past the request)
    auto write_out = [&](int v) {
      if (!(ok = wait_or_fail(o_staged(v), q_par(v)))) return;
      const int k = v % C::Q_SLOTS;
      const int ob = __shfl_sync(kFullMask, pend_b, k), pos = __shfl_sync(kFullMask, pend_pos, k);
      const int head = __shfl_sync(kFullMask, pend_head, k), rows = __shfl_sync(kFullMask, pend_rows, k);
      const uint32_t src = q_slot(v);
      if (rows == C::M) {
        if (lane == 0) {
          for (int cb = 0; cb < C::NCB; ++cb) {
            if (o_padded)
              tc::tma_store_4d_hint(&o_map, src + cb * (C::M * C::SW_BYTES), cb * C::CB_ELEMS, head, pos, ob, once);
            else
              tc::tma_store_3d_hint(&o_map, src + cb * (C::M * C::SW_BYTES), cb * C::CB_ELEMS, head, pos, once);
          }
          tc::bulk_commit();
          tc::bulk_wait_read_all();  // the slot may be refilled once the stores have read it
        }
      } else {
        // row r of the tile is position pos + r / G, head head + r % G
        const int64_t orow0 = (o_padded ? (int64_t)ob * p.o_batch : 0) + (int64_t)pos * p.o_token;
        uint16_t* obase = p.out + orow0 + (int64_t)head * p.o_head;
        for (int i = 0; i < C::M * C::CPR / 32; ++i) {
          const int flat = i * 32 + lane, r = flat / C::CPR, c = flat % C::CPR;
          if (r < rows) {
            const uint4 x = lds128(src + swz<C::SW_BYTES>(r, c, C::M));
            *reinterpret_cast<uint4*>(obase + (int64_t)(r / G) * p.o_token + (int64_t)(r % G) * p.o_head + c * 8) = x;
          }
        }
        tc::fence_proxy_async_smem();  // the next TMA write of this slot follows these reads
      }
      __syncwarp();
    };
    PrefillItem it;
    for (int n_item = 0; ok; ++n_item) {
      if (!get_item(n_item, it)) break;
      for (int t = 0; ok && t < it.nq; ++t, ++u) {
        if (u >= C::Q_SLOTS) {
          write_out(u - C::Q_SLOTS);
          if (!ok || !(ok = wait_or_fail(q_free(u), q_par(u) ^ 1u))) break;
        }
        const int qf = it.first0 + t * C::BQ;
        if (lane == u % C::Q_SLOTS) {
          pend_b = it.b;
          pend_pos = o_padded ? qf : it.q0 + qf;
          pend_head = it.kvh * G;
          pend_rows = (min(it.q_len, qf + C::BQ) - qf) * G;
        }
        if (lane == 0) {
          tc::mbar_arrive_expect_tx(q_full(u), (uint32_t)C::Q_BYTES);
          for (int cb = 0; cb < C::NCB; ++cb) {
            const uint32_t dst = q_slot(u) + cb * (C::M * C::SW_BYTES);
            if (q_padded)
              tc::tma_load_4d_hint(dst, &q_map, cb * C::CB_ELEMS, it.kvh * G, qf, it.b, q_full(u), once);
            else
              tc::tma_load_3d_hint(dst, &q_map, cb * C::CB_ELEMS, it.kvh * G, it.q0 + qf, q_full(u), once);
          }
        }
        __syncwarp();
      }
    }
    for (int v = max(0, u - C::Q_SLOTS); ok && v < u; ++v) write_out(v);  // the last tiles
    if (lane == 0) tc::bulk_wait_all();
    if (!ok) {
      // a wait gave up: let the query loads still in flight (the last tiles issued, one phase
      // per slot) land before the CTA's shared memory goes away
      for (int v = max(0, u - C::Q_SLOTS); v < u; ++v) tc::mbar_wait(q_full(v), q_par(v), tc::kWaitLimit);
    }
    __syncwarp();
  } else if (warp >= C::KV_WARP0) {
    // ======================= K/V gathers: warp KV_WARP0 + s fills stage s with every KV tile
    //                         g = s mod STAGES (g counts over all items)
    const int st = warp - C::KV_WARP0;
    const size_t head_stride = (size_t)p.num_kv_heads * D;
    const unsigned nslots = (unsigned)p.num_slots;
    const uint32_t kdst = sbase + C::K_OFF + st * C::KV_BYTES, vdst = sbase + C::V_OFF + st * C::KV_BYTES;
    int g_base = 0;  // global index of the current item's KV tile 0
    bool ok = true, bad_input = false;
    PrefillItem it;
    for (int n_item = 0; ok; ++n_item) {
      if (!get_item(n_item, it)) break;
      const int kvh = it.kvh;
      const int32_t* r2t = p.req_to_token + (size_t)it.b * p.r2t_stride;
      const int kv_end = min(it.cb + min(it.q_len, it.first0 + BQ2), it.kvn);
      const int j_first = (st - g_base % C::STAGES + C::STAGES) % C::STAGES;
      // slot id of key 32 half + lane of item tile j, or -1 past the keys the item reads;
      // `real`: a key of the request whose id is checked against the pool when it is used (a
      // position past the table row is not read and is reported at once)
      auto ids_of = [&](int j, int half, bool& real) {
        const int key = j * C::BN + half * 32 + lane;
        real = j < it.n_tiles && key < kv_end;
        if constexpr (CONTIG) {
          const int pos = real ? key : -1;  // contiguous cache: the position itself
          real = false;
          return pos;
        } else {
          if (real && key >= p.r2t_stride) {
            bad_input = true;
            real = false;
          }
          return real ? ldg_nc_i32(r2t + key) : -1;
        }
      };
      // one K/V tile: row `key` comes from the slot id held by lane key % 32 of id0 (keys
      // 0-31) or id1 (keys 32-63); padding and out-of-range ids read as zeros.  K and V share
      // each lane's address arithmetic (one loop over both costs the softmax warps on the
      // same schedulers noticeably fewer issue slots than two)
      auto gather = [&](int id0, int id1) {
#pragma unroll 8
        for (int i = 0; i < C::KV_IT; ++i) {
          const int flat = i * 32 + lane;
          const int key = flat / C::CPR, c = flat % C::CPR;  // key < 32 exactly for the first half of `i`
          const int id = __shfl_sync(kFullMask, (i < C::KV_IT / 2) ? id0 : id1, key & 31);
          bool valid;
          size_t off;
          if constexpr (CONTIG) {  // id = key position in request b's contiguous rows
            valid = (unsigned)id < (unsigned)p.kv.max_len;
            off = valid ? (size_t)it.b * p.kv.batch + (size_t)id * p.kv.token + (size_t)kvh * p.kv.head + c * 8 : 0;
          } else {
            valid = (unsigned)id < nslots;
            off = valid ? (size_t)id * head_stride + (size_t)kvh * D + c * 8 : 0;
          }
          const uint32_t o = swz<C::SW_BYTES>(key, c, C::BN);
          cp_async16(kdst + o, p.k_pool + off, valid);
          cp_async16(vdst + o, p.v_pool + off, valid);
        }
        cp_async_commit();
      };
      bool real0, real1;
      int id0 = ids_of(j_first, 0, real0), id1 = ids_of(j_first, 1, real1);
      for (int j = j_first; j < it.n_tiles; j += C::STAGES) {
        const int g = g_base + j;
        const uint32_t par = (uint32_t)(((g / C::STAGES) - 1) & 1);  // phase of tile g - STAGES
        if (g >= C::STAGES && !(ok = wait_or_fail(kv_empty(st), par))) break;
        if constexpr (!CONTIG) bad_input |= (real0 && (unsigned)id0 >= nslots) || (real1 && (unsigned)id1 >= nslots);
        gather(id0, id1);
        id0 = ids_of(j + C::STAGES, 0, real0);  // next tile of this stage: its slot ids load meanwhile
        id1 = ids_of(j + C::STAGES, 1, real1);
        cp_async_wait<0>();
        tc::fence_proxy_async_smem();  // the tensor core reads the tiles through the async proxy
        tc::mbar_arrive(kv_full(st));  // K landed: S may start
        // P V runs in fp16: each lane turns the V chunks it copied into fp16 in place, same layout
#pragma unroll 4
        for (int i = 0; i < C::KV_IT; ++i) {
          const int flat = i * 32 + lane;
          const uint32_t a = vdst + swz<C::SW_BYTES>(flat / C::CPR, flat % C::CPR, C::BN);
          uint4 x = lds128(a);
          float2 f;
          f = bf16x2_to_float2(x.x); x.x = float2_to_f16x2_rn(f.x, f.y);
          f = bf16x2_to_float2(x.y); x.y = float2_to_f16x2_rn(f.x, f.y);
          f = bf16x2_to_float2(x.z); x.z = float2_to_f16x2_rn(f.x, f.y);
          f = bf16x2_to_float2(x.w); x.w = float2_to_f16x2_rn(f.x, f.y);
          sts128(a, x);
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(v_full(st));
      }
      g_base += it.n_tiles;
    }
    cp_async_wait<0>();
    if (p.status != nullptr && __any_sync(kFullMask, bad_input) && lane == 0) atomicOr(p.status, kStatusBadInput);

  } else if (warp >= C::MMA_WARP) {
    // ======================= MMA issue: warp MMA_WARP + t for query tile t; the whole warp runs
    // the loop and its waits, one elected lane issues each MMA and commit.
    // tcgen05.mma issue runs nearly in step with execution, so whatever the issuing warp does
    // between MMAs (waits, fences, commits) idles the tensor core unless another warp has MMAs
    // queued: the two query tiles therefore have their own issuing warps, and the barriers each
    // group needs are tested (without blocking) in the middle of the group before it.  Per KV
    // tile j: S_t(j+1) = Q_t K_{j+1}^T into the other S buffer, then O_t += P_t(j) V_j once the
    // softmax warps of tile t have written P_t(j).  Both warps release every KV tile (after it
    // has landed), used or not, so the shared empty barriers count two arrivals per phase.
    const int t = warp - C::MMA_WARP;
    // descriptor halves of query slot 0, K stage 0 (K-major) and V stage 0 (MN-major)
    const uint64_t qd0 = tc::smem_desc_swz(sbase + C::Q_OFF, 16, C::ATOM, C::SW_MODE);
    const uint64_t kd0 = tc::smem_desc_swz(sbase + C::K_OFF, 16, C::ATOM, C::SW_MODE);
    const uint64_t vd0 = tc::smem_desc_swz(sbase + C::V_OFF, C::BN * C::SW_BYTES, C::ATOM, C::SW_MODE);
    const uint32_t q_hi = (uint32_t)(qd0 >> 32), k_hi = (uint32_t)(kd0 >> 32), v_hi = (uint32_t)(vd0 >> 32);
    const uint32_t k_lo = (uint32_t)kd0, v_lo = (uint32_t)vd0;
    const uint32_t od = tmem + t * C::TMEM_TILE;  // O of tile t; S / P buffers at od + D + {0, BN}
    int g_base = 0;   // global index of the item's KV tile 0
    int gs = 0;       // KV tiles of tile t so far (S buffer / phase counter)
    int n_used = 0;   // items so far that had tile t (o_done / o_free phases)
    int u0 = 0;       // query tiles of the items before this one
    int uw = 0;       // query tiles waited for so far (every warp waits for all, in order)
    bool ok = true;   // warp-uniform
    PrefillItem it;
    for (int n_item = 0; ok; ++n_item) {
      if (!get_item(n_item, it)) break;
      const int nk =
          (t < it.nq) ? (min(it.cb + min(it.q_len, it.first0 + (t + 1) * C::BQ), it.kvn) + C::BN - 1) / C::BN : 0;
      const int n = it.n_tiles;
      const uint32_t q_lo = (uint32_t)qd0 + (uint32_t)((((u0 + t) % C::Q_SLOTS) * C::Q_BYTES) >> 4);
      // blocking only if not pre-tested ready; gives up (and stops this warp's issue) on a
      // timeout or once another warp has given up; the whole warp agrees
      auto wait_one = [&](uint32_t bar, uint32_t parity, bool ready) {
        if (ok) {
          const bool good = *err == 0 && (ready || tc::mbar_wait(bar, parity, p.wait_limit));
          ok = __all_sync(kFullMask, good);
          if (!ok) *err = 1;
        }
        tc::fence_after_sync();
      };
      auto stage = [&](int j) { return (g_base + j) % C::STAGES; };
      auto kv_par = [&](int j) { return (uint32_t)(((g_base + j) / C::STAGES) & 1); };
      auto sbuf = [&](int j) { return (gs + j) & 1; };
      auto s_par = [&](int j) { return (uint32_t)(((gs + j) >> 1) & 1); };
      // issue S_t(j); while it runs, test barrier `nb` (parity `np`); returns that test (agreed
      // by the warp).
      auto issue_s = [&](int j, uint32_t nb, uint32_t np) -> bool {
        if (!ok) return false;  // a wait gave up: issue nothing more
        const uint32_t sd = od + D + sbuf(j) * C::BN;
        const uint32_t klo = k_lo + (uint32_t)((stage(j) * C::KV_BYTES) >> 4);
        bool r = false;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          mma_ss_e(sd, q_lo + (uint32_t)(((kk / C::KPB) * (C::M * C::SW_BYTES) + (kk % C::KPB) * 32) >> 4), q_hi,
                   klo + (uint32_t)(((kk / C::KPB) * (C::BN * C::SW_BYTES) + (kk % C::KPB) * 32) >> 4), k_hi,
                   C::IDESC_S, kk > 0 ? 1u : 0u);
          if (kk == D / 32) r = nb != 0u && tc::mbar_test(nb, np);
        }
        mma_commit_e(s_full(t, sbuf(j)));
        return __all_sync(kFullMask, r);
      };
      auto issue_pv = [&](int j, uint32_t nb, uint32_t np) -> bool {
        if (!ok) return false;  // a wait gave up: issue nothing more
        const uint32_t pa = od + D + sbuf(j) * C::BN;  // P (fp16 pairs) in columns [0, 32)
        const uint32_t vlo = v_lo + (uint32_t)((stage(j) * C::KV_BYTES) >> 4);
        const uint32_t acc0 = j > 0 ? 1u : 0u;
        bool r = false;
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          mma_ts_e(od, pa + kk * 8, vlo + (uint32_t)((kk * 16 * C::SW_BYTES) >> 4), v_hi, C::IDESC_PV,
                   kk > 0 ? 1u : acc0);
          if (kk == 1) r = nb != 0u && tc::mbar_test(nb, np);
        }
        mma_commit_e(kv_empty(stage(j)));  // the stage may be refilled once P V_j is done
        if (j == nk - 1) mma_commit_e(o_done(t));
        return __all_sync(kFullMask, r);
      };

      // the query tiles are waited for in order, this warp's own and the other's, up to its
      // own (so no wait is ever more than one phase of a slot away); a tile seen is released
      // at once: the tensor core's reads of it are covered by its epilogue's o_done wait
      for (; ok && uw < u0 + min(t + 1, it.nq); ++uw) {
        wait_one(q_full(uw), q_par(uw), false);
        if (ok && lane == 0) tc::mbar_arrive(q_free(uw));  // (a tile not seen landing is never released)
      }
      bool ready = false;  // pre-test result for the next wait
      if (nk > 0) {
        wait_one(kv_full(stage(0)), kv_par(0), false);
        ready = issue_s(0, nk > 1 ? kv_full(stage(1)) : 0u, kv_par(1));
      }
      for (int j = 0; ok && j < n; ++j) {
        if (j < nk) {
          if (j + 1 < nk) {  // S of KV tile j + 1 into the other buffer
            wait_one(kv_full(stage(j + 1)), kv_par(j + 1), ready);
            ready = issue_s(j + 1, p_full(t, sbuf(j)), s_par(j));
          }
          // O_t += P_t(j) V_j (the item's first P V overwrites O once the epilogue of the
          // item before has read it)
          if (j == 0 && n_used > 0) wait_one(o_free(t), (uint32_t)((n_used - 1) & 1), false);
          wait_one(v_full(stage(j)), kv_par(j), false);
          wait_one(p_full(t, sbuf(j)), s_par(j), ready);
          ready = issue_pv(j, j + 2 < nk ? kv_full(stage(j + 2)) : 0u, kv_par(j + 2));
        } else {
          // a KV tile this query tile does not need is still released by this warp, but only
          // once it has landed: otherwise the release could run ahead and count toward an
          // earlier phase of the stage's empty barrier
          wait_one(kv_full(stage(j)), kv_par(j), false);
          if (ok) mma_commit_e(kv_empty(stage(j)));
        }
      }
      gs += nk;
      if (nk > 0) ++n_used;
      g_base += it.n_tiles;
      u0 += it.nq;
    }
    // every MMA this warp issued has completed before the CTA may release tensor memory
    // (MMAs always complete, so this wait takes the default limit whatever the caller's)
    mma_commit_e(fin);
    if (!__all_sync(kFullMask, tc::mbar_wait(fin, 0, tc::kWaitLimit))) *err = 1;
    __syncwarp();
  } else {
    // ======================= softmax: warp group t = warp / 4; thread owns row tid % 128
    const int t = warp >> 2;
    const int row = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t o_col = tmem + lane_base + t * C::TMEM_TILE;
    const float scale = p.scale_log2;
    const bool pos_scale = scale >= 0.f;
    constexpr bool has_mask = MASK;
    int gs = 0, n_used = 0;  // same counters as the MMA thread, for this query tile
    int g_base = 0;          // global index of the item's KV tile 0
    int u0 = 0;              // query tiles of the items before this one
    bool ok = true;
    PrefillItem it;
    for (int n_item = 0; ok; ++n_item) {
      if (!get_item(n_item, it)) break;
      const int u = u0 + t;  // this tile's query-tile number
      u0 += it.nq;
      if (t >= it.nq) {
        g_base += it.n_tiles;
        continue;
      }
      const int qf = it.first0 + t * C::BQ, ql = min(it.q_len, qf + C::BQ) - 1;
      const int n_keys = (min(it.cb + ql + 1, it.kvn) + C::BN - 1) / C::BN;
      const int qi = qf + row / G;                              // this thread's query position
      const int limit = min(it.cb + min(qi, ql), it.kvn - 1);   // last key this row attends
      const int mask_from = min(it.cb + qf + 1, it.kvn) / C::BN;  // tiles >= this one hold a masked key for some row
      // explicit mask: this row's bytes (padded rows past the tile's last position reuse it)
      const uint8_t* mrow = has_mask ? p.mask + (int64_t)it.b * p.mask_req_pitch + (int64_t)min(qi, ql) * p.mask_row_pitch
                                     : nullptr;
      float m_run = -CUDART_INF_F, l_run = 0.f;
      for (int j = 0; j < n_keys; ++j) {
        const int gb = gs + j;
        const uint32_t sb = o_col + D + (gb & 1) * C::BN;  // S_t(j), then P_t(j)
        // the tile's 64 mask bytes load while S is computed; a 16-byte chunk that starts inside
        // the row (pitch a multiple of 16) lies inside it, later ones read as masked
        uint4 mw[4];
        if (has_mask) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            mw[c] = (j * C::BN + 16 * c < p.mask_kv_pitch) ? ldg_nc_v4(mrow + j * C::BN + 16 * c) : make_uint4(0, 0, 0, 0);
        }
        if (!(ok = wait_or_fail(s_full(t, gb & 1), (uint32_t)((gb >> 1) & 1)))) break;
        tc::fence_after_sync();
        float s[C::BN];
        {
          uint32_t raw[32];
#pragma unroll
          for (int half = 0; half < C::BN / 32; ++half) {
            tc::tmem_ld32(sb + half * 32, raw);
            tc::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) s[half * 32 + c] = __uint_as_float(raw[c]);
          }
        }
        // Keys past this row's limit (tiles that cross the causal edge) or hidden by the explicit
        // mask are set to the extreme that the row max / min ignores, and get p = 0 below.
        const bool masked = has_mask || j >= mask_from;
        const int j0 = j * C::BN;
        const float skip = pos_scale ? -CUDART_INF_F : CUDART_INF_F;
        // explicit mask: bit c of vb = key j0 + c visible (mask byte nonzero, key <= limit)
        uint64_t vb = 0;
        if (has_mask) {
          vb = mask_bits64(mw);
          const int n_in = limit - j0 + 1;  // keys of the tile within the row's window
          vb = (n_in >= 64) ? vb : (n_in <= 0 ? 0ull : vb & ((1ull << n_in) - 1ull));
#pragma unroll
          for (int c = 0; c < C::BN; ++c) s[c] = ((vb >> c) & 1ull) ? s[c] : skip;
        } else if (masked) {
#pragma unroll
          for (int c = 0; c < C::BN; ++c) s[c] = (j0 + c <= limit) ? s[c] : skip;
        }
        // P = 2^(sm_scale s - m_run + kPOffset) as fp16 pairs (P V runs in fp16: 11 significant
        // bits, so the only rounding that matters is the output's).  The row max (min for a
        // negative scale) is taken only on a row's first visible tile and when the tile's row
        // sum exceeds kPSumLimit (then some p may be near the fp16 limit): the reference moves
        // up, O and l are rescaled, and P is recomputed.
        bool do_max = __any_sync(kFullMask, m_run == -CUDART_INF_F);
        uint32_t ph[C::BN / 2];
        float lsum = 0.f;
        for (;;) {
          if (do_max) {
            float e4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // four independent 3-input chains over 16 scores each
              float e = skip;
#pragma unroll
              for (int c = q * 16; c < q * 16 + 16; c += 2)
                e = pos_scale ? max3(e, s[c], s[c + 1]) : min3(e, s[c], s[c + 1]);
              e4[q] = e;
            }
            const float ext = pos_scale ? max3(max3(e4[0], e4[1], e4[2]), e4[3], skip)
                                        : min3(min3(e4[0], e4[1], e4[2]), e4[3], skip);
            const bool none = has_mask ? vb == 0ull : j0 > limit;
            const float m_tile = none ? -CUDART_INF_F : ext * scale;  // -inf: no visible key
            const bool need = m_tile > m_run + C::kRescaleThreshold;  // true on the first visible tile
            if (__any_sync(kFullMask, need)) {
              const float alpha = need ? fast_exp2(m_run - m_tile) : 1.f;  // 0 while m_run = -inf
              if (j > 0) {
                // O holds P V of KV tiles < j once P V_{j-1} completes; the issuing thread commits
                // that KV tile's empty barrier right after it, so wait for that phase (rare: only
                // when the row max grows past the threshold)
                const int gp = g_base + j - 1;
                if (!(ok = wait_or_fail(kv_empty(gp % C::STAGES), (uint32_t)((gp / C::STAGES) & 1)))) break;
                tc::fence_after_sync();
#pragma unroll 1
                for (int cc = 0; cc < D / 16; ++cc) {
                  uint32_t o[16];
                  tc::tmem_ld16(o_col + cc * 16, o);
                  tc::tmem_ld_wait();
#pragma unroll
                  for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                  tc::tmem_st16(o_col + cc * 16, o);
                }
              }
              l_run *= alpha;
              if (need) m_run = m_tile;
            }
          }
          // pairs of scores through packed fp32x2 arithmetic
          const float neg_m = (m_run == -CUDART_INF_F) ? 0.f : C::kPOffset - m_run;
          const uint64_t sc2 = pk2(scale, scale), nm2 = pk2(neg_m, neg_m);
          uint64_t lsum2 = pk2(0.f, 0.f);
          if (has_mask || masked) {  // a tile with hidden keys: their p is forced to 0
#pragma unroll
            for (int e = 0; e < C::BN / 2; ++e) {
              const int c0 = 2 * e;
              float x0, x1;
              upk2(fma2(pk2(s[c0], s[c0 + 1]), sc2, nm2), x0, x1);
              float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              if (has_mask) {
                p0 = ((vb >> c0) & 1ull) ? p0 : 0.f;
                p1 = ((vb >> (c0 + 1)) & 1ull) ? p1 : 0.f;
              } else {
                p0 = (j0 + c0 <= limit) ? p0 : 0.f;
                p1 = (j0 + c0 + 1 <= limit) ? p1 : 0.f;
              }
              lsum2 = add2(lsum2, pk2(p0, p1));
              ph[e] = float2_to_f16x2_rn(p0, p1);
            }
          } else {  // every key of the tile is visible to every row
#pragma unroll
            for (int e = 0; e < C::BN / 2; ++e) {
              const int c0 = 2 * e;
              float x0, x1;
              upk2(fma2(pk2(s[c0], s[c0 + 1]), sc2, nm2), x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              lsum2 = add2(lsum2, pk2(p0, p1));
              ph[e] = float2_to_f16x2_rn(p0, p1);
            }
          }
          float ls0, ls1;
          upk2(lsum2, ls0, ls1);
          lsum = ls0 + ls1;
          if (do_max || !__any_sync(kFullMask, lsum > C::kPSumLimit)) break;
          do_max = true;
        }
        if (!ok) break;
        l_run += lsum;
        tc::tmem_st32(sb, ph);  // P over the S columns just read (fp16 pairs: 32 columns)
        tc::tmem_st_wait();
        tc::fence_before_sync();
        tc::mbar_arrive(p_full(t, gb & 1));
      }
      if (!ok) break;

      // ---- epilogue, once the last P V of this tile has landed: O / l as bf16 into the
      // tile's query slot (free: every S that read it is complete), release O, and hand the
      // slot to the query warp, which writes the rows out while these warps go on
      ok = wait_or_fail(o_done(t), (uint32_t)(n_used & 1));
      tc::fence_after_sync();
      tc::fence_proxy_async_smem();  // the tensor core's reads of this buffer precede the writes below
      // a timed-out wait poisons the tile; a row with no visible key (explicit mask) is zero
      const float inv = (ok && !*err) ? (l_run > 0.f ? 1.f / l_run : 0.f) : CUDART_NAN_F;
      const uint32_t stg = q_slot(u);
      bool nonfinite = false;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tc::tmem_ld32(o_col + cc * 32, o);
        tc::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) nonfinite |= !(fabsf(__uint_as_float(o[c])) <= 3.4e38f);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 v;
          v.x = float2_to_bf16x2_rn(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv);
          v.y = float2_to_bf16x2_rn(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv);
          v.z = float2_to_bf16x2_rn(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv);
          v.w = float2_to_bf16x2_rn(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv);
          sts128(stg + swz<C::SW_BYTES>(row, cc * 4 + q4, C::M), v);
        }
      }
      if (ok && !*err && p.status != nullptr && __any_sync(kFullMask, nonfinite) && lane == 0)
        atomicOr(p.status, kStatusRange);
      tc::fence_before_sync();
      tc::mbar_arrive(o_free(t));    // O of this tile may be overwritten by the next item
      tc::fence_proxy_async_smem();  // the staged rows are read by TMA stores (async proxy)
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(o_staged(u));
      gs += n_keys;
      ++n_used;
      g_base += it.n_tiles;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc<C::TMEM_COLS>(tmem);
    if (lane == 0 && *err != 0 && p.status != nullptr) atomicOr(p.status, kStatusTimeout);
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against libcuda)
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult status{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &status) !=
            cudaSuccess ||
        status != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

template <int D, int G, bool MASK, bool CONTIG>
cudaError_t launch_prefill_t(const PrefillParams& p, cudaStream_t stream) {
  using C = PrefillCfg<D, G>;
  static std::atomic<bool> attr_done[kMaxDevices];
  const cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(prefill_kernel<D, G, MASK, CONTIG>),
                                            C::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  // persistent CTAs, one per SM, each walking its share of the items
  const int64_t items = (int64_t)p.num_q_tiles * p.num_kv_heads;
  const int grid = (int)(items < p.num_ctas ? items : p.num_ctas);
  if (grid <= 0) return cudaSuccess;
  // q as [total_q][Hq][D] bf16; one box = BQ positions x the G heads of a KV head x one column
  // block (64 columns with 128-byte swizzle; 32 with 64-byte swizzle for D = 32)
  const PFN_cuTensorMapEncodeTiled_v12000 encode = encode_tiled();
  if (encode == nullptr) return cudaErrorNotSupported;
  // (out has the same layout; its map writes whole tiles of one request)
  // packed rows: [total_q rows][Hq][D] by (row stride, head stride); padded: [B][q_rows][Hq][D]
  // by (batch, row, head strides) -- a 4-D map addressed by (column, head, local row, request)
  CUtensorMap q_map, o_map;
  const CUtensorMapSwizzle swz_mode = C::SW_BYTES == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const cuuint32_t box[4] = {(cuuint32_t)C::CB_ELEMS, (cuuint32_t)G, (cuuint32_t)C::BQ, 1u};
  const cuuint32_t elem_strides[4] = {1u, 1u, 1u, 1u};
  auto make_map = [&](CUtensorMap* map, const uint16_t* base, int64_t bstride, int64_t tstride, int64_t hstride,
                      CUtensorMapL2promotion promo) {
    const bool padded = bstride > 0;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)p.num_qo_heads,
                                (cuuint64_t)(padded ? p.q_rows : p.total_q), (cuuint64_t)p.batch};
    const cuuint64_t strides[3] = {(cuuint64_t)hstride * 2, (cuuint64_t)tstride * 2, (cuuint64_t)bstride * 2};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, padded ? 4 : 3, const_cast<uint16_t*>(base), dims, strides,
                  box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swz_mode, promo,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  if (!make_map(&q_map, p.q, p.q_batch, p.q_token, p.q_head, CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
      !make_map(&o_map, p.out, p.o_batch, p.o_token, p.o_head, CU_TENSOR_MAP_L2_PROMOTION_NONE))
    return cudaErrorInvalidValue;
  prefill_kernel<D, G, MASK, CONTIG><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(p, q_map, o_map);
  return cudaGetLastError();
}

template <bool MASK, bool CONTIG>
cudaError_t dispatch_prefill(const PrefillParams& p, cudaStream_t stream) {
  const int G = p.num_qo_heads / p.num_kv_heads;
#define ASTR_PF_CASE(DD, GG) \
  if (p.head_dim == DD && G == GG) return launch_prefill_t<DD, GG, MASK, CONTIG>(p, stream);
  ASTR_PF_CASE(128, 4) ASTR_PF_CASE(128, 1) ASTR_PF_CASE(128, 2) ASTR_PF_CASE(128, 8) ASTR_PF_CASE(128, 16)
  ASTR_PF_CASE(64, 4) ASTR_PF_CASE(64, 1) ASTR_PF_CASE(64, 2) ASTR_PF_CASE(64, 8) ASTR_PF_CASE(64, 16)
  ASTR_PF_CASE(32, 4) ASTR_PF_CASE(32, 1) ASTR_PF_CASE(32, 2) ASTR_PF_CASE(32, 8) ASTR_PF_CASE(32, 16)
#undef ASTR_PF_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

// The kernels with an explicit mask and those over a contiguous K/V cache are further
// instantiations of the same template, compiled in translation units of their own
// (prefill_masked.cu and prefill_contig.cu include this file with ASTR_PREFILL_MASKED_TU or
// ASTR_PREFILL_CONTIG_TU defined) so the sets build in parallel.
#if defined(ASTR_PREFILL_MASKED_TU)
cudaError_t launch_prefill_masked(const PrefillParams& p, cudaStream_t stream) {
  return dispatch_prefill<true, false>(p, stream);
}
#elif defined(ASTR_PREFILL_CONTIG_TU)
cudaError_t launch_prefill_contig(const PrefillParams& p, cudaStream_t stream) {
  return p.mask != nullptr ? dispatch_prefill<true, true>(p, stream) : dispatch_prefill<false, true>(p, stream);
}
#else
int prefill_rows_per_cta() { return 256; }

bool prefill_supported(int head_dim, int group) {
  return (head_dim == 32 || head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream) {
  if (p.contig) return launch_prefill_contig(p, stream);
  if (p.mask != nullptr) return launch_prefill_masked(p, stream);
  return dispatch_prefill<false, false>(p, stream);
}
#endif

}  // namespace astr
