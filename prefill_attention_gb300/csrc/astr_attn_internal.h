// astr_attn_internal.h -- parameter blocks and launcher declarations shared between the
// C-ABI layer (api.cu) and the kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace astr {

constexpr int kMaxDevices = 64;

// Raises func's dynamic shared-memory limit to `bytes` on the current device, once per device
// (the attribute belongs to the device that is current when it is set).  `done` is the
// caller's table for this kernel.  Thread-safe.
cudaError_t set_smem_limit_once(const void* func, int bytes, std::atomic<bool> (&done)[kMaxDevices]);

// Status-word bits (the ASTR_KSTATUS_* values of the C header).
constexpr int kStatusTimeout = 1, kStatusBadInput = 2, kStatusSmem = 4, kStatusRange = 8, kStatusPlan = 16;

// Prefill work plan (int32 words): a header, then one row per CTA of the launch -- the item
// count and up to kPlanMaxItems items, each (request, pair << 16 | KV head).
constexpr int kPlanMagic = 0x41535450;  // "ASTP"
constexpr int kPlanVersion = 1;
constexpr int kPlanHeader = 8;          // magic, version, batch, Hkv, pair height, grid, checksum, causal
constexpr int kPlanMaxItems = 128;
constexpr int kPlanRow = 1 + 2 * kPlanMaxItems;

// Checksum of a call's qo_indptr [batch + 1] and seq_lens [batch], the same on the host and in
// the kernel: a sum of per-element mixes (an integer hash of the index and the value), so
// threads can add their shares in any order.
__host__ __device__ inline uint32_t plan_mix(uint32_t i, uint32_t v) {
  uint32_t h = v * 0x9E3779B1u + i * 0x85EBCA77u + 0x165667B1u;
  h ^= h >> 15;
  h *= 0x2C1B3C6Du;
  h ^= h >> 12;
  h *= 0x297A2D39u;
  h ^= h >> 15;
  return h;
}
constexpr uint32_t kPlanSeqTag = 0x40000000u;  // index offset of the seq_lens elements

// Decode split kernel: a CTA runs this many independent warp pairs, one key chunk each.
constexpr int kDecodeChunksPerCta = 4;

// Contiguous (stride-addressed) K/V cache instead of pool + slot table: element e of key
// position j, KV head h, request b sits at b * batch + j * token + h * head + e (elements; all
// three strides multiples of 8, i.e. 16 bytes).  Positions up to max_len - 1 exist.
struct KvStrides {
  int64_t batch, token, head;
  int max_len;
};

// Decode: one launch of the split kernel followed by one launch of the combine kernel.
struct DecodeParams {
  const uint16_t* q;             // [B, Hq, D]
  const uint16_t* k_pool;        // [num_slots, Hkv, D]
  const uint16_t* v_pool;
  const int32_t* req_to_token;   // [B, r2t_stride]
  const int32_t* seq_lens;       // [B]
  const int32_t* kv_indptr;      // [B + 1] exclusive prefix sum of seq_lens
  float* o_part;                 // [B, Hq, part_pitch, D]
  float* ml_part;                // [B, Hq, part_pitch, 2]
  uint16_t* out;                 // [B, Hq, D]
  int64_t r2t_stride;
  int64_t num_slots;             // rows of k_pool / v_pool (sizes the gather tensor maps)
  int batch, num_qo_heads, num_kv_heads, head_dim;
  int num_splits;                // chunks per KV head (kDecodeChunksPerCta per CTA)
  int part_pitch;                // partial slots per (b, h) row of o_part (= max_splits)
  int min_chunk;                 // floor on the chunk length (32-key slots) so no request needs
                                 // more than part_pitch partial slots
  float scale_log2;              // sm_scale * log2(e): logits are kept in base-2 units on chip
  int combine_all;               // combine even single-chunk requests (partials supplied by the caller)
  int indptr_before_wait;        // combine: kv_indptr may be read before the dependency wait (the
                                 // previous kernel is this call's split kernel, which does not write it)
  int early_index;               // split: plan the chunks before the dependency wait (the caller's
                                 // index arrays are not written by the preceding kernel)
  int32_t* status;               // optional status word (kStatus* bits, OR-ed in); may be null
  uint32_t wait_limit;           // polls per pipeline wait before giving up
};

// Decode query / output rows by strides: request b, head h at q + b * q_req + h * q_head
// (elements), the same for out.  The packed [B, Hq, D] layout is q_req = Hq * D, q_head = D;
// the kernels take it at compile time when no strides are given.
struct QoStrides {
  int64_t q_req, q_head, o_req, o_head;
};

// Decode with an explicit mask: request b's bytes start at mask + b * req_pitch, one byte per
// key position.  Kept out of DecodeParams so the unmasked kernels' parameter block is unchanged.
struct DecodeMask {
  const uint8_t* mask;
  int64_t req_pitch;
  int kv_pitch;                  // bytes in a mask row (a multiple of 16)
};

// Prefill/extend: one launch of the tensor-core kernel.
struct PrefillParams {
  const uint16_t* q;             // [total_q, Hq, D]
  const int32_t* qo_indptr;      // [B + 1]
  const uint16_t* k_pool;        // [num_slots, Hkv, D]
  const uint16_t* v_pool;
  const int32_t* req_to_token;   // [B, r2t_stride]
  const int32_t* seq_lens;       // [B]
  uint16_t* out;                 // [total_q, Hq, D]
  int64_t r2t_stride;
  int64_t num_slots;             // rows of k_pool / v_pool (slot ids outside read as zeros)
  int batch, num_qo_heads, num_kv_heads, head_dim;
  int total_q;
  int num_q_tiles;               // upper bound on (request, query-tile pair) work items per KV head
  int num_ctas;                  // persistent CTAs to launch (one per SM)
  float scale_log2;
  int causal;                    // 1: key j visible to local row i iff j <= seq_len - q_len + i; 0: off
  const uint8_t* mask;           // explicit mask or nullptr: row i of request b at
                                 // mask + b * mask_req_pitch + i * mask_row_pitch (0 for 2-D masks)
  int64_t mask_req_pitch, mask_row_pitch;
  int mask_kv_pitch;             // bytes in a mask row (a multiple of 16)
  int contig;                    // 1: K/V rows come from a contiguous cache addressed by kv
  KvStrides kv;
  int32_t* status;               // optional status word (kStatus* bits, OR-ed in); may be null
  uint32_t wait_limit;           // polls per pipeline wait before giving up
  // query row i of request b, head h (elements): q_batch == 0 -> (qo_indptr[b] + i) * q_token +
  // h * q_head (packed; [total_q, Hq, D] is q_token = Hq * D, q_head = D); q_batch > 0 ->
  // b * q_batch + i * q_token + h * q_head (padded, q_rows positions per request).  Same for out.
  int64_t q_batch, q_token, q_head, o_batch, o_token, o_head;
  int q_rows;
  const int32_t* plan;           // work plan (kPlan* layout) the host found large enough, or null
  int plan_rejected;             // 1: the call had a plan too small for its grid (reported, not read)
};

// KV append: one launch, one warp per new token.
struct AppendParams {
  const uint16_t* k_new;         // [total_q, Hkv, D]
  const uint16_t* v_new;
  const int32_t* qo_indptr;      // [B + 1]
  const int32_t* req_to_token;   // [B, r2t_stride]
  const int32_t* seq_lens;       // [B]
  uint16_t* k_pool;              // [num_slots, Hkv, D]
  uint16_t* v_pool;
  int64_t r2t_stride;
  int64_t num_slots;             // slot ids outside [0, num_slots) are skipped
  int batch, total_q;
  int row_vecs;                  // 16-byte vectors per slot row (Hkv * D * 2 / 16)
  int32_t* status;               // optional status word (kStatus* bits, OR-ed in); may be null
};

// Launchers return cudaSuccess or the launch error; they never synchronise.
// mask / strides may be null (no explicit mask / the paged pool through req_to_token)
// qo may be null as well (the packed query / output layout)
cudaError_t launch_decode_split(const DecodeParams& p, const DecodeMask* mask, const KvStrides* strides,
                                const QoStrides* qo, cudaStream_t stream);
cudaError_t launch_decode_combine(const DecodeParams& p, const QoStrides* qo, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream);         // dispatches on p.mask
cudaError_t launch_prefill_masked(const PrefillParams& p, cudaStream_t stream);  // the explicit-mask kernels
cudaError_t launch_prefill_contig(const PrefillParams& p, cudaStream_t stream);  // the contiguous-cache kernels
cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream);

// Whether the kernels exist for this (head_dim, group size).
bool decode_supported(int head_dim, int group);
bool prefill_supported(int head_dim, int group);
int prefill_rows_per_cta();  // query-head rows per CTA (two tensor-core tiles of M = 128)

}  // namespace astr
