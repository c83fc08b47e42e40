// api.cu -- the C ABI declared in include/astr_attn.h: argument checks, split planning
// and kernel launches on the caller's stream.  No allocation, no synchronisation, no
// device-memory reads on the host, so every entry point can be captured in a CUDA graph.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "astr_attn.h"
#include "astr_attn_internal.h"

namespace astr {

cudaError_t set_smem_limit_once(const void* func, int bytes, std::atomic<bool> (&done)[kMaxDevices]) {
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  done[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

}  // namespace astr

namespace {

using astr::kMaxDevices;
constexpr int kDecodeCtasPerSm = 1;     // the split kernel is persistent: one CTA per SM
constexpr uint32_t kDefaultWaitLimit = 1u << 20;  // polls per pipeline wait (dims->wait_limit = 0)

std::mutex g_mu;
int g_sm_count[kMaxDevices] = {0};

int sm_count(int device, int* out) {
  if (device < 0 || device >= kMaxDevices) return ASTR_ERR_DEVICE;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[device] > 0) {
      *out = g_sm_count[device];
      return ASTR_OK;
    }
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0) {
    cudaGetLastError();  // clear the sticky-free error so later launches are not blamed
    return ASTR_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_sm_count[device] = n;
  *out = n;
  return ASTR_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape checks common to both paths.
int check_common(const astr_attn_dims* d) {
  if (d == nullptr) return ASTR_ERR_INVALID_ARG;
  if (d->batch < 0 || d->num_qo_heads < 1 || d->num_kv_heads < 1 || d->head_dim < 1 || d->num_slots < 0 ||
      d->r2t_stride < 0 || d->max_seq_len < 0)
    return ASTR_ERR_INVALID_ARG;
  if (d->num_qo_heads % d->num_kv_heads != 0) return ASTR_ERR_UNSUPPORTED;
  if (d->head_dim != 32 && d->head_dim != 64 && d->head_dim != 128) return ASTR_ERR_UNSUPPORTED;
  if (d->r2t_stride < d->max_seq_len) return ASTR_ERR_INVALID_ARG;
  if (d->batch > 0 && d->max_seq_len > 0 && d->num_slots < 1) return ASTR_ERR_INVALID_ARG;
  if (d->num_kv_heads > 65535 || d->batch > 65535) return ASTR_ERR_INVALID_ARG;  // grid y / z limits
  if (d->status != nullptr && !aligned(d->status, 4)) return ASTR_ERR_MISALIGNED;
  if ((d->flags & ~ASTR_DIMS_STABLE_INDICES) != 0) return ASTR_ERR_INVALID_ARG;  // an undefined flag bit
  return ASTR_OK;
}

uint32_t wait_limit_of(const astr_attn_dims* d) { return d->wait_limit != 0 ? d->wait_limit : kDefaultWaitLimit; }

// Key chunks per KV head: one wave of persistent CTAs (kv heads x CTAs = SMs), each CTA
// running kDecodeChunksPerCta chunks.
int plan_splits(const astr_attn_dims* d, int sms) {
  if (d->num_splits > 0) return d->num_splits;
  const int64_t target = (int64_t)sms * kDecodeCtasPerSm;
  int64_t s = (target + d->num_kv_heads - 1) / d->num_kv_heads;
  if (s < 1) s = 1;
  return (int)(s * astr::kDecodeChunksPerCta);
}

// Floor on the chunk length in 32-key slots: a request of max_seq_len keys has
// m = ceil(max_seq_len / 32) slots and overlaps at most ceil(m / C) + 1 chunks, which must
// fit in max_splits partial slots.
int plan_min_chunk(const astr_attn_dims* d) {
  if (d->max_splits <= 1) return 1;  // single chunk per KV head (the kernel uses all slots)
  const int64_t m = ((int64_t)d->max_seq_len + 31) / 32;
  int64_t c = (m + d->max_splits - 2) / (d->max_splits - 1);
  if (c < 1) c = 1;
  return (int)c;
}

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return ASTR_ERR_DEVICE;
  }
  return ASTR_OK;
}

// Prefill launch size: pairs of query tiles per KV head (an upper bound from host-known
// values) and the persistent grid, min(items, SMs).  Shared by the call and the planner so a
// plan is made for exactly the grid the call launches.
int64_t prefill_q_tiles(const astr_attn_dims* d) {
  const int G = d->num_qo_heads / d->num_kv_heads;
  const int bq = astr::prefill_rows_per_cta() / G;  // query positions per pair
  const int64_t by_total = ((int64_t)d->total_q + bq - 1) / bq + d->batch;
  const int64_t by_max = (int64_t)d->batch * (((int64_t)d->max_q_len + bq - 1) / bq);
  return by_total < by_max ? by_total : by_max;
}
int prefill_grid(const astr_attn_dims* d, int sms) {
  const int64_t items = prefill_q_tiles(d) * d->num_kv_heads;
  return (int)(items < sms ? items : sms);
}

}  // namespace

extern "C" {

const char* astr_attn_status_string(int status) {
  switch (status) {
    case ASTR_OK: return "ok";
    case ASTR_ERR_INVALID_ARG: return "invalid argument (null pointer, negative or inconsistent dims, non-finite scale)";
    case ASTR_ERR_UNSUPPORTED: return "unsupported shape (head_dim must be 32, 64 or 128; Hq % Hkv == 0; supported group size)";
    case ASTR_ERR_MISALIGNED: return "misaligned pointer (bf16/fp32 arrays need 16-byte, int32 arrays 4-byte alignment)";
    case ASTR_ERR_WORKSPACE_TOO_SMALL: return "workspace too small (num_splits above max_splits)";
    case ASTR_ERR_LAUNCH_FAILED: return "CUDA launch failed";
    case ASTR_ERR_DEVICE: return "CUDA device query failed";
    default: return "unknown status";
  }
}

int astr_attn_version(void) { return 20100; }

int astr_attn_decode_workspace_bytes(const astr_attn_dims* d, size_t* o_bytes, size_t* ml_bytes) {
  if (d == nullptr || o_bytes == nullptr || ml_bytes == nullptr) return ASTR_ERR_INVALID_ARG;
  if (d->batch < 0 || d->num_qo_heads < 1 || d->head_dim < 1 || d->max_splits < 1) return ASTR_ERR_INVALID_ARG;
  const size_t rows = (size_t)d->batch * (size_t)d->num_qo_heads * (size_t)d->max_splits;
  *o_bytes = rows * (size_t)d->head_dim * sizeof(float);
  *ml_bytes = rows * 2 * sizeof(float);
  return ASTR_OK;
}

int astr_attn_decode_num_splits(const astr_attn_dims* d, int device, int* num_splits) {
  if (num_splits == nullptr) return ASTR_ERR_INVALID_ARG;
  int st = check_common(d);
  if (st != ASTR_OK) return st;
  if (d->max_splits < 1 || d->num_splits < 0) return ASTR_ERR_INVALID_ARG;
  int sms = 0;
  st = sm_count(device, &sms);
  if (st != ASTR_OK) return st;
  *num_splits = plan_splits(d, sms);
  return ASTR_OK;
}

static int decode_prepare(const astr_attn_dims* d, float sm_scale, astr::DecodeParams* p, bool* nothing) {
  int st = check_common(d);
  if (st != ASTR_OK) return st;
  if (d->max_splits < 1 || d->num_splits < 0) return ASTR_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return ASTR_ERR_INVALID_ARG;
  const int G = d->num_qo_heads / d->num_kv_heads;
  if (!astr::decode_supported(d->head_dim, G)) return ASTR_ERR_UNSUPPORTED;
  *nothing = (d->batch == 0);
  int dev = 0, sms = 0;
  if ((st = current_device(&dev)) != ASTR_OK) return st;
  if ((st = sm_count(dev, &sms)) != ASTR_OK) return st;
  if (d->num_slots * (int64_t)d->num_kv_heads > 0x7fffffffLL) return ASTR_ERR_INVALID_ARG;  // TMA row index
  p->r2t_stride = d->r2t_stride;
  p->num_slots = d->num_slots;
  p->batch = d->batch;
  p->num_qo_heads = d->num_qo_heads;
  p->num_kv_heads = d->num_kv_heads;
  p->head_dim = d->head_dim;
  p->num_splits = plan_splits(d, sms);
  p->part_pitch = d->max_splits;
  p->min_chunk = plan_min_chunk(d);
  p->scale_log2 = sm_scale * 1.4426950408889634f;
  p->status = d->status;
  p->wait_limit = wait_limit_of(d);
  p->early_index = (d->flags & ASTR_DIMS_STABLE_INDICES) ? 1 : 0;
  if (p->num_splits > 0x7fffffff / 2) return ASTR_ERR_INVALID_ARG;
  return ASTR_OK;
}

// Query / output strides: non-negative multiples of 8 elements (16-byte rows); NULL = packed.
static int check_qo_layout(const astr_attn_qo_layout* l, const astr_attn_dims* d, astr_attn_qo_layout* out) {
  const int64_t row = (int64_t)d->num_qo_heads * d->head_dim;
  *out = astr_attn_qo_layout{0, row, d->head_dim, 0, row, d->head_dim};
  if (l == nullptr) return ASTR_OK;
  const int64_t v[6] = {l->q_batch_stride, l->q_token_stride, l->q_head_stride,
                        l->o_batch_stride, l->o_token_stride, l->o_head_stride};
  for (int64_t x : v)
    if (x < 0) return ASTR_ERR_INVALID_ARG;
  for (int64_t x : v)
    if (x % 8 != 0) return ASTR_ERR_MISALIGNED;
  *out = *l;
  return ASTR_OK;
}

// Contiguous-cache layout: strides non-negative multiples of 8 elements (16-byte rows).
static int check_layout(const astr_attn_kv_layout* l, const astr_attn_dims* d, astr::KvStrides* ks) {
  if (l == nullptr || d == nullptr) return ASTR_ERR_INVALID_ARG;
  if (l->batch_stride < 0 || l->token_stride < 0 || l->head_stride < 0) return ASTR_ERR_INVALID_ARG;
  if (l->batch_stride % 8 != 0 || l->token_stride % 8 != 0 || l->head_stride % 8 != 0) return ASTR_ERR_MISALIGNED;
  *ks = astr::KvStrides{l->batch_stride, l->token_stride, l->head_stride, d->max_seq_len};
  return ASTR_OK;
}

// The dims as the shared checks expect them when K/V come from a contiguous cache: no slot
// table (its pitch taken as max_seq_len) and no pool (one nominal slot).
static astr_attn_dims contiguous_dims(const astr_attn_dims* d) {
  astr_attn_dims c = *d;
  c.r2t_stride = d->max_seq_len;
  c.num_slots = 1;
  return c;
}

// Explicit-mask arguments: shape rules, then the pitches of request b's bytes (and of its rows).
static int check_mask(const astr_attn_mask* m, const astr_attn_dims* d, bool decode, int64_t* req_pitch,
                      int64_t* row_pitch) {
  if (m == nullptr || d == nullptr) return ASTR_ERR_INVALID_ARG;
  if (m->causal != 0 && m->causal != 1) return ASTR_ERR_INVALID_ARG;
  *req_pitch = *row_pitch = 0;
  if (m->mask == nullptr) return ASTR_OK;
  if (!aligned(m->mask, 16)) return ASTR_ERR_MISALIGNED;
  if (m->dims != 2 && m->dims != 3) return ASTR_ERR_INVALID_ARG;
  if (m->kv_pitch < 16 || m->kv_pitch % 16 != 0 || m->kv_pitch < d->max_seq_len) return ASTR_ERR_INVALID_ARG;
  if (m->dims == 3 && (m->q_pitch < 1 || (!decode && m->q_pitch < d->max_q_len))) return ASTR_ERR_INVALID_ARG;
  *req_pitch = (m->dims == 3) ? (int64_t)m->q_pitch * m->kv_pitch : (int64_t)m->kv_pitch;
  *row_pitch = (m->dims == 3) ? (int64_t)m->kv_pitch : 0;
  return ASTR_OK;
}

static int paged_decode_impl(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                             const int32_t* req_to_token, const int32_t* seq_lens, const int32_t* kv_indptr,
                             const astr_attn_mask* mask, const astr_attn_kv_layout* layout,
                             const astr_attn_qo_layout* qo_layout, float* o_part, float* ml_part, uint16_t* out,
                             const astr_attn_dims* dims, float sm_scale, void* stream) {
  const bool contig = layout != nullptr;  // K/V from a contiguous cache: no slot table
  if (!q || !k_pool || !v_pool || (!contig && !req_to_token) || !seq_lens || !kv_indptr || !o_part || !ml_part || !out)
    return ASTR_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o_part, 16) ||
      !aligned(ml_part, 16) || !aligned(out, 16) || !aligned(req_to_token, 4) || !aligned(seq_lens, 4) ||
      !aligned(kv_indptr, 4))
    return ASTR_ERR_MISALIGNED;
  if (dims == nullptr) return ASTR_ERR_INVALID_ARG;
  int64_t mask_req_pitch = 0, mask_row_pitch = 0;
  int st = ASTR_OK;
  if (mask != nullptr && (st = check_mask(mask, dims, true, &mask_req_pitch, &mask_row_pitch)) != ASTR_OK) return st;
  astr::KvStrides ks{0, 0, 0, 0};
  if (contig && (st = check_layout(layout, dims, &ks)) != ASTR_OK) return st;
  astr_attn_qo_layout qo{};
  if ((st = check_qo_layout(qo_layout, dims, &qo)) != ASTR_OK) return st;
  const astr_attn_dims cdims = contig ? contiguous_dims(dims) : *dims;
  astr::DecodeParams p{};
  bool nothing = false;
  st = decode_prepare(&cdims, sm_scale, &p, &nothing);
  if (st != ASTR_OK || nothing) return st;
  // one row per request: a packed tensor steps by its row stride, a padded one by its batch stride
  const astr::QoStrides qs{qo.q_batch_stride > 0 ? qo.q_batch_stride : qo.q_token_stride, qo.q_head_stride,
                           qo.o_batch_stride > 0 ? qo.o_batch_stride : qo.o_token_stride, qo.o_head_stride};
  const int64_t row = (int64_t)dims->num_qo_heads * dims->head_dim;
  const bool packed = qs.q_req == row && qs.q_head == dims->head_dim && qs.o_req == row && qs.o_head == dims->head_dim;
  astr::DecodeMask dm{nullptr, 0, 0};
  if (mask != nullptr && mask->mask != nullptr) dm = astr::DecodeMask{mask->mask, mask_req_pitch, mask->kv_pitch};
  p.q = q; p.k_pool = k_pool; p.v_pool = v_pool; p.req_to_token = req_to_token; p.seq_lens = seq_lens;
  p.kv_indptr = kv_indptr; p.o_part = o_part; p.ml_part = ml_part; p.out = out;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (astr::launch_decode_split(p, dm.mask != nullptr ? &dm : nullptr, contig ? &ks : nullptr, packed ? nullptr : &qs,
                                s) != cudaSuccess)
    return ASTR_ERR_LAUNCH_FAILED;
  p.indptr_before_wait = 1;  // the combine follows this call's split kernel directly
  if (astr::launch_decode_combine(p, packed ? nullptr : &qs, s) != cudaSuccess) return ASTR_ERR_LAUNCH_FAILED;
  return ASTR_OK;
}

int astr_attn_paged_decode(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                           const int32_t* req_to_token, const int32_t* seq_lens, const int32_t* kv_indptr,
                           float* o_part, float* ml_part, uint16_t* out, const astr_attn_dims* dims, float sm_scale,
                           void* stream) {
  return paged_decode_impl(q, k_pool, v_pool, req_to_token, seq_lens, kv_indptr, nullptr, nullptr, nullptr, o_part,
                           ml_part, out, dims, sm_scale, stream);
}

int astr_attn_paged_decode_masked(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                                  const int32_t* req_to_token, const int32_t* seq_lens, const int32_t* kv_indptr,
                                  const astr_attn_mask* mask, float* o_part, float* ml_part, uint16_t* out,
                                  const astr_attn_dims* dims, float sm_scale, void* stream) {
  if (mask == nullptr) return ASTR_ERR_INVALID_ARG;
  return paged_decode_impl(q, k_pool, v_pool, req_to_token, seq_lens, kv_indptr, mask, nullptr, nullptr, o_part,
                           ml_part, out, dims, sm_scale, stream);
}

int astr_attn_decode_contiguous(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                const astr_attn_kv_layout* layout, const int32_t* seq_lens, const int32_t* kv_indptr,
                                const astr_attn_mask* mask, float* o_part, float* ml_part, uint16_t* out,
                                const astr_attn_dims* dims, float sm_scale, void* stream) {
  if (layout == nullptr) return ASTR_ERR_INVALID_ARG;
  return paged_decode_impl(q, k_cache, v_cache, nullptr, seq_lens, kv_indptr, mask, layout, nullptr, o_part, ml_part,
                           out, dims, sm_scale, stream);
}

int astr_attn_decode_strided(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* req_to_token,
                             const astr_attn_kv_layout* kv_layout, const astr_attn_qo_layout* qo_layout,
                             const int32_t* seq_lens, const int32_t* kv_indptr, const astr_attn_mask* mask,
                             float* o_part, float* ml_part, uint16_t* out, const astr_attn_dims* dims, float sm_scale,
                             void* stream) {
  return paged_decode_impl(q, k, v, kv_layout != nullptr ? nullptr : req_to_token, seq_lens, kv_indptr, mask,
                           kv_layout, qo_layout, o_part, ml_part, out, dims, sm_scale, stream);
}

int astr_attn_decode_split(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                           const int32_t* req_to_token, const int32_t* seq_lens, const int32_t* kv_indptr,
                           float* o_part, float* ml_part, const astr_attn_dims* dims, float sm_scale, void* stream) {
  if (!q || !k_pool || !v_pool || !req_to_token || !seq_lens || !kv_indptr || !o_part || !ml_part)
    return ASTR_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(o_part, 16) ||
      !aligned(ml_part, 16) || !aligned(req_to_token, 4) || !aligned(seq_lens, 4) || !aligned(kv_indptr, 4))
    return ASTR_ERR_MISALIGNED;
  astr::DecodeParams p{};
  bool nothing = false;
  int st = decode_prepare(dims, sm_scale, &p, &nothing);
  if (st != ASTR_OK || nothing) return st;
  p.q = q; p.k_pool = k_pool; p.v_pool = v_pool; p.req_to_token = req_to_token; p.seq_lens = seq_lens;
  p.kv_indptr = kv_indptr; p.o_part = o_part; p.ml_part = ml_part;
  if (astr::launch_decode_split(p, nullptr, nullptr, nullptr, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ASTR_ERR_LAUNCH_FAILED;
  return ASTR_OK;
}

int astr_attn_decode_combine(const float* o_part, const float* ml_part, const int32_t* seq_lens,
                             const int32_t* kv_indptr, uint16_t* out, const astr_attn_dims* dims, void* stream) {
  (void)seq_lens;
  if (!o_part || !ml_part || !out) return ASTR_ERR_INVALID_ARG;
  if (!aligned(o_part, 16) || !aligned(ml_part, 16) || !aligned(out, 16) ||
      (kv_indptr != nullptr && !aligned(kv_indptr, 4)))
    return ASTR_ERR_MISALIGNED;
  if (kv_indptr == nullptr && dims != nullptr) {  // explicit layout: num_splits partials per (b, h)
    if (dims->num_splits < 1) return ASTR_ERR_INVALID_ARG;
    if (dims->num_splits > dims->max_splits) return ASTR_ERR_WORKSPACE_TOO_SMALL;
  }
  astr::DecodeParams p{};
  bool nothing = false;
  int st = decode_prepare(dims, 1.0f, &p, &nothing);
  if (st != ASTR_OK || nothing) return st;
  p.kv_indptr = kv_indptr;
  p.combine_all = 1;  // standalone combine: every request's partials come from the caller
  p.o_part = const_cast<float*>(o_part);
  p.ml_part = const_cast<float*>(ml_part);
  p.out = out;
  if (astr::launch_decode_combine(p, nullptr, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ASTR_ERR_LAUNCH_FAILED;
  return ASTR_OK;
}

static int prefill_impl(const uint16_t* q, const int32_t* qo_indptr, const uint16_t* k_pool, const uint16_t* v_pool,
                        const int32_t* req_to_token, const int32_t* seq_lens, const int32_t* kv_indptr,
                        const astr_attn_mask* mask, const astr_attn_kv_layout* layout,
                        const astr_attn_qo_layout* qo_layout, uint16_t* out, const astr_attn_dims* dims,
                        float sm_scale, void* stream) {
  (void)kv_indptr;
  const bool contig = layout != nullptr;  // K/V from a contiguous cache: no slot table
  if (!q || !qo_indptr || !k_pool || !v_pool || (!contig && !req_to_token) || !seq_lens || !out || !dims)
    return ASTR_ERR_INVALID_ARG;
  astr::KvStrides ks{0, 0, 0, 0};
  if (contig) {
    const int lst = check_layout(layout, dims, &ks);
    if (lst != ASTR_OK) return lst;
  }
  const astr_attn_dims cdims = contig ? contiguous_dims(dims) : *dims;
  const astr_attn_dims* d = &cdims;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(qo_indptr, 4) || !aligned(req_to_token, 4) || !aligned(seq_lens, 4) ||
      (kv_indptr != nullptr && !aligned(kv_indptr, 4)))
    return ASTR_ERR_MISALIGNED;
  int st = check_common(d);
  if (st != ASTR_OK) return st;
  if (d->total_q < 0 || d->max_q_len < 0 || d->max_q_len > d->max_seq_len) return ASTR_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return ASTR_ERR_INVALID_ARG;
  const int G = d->num_qo_heads / d->num_kv_heads;
  if (!astr::prefill_supported(d->head_dim, G)) return ASTR_ERR_UNSUPPORTED;
  int64_t mask_req_pitch = 0, mask_row_pitch = 0;
  if (mask != nullptr && (st = check_mask(mask, d, false, &mask_req_pitch, &mask_row_pitch)) != ASTR_OK) return st;
  astr_attn_qo_layout qo{};
  if ((st = check_qo_layout(qo_layout, d, &qo)) != ASTR_OK) return st;
  if (d->batch == 0 || d->total_q == 0 || d->max_q_len == 0) return ASTR_OK;
  int dev = 0;
  if ((st = current_device(&dev)) != ASTR_OK) return st;
  astr::PrefillParams p{};
  p.q = q; p.qo_indptr = qo_indptr; p.k_pool = k_pool; p.v_pool = v_pool; p.req_to_token = req_to_token;
  p.seq_lens = seq_lens; p.out = out;
  p.r2t_stride = d->r2t_stride;
  p.batch = d->batch;
  p.num_qo_heads = d->num_qo_heads;
  p.num_kv_heads = d->num_kv_heads;
  p.head_dim = d->head_dim;
  p.num_slots = d->num_slots;
  p.total_q = d->total_q;
  const int64_t tiles = prefill_q_tiles(d);
  if (tiles > 0x7fffffffLL) return ASTR_ERR_INVALID_ARG;
  p.num_q_tiles = (int)tiles;
  int sms = 0;
  if ((st = sm_count(dev, &sms)) != ASTR_OK) return st;
  p.num_ctas = sms;
  // a plan is read only if it holds a row for every CTA of this launch
  if (d->prefill_plan != nullptr) {
    if (!aligned(d->prefill_plan, 4)) return ASTR_ERR_MISALIGNED;
    const int64_t need = astr::kPlanHeader + (int64_t)prefill_grid(d, sms) * astr::kPlanRow;
    if (d->prefill_plan_words >= need)
      p.plan = d->prefill_plan;
    else
      p.plan_rejected = 1;
  }
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.causal = (mask == nullptr) ? 1 : mask->causal;
  if (mask != nullptr && mask->mask != nullptr) {
    p.mask = mask->mask;
    p.mask_req_pitch = mask_req_pitch;
    p.mask_row_pitch = mask_row_pitch;
    p.mask_kv_pitch = mask->kv_pitch;
  }
  p.contig = contig ? 1 : 0;
  p.kv = ks;
  p.q_batch = qo.q_batch_stride; p.q_token = qo.q_token_stride; p.q_head = qo.q_head_stride;
  p.o_batch = qo.o_batch_stride; p.o_token = qo.o_token_stride; p.o_head = qo.o_head_stride;
  p.q_rows = d->max_q_len;
  p.status = d->status;
  p.wait_limit = wait_limit_of(d);
  if (astr::launch_prefill(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ASTR_ERR_LAUNCH_FAILED;
  return ASTR_OK;
}

int astr_attn_prefill_ragged(const uint16_t* q, const int32_t* qo_indptr, const uint16_t* k_pool,
                             const uint16_t* v_pool, const int32_t* req_to_token, const int32_t* seq_lens,
                             const int32_t* kv_indptr, uint16_t* out, const astr_attn_dims* d, float sm_scale,
                             void* stream) {
  return prefill_impl(q, qo_indptr, k_pool, v_pool, req_to_token, seq_lens, kv_indptr, nullptr, nullptr, nullptr,
                      out, d, sm_scale, stream);
}

int astr_attn_prefill_ragged_masked(const uint16_t* q, const int32_t* qo_indptr, const uint16_t* k_pool,
                                    const uint16_t* v_pool, const int32_t* req_to_token, const int32_t* seq_lens,
                                    const int32_t* kv_indptr, const astr_attn_mask* mask, uint16_t* out,
                                    const astr_attn_dims* d, float sm_scale, void* stream) {
  if (mask == nullptr) return ASTR_ERR_INVALID_ARG;
  return prefill_impl(q, qo_indptr, k_pool, v_pool, req_to_token, seq_lens, kv_indptr, mask, nullptr, nullptr, out,
                      d, sm_scale, stream);
}

int astr_attn_prefill_contiguous(const uint16_t* q, const int32_t* qo_indptr, const uint16_t* k_cache,
                                 const uint16_t* v_cache, const astr_attn_kv_layout* layout, const int32_t* seq_lens,
                                 const int32_t* kv_indptr, const astr_attn_mask* mask, uint16_t* out,
                                 const astr_attn_dims* d, float sm_scale, void* stream) {
  if (layout == nullptr) return ASTR_ERR_INVALID_ARG;
  return prefill_impl(q, qo_indptr, k_cache, v_cache, nullptr, seq_lens, kv_indptr, mask, layout, nullptr, out, d,
                      sm_scale, stream);
}

int astr_attn_prefill_strided(const uint16_t* q, const int32_t* qo_indptr, const uint16_t* k, const uint16_t* v,
                              const int32_t* req_to_token, const astr_attn_kv_layout* kv_layout,
                              const astr_attn_qo_layout* qo_layout, const int32_t* seq_lens, const int32_t* kv_indptr,
                              const astr_attn_mask* mask, uint16_t* out, const astr_attn_dims* d, float sm_scale,
                              void* stream) {
  return prefill_impl(q, qo_indptr, k, v, kv_layout != nullptr ? nullptr : req_to_token, seq_lens, kv_indptr, mask,
                      kv_layout, qo_layout, out, d, sm_scale, stream);
}

// Host work plan.  Items (request b, pair pr, KV head) carry the cost estimate the kernel's own
// order uses, 53 n_tiles + 13 units + 260 (about 10 ns each: a KV tile streamed, a (query tile,
// KV tile) MMA unit, and an item's fill, drain and epilogue; fitted to measured per-CTA busy
// times); longest first, each to the least-loaded CTA (ties: lowest CTA index), items of a CTA
// in the order dealt.
int astr_attn_prefill_plan(const int32_t* qo_indptr_host, const int32_t* seq_lens_host, const astr_attn_dims* d,
                           int32_t causal, int32_t num_ctas, int device, int32_t* plan, size_t plan_words,
                           size_t* words_needed) {
  if (qo_indptr_host == nullptr || seq_lens_host == nullptr || words_needed == nullptr) return ASTR_ERR_INVALID_ARG;
  int st = check_common(d);
  if (st != ASTR_OK) return st;
  if (d->total_q < 0 || d->max_q_len < 0 || num_ctas < 0) return ASTR_ERR_INVALID_ARG;
  const int G = d->num_qo_heads / d->num_kv_heads;
  if (!astr::prefill_supported(d->head_dim, G)) return ASTR_ERR_UNSUPPORTED;
  if (d->batch > 1024 || d->num_kv_heads >= 32768) return ASTR_ERR_UNSUPPORTED;  // the kernel's shared tables
  const int B = d->batch, H = d->num_kv_heads;
  const int bq2 = astr::prefill_rows_per_cta() / G, bq = bq2 / 2, bn = 64;
  for (int b = 0; b < B; ++b) {
    const int64_t ql = (int64_t)qo_indptr_host[b + 1] - qo_indptr_host[b];
    if (ql < 0 || seq_lens_host[b] < 0 || (causal && ql > seq_lens_host[b])) return ASTR_ERR_INVALID_ARG;
  }
  int sms = num_ctas;
  if (sms == 0 && (st = sm_count(device, &sms)) != ASTR_OK) return st;
  const int grid = prefill_grid(d, sms);
  struct Item {
    int64_t cost;
    int b, pair, kvh;
  };
  std::vector<Item> items;
  for (int b = 0; b < B; ++b) {
    const int q_len = qo_indptr_host[b + 1] - qo_indptr_host[b], kvn = seq_lens_host[b];
    const int cb = causal ? kvn - q_len : kvn - 1;
    const int pairs = (q_len + bq2 - 1) / bq2;
    if (pairs > 65535) return ASTR_ERR_UNSUPPORTED;
    for (int pr = 0; pr < pairs; ++pr) {
      const int first0 = pr * bq2;
      const int nq = std::min(2, (q_len - first0 + bq - 1) / bq);
      const int last = std::min(q_len, first0 + nq * bq) - 1;
      const int64_t n_tiles = (std::min<int64_t>((int64_t)cb + last + 1, kvn) + bn - 1) / bn;
      int64_t units = 0;
      for (int t = 0; t < nq; ++t)
        units += (std::min<int64_t>((int64_t)cb + std::min(q_len, first0 + (t + 1) * bq), kvn) + bn - 1) / bn;
      const int64_t cost = 53 * n_tiles + 13 * units + 260;
      for (int h = 0; h < H; ++h) items.push_back({cost, b, pr, h});
    }
  }
  std::vector<int> order(items.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return items[x].cost > items[y].cost; });
  std::vector<std::vector<int>> rows(grid > 0 ? grid : 0);
  if (grid > 0) {
    using Load = std::pair<int64_t, int>;  // (estimated load, CTA): the smallest first
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int c = 0; c < grid; ++c) heap.push({0, c});
    for (const int i : order) {
      const Load l = heap.top();
      heap.pop();
      rows[l.second].push_back(i);
      if (rows[l.second].size() > (size_t)astr::kPlanMaxItems) return ASTR_ERR_UNSUPPORTED;
      heap.push({l.first + items[i].cost, l.second});
    }
  }
  const size_t words = (size_t)astr::kPlanHeader + (size_t)(grid > 0 ? grid : 0) * astr::kPlanRow;
  *words_needed = words;
  if (plan == nullptr) return ASTR_OK;
  if (plan_words < words) return ASTR_ERR_INVALID_ARG;
  uint32_t h = 0;
  for (int i = 0; i <= B; ++i) h += astr::plan_mix((uint32_t)i, (uint32_t)qo_indptr_host[i]);
  for (int i = 0; i < B; ++i) h += astr::plan_mix(astr::kPlanSeqTag + (uint32_t)i, (uint32_t)seq_lens_host[i]);
  const int32_t header[astr::kPlanHeader] = {astr::kPlanMagic, astr::kPlanVersion, B, H, bq2, grid, (int32_t)h,
                                             causal ? 1 : 0};
  std::copy(header, header + astr::kPlanHeader, plan);
  for (int c = 0; c < grid; ++c) {
    int32_t* row = plan + astr::kPlanHeader + (size_t)c * astr::kPlanRow;
    std::fill(row, row + astr::kPlanRow, 0);
    row[0] = (int32_t)rows[c].size();
    for (size_t k = 0; k < rows[c].size(); ++k) {
      const Item& it = items[rows[c][k]];
      row[1 + 2 * k] = it.b;
      row[2 + 2 * k] = (int32_t)(((uint32_t)it.pair << 16) | (uint32_t)it.kvh);
    }
  }
  return ASTR_OK;
}

int astr_attn_kv_append(const uint16_t* k_new, const uint16_t* v_new, const int32_t* qo_indptr,
                        const int32_t* req_to_token, const int32_t* seq_lens, uint16_t* k_pool, uint16_t* v_pool,
                        const astr_attn_dims* d, void* stream) {
  if (!k_new || !v_new || !qo_indptr || !req_to_token || !seq_lens || !k_pool || !v_pool) return ASTR_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
      !aligned(qo_indptr, 4) || !aligned(req_to_token, 4) || !aligned(seq_lens, 4))
    return ASTR_ERR_MISALIGNED;
  int st = check_common(d);
  if (st != ASTR_OK) return st;
  if (d->total_q < 0) return ASTR_ERR_INVALID_ARG;
  if (d->batch == 0 || d->total_q == 0) return ASTR_OK;
  if (d->num_slots < 1) return ASTR_ERR_INVALID_ARG;
  astr::AppendParams p{};
  p.k_new = k_new; p.v_new = v_new; p.qo_indptr = qo_indptr; p.req_to_token = req_to_token;
  p.seq_lens = seq_lens; p.k_pool = k_pool; p.v_pool = v_pool;
  p.r2t_stride = d->r2t_stride;
  p.num_slots = d->num_slots;
  p.batch = d->batch;
  p.total_q = d->total_q;
  p.row_vecs = d->num_kv_heads * d->head_dim * 2 / 16;
  p.status = d->status;
  if (astr::launch_kv_append(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ASTR_ERR_LAUNCH_FAILED;
  return ASTR_OK;
}

}  // extern "C"
