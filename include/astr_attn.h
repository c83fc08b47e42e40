/*
 * astr_attn.h -- C ABI of the GB300 (sm_103a) paged-attention library libastr_attn.so.
 *
 * One hot path of an LLM serving engine: batched bf16 attention with grouped KV heads
 * over a KV-cache pool addressed through a req_to_token slot table at page_size = 1.
 * Sources (AstrAI commit log pages; "P3" = page "astrai/extension @6f67ba8",
 * "P1" = page "astrai/extension/backend/attention.py @c9ceca1",
 * "P2" = page "astrai/extension/backend @c9ceca1",
 * "P5" = page "astrai/extension/attention_backend.py @47b3ed4"):
 *   - P3, CUDA-backend commit: decode goes through attn_paged_decode and prefill through
 *     attn_prefill; req_to_token serves as the page table with one token per page.
 *   - P3, kernel-rename commit: decode is split-KV only -- every split writes an
 *     unnormalised partial (o_part) and its (m, l) pair (ml_part), and one combine kernel
 *     merges them with a log-sum-exp rescale.
 *   - P1, batched-SDPA commit: prefill/extend rows are packed flat by qo_indptr and use the
 *     per-request causal offset seq_len - q_len; masked keys get exactly zero weight.
 *   - P3, workspace and kv_indptr commits; P5, graph-workspace commit: the caller owns
 *     o_part, ml_part and out, allocated once, so the decode loop allocates nothing and
 *     can be captured into a CUDA graph; kv_indptr (exclusive prefix sum of seq_lens) is
 *     built once per step by the caller.
 *
 * Conventions for every entry point below:
 *   - Return value: ASTR_OK (0) or a negative astr_status.  Argument checks run on the
 *     host from the arguments alone; no device memory is read on the host, nothing is
 *     allocated, nothing synchronises, and no work goes to the legacy default stream
 *     unless the caller passes stream 0.  The calls are therefore capturable in a CUDA
 *     graph.  On an error status nothing has been launched.
 *   - All array pointers are DEVICE pointers owned by the caller; the library keeps no
 *     pointer after the call returns.  The dims struct is a HOST pointer read during the
 *     call only.
 *   - `stream` is a cudaStream_t passed as void*; all work is enqueued on it.
 *   - bf16 arrays hold IEEE bfloat16 bit patterns (uint16_t storage).  bf16 and fp32
 *     arrays must be 16-byte aligned; int32 arrays 4-byte aligned (ASTR_ERR_MISALIGNED).
 *   - Layouts (row-major, innermost last):
 *       q (decode)        [batch, num_qo_heads, head_dim]            bf16
 *       q (prefill)       [total_q, num_qo_heads, head_dim]          bf16
 *       k_pool, v_pool    [num_slots, num_kv_heads, head_dim]        bf16
 *       req_to_token      [batch, r2t_stride]                        int32 slot ids
 *       seq_lens          [batch]                                    int32
 *       kv_indptr         [batch + 1]   kv_indptr[b] = sum_{b'<b} seq_lens[b']   int32
 *       qo_indptr         [batch + 1]   flat query row range of request b        int32
 *       out (decode)      [batch, num_qo_heads, head_dim]            bf16
 *       out (prefill)     [total_q, num_qo_heads, head_dim]          bf16
 *       o_part            [batch, num_qo_heads, max_splits, head_dim] fp32
 *       ml_part           [batch, num_qo_heads, max_splits, 2]       fp32 (m, l)
 *   - Query head h reads KV head h / (num_qo_heads / num_kv_heads) (consecutive groups).
 *   - Caller preconditions (not checked on the host, as that would need device reads): every
 *     slot id in row b's first seq_lens[b] entries is in [0, num_slots); 0 <= seq_lens[b] <=
 *     max_seq_len <= r2t_stride; kv_indptr is the exclusive prefix sum of seq_lens;
 *     for prefill 0 <= qo_indptr[b+1] - qo_indptr[b] <= seq_lens[b], qo_indptr[0] = 0 and
 *     qo_indptr[batch] = total_q.  Violations give wrong results but no out-of-bounds access:
 *     a slot id outside the pool, or a key position past the table row, reads as a zero row
 *     (the KV append skips that token) and raises ASTR_KSTATUS_BAD_INPUT in the status word.
 *   - Errors found on the GPU (P1, input-validation bullet; P2, misaligned-input bullet: bad
 *     inputs are rejected with a clear error) cannot be returned by an asynchronous call.  When
 *     dims->status points to a device int32, the kernels OR the ASTR_KSTATUS_* bits below into
 *     it; the caller zeroes it before the call and reads it after synchronising the stream.
 *     Every wait of a kernel's pipeline is bounded (dims->wait_limit polls); a wait that runs
 *     out makes the kernel give up, write the outputs it still owns as NaN (prefill: the tiles
 *     it has not finished stay unwritten), raise ASTR_KSTATUS_TIMEOUT and return, leaving the
 *     CUDA context usable.  Outputs are valid only when the status word stays 0.
 */
#ifndef ASTR_ATTN_H
#define ASTR_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum astr_status {
  ASTR_OK = 0,
  ASTR_ERR_INVALID_ARG = -1,          /* null pointer, negative or inconsistent dims, non-finite sm_scale */
  ASTR_ERR_UNSUPPORTED = -2,          /* head_dim not 32/64/128, Hq % Hkv != 0, group size not supported */
  ASTR_ERR_MISALIGNED = -3,           /* a pointer breaks the alignment rule above */
  ASTR_ERR_WORKSPACE_TOO_SMALL = -4,  /* explicit combine layout: num_splits above max_splits */
  ASTR_ERR_LAUNCH_FAILED = -5,        /* a CUDA launch or attribute call failed (cudaGetLastError) */
  ASTR_ERR_DEVICE = -6                /* querying the current device failed */
} astr_status;

/* Status-word bits set by the kernels (see the conventions above). */
#define ASTR_KSTATUS_TIMEOUT 1    /* a pipeline wait ran out: the call's outputs are invalid */
#define ASTR_KSTATUS_BAD_INPUT 2  /* an out-of-pool slot id or a key position past r2t_stride was met */
#define ASTR_KSTATUS_SMEM 4       /* the shared-memory window was not 1024-byte aligned: no work done */
#define ASTR_KSTATUS_RANGE 8      /* prefill: an output row came out non-finite -- P V runs in fp16, so a
                                     V element beyond 65504 (or a non-finite input) makes it so */
#define ASTR_KSTATUS_PLAN 16      /* prefill: dims->prefill_plan does not match the call and was not used
                                     (the kernel ordered the work itself; the results are valid) */

/* Shapes and capacities; host struct read during the call only.  Zero-initialise it: the
 * trailing fields then take their defaults. */
typedef struct astr_attn_dims {
  int32_t batch;         /* requests in the batch (0 = nothing to do) */
  int32_t num_qo_heads;  /* Hq */
  int32_t num_kv_heads;  /* Hkv; Hq % Hkv == 0; group size Hq/Hkv in {1,2,4,8,16} */
  int32_t head_dim;      /* 32, 64 or 128 */
  int64_t num_slots;     /* rows of k_pool / v_pool */
  int32_t r2t_stride;    /* elements between consecutive req_to_token rows */
  int32_t max_seq_len;   /* host-known upper bound of seq_lens (bounds the partials per request) */
  int32_t total_q;       /* prefill: flat query rows (= qo_indptr[batch]); ignored by decode */
  int32_t max_q_len;     /* prefill: upper bound of q_len (sizes the grid); ignored by decode */
  int32_t max_splits;    /* decode: partial slots per (request, head) in o_part / ml_part (>= 1) */
  int32_t num_splits;    /* decode: key chunks per KV head; 0 = plan automatically (one wave) */
  int32_t* status;       /* optional DEVICE int32, 4-byte aligned: kernels OR ASTR_KSTATUS_* bits
                            into it (NULL = not reported); owned by the caller */
  uint32_t wait_limit;   /* polls per pipeline wait before a kernel gives up (the first poll does not
                            block, later ones may suspend the thread briefly); 0 = default (2^20) */
  const int32_t* prefill_plan;  /* prefill: optional DEVICE copy of a work plan written by
                                   astr_attn_prefill_plan for this call (NULL = the kernel orders the
                                   work itself); ignored by decode; owned by the caller */
  int64_t prefill_plan_words;   /* int32 words readable at prefill_plan (the plan's words_needed) */
  uint32_t flags;               /* ASTR_DIMS_* bits below; 0 = none */
} astr_attn_dims;

/* dims->flags.  STABLE_INDICES: req_to_token, seq_lens and kv_indptr were written before the
 * kernel that precedes this call in its stream (true for every layer of a decode step once the
 * step's tables are in place).  The decode split step then plans its chunks from them before it
 * waits for that kernel (a programmatic dependent launch), so the planning overlaps the
 * preceding kernel instead of following it; K, V and q are still read only after the wait.
 * Wrong results if the preceding kernel does write one of the three arrays. */
#define ASTR_DIMS_STABLE_INDICES 1u

/*
 * Decode split schedule (P3, shared-helpers commit: the split count is chosen per call;
 * P3, kv_indptr commit: kv_indptr is built once per step and drives it here).
 * Each request's keys are cut into slots of 32 keys from its first key (the last slot
 * possibly short); the batch's slots are laid end to end in request order (request b's first
 * slot SP_b = sum over b' < b of ceil(seq_len_b' / 32), S = SP_batch) and, for every KV head,
 * cut into `num_splits` chunks of C slots, each read by one warp pair (a producer and a
 * consumer warp; four chunks per CTA):
 *   C = max(ceil(S / num_splits), F),  F = max(1, ceil(ceil(max_seq_len / 32) / (max_splits - 1)))
 *   (C = S when max_splits == 1), so every chunk holds the same number of 32-key slots (the
 *   gather pipeline keeps a fixed number of slots in flight, so slots, not keys, set a
 *   chunk's time).
 * Request b overlaps chunks SP_b / C .. (SP_b + ceil(seq_len_b / 32) - 1) / C; the piece of it
 * in chunk c becomes partial slot c - SP_b / C of (b, h), and the floor F keeps the count at
 * or below max_splits (a request longer than max_seq_len keys would need more; its pieces
 * past max_splits are not written, which leaves its output wrong but memory intact).
 * This call returns num_splits as planned for `device`: the
 * forced dims->num_splits if > 0, else 4 * ceil(#SMs / Hkv) (one persistent CTA per SM).
 * Depends only on host-known values, never on the contents of seq_lens.
 * Errors: INVALID_ARG (null, bad dims), DEVICE (device query failed).
 */
int astr_attn_decode_num_splits(const astr_attn_dims* dims, int device, int* num_splits);

/*
 * Bytes the caller must provide for o_part and ml_part: batch * Hq * max_splits *
 * head_dim * 4 and batch * Hq * max_splits * 2 * 4.  Errors: INVALID_ARG.
 */
int astr_attn_decode_workspace_bytes(const astr_attn_dims* dims, size_t* o_part_bytes, size_t* ml_part_bytes);

/*
 * Split-KV paged decode (one query row per request).
 *   out[b, h, :] = sum_{j < seq_lens[b]} softmax_j(sm_scale * <q[b,h], K_j>) V_j,
 *   K_j, V_j = pool[req_to_token[b * r2t_stride + j], h / G, :].
 * Launches the split kernel (schedule as for astr_attn_decode_num_splits; each chunk serves
 * all G query heads of its KV head from one K/V load; a request that lies entirely inside
 * one chunk has its output written directly; every other request piece writes its partial
 * slot: o_part unnormalised, ml_part = (max scaled logit in natural-log units, sum of
 * exponentials)) and then the combine kernel for the requests that span several chunks.
 * Slots that no piece maps to are left untouched.  seq_lens[b] = 0 gives a zero output
 * row.  Deterministic for fixed dims (no atomics).
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, DEVICE, LAUNCH_FAILED.
 */
int astr_attn_paged_decode(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                           const int32_t* req_to_token, const int32_t* seq_lens, const int32_t* kv_indptr,
                           float* o_part, float* ml_part, uint16_t* out, const astr_attn_dims* dims,
                           float sm_scale, void* stream);

/*
 * The split step alone: the first of the two launches of astr_attn_paged_decode, except that
 * every request piece (also single-chunk requests) writes its partial slot; nothing else is
 * written.  astr_attn_decode_combine with the same kv_indptr then produces `out`.  Same
 * arguments, rules and errors as astr_attn_paged_decode minus `out`.
 */
int astr_attn_decode_split(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                           const int32_t* req_to_token, const int32_t* seq_lens, const int32_t* kv_indptr,
                           float* o_part, float* ml_part, const astr_attn_dims* dims, float sm_scale, void* stream);

/*
 * The combine step alone (P3, kernel-rename commit: the log-sum-exp merge shared by the
 * split paths): for each (b, h) over its S partial slots,
 *   M = max_s m_s,  w_s = exp(m_s - M),  out = (sum_s w_s o_s) / (sum_s w_s l_s)  -> bf16.
 * With kv_indptr given, S is the number of chunks request b overlaps under the schedule
 * of astr_attn_decode_num_splits (the layout astr_attn_decode_split writes).  With
 * kv_indptr NULL, every row holds S = dims->num_splits slots (1 <= S <= max_splits, else
 * INVALID_ARG / WORKSPACE_TOO_SMALL).  A row with S = 0 or all m_s = -inf is written as
 * zeros.  seq_lens is not read (may be NULL).  Errors as astr_attn_paged_decode.
 */
int astr_attn_decode_combine(const float* o_part, const float* ml_part, const int32_t* seq_lens,
                             const int32_t* kv_indptr, uint16_t* out, const astr_attn_dims* dims, void* stream);

/*
 * Work plan for the prefill calls (optional: it orders the work and changes no result; not a
 * step of the pages' method).  Without a plan, every CTA of a prefill launch first derives the
 * work order from qo_indptr and seq_lens in shared memory (a few microseconds of every call).
 * A plan is made once on the host, from host copies of the same two arrays, and serves every
 * call of the batch (one per layer): it holds each CTA's work items (KV head x pair of query
 * tiles), dealt longest-estimated-first to the least-loaded CTA.  The kernel checks the plan
 * against the call -- batch, num_kv_heads, group size, grid, causal flag and a checksum of
 * qo_indptr and seq_lens -- and ignores one that does not match (ASTR_KSTATUS_PLAN).
 *   qo_indptr_host [batch + 1], seq_lens_host [batch]: HOST int32 copies of the call's arrays.
 *   dims: the call's dims (batch, heads, head_dim, total_q and max_q_len as the call passes them).
 *   causal: 1 for astr_attn_prefill_ragged / _contiguous / _strided without a mask, else the
 *     mask's causal flag.
 *   num_ctas: CTAs the call launches on; 0 = the SM count of `device` (what the call uses).
 *   plan: HOST buffer of plan_words int32 words to write (the caller copies it to the device and
 *     sets dims->prefill_plan and dims->prefill_plan_words); NULL = only report the size.
 *   *words_needed: the plan's size in int32 words.
 * Returns OK; INVALID_ARG (a null pointer, bad dims, a negative q_len or seq_len, q_len above
 * seq_len for a causal call, plan_words below words_needed); UNSUPPORTED (head_dim / group size
 * as for the prefill calls, more than 1024 requests, or more than 128 items on one CTA: the
 * kernel then deals the items in their natural order and no plan applies); DEVICE.
 */
int astr_attn_prefill_plan(const int32_t* qo_indptr_host, const int32_t* seq_lens_host, const astr_attn_dims* dims,
                           int32_t causal, int32_t num_ctas, int device, int32_t* plan, size_t plan_words,
                           size_t* words_needed);

/*
 * Ragged packed prefill/extend over the same pool (P1, batched-SDPA commit; P3,
 * CUDA-backend and unified-causal-offset commits).  For request b with q_len_b =
 * qo_indptr[b+1] - qo_indptr[b] and causal offset c_b = seq_lens[b] - q_len_b, flat row
 * r = qo_indptr[b] + i (0 <= i < q_len_b) and query head h:
 *   out[r, h, :] = sum_{j <= c_b + i} softmax_j(sm_scale * <q[r,h], K_j>) V_j.
 * The new tokens' K/V must already be in the pool (positions c_b .. seq_len_b - 1).
 * Requests with q_len = 0 write nothing.  kv_indptr is accepted for interface symmetry
 * with decode and is not read (may be NULL).  Tensor cores (tcgen05, accumulators in
 * tensor memory) compute Q K^T and P V.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, DEVICE, LAUNCH_FAILED.
 */
int astr_attn_prefill_ragged(const uint16_t* q, const int32_t* qo_indptr, const uint16_t* k_pool,
                             const uint16_t* v_pool, const int32_t* req_to_token, const int32_t* seq_lens,
                             const int32_t* kv_indptr, uint16_t* out, const astr_attn_dims* dims, float sm_scale,
                             void* stream);

/*
 * Explicit attention mask (P3, prefill-mask commit: 2-D [batch, kv_len] and 3-D
 * [batch, q_len, kv_len] masks, causal and mask may coexist; unified-causal-offset commit:
 * the causal offset can be switched off).  Host struct read during the call only.  Key j of
 * request b is visible to its local query row i iff j < seq_lens[b], the causal rule holds
 * (causal = 1: j <= seq_lens[b] - q_len_b + i; causal = 0: always) and, when `mask` is not
 * NULL, its byte for (b, i, j) is nonzero:
 *   dims = 2:  mask[b * kv_pitch + j]                      (the same for every row i)
 *   dims = 3:  mask[(b * q_pitch + i) * kv_pitch + j]
 * A query row with no visible key is written as zeros.  Decode has one row per request
 * (i = 0) and no causal rule (its row sees every key).
 */
typedef struct astr_attn_mask {
  const uint8_t* mask;   /* DEVICE bytes, nonzero = visible, 16-byte aligned; NULL = no explicit mask */
  int32_t dims;          /* 2 or 3 (read only when mask is not NULL) */
  int32_t kv_pitch;      /* bytes per mask row: a multiple of 16, >= max_seq_len */
  int32_t q_pitch;       /* dims = 3: rows per request, >= max_q_len for prefill, >= 1 for decode */
  int32_t causal;        /* prefill: 1 = causal offset seq_len - q_len, 0 = off; decode ignores it */
} astr_attn_mask;

/*
 * astr_attn_paged_decode with an explicit mask (struct above; mask->causal is not read).  The
 * split kernel reads each 32-key slot's mask bytes next to its slot ids; masked keys get
 * exactly zero weight.  Same arguments, rules and errors as astr_attn_paged_decode, plus
 * INVALID_ARG for a NULL `mask` struct or bad dims / pitches and MISALIGNED for mask->mask.
 */
int astr_attn_paged_decode_masked(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                                  const int32_t* req_to_token, const int32_t* seq_lens, const int32_t* kv_indptr,
                                  const astr_attn_mask* mask, float* o_part, float* ml_part, uint16_t* out,
                                  const astr_attn_dims* dims, float sm_scale, void* stream);

/*
 * astr_attn_prefill_ragged with an explicit mask and/or the causal offset switched off
 * (struct above).  mask->mask = NULL with causal = 1 is astr_attn_prefill_ragged itself; with
 * causal = 0 every row attends over all seq_lens[b] keys of its request.  Each softmax thread
 * reads its row's 64 mask bytes per key tile while the tile's scores are computed.  Same
 * arguments, rules and errors as astr_attn_prefill_ragged, plus INVALID_ARG for a NULL `mask`
 * struct, bad dims / pitches or causal not 0/1, and MISALIGNED for mask->mask.
 */
int astr_attn_prefill_ragged_masked(const uint16_t* q, const int32_t* qo_indptr, const uint16_t* k_pool,
                                    const uint16_t* v_pool, const int32_t* req_to_token, const int32_t* seq_lens,
                                    const int32_t* kv_indptr, const astr_attn_mask* mask, uint16_t* out,
                                    const astr_attn_dims* dims, float sm_scale, void* stream);

/*
 * Contiguous K/V cache layout (P3, stride-addressing and layout commits: Q/KV/O addressed
 * through strides so "bhld" and "blhd" caches work without copies).  Host struct read during
 * the call only.  Element e of key position j, KV head h, request b of a contiguous cache sits
 * at cache[b * batch_stride + j * token_stride + h * head_stride + e]; all strides are in
 * elements, non-negative and multiples of 8 (16-byte rows).  For a cache of L positions:
 *   bhld  [batch, Hkv, L, head_dim]:  batch_stride = Hkv*L*d, head_stride = L*d, token_stride = d
 *   blhd  [batch, L, Hkv, head_dim]:  batch_stride = L*Hkv*d, token_stride = Hkv*d, head_stride = d
 * Positions 0 .. dims->max_seq_len - 1 of every request must lie inside the cache.
 */
typedef struct astr_attn_kv_layout {
  int64_t batch_stride;
  int64_t token_stride;
  int64_t head_stride;
} astr_attn_kv_layout;

/*
 * Decode over a contiguous K/V cache: astr_attn_paged_decode (and, with `mask` not NULL,
 * astr_attn_paged_decode_masked) with key j of request b read from the cache rows of layout
 * `layout` instead of pool[req_to_token[b][j]].  dims->r2t_stride and num_slots are not read;
 * dims->max_seq_len bounds the positions read (a key at or past it reads as zeros).  Same
 * schedule, partial layout, rules and errors otherwise, plus INVALID_ARG for a NULL layout or
 * negative strides and MISALIGNED for strides that are not multiples of 8.
 */
int astr_attn_decode_contiguous(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                const astr_attn_kv_layout* layout, const int32_t* seq_lens, const int32_t* kv_indptr,
                                const astr_attn_mask* mask, float* o_part, float* ml_part, uint16_t* out,
                                const astr_attn_dims* dims, float sm_scale, void* stream);

/*
 * Ragged prefill over a contiguous K/V cache: astr_attn_prefill_ragged (with `mask` not NULL,
 * astr_attn_prefill_ragged_masked, causal switch included) with key j of request b read from
 * the cache rows of `layout`.  Query rows and outputs keep the packed [total_q, Hq, head_dim]
 * layout.  dims->r2t_stride and num_slots are not read; dims->max_seq_len bounds the positions
 * read.  Errors as astr_attn_decode_contiguous.
 */
int astr_attn_prefill_contiguous(const uint16_t* q, const int32_t* qo_indptr, const uint16_t* k_cache,
                                 const uint16_t* v_cache, const astr_attn_kv_layout* layout, const int32_t* seq_lens,
                                 const int32_t* kv_indptr, const astr_attn_mask* mask, uint16_t* out,
                                 const astr_attn_dims* dims, float sm_scale, void* stream);

/*
 * Query and output addressed by strides (P3, stride-addressing and layout commits: Q, KV and O
 * addressed through strides, so "bhld" / "blhd" tensors work without copies).  Host struct
 * read during the call only.  Strides are in elements, non-negative multiples of 8 (16-byte
 * rows); head_dim is contiguous.  Element e of query head h in request-local query row i of
 * request b sits at
 *   q_batch_stride == 0 (rows packed flat):  q[(r0_b + i) * q_token_stride + h * q_head_stride + e],
 *                                            r0_b = qo_indptr[b] for prefill, b for decode;
 *   q_batch_stride  > 0 (rows padded per request):
 *                                            q[b * q_batch_stride + i * q_token_stride + h * q_head_stride + e],
 * and the output element likewise with the o_* strides.  Decode has one row per request (i = 0).
 *   packed [rows, Hq, d]:        {0, Hq*d, d} (the layout of the entry points above)
 *   padded bhld [B, Hq, L, d]:   {Hq*L*d, d, L*d}        padded blhd [B, L, Hq, d]: {L*Hq*d, Hq*d, d}
 * A padded prefill tensor holds at least dims->max_q_len positions per request.
 */
typedef struct astr_attn_qo_layout {
  int64_t q_batch_stride, q_token_stride, q_head_stride;
  int64_t o_batch_stride, o_token_stride, o_head_stride;
} astr_attn_qo_layout;

/*
 * Decode with every layout choice at once: K/V from the paged pool through req_to_token
 * (kv_layout NULL) or from a contiguous cache (kv_layout given; req_to_token not read), query
 * and output by the strides of qo_layout (NULL: packed [B, Hq, d]), an optional explicit mask
 * (NULL: none).  The same computation, schedule, partial layout, rules and errors as
 * astr_attn_paged_decode / _masked / astr_attn_decode_contiguous, plus INVALID_ARG for
 * negative strides and MISALIGNED for strides that are not multiples of 8.
 */
int astr_attn_decode_strided(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* req_to_token,
                             const astr_attn_kv_layout* kv_layout, const astr_attn_qo_layout* qo_layout,
                             const int32_t* seq_lens, const int32_t* kv_indptr, const astr_attn_mask* mask,
                             float* o_part, float* ml_part, uint16_t* out, const astr_attn_dims* dims, float sm_scale,
                             void* stream);

/*
 * Ragged prefill with every layout choice at once (as astr_attn_decode_strided): K/V paged or
 * contiguous, query rows and outputs by the strides of qo_layout (NULL: packed [total_q, Hq, d];
 * padded tensors are addressed by (request, local row), packed ones by qo_indptr[b] + row),
 * optional mask and causal switch.  qo_indptr always gives each request's q_len.  Only the rows
 * of each request's q_len are written.  Errors as astr_attn_decode_strided.
 */
int astr_attn_prefill_strided(const uint16_t* q, const int32_t* qo_indptr, const uint16_t* k, const uint16_t* v,
                              const int32_t* req_to_token, const astr_attn_kv_layout* kv_layout,
                              const astr_attn_qo_layout* qo_layout, const int32_t* seq_lens, const int32_t* kv_indptr,
                              const astr_attn_mask* mask, uint16_t* out, const astr_attn_dims* dims, float sm_scale,
                              void* stream);

/*
 * Paged decode that allocates nothing (no counterpart in the source pages; this is a
 * service of this library).  Same computation, arguments, rules and errors as
 * astr_attn_paged_decode minus o_part / ml_part: the split-KV partials go to a 16 MiB
 * array compiled into the library instead of caller memory.  It is for callers that
 * cannot hand the library a workspace -- an operator inside an inference runtime whose
 * memory planner owns all device memory and forwards only inputs and outputs, or a
 * process that must not grow device memory after start-up.  Every GPU that loads the
 * library holds the array until the process exits.
 *   - Size limit: batch * Hq * max_splits * (head_dim + 2) * 4 bytes (plus alignment
 *     padding of at most 255 bytes) must fit in 16 MiB, else WORKSPACE_TOO_SMALL before
 *     anything is launched.
 *   - The first call on a device resolves the array's device address with that device
 *     current; make that first call before any stream capture.
 *   - All calls share the one array: calls that overlap on the GPU race and must be
 *     serialised by the caller.  The array keeps the previous call's contents; nothing in
 *     it needs to start at zero.
 *   - Calls no cudaMalloc / cudaFree or any allocating routine.
 */
int astr_attn_paged_decode_noalloc(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                                   const int32_t* req_to_token, const int32_t* seq_lens, const int32_t* kv_indptr,
                                   uint16_t* out, const astr_attn_dims* dims, float sm_scale, void* stream);

/*
 * KV append: write the new tokens' K and V into their pool slots (P5, write-then-gather
 * helper commit: the new K/V go into the pool before attention gathers from it).  Request b
 * has q_len_b = qo_indptr[b+1] - qo_indptr[b] new tokens, which are its key positions
 * c_b .. seq_lens[b] - 1 (c_b = seq_lens[b] - q_len_b, the prefill's causal offset; seq_lens
 * already counts them).  For flat row r = qo_indptr[b] + i:
 *   slot = req_to_token[b * r2t_stride + c_b + i],
 *   k_pool[slot, :, :] = k_new[r, :, :],  v_pool[slot, :, :] = v_new[r, :, :]   (bit copies).
 * Decode appends one token per request: qo_indptr[b] = b, the current token being the last
 * key (position seq_lens[b] - 1).  Call it before astr_attn_prefill_ragged /
 * astr_attn_paged_decode on the same stream.
 *   - k_new, v_new: [total_q, num_kv_heads, head_dim] bf16 (dims->total_q rows), device,
 *     16-byte aligned, not overlapping the pools.  k_pool / v_pool are written in place.
 *   - Only the new tokens' slots change.  Distinct new tokens must map to distinct slots
 *     (else which write lands is undefined).  A slot id outside [0, num_slots), or a
 *     position outside the table row, is skipped (nothing written for that token).
 *   - Reads dims->batch, num_kv_heads, head_dim, num_slots, r2t_stride, total_q (and checks
 *     the shape fields as the attention calls do); batch = 0 or total_q = 0 does nothing.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, LAUNCH_FAILED.
 */
int astr_attn_kv_append(const uint16_t* k_new, const uint16_t* v_new, const int32_t* qo_indptr,
                        const int32_t* req_to_token, const int32_t* seq_lens, uint16_t* k_pool, uint16_t* v_pool,
                        const astr_attn_dims* dims, void* stream);

/* Static description of a status code (never NULL). */
const char* astr_attn_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int astr_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ASTR_ATTN_H */
