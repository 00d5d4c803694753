/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged-KV grouped-query attention library.
 *
 * Operations (cited by page title and section):
 *   - decode, split-KV: "vllm/attention/ops/triton_decode_attention.py",
 *     _fwd_grouped_kernel_stage1 (per-split partial output and log-sum-exp)
 *     and _fwd_kernel_stage2 (merge of the splits by LSE);
 *   - prefix-prefill / extend: "vllm/attention/ops/prefix_prefill.py",
 *     context_attention_fwd / _fwd_kernel (new queries see the cached context
 *     unmasked and the new tokens causally);
 *   - sinks, window_left, fp8 descales, plan/bind/run split and the
 *     caller-owned scratch workspace: "vllm/v1/attention/backends/b12x",
 *     B12xPagedAttentionImpl (__init__, forward, _prepare_fp8_descales).
 *
 * What every call computes, for request b, query row at sequence position
 * pos_q, q head h and kv head g = h / (Hq / Hkv):
 *   J      = { j : 0 <= j <= pos_q, and (window <= 0 or pos_q - j < window) }
 *   K_j    = k_cache[block_table[b][j / page_size]][j % page_size][g][:]
 *   s_j    = scale * (q . K_j);  s_j = cap * tanh(s_j / cap) when soft_cap > 0
 *   m      = max(max_J s_j, sink_h)            (sink only when sinks != NULL)
 *   Z      = sum_J exp(s_j - m) + exp(sink_h - m)
 *   out    = sum_J exp(s_j - m) V_j / Z        (bf16)
 *   lse    = m + ln Z                          (fp32, natural log)
 * Decode has one query per request at pos_q = seq_lens[b] - 1.  Extend packs
 * the new queries of request b in rows [query_start_loc[b], query_start_loc[b+1]),
 * row i of the request at pos_q = ctx_b + i with
 * ctx_b = seq_lens[b] - (query_start_loc[b+1] - query_start_loc[b]); the new
 * tokens' K/V must already be in the pages.
 * fp8 KV: element value = bf16( float(e4m3) * k_scale ) (same for V with
 * v_scale; per-request scales k_scales[b] / v_scales[b] replace them when
 * given), as the prefix-prefill page dequantises.
 *
 * Conventions
 *   - Pointers named "device" must be device memory of the current device;
 *     the caller owns every buffer, including the scratch workspace.  No call
 *     allocates device memory.
 *   - Calls enqueue work on `stream` (a cudaStream_t, NULL = legacy default
 *     stream) and return without synchronising.
 *   - Strides are in ELEMENTS; the innermost (head_dim) dimension is
 *     contiguous.  KV base pointers and the byte strides of pages, slots and
 *     kv heads must be multiples of 16 bytes (they feed TMA tensor maps).
 *   - Metadata (block_table, seq_lens, query_start_loc) is int32, in device
 *     memory.  Block-table entries past ceil(seq_lens[b] / page_size) are
 *     never read.
 *   - Errors: no exceptions cross the ABI.  Argument errors return
 *     PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED before anything is enqueued.
 *     Kernels never trap: a bounded wait that expires sets an error word in
 *     the scratch header, which pa_check reports as PA_ERR_DEVICE.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,       /* null pointer, negative size, inconsistent shape */
  PA_ERR_UNSUPPORTED = 2,       /* valid but outside what the kernels implement */
  PA_ERR_SCRATCH_TOO_SMALL = 3, /* scratch_bytes < plan->scratch_bytes */
  PA_ERR_CUDA = 4,              /* a CUDA runtime/driver call failed */
  PA_ERR_DEVICE = 5             /* a kernel reported an error in the scratch header */
} pa_status;

/* Bits of the device error code that pa_check returns in *device_code.  A
 * kernel ORs one into the scratch header when it meets the condition; it never
 * traps.  Only an expired wait makes the other CTAs of the call give up; after
 * any other bit the rest of the call still runs and writes its results. */
typedef enum {
  PA_DEVICE_WAIT_TIMEOUT = 1,   /* a bounded device-side wait ran out of time */
  PA_DEVICE_WORK_OVERFLOW = 2,  /* a work list or block-table slice exceeded its planned capacity */
  PA_DEVICE_CAPACITY = 4,       /* a length or query packing beyond what the plan allows; that
                                   request's rows are left untouched */
  PA_DEVICE_PAGE_ID = 8         /* a block-table entry of a page holding attended keys lies outside
                                   [0, num_pages) (or an append slot's page does); that page reads
                                   as zeros (is not written), every other page is unaffected */
} pa_device_code;

typedef enum { PA_KV_BF16 = 0, PA_KV_FP8_E4M3 = 1 } pa_kv_dtype;
/* VERIFY: extend where every request brings the same small number q_len of
 * new tokens (1 + speculative tokens) over a long context; planned and run
 * like decode (split-KV + merge), entered through pa_extend. */
typedef enum { PA_MODE_DECODE = 0, PA_MODE_EXTEND = 1, PA_MODE_VERIFY = 2 } pa_mode;

/* Static problem description (capacities, never live lengths, except for the
 * optional host seq_lens hint given to pa_plan). */
typedef struct {
  int32_t mode;               /* pa_mode */
  int32_t num_q_heads;        /* Hq; Hq % Hkv == 0 and Hq / Hkv <= 128 */
  int32_t num_kv_heads;       /* Hkv */
  int32_t head_dim;           /* D in {64, 128, 256} */
  int32_t page_size;          /* ps in {16, 32, 64} */
  int32_t kv_dtype;           /* pa_kv_dtype */
  int32_t max_batch;          /* capacity: requests per call */
  int32_t max_pages_per_seq;  /* capacity: block-table row width */
  int32_t max_total_q;        /* extend: capacity of packed query rows */
  int32_t window;             /* sliding window W; 0 = off */
  int32_t has_sinks;          /* 1: calls pass a [Hq] fp32 sink logit array */
  float soft_cap;             /* 0 = off; else s = cap * tanh(s / cap) */
  int32_t num_splits;         /* decode: 0 = planner's choice, >0 = max KV splits per request */
  int32_t num_sms;            /* SMs to plan for; 0 = query the current device */
  int32_t q_len;              /* verify: new tokens per request (q_len * Hq/Hkv <= 16); else ignored */
} pa_shape;

/* Plan produced by pa_plan; plain data, may be copied.  Fields other than
 * scratch_bytes are the planner's launch choices, exposed for inspection. */
typedef struct {
  pa_shape shape;
  int32_t tile_tokens;        /* keys per pipeline stage */
  int32_t split_tiles;        /* decode: stages per KV split (0 when num_splits is fixed) */
  int32_t max_splits;         /* decode: largest split count a request can get */
  int32_t stages;             /* pipeline depth per warp */
  int32_t warps;              /* compute warps per CTA */
  int32_t bt_cache;           /* block-table entries staged in shared memory per CTA */
  int32_t smem_bytes;         /* dynamic shared memory per CTA */
  int32_t grid[3];            /* main kernel grid */
  int64_t scratch_bytes;      /* device scratch the calls need (>= 65536, the header) */
  int32_t launches;           /* kernel launches one call makes */
  int32_t kv_copy;            /* extend over an e4m3 cache: 1 = each call first dequantises the
                                 pages it reads, once, into a bf16 copy inside the scratch
                                 workspace and attends over the copy (chosen while the copy
                                 for max_batch x max_pages_per_seq pages fits in 2 GiB);
                                 0 = every attention CTA dequantises its tiles in shared memory */
  int32_t split_merge;        /* decode / verify with max_splits > 1: 1 = the split that finishes
                                 last for a (request, kv head) merges that pair's splits, counted
                                 by arrival counters in the scratch header (one launch; chosen
                                 while max_batch x Hkv x head groups <= 16320); 0 = a merge
                                 kernel follows */
  int32_t reserved[5];
} pa_plan_t;

/* Plan a decode or extend call from capacities.  host_seq_lens (host memory,
 * `batch` entries, may be NULL) lets the decode planner size KV splits to the
 * actual lengths; without it the plan assumes every request is at capacity.
 * Pure host code: no CUDA call is made unless shape->num_sms == 0.
 * Returns PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED for shapes it cannot run. */
pa_status pa_plan(const pa_shape* shape, const int32_t* host_seq_lens, int32_t batch,
                  pa_plan_t* plan);

/* Split-KV paged decode: stage 1 (per-split partial output and LSE, written to
 * the scratch workspace) followed by the LSE merge (final out / lse).  When
 * the plan gives every request a single split (plan->max_splits == 1) stage 1
 * writes out / lse itself; with plan->split_merge the stage-1 CTA that
 * finishes last for a (request, kv head) merges its splits; otherwise a merge
 * kernel follows (plan->launches).
 *   q            device bf16, [batch, Hq, D], strides q_stride_tok / q_stride_head
 *   k_cache, v_cache  device, [num_pages, page_size, Hkv, D] bf16 or e4m3 bytes,
 *                strides kv_stride_page / kv_stride_tok / kv_stride_head
 *                (both caches share the strides; K and V may be the two halves
 *                of one [num_pages, 2, page_size, Hkv*D] allocation)
 *   block_table  device int32 [batch, bt_stride] (bt_stride >= pages used)
 *   seq_lens     device int32 [batch]; keys per request (>= 0)
 *   scale        softmax scale applied to q.K before the soft-cap
 *   sinks        device fp32 [Hq] when plan->shape.has_sinks, else NULL
 *   k_scale, v_scale  per-tensor fp8 scales (ignored for bf16 KV)
 *   k_scales, v_scales  device fp32 [batch] per-request fp8 descales, or NULL;
 *                each one given replaces its per-tensor scale (request b's
 *                pages dequantise as bf16(float(code) * k_scales[b])), as the
 *                b12x backend page's descales may be one value per request
 *                ("vllm/v1/attention/backends/b12x", _prepare_fp8_descales);
 *                ignored for bf16 KV
 *   out          device bf16 [batch, Hq, D], strides out_stride_tok / out_stride_head
 *   lse          device fp32 [batch, Hq] contiguous, or NULL
 *   scratch      device, >= plan->scratch_bytes bytes, 256-byte aligned; its
 *                first 64 KiB are the header (error word and split-arrival
 *                counters; zero it once with pa_scratch_init).  The rest is
 *                overwritten by every call.
 * Concurrent calls must not share a scratch buffer. */
pa_status pa_decode(const pa_plan_t* plan,
                    const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                    const void* k_cache, const void* v_cache,
                    int64_t kv_stride_page, int64_t kv_stride_tok, int64_t kv_stride_head,
                    int32_t num_pages,
                    const int32_t* block_table, int64_t bt_stride,
                    const int32_t* seq_lens, int32_t batch,
                    float scale, const float* sinks, float k_scale, float v_scale,
                    const float* k_scales, const float* v_scales,
                    void* out, int64_t out_stride_tok, int64_t out_stride_head,
                    float* lse,
                    void* scratch, int64_t scratch_bytes, void* stream);

/* pa_decode without a caller-provided workspace.  The source pages have no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * device memory for a scratch buffer -- for example a plugin or host runtime
 * with no device allocator of its own, a process whose memory pool already
 * owns the whole GPU, or code that must never allocate so that its latency
 * stays fixed.  Arguments and results are those of pa_decode, minus scratch
 * and the per-request scales (per-tensor k_scale / v_scale only).
 *   - The workspace is a 16 MiB array inside the library's device image,
 *     present on every GPU that loads the library until the process exits.
 *     Plans whose scratch_bytes exceed 16 MiB return PA_ERR_SCRATCH_TOO_SMALL.
 *   - Every call made outside a stream capture looks up the array's device
 *     address on the current device (a runtime query, no allocation); a call
 *     made while its stream is being captured reuses the address the last
 *     uncaptured call on that device found, so make the first call on each
 *     device before any stream capture (without one, a captured call returns
 *     PA_ERR_CUDA).  Nothing is allocated, by this call or any later one.
 *   - Every call on a device shares the one array and clears its error header
 *     first; calls that overlap on the GPU race on it, so the caller must
 *     serialise them.
 *   - Device-side errors are not reported: the header that records them is
 *     cleared by the next call and no call reads it.  In particular a request
 *     whose seq_lens entry needs more KV splits than the plan allows (a length
 *     beyond the capacity the plan was made for) is skipped on the device and
 *     its rows of out and lse are LEFT UNTOUCHED, and the call still returns
 *     PA_OK.  Callers that cannot rule this out on the host should use
 *     pa_decode with pa_check, which reports it. */
pa_status pa_decode_static_scratch(const pa_plan_t* plan,
                                   const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                                   const void* k_cache, const void* v_cache,
                                   int64_t kv_stride_page, int64_t kv_stride_tok, int64_t kv_stride_head,
                                   int32_t num_pages,
                                   const int32_t* block_table, int64_t bt_stride,
                                   const int32_t* seq_lens, int32_t batch,
                                   float scale, const float* sinks, float k_scale, float v_scale,
                                   void* out, int64_t out_stride_tok, int64_t out_stride_head,
                                   float* lse, void* stream);

/* Prefix-prefill / extend over the paged cache (all keys, cached and new,
 * are read from the pages).
 *   q               device bf16 [total_q, Hq, D] (strides as for decode)
 *   seq_lens        device int32 [batch]: cached + new tokens per request
 *   query_start_loc device int32 [batch + 1], query_start_loc[0] = 0,
 *                   non-decreasing, query_start_loc[batch] = total_q
 *   out             device bf16 [total_q, Hq, D]; lse device fp32 [total_q, Hq] or NULL
 * A scheduler kernel builds the (request, kv head, query tile) work list in
 * the scratch workspace from the device metadata, longest first; the
 * attention kernel takes items from that list.  total_q must not exceed
 * plan->shape.max_total_q.  With a PA_MODE_VERIFY plan every request must
 * hold exactly plan->shape.q_len rows (query_start_loc[b] = b * q_len,
 * total_q = batch * q_len); the call runs the split-KV kernels and a bad
 * packing sets the device error word.  With an e4m3 cache and plan->kv_copy
 * the call first writes bf16(float(code) * scale) of every page a request
 * reads into the scratch workspace (pages before the sliding window are
 * skipped) and attends over that copy; the values the attention sees are the
 * same either way.  The work list and the copy are laid out from the plan's
 * shape: a plan whose grid no longer matches that shape returns
 * PA_ERR_INVALID_ARG, and a scratch smaller than the layout (the copy
 * included) PA_ERR_SCRATCH_TOO_SMALL, before anything is enqueued.  Other
 * arguments as for pa_decode. */
pa_status pa_extend(const pa_plan_t* plan,
                    const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                    const void* k_cache, const void* v_cache,
                    int64_t kv_stride_page, int64_t kv_stride_tok, int64_t kv_stride_head,
                    int32_t num_pages,
                    const int32_t* block_table, int64_t bt_stride,
                    const int32_t* seq_lens, const int32_t* query_start_loc,
                    int32_t batch, int32_t total_q,
                    float scale, const float* sinks, float k_scale, float v_scale,
                    const float* k_scales, const float* v_scales,
                    void* out, int64_t out_stride_tok, int64_t out_stride_head,
                    float* lse,
                    void* scratch, int64_t scratch_bytes, void* stream);

/* Append new tokens' K and V to the paged cache -- the write side the
 * attention calls read ("vllm/v1/attention/backends/b12x",
 * do_kv_cache_update, which passes these arguments to reshape_and_cache_flash).
 *   k_new, v_new   device bf16 [num_tokens, Hkv, head_dim], strides
 *                  new_stride_tok / new_stride_head (16-byte aligned rows)
 *   k_cache, v_cache, kv strides, num_pages, page_size   as for pa_decode
 *   slot_mapping   device int64 [num_tokens]: token t goes to page
 *                  slot / page_size, slot slot % page_size; negative = padding, skipped
 *   kv_dtype       PA_KV_BF16 stores the values; PA_KV_FP8_E4M3 stores
 *                  e4m3(x / scale) (round to nearest even, saturated to +-448)
 *   scratch        optional (may be NULL): a scratch buffer whose error header
 *                  records slots outside the pool (those tokens are not written)
 * One call moves fewer than 2^31 eight-element vectors (num_tokens * Hkv *
 * head_dim / 8), else PA_ERR_UNSUPPORTED.
 * Asynchronous on `stream`; one kernel launch. */
pa_status pa_append_kv(const void* k_new, const void* v_new, int64_t new_stride_tok, int64_t new_stride_head,
                       void* k_cache, void* v_cache,
                       int64_t kv_stride_page, int64_t kv_stride_tok, int64_t kv_stride_head,
                       int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim,
                       int32_t kv_dtype, const int64_t* slot_mapping, int32_t num_tokens,
                       float k_scale, float v_scale, void* scratch, void* stream);

/* Zero the 64 KiB header at the start of a scratch buffer (enqueued on
 * `stream`): the error word, and the split-arrival counters that decode
 * calls leave at zero when they finish.  Call once after allocating the
 * scratch. */
pa_status pa_scratch_init(void* scratch, void* stream);

/* Synchronise `stream`, read the scratch error word and, if it is set,
 * zero the whole header (a failed call can leave arrival counters behind:
 * call pa_check, or pa_scratch_init, before reusing a scratch buffer after
 * a device error).  Returns
 * PA_OK, PA_ERR_DEVICE (a kernel reported an error: a bounded wait expired,
 * a length or packing beyond what the plan allows, a work list over its
 * capacity, a block-table entry or append slot outside the pool; the
 * header's pa_device_code bits are stored in *device_code when non-NULL)
 * or PA_ERR_CUDA. */
pa_status pa_check(void* scratch, void* stream, uint32_t* device_code);

/* Test hook for the device-side error reporting; callers of the attention
 * calls never need it.  Enqueues one single-warp kernel that waits, through
 * one of the bounded wait helpers the library's kernels use, on an mbarrier
 * nothing arrives on, with no copy or tensor-core work in flight:
 *   which 0: the decode kernels' suspending wait;
 *         1: the extend kernel's suspending wait;  2: its polling wait;
 *         3, 4: the same two after PA_DEVICE_WAIT_TIMEOUT is already set in
 *               the header (as when another CTA's wait expired): they must
 *               give up at once instead of waiting out their limit.
 * The wait ends after limit_ns (1e3 .. 1e8 ns) of %globaltimer and sets
 * PA_DEVICE_WAIT_TIMEOUT in the scratch header, which pa_check reports.  It
 * also writes two int64 at byte 64 of the scratch: 1 if the wait saw the
 * phase complete (never expected here) else 0, and the nanoseconds it waited.
 * scratch: device, >= 65536 bytes, 256-byte aligned, header zeroed. */
pa_status pa_debug_wait_expiry(void* scratch, int32_t which, int64_t limit_ns, void* stream);

/* Static string for a status code. */
const char* pa_status_string(pa_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
