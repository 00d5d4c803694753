// Internal declarations shared by the CUDA translation units of the library.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa.h"

namespace pa {

// Scratch header at the start of every scratch workspace: the error word,
// then (from byte 256) one split-arrival counter per (request, kv head group)
// for decode plans whose last split merges the others.  Zero when a call
// starts; every call leaves it zero unless it reported a device error.
constexpr int64_t kScratchHeaderBytes = 65536;
constexpr int64_t kMergeCounterOffset = 256;
constexpr int64_t kMergeCounters = (kScratchHeaderBytes - kMergeCounterOffset) / 4;
// Device error codes OR-ed into the header's first word (pa_device_code).
constexpr uint32_t kErrWaitTimeout = PA_DEVICE_WAIT_TIMEOUT;     // an mbarrier wait ran out of time
constexpr uint32_t kErrSchedOverflow = PA_DEVICE_WORK_OVERFLOW;  // a work list exceeded its capacity
constexpr uint32_t kErrCapacity = PA_DEVICE_CAPACITY;            // a length exceeded the plan's capacity
constexpr uint32_t kErrPageId = PA_DEVICE_PAGE_ID;               // a page id outside the pool
// Wall-clock bound on every device-side wait (nanoseconds of %globaltimer).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Decode launch parameters (by value to both decode kernels).
struct DecodeParams {
  const uint16_t* q;          // bf16 [B, Hq, D]
  int64_t q_stride_tok, q_stride_head;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* seq_lens;
  int batch, num_q_heads, num_kv_heads, group, page_size;
  int num_pages;              // pool size: block-table entries must lie in [0, num_pages)
  float scale_log2;           // scale * log2(e)
  float cap_log2;             // soft_cap * log2(e); 0 = off
  float scale_over_cap;       // scale / soft_cap
  int window;                 // 0 = off
  const float* sinks;         // [Hq] or null
  float k_scale, v_scale;
  const float* k_scales;      // fp8: [B] per-request scales replacing k_scale, or null
  const float* v_scales;
  uint16_t* out;              // bf16 [B, Hq, D]
  int64_t out_stride_tok, out_stride_head;
  float* lse;                 // [B, Hq] or null
  float* o_part;              // [B, Hq, max_splits, D] normalised split outputs
  float* lse_part;            // [B, Hq, max_splits] split LSE (natural log)
  int tile_tokens;            // keys per pipeline stage
  int max_splits;
  int split_tiles;            // >0: tiles per split (planner mode)
  int fixed_splits;           // >0: split count per request (fixed mode)
  int bt_cache;               // block-table entries staged per CTA
  int q_len;                  // query tokens per request: 1 (decode) or 1 + speculative (verify)
  int head_groups;            // CTAs per kv head: ceil(group / 16) for decode groups above 16, else 1
  const int32_t* qsl;         // verify: query_start_loc, checked to be b * q_len; null for decode
  uint32_t* merge_cnt;        // [B, Hkv * head_groups] split-arrival counters: the last split of a
                              // request's kv head merges its splits; null = a merge kernel follows
  uint32_t* err;              // scratch header error word
};

struct DecodeConfig {
  int head_dim;
  bool fp8;
  int nh8;                    // ceil(query rows per kv head / 8)
  int tile_tokens;
  int stages;
  int warps;
  int smem_bytes;
};

// Host helpers shared by the entry points (api.cu).
pa_status validate_shape(const pa_shape& s);
pa_status check_kv(const pa_shape& s, const void* k, const void* v, int64_t st_page, int64_t st_tok,
                   int64_t st_head, int32_t num_pages);
pa_status make_kv_map(CUtensorMap* map, const void* base, bool fp8, int D, int Hkv, int ps, int num_pages,
                      int64_t st_page, int64_t st_tok, int64_t st_head, int box_rows);
pa_status make_q_map(CUtensorMap* map, const void* base, int D, int Hq, int rows, int64_t st_tok, int64_t st_head,
                     int group, int rows_per_box);

// Split-KV path for decode (q_len = 1, qsl = null) and verify (equal q_len
// per request, qsl checked on the device).
pa_status run_split_kv(const pa_plan_t* plan, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                       const void* k_cache, const void* v_cache, int64_t kv_stride_page, int64_t kv_stride_tok,
                       int64_t kv_stride_head, int32_t num_pages, const int32_t* block_table, int64_t bt_stride,
                       const int32_t* seq_lens, const int32_t* qsl, int32_t batch, float scale, const float* sinks,
                       float k_scale, float v_scale, const float* k_scales, const float* v_scales, void* out,
                       int64_t out_stride_tok, int64_t out_stride_head, float* lse, void* scratch,
                       int64_t scratch_bytes, void* stream);

// Kernel-variant table shared by the planner and the launcher.
DecodeConfig decode_config(int head_dim, bool fp8, int rows, int bt_cache);

cudaError_t launch_decode(const DecodeConfig& cfg, const CUtensorMap& tmk, const CUtensorMap& tmv,
                          const DecodeParams& p, dim3 grid, cudaStream_t stream);

}  // namespace pa
