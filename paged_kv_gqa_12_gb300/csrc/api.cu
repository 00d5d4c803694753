// C-ABI entry points (include/pa.h): planning, argument validation, TMA
// tensor-map construction and kernel launches.  Host code only.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"
#include "extend.h"

namespace pa {
namespace {

constexpr int kMaxSmemPerCta = 232448;  // 227 KB opt-in dynamic shared memory on sm_103a
constexpr float kLog2eHost = 1.4426950408889634f;

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
  });
  return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

pa_status validate_shape(const pa_shape& s) {
  if (s.mode != PA_MODE_DECODE && s.mode != PA_MODE_EXTEND && s.mode != PA_MODE_VERIFY) return PA_ERR_INVALID_ARG;
  if (s.num_q_heads <= 0 || s.num_kv_heads <= 0 || s.num_q_heads % s.num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (s.max_batch < 0 || s.max_pages_per_seq < 0 || s.max_total_q < 0 || s.window < 0 || s.num_splits < 0 ||
      s.num_sms < 0)
    return PA_ERR_INVALID_ARG;
  if (!(s.soft_cap >= 0.f) || !std::isfinite(s.soft_cap)) return PA_ERR_INVALID_ARG;
  if (s.kv_dtype != PA_KV_BF16 && s.kv_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
  if (s.has_sinks != 0 && s.has_sinks != 1) return PA_ERR_INVALID_ARG;
  if (s.head_dim != 64 && s.head_dim != 128 && s.head_dim != 256) return PA_ERR_UNSUPPORTED;
  if (s.page_size != 16 && s.page_size != 32 && s.page_size != 64) return PA_ERR_UNSUPPORTED;
  // decode splits larger groups over several CTAs (16 heads each); extend
  // packs 128 / group tokens per query tile
  if (s.num_q_heads / s.num_kv_heads > 128) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(s.max_pages_per_seq) * s.page_size > (int64_t{1} << 30)) return PA_ERR_UNSUPPORTED;
  if (s.mode == PA_MODE_VERIFY) {
    if (s.q_len < 1) return PA_ERR_INVALID_ARG;
    if (s.q_len * (s.num_q_heads / s.num_kv_heads) > 16) return PA_ERR_UNSUPPORTED;  // rows per kv head
  }
  return PA_OK;
}

// Query tokens per request on the split-KV path.
int split_kv_qlen(const pa_shape& s) { return s.mode == PA_MODE_VERIFY ? s.q_len : 1; }

// CTAs per kv head on the split-KV path: each covers at most 16 query rows.
int split_kv_head_groups(const pa_shape& s) {
  const int G = s.num_q_heads / s.num_kv_heads;
  return (s.mode == PA_MODE_DECODE && G > 16) ? (G + 15) / 16 : 1;
}

// Scratch bytes a split-KV plan needs: the header, then the normalised split
// outputs o_part [max_batch, q_len, Hq, max_splits, D] and their LSEs, each
// region 256-byte aligned.
int64_t split_kv_scratch_bytes(const pa_shape& s, int64_t max_splits) {
  const int64_t prow = static_cast<int64_t>(s.max_batch) * split_kv_qlen(s) * s.num_q_heads * max_splits;
  return kScratchHeaderBytes + align_up(prow * s.head_dim * 4, 256) + align_up(prow * 4, 256);
}

namespace {

// Keys a split-KV request attends to (union over its q_len queries): the
// window of the first query reaches W keys back, the last query adds q_len - 1.
int64_t decode_keys(int64_t L, int window, int q_len) {
  return window > 0 ? std::min<int64_t>(L, static_cast<int64_t>(window) + q_len - 1) : L;
}

pa_status plan_decode(const pa_shape& s, const int32_t* host_lens, int32_t batch, int num_sms, pa_plan_t* out) {
  const int G = s.num_q_heads / s.num_kv_heads;
  const int qlen = split_kv_qlen(s);
  const int hgroups = split_kv_head_groups(s);
  const int rows = hgroups > 1 ? 16 : G * qlen;
  const bool fp8 = s.kv_dtype == PA_KV_FP8_E4M3;
  DecodeConfig cfg = decode_config(s.head_dim, fp8, rows, 0);
  const int TS = cfg.tile_tokens;
  const int64_t max_len = static_cast<int64_t>(s.max_pages_per_seq) * s.page_size;
  const int64_t max_n = decode_keys(max_len, s.window, qlen);
  // +1: a window start that is not tile-aligned adds one partial tile
  const int64_t max_tiles = max_n > 0 ? cdiv64(max_n, TS) + 1 : 1;
  int64_t split_tiles = 0, tps_max, max_splits;
  if (s.num_splits > 0) {
    max_splits = std::min<int64_t>(s.num_splits, max_tiles);
    tps_max = cdiv64(max_tiles, max_splits);
  } else {
    int64_t units = 0;
    if (host_lens) {
      for (int b = 0; b < batch; ++b) {
        const int64_t L = host_lens[b];
        const int64_t n = decode_keys(L, s.window, qlen);
        if (n > 0) units += cdiv64(L, TS) - (L - n) / TS;
      }
      units *= static_cast<int64_t>(s.num_kv_heads) * hgroups;
    } else {
      units = static_cast<int64_t>(s.max_batch) * s.num_kv_heads * hgroups * max_tiles;
    }
    const int ctas_per_sm = (decode_config(s.head_dim, fp8, rows, 64).smem_bytes * 2 <= kMaxSmemPerCta) ? 2 : 1;
    const int64_t slots = static_cast<int64_t>(num_sms) * ctas_per_sm;
    const int64_t pairs = static_cast<int64_t>(host_lens ? batch : s.max_batch) * s.num_kv_heads * hgroups;
    // Splits per CTA slot: about four; once the (request, head) pairs alone
    // fill a wave, about eight, but each split then holds at least 1024 keys
    // per 8 query rows (fewer, longer splits cost less in prologues, partial
    // outputs and merging than they gain in balance).  Measured, with equal
    // splits per request: Llama-3-8B-shaped decode 0.1897 ms at four,
    // 0.1863 at eight (1024-key splits); its first 16 requests 0.0681 at
    // four, 0.0748 at eight; its verify form (4 tokens, 16 rows) 0.2127 with
    // 118-tile splits, 0.2196 with 1024-key ones; e4m3 window-1024 workload:
    // one split 2.30 TB/s, two 2.05.
    const bool wave = pairs >= slots;
    const int64_t target = slots * (wave ? 8 : 4);
    split_tiles = std::max<int64_t>(8, cdiv64(units, std::max<int64_t>(target, 1)));
    if (wave) split_tiles = std::max<int64_t>(split_tiles, cdiv64(1024 * std::max(1, rows / 8), TS));
    // no second split of a single tile (a window start off the tile grid)
    if (split_tiles + 1 >= max_tiles) split_tiles = max_tiles;
    split_tiles = std::min<int64_t>(split_tiles, max_tiles);
    max_splits = cdiv64(max_tiles, split_tiles);
    tps_max = split_tiles;
  }
  const int64_t bt_cache = cdiv64(tps_max * TS, s.page_size) + 2;
  if (bt_cache > (1 << 15)) return PA_ERR_UNSUPPORTED;
  cfg = decode_config(s.head_dim, fp8, rows, static_cast<int>(bt_cache));
  if (cfg.smem_bytes > kMaxSmemPerCta) return PA_ERR_UNSUPPORTED;

  out->tile_tokens = TS;
  out->split_tiles = static_cast<int32_t>(split_tiles);
  out->max_splits = static_cast<int32_t>(max_splits);
  out->stages = cfg.stages;
  out->warps = cfg.warps;
  out->bt_cache = static_cast<int32_t>(bt_cache);
  out->smem_bytes = cfg.smem_bytes;
  out->grid[0] = static_cast<int32_t>(max_splits);
  out->grid[1] = s.num_kv_heads * hgroups;
  out->grid[2] = s.max_batch;
  out->scratch_bytes = split_kv_scratch_bytes(s, max_splits);
  // several splits: the last split of each (request, kv head group) merges
  // them while the header has a counter for every such pair, else a merge
  // kernel follows the split kernel
  const int64_t pairs_cap = static_cast<int64_t>(s.max_batch) * s.num_kv_heads * hgroups;
  out->split_merge = (max_splits > 1 && pairs_cap <= kMergeCounters) ? 1 : 0;
  out->launches = (max_splits > 1 && !out->split_merge) ? 2 : 1;
  return PA_OK;
}

}  // namespace

// 4-D tensor map over a paged cache [pages, page_size, kv_heads, head_dim]:
// dims (innermost first) head_dim, kv head, slot, page.  Box: `box_bytes`
// of head_dim, one head, `box_rows` slots, one page, swizzled so that the
// kernels' ldmatrix / vector reads are bank-conflict free.
pa_status make_kv_map(CUtensorMap* map, const void* base, bool fp8, int D, int Hkv, int ps, int num_pages,
                      int64_t st_page, int64_t st_tok, int64_t st_head, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  const int e = fp8 ? 1 : 2;
  const int row_bytes = D * e;
  const int box_bytes = row_bytes < 128 ? row_bytes : 128;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(ps),
                        static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st_head * e), static_cast<cuuint64_t>(st_tok * e),
                           static_cast<cuuint64_t>(st_page * e)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_bytes / e), 1u, static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapSwizzle sw = box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_UNSUPPORTED;
}

// 3-D tensor map over packed queries [rows, Hq, D] (bf16): dims head_dim,
// q head, row; box 64 dims x `group` heads x `rows_per_box` rows, 128-byte
// swizzle, so one box per 64-dim chunk lands as a [rows*group, 64] K-major tile.
pa_status make_q_map(CUtensorMap* map, const void* base, int D, int Hq, int rows, int64_t st_tok, int64_t st_head,
                     int group, int rows_per_box) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(st_head * 2), static_cast<cuuint64_t>(st_tok * 2)};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(rows_per_box)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_UNSUPPORTED;
}

pa_status check_kv(const pa_shape& s, const void* k, const void* v, int64_t st_page, int64_t st_tok,
                   int64_t st_head, int32_t num_pages) {
  if (!k || !v || num_pages <= 0) return PA_ERR_INVALID_ARG;
  if (st_page <= 0 || st_tok <= 0 || st_head <= 0) return PA_ERR_INVALID_ARG;
  const int e = s.kv_dtype == PA_KV_FP8_E4M3 ? 1 : 2;
  if (!aligned(k, 16) || !aligned(v, 16)) return PA_ERR_UNSUPPORTED;
  if ((st_page * e) % 16 || (st_tok * e) % 16 || (st_head * e) % 16) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

namespace {

pa_status check_rows(const void* p, int64_t st_tok, int64_t st_head, bool required) {
  if (!p) return required ? PA_ERR_INVALID_ARG : PA_OK;
  if (st_tok <= 0 || st_head <= 0) return PA_ERR_INVALID_ARG;
  // rows are accessed as bf16 pairs: 4-byte alignment of every (row, head)
  if (!aligned(p, 4) || (st_tok % 2) || (st_head % 2)) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

int query_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

int32_t pa_version(void) { return 104; }

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape, layout or alignment";
    case PA_ERR_SCRATCH_TOO_SMALL: return "scratch workspace smaller than the plan requires";
    case PA_ERR_CUDA: return "CUDA call failed";
    case PA_ERR_DEVICE: return "a kernel reported a device-side error";
  }
  return "unknown status";
}

pa_status pa_plan(const pa_shape* shape, const int32_t* host_seq_lens, int32_t batch, pa_plan_t* plan) {
  if (!shape || !plan) return PA_ERR_INVALID_ARG;
  pa_status st = validate_shape(*shape);
  if (st != PA_OK) return st;
  if (host_seq_lens) {
    if (batch < 0 || batch > shape->max_batch) return PA_ERR_INVALID_ARG;
    const int64_t cap = static_cast<int64_t>(shape->max_pages_per_seq) * shape->page_size;
    for (int b = 0; b < batch; ++b)
      if (host_seq_lens[b] < 0 || host_seq_lens[b] > cap) return PA_ERR_INVALID_ARG;
  }
  int num_sms = shape->num_sms;
  if (num_sms == 0) {
    num_sms = query_sms();
    if (num_sms <= 0) return PA_ERR_CUDA;
  }
  pa_plan_t p;
  std::memset(&p, 0, sizeof p);
  p.shape = *shape;
  p.shape.num_sms = num_sms;
  if (shape->mode == PA_MODE_DECODE || shape->mode == PA_MODE_VERIFY) {
    st = plan_decode(*shape, host_seq_lens, batch, num_sms, &p);
  } else {
    st = plan_extend(*shape, num_sms, &p);
  }
  if (st != PA_OK) return st;
  *plan = p;
  return PA_OK;
}

pa_status pa_decode(const pa_plan_t* plan, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                    const void* k_cache, const void* v_cache, int64_t kv_stride_page, int64_t kv_stride_tok,
                    int64_t kv_stride_head, int32_t num_pages, const int32_t* block_table, int64_t bt_stride,
                    const int32_t* seq_lens, int32_t batch, float scale, const float* sinks, float k_scale,
                    float v_scale, const float* k_scales, const float* v_scales, void* out,
                    int64_t out_stride_tok, int64_t out_stride_head, float* lse, void* scratch,
                    int64_t scratch_bytes, void* stream) {
  if (!plan || plan->shape.mode != PA_MODE_DECODE) return PA_ERR_INVALID_ARG;
  return run_split_kv(plan, q, q_stride_tok, q_stride_head, k_cache, v_cache, kv_stride_page, kv_stride_tok,
                      kv_stride_head, num_pages, block_table, bt_stride, seq_lens, nullptr, batch, scale, sinks,
                      k_scale, v_scale, k_scales, v_scales, out, out_stride_tok, out_stride_head, lse, scratch,
                      scratch_bytes, stream);
}

}  // extern "C"

namespace pa {

pa_status run_split_kv(const pa_plan_t* plan, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                       const void* k_cache, const void* v_cache, int64_t kv_stride_page, int64_t kv_stride_tok,
                       int64_t kv_stride_head, int32_t num_pages, const int32_t* block_table, int64_t bt_stride,
                       const int32_t* seq_lens, const int32_t* qsl, int32_t batch, float scale, const float* sinks,
                       float k_scale, float v_scale, const float* k_scales, const float* v_scales, void* out,
                       int64_t out_stride_tok, int64_t out_stride_head, float* lse, void* scratch,
                       int64_t scratch_bytes, void* stream) {
  if (!plan) return PA_ERR_INVALID_ARG;
  const pa_shape& s = plan->shape;
  if ((s.mode != PA_MODE_DECODE && s.mode != PA_MODE_VERIFY) || validate_shape(s) != PA_OK) return PA_ERR_INVALID_ARG;
  if (s.mode == PA_MODE_VERIFY && !qsl) return PA_ERR_INVALID_ARG;
  if (batch < 0 || batch > s.max_batch) return PA_ERR_INVALID_ARG;
  if (batch > 65535) return PA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale)) return PA_ERR_INVALID_ARG;
  if ((sinks != nullptr) != (s.has_sinks != 0)) return PA_ERR_INVALID_ARG;
  if (!scratch || scratch_bytes < plan->scratch_bytes) return !scratch ? PA_ERR_INVALID_ARG : PA_ERR_SCRATCH_TOO_SMALL;
  if (scratch_bytes < kScratchHeaderBytes) return PA_ERR_SCRATCH_TOO_SMALL;
  if (!aligned(scratch, 256)) return PA_ERR_UNSUPPORTED;
  // a plan edited by hand must not index arrival counters past the header,
  // nor lay split partials out past the scratch_bytes it states, nor run a
  // tile size the kernels were not compiled for
  if (plan->split_merge != 0 &&
      static_cast<int64_t>(s.max_batch) * s.num_kv_heads * split_kv_head_groups(s) > kMergeCounters)
    return PA_ERR_INVALID_ARG;
  if (plan->max_splits < 1 || plan->split_tiles < 0 || plan->bt_cache < 1 ||
      plan->scratch_bytes < split_kv_scratch_bytes(s, plan->max_splits))
    return PA_ERR_INVALID_ARG;
  if (batch == 0) return PA_OK;
  if (!block_table || !seq_lens || bt_stride < 0) return PA_ERR_INVALID_ARG;
  pa_status st = check_rows(q, q_stride_tok, q_stride_head, true);
  if (st != PA_OK) return st;
  if ((st = check_rows(out, out_stride_tok, out_stride_head, true)) != PA_OK) return st;
  if (lse && !aligned(lse, 4)) return PA_ERR_UNSUPPORTED;
  if ((st = check_kv(s, k_cache, v_cache, kv_stride_page, kv_stride_tok, kv_stride_head, num_pages)) != PA_OK)
    return st;

  const bool fp8 = s.kv_dtype == PA_KV_FP8_E4M3;
  const int G = s.num_q_heads / s.num_kv_heads;
  const int qlen = split_kv_qlen(s);
  const int hgroups = split_kv_head_groups(s);
  const DecodeConfig cfg = decode_config(s.head_dim, fp8, hgroups > 1 ? 16 : G * qlen, plan->bt_cache);
  if (plan->tile_tokens != cfg.tile_tokens || cfg.smem_bytes > kMaxSmemPerCta) return PA_ERR_INVALID_ARG;
  const int box_rows = std::min(s.page_size, plan->tile_tokens);
  CUtensorMap tmk, tmv;
  if ((st = make_kv_map(&tmk, k_cache, fp8, s.head_dim, s.num_kv_heads, s.page_size, num_pages, kv_stride_page,
                        kv_stride_tok, kv_stride_head, box_rows)) != PA_OK)
    return st;
  if ((st = make_kv_map(&tmv, v_cache, fp8, s.head_dim, s.num_kv_heads, s.page_size, num_pages, kv_stride_page,
                        kv_stride_tok, kv_stride_head, box_rows)) != PA_OK)
    return st;

  DecodeParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.q_stride_tok = q_stride_tok;
  p.q_stride_head = q_stride_head;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = seq_lens;
  p.batch = batch;
  p.num_q_heads = s.num_q_heads;
  p.num_kv_heads = s.num_kv_heads;
  p.group = G;
  p.page_size = s.page_size;
  p.num_pages = num_pages;
  p.scale_log2 = scale * kLog2eHost;
  p.cap_log2 = s.soft_cap > 0.f ? s.soft_cap * kLog2eHost : 0.f;
  p.scale_over_cap = s.soft_cap > 0.f ? scale / s.soft_cap : 0.f;
  p.window = s.window;
  p.sinks = sinks;
  p.k_scale = fp8 ? k_scale : 1.f;
  p.v_scale = fp8 ? v_scale : 1.f;
  p.k_scales = fp8 ? k_scales : nullptr;
  p.v_scales = fp8 ? v_scales : nullptr;
  p.out = static_cast<uint16_t*>(out);
  p.out_stride_tok = out_stride_tok;
  p.out_stride_head = out_stride_head;
  p.lse = lse;
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  const int64_t rows = static_cast<int64_t>(s.max_batch) * qlen * s.num_q_heads * plan->max_splits;
  p.o_part = reinterpret_cast<float*>(sc + kScratchHeaderBytes);
  p.lse_part = reinterpret_cast<float*>(sc + kScratchHeaderBytes + align_up(rows * s.head_dim * 4, 256));
  p.tile_tokens = plan->tile_tokens;
  p.max_splits = plan->max_splits;
  p.split_tiles = plan->split_tiles;
  p.fixed_splits = s.num_splits > 0 ? plan->max_splits : 0;
  p.bt_cache = plan->bt_cache;
  p.q_len = qlen;
  p.head_groups = hgroups;
  p.qsl = qsl;
  p.merge_cnt = plan->split_merge ? reinterpret_cast<uint32_t*>(sc + kMergeCounterOffset) : nullptr;
  p.err = reinterpret_cast<uint32_t*>(sc);
  const dim3 grid(plan->max_splits, s.num_kv_heads * hgroups, batch);
  const cudaError_t e = launch_decode(cfg, tmk, tmv, p, grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa

extern "C" {

pa_status pa_scratch_init(void* scratch, void* stream) {
  if (!scratch) return PA_ERR_INVALID_ARG;
  const cudaError_t e = cudaMemsetAsync(scratch, 0, kScratchHeaderBytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_check(void* scratch, void* stream, uint32_t* device_code) {
  if (!scratch) return PA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, scratch, sizeof word, cudaMemcpyDeviceToHost, st) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  if (device_code) *device_code = word;
  if (word == 0) return PA_OK;
  // a failed call may leave split-arrival counters behind: clear the whole header
  if (cudaMemsetAsync(scratch, 0, kScratchHeaderBytes, st) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  return PA_ERR_DEVICE;
}

}  // extern "C"
