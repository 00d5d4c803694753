// Append new tokens' K/V to the paged cache: the write side of the cache.
//
// Operation: "vllm/v1/attention/backends/b12x", do_kv_cache_update, which
// hands key, value, the two caches, slot_mapping, the cache dtype and the
// per-tensor k_scale / v_scale to reshape_and_cache_flash: token t goes to
// page slot_mapping[t] / page_size, slot slot_mapping[t] % page_size; a
// negative slot is padding.  An e4m3 cache stores e4m3(x / scale), rounded
// to nearest even and saturated to +-448.
//
// One thread moves 8 consecutive head_dim elements of one (token, kv head):
// a 16-byte load of the new bf16 values, a 16-byte (bf16) or 8-byte (e4m3)
// store into the page; the kernel is a pure HBM stream.
#include <cstdint>

#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

struct AppendParams {
  const uint16_t* k_new;
  const uint16_t* v_new;
  int64_t new_stride_tok, new_stride_head;
  uint8_t* k_cache;
  uint8_t* v_cache;
  int64_t stride_page, stride_tok, stride_head;   // bytes
  int num_pages, page_size, num_kv_heads, head_dim, num_tokens;
  int vpr_log2;        // log2(head_dim / 8): 8-element vectors per row
  int ps_log2;         // log2(page_size) when it is a power of two, else -1
  const int64_t* slot_mapping;
  float k_scale, v_scale;
  uint32_t* err;   // optional error word
};

// (the host guarantees tokens x heads x head_dim / 8 < 2^31, so the thread
// index and its row split stay in 32 bits; head_dim / 8 is a power of two)
template <bool FP8>
__global__ void __launch_bounds__(256) append_kv_kernel(const AppendParams p) {
  const uint32_t total = static_cast<uint32_t>(p.num_tokens) * static_cast<uint32_t>(p.num_kv_heads)
                         << p.vpr_log2;
  const uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int vv = static_cast<int>(idx & ((1u << p.vpr_log2) - 1u));
  const uint32_t th = idx >> p.vpr_log2;
  const uint32_t nh = static_cast<uint32_t>(p.num_kv_heads);
  const int t = static_cast<int>(th / nh);
  const int h = static_cast<int>(th - static_cast<uint32_t>(t) * nh);
  const int64_t slot = p.slot_mapping[t];
  if (slot < 0) return;                                   // padding token
  int64_t page, off;
  if (p.ps_log2 >= 0) {
    page = slot >> p.ps_log2;
    off = slot & ((int64_t{1} << p.ps_log2) - 1);
  } else {
    page = slot / p.page_size;
    off = slot - page * p.page_size;
  }
  if (page >= p.num_pages) {                              // outside the pool: nothing written
    if (p.err != nullptr && vv == 0 && h == 0) atomicOr(p.err, kErrPageId);
    return;
  }
  const int64_t src = static_cast<int64_t>(t) * p.new_stride_tok + static_cast<int64_t>(h) * p.new_stride_head + vv * 8;
  const uint4 kx = *reinterpret_cast<const uint4*>(p.k_new + src);
  const uint4 vx = *reinterpret_cast<const uint4*>(p.v_new + src);
  const int64_t dst = page * p.stride_page + off * p.stride_tok + static_cast<int64_t>(h) * p.stride_head;
  if constexpr (!FP8) {
    *reinterpret_cast<uint4*>(p.k_cache + dst + vv * 16) = kx;
    *reinterpret_cast<uint4*>(p.v_cache + dst + vv * 16) = vx;
  } else {
    auto quant8 = [](const uint4& w, float scale) {
      const uint32_t in[4] = {w.x, w.y, w.z, w.w};
      uint32_t out[2] = {0u, 0u};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float lo = __fdiv_rn(bf16_to_f32(static_cast<uint16_t>(in[k] & 0xffffu)), scale);
        const float hi = __fdiv_rn(bf16_to_f32(static_cast<uint16_t>(in[k] >> 16)), scale);
        const uint32_t pair = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
        out[k >> 1] |= pair << (16 * (k & 1));
      }
      return make_uint2(out[0], out[1]);
    };
    *reinterpret_cast<uint2*>(p.k_cache + dst + vv * 8) = quant8(kx, p.k_scale);
    *reinterpret_cast<uint2*>(p.v_cache + dst + vv * 8) = quant8(vx, p.v_scale);
  }
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_append_kv(const void* k_new, const void* v_new, int64_t new_stride_tok,
                                  int64_t new_stride_head, void* k_cache, void* v_cache, int64_t kv_stride_page,
                                  int64_t kv_stride_tok, int64_t kv_stride_head, int32_t num_pages,
                                  int32_t page_size, int32_t num_kv_heads, int32_t head_dim, int32_t kv_dtype,
                                  const int64_t* slot_mapping, int32_t num_tokens, float k_scale, float v_scale,
                                  void* scratch, void* stream) {
  using namespace pa;
  if (num_tokens < 0 || num_kv_heads <= 0 || page_size <= 0 || num_pages <= 0) return PA_ERR_INVALID_ARG;
  if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
  const bool fp8 = kv_dtype == PA_KV_FP8_E4M3;
  if (fp8 && !(k_scale > 0.f && v_scale > 0.f)) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (new_stride_tok <= 0 || new_stride_head <= 0 || kv_stride_page <= 0 || kv_stride_tok <= 0 || kv_stride_head <= 0)
    return PA_ERR_INVALID_ARG;
  const int e = fp8 ? 1 : 2;
  auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  // 16-byte vector loads of the new values, 8/16-byte vector stores into pages
  if (!a16(k_new) || !a16(v_new) || (new_stride_tok % 8) || (new_stride_head % 8)) return PA_ERR_UNSUPPORTED;
  if (!a16(k_cache) || !a16(v_cache) || (kv_stride_page * e) % 16 || (kv_stride_tok * e) % 16 ||
      (kv_stride_head * e) % 16)
    return PA_ERR_UNSUPPORTED;
  AppendParams p{};
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.new_stride_tok = new_stride_tok;
  p.new_stride_head = new_stride_head;
  p.k_cache = static_cast<uint8_t*>(k_cache);
  p.v_cache = static_cast<uint8_t*>(v_cache);
  p.stride_page = kv_stride_page * e;
  p.stride_tok = kv_stride_tok * e;
  p.stride_head = kv_stride_head * e;
  p.num_pages = num_pages;
  p.page_size = page_size;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.num_tokens = num_tokens;
  p.vpr_log2 = head_dim == 64 ? 3 : (head_dim == 128 ? 4 : 5);
  p.ps_log2 = (page_size & (page_size - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(page_size)) : -1;
  p.slot_mapping = slot_mapping;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.err = static_cast<uint32_t*>(scratch);
  const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * (head_dim / 8);
  if (total >= (int64_t{1} << 31)) return PA_ERR_UNSUPPORTED;   // one call moves < 2^31 vectors
  const unsigned blocks = static_cast<unsigned>((total + 255) / 256);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (fp8) {
    append_kv_kernel<true><<<blocks, 256, 0, st>>>(p);
  } else {
    append_kv_kernel<false><<<blocks, 256, 0, st>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
