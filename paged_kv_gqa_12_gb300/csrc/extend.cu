// Prefix-prefill / extend over the paged cache (placeholder until the
// tensor-core kernel lands).
#include "extend.h"
#include "pa_internal.h"

namespace pa {

pa_status plan_extend(const pa_shape& s, int num_sms, pa_plan_t* out) {
  (void)s;
  (void)num_sms;
  (void)out;
  return PA_ERR_UNSUPPORTED;
}

}  // namespace pa

extern "C" pa_status pa_extend(const pa_plan_t* plan, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                               const void* k_cache, const void* v_cache, int64_t kv_stride_page,
                               int64_t kv_stride_tok, int64_t kv_stride_head, int32_t num_pages,
                               const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens,
                               const int32_t* query_start_loc, int32_t batch, int32_t total_q, float scale,
                               const float* sinks, float k_scale, float v_scale, void* out, int64_t out_stride_tok,
                               int64_t out_stride_head, float* lse, void* scratch, int64_t scratch_bytes,
                               void* stream) {
  return PA_ERR_UNSUPPORTED;
}
