// Extend (prefix-prefill) planning, shared between the C-ABI and the kernels.
#pragma once

#include "pa.h"

namespace pa {

pa_status plan_extend(const pa_shape& s, int num_sms, pa_plan_t* out);

}  // namespace pa
