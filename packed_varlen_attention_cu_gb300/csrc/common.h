// common.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <stdint.h>

#include "../../include/pva.h"

namespace pva {

// Persistent CTA count: `requested` if positive, else the SM count of the
// current device (-1 when no device can be queried).
int32_t resolve_num_ctas(int32_t requested);

// Byte offset of the D scratch inside a backward plan for this problem, or -1
// when the problem has no backward plan (see pva_bwd_plan_bytes).
int64_t bwd_plan_dvec_offset(int32_t num_docs, const pva_mask_desc* mask,
                             const pva_worklist_params* params);

}  // namespace pva
