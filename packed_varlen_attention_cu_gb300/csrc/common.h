// common.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <stdint.h>

namespace pva {

// Persistent CTA count: `requested` if positive, else the SM count of the
// current device (-1 when no device can be queried).
int32_t resolve_num_ctas(int32_t requested);

}  // namespace pva
