// Tensor-core two-segment denoise attention (placeholder until the tcgen05 kernel lands).

#include "tt_internal.h"

namespace tt {

bool attn_tc_supported(int, int, int, int, int, tt_dtype) { return false; }
size_t attn_tc_ws_bytes(int, int, int, int, int) { return 0; }
tt_status launch_attn_tc(const AttnArgs &) { return TT_ERR_UNSUPPORTED; }

}  // namespace tt
