#include "tc_fused.h"

namespace ttc {

bool tc_supported(const LayerPlan&) { return false; }
size_t tc_operand_bytes(const LayerPlan&) { return 256; }
tt_status tc_forward(const LayerPlan&, int64_t, const void*, const float*, const float*,
                     const float*, void*, void*, size_t, cudaStream_t) {
  return TT_ERR_UNSUPPORTED;
}
tt_status tc_backward(const LayerPlan&, int64_t, const void*, const void*, const float*,
                      const float*, const float*, void*, float*, bool, float*, float*, void*,
                      size_t, cudaStream_t) {
  return TT_ERR_UNSUPPORTED;
}

}  // namespace ttc
