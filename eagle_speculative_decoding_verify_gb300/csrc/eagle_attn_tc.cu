// Tensor-core (tcgen05) path of eagle_tree_attn: not enabled yet.
#include "eagle_attn.h"

namespace eagle {
bool tc_supported(int) { return false; }
int attn_tc_num_launches(const eagle_attn_item*, int, int, int, int) { return 0; }
size_t attn_tc_ws_size(const eagle_attn_item*, int, int, int, int, int) { return 0; }
eagle_status attn_tc_launch(const eagle_attn_item*, int, int, int, int, float, void*, size_t,
                            cudaStream_t, int) {
  return EAGLE_ERR_UNSUPPORTED_SHAPE;
}
}  // namespace eagle
