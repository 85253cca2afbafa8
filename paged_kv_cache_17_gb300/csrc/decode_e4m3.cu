// Instantiations of the paged decode kernel for a E4M3 KV pool (plain decode),
// head_dim 64 / 128, query-group sizes 1, 2, 4, 8.
#include "decode_launch.cuh"

namespace pkv {
PKV_FOR_EACH_GROUP(PKV_DEFINE_DECODE, 64, true, false)
PKV_FOR_EACH_GROUP(PKV_DEFINE_DECODE, 128, true, false)
}  // namespace pkv
