// Instantiations of the paged decode kernel for a E4M3 KV pool, cascade variant (merges shared-prefix records),
// head_dim 64 / 128, query-group sizes 1, 2, 4, 8.
#include "decode_launch.cuh"

namespace pkv {
PKV_FOR_EACH_GROUP(PKV_DEFINE_DECODE, 64, true, true)
PKV_FOR_EACH_GROUP(PKV_DEFINE_DECODE, 128, true, true)
}  // namespace pkv
