// Instantiations of the paged decode kernel for an OCP E4M3 KV pool with per-(K|V, kv head)
// fp32 scales (head_dim 64 / 128, query-group sizes 1, 2, 4, 8).
#include "decode_launch.cuh"

namespace pkv {
PKV_FOR_EACH_GROUP(PKV_DEFINE_DECODE, 64, true)
PKV_FOR_EACH_GROUP(PKV_DEFINE_DECODE, 128, true)
}  // namespace pkv
