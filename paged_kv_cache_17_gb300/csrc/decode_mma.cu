// Instantiations of the tensor-core decode kernel (bf16 KV pool), head_dim 64 / 128,
// query-group sizes 1, 2, 4, 8: the plain form and the cascade form (merges shared-prefix
// records).
#include "decode_launch.cuh"

namespace pkv {
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 64, false)
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 128, false)
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 64, true)
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 128, true)
}  // namespace pkv
