// Instantiations of the tensor-core decode kernel, E4M3 KV pool: head_dim 64 / 128, query
// groups of 1, 2, 4, 8, plain and cascade forms.
#include "decode_launch.cuh"

namespace pkv {
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 64, true, false)
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 128, true, false)
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 64, true, true)
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 128, true, true)
}  // namespace pkv
