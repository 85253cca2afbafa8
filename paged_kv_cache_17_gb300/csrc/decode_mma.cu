// Instantiations of the tensor-core decode kernel, bf16 KV pool: head_dim 64 / 128, query
// groups of 1, 2, 4, 8, plain and cascade forms.
#include "decode_launch.cuh"

namespace pkv {
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 64, false, false)
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 128, false, false)
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 64, false, true)
PKV_FOR_EACH_GROUP_MMA(PKV_DEFINE_DECODE_MMA, 128, false, true)
}  // namespace pkv
