// The persistent decode kernel built with 8 compute warps (for rows wider
// than 2048 inputs; decode_plan picks the build): the same source as
// moe_layer.cu.
#define MOE_NCW 8
#include "moe_layer.cu"
