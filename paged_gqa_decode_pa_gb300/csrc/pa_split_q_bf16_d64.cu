// Instantiations of the split kernel for several query tokens per sequence
// (one warp per tile stream, warp pairs, and wide rows),
// bf16 storage, head_dim 64.
#include "pa_split.cuh"

PA_INSTANTIATE_SPLIT(__nv_bfloat16, 64, pa::kMmaQ)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, 64, pa::kMmaP)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, 64, pa::kMmaW)
