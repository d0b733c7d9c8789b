// Instantiations of the split kernel for several query tokens per sequence
// (one warp per tile stream, warp pairs, and wide rows),
// bf16 storage, head_dim 128.
#include "pa_split.cuh"

PA_INSTANTIATE_SPLIT(__nv_bfloat16, 128, pa::kMmaQ)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, 128, pa::kMmaP)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, 128, pa::kMmaW)
