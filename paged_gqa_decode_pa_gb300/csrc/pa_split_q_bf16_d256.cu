// Instantiations of the split kernel for several query tokens per sequence
// (one warp per tile stream, and warp pairs),
// bf16 storage, head_dim 256.
#include "pa_split.cuh"

PA_INSTANTIATE_SPLIT(__nv_bfloat16, 256, pa::kMmaQ)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, 256, pa::kMmaP)
