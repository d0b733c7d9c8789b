// Instantiations of the split kernel for bf16 storage, head_dim 256.
#include "pa_split.cuh"

PA_INSTANTIATE_SPLIT(__nv_bfloat16, 256, pa::kMma)
PA_INSTANTIATE_SPLIT(__nv_bfloat16, 256, pa::kSimt)
