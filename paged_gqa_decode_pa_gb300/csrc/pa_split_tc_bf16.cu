// Instantiations of the tcgen05 split kernel for bf16 storage, head_dim 128.
#include "pa_split_tc.cuh"

PA_INSTANTIATE_SPLIT_TC(__nv_bfloat16, false)
PA_INSTANTIATE_SPLIT_TC(__nv_bfloat16, true)
