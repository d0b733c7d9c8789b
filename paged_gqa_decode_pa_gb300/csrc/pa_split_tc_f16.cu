// Instantiations of the tcgen05 split kernel for fp16 storage, head_dim 128.
#include "pa_split_tc.cuh"

PA_INSTANTIATE_SPLIT_TC(__half, false)
PA_INSTANTIATE_SPLIT_TC(__half, true)
