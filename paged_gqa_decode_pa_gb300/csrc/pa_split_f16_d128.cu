// Instantiations of the split kernel for f16 storage, head_dim 128.
#include "pa_split.cuh"

PA_INSTANTIATE_SPLIT(__half, 128, pa::kMma)
PA_INSTANTIATE_SPLIT(__half, 128, pa::kSimt)
