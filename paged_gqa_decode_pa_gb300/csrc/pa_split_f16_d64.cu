// Instantiations of the split kernel for f16 storage, head_dim 64.
#include "pa_split.cuh"

PA_INSTANTIATE_SPLIT(__half, 64, pa::kMma)
PA_INSTANTIATE_SPLIT(__half, 64, pa::kSimt)
