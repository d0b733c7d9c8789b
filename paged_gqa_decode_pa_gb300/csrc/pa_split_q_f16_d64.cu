// Instantiations of the split kernel for several query tokens per sequence
// (one warp per tile stream, warp pairs, and wide rows),
// f16 storage, head_dim 64.
#include "pa_split.cuh"

PA_INSTANTIATE_SPLIT(__half, 64, pa::kMmaQ)
PA_INSTANTIATE_SPLIT(__half, 64, pa::kMmaP)
PA_INSTANTIATE_SPLIT(__half, 64, pa::kMmaW)
