// Instantiations of the cluster kernel for bf16 storage, every head dimension.
#include "pa_cluster.cuh"

PA_INSTANTIATE_CLUSTER(__nv_bfloat16, 64)
PA_INSTANTIATE_CLUSTER(__nv_bfloat16, 128)
PA_INSTANTIATE_CLUSTER(__nv_bfloat16, 256)
