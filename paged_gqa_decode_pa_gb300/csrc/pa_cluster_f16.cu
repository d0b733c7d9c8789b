// Instantiations of the cluster kernel for f16 storage, every head dimension.
#include "pa_cluster.cuh"

PA_INSTANTIATE_CLUSTER(__half, 64)
PA_INSTANTIATE_CLUSTER(__half, 128)
PA_INSTANTIATE_CLUSTER(__half, 256)
