// The dgrad kernels whose epilogue also takes the per-channel sums of the output.
#include "dgrad_variant.cuh"

template cudaError_t cdg_dgrad_prepare_variant<1>(int, int, bool);
template cudaError_t cdg_dgrad_launch_variant<1>(const CdgParams &, int, int, bool, int, size_t, cudaStream_t);
template int cdg_dgrad_max_pairs_variant<1>(int, int, bool, size_t);
