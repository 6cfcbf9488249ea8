// Instantiations of the fused kernels for the Hadamard variant (q and k
// rotated by H_128 / sqrt(128) after RoPE), compiled apart from the plain
// ones so the two sets build in parallel.
#include "dsa_prep_kernels.cuh"

namespace dsa_prep_impl {

const KernelFn kPipelineHad[2][5] = {
    {pipeline_fn<true, 0, 0>(), pipeline_fn<true, 0, 1>(), pipeline_fn<true, 0, 2>(),
     pipeline_fn<true, 0, 4>(), pipeline_fn<true, 0, 8>()},
    {pipeline_fn<true, 1, 0>(), pipeline_fn<true, 1, 1>(), pipeline_fn<true, 1, 2>(),
     pipeline_fn<true, 1, 4>(), pipeline_fn<true, 1, 8>()}};
const KernelFn kPipelineMultiHad[2][5] = {
    {pipeline_fn<true, 0, 0, true>(), pipeline_fn<true, 0, 1, true>(), pipeline_fn<true, 0, 2, true>(),
     pipeline_fn<true, 0, 4, true>(), pipeline_fn<true, 0, 8, true>()},
    {pipeline_fn<true, 1, 0, true>(), pipeline_fn<true, 1, 1, true>(), pipeline_fn<true, 1, 2, true>(),
     pipeline_fn<true, 1, 4, true>(), pipeline_fn<true, 1, 8, true>()}};
const KernelFn kDirectHad[2][5] = {
    {direct_fn<true, 0, 0>(), direct_fn<true, 0, 1>(), direct_fn<true, 0, 2>(),
     direct_fn<true, 0, 4>(), direct_fn<true, 0, 8>()},
    {direct_fn<true, 1, 0>(), direct_fn<true, 1, 1>(), direct_fn<true, 1, 2>(),
     direct_fn<true, 1, 4>(), direct_fn<true, 1, 8>()}};
const KernelFn kStreamHad[2][5] = {
    {kstream_fn<true, 0, 0>(), kstream_fn<true, 0, 1>(), kstream_fn<true, 0, 2>(),
     kstream_fn<true, 0, 4>(), kstream_fn<true, 0, 8>()},
    {kstream_fn<true, 1, 0>(), kstream_fn<true, 1, 1>(), kstream_fn<true, 1, 2>(),
     kstream_fn<true, 1, 4>(), kstream_fn<true, 1, 8>()}};

}  // namespace dsa_prep_impl
