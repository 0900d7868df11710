// combine_f16.cu -- the combine kernels for fp16 inputs and outputs
// (Struct_ep_combine_skip_a2a: combine_dtype; trtllm_moe_allreduce_fusion:
// "fp16/bf16 -> fp4"), compiled apart from the bf16 ones to build in parallel.
#include "combine_impl.cuh"

namespace nqg {
namespace combine_detail {

template moe_status launch_io<1>(const Params &, const Plan &, int32_t, cudaStream_t);

} // namespace combine_detail
} // namespace nqg
