// combine_f16w.cu -- the combine kernels for fp16 inputs and outputs with
// fp16 router weights (Struct_ep_combine_skip_a2a: combine_dtype,
// router_weights_dtype): each row element is multiplied by its weight in one
// mixed-precision fma instead of being widened to fp32 first.  Compiled in
// its own unit to build in parallel.
#include "combine_impl.cuh"

namespace nqg {
namespace combine_detail {

template moe_status launch_io<2>(const Params &, const Plan &, int32_t, cudaStream_t);

} // namespace combine_detail
} // namespace nqg
