// The streaming kernel's fused instantiations for 16-bit gradients reduced
// through the compression hook: every ring term and partial sum rounded to the
// 16-bit wire type.
#include "stream_impl.cuh"

namespace ddpk {
ddp_status launch_stream_fused_wire(StreamArgs& a, int dtype, void* stream)
{
    return launch_op<OP_FUSED, true>(a, dtype, stream);
}
}  // namespace ddpk
