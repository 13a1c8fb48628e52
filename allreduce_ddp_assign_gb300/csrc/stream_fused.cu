// The streaming kernel's fused pack + ring-reduce (+ copy-back) instantiations
// (those for 16-bit gradients reduced through a 16-bit wire type are in
// stream_fused_wire.cu).
#include "stream_impl.cuh"

namespace ddpk {
ddp_status launch_stream_fused_wire(StreamArgs& a, int dtype, void* stream);  // stream_fused_wire.cu

ddp_status launch_stream_fused(StreamArgs& a, int dtype, void* stream)
{
    if (a.wire != DDP_F32 && dtype != DDP_F32) return launch_stream_fused_wire(a, dtype, stream);
    return launch_op<OP_FUSED, false>(a, dtype, stream);
}
}  // namespace ddpk
