// The streaming kernel's no_sync pack instantiations.
#include "stream_impl.cuh"

namespace ddpk {
ddp_status launch_stream_pack(StreamArgs& a, int dtype, void* stream) { return launch_op<OP_PACK, false>(a, dtype, stream); }
}  // namespace ddpk
