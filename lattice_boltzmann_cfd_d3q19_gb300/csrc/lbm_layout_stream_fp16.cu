// Kernels instantiated for the stream layout with half-precision population storage.
#define LBM_LAYOUT LAYOUT_STREAM_FP16
#include "lbm_layout_impl.cuh"

namespace lbm {
const LayoutOps& layout_ops_stream_fp16() { return kOps; }
}  // namespace lbm
