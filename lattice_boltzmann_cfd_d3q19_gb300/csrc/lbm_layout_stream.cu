// Kernels instantiated for the stream population layout.
#define LBM_LAYOUT LAYOUT_STREAM
#include "lbm_layout_impl.cuh"

namespace lbm {
const LayoutOps& layout_ops_stream() { return kOps; }
}  // namespace lbm
