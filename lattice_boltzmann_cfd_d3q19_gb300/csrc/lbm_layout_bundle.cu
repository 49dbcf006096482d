// Kernels instantiated for the bundle population layout.
#define LBM_LAYOUT LAYOUT_BUNDLE
#include "lbm_layout_impl.cuh"

namespace lbm {
const LayoutOps& layout_ops_bundle() { return kOps; }
}  // namespace lbm
