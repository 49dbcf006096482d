// Kernels instantiated for the collision population layout.
#define LBM_LAYOUT LAYOUT_COLLISION
#include "lbm_layout_impl.cuh"

namespace lbm {
const LayoutOps& layout_ops_collision() { return kOps; }
}  // namespace lbm
