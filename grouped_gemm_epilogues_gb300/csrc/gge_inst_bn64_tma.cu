// Kernel instantiation: 128 x 64 tiles (narrow outputs, e.g. a small M under swap_ab), TMA A producer.
#include "gge_inst.cuh"

namespace gge {
GGE_INSTANTIATE(64, false, 1)
GGE_INSTANTIATE_TRANS(64)
}  // namespace gge
