// Kernel instantiation: 256-column tiles, tma A producer.
#include "gge_inst.cuh"

namespace gge {
GGE_INSTANTIATE(256, false, 1)
GGE_INSTANTIATE_TRANS(256)
}  // namespace gge
