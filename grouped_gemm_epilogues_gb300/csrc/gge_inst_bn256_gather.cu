// Kernel instantiation: 256-column tiles, gather A producer.
#include "gge_inst.cuh"

namespace gge {
GGE_INSTANTIATE(256, true, 1)
}  // namespace gge
