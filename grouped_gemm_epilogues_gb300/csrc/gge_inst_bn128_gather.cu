// Kernel instantiation: 128-column tiles, gather A producer.
#include "gge_inst.cuh"

namespace gge {
GGE_INSTANTIATE(128, true, 1)
}  // namespace gge
