// Kernel instantiation: 128-column tiles, tma A producer.
#include "gge_inst.cuh"

namespace gge {
GGE_INSTANTIATE(128, false, 1)
GGE_INSTANTIATE_TRANS(128)
}  // namespace gge
