// Kernel instantiation: 256 x 224 tiles on a CTA pair (tcgen05 cta_group::2), TMA A producer.
#include "gge_inst.cuh"

namespace gge {
GGE_INSTANTIATE(224, false, 2)
}  // namespace gge
