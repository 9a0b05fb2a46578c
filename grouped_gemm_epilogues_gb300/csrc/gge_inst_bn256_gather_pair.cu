// Kernel instantiation: 256 x 256 tiles on a CTA pair (tcgen05 cta_group::2), gathered A rows.
#include "gge_inst.cuh"

namespace gge {
GGE_INSTANTIATE(256, true, 2)
}  // namespace gge
