// FP16, row-major B: the two-pair kernels (A shared by multicast) of this operand kind and layout.
#include "launch.h"
namespace dgt {
#if !DGT_NO_MULTICAST
DGT_DEFINE_QUAD_VARIANTS(f16_rm, KIND_F16, false)
#else
DGT_DEFINE_NO_QUAD(f16_rm)
#endif
}  // namespace dgt
