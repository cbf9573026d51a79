// TF32, row-major B: the two-pair kernels (A shared by multicast) of this operand kind and layout.
#include "launch.h"
namespace dgt {
#if !DGT_NO_MULTICAST
DGT_DEFINE_QUAD_VARIANTS(tf32_rm, KIND_TF32, false)
#else
DGT_DEFINE_NO_QUAD(tf32_rm)
#endif
}  // namespace dgt
