// TF32, K-major B: the two-pair kernels (A shared by multicast) of this operand kind and layout.
#include "launch.h"
namespace dgt {
#if !DGT_NO_MULTICAST
DGT_DEFINE_QUAD_VARIANTS(tf32_km, KIND_TF32, true)
#else
DGT_DEFINE_NO_QUAD(tf32_km)
#endif
}  // namespace dgt
