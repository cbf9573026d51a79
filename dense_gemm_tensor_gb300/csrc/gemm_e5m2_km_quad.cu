// FP8 E5M2 (kind::f8f6f4, bfloat16 C), K-major B: the two-pair kernels (A shared by multicast) of this operand kind and layout.
#include "launch.h"
namespace dgt {
#if !DGT_NO_MULTICAST
DGT_DEFINE_QUAD_VARIANTS(e5m2_km, KIND_E5M2, true)
#else
DGT_DEFINE_NO_QUAD(e5m2_km)
#endif
}  // namespace dgt
