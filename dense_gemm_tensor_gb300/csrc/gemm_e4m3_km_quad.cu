// FP8 E4M3 (kind::f8f6f4, bfloat16 C), K-major B: the two-pair kernels (A shared by multicast) of this operand kind and layout.
#include "launch.h"
namespace dgt {
#if !DGT_NO_MULTICAST
DGT_DEFINE_QUAD_VARIANTS(e4m3_km, KIND_E4M3, true)
#else
DGT_DEFINE_NO_QUAD(e4m3_km)
#endif
}  // namespace dgt
