// FP8 E5M2 (kind::f8f6f4, bfloat16 C), K-major B: the single-CTA kernels of this operand kind and layout.
#include "launch.h"
namespace dgt {
DGT_DEFINE_VARIANTS(e5m2_km, KIND_E5M2, true)
}  // namespace dgt
