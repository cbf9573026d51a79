// FP8 E4M3 (kind::f8f6f4, bfloat16 C), K-major B: the single-CTA kernels of this operand kind and layout.
#include "launch.h"
namespace dgt {
DGT_DEFINE_VARIANTS(e4m3_km, KIND_E4M3, true)
}  // namespace dgt
