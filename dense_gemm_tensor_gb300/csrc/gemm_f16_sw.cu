// FP16, row-major B: the CTA-pair kernel on the transposed product C^T = B^T A^T, each tile width.
#include "launch.h"
namespace dgt {
DGT_DEFINE_SWAP_VARIANTS(f16_sw, KIND_F16)
}  // namespace dgt
