// BF16, row-major B: the CTA-pair kernel on the transposed product C^T = B^T A^T, each tile width.
#include "launch.h"
namespace dgt {
DGT_DEFINE_SWAP_VARIANTS(bf16_sw, KIND_BF16)
}  // namespace dgt
