// Main-kernel instantiation for tile configuration 30: 128 x 256 output
// tile, eight consumer warps in one CTA per SM, BK=32, 4 stages, the inner
// loop of configuration 28, C from registers.  The wide-product form of
// configuration 29.
#include "kernel_table.h"

namespace sg {
using CfgAlgo30 = FfmaConfig<128,256,32,4,2,4,8,4,1,4,0>;
void fill_algo30(KernelEntry *v) { fill_variants<CfgAlgo30>(v); }
}  // namespace sg
