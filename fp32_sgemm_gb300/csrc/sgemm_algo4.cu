// Main-kernel instantiation for tile configuration 4: 128 x 128 output tile,
// BK=16, 6 stages, 8-byte A reads, 4 compute warps + 1 TMA producer warp, one CTA per SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo4 = FfmaConfig<128,128,16,6,2,2,8,1,1,2>;
void fill_algo4(KernelEntry *v) { fill_variants<CfgAlgo4>(v); }
}  // namespace sg
