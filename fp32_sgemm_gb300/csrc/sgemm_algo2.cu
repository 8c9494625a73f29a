// Main-kernel instantiation for tile configuration 2: 128 x 128 output tile,
// BK=32, 4 stages, 8-byte A reads, 4 compute warps + 1 TMA producer warp, one CTA per SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo2 = FfmaConfig<128,128,32,4,2,2,8,1,1,2>;
void fill_algo2(KernelEntry *v) { fill_variants<CfgAlgo2>(v); }
}  // namespace sg
