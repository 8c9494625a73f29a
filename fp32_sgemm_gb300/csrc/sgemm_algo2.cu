// Main-kernel instantiation for tile configuration 2: 128 x 128 output
// tile, BK=32, 4 stages, dedicated TMA producer warp, double-buffered fragments, 1 CTA/SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo2 = FfmaConfig<128,128,32,4,2,2,8,2,1,4,1,1>;
void fill_algo2(KernelEntry *v) { fill_variants<CfgAlgo2>(v); }
}  // namespace sg
