// Main-kernel instantiation for tile configuration 1: 128 x 128 output
// tile, BK=32, 4 stages, dedicated TMA producer warp, compiler-scheduled fragments, 1 CTA/SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo1 = FfmaConfig<128,128,32,4,2,2,8,1,1,4,1,0>;
void fill_algo1(KernelEntry *v) { fill_variants<CfgAlgo1>(v); }
}  // namespace sg
