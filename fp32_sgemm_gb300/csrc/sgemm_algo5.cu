// Main-kernel instantiation for tile configuration 5: 128 x 128 output
// tile, BK=32, 3 stages, TMA issued by thread 0, double-buffered fragments, 2 CTAs/SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo5 = FfmaConfig<128,128,32,3,2,2,8,2,2,4,0,1>;
void fill_algo5(KernelEntry *v) { fill_variants<CfgAlgo5>(v); }
}  // namespace sg
