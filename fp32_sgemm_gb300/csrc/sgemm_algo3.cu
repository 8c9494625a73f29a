// Main-kernel instantiation for tile configuration 3: 128 x 128 output
// tile, BK=16, 4 stages, TMA issued by thread 0, double-buffered fragments, 2 CTAs/SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo3 = FfmaConfig<128,128,16,4,2,2,8,2,2,4,0,1>;
void fill_algo3(KernelEntry *v) { fill_variants<CfgAlgo3>(v); }
}  // namespace sg
