// Main-kernel instantiation for tile configuration 7: 128 x 128 output
// tile, BK=32, 3 stages, TMA issued by thread 0, compiler-scheduled fragments, 2 CTAs/SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo7 = FfmaConfig<128,128,32,3,2,2,8,1,2,4,0,0>;
void fill_algo7(KernelEntry *v) { fill_variants<CfgAlgo7>(v); }
}  // namespace sg
