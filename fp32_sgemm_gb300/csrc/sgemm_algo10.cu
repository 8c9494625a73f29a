// Main-kernel instantiation for tile configuration 10: 128 x 128 output
// tile, BK=32, 3 stages, TMA issued by thread 0, double-buffered 8-byte A
// fragments (unrolled by 4 A groups), 2 CTAs/SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo10 = FfmaConfig<128,128,32,3,2,2,8,4,2,2,0,1>;
void fill_algo10(KernelEntry *v) { fill_variants<CfgAlgo10>(v); }
}  // namespace sg
