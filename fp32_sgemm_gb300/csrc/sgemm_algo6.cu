// Main-kernel instantiation for tile configuration 6: 128 x 128 output
// tile, BK=32, 3 stages, TMA issued by thread 0, double-buffered 8-byte A fragments, 2 CTAs/SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo6 = FfmaConfig<128,128,32,3,2,2,8,2,2,2,0,1>;
void fill_algo6(KernelEntry *v) { fill_variants<CfgAlgo6>(v); }
}  // namespace sg
