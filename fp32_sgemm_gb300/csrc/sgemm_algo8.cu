// Main-kernel instantiation for tile configuration 8: 128 x 128 output
// tile, BK=32, 3 stages, TMA issued by thread 0, double-buffered fragments (slice fully unrolled), 2 CTAs/SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo8 = FfmaConfig<128,128,32,3,2,2,8,8,2,4,0,1>;
void fill_algo8(KernelEntry *v) { fill_variants<CfgAlgo8>(v); }
}  // namespace sg
