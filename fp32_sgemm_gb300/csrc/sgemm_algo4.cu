// Main-kernel instantiation for tile configuration 4: 128 x 128 output
// tile, BK=16, 4 stages, TMA issued by thread 0, double-buffered fragments (slice fully unrolled), 2 CTAs/SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo4 = FfmaConfig<128,128,16,4,2,2,8,4,2,4,0,1>;
void fill_algo4(KernelEntry *v) { fill_variants<CfgAlgo4>(v); }
}  // namespace sg
