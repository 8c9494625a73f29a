// Main-kernel instantiation for tile configuration 9: 128 x 128 output
// tile, BK=32, 3 stages, TMA issued by thread 0, double-buffered 8-byte A
// fragments (slice fully unrolled), 2 CTAs/SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo9 = FfmaConfig<128,128,32,3,2,2,8,8,2,2,0,1>;
void fill_algo9(KernelEntry *v) { fill_variants<CfgAlgo9>(v); }
}  // namespace sg
