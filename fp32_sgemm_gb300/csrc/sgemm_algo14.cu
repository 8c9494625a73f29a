// Main-kernel instantiation for tile configuration 14: 128 x 256 output
// tile, eight consumer warps (2 x 4 warp tiles of 64 x 64) in one CTA per SM,
// BK=32, 4 stages, TMA issued by thread 0, double-buffered fragments.  Two
// warps of the same CTA share each SM sub-partition, so neither can run
// ahead of the other by more than the ring depth.
#include "kernel_table.h"

namespace sg {
using CfgAlgo14 = FfmaConfig<128,256,32,4,2,4,8,4,1,2,0,1>;
void fill_algo14(KernelEntry *v) { fill_variants<CfgAlgo14>(v); }
}  // namespace sg
