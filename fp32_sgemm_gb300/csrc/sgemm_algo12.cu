// Main-kernel instantiation for tile configuration 12: 64 x 256 output
// tile (one warp row of four 64 x 64 warp tiles), BK=32, 2 stages, TMA
// issued by thread 0, double-buffered fragments, 2 CTAs/SM.  For products
// with at most 64 rows, where a 128-row tile would compute padding rows.
#include "kernel_table.h"

namespace sg {
using CfgAlgo12 = FfmaConfig<64,256,32,2,1,4,8,4,2,2,0,1>;
void fill_algo12(KernelEntry *v) { fill_variants<CfgAlgo12>(v); }
}  // namespace sg
