// Main-kernel instantiation for tile configuration 1: 128 x 128 output tile,
// BK=32, 4 stages, 16-byte A reads, 4 compute warps + 1 TMA producer warp, one CTA per SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo1 = FfmaConfig<128,128,32,4,2,2,8,1,1,4>;
void fill_algo1(KernelEntry *v) { fill_variants<CfgAlgo1>(v); }
}  // namespace sg
