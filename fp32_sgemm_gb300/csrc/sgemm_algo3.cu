// Main-kernel instantiation for tile configuration 3: 128 x 128 output tile,
// BK=16, 6 stages, 16-byte A reads, 4 compute warps + 1 TMA producer warp, one CTA per SM.
#include "kernel_table.h"

namespace sg {
using CfgAlgo3 = FfmaConfig<128,128,16,6,2,2,8,1,1,4>;
void fill_algo3(KernelEntry *v) { fill_variants<CfgAlgo3>(v); }
}  // namespace sg
