// Main-kernel instantiation for tile configuration 11: configuration 10
// (128 x 128 tile, BK=32, 3 stages, TMA issued by thread 0, double-buffered
// 8-byte A fragments, 2 CTAs/SM) with scalar FP32 FMAs instead of packed
// two-wide ones.
#include "kernel_table.h"

namespace sg {
using CfgAlgo11 = FfmaConfig<128,128,32,3,2,2,8,4,2,2,0,1,1>;
void fill_algo11(KernelEntry *v) { fill_variants<CfgAlgo11>(v); }
}  // namespace sg
