// Main-kernel instantiation for tile configuration 30: configuration 14
// (128 x 256, 4 stages, C read and written from registers) with 16-byte A
// reads and only the A fragments double buffered (configuration 28's loop).
#include "kernel_table.h"

namespace sg {
using CfgAlgo30 = FfmaConfig<128,256,32,4,2,4,8,4,1,4,0,2>;
void fill_algo30(KernelEntry *v) { fill_variants<CfgAlgo30>(v); }
}  // namespace sg
