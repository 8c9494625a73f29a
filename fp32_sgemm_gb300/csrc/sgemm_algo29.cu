// Main-kernel instantiation for tile configuration 29: configuration 15
// (256 x 128, 4 stages, C read and written from registers) with 16-byte A
// reads and only the A fragments double buffered (configuration 28's loop).
#include "kernel_table.h"

namespace sg {
using CfgAlgo29 = FfmaConfig<256,128,32,4,4,2,8,4,1,4,0,2>;
void fill_algo29(KernelEntry *v) { fill_variants<CfgAlgo29>(v); }
}  // namespace sg
