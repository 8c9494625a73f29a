// Main-kernel instantiation for tile configuration 27: configuration 26
// (128 x 256, 2 stages, C through shared-memory staging) with 16-byte A
// reads and only the A fragments double buffered (configuration 28's loop).
#include "kernel_table.h"

namespace sg {
using CfgAlgo27 = FfmaConfig<128,256,32,2,2,4,8,4,1,4,0,2,0,1,0>;
void fill_algo27(KernelEntry *v) { fill_variants<CfgAlgo27>(v); }
}  // namespace sg
