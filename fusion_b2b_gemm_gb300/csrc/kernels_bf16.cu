// bf16-input tcgen05 chain kernels (bf16 or fp32 output).
#include "registry.h"

namespace b2b {
namespace {
const ChainKernelEntry kEntries[] = {
    // three-stage
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 3, 256, 256, 256, false),
    // single GEMM (unfused reference chain)
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 1, 64, 64, 256, false),
};
}  // namespace
ChainTable chain_table_bf16() { return {kEntries, static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]))}; }
}  // namespace b2b
