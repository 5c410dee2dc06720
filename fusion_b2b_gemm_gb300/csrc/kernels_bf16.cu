// bf16-input tcgen05 chain kernels, one and two stages (bf16 or fp32 output).
#include "registry.h"

namespace b2b {
namespace {
const ChainKernelEntry kEntries[] = {
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 1, 64, 64, 64, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 1, 64, 64, 128, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 1, 64, 64, 256, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 1, 64, 64, 64, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 1, 64, 64, 128, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 1, 64, 64, 256, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 64, 64, 64, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 64, 64, 128, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 64, 64, 256, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 128, 64, 64, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 128, 64, 128, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 128, 64, 256, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 256, 64, 64, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 256, 64, 128, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 256, 64, 256, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 64, 64, 64, true),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 64, 64, 128, true),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 128, 64, 64, true),
    B2B_CHAIN_ENTRY(kInBF16, kOutBF16, 2, 128, 64, 128, true),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 64, 64, 64, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 64, 64, 128, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 64, 64, 256, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 128, 64, 64, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 128, 64, 128, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 128, 64, 256, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 256, 64, 64, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 256, 64, 128, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 256, 64, 256, false),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 64, 64, 64, true),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 64, 64, 128, true),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 128, 64, 64, true),
    B2B_CHAIN_ENTRY(kInBF16, kOutF32, 2, 128, 64, 128, true),
};
}  // namespace
ChainTable chain_table_bf16() { return {kEntries, static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]))}; }
}  // namespace b2b
