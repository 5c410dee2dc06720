// fp16-input tcgen05 chain kernels, one and two stages (fp32 or fp16 output).
#include "registry.h"

namespace b2b {
namespace {
const ChainKernelEntry kEntries[] = {
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 1, 64, 64, 64, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 1, 64, 64, 128, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 1, 64, 64, 256, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 1, 64, 64, 64, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 1, 64, 64, 128, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 1, 64, 64, 256, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 64, 64, 64, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 64, 64, 128, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 64, 64, 256, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 128, 64, 64, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 128, 64, 128, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 128, 64, 256, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 256, 64, 64, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 256, 64, 128, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 256, 64, 256, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 64, 64, 64, true),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 64, 64, 128, true),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 128, 64, 64, true),
    B2B_CHAIN_ENTRY(kInF16, kOutF32, 2, 128, 64, 128, true),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 64, 64, 64, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 64, 64, 128, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 64, 64, 256, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 128, 64, 64, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 128, 64, 128, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 128, 64, 256, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 256, 64, 64, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 256, 64, 128, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 256, 64, 256, false),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 64, 64, 64, true),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 64, 64, 128, true),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 128, 64, 64, true),
    B2B_CHAIN_ENTRY(kInF16, kOutF16, 2, 128, 64, 128, true),
};
}  // namespace
ChainTable chain_table_f16() { return {kEntries, static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]))}; }
}  // namespace b2b
