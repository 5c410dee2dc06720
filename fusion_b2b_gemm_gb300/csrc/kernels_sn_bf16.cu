// Cascades of 16-bit GEMMs on CTA pairs (chainn_kernel), bf16 inputs.
#include "registry.h"

namespace b2b {
namespace {
const ChainNEntry kEntries[] = {
    B2B_CHAINN_ENTRY(kInBF16, kOutBF16, 128),
    B2B_CHAINN_ENTRY(kInBF16, kOutBF16, 256),
    B2B_CHAINN_ENTRY(kInBF16, kOutF32, 128),
    B2B_CHAINN_ENTRY(kInBF16, kOutF32, 256),
};
}  // namespace
ChainNTable chainn_table_bf16() { return {kEntries, static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]))}; }
}  // namespace b2b
