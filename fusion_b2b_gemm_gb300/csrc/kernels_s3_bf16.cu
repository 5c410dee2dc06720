// Three-stage chain kernels (CTA pairs), bf16 inputs.
#include "registry.h"

namespace b2b {
namespace {
const Chain3Entry kEntries[] = {
    B2B_CHAIN3_ENTRY(kInBF16, kOutBF16, 128, 128, 128),
    B2B_CHAIN3_ENTRY(kInBF16, kOutBF16, 128, 128, 256),
    B2B_CHAIN3_ENTRY(kInBF16, kOutBF16, 128, 256, 128),
    B2B_CHAIN3_ENTRY(kInBF16, kOutBF16, 128, 256, 256),
    B2B_CHAIN3_ENTRY(kInBF16, kOutBF16, 256, 128, 128),
    B2B_CHAIN3_ENTRY(kInBF16, kOutBF16, 256, 128, 256),
    B2B_CHAIN3_ENTRY(kInBF16, kOutBF16, 256, 256, 128),
    B2B_CHAIN3_ENTRY(kInBF16, kOutBF16, 256, 256, 256),
    B2B_CHAIN3_ENTRY(kInBF16, kOutF32, 128, 128, 128),
    B2B_CHAIN3_ENTRY(kInBF16, kOutF32, 128, 128, 256),
    B2B_CHAIN3_ENTRY(kInBF16, kOutF32, 128, 256, 128),
    B2B_CHAIN3_ENTRY(kInBF16, kOutF32, 128, 256, 256),
    B2B_CHAIN3_ENTRY(kInBF16, kOutF32, 256, 128, 128),
    B2B_CHAIN3_ENTRY(kInBF16, kOutF32, 256, 128, 256),
    B2B_CHAIN3_ENTRY(kInBF16, kOutF32, 256, 256, 128),
    B2B_CHAIN3_ENTRY(kInBF16, kOutF32, 256, 256, 256),
};
}  // namespace
Chain3Table chain3_table_bf16() { return {kEntries, static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]))}; }
}  // namespace b2b
