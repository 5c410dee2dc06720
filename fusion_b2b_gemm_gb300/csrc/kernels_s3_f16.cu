// Three-stage chain kernels (CTA pairs), fp16 inputs.
#include "registry.h"

namespace b2b {
namespace {
const Chain3Entry kEntries[] = {
    B2B_CHAIN3_ENTRY(kInF16, kOutF16, 128, 128, 128),
    B2B_CHAIN3_ENTRY(kInF16, kOutF16, 128, 128, 256),
    B2B_CHAIN3_ENTRY(kInF16, kOutF16, 128, 256, 128),
    B2B_CHAIN3_ENTRY(kInF16, kOutF16, 128, 256, 256),
    B2B_CHAIN3_ENTRY(kInF16, kOutF16, 256, 128, 128),
    B2B_CHAIN3_ENTRY(kInF16, kOutF16, 256, 128, 256),
    B2B_CHAIN3_ENTRY(kInF16, kOutF16, 256, 256, 128),
    B2B_CHAIN3_ENTRY(kInF16, kOutF16, 256, 256, 256),
    B2B_CHAIN3_ENTRY(kInF16, kOutF32, 128, 128, 128),
    B2B_CHAIN3_ENTRY(kInF16, kOutF32, 128, 128, 256),
    B2B_CHAIN3_ENTRY(kInF16, kOutF32, 128, 256, 128),
    B2B_CHAIN3_ENTRY(kInF16, kOutF32, 128, 256, 256),
    B2B_CHAIN3_ENTRY(kInF16, kOutF32, 256, 128, 128),
    B2B_CHAIN3_ENTRY(kInF16, kOutF32, 256, 128, 256),
    B2B_CHAIN3_ENTRY(kInF16, kOutF32, 256, 256, 128),
    B2B_CHAIN3_ENTRY(kInF16, kOutF32, 256, 256, 256),
};
}  // namespace
Chain3Table chain3_table_f16() { return {kEntries, static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]))}; }
}  // namespace b2b
