// Cascades of 16-bit GEMMs on CTA pairs (chainn_kernel), f16 operands (after a
// tf32 first GEMM in the mixed-type entries).
#include "registry.h"

namespace b2b {
namespace {
const ChainNEntry kEntries[] = {
    B2B_CHAINN_ENTRY(kInF16, kOutF16, 128, false),
    B2B_CHAINN_ENTRY(kInF16, kOutF16, 256, false),
    B2B_CHAINN_ENTRY(kInF16, kOutF32, 128, false),
    B2B_CHAINN_ENTRY(kInF16, kOutF32, 256, false),
    // tf32 first GEMM, f16 after it, fp32 out
    B2B_CHAINN_ENTRY(kInF16, kOutF32, 128, true),
    B2B_CHAINN_ENTRY(kInF16, kOutF32, 256, true),
};
}  // namespace
ChainNTable chainn_table_f16() { return {kEntries, static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]))}; }
}  // namespace b2b
