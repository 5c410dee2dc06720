// Two-GEMM tf32 chains on CTA pairs (chainn_kernel): the intermediate kept in
// tensor memory, fp32 out.
#include "registry.h"

namespace b2b {
namespace {
const ChainNEntry kEntries[] = {
    B2B_CHAINN_ENTRY(kInTF32, kOutF32, 128, true),
    B2B_CHAINN_ENTRY(kInTF32, kOutF32, 256, true),
};
}  // namespace
ChainNTable chainn_table_tf32() { return {kEntries, static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]))}; }
}  // namespace b2b
