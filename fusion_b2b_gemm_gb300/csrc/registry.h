// Table of compiled tcgen05 chain kernels.  Each kernels_*.cu translation
// unit instantiates a set of chain_tc_kernel specialisations and returns its
// table; the plan picks the entry that matches the padded widths it chose.
#pragma once

#include "chain_tc.cuh"

namespace b2b {

struct ChainKernelEntry {
  int in, out, S, n1p, n2p, nf;
  bool res;
  const void* fn;
};

struct ChainTable {
  const ChainKernelEntry* entries;
  int count;
};

ChainTable chain_table_f16();
ChainTable chain_table_bf16();
ChainTable chain_table_tf32();
ChainTable chain_table_s3_f16();
ChainTable chain_table_s3_bf16();

}  // namespace b2b

#define B2B_CHAIN_ENTRY(IN, OUT, S, A, B, F, R) \
  { IN, OUT, S, A, B, F, R, reinterpret_cast<const void*>(&::b2b::chain_tc_kernel<IN, OUT, S, A, B, F, R>) }
