// Table of compiled tcgen05 chain kernels.  Each kernels_*.cu translation
// unit instantiates a set of chain_tc_kernel specialisations and returns its
// table; the plan picks the entry that matches the padded widths it chose.
#pragma once

#include "chain3.cuh"
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

// Three-stage 16-bit chains (chain3_kernel, CTA pairs).
struct Chain3Entry {
  int in, out, n1p, n2p, nf;
  const void* fn;
};
struct Chain3Table {
  const Chain3Entry* entries;
  int count;
};
Chain3Table chain3_table_f16();
Chain3Table chain3_table_bf16();

}  // namespace b2b

#define B2B_CHAIN_ENTRY(IN, OUT, S, A, B, F, R) \
  { IN, OUT, S, A, B, F, R, reinterpret_cast<const void*>(&::b2b::chain_tc_kernel<IN, OUT, S, A, B, F, R>) }
#define B2B_CHAIN3_ENTRY(IN, OUT, A, B, F) \
  { IN, OUT, A, B, F, reinterpret_cast<const void*>(&::b2b::chain3_kernel<IN, OUT, A, B, F>) }
