// Table of compiled tcgen05 chain kernels.  Each kernels_*.cu translation
// unit instantiates a set of chain_tc_kernel specialisations and returns its
// table; the plan picks the entry that matches the padded widths it chose.
#pragma once

#include "chainn.cuh"
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

// Cascades on CTA pairs (chainn_kernel): 16-bit GEMMs in three or more
// stages, or two with an intermediate wider than 256 columns; mixed-type
// cascades; two-GEMM tf32 chains.
struct ChainNEntry {
  int in, out, nf;
  bool tf0;  // first GEMM on tf32 operands (mixed-type cascade)
  const void* fn;
};
struct ChainNTable {
  const ChainNEntry* entries;
  int count;
};
ChainNTable chainn_table_f16();
ChainNTable chainn_table_bf16();
ChainNTable chainn_table_tf32();

}  // namespace b2b

#define B2B_CHAIN_ENTRY(IN, OUT, S, A, B, F, R) \
  { IN, OUT, S, A, B, F, R, reinterpret_cast<const void*>(&::b2b::chain_tc_kernel<IN, OUT, S, A, B, F, R>) }
#define B2B_CHAINN_ENTRY(IN, OUT, F, T) \
  { IN, OUT, F, T, reinterpret_cast<const void*>(&::b2b::chainn_kernel<IN, OUT, F, T>) }
