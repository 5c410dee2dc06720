// Fused cascaded GEMM on the 5th-generation tensor cores (tcgen05), sm_103a.
//
//   P1 = A.W0  ->  rearrange/round  ->  P2 = P1.W1  [->  rearrange  ->  E = P2.W2]
//
// Source of the method: patent "数据处理方法、装置、设备及介质" (Alibaba, 2023),
// Detailed description para. 35-37 (steps 101-103), para. 54-60 (the result
// of operator 1 is held by rule 1, rearranged, and handed to operator 2 by
// rule 2 without going through memory), para. 103-110 (rearrangement through
// shared memory) and para. 41 (three cascaded operators).
//
// On this hardware rule 1 is the tcgen05 accumulator layout in tensor memory
// (row m of the 128-row tile in TMEM lane m, column n in TMEM column n, fp32)
// and rule 2 is the K-major 128-byte-swizzled shared-memory operand image that
// a tcgen05.mma A-descriptor reads.  Because a row stays in one lane, the
// rearrangement needs no cross-thread exchange: each converter thread loads
// its row with tcgen05.ld, rounds it to the operand type and writes it into
// the swizzled image with 16-byte st.shared.  For tf32 the rounded operand is
// written back into the accumulator's own columns (tcgen05.st), because the
// tf32 MMA can take its A operand from tensor memory, where the layout of
// rule 2 equals rule 1.
//
// CTA roles (352 threads, one CTA per SM, persistent over 128-row tiles):
//   warp 0     TMA producer: A panels and weight panels into a ring of stages
//   warp 1     TMEM allocator and the MMA-issuing thread (GEMM1 only when the
//              weights are resident; then warp 10 issues GEMM2)
//   warps 2-5  converters: accumulator -> operand (the rearrangement)
//   warps 6-9  epilogue: accumulator -> output type -> swizzled staging -> TMA store
//   warp 10    second MMA-issuing thread (resident-weight chains), or the
//              producer of the A ring (streamed weights: the A panels have a
//              ring of their own, so that the next tile's A is read from HBM
//              while the current tile's later GEMMs run)
// Every wait is bounded (ptx::BoundedWait); on a timeout the CTA raises an
// abort flag, every role leaves its loop, in-flight copies and MMAs are
// drained, tensor memory is freed and the status word reports the timeout.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

namespace b2b {

enum : int { kInF16 = 0, kInBF16 = 1, kInTF32 = 2 };
enum : int { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2 };

constexpr int kChainThreads = 352;
constexpr int kPanelBytes = 128 * 128;  // one 128-row x 128-byte swizzled panel
constexpr int kBarBytes = 512;
constexpr int kTimeoutCode = 7;         // B2B_ERR_TIMEOUT

// Barrier slots (8 bytes each) at ChainParams::off_bar.
enum : int {
  kBarFull = 0,     // [8] ring stage filled by TMA
  kBarEmpty = 8,    // [8] ring stage consumed by the MMAs
  kBarWFull = 16,   // resident weights landed
  kBarWEmpty = 17,  // resident weights no longer read
  kBarRFull = 18,   // [4] region holds a final product for the epilogue
  kBarREmpty = 22,  // [4] tensor-memory region drained by a warpgroup
  kBarPFull = 26,   // operand image of the intermediate written
  kBarPEmpty = 27,  // operand image of the intermediate no longer read
  kBarEpiSync = 28,
  kBarDrain = 29,
  kBarCFull = 30,   // [2] region X / Y holds an intermediate for the converters
  kBarDrain2 = 32,
  kBarPFull1 = 33,  // second operand image (double-buffered intermediate)
  kBarPEmpty1 = 34,
  kSlotTmem = 35,   // uint32 TMEM base address, then the int abort flag
  kBarAFull = 36,   // [8] A-ring stage filled by TMA (streamed weights)
  kBarAEmpty = 44,  // [8] A-ring stage consumed by the MMAs
};
// Each consumer warpgroup has its own "full" barrier per region, so that it
// sees every completion of that barrier in order: when the last GEMM reuses
// X and Y, the converters and the epilogue take turns on the same region,
// and a parity wait could not tell a waiter's own phase from the other's.

struct ChainParams {
  int batch, M, K;
  int m_tiles, total_tiles;
  int npass;          // passes of the final GEMM (NF columns each)
  int kpan0;          // 128-byte K panels of A (ceil(K / panel width))
  int nst;            // ring depth (weight panels when streamed, A tiles when resident)
  int nsta;           // streamed weights: depth of the separate ring of A panels (0: A shares
                      // each GEMM1 stage with its weight panel)
  int nstg;           // output staging buffers (1 or 2)
  uint32_t off_ring, stage_bytes, off_aring, off_wres0, off_wres1, off_p, off_stg, off_bar;
  uint32_t tmem_cols;
  int region_col[4];  // X, Y, Z0, Z1 (TMEM column offsets)
  int nz;             // Z buffers for the final accumulator; 0 = reuse X/Y in turn
  int lookahead;      // two-stage only: GEMM1 double-buffered (X, Y) and issued a tile ahead
  int dbl_p;          // two operand buffers for the intermediate (tile parity), own barriers
  uint32_t p_bytes;   // bytes of one shared-memory operand image (0: kept in tensor memory)
  int p_tmem;         // 16-bit intermediate kept in tensor memory (tf32 always is)
  int w_merged;       // bit s: weight s is mapped 4-D (128-byte column blocks, K, blocks,
                      // batch), so a whole panel (all its column blocks) arrives as one TMA box
  int w_kmajor;       // tf32 only: the weights arrive transposed ([N][K], K-major) instead of
                      // as stored ([K][N], MN-major with 32-byte swizzle atoms)
  uint32_t debug;     // test support: bit 0 = arm the first ring stage but never fill it
  int* status;
  unsigned long long budget_ns;
  // Resident weights: optional tile schedule, kSchedStride ints per CTA:
  // the number of segments, then (first tile, tile count) of each, tiles
  // numbered batch-major; null = one contiguous range per CTA.
  const int* sched;
};
constexpr int kSchedSegs = 4;
constexpr int kSchedStride = 1 + 2 * kSchedSegs;

// Which tensor-memory region phase `ph` of local tile `it` writes, and how
// many times that region has been written before (its use index, which the
// MMA thread waits on through the region's "empty" barrier).
// Phases 0..S-2 are the intermediate GEMMs (X, then Y); the rest are the
// passes of the final GEMM (Z buffers in turn, or X/Y in turn when nz == 0).
__host__ __device__ __forceinline__ void region_use(const ChainParams& p, int S, int it, int ph,
                                                    int& r, uint32_t& u) {
  const int ux = 1 + (p.npass + 1) / 2, uy = 1 + p.npass / 2;
  if (p.lookahead && ph == 0) {  // GEMM1 alternates between two buffers
    r = it & 1;
    u = static_cast<uint32_t>(it) >> 1;
    return;
  }
  if (ph < S - 1) {
    r = ph;
    u = (p.nz > 0) ? static_cast<uint32_t>(it)
                   : static_cast<uint32_t>(it) * static_cast<uint32_t>(ph == 0 ? ux : uy);
    return;
  }
  const int pass = ph - (S - 1);
  if (p.nz > 0) {
    const uint32_t g = static_cast<uint32_t>(it) * p.npass + pass;
    r = 2 + static_cast<int>(g % p.nz);
    u = g / p.nz;
  } else {
    r = pass & 1;
    u = static_cast<uint32_t>(it) * static_cast<uint32_t>(r == 0 ? ux : uy) + 1 + pass / 2;
  }
}

// ------------------------------------------------------------ rearrangement
// One converter thread holds 32 consecutive fp32 accumulator columns
// [c0, c0 + 32) of its row.  Round them to the operand type and store them
// into the K-major 128B-swizzled operand image at `img` (panels of 128 rows x
// 128 bytes): 16-byte unit u of row r lands at unit u ^ (r % 8).
template <int IN>
__device__ __forceinline__ void store_operand_row(uint32_t img, int row, int c0,
                                                  const uint32_t (&v)[32]) {
  using namespace ptx;
  const uint32_t sw = static_cast<uint32_t>(row & 7);
  if constexpr (IN == kInTF32) {
    const uint32_t rbase = img + static_cast<uint32_t>(c0 / 32) * kPanelBytes + row * 128u;
#pragma unroll
    for (uint32_t u = 0; u < 8; ++u)
      st_shared_v4(rbase + ((u ^ sw) << 4), to_tf32_rna(v[4 * u]), to_tf32_rna(v[4 * u + 1]),
                   to_tf32_rna(v[4 * u + 2]), to_tf32_rna(v[4 * u + 3]));
  } else {
    const uint32_t rbase = img + static_cast<uint32_t>(c0 / 64) * kPanelBytes + row * 128u;
    const uint32_t unit0 = static_cast<uint32_t>((c0 % 64) / 8);
#pragma unroll
    for (uint32_t u = 0; u < 4; ++u) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = (IN == kInF16) ? pack_f16x2(v[8 * u + 2 * i], v[8 * u + 2 * i + 1])
                              : pack_bf16x2(v[8 * u + 2 * i], v[8 * u + 2 * i + 1]);
      st_shared_v4(rbase + (((unit0 + u) ^ sw) << 4), w[0], w[1], w[2], w[3]);
    }
  }
}

// Output staging: 32 fp32 accumulator columns [c, c + 32) of a store box
// (128 bytes wide) -> output type -> 128B-swizzled box image.
template <int OUT>
__device__ __forceinline__ void store_output_row(uint32_t img, int row, int c,
                                                 const uint32_t (&v)[32]) {
  using namespace ptx;
  const uint32_t sw = static_cast<uint32_t>(row & 7);
  const uint32_t rbase = img + row * 128u;
  if constexpr (OUT == kOutF32) {
#pragma unroll
    for (uint32_t u = 0; u < 8; ++u)
      st_shared_v4(rbase + ((u ^ sw) << 4), v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
  } else {
    const uint32_t unit0 = static_cast<uint32_t>(c / 8);
#pragma unroll
    for (uint32_t u = 0; u < 4; ++u) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = (OUT == kOutF16) ? pack_f16x2(v[8 * u + 2 * i], v[8 * u + 2 * i + 1])
                                : pack_bf16x2(v[8 * u + 2 * i], v[8 * u + 2 * i + 1]);
      st_shared_v4(rbase + (((unit0 + u) ^ sw) << 4), w[0], w[1], w[2], w[3]);
    }
  }
}

// The rearrangement of one accumulator row (step 103 on this hardware).
// `tsrc` is the TMEM address of this warp's lane quadrant at the first
// accumulator column; the thread owns row `row` of the tile.  16-bit types:
// round and store into the swizzled shared-memory operand image `p_img`.
// tf32: round in place; the MMA then reads the operand from tensor memory.
template <int IN>
__device__ __forceinline__ void rearrange_accumulator(uint32_t tsrc, int width, int row,
                                                      uint32_t p_img) {
  using namespace ptx;
  // two 32-column loads in flight per wait (widths are multiples of 64)
#pragma unroll 1
  for (int c0 = 0; c0 < width; c0 += 64) {
    uint32_t v0[32], v1[32];
    tmem_ld32(tsrc + static_cast<uint32_t>(c0), v0);
    tmem_ld32(tsrc + static_cast<uint32_t>(c0 + 32), v1);
    tmem_wait_ld();
    if constexpr (IN == kInTF32) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v0[i] = to_tf32_rna(v0[i]);
        v1[i] = to_tf32_rna(v1[i]);
      }
      tmem_st32(tsrc + static_cast<uint32_t>(c0), v0);
      tmem_st32(tsrc + static_cast<uint32_t>(c0 + 32), v1);
    } else {
      store_operand_row<IN>(p_img, row, c0, v0);
      store_operand_row<IN>(p_img, row, c0 + 32, v1);
    }
  }
  if constexpr (IN == kInTF32) {
    tmem_wait_st();
  } else {
    fence_proxy_async_smem();
  }
}

// 16-bit intermediate kept in tensor memory as the A operand of the next
// GEMM: the accumulator row is rounded and packed in place, two K elements
// per 32-bit column (even K in the low half), so `width` columns of fp32 at
// tsrc become width/2 columns of the operand at tdst (tdst <= tsrc, in the
// same lanes).  Chunk c0 is read before its packed form is written to
// columns [tdst + c0/2, tdst + c0/2 + 32), which never reach an unread chunk.
template <int IN>
__device__ __forceinline__ void rearrange_accumulator_tmem16(uint32_t tsrc, int width, uint32_t tdst) {
  using namespace ptx;
#pragma unroll 1
  for (int c0 = 0; c0 < width; c0 += 64) {
    uint32_t v0[32], v1[32], w[32];
    tmem_ld32(tsrc + static_cast<uint32_t>(c0), v0);
    tmem_ld32(tsrc + static_cast<uint32_t>(c0 + 32), v1);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      w[i] = (IN == kInF16) ? pack_f16x2(v0[2 * i], v0[2 * i + 1]) : pack_bf16x2(v0[2 * i], v0[2 * i + 1]);
      w[16 + i] =
          (IN == kInF16) ? pack_f16x2(v1[2 * i], v1[2 * i + 1]) : pack_bf16x2(v1[2 * i], v1[2 * i + 1]);
    }
    tmem_st32(tdst + static_cast<uint32_t>(c0 / 2), w);
  }
  tmem_wait_st();
}
template <int IN>
__device__ __forceinline__ void rearrange_accumulator_tmem16(uint32_t tsrc, int width) {
  rearrange_accumulator_tmem16<IN>(tsrc, width, tsrc);
}

// Warp-uniform bounded wait: the warp goes on only if every lane saw the phase.
__device__ __forceinline__ bool warp_wait(const ptx::BoundedWait& bw, uint32_t bar,
                                          uint32_t parity) {
  const bool ok = bw.wait(bar, parity);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Barrier among the 128 threads of one warpgroup, built on an mbarrier so
// that it is bounded like every other wait.
__device__ __forceinline__ bool group_sync(const ptx::BoundedWait& bw, uint32_t bar,
                                           uint32_t& uses) {
  ptx::mbar_arrive(bar);
  const bool ok = warp_wait(bw, bar, uses & 1u);
  ++uses;
  return ok;
}

// Wait used while draining after an abort: ignores the abort flag (the copy
// or MMA being waited for completes on its own) but still has a budget.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t budget_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > budget_ns) return;
  }
}

// Tiles of one CTA, walked without divisions: batch b and 128-row tile mt.
// A scheduled CTA walks a list of contiguous segments instead (`segs`: tile
// count of the current one in `left`, then (first, count) pairs).
struct TileCursor {
  int b, mt, db, dmt, m_tiles;
  int left, seg, nseg;
  const int* segs;
  __device__ __forceinline__ void init(int tile, int step, int mtiles) {
    m_tiles = mtiles;
    b = tile / mtiles;
    mt = tile - b * mtiles;
    db = step / mtiles;
    dmt = step - db * mtiles;
    segs = nullptr;
  }
  __device__ __forceinline__ void init_segments(const int* s, int n, int mtiles) {
    init(n > 0 ? s[0] : 0, 1, mtiles);
    segs = s;
    nseg = n;
    seg = 0;
    left = n > 0 ? s[1] : 0;
  }
  __device__ __forceinline__ void next() {
    if (segs != nullptr && --left == 0) {
      if (++seg < nseg) {
        const int t = segs[2 * seg];
        b = t / m_tiles;
        mt = t - b * m_tiles;
        left = segs[2 * seg + 1];
      }
      return;
    }
    mt += dmt;
    b += db;
    if (mt >= m_tiles) {
      mt -= m_tiles;
      ++b;
    }
  }
};

template <int IN, int OUT, int S, int N1P, int N2P, int NF, bool RES>
__global__ void __launch_bounds__(kChainThreads, 1)
    chain_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmW0,
                    const __grid_constant__ CUtensorMap tmW1,
                    const __grid_constant__ CUtensorMap tmW2,
                    const __grid_constant__ CUtensorMap tmOut,
                    const __grid_constant__ ChainParams p) {
  using namespace ptx;
  constexpr bool TF32 = (IN == kInTF32);
  constexpr int ESZ = TF32 ? 4 : 2;
  constexpr int OSZ = (OUT == kOutF32) ? 4 : 2;
  constexpr int CK = 128 / ESZ;       // K elements per 128-byte panel
  constexpr int KSTEP = 32 / ESZ;     // K of one tcgen05.mma
  constexpr int WBOX_N = 128 / ESZ;   // weight columns per TMA box
  constexpr int WBOX_BYTES = CK * 128;
  constexpr int OBOX_N = 128 / OSZ;   // output columns per TMA store box
  constexpr bool P_TMEM = TF32;
  // Weights are read as stored ([K][N]: an MN-major B operand), in blocks of
  // 128 bytes of N (64 16-bit or 32 tf32 columns) by K rows.  16-bit blocks
  // use the 128-byte swizzle; tf32 blocks the 128-byte swizzle of 32-byte
  // atoms, the only MN-major form the tf32 MMA reads.  With w_kmajor (tf32
  // only) the weights arrive transposed instead ([N][K], K-major).
  const bool W_KMAJOR = TF32 && p.w_kmajor != 0;
  // With resident weights (16-bit), GEMM1 and GEMM2 are issued by two
  // threads (warps 1 and 10): the tensor pipe holds little more than the MMA
  // being executed, so every wait of a single issuing thread would leave it
  // idle; with two issuers one waits while the other issues.
  constexpr bool SPLIT = RES && !TF32;
  constexpr uint32_t FMT = (IN == kInF16) ? 0u : (IN == kInBF16 ? 1u : 2u);
  constexpr int NPH_FIXED = S - 1;    // intermediate phases per tile
  static_assert(S >= 1 && S <= 3, "one to three cascaded GEMMs");
  static_assert(!(TF32 && S == 3), "tf32 chains have two stages");
  static_assert(!RES || S == 2, "resident weights only for two-stage chains");
  static_assert(N1P % 64 == 0 && N2P % 64 == 0 && NF % 64 == 0, "panel widths");
  static_assert(N1P <= 256 && N2P <= 256 && NF <= 256, "one MMA covers at most 256 columns");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + p.off_bar;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + p.off_bar + 8 * kSlotTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Tiles of this CTA: a contiguous range when the weights stay resident
  // (few batch changes), otherwise strided so that concurrent CTAs share the
  // same weights in L2.
  int t_begin, t_step, t_count;
  const int* my_segs = nullptr;
  int my_nseg = 0;
  if constexpr (RES) {
    if (p.sched != nullptr) {
      // a schedule that keeps most CTAs within one batch (see the plan)
      my_segs = p.sched + blockIdx.x * kSchedStride + 1;
      my_nseg = p.sched[blockIdx.x * kSchedStride];
      t_count = 0;
      for (int i = 0; i < my_nseg; ++i) t_count += my_segs[2 * i + 1];
      t_begin = my_nseg > 0 ? my_segs[0] : 0;
      t_step = 1;
    } else {
      const long long T = p.total_tiles, G = gridDim.x;
      const int b0 = static_cast<int>((blockIdx.x * T) / G);
      const int b1 = static_cast<int>(((blockIdx.x + 1) * T) / G);
      t_begin = b0;
      t_step = 1;
      t_count = b1 - b0;
    }
  } else {
    t_begin = blockIdx.x;
    t_step = gridDim.x;
    t_count = (static_cast<int>(blockIdx.x) < p.total_tiles)
                  ? (p.total_tiles - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x
                  : 0;
  }
  TileCursor first;
  if (my_segs != nullptr)
    first.init_segments(my_segs, my_nseg, p.m_tiles);
  else
    first.init(t_begin, t_step, p.m_tiles);
  // Everything up to the dependency wait may overlap the previous kernel in
  // the stream: it reads only the plan's own tile schedule.  Before waiting
  // for that kernel, and while the other warps set up barriers and tensor
  // memory, one thread pulls this CTA's first A tile into L2 (measured: the
  // TMA prefetch instructions of a tile take about half a microsecond to
  // issue).  A may be that kernel's output, but a prefetch touches L2 only,
  // where its writes land too, and every load into shared memory comes after
  // the wait, so no stale value is read.
  if (warp == 3 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmW0);
    if (S >= 2) prefetch_tmap(&tmW1);
    if (S >= 3) prefetch_tmap(&tmW2);
    prefetch_tmap(&tmOut);
  }
  if (warp == 3 && lane == 0 && t_count > 0) {
    for (int kb = 0; kb < p.kpan0; ++kb) tma_prefetch_l2_3d(&tmA, kb * CK, first.mt * 128, first.b);
    if constexpr (RES) {
      // the weights of the first batch, and the second tile's A
      const int b = first.b;
      for (int kb = 0; kb < p.kpan0; ++kb) {
        if (W_KMAJOR)
          tma_prefetch_l2_3d(&tmW0, kb * CK, 0, b);
        else if (p.w_merged & 1)
          tma_prefetch_l2_4d(&tmW0, 0, kb * CK, 0, b);
        else
          for (int j = 0; j < N1P / WBOX_N; ++j) tma_prefetch_l2_3d(&tmW0, j * WBOX_N, kb * CK, b);
      }
      for (int kb = 0; kb < N1P / CK; ++kb) {
        if (W_KMAJOR)
          tma_prefetch_l2_3d(&tmW1, kb * CK, 0, b);
        else if (p.w_merged & 2)
          tma_prefetch_l2_4d(&tmW1, 0, kb * CK, 0, b);
        else
          for (int j = 0; j < NF / WBOX_N; ++j) tma_prefetch_l2_3d(&tmW1, j * WBOX_N, kb * CK, b);
      }
      if (t_count > 1) {
        TileCursor second = first;
        second.next();
        for (int kb = 0; kb < p.kpan0; ++kb) tma_prefetch_l2_3d(&tmA, kb * CK, second.mt * 128, second.b);
      }
    }
  }
  // Barriers, set up by the lanes of warp 0 in parallel (each lane fences
  // its own initialisations), while warp 1 allocates tensor memory.
  if (warp == 0) {
    if (lane < 8) {
      mbar_init(bar(kBarFull + lane), 1);
      mbar_init(bar(kBarEmpty + lane), 1);
      mbar_init(bar(kBarAFull + lane), 1);
      mbar_init(bar(kBarAEmpty + lane), 1);
    } else if (lane < 12) {
      mbar_init(bar(kBarRFull + lane - 8), 1);
      mbar_init(bar(kBarREmpty + lane - 8), 128);
    } else if (lane == 12) {
      mbar_init(bar(kBarWFull), 1);
      mbar_init(bar(kBarWEmpty), SPLIT ? 2 : 1);
      mbar_init(bar(kBarCFull), 1);
      mbar_init(bar(kBarCFull + 1), 1);
    } else if (lane == 13) {
      mbar_init(bar(kBarPFull), 128);
      mbar_init(bar(kBarPEmpty), 1);
      mbar_init(bar(kBarPFull1), 128);
      mbar_init(bar(kBarPEmpty1), 1);
    } else if (lane == 14) {
      mbar_init(bar(kBarEpiSync), 128);
      mbar_init(bar(kBarDrain), 1);
      mbar_init(bar(kBarDrain2), 1);
      *abort_flag = 0;
    }
    if (lane < 15) fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  BoundedWait bw{abort_flag, p.status, p.budget_ns, kTimeoutCode};
  // L2 policy of the streams read or written once (resident-weight A tiles,
  // the output)
  const uint64_t pol_stream = l2_policy_evict_first();

  grid_launch_dependents();
  grid_dependency_wait();
  const int nph = NPH_FIXED + p.npass;
  const bool lookahead = p.lookahead != 0;
  // streamed weights with CTAs that run several tiles: A panels come through
  // a ring of their own (warp 10), so the next tile's A is read from HBM
  // while this tile's later GEMMs run
  const bool split_a = !RES && p.nsta > 0;

  auto stage_width = [](int s) -> int { return s < S - 1 ? (s == 0 ? N1P : N2P) : NF; };
  auto stage_kpan = [&](int s) -> int { return s == 0 ? p.kpan0 : (s == 1 ? N1P / CK : N2P / CK); };
  // With resident weights the ring carries whole A tiles (kpan0 panels per
  // stage); otherwise one panel (A and/or weight) per stage.
  auto panels_per_stage = [&](int s) -> int { return (RES && s == 0) ? p.kpan0 : 1; };
  // Final-pass region index without divisions (nz is 1 or 2).
  auto zregion = [&](int it, int pass, int& r, uint32_t& u) {
    const uint32_t g = static_cast<uint32_t>(it) * static_cast<uint32_t>(p.npass) + pass;
    r = 2 + ((p.nz == 2) ? static_cast<int>(g & 1u) : 0);
    u = (p.nz == 2) ? (g >> 1) : g;
  };

  // Order in which the producer loads and a single MMA thread computes the
  // phases.  Plain order: every phase of tile 0, then of tile 1, ...  With
  // lookahead (two-stage chains whose first accumulator is double-buffered in
  // tensor memory), GEMM1 of tile it+1 comes before GEMM2 of tile it.  Across a
  // change of batch with resident weights there is no lookahead: the new
  // weights may only land after GEMM2 of the old batch.
  auto for_each_phase = [&](auto&& fn) {
    TileCursor cur = first;
    if (!lookahead) {
      for (int it = 0; it < t_count; ++it, cur.next())
        for (int ph = 0; ph < nph; ++ph)
          if (!fn(it, ph, cur)) return;
      return;
    }
    TileCursor nxt = first;
    if (t_count > 0 && !fn(0, 0, cur)) return;
    nxt.next();
    for (int it = 0; it < t_count; ++it, cur.next(), nxt.next()) {
      const bool more = it + 1 < t_count;
      const bool ahead = more && (!RES || nxt.b == cur.b);
      if (ahead && !fn(it + 1, 0, nxt)) return;
      for (int ph = 1; ph < nph; ++ph)
        if (!fn(it, ph, cur)) return;
      if (!ahead && more && !fn(it + 1, 0, nxt)) return;
    }
  };

  // One GEMM phase issued by the calling thread: operands from the ring
  // and/or resident weights and/or the intermediate, accumulator in region r.
  // `stage`/`phase` track the ring; returns false on abort.
  auto issue_phase = [&](int it, int ph, int r, uint32_t& stage, uint32_t& phase, uint32_t& astage,
                         uint32_t& aphase) -> bool {
    const int s = ph < S - 1 ? ph : S - 1;
    const int width = stage_width(s);
    const int kpan = stage_kpan(s);
    const int ppst = panels_per_stage(s);
    const bool ring = (s == 0) || !RES;
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(p.region_col[r]);
    const uint32_t idesc = make_idesc(FMT, static_cast<uint32_t>(width), 128u, !W_KMAJOR);
    const uint32_t wres = (s == 0) ? p.off_wres0 : p.off_wres1;
    // the operand of a later stage: which region holds the intermediate
    const uint32_t a_tmem =
        tmem_base + static_cast<uint32_t>(p.region_col[(lookahead && s >= 1) ? (it & 1) : 0]);
    const uint32_t p_img = base + p.off_p + ((p.dbl_p && (it & 1)) ? p.p_bytes : 0u);
    const bool a_in_tmem = P_TMEM || p.p_tmem;
    int kin = 0;
    for (int kb = 0; kb < kpan; ++kb) {
      const uint32_t sbase = base + p.off_ring + stage * p.stage_bytes;
      if (ring && kin == 0) {
        if (!bw.wait(bar(kBarFull + stage), phase)) return false;
        if (split_a && s == 0 && !bw.wait(bar(kBarAFull + astage), aphase)) return false;
        tc_fence_after();
      }
      // resident weights: the stage is a whole A tile; streamed: the stage is
      // one weight panel, with A from its own ring or (GEMM1 without an A
      // ring) in front of the weight panel
      const uint32_t sa = RES ? sbase + static_cast<uint32_t>(kin) * kPanelBytes
                              : (split_a ? base + p.off_aring + astage * static_cast<uint32_t>(kPanelBytes) : sbase);
      const uint32_t b_base = RES ? base + wres + static_cast<uint32_t>(kb) * 128u * width
                                  : sbase + (split_a || s != 0 ? 0u : static_cast<uint32_t>(kPanelBytes));
      // B descriptor of the panel's first K step and its increment per step
      // (the start address field counts 16-byte units; a K step moves
      // KSTEP rows of 128 bytes, or 32 bytes along a K-major row)
      uint64_t bd0;
      uint32_t bstep;
      if constexpr (TF32) {
        bd0 = W_KMAJOR ? desc_sw128(b_base, 16u, 1024u) : desc_mn32(b_base, WBOX_BYTES, 512u);
        bstep = W_KMAJOR ? 2u : (KSTEP * 128u) >> 4;
      } else {
        bd0 = desc_sw128(b_base, WBOX_BYTES, 1024u);
        bstep = (KSTEP * 128u) >> 4;
      }
      auto bdesc = [&](int kk) -> uint64_t { return bd0 + static_cast<uint64_t>(kk) * bstep; };
      const uint32_t acc0 = kb != 0 ? 1u : 0u;
      // The MMAs of one panel are issued back to back, with the choice of
      // operand source made once per panel: a branch between consecutive
      // tcgen05.mma instructions was measured to cost a third of the
      // tensor-pipe rate (M=128, N=256: 171 instead of 128 cycles per MMA).
      if (s == 0) {
#pragma unroll
        for (int kk = 0; kk < CK / KSTEP; ++kk)
          mma_ss<TF32>(d_tmem, desc_sw128(sa + kk * 32u, 16u, 1024u), bdesc(kk), idesc, kk ? 1u : acc0);
      } else if (a_in_tmem) {
        // 32 bits per column: one tf32 element or two 16-bit elements of K
        const uint32_t ak = a_tmem + static_cast<uint32_t>(kb * CK * ESZ / 4);
#pragma unroll
        for (int kk = 0; kk < CK / KSTEP; ++kk)
          mma_ts<TF32>(d_tmem, ak + static_cast<uint32_t>(kk * KSTEP * ESZ / 4), bdesc(kk), idesc,
                       kk ? 1u : acc0);
      } else {
        const uint32_t pk = p_img + static_cast<uint32_t>(kb) * kPanelBytes;
#pragma unroll
        for (int kk = 0; kk < CK / KSTEP; ++kk)
          mma_ss<TF32>(d_tmem, desc_sw128(pk + kk * 32u, 16u, 1024u), bdesc(kk), idesc, kk ? 1u : acc0);
      }
      if (ring && ++kin == ppst) {
        kin = 0;
        tc_commit(bar(kBarEmpty + stage));
        if (++stage == static_cast<uint32_t>(p.nst)) {
          stage = 0;
          phase ^= 1u;
        }
        if (split_a && s == 0) {
          tc_commit(bar(kBarAEmpty + astage));
          if (++astage == static_cast<uint32_t>(p.nsta)) {
            astage = 0;
            aphase ^= 1u;
          }
        }
      }
    }
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmW0);
      if (S >= 2) prefetch_tmap(&tmW1);
      if (S >= 3) prefetch_tmap(&tmW2);
      prefetch_tmap(&tmOut);
      uint32_t stage = 0, phase = 0, wl = 0;
      uint64_t issued = 0;
      int cur_b = -1;
      for_each_phase([&](int it, int ph, const TileCursor& c) -> bool {
        const int b = c.b;
        const int m0 = c.mt * 128;
        if constexpr (RES) {
          if (ph == 0 && b != cur_b) {
            if (wl > 0 && !bw.wait(bar(kBarWEmpty), (wl - 1) & 1u)) return false;
            const uint32_t bytes = static_cast<uint32_t>(p.kpan0) * 128u * N1P +
                                   static_cast<uint32_t>(N1P / CK) * 128u * NF;
            mbar_arrive_expect_tx(bar(kBarWFull), bytes);
            for (int kb = 0; kb < p.kpan0; ++kb) {
              const uint32_t dst = base + p.off_wres0 + kb * 128u * N1P;
              if (W_KMAJOR) {
                tma_load_3d(dst, &tmW0, bar(kBarWFull), kb * CK, 0, b);
              } else if (p.w_merged & 1) {
                tma_load_4d(dst, &tmW0, bar(kBarWFull), 0, kb * CK, 0, b);
              } else {
                for (int j = 0; j < N1P / WBOX_N; ++j)
                  tma_load_3d(dst + j * WBOX_BYTES, &tmW0, bar(kBarWFull), j * WBOX_N, kb * CK, b);
              }
            }
            for (int kb = 0; kb < N1P / CK; ++kb) {
              const uint32_t dst = base + p.off_wres1 + kb * 128u * NF;
              if (W_KMAJOR) {
                tma_load_3d(dst, &tmW1, bar(kBarWFull), kb * CK, 0, b);
              } else if (p.w_merged & 2) {
                tma_load_4d(dst, &tmW1, bar(kBarWFull), 0, kb * CK, 0, b);
              } else {
                for (int j = 0; j < NF / WBOX_N; ++j)
                  tma_load_3d(dst + j * WBOX_BYTES, &tmW1, bar(kBarWFull), j * WBOX_N, kb * CK, b);
              }
            }
            cur_b = b;
            ++wl;
          }
        }
        const int s = ph < S - 1 ? ph : S - 1;
        if (RES && s != 0) return true;
        const int width = stage_width(s);
        const int n0 = ph < S - 1 ? 0 : (ph - (S - 1)) * NF;
        const int kpan = stage_kpan(s);
        const int ppst = panels_per_stage(s);
        const CUtensorMap* wm = s == 0 ? &tmW0 : (s == 1 ? &tmW1 : &tmW2);
        for (int kb0 = 0; kb0 < kpan; kb0 += ppst) {
          if (!bw.wait(bar(kBarEmpty + stage), phase ^ 1u)) return false;
          const uint32_t dst = base + p.off_ring + stage * p.stage_bytes;
          // (resident weights: the stage is an A tile; streamed: a weight panel,
          // behind its A panel in GEMM1 stages when A has no ring of its own)
          const bool a_here = !RES && !split_a && s == 0;
          const uint32_t wofs = a_here ? static_cast<uint32_t>(kPanelBytes) : 0u;
          const uint32_t bytes = RES ? kPanelBytes * static_cast<uint32_t>(ppst)
                                     : 128u * static_cast<uint32_t>(width) + wofs;
          const uint32_t fb = bar(kBarFull + stage);
          mbar_arrive_expect_tx(fb, bytes);
          // test support: the very first stage is armed but never filled, so
          // the MMA thread's bounded wait on it must run out
          const bool drop = (p.debug & 1u) && issued == 0;
          for (int q = 0; q < ppst && !drop; ++q) {
            const int kb = kb0 + q;
            if constexpr (RES) {
              // A is read once: first out of L2 (measured with the output
              // stores likewise hinted: batched_f16 24.0 -> 23.4 us)
              tma_load_3d_hint(dst + q * kPanelBytes, &tmA, fb, kb * CK, m0, b, pol_stream);
            } else {
              if (a_here) tma_load_3d(dst, &tmA, fb, kb * CK, m0, b);
              if (W_KMAJOR) {
                // one box: `width` rows of the transposed weight, 128 bytes of K
                tma_load_3d(dst + wofs, wm, fb, kb * CK, n0, b);
              } else if ((p.w_merged >> s) & 1) {
                // one box: all 64-column blocks of this panel
                tma_load_4d(dst + wofs, wm, fb, 0, kb * CK, n0 / WBOX_N, b);
              } else {
                for (int j = 0; j < width / WBOX_N; ++j)
                  tma_load_3d(dst + wofs + j * WBOX_BYTES, wm, fb, n0 + j * WBOX_N, kb * CK, b);
              }
            }
          }
          ++issued;
          if (++stage == static_cast<uint32_t>(p.nst)) {
            stage = 0;
            phase ^= 1u;
          }
        }
        return true;
      });
      // Wait for every copy still in flight before the CTA may exit.
      const uint64_t nst = static_cast<uint64_t>(p.nst);
      const uint64_t tail = issued < nst ? issued : nst;
      for (uint64_t j = 0; j < tail; ++j) {
        const uint64_t idx = issued - 1 - j;
        drain_wait(bar(kBarFull + static_cast<int>(idx % nst)),
                   static_cast<uint32_t>((idx / nst) & 1u), p.budget_ns);
      }
      if (RES && wl > 0) drain_wait(bar(kBarWFull), (wl - 1) & 1u, p.budget_ns);
    }
  } else if (warp == 1 && !SPLIT) {
    // ---------------------------------------------- MMA (single issuer)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, pf = 0, wl = 0, astage = 0, aphase = 0;
      int cur_b = -1;
      for_each_phase([&](int it, int ph, const TileCursor& c) -> bool {
        if (ph == 0) {
          if constexpr (RES) {
            if (c.b != cur_b) {
              if (!bw.wait(bar(kBarWFull), wl & 1u)) return false;
              ++wl;
              cur_b = c.b;
              tc_fence_after();
            }
          }
          if constexpr (P_TMEM && S >= 2) {
            // The intermediate of the previous tile (in region X) must be fully
            // read by GEMM2 before GEMM1 of this tile overwrites X.  (A single
            // GEMM has no intermediate, and nothing completes this barrier.)
            if (it > 0 && !bw.wait(bar(kBarPEmpty), static_cast<uint32_t>(it - 1) & 1u)) return false;
          }
        }
        const int s = ph < S - 1 ? ph : S - 1;
        // The first phase that reads an intermediate waits for its operand
        // (the later passes of the last GEMM read the same operand).
        if (s >= 1 && ph == s) {
          if (!bw.wait(bar(kBarPFull), pf & 1u)) return false;
          ++pf;
          tc_fence_after();
        }
        int r;
        uint32_t u;
        region_use(p, S, it, ph, r, u);
        if (!bw.wait(bar(kBarREmpty + r), (u & 1u) ^ 1u)) return false;
        tc_fence_after();
        if (!issue_phase(it, ph, r, stage, phase, astage, aphase)) return false;
        tc_commit(bar(ph < S - 1 ? kBarCFull + r : kBarRFull + r));
        if (S >= 2 && ph == nph - 1) tc_commit(bar(kBarPEmpty));
        if (RES && ph == nph - 1 && it + 1 < t_count) {
          TileCursor n = c;
          n.next();
          if (n.b != c.b) tc_commit(bar(kBarWEmpty));  // end of a batch segment
        }
        return true;
      });
      // Every MMA issued so far must be complete before tensor memory is freed.
      tc_commit(bar(kBarDrain));
      drain_wait(bar(kBarDrain), 0, p.budget_ns);
    }
  } else if (SPLIT && (warp == 1 || warp == 10)) {
    // ------------------------------- MMA, GEMM1 issuer (warp 1) and GEMM2 issuer (warp 10)
    if (lane == 0) {
      const bool g1 = (warp == 1);
      uint32_t stage = 0, phase = 0, pf = 0, wl = 0, astage = 0, aphase = 0;
      int cur_b = -1;
      TileCursor c = first;
      bool ok = true;
      for (int it = 0; it < t_count && ok; ++it, c.next()) {
        if (c.b != cur_b) {  // new resident weights
          if (!bw.wait(bar(kBarWFull), wl & 1u)) break;
          ++wl;
          cur_b = c.b;
          tc_fence_after();
        }
        if (g1) {
          const int r = lookahead ? (it & 1) : 0;
          const uint32_t u = lookahead ? static_cast<uint32_t>(it) >> 1 : static_cast<uint32_t>(it);
          if (!bw.wait(bar(kBarREmpty + r), (u & 1u) ^ 1u)) break;
          if (p.p_tmem) {
            // region r also holds the operand of GEMM2 two tiles back: wait
            // until that GEMM2 has completed (its own barrier per region)
            if (!bw.wait(bar(r ? kBarPEmpty1 : kBarPEmpty), (u & 1u) ^ 1u)) break;
          }
          tc_fence_after();
          if (!issue_phase(it, 0, r, stage, phase, astage, aphase)) break;
          tc_commit(bar(kBarCFull + r));
        } else {
          for (int pass = 0; pass < p.npass && ok; ++pass) {
            if (pass == 0) {
              // with two operand images each has its own barriers, so that
              // every wait sees the completions of its barrier in order
              const bool w = p.dbl_p ? bw.wait(bar((it & 1) ? kBarPFull1 : kBarPFull),
                                               (static_cast<uint32_t>(it) >> 1) & 1u)
                                     : bw.wait(bar(kBarPFull), pf & 1u);
              if (!w) {
                ok = false;
                break;
              }
              ++pf;
              tc_fence_after();
            }
            int r;
            uint32_t u;
            zregion(it, pass, r, u);
            if (!bw.wait(bar(kBarREmpty + r), (u & 1u) ^ 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (!issue_phase(it, 1 + pass, r, stage, phase, astage, aphase)) {
              ok = false;
              break;
            }
            tc_commit(bar(kBarRFull + r));
          }
          if (!ok) break;
          tc_commit(bar((p.dbl_p && (it & 1)) ? kBarPEmpty1 : kBarPEmpty));
        }
        if (it + 1 < t_count) {
          TileCursor n = c;
          n.next();
          if (n.b != c.b) tc_commit(bar(kBarWEmpty));  // this issuer is done with the batch
        }
      }
      const int db = g1 ? kBarDrain : kBarDrain2;
      tc_commit(bar(db));
      drain_wait(bar(db), 0, p.budget_ns);
    }
  } else if (!RES && warp == 10) {
    // ------------------------------------------------- A-ring producer
    // The A panels of every tile, in order, as far ahead as the A ring
    // allows: the next tile's A arrives while this tile's later GEMMs run.
    if (lane == 0 && split_a) {
      uint32_t as = 0, aph = 0;
      uint64_t aissued = 0;
      TileCursor c = first;
      bool ok = true;
      // (a single GEMM reads A once per pass of its N columns)
      const int reads = (S == 1) ? p.npass : 1;
      for (int it = 0; it < t_count && ok; ++it, c.next()) {
        const int m0 = c.mt * 128;
        for (int kq = 0; kq < reads * p.kpan0 && ok; ++kq) {
          const int kb = kq % p.kpan0;
          if (!bw.wait(bar(kBarAEmpty + as), aph ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar(kBarAFull + as);
          mbar_arrive_expect_tx(fb, kPanelBytes);
          tma_load_3d(base + p.off_aring + as * static_cast<uint32_t>(kPanelBytes), &tmA, fb, kb * CK, m0, c.b);
          ++aissued;
          if (++as == static_cast<uint32_t>(p.nsta)) {
            as = 0;
            aph ^= 1u;
          }
        }
      }
      // copies still in flight must land before the CTA exits
      const uint64_t n = static_cast<uint64_t>(p.nsta);
      const uint64_t tail = aissued < n ? aissued : n;
      for (uint64_t j = 0; j < tail; ++j) {
        const uint64_t idx = aissued - 1 - j;
        drain_wait(bar(kBarAFull + static_cast<int>(idx % n)), static_cast<uint32_t>((idx / n) & 1u),
                   p.budget_ns);
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ---------------------------------------------------------- converters
    if constexpr (S >= 2) {
      const int q = warp & 3;
      const int row = q * 32 + lane;
      const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
      bool ok = true;
      for (int it = 0; it < t_count && ok; ++it) {
        for (int s = 0; s < S - 1 && ok; ++s) {
          int r;
          uint32_t u;
          region_use(p, S, it, s, r, u);
          // the previous tile's intermediate must be consumed before this
          // tile's is written (and the converters never run two tiles ahead)
          const bool odd = p.dbl_p && (it & 1);
          if (s == 0 && ok) {
            ok = p.dbl_p ? warp_wait(bw, bar(odd ? kBarPEmpty1 : kBarPEmpty),
                                     ((static_cast<uint32_t>(it) >> 1) & 1u) ^ 1u)
                         : warp_wait(bw, bar(kBarPEmpty), (static_cast<uint32_t>(it) & 1u) ^ 1u);
          }
          // region r receives one intermediate per tile (per two tiles for
          // each of the two buffers of a lookahead chain)
          const uint32_t cu = lookahead ? static_cast<uint32_t>(it) >> 1 : static_cast<uint32_t>(it);
          if (ok) ok = warp_wait(bw, bar(kBarCFull + r), cu & 1u);
          if (ok) {
            tc_fence_after();
            const int width = (s == 0) ? N1P : N2P;
            const uint32_t tsrc = tmem_base + lane_off + static_cast<uint32_t>(p.region_col[r]);
            if (!TF32 && p.p_tmem)
              rearrange_accumulator_tmem16<IN>(tsrc, width);
            else
              rearrange_accumulator<IN>(tsrc, width, row, base + p.off_p + (odd ? p.p_bytes : 0u));
            tc_fence_before();
          }
          if (ok) {
            mbar_arrive(bar(odd ? kBarPFull1 : kBarPFull));
            mbar_arrive(bar(kBarREmpty + r));
          }
        }
      }
    }
  } else if (warp >= 6 && warp < 10) {
    // ------------------------------------------------------------ epilogue
    // One named barrier (id 1, 128 threads) per output box.  The loop trip
    // counts do not depend on data, so after an abort every warp keeps
    // walking the same loops and reaching the same barriers while skipping
    // the work: the barriers stay matched and nothing waits forever.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const bool elected = (warp == 6 && lane == 0);
    constexpr int NBOX = NF / OBOX_N;
    constexpr int LDS = OBOX_N / 32;  // 32-column TMEM loads per box (1 or 2)
    uint32_t nbox = 0;
    bool ok = true;
    TileCursor c = first;
    // A CTA with one tile and a single final pass stages its output boxes in
    // the ring, idle by then (the pass completing means every MMA, and so
    // every read of a stage, is done, and nothing more is loaded), one box
    // per 16 KB, so that their stores run concurrently instead of each
    // waiting for the previous one to have read its staging buffer: the
    // epilogue is that CTA's last step and nothing else hides it.
    const int ring_boxes = static_cast<int>((static_cast<uint32_t>(p.nst) * p.stage_bytes) / kPanelBytes);
    // (streamed weights only: in the resident-weight kernels, whose CTAs run
    // many tiles, the extra choice per box measured 1 % slower)
    const bool ring_last = !RES && p.npass == 1 && t_count == 1 && NBOX <= ring_boxes;
    for (int it = 0; it < t_count; ++it, c.next()) {
      const int b = c.b;
      const int m0 = c.mt * 128;
      const bool in_ring = ring_last && it == t_count - 1;
      for (int pass = 0; pass < p.npass; ++pass) {
        int r;
        uint32_t u;
        region_use(p, S, it, NPH_FIXED + pass, r, u);
        // how many final products this region held before (epilogue's own count)
        const uint32_t eu =
            p.nz > 0 ? u
                     : static_cast<uint32_t>(it) * static_cast<uint32_t>(r == 0 ? (p.npass + 1) / 2 : p.npass / 2) +
                           static_cast<uint32_t>(pass / 2);
        if (ok) ok = warp_wait(bw, bar(kBarRFull + r), eu & 1u);
        tc_fence_after();
        const uint32_t tsrc = tmem_base + lane_off + static_cast<uint32_t>(p.region_col[r]);
        const int n0 = pass * NF;
        // The TMEM load of box j+1 is issued as soon as box j is in shared
        // memory, so its latency overlaps box j's barrier and store.
        uint32_t v[LDS][32];
        if (ok) {
#pragma unroll
          for (int l = 0; l < LDS; ++l) tmem_ld32(tsrc + static_cast<uint32_t>(l * 32), v[l]);
        }
#pragma unroll 1
        for (int j = 0; j < NBOX; ++j) {
          const uint32_t buf = (p.nstg == 2) ? (nbox & 1u) : 0u;
          const uint32_t stg = in_ring ? base + p.off_ring + static_cast<uint32_t>(pass * NBOX + j) * kPanelBytes
                                       : base + p.off_stg + buf * kPanelBytes;
          if (ok) {
            tmem_wait_ld();
            if (j == NBOX - 1) {
              tc_fence_before();
              mbar_arrive(bar(kBarREmpty + r));
            }
#pragma unroll
            for (int l = 0; l < LDS; ++l) store_output_row<OUT>(stg, row, l * 32, v[l]);
            fence_proxy_async_smem();
            if (j + 1 < NBOX) {
#pragma unroll
              for (int l = 0; l < LDS; ++l)
                tmem_ld32(tsrc + static_cast<uint32_t>((j + 1) * OBOX_N + l * 32), v[l]);
            }
          }
          // The store issued for the previous box must have read its staging
          // buffer before anyone fills that buffer again (next box).  (Boxes
          // in the ring each have their own buffer.)
          if (elected && ok && !in_ring) {
            if (p.nstg == 2)
              bulk_wait_read<0>();
          }
          named_bar_sync(1, 128);
          if (elected && ok) {
            // (the output is not read again here: first out of L2)
            tma_store_3d_hint(&tmOut, stg, n0 + j * OBOX_N, m0, b, pol_stream);
            bulk_commit();
            if (p.nstg == 1 && !in_ring) bulk_wait_read<0>();
          }
          if (p.nstg == 1 && !in_ring) named_bar_sync(1, 128);
          ++nbox;
        }
      }
    }
    if (elected) bulk_wait_all();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace b2b

namespace b2b {

// Test support: run the converter routine of the fused kernel on one 128-row
// tile.  `acc` holds the tile's fp32 bit patterns [128][width]; they are put
// into tensor memory in the accumulator layout, rearranged by
// rearrange_accumulator<IN>, and the resulting operand (the swizzled
// shared-memory image, or for tf32 the tensor-memory operand) is copied out.
template <int IN>
__global__ void __launch_bounds__(128, 1)
    probe_operand_kernel(const uint32_t* __restrict__ acc, uint32_t* __restrict__ out, int width,
                         uint32_t tmem_cols) {
  using namespace ptx;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tslot;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t img = (raw + 1023u) & ~1023u;
  const uint8_t* gimg = smem_raw + (img - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = warp * 32 + lane;
  if (warp == 0) {
    tmem_alloc(smem_u32(&tslot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tslot;
  const uint32_t tsrc = tbase + (static_cast<uint32_t>(warp * 32) << 16);
  for (int c0 = 0; c0 < width; c0 += 32) {
    uint32_t v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = acc[row * width + c0 + i];
    tmem_st32(tsrc + static_cast<uint32_t>(c0), v);
  }
  tmem_wait_st();
  rearrange_accumulator<IN>(tsrc, width, row, img);
  if constexpr (IN == kInTF32) {
    for (int c0 = 0; c0 < width; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tsrc + static_cast<uint32_t>(c0), v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) out[row * width + c0 + i] = v[i];
    }
  } else {
    __syncthreads();
    const int words = width * 256 / 4;
    const uint32_t* src = reinterpret_cast<const uint32_t*>(gimg);
    for (int i = threadIdx.x; i < words; i += blockDim.x) out[i] = src[i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, tmem_cols);
}

}  // namespace b2b
