// A cascade of S GEMMs (2 <= S <= 8) with 16-bit operands on pairs of SMs
// (tcgen05, cta_group::2, sm_103a):
//
//   P_1 = A.W_0 -> round -> P_2 = P_1.W_1 -> round -> ... -> E = P_{S-1}.W_{S-1}
//
// Source of the method: patent "数据处理方法、装置、设备及介质" (Alibaba, 2023),
// Detailed description para. 41 (several cascaded operators, each one's
// output the next one's input), para. 54-60 (the result of one operator is
// rearranged and handed to the next without going through memory) and
// para. 103-110 (rearrangement through shared memory).
//
// Every weight is streamed through the SMs once per 256-row tile, so the
// weights, not A, dominate the bytes an SM must load.  Two CTAs of a cluster
// share each MMA (M = 256): each holds its own 128 rows of A, of the
// intermediates and of every accumulator, and half of the columns of every
// weight panel, which halves the weight traffic and the shared memory a
// weight slot needs per SM.  The converters turn an accumulator row into the
// K-major 128-byte-swizzled operand image of the next GEMM in shared memory
// (one image, overwritten stage after stage).
//
// Every GEMM runs in passes of at most 256 output columns.  Tensor memory
// (512 columns) holds two 256-column regions, X and Y.  An intermediate of
// at most 256 columns takes the region not used last, so a GEMM writes one
// region while the converters still read the other, and starts on the first
// 128-column chunk of its operand image as soon as that chunk is written.
// A wider intermediate (up to 512 columns) starts in the region not used
// last and continues in the other; the next GEMM writes the first one again
// once its converters have freed it.  The passes of the first GEMM are
// converted one by one as they complete (it reads no operand image); a later
// GEMM's result only once the whole GEMM, which reads the image, is done.
// The passes of the last GEMM alternate between the regions, so the
// epilogue of one pass overlaps the MMAs of the next.  Whether a region is
// free is counted by one barrier per region that its reader (the converters
// or the epilogue) releases.
//
// Roles (384 threads, one CTA per SM, persistent over 256-row tiles):
//   warp 0     producer: one ring of 16 KB slots in the order the MMAs read
//              them (the first GEMM: an A panel and this CTA's half of a
//              weight panel; every later GEMM: a weight half panel)
//   warp 1     TMEM allocation (both CTAs); the even CTA's lane 0 issues MMAs
//   warps 2-9  converters (accumulator -> operand image), half of each
//              128-column chunk for each of the two warps that share a TMEM
//              lane quadrant
//   warps 6-9  also the epilogue (accumulator -> output type -> staging ->
//              TMA store, each warp its own 32 rows)
//   warp 11    slot watcher (even CTA): waits for every slot's copies in
//              the MMAs' order and publishes the count in shared memory,
//              which the MMA thread polls at a fraction of the cost of an
//              mbarrier wait (the tensor pipe queues only about two MMAs, so
//              the MMA thread's own waits would leave it idle)
// Every wait is bounded; after an abort the converter and epilogue loops are
// still walked to the end with the work skipped, so that named barriers stay
// matched, and the two CTAs meet at a cluster barrier before exit.
#pragma once

#include "chain_tc.cuh"

namespace b2b {

constexpr int kMaxStages = 8;

// Barrier slots (8 bytes each) at ChainNParams::off_bar.
enum : int {
  knFull = 0,        // [16] ring slot filled (even CTA's: armed by it for both CTAs' copies)
  knEmpty = 16,      // [16] ring slot consumed
  knCFull = 32,      // an intermediate GEMM after the first complete (all its
                     // passes): converters
  knPChunk = 33,     // [2][4] 128-column chunk c of intermediate k's operand image
                     //        (set k & 1) written in both CTAs (even CTA's)
  knRFull = 41,      // [2] X / Y holds a pass of the last GEMM (epilogue)
  knREmpty = 43,     // [2] X / Y read in both CTAs, by the converters or the
                     //     epilogue (even CTA's)
  knDrain = 45,      // every MMA complete (exit)
  knSlotTmem = 46,   // uint32 TMEM base, then the int abort flag
  knSlotReady = 47,  // uint32: ring slots whose copies have landed (even CTA)
  knCFull0 = 48,     // [4] pass j of the first GEMM complete: converters
};

constexpr int kChainNThreads = 384;

struct ChainNParams {
  int batch, M, K;
  int S;                     // GEMMs in the cascade
  int m_tiles, total_tiles;  // 256-row tiles per batch, in all
  int wpad[kMaxStages];      // intermediate s < S-1: padded width (128, 256, 384 or 512)
  int pw[kMaxStages];        // pass width: 128 or 256 (intermediates), NF (last GEMM)
  int kpan[kMaxStages];      // 64-element K panels GEMM s reads
  int npass;                 // NF-column passes of the last GEMM
  int slots0;                // ring slots of the intermediate GEMMs of one tile
  int nslot, nstg;           // ring slots (16 KB each) and staging buffers per warp
  uint32_t off_ring, off_p, off_stg, off_bar;
  int w_merged;              // bit s: weight s is read as one 4-D box per half panel
  int split;                 // leftover tiles whose passes are split between two clusters
  int ptm;                   // bit s: 16-bit intermediate s is packed in tensor memory (two
                             // K per 32-bit column, in place in its accumulator's region)
                             // and read from there by the next GEMM instead of from the
                             // operand image.  Plans set it for an intermediate of at most
                             // 256 columns whose region the GEMM after next may overwrite:
                             // the next intermediate fits one region, or, for the last one,
                             // the last GEMM runs in one pass.
  int w_kmajor;              // tf32 weights arrive transposed ([N][K], K-major) instead of as
                             // stored ([K][N], MN-major with 32-byte swizzle atoms)
  uint32_t debug;            // test support: bit 0 = the first ring slot is never filled
  int* status;
  unsigned long long budget_ns;
};

// Tensor maps of one run: A, the output, and every weight.
struct ChainNMaps {
  CUtensorMap a, out;
  CUtensorMap w[kMaxStages];
};

// Work units of a cluster.  Tiles are dealt to the clusters in strides; when
// they do not divide evenly, the `split` leftover tiles are each shared by two
// clusters, one taking the first half of the last GEMM's passes and the other
// the rest (both compute the intermediates), and these half units come first.
// That shortens the longest cluster's work and starts half of the clusters
// out of step with the others, which spreads their HBM-bound first GEMMs.
struct ChainNUnit {
  int b, mt, p0, p1;  // batch, 256-row tile, passes [p0, p1) of the last GEMM
};
__host__ __device__ __forceinline__ int chainn_units(const ChainNParams& p, int cid, int ncl) {
  if (p.split > 0) return p.total_tiles / ncl + (cid < 2 * p.split ? 1 : 0);
  return cid < p.total_tiles ? (p.total_tiles - cid + ncl - 1) / ncl : 0;
}
__host__ __device__ __forceinline__ ChainNUnit chainn_unit(const ChainNParams& p, int cid, int ncl, int i) {
  int tile, p0 = 0, p1 = p.npass;
  if (p.split > 0 && cid < 2 * p.split) {
    if (i == 0) {
      tile = (p.total_tiles / ncl) * ncl + (cid >> 1);
      const int h = (p.npass + 1) / 2;
      p0 = (cid & 1) ? h : 0;
      p1 = (cid & 1) ? p.npass : h;
    } else {
      tile = cid + (i - 1) * ncl;
    }
  } else {
    tile = cid + i * ncl;
  }
  ChainNUnit u;
  u.b = tile / p.m_tiles;
  u.mt = tile - u.b * p.m_tiles;
  u.p0 = p0;
  u.p1 = p1;
  return u;
}

// Tensor-memory placement, walked identically by the MMA thread, the
// converters and the epilogue.  Every accumulator starts in the region not
// used last (r0); a wider one continues in the other region, and the next
// accumulator then starts in r0 again, which its converters free first.
// Column c of an accumulator that starts in r0 lives at tmem_col(r0, c).
template <int V>
struct integral_constant_int {
  static constexpr int value = V;
};

struct RegionCursor {
  uint32_t last = 1;
  __host__ __device__ __forceinline__ uint32_t take(int width) {
    const uint32_t r0 = last ^ 1u;
    last = width <= 256 ? r0 : r0 ^ 1u;
    return r0;
  }
};
__host__ __device__ __forceinline__ uint32_t tmem_col(uint32_t r0, int c) {
  return ((((static_cast<uint32_t>(c) >> 8) ^ r0) & 1u) << 8) | (static_cast<uint32_t>(c) & 255u);
}

// One converter warp's share of 128-column chunk `ch` of an intermediate
// whose accumulator starts in region r0: the two warps that share a TMEM lane
// quadrant take 64 columns each (h = 0: the low half, h = 1: the high half),
// rounded into the K-major swizzled operand image `p_img` (128-byte panels
// of 64 K elements, one per 64 columns).  `lane_off` selects the warp's lane
// quadrant, `row` is the thread's row of the tile.
template <int IN>
__device__ __forceinline__ void convert_chunk_half(uint32_t tmem_base, uint32_t lane_off, uint32_t r0, int ch,
                                                   int h, int row, uint32_t p_img) {
  const int pcol = ch * 128 + h * 64;
  rearrange_accumulator<IN>(tmem_base + lane_off + tmem_col(r0, pcol), 64, row,
                            p_img + static_cast<uint32_t>(pcol / 64) * kPanelBytes);
}

// TF0: the first GEMM takes fp32 A and W0 as tf32 operands (W0 read as
// stored, an MN-major B operand in 128-byte rows swizzled in 32-byte atoms,
// or, with w_kmajor, transposed to [N][K]), and its result is rounded to
// the 16-bit type IN of every later GEMM: a mixed-type cascade, where the
// accumulator and operand layouts of the first hand-over differ in element
// size as well as in order.
//
// IN = tf32 (with TF0): a two-GEMM tf32 chain.  The intermediate (at most
// 256 columns) is rounded to tf32 in place in tensor memory, one K element
// per 32-bit column, and the second GEMM (one pass, its weight read like
// W0) reads it from there as its A operand, so no operand image is kept.
// The next GEMM to write that region is the next unit's first GEMM, which
// the tensor pipe runs after every MMA that reads it.
template <int IN, int OUT, int NF, bool TF0 = false>
__global__ void __launch_bounds__(kChainNThreads, 1)
    chainn_kernel(const __grid_constant__ ChainNMaps maps, const __grid_constant__ ChainNParams p) {
  using namespace ptx;
  static_assert(IN == kInF16 || IN == kInBF16 || (IN == kInTF32 && TF0), "16-bit or tf32 operands");
  static_assert(NF == 128 || NF == 256, "pass width of the last GEMM");
  constexpr bool PT = IN == kInTF32;  // tf32 intermediate, kept in tensor memory
  constexpr int CG = 2;
  constexpr int CK = 64;           // K elements per 128-byte panel
  constexpr int CK0 = TF0 ? 32 : CK;  // of the first GEMM's operands
  constexpr int KSTEP = 16;        // K of one MMA
  constexpr int WBOX_N = 64;       // weight columns per 128-byte block
  constexpr int WBOX_BYTES = CK * 128;
  constexpr int OSZ = (OUT == kOutF32) ? 4 : 2;
  constexpr int OBOX_N = 128 / OSZ;
  constexpr uint32_t FMT = (IN == kInF16) ? 0u : (IN == kInBF16 ? 1u : 2u);
  constexpr uint32_t kCols = 512;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + p.off_bar;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + p.off_bar + 8 * knSlotTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const int S = p.S;
  const bool wk = p.w_kmajor != 0;  // tf32 weights transposed (K-major)

  // Before waiting for the previous kernel in the stream, and while the
  // other warps set up barriers and tensor memory, one thread pulls the first
  // unit's A into L2 (the TMA prefetch instructions take a good part of a
  // microsecond to issue).  A may be that kernel's output, but a prefetch
  // touches L2 only, where its writes land too, and every load into shared
  // memory comes after the wait, so no stale value is read.  At most four K
  // panels (more only compete with that kernel's tail).  In a tf32 chain
  // whose cluster runs a single unit, where the set-up is on the critical
  // path, the prefetching warp arrives on the cluster barrier first, so the
  // barrier does not wait for the prefetches (16384 rows: set-up 1.9 -> 0.8
  // us, 13.5 -> 13.1 us per call; the 16-bit cascades, with several units
  // per cluster, keep one barrier after the prefetches: the split one
  // measured 1-3 % slower there).
  //
  // Work units (256-row tiles, or halves of their last GEMM) of this
  // cluster.
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);
  const int t_count = chainn_units(p, cid, ncl);
  const bool early = PT && t_count == 1;
  if (warp == 3 && early) cluster_arrive();
  if (warp == 3 && lane == 0) {
    prefetch_tmap(&maps.a);
    for (int s = 0; s < S; ++s) prefetch_tmap(&maps.w[s]);
    prefetch_tmap(&maps.out);
  }
  if (warp == 3 && lane == 0 && t_count > 0) {
    const ChainNUnit c = chainn_unit(p, cid, ncl, 0);
    const int m0 = c.mt * 256 + static_cast<int>(rank) * 128;
    const int npf = p.kpan[0] < 4 ? p.kpan[0] : 4;
    for (int q = 0; q < npf; ++q) tma_prefetch_l2_3d(&maps.a, q * CK0, m0, c.b);
    // and this CTA's half of the first GEMM's first weight panels (as
    // stored; a transposed tf32 weight is the transpose kernel's output, not
    // yet written)
    if (!p.w_kmajor) {
      const int n0 = static_cast<int>(rank) * (p.pw[0] / 2);
      const int blk = TF0 ? 32 : WBOX_N;  // columns per 128-byte block
      for (int q = 0; q < npf; ++q) {
        if (p.w_merged & 1)
          tma_prefetch_l2_4d(&maps.w[0], 0, q * CK0, n0 / blk, c.b);
        else
          for (int j = 0; j < p.pw[0] / 2 / blk; ++j) tma_prefetch_l2_3d(&maps.w[0], n0 + j * blk, q * CK0, c.b);
      }
    }
  }
  // Barriers, set up by the lanes of warp 0 in parallel (each lane fences
  // its own initialisations), while warp 1 allocates tensor memory.
  if (warp == 0) {
    if (lane < 16) {
      mbar_init(bar(knFull + lane), 1);
      mbar_init(bar(knEmpty + lane), 1);
    } else if (lane < 24) {
      mbar_init(bar(knPChunk + lane - 16), 2);
    } else if (lane < 28) {
      mbar_init(bar(knCFull0 + lane - 24), 1);
    } else if (lane < 30) {
      mbar_init(bar(knRFull + lane - 28), 1);
      mbar_init(bar(knREmpty + lane - 28), 2);
    } else if (lane == 30) {
      mbar_init(bar(knCFull), 1);
      mbar_init(bar(knDrain), 1);
    } else {
      *abort_flag = 0;
      *reinterpret_cast<volatile uint32_t*>(gbase + p.off_bar + 8 * knSlotReady) = 0u;
    }
    if (lane < 31) fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(tmem_slot), kCols);
    tmem_relinquish<CG>();
  }
  // (every thread of both CTAs: the peer's barriers exist before anything
  // arrives on them)
  tc_fence_before();
  if constexpr (PT) {
    __syncwarp();
    if (warp != 3 || !early) cluster_arrive();
    cluster_wait();
  } else {
    __syncthreads();
    cluster_sync();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_launch_dependents();
  grid_dependency_wait();

  BoundedWait bw{abort_flag, p.status, p.budget_ns, kTimeoutCode};
  // The output is written with an L2 evict-first policy (three_stage_bf16
  // 40.7 -> 40.4 us, mixed_tf32_bf16 35.9 -> 35.7 us); A is read with it
  // only by a cluster with a single unit (the tf32 workload 13.1 -> 12.9
  // us): with several units per cluster, whose next A is pulled into L2
  // ahead, hinted A loads made every cascade slower (three_stage_bf16
  // 40.7 -> 42.7 us).
  const bool hint_a = t_count == 1;
  const uint64_t pol_stream = l2_policy_evict_first();
  // Waits on barriers that threads of the peer CTA arrive on (the same
  // default-scope wait: the remote arrives are ordered by the barrier itself).
  BoundedWait bwm = bw;
  auto lbar = [&](int i) -> uint32_t { return mapa_shared(bar(i), 0); };

  // This CTA's 128 rows of each unit.
  auto row0 = [&](int mt) -> int { return mt * 256 + static_cast<int>(rank) * 128; };
  const uint32_t p_img = base + p.off_p;
  const int kpan_last = p.kpan[S - 1];
  // K panels per ring slot: a weight half panel of 64 columns (pass width
  // 128) takes 8 KB, so a slot holds two K panels of it; GEMM s > 0 only
  // (its K panel count, a multiple of 128 / 64, is even); tf32 weights: one
  auto kps_of = [&](int s) -> int { return (!PT && s > 0 && p.pw[s] == 128) ? 2 : 1; };
  const int kps_last = kps_of(S - 1);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&maps.a);
      prefetch_tmap(&maps.out);
      for (int s = 0; s < S; ++s) prefetch_tmap(&maps.w[s]);
      uint32_t slot = 0, phase = 0;
      uint64_t issued = 0;
      bool ok = true;
      // one ring slot: an A panel (s < 0), or this CTA's half of `npan`
      // weight K panels (kb, kb + 1, ...)
      auto load = [&](int s, int b, int m0, int kb, int col0, int pw, int npan) -> bool {
        if (!bw.wait(bar(knEmpty + slot), phase ^ 1u)) return false;
        const uint32_t dst = base + p.off_ring + slot * static_cast<uint32_t>(kPanelBytes);
        const uint32_t fb = lbar(knFull + slot);
        const int wcols = pw / 2;
        const uint32_t bytes =
            s < 0 ? static_cast<uint32_t>(kPanelBytes) : 128u * static_cast<uint32_t>(wcols * npan);
        // Only the even CTA arms its barrier, for both CTAs' copies; the odd
        // CTA's copies may land first (the transaction count then dips
        // below zero until the arming, which the barrier allows).
        if (leader) mbar_arrive_expect_tx(bar(knFull + slot), 2u * bytes);
        // test support: the very first slot is armed but never filled
        if (!((p.debug & 1u) && issued == 0)) {
          if (s < 0) {
            if (hint_a)
              tma_load_3d_pair_hint(dst, &maps.a, fb, kb * CK0, m0, b, pol_stream);
            else
              tma_load_3d_pair(dst, &maps.a, fb, kb * CK0, m0, b);
          } else {
            const CUtensorMap* wm = &maps.w[s];
            const int n0 = col0 + static_cast<int>(rank) * wcols;
            if (((TF0 && s == 0) || PT) && p.w_kmajor) {
              // a tf32 weight transposed: this CTA's wcols rows of 32 K elements
              tma_load_3d_pair(dst, wm, fb, kb * CK0, n0, b);
            } else if ((TF0 && s == 0) || PT) {
              // a tf32 weight as stored: 32 K rows of this CTA's wcols columns,
              // in blocks of 32 columns (4 KB each)
              if ((p.w_merged >> s) & 1)
                tma_load_4d_pair(dst, wm, fb, 0, kb * CK0, n0 / 32, b);
              else
                for (int j = 0; j < wcols / 32; ++j) tma_load_3d_pair(dst + j * 4096u, wm, fb, n0 + j * 32, kb * CK0, b);
            } else if ((p.w_merged >> s) & 1) {
              // one box of npan * 64 K rows and wcols / 64 column blocks
              tma_load_4d_pair(dst, wm, fb, 0, kb * CK, n0 / WBOX_N, b);
            } else {
              for (int i = 0; i < npan; ++i)
                for (int j = 0; j < wcols / WBOX_N; ++j)
                  tma_load_3d_pair(dst + (i * (wcols / WBOX_N) + j) * WBOX_BYTES, wm, fb, n0 + j * WBOX_N,
                                   (kb + i) * CK, b);
            }
          }
        }
        ++issued;
        if (++slot == static_cast<uint32_t>(p.nslot)) {
          slot = 0;
          phase ^= 1u;
        }
        return true;
      };
      for (int it = 0; it < t_count && ok; ++it) {
        const ChainNUnit c = chainn_unit(p, cid, ncl, it);
        const int m0 = row0(c.mt);
        // the ring reaches only a few panels into the next unit's first
        // GEMM: pull the next unit's A into L2 now
        if (it + 1 < t_count) {
          const ChainNUnit n = chainn_unit(p, cid, ncl, it + 1);
          for (int q = 0; q < p.kpan[0]; ++q) tma_prefetch_l2_3d(&maps.a, q * CK0, row0(n.mt), n.b);
        }
        for (int s = 0; s < S - 1 && ok; ++s) {
          const int pw = p.pw[s], kps = kps_of(s);
          for (int col0 = 0; col0 < p.wpad[s] && ok; col0 += pw)
            for (int kb = 0; kb < p.kpan[s] && ok; kb += kps) {
              if (s == 0) ok = load(-1, c.b, m0, kb, 0, 0, 1);
              if (ok) ok = load(s, c.b, m0, kb, col0, pw, kps);
            }
        }
        for (int j = c.p0; j < c.p1 && ok; ++j)
          for (int kb = 0; kb < kpan_last && ok; kb += kps_last)
            ok = load(S - 1, c.b, m0, kb, j * NF, NF, kps_last);
      }
      // copies in flight land before exit (the even CTA's barriers count both
      // CTAs' copies; the odd CTA waits at the cluster barrier before exit)
      const uint64_t n = static_cast<uint64_t>(p.nslot);
      const uint64_t tail = !leader ? 0 : (issued < n ? issued : n);
      for (uint64_t j = 0; j < tail; ++j) {
        const uint64_t idx = issued - 1 - j;
        drain_wait(bar(knFull + static_cast<int>(idx % n)), static_cast<uint32_t>((idx / n) & 1u),
                   p.budget_ns);
      }
    }
  } else if (warp == 11) {
    // ------------------------------------------- slot watcher (even CTA)
    if (lane == 0 && leader) {
      uint32_t slot = 0, phase = 0, n = 0;
      const uint32_t ready = bar(knSlotReady);
      bool ok = true;
      for (int it = 0; it < t_count && ok; ++it) {
        const ChainNUnit c = chainn_unit(p, cid, ncl, it);
        const int per_unit = p.slots0 + (c.p1 - c.p0) * (kpan_last / kps_last);
        for (int q = 0; q < per_unit && ok; ++q) {
          ok = bw.wait(bar(knFull + slot), phase);
          if (!ok) break;
          if (++slot == static_cast<uint32_t>(p.nslot)) {
            slot = 0;
            phase ^= 1u;
          }
          st_release_shared(ready, ++n);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------- MMA (even CTA, lane 0)
    if (lane == 0 && leader) {
      uint32_t slot = 0;
      uint32_t ux = 0, uy = 0;  // products written to X / Y so far
      bool ok = true;
      // region r's previous product has been read in both CTAs
      auto take_region = [&](int r) -> bool {
        const uint32_t ur = r ? uy : ux;
        const bool done = ur == 0 || bwm.wait(bar(knREmpty + r), (ur - 1u) & 1u);
        if (r) ++uy; else ++ux;
        return done;
      };
      // the next `need` slots have landed once the watcher's count reaches
      // consumed + need
      uint32_t consumed = 0, seen = 0;
      const uint32_t ready = bar(knSlotReady);
      // tf32 chains: the tensor-memory column of the intermediate the next
      // GEMM reads
      uint32_t p_tmem = 0;
      // 16-bit chains: whether the intermediate the next GEMM reads is packed
      // in tensor memory (at p_tmem) rather than in the operand image
      bool a_tm = false;
      auto stage_ready = [&](uint32_t need) -> bool {
        if (seen >= consumed + need) return true;
        seen = ld_acquire_shared(ready);
        if (seen >= consumed + need) return true;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
          for (int i = 0; i < 32; ++i) {
            seen = ld_acquire_shared(ready);
            if (seen >= consumed + need) return true;
          }
          if (*abort_flag) return false;
          if (globaltimer_ns() - t0 > p.budget_ns) {
            bw.raise();
            return false;
          }
        }
      };
      auto next_slot = [&](uint32_t x) -> uint32_t {
        return x + 1u == static_cast<uint32_t>(p.nslot) ? 0u : x + 1u;
      };
      // The MMAs of one K-panel group: four per 128-byte K panel.  First
      // GEMM (npan == 0): the A panel in slot sa_slot, the weight half panel
      // in slot w_slot; later GEMMs read K panels kb .. kb + npan - 1 of the
      // operand image (their weight half panels share slot w_slot).
      // (straight-line MMAs: a branch between two of them costs more than
      // the tensor pipe's queue hides)
      auto group_mmas = [&](auto npan_c, uint32_t d, uint32_t idesc, int kb, uint32_t sa_slot, uint32_t w_slot,
                            uint32_t acc0) {
        constexpr int npan = decltype(npan_c)::value;
        constexpr bool a_smem = npan == 0;
        const uint32_t wb = base + p.off_ring + w_slot * static_cast<uint32_t>(kPanelBytes);
        const uint32_t sa = a_smem ? base + p.off_ring + sa_slot * static_cast<uint32_t>(kPanelBytes)
                                   : p_img + static_cast<uint32_t>(kb) * kPanelBytes;
        // a tf32 weight: 8 K elements per MMA, B as stored (MN-major, 32-column
        // blocks of 4 KB, 32-byte swizzle atoms: a K step is 8 rows of 128
        // bytes) or transposed (K-major: a K step is 32 bytes along a row)
        const uint64_t tb0 = wk ? desc_sw128(wb, 16u, 1024u) : desc_mn32(wb, 4096u, 512u);
        const uint32_t tbs = wk ? 2u : 64u;
        if constexpr (a_smem && TF0) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss<true, CG>(d, desc_sw128(sa + kk * 32u, 16u, 1024u), tb0 + kk * tbs, idesc, kk ? 1u : acc0);
        } else if constexpr (PT) {
          // tf32 intermediate in tensor memory: K panel kb is its columns
          // [32 kb, 32 kb + 32), 8 per MMA
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts<true, CG>(d, p_tmem + static_cast<uint32_t>(kb * 32 + kk * 8), tb0 + kk * tbs, idesc,
                             kk ? 1u : acc0);
        } else if constexpr (npan == 2) {
          if (a_tm) {
            // the intermediate packed in tensor memory: K panel kb is its
            // columns [32 kb, 32 kb + 32), 8 per MMA
#pragma unroll
            for (int kk = 0; kk < 2 * (CK / KSTEP); ++kk) {
              const uint32_t pa = static_cast<uint32_t>(kk >> 2), ks = static_cast<uint32_t>(kk & 3);
              mma_ts<false, CG>(d, p_tmem + static_cast<uint32_t>(kb * 32) + pa * 32u + ks * 8u,
                                desc_sw128(wb + pa * WBOX_BYTES + ks * KSTEP * 128u, WBOX_BYTES, 1024u), idesc,
                                kk ? 1u : acc0);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 2 * (CK / KSTEP); ++kk) {
              const uint32_t pa = static_cast<uint32_t>(kk >> 2), ks = static_cast<uint32_t>(kk & 3);
              mma_ss<false, CG>(d, desc_sw128(sa + pa * kPanelBytes + ks * 32u, 16u, 1024u),
                                desc_sw128(wb + pa * WBOX_BYTES + ks * KSTEP * 128u, WBOX_BYTES, 1024u), idesc,
                                kk ? 1u : acc0);
            }
          }
        } else {
          if (!a_smem && a_tm) {
#pragma unroll
            for (int kk = 0; kk < CK / KSTEP; ++kk)
              mma_ts<false, CG>(d, p_tmem + static_cast<uint32_t>(kb * 32 + kk * 8),
                                desc_sw128(wb + kk * KSTEP * 128u, WBOX_BYTES, 1024u), idesc, kk ? 1u : acc0);
          } else {
#pragma unroll
            for (int kk = 0; kk < CK / KSTEP; ++kk)
              mma_ss<false, CG>(d, desc_sw128(sa + kk * 32u, 16u, 1024u),
                                desc_sw128(wb + kk * KSTEP * 128u, WBOX_BYTES, 1024u), idesc, kk ? 1u : acc0);
          }
        }
      };
      // One stage: one K-panel group, or (pair) two consecutive ones, whose
      // slots are waited for and released together, so that the per-stage
      // work of this thread (the readiness check, a chunk wait, the fence)
      // is paid once per eight MMAs instead of four (measured: 1-2 % on the
      // cascades; the tensor pipe queues only about two MMAs, so that work
      // can show up as idle pipe time).  A chunk wait (chunk >= 0, parity
      // cpar) is for the operand image chunk holding K panel kb (a pair
      // never spans two chunks: it starts at an even panel).
      auto stage_mmas = [&](auto npan_c, auto pair_c, uint32_t d, uint32_t idesc, int kb, int chunk,
                            uint32_t cpar) -> bool {
        constexpr int npan = decltype(npan_c)::value;
        constexpr bool pair = decltype(pair_c)::value != 0;
        constexpr bool a_smem = npan == 0;
        constexpr uint32_t per = a_smem ? 2u : 1u;  // slots per K-panel group
        constexpr uint32_t need = pair ? 2u * per : per;
        if (!stage_ready(need)) return false;
        if (chunk >= 0 && !bwm.wait(bar(chunk), cpar)) return false;
        consumed += need;
        tc_fence_after();
        const uint32_t s0 = slot;
        const uint32_t s1 = a_smem ? next_slot(s0) : s0;
        group_mmas(npan_c, d, idesc, kb, s0, s1, kb != 0 ? 1u : 0u);
        uint32_t last = s1;
        if constexpr (pair) {
          const uint32_t s2 = next_slot(s1);
          const uint32_t s3 = a_smem ? next_slot(s2) : s2;
          group_mmas(npan_c, d, idesc, kb + 1, s2, s3, 1u);
          last = s3;
        }
        uint32_t x = s0;
#pragma unroll
        for (uint32_t q = 0; q < need; ++q) {
          tc_commit<CG>(bar(knEmpty + x));
          x = next_slot(x);
        }
        slot = next_slot(last);
        return true;
      };
      // the K panels of GEMM s > 0 from kb on need chunk kb / 2 (tf32:
      // kb / 4) of the previous intermediate (global index k - 1), on its
      // first pass only
      RegionCursor rc;
      uint32_t k = 0;  // intermediates started so far
      constexpr int kpc = PT ? 4 : 2;  // K panels per 128-column chunk
      auto chunk_of = [&](bool first_pass, int kb) -> int {
        if (!first_pass || (kb % kpc)) return -1;
        return knPChunk + static_cast<int>(((k - 1u) & 1u) * 4u) + kb / kpc;
      };
      // one pass: kpan K panels, npan of them per ring slot (0: the first
      // GEMM, one K panel and two slots)
      // (after the first GEMM, one-panel groups go in pairs while two
      // panels are left; a chunk wait falls on an even panel, so on the
      // first of a pair.  The first GEMM, which waits on its loads, keeps
      // single groups: a pair would hold back its MMAs until four slots
      // have landed.)
      auto run_pass = [&](auto npan_c, uint32_t d, uint32_t idesc, int kpan, bool first, uint32_t cpar) -> bool {
        constexpr int npan = decltype(npan_c)::value;
        constexpr int step = npan == 0 ? 1 : npan;
        using Single = integral_constant_int<0>;
        using Pair = integral_constant_int<1>;
        int kb = 0;
        if constexpr (npan == 1) {
          for (; kb + 1 < kpan; kb += 2)
            if (!stage_mmas(npan_c, Pair{}, d, idesc, kb, npan == 0 ? -1 : chunk_of(first, kb), cpar)) return false;
        }
        for (; kb < kpan; kb += step)
          if (!stage_mmas(npan_c, Single{}, d, idesc, kb, npan == 0 ? -1 : chunk_of(first, kb), cpar)) return false;
        return true;
      };
      using First = integral_constant_int<0>;
      using One = integral_constant_int<1>;
      using Two = integral_constant_int<2>;
      for (int it = 0; it < t_count && ok; ++it) {
        const ChainNUnit c = chainn_unit(p, cid, ncl, it);
        for (int s = 0; s < S - 1 && ok; ++s) {
          const int pw = p.pw[s];
          const uint32_t r0 = rc.take(p.wpad[s]);
          const uint32_t idesc = ((TF0 && s == 0) || PT) ? make_idesc(2u, static_cast<uint32_t>(pw), 256u, !wk)
                                                         : make_idesc(FMT, static_cast<uint32_t>(pw), 256u, true);
          const uint32_t cpar = ((k - 1u) >> 1) & 1u;
          int touched = 0;
          for (int col0 = 0; col0 < p.wpad[s] && ok; col0 += pw) {
            const uint32_t col = tmem_col(r0, col0);
            const int r = static_cast<int>(col >> 8);
            if (!((touched >> r) & 1)) {
              touched |= 1 << r;
              ok = take_region(r);
              if (!ok) break;
              tc_fence_after();
            }
            if (s == 0)
              ok = run_pass(First{}, tmem_base + col, idesc, p.kpan[s], col0 == 0, cpar);
            else if (kps_of(s) == 2)
              ok = run_pass(Two{}, tmem_base + col, idesc, p.kpan[s], col0 == 0, cpar);
            else
              ok = run_pass(One{}, tmem_base + col, idesc, p.kpan[s], col0 == 0, cpar);
            // the first GEMM reads no operand image, so each of its passes
            // can be converted as soon as it completes (every MMA that read
            // the image, the previous tile's last GEMM, completed before it)
            if (ok && s == 0) tc_commit<CG>(bar(knCFull0 + (col0 >> (pw == 256 ? 8 : 7))));
          }
          if (!ok) break;
          if (s > 0) tc_commit<CG>(bar(knCFull));
          p_tmem = tmem_base + (r0 << 8);
          a_tm = !PT && ((p.ptm >> s) & 1);
          ++k;
        }
        if (!ok) break;
        // the unit's passes of the last GEMM, each in the next region
        const uint32_t idesc = make_idesc(FMT, NF, 256u, !(PT && wk));
        const uint32_t cpar = ((k - 1u) >> 1) & 1u;
        for (int j = c.p0; j < c.p1 && ok; ++j) {
          const int r = static_cast<int>(rc.take(NF));
          const uint32_t col = static_cast<uint32_t>(r) * 256u;
          ok = take_region(r);
          if (!ok) break;
          tc_fence_after();
          ok = kps_last == 2 ? run_pass(Two{}, tmem_base + col, idesc, kpan_last, j == c.p0, cpar)
                             : run_pass(One{}, tmem_base + col, idesc, kpan_last, j == c.p0, cpar);
          if (!ok) break;
          tc_commit<CG>(bar(knRFull + r));
        }
      }
      tc_commit<CG>(bar(knDrain));
      drain_wait(bar(knDrain), 0, p.budget_ns);
    }
  } else if (warp >= 2 && warp < 10) {
    // ----------------------------------------- converters (warps 2-9) and
    // ---------------------------------------------------- epilogue (6-9)
    // Every tile: each intermediate accumulator into the operand image, in
    // 128-column chunks, by all eight warps (warp w reads TMEM lanes
    // 32 (w % 4) .. + 31; warps 2-5 take the low 64 columns of a chunk,
    // warps 6-9 the high 64) -- or, ptm bit s set, packed in place by warps 2-5 --
    // then warps 6-9 store the passes of the last GEMM.  An intermediate's completion barrier also means that every
    // earlier MMA, and so every read of the image it overwrites, is done.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int h = warp < 6 ? 0 : 1;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const bool epi = (warp >= 6);
    // epilogue: each warp converts and stores its own 32 rows (boxes of 32
    // rows x 128 bytes) through two staging buffers of its own, so the warps
    // never wait for each other except once per pass, when the region has
    // been read
    const bool two_stg = p.nstg == 2;
    const uint32_t wstg = base + p.off_stg + static_cast<uint32_t>(q * p.nstg) * 4096u;
    const bool elected = (warp == 6 && lane == 0);
    constexpr int NBOX = NF / OBOX_N;
    constexpr int LDS = OBOX_N / 32;
    RegionCursor rc;
    uint32_t k = 0;             // intermediates converted so far
    uint32_t kl = 0;            // of them, intermediates after the first
    uint32_t krx = 0, kry = 0;  // last-GEMM passes read from X / Y so far
    uint32_t nbox = 0;
    bool ok = true;
    for (int it = 0; it < t_count; ++it) {
      const ChainNUnit c = chainn_unit(p, cid, ncl, it);
      for (int s = 0; s < S - 1; ++s) {
        const uint32_t r0 = rc.take(p.wpad[s]);
        // the first GEMM: one completion barrier per pass; later GEMMs: one
        if (s > 0) {
          if (ok) ok = warp_wait(bw, bar(knCFull), kl & 1u);
          ++kl;
          if (ok) tc_fence_after();
        }
        const int nch = p.wpad[s] / 128;
        const int cpp = p.pw[s] / 128;  // chunks per pass
        for (int ch = 0; ch < nch; ++ch) {
          if (s == 0 && (cpp == 1 || !(ch & 1))) {
            if (ok) ok = warp_wait(bw, bar(knCFull0 + (cpp == 1 ? ch : ch >> 1)), static_cast<uint32_t>(it) & 1u);
            if (ok) tc_fence_after();
          }
          if (ok) {
            // packed in tensor memory by the four warps 2-5 (one per lane
            // quadrant: the packing moves columns, which two warps on the
            // same lanes could not share), or into the image by all eight
            if (PT || !((p.ptm >> s) & 1))
              convert_chunk_half<IN>(tmem_base, lane_off, r0, ch, h, row, p_img);
            else if (h == 0) {
              // accumulator columns [128 ch, +128) packed into [64 ch, +64);
              // chunks go in order, so no write reaches an unread column
              const uint32_t treg = tmem_base + lane_off + (r0 << 8);
              rearrange_accumulator_tmem16<IN>(treg + static_cast<uint32_t>(ch * 128), 128,
                                               treg + static_cast<uint32_t>(ch * 64));
            }
            tc_fence_before();
          }
          named_bar_sync(2, 256);
          if (warp == 2 && lane == 0 && ok) {
            // every chunk barrier of the set completes once per intermediate
            // (the MMA thread derives its parities from that): after the last
            // chunk, the ones this width does not use complete too
            const int set = knPChunk + static_cast<int>((k & 1u) * 4u);
            mbar_arrive_cluster(lbar(set + ch));
            if (ch + 1 == nch)
              for (int c2 = nch; c2 < 4; ++c2) mbar_arrive_cluster(lbar(set + c2));
            // the chunk was the last one in its region: the region is free
            const uint32_t r = tmem_col(r0, ch * 128) >> 8;
            if (ch + 1 == nch || (tmem_col(r0, ch * 128 + 128) >> 8) != r)
              mbar_arrive_cluster(lbar(knREmpty + static_cast<int>(r)));
          }
        }
        ++k;
      }
      const int mw = row0(c.mt) + q * 32;  // this warp's first row
      for (int j = c.p0; j < c.p1; ++j) {
        const int r = static_cast<int>(rc.take(NF));
        if (!epi) continue;
        const uint32_t col = static_cast<uint32_t>(r) * 256u;
        if (ok) ok = warp_wait(bw, bar(knRFull + r), (r ? kry : krx) & 1u);
        if (r) ++kry; else ++krx;
        tc_fence_after();
        const uint32_t tsrc = tmem_base + lane_off + col;
        uint32_t v[LDS][32];
        if (ok) {
#pragma unroll
          for (int l = 0; l < LDS; ++l) tmem_ld32(tsrc + static_cast<uint32_t>(l * 32), v[l]);
        }
#pragma unroll 1
        for (int x = 0; x < NBOX; ++x) {
          const uint32_t stg = wstg + (two_stg ? (nbox & 1u) * 4096u : 0u);
          // the store issued two boxes ago (same buffer) has read it
          if (lane == 0 && ok) {
            if (two_stg) bulk_wait_read<1>(); else bulk_wait_read<0>();
          }
          __syncwarp();
          if (ok) {
            tmem_wait_ld();
#pragma unroll
            for (int l = 0; l < LDS; ++l) store_output_row<OUT>(stg, lane, l * 32, v[l]);
            fence_proxy_async_smem();
            if (x + 1 < NBOX) {
#pragma unroll
              for (int l = 0; l < LDS; ++l)
                tmem_ld32(tsrc + static_cast<uint32_t>((x + 1) * OBOX_N + l * 32), v[l]);
            }
          }
          if (x == NBOX - 1) {
            // every warp has read the region: one arrival per CTA on the even CTA
            if (ok) tc_fence_before();
            named_bar_sync(1, 128);
            if (elected && ok) mbar_arrive_cluster(lbar(knREmpty + r));
          }
          __syncwarp();
          // (the odd CTA's rows of the last tile may lie past M)
          if (lane == 0 && ok && mw < p.M) {
            tma_store_3d_hint(&maps.out, stg, j * NF + x * OBOX_N, mw, c.b, pol_stream);
            bulk_commit();
          }
          ++nbox;
        }
      }
    }
    if (epi && lane == 0) bulk_wait_all();
  }

  __syncthreads();
  // neither CTA leaves (or frees tensor memory) while the other may still
  // arrive on its barriers or the even CTA's MMAs may still write it
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, kCols);
  }
}

// Test support: the layout probes of the rearrangement code that tensor
// memory holds an operand for, or that two warps share per lane quadrant.
//   FORM 1: the 16-bit intermediate kept in tensor memory (two-stage chains
//           with resident weights): `acc` [128][width] goes into columns
//           [0, width) in the accumulator layout, rearrange_accumulator_tmem16
//           packs it in place, and columns [0, width / 2) are copied to `out`
//           ([128][width / 2] 32-bit words, row-major).
//   FORM 2: the converters of the pair kernel: `acc` goes into tensor memory
//           as an accumulator that starts in region r0 (column c at
//           tmem_col(r0, c)), eight warps convert it chunk by chunk with
//           convert_chunk_half, and the operand image (width * 256 bytes) is
//           copied to `out`.
// One CTA of 256 threads (FORM 1 uses the first 128).
template <int IN, int FORM>
__global__ void __launch_bounds__(256, 1)
    probe_layout_kernel(const uint32_t* __restrict__ acc, uint32_t* __restrict__ out, int width, uint32_t r0,
                        uint32_t tmem_cols) {
  using namespace ptx;
  static_assert(IN == kInF16 || IN == kInBF16, "16-bit operands");
  static_assert(FORM == 1 || FORM == 2, "probe form");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tslot;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t img = (raw + 1023u) & ~1023u;
  const uint8_t* gimg = smem_raw + (img - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;
  const int row = q * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
  if (warp == 0) {
    tmem_alloc(smem_u32(&tslot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tslot;
  if (warp < 4) {
    for (int c0 = 0; c0 < width; c0 += 32) {
      uint32_t v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = acc[row * width + c0 + i];
      const uint32_t col = FORM == 2 ? tmem_col(r0, c0) : static_cast<uint32_t>(c0);
      tmem_st32(tbase + lane_off + col, v);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (FORM == 1) {
    if (warp < 4) {
      rearrange_accumulator_tmem16<IN>(tbase + lane_off, width);
      for (int c0 = 0; c0 < width / 2; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + static_cast<uint32_t>(c0), v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c0 + i < width / 2) out[row * (width / 2) + c0 + i] = v[i];
      }
    }
  } else {
    const int h = warp >> 2;
    for (int ch = 0; ch < width / 128; ++ch) convert_chunk_half<IN>(tbase, lane_off, r0, ch, h, row, img);
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
