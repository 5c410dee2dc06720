// Three cascaded GEMMs with 16-bit operands on pairs of SMs (tcgen05,
// cta_group::2, sm_103a):
//
//   P1 = A.W0 -> round -> P2 = P1.W1 -> round -> E = P2.W2
//
// Source of the method: patent "数据处理方法、装置、设备及介质" (Alibaba, 2023),
// Detailed description para. 41 (three cascaded operators), para. 54-60 (the
// result of one operator is rearranged and handed to the next without going
// through memory) and para. 103-110 (rearrangement through shared memory).
//
// Every weight is streamed through the SMs once per 256-row tile, so the
// weights, not A, dominate the bytes an SM must load.  Two CTAs of a cluster
// share each MMA (M = 256): each holds its own 128 rows of A, of the
// intermediate and of every accumulator, and half of the columns of every
// weight panel, which halves the weight traffic and the shared memory a
// weight stage needs per SM.  The converters turn an accumulator row into the
// K-major 128-byte-swizzled operand image of the next GEMM in shared memory
// (one image, P1 then P2).  Tensor memory holds two 256-column regions, X and
// Y: GEMM1 writes X, GEMM2 writes Y, and the passes of the last GEMM
// (NF columns each) alternate X, Y, so that the epilogue of one pass overlaps
// the MMAs of the next.
//
// Roles (352 threads, one CTA per SM, persistent over 256-row tiles):
//   warp 0     producer: one ring of 16 KB slots in the order the MMAs read
//              them (GEMM1: an A panel and this CTA's half of a weight panel;
//              GEMM2 and the passes: a weight half panel), so the weights of
//              GEMM2 and of the passes can have the whole ring in flight
//   warp 1     TMEM allocation (both CTAs); the even CTA's lane 0 issues MMAs
//   warps 2-9  converters (accumulator -> operand image), half of the
//              columns each for the two warps that share a TMEM lane quadrant
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

// Barrier slots (8 bytes each) at Chain3Params::off_bar.
enum : int {
  k3Full = 0,       // [16] ring slot filled (even CTA's: armed by it for both CTAs' copies)
  k3Empty = 16,     // [16] ring slot consumed
  k3CFull = 32,     // [2] GEMM1 (X) / GEMM2 (Y) accumulator complete (converters)
  k3PChunk = 34,    // [2][2] half c of P1 / P2 written in both CTAs (even CTA's)
  k3PEmpty = 38,    // last pass of a tile complete: the operand image is free
  k3RFull = 39,     // [2] X / Y holds a pass product (epilogue)
  k3REmpty = 41,    // [2] X / Y pass product drained in both CTAs (even CTA's)
  k3Drain = 43,     // every MMA complete (exit)
  k3SlotTmem = 44,  // uint32 TMEM base, then the int abort flag
  k3SlotReady = 45, // uint32: ring slots whose copies have landed (even CTA)
};

constexpr int kChain3Threads = 384;

struct Chain3Params {
  int batch, M, K;
  int m_tiles, total_tiles;  // 256-row tiles per batch, in all
  int npass;                 // NF-column passes of the last GEMM
  int kpan0;                 // 64-element K panels of A
  int nslot, nstg;           // ring slots (16 KB each) and staging buffers per warp
  uint32_t off_ring, off_p, off_stg, off_bar;
  int w_merged;              // bit s: weight s is read as one 4-D box per half panel
  int split;                 // leftover tiles whose passes are split between two clusters
  uint32_t debug;            // test support: bit 0 = the first weight stage is never filled
  int* status;
  unsigned long long budget_ns;
};

// Work units of a cluster.  Tiles are dealt to the clusters in strides; when
// they do not divide evenly, the `split` leftover tiles are each shared by two
// clusters, one taking the first half of the last GEMM's passes and the other
// the rest (both compute GEMM1 and GEMM2), and these half units come first.
// That shortens the longest cluster's work and starts half of the clusters
// out of step with the others, which spreads their HBM-bound GEMM1 phases.
struct Chain3Unit {
  int b, mt, p0, p1;  // batch, 256-row tile, passes [p0, p1)
};
__device__ __forceinline__ int chain3_units(const Chain3Params& p, int cid, int ncl) {
  if (p.split > 0) return p.total_tiles / ncl + (cid < 2 * p.split ? 1 : 0);
  return cid < p.total_tiles ? (p.total_tiles - cid + ncl - 1) / ncl : 0;
}
__device__ __forceinline__ Chain3Unit chain3_unit(const Chain3Params& p, int cid, int ncl, int i) {
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
  Chain3Unit u;
  u.b = tile / p.m_tiles;
  u.mt = tile - u.b * p.m_tiles;
  u.p0 = p0;
  u.p1 = p1;
  return u;
}

template <int IN, int OUT, int N1P, int N2P, int NF>
__global__ void __launch_bounds__(kChain3Threads, 1)
    chain3_kernel(const __grid_constant__ CUtensorMap tmA,
                  const __grid_constant__ CUtensorMap tmW0,
                  const __grid_constant__ CUtensorMap tmW1,
                  const __grid_constant__ CUtensorMap tmW2,
                  const __grid_constant__ CUtensorMap tmOut,
                  const __grid_constant__ Chain3Params p) {
  using namespace ptx;
  static_assert(IN == kInF16 || IN == kInBF16, "16-bit operands");
  static_assert((N1P == 128 || N1P == 256) && (N2P == 128 || N2P == 256) && (NF == 128 || NF == 256),
                "padded widths");
  constexpr int CG = 2;
  constexpr int CK = 64;           // K elements per 128-byte panel
  constexpr int KSTEP = 16;        // K of one MMA
  constexpr int WBOX_N = 64;       // weight columns per 128-byte block
  constexpr int WBOX_BYTES = CK * 128;
  constexpr int OSZ = (OUT == kOutF32) ? 4 : 2;
  constexpr int OBOX_N = 128 / OSZ;
  constexpr uint32_t FMT = (IN == kInF16) ? 0u : 1u;
  constexpr uint32_t kCols = 512;
  constexpr uint32_t kX = 0, kY = 256;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + p.off_bar;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + p.off_bar + 8 * k3SlotTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 16; ++i) {
      mbar_init(bar(k3Full + i), 1);
      mbar_init(bar(k3Empty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(k3CFull + i), 1);
      mbar_init(bar(k3PChunk + 2 * i), 2);
      mbar_init(bar(k3PChunk + 2 * i + 1), 2);
      mbar_init(bar(k3RFull + i), 1);
      mbar_init(bar(k3REmpty + i), 2);
    }
    mbar_init(bar(k3PEmpty), 1);
    mbar_init(bar(k3Drain), 1);
    *abort_flag = 0;
    *reinterpret_cast<volatile uint32_t*>(gbase + p.off_bar + 8 * k3SlotReady) = 0u;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(tmem_slot), kCols);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before anything arrives on them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_launch_dependents();
  grid_dependency_wait();

  BoundedWait bw{abort_flag, p.status, p.budget_ns, kTimeoutCode};
  // Waits on barriers that threads of the peer CTA arrive on (the same
  // default-scope wait: the cluster-scope acquire form costs more and the
  // remote arrives are ordered by the barrier itself).
  BoundedWait bwm = bw;
  auto lbar = [&](int i) -> uint32_t { return mapa_shared(bar(i), 0); };

  // Work units (256-row tiles, or halves of their last GEMM) of this
  // cluster; this CTA's 128 rows of each.
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);
  const int t_count = chain3_units(p, cid, ncl);
  auto row0 = [&](int mt) -> int { return mt * 256 + static_cast<int>(rank) * 128; };
  const uint32_t p_img = base + p.off_p;

  // Ring slots of one unit, in the order the MMAs read them: GEMM1 (kpan0
  // panels, two slots each: A, weight), GEMM2 (N1P / 64 slots), then every
  // pass of the unit (N2P / 64 slots each).
  const int np1 = p.kpan0, np2 = N1P / CK, np3 = N2P / CK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmW0);
      prefetch_tmap(&tmW1);
      prefetch_tmap(&tmW2);
      prefetch_tmap(&tmOut);
      uint32_t slot = 0, phase = 0;
      uint64_t issued = 0;
      bool ok = true;
      for (int it = 0; it < t_count && ok; ++it) {
        const Chain3Unit c = chain3_unit(p, cid, ncl, it);
        const int m0 = row0(c.mt);
        // the ring reaches only a few panels into the next unit's GEMM1: pull
        // the next unit's A into L2 now
        if (it + 1 < t_count) {
          const Chain3Unit n = chain3_unit(p, cid, ncl, it + 1);
          for (int q = 0; q < np1; ++q) tma_prefetch_l2_3d(&tmA, q * CK, row0(n.mt), n.b);
        }
        const int per_unit = 2 * np1 + np2 + (c.p1 - c.p0) * np3;
        for (int q = 0; q < per_unit; ++q) {
          if (!bw.wait(bar(k3Empty + slot), phase ^ 1u)) {
            ok = false;
            break;
          }
          // which operand, K panel and (weights) this CTA's columns
          const CUtensorMap* wm = nullptr;
          int kb, n0 = 0, wcols = 0, s = -1;
          if (q < 2 * np1) {
            kb = q >> 1;
            if (q & 1) {
              s = 0; wm = &tmW0; wcols = N1P / 2; n0 = static_cast<int>(rank) * wcols;
            }
          } else if (q < 2 * np1 + np2) {
            s = 1; wm = &tmW1; kb = q - 2 * np1; wcols = N2P / 2; n0 = static_cast<int>(rank) * wcols;
          } else {
            const int r = q - 2 * np1 - np2;
            const int j = r / np3;
            s = 2; wm = &tmW2; kb = r - j * np3; wcols = NF / 2;
            n0 = (c.p0 + j) * NF + static_cast<int>(rank) * wcols;
          }
          const uint32_t dst = base + p.off_ring + slot * static_cast<uint32_t>(kPanelBytes);
          const uint32_t fb = lbar(k3Full + slot);
          const uint32_t bytes = s < 0 ? static_cast<uint32_t>(kPanelBytes) : 128u * static_cast<uint32_t>(wcols);
          // Only the even CTA arms its barrier, for both CTAs' copies; the odd
          // CTA's copies may land first (the transaction count then dips
          // below zero until the arming, which the barrier allows).
          if (leader) mbar_arrive_expect_tx(bar(k3Full + slot), 2u * bytes);
          // test support: the very first slot is armed but never filled
          if (!((p.debug & 1u) && issued == 0)) {
            if (s < 0) {
              tma_load_3d_pair(dst, &tmA, fb, kb * CK, m0, c.b);
            } else if ((p.w_merged >> s) & 1) {
              tma_load_4d_pair(dst, wm, fb, 0, kb * CK, n0 / WBOX_N, c.b);
            } else {
              for (int j = 0; j < wcols / WBOX_N; ++j)
                tma_load_3d_pair(dst + j * WBOX_BYTES, wm, fb, n0 + j * WBOX_N, kb * CK, c.b);
            }
          }
          ++issued;
          if (++slot == static_cast<uint32_t>(p.nslot)) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      // copies in flight land before exit (the even CTA's barriers count both
      // CTAs' copies; the odd CTA waits at the cluster barrier before exit)
      const uint64_t n = static_cast<uint64_t>(p.nslot);
      const uint64_t tail = !leader ? 0 : (issued < n ? issued : n);
      for (uint64_t j = 0; j < tail; ++j) {
        const uint64_t idx = issued - 1 - j;
        drain_wait(bar(k3Full + static_cast<int>(idx % n)), static_cast<uint32_t>((idx / n) & 1u),
                   p.budget_ns);
      }
    }
  } else if (warp == 11) {
    // ------------------------------------------- slot watcher (even CTA)
    if (lane == 0 && leader) {
      uint32_t slot = 0, phase = 0, n = 0;
      const uint32_t ready = bar(k3SlotReady);
      bool ok = true;
      for (int it = 0; it < t_count && ok; ++it) {
        const Chain3Unit c = chain3_unit(p, cid, ncl, it);
        const int per_unit = 2 * np1 + np2 + (c.p1 - c.p0) * np3;
        for (int q = 0; q < per_unit && ok; ++q) {
          ok = bw.wait(bar(k3Full + slot), phase);
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
      uint32_t u[2] = {0u, 0u};  // pass products written to X / Y so far
      bool ok = true;
      // region r's last pass product has been drained by the epilogue in
      // both CTAs (an accumulator of GEMM1 / GEMM2 there has been read once
      // the converters reported its operand image complete)
      auto drained = [&](int r) -> bool { return u[r] == 0 || bwm.wait(bar(k3REmpty + r), (u[r] - 1u) & 1u); };
      // One weight stage: four MMAs with A from the A ring (a_smem) or from
      // the operand image (K panel kb)
      // the next `need` slots have landed once the watcher's count reaches
      // consumed + need
      uint32_t consumed = 0, seen = 0;
      const uint32_t ready = bar(k3SlotReady);
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
      // chunk >= 0: the K panels from kb on need half `chunk` of the operand
      // image, whose barrier is waited for here.  GEMM1 (a_smem): the A panel
      // is in this slot and the weight half panel in the next.
      auto stage_mmas = [&](uint32_t d, uint32_t idesc, bool a_smem, int kb, int chunk = -1,
                            uint32_t cpar = 0) -> bool {
        const uint32_t need = a_smem ? 2u : 1u;
        if (!stage_ready(need)) return false;
        if (chunk >= 0 && !bwm.wait(bar(chunk), cpar)) return false;
        consumed += need;
        tc_fence_after();
        const uint32_t s0 = slot;
        const uint32_t s1 = a_smem ? (slot + 1u == static_cast<uint32_t>(p.nslot) ? 0u : slot + 1u) : slot;
        const uint32_t wb = base + p.off_ring + s1 * static_cast<uint32_t>(kPanelBytes);
        const uint32_t sa = a_smem ? base + p.off_ring + s0 * static_cast<uint32_t>(kPanelBytes)
                                   : p_img + static_cast<uint32_t>(kb) * kPanelBytes;
        const uint32_t acc0 = kb != 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < CK / KSTEP; ++kk)
          mma_ss<false, CG>(d, desc_sw128(sa + kk * 32u, 16u, 1024u),
                            desc_sw128(wb + kk * KSTEP * 128u, WBOX_BYTES, 1024u), idesc, kk ? 1u : acc0);
        tc_commit<CG>(bar(k3Empty + s0));
        if (a_smem) tc_commit<CG>(bar(k3Empty + s1));
        slot = s1 + 1u == static_cast<uint32_t>(p.nslot) ? 0u : s1 + 1u;
        return true;
      };
      for (int it = 0; it < t_count && ok; ++it) {
        const Chain3Unit c = chain3_unit(p, cid, ncl, it);
        const uint32_t par = static_cast<uint32_t>(it) & 1u;
        // GEMM1 -> X
        ok = drained(0);
        if (!ok) break;
        tc_fence_after();
        {
          const uint32_t idesc = make_idesc(FMT, N1P, 256u, true);
          for (int kb = 0; kb < np1 && ok; ++kb) ok = stage_mmas(tmem_base + kX, idesc, true, kb);
        }
        if (!ok) break;
        tc_commit<CG>(bar(k3CFull + 0));
        // GEMM2 -> Y, A = P1, each half as soon as the converters finish it
        ok = drained(1);
        if (!ok) break;
        {
          const uint32_t idesc = make_idesc(FMT, N2P, 256u, true);
          for (int kb = 0; kb < np2 && ok; ++kb)
            ok = stage_mmas(tmem_base + kY, idesc, false, kb,
                            kb == 0 ? k3PChunk : (kb == np2 / 2 ? k3PChunk + 1 : -1), par);
        }
        if (!ok) break;
        tc_commit<CG>(bar(k3CFull + 1));
        // the unit's passes of GEMM3 -> X, Y, X, ..., A = P2 (the first pass
        // writes X, drained long ago, and takes each half of P2 as soon as
        // the converters finish it)
        const uint32_t idesc = make_idesc(FMT, NF, 256u, true);
        for (int j = c.p0; j < c.p1 && ok; ++j) {
          const int r = (j - c.p0) & 1;
          ok = drained(r);
          if (!ok) break;
          for (int kb = 0; kb < np3 && ok; ++kb)
            ok = stage_mmas(tmem_base + (r ? kY : kX), idesc, false, kb,
                            j != c.p0 ? -1 : (kb == 0 ? k3PChunk + 2 : (kb == np3 / 2 ? k3PChunk + 3 : -1)), par);
          if (!ok) break;
          tc_commit<CG>(bar(k3RFull + r));
          ++u[r];
        }
        if (!ok) break;
        tc_commit<CG>(bar(k3PEmpty));
      }
      tc_commit<CG>(bar(k3Drain));
      drain_wait(bar(k3Drain), 0, p.budget_ns);
    }
  } else if (warp >= 2 && warp < 10) {
    // ----------------------------------------- converters (warps 2-9) and
    // ---------------------------------------------------- epilogue (6-9)
    // Every tile: GEMM1's accumulator (X) then GEMM2's (Y) into the operand
    // image, by all eight warps (warp w reads TMEM lanes 32 (w % 4) .. + 31;
    // warps 2-5 take the low half of the columns, warps 6-9 the high half),
    // then warps 6-9 store the passes of the last GEMM.  The image is free
    // once the previous tile's last pass has completed (P1) or once GEMM2 has
    // (P2, implied by GEMM2's completion barrier).
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int h = warp < 6 ? 0 : 1;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const bool epi = (warp >= 6);
    // epilogue: each warp converts and stores its own 32 rows (boxes of 32
    // rows x 128 bytes) through two staging buffers of its own, so the warps
    // never wait for each other except once per pass, when the region has
    // been read
    const uint32_t wstg = base + p.off_stg + static_cast<uint32_t>(q) * 2u * 4096u;
    const bool elected = (warp == 6 && lane == 0);
    constexpr int NBOX = NF / OBOX_N;
    constexpr int LDS = OBOX_N / 32;
    uint32_t k[2] = {0u, 0u};
    uint32_t nbox = 0;
    bool ok = true;
    for (int it = 0; it < t_count; ++it) {
      const Chain3Unit c = chain3_unit(p, cid, ncl, it);
      const uint32_t par = static_cast<uint32_t>(it) & 1u;
      for (int g = 0; g < 2; ++g) {
        if (g == 0 && it > 0 && ok) ok = warp_wait(bw, bar(k3PEmpty), par ^ 1u);
        if (ok) ok = warp_wait(bw, bar(k3CFull + g), par);
        if (ok) tc_fence_after();
        // a 256-column accumulator in two halves (each warp 64 columns of
        // each), reported one at a time; a 128-column one in one step
        const int width = g == 0 ? N1P : N2P;
        const int nch = width == 256 ? 2 : 1;
        const int cw = width / (2 * nch);  // columns per warp and chunk
        for (int ch = 0; ch < nch; ++ch) {
          if (ok) {
            const int c0 = ch * (width / nch) + h * cw;
            rearrange_accumulator<IN>(tmem_base + lane_off + (g == 0 ? kX : kY) + static_cast<uint32_t>(c0), cw,
                                      row, p_img + static_cast<uint32_t>(c0 / 64) * kPanelBytes);
            tc_fence_before();
          }
          named_bar_sync(2, 256);
          if (warp == 2 && lane == 0 && ok) {
            mbar_arrive_cluster(lbar(k3PChunk + 2 * g + ch));
            if (nch == 1) mbar_arrive_cluster(lbar(k3PChunk + 2 * g + 1));
          }
        }
      }
      if (!epi) continue;
      const int mw = row0(c.mt) + q * 32;  // this warp's first row
      for (int j = c.p0; j < c.p1; ++j) {
        const int r = (j - c.p0) & 1;
        if (ok) ok = warp_wait(bw, bar(k3RFull + r), k[r] & 1u);
        ++k[r];
        tc_fence_after();
        const uint32_t tsrc = tmem_base + lane_off + (r ? kY : kX);
        uint32_t v[LDS][32];
        if (ok) {
#pragma unroll
          for (int l = 0; l < LDS; ++l) tmem_ld32(tsrc + static_cast<uint32_t>(l * 32), v[l]);
        }
#pragma unroll 1
        for (int x = 0; x < NBOX; ++x) {
          const uint32_t stg = wstg + (nbox & 1u) * 4096u;
          // the store issued two boxes ago (same buffer) has read it
          if (lane == 0 && ok) bulk_wait_read<1>();
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
            if (elected && ok) mbar_arrive_cluster(lbar(k3REmpty + r));
          }
          __syncwarp();
          // (the odd CTA's rows of the last tile may lie past M)
          if (lane == 0 && ok && mw < p.M) {
            tma_store_3d(&tmOut, stg, j * NF + x * OBOX_N, mw, c.b);
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

}  // namespace b2b
