// Fused cascaded fp64 GEMM D = (A.B).C on the warp-level fp64 MMA
// (mma.sync.m8n8k4.f64), with the accumulator-to-operand rearrangement done
// in registers by warp shuffles scheduled by a coordination matrix.
//
// Source: patent "数据处理方法、装置、设备及介质" (Alibaba, 2023), Detailed
// description para. 61-74 (split into 4-thread groups, relation per group,
// other groups by an offset), para. 75-91 (coordination matrix: in round j
// thread i takes value q of thread p into its slot r; the p's of a round are
// distinct) and para. 92-102 (encode p, q, r as unary functions of i per
// round built from add / shift / and operations, then emit the exchange code).
//
// Rule 1 here is the m8n8k4 fp64 accumulator fragment: lane 4g+t holds row g,
// columns 2t and 2t+1 of an 8x8 tile.  Rule 2 is the m8n8k4 A fragment: lane
// 4g+t holds row g, column t of an 8x4 slice.  Two k4 slices cover one 8-col
// accumulator tile, so each 4-lane group exchanges 8 values in 2 rounds.  The
// host derives the relation from the two layouts, builds the coordination
// matrix and packs each round's functions f_j (source lane), the sender-side
// value index and h_j (destination slot) as 2-bit tables indexed by t.
#pragma once

#include <cstdint>

namespace b2b {

struct F64Params {
  int batch, M, K;
  int m8_tiles;           // ceil(M / 8)
  long long total;        // batch * m8_tiles warp tasks
  uint32_t fsrc[2];       // round j: source lane (in the group) of receiver t, bits 2t..2t+1
  uint32_t qsend[2];      // round j: which of its two values sender t offers
  uint32_t hslot[2];      // round j: slot of receiver t that the value fills
};

__device__ __forceinline__ void dmma_m8n8k4(double& d0, double& d1, double a, double b) {
  asm volatile("mma.sync.aligned.m8n8k4.row.col.f64.f64.f64.f64 {%0, %1}, {%2}, {%3}, {%0, %1};"
               : "+d"(d0), "+d"(d1)
               : "d"(a), "d"(b));
}

// Rearrange one 8-column accumulator tile (c0, c1 of this lane) into the two
// A fragments of the k4 slices that cover it (a0: first slice, a1: second).
__device__ __forceinline__ void f64_rearrange_tile(const F64Params& p, double c0, double c1,
                                                   double& a0, double& a1) {
  const int lane = threadIdx.x & 31;
  const int t = lane & 3;
  const int grp = lane & ~3;
  a0 = 0.0;
  a1 = 0.0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int src = grp | static_cast<int>((p.fsrc[j] >> (2 * t)) & 3u);
    const double offer = ((p.qsend[j] >> (2 * t)) & 1u) ? c1 : c0;
    const double got = __shfl_sync(0xffffffffu, offer, src);
    if ((p.hslot[j] >> (2 * t)) & 1u)
      a1 = got;
    else
      a0 = got;
  }
}

// One warp per 8-row task (batch b, rows m0..m0+7), grid-strided.
// STAGES == 1 computes the single GEMM D = A.B (N2 unused).
template <int N1, int N2, int STAGES>
__global__ void __launch_bounds__(128) chain_f64_kernel(const double* __restrict__ A,
                                                        const double* __restrict__ B,
                                                        const double* __restrict__ C,
                                                        double* __restrict__ D, const F64Params p) {
  static_assert(N1 % 8 == 0 && N2 % 8 == 0, "8-column tiles");
  // Wait for the previous kernel in the stream (programmatic launch).  No
  // early trigger here: this grid has many more CTAs than fit at once, and
  // waiting CTAs of the next launch would take their slots.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       w < p.total; w += nwarps) {
    const int b = static_cast<int>(w / p.m8_tiles);
    const int m0 = static_cast<int>(w % p.m8_tiles) * 8;
    const double* Ab = A + static_cast<size_t>(b) * p.M * p.K;
    const double* Bb = B + static_cast<size_t>(b) * p.K * N1;
    const int row = m0 + g;
    const bool valid = row < p.M;

    double c[N1 / 8][2];
#pragma unroll
    for (int j = 0; j < N1 / 8; ++j) c[j][0] = c[j][1] = 0.0;
#pragma unroll 2
    for (int s = 0; s < p.K / 4; ++s) {
      const double a = valid ? __ldg(Ab + static_cast<size_t>(row) * p.K + 4 * s + t) : 0.0;
#pragma unroll
      for (int j = 0; j < N1 / 8; ++j)
        dmma_m8n8k4(c[j][0], c[j][1], a, __ldg(Bb + static_cast<size_t>(4 * s + t) * N1 + 8 * j + g));
    }

    if constexpr (STAGES == 1) {
      if (valid) {
        double* Dr = D + (static_cast<size_t>(b) * p.M + row) * N1;
#pragma unroll
        for (int j = 0; j < N1 / 8; ++j)
          *reinterpret_cast<double2*>(Dr + 8 * j + 2 * t) = make_double2(c[j][0], c[j][1]);
      }
    } else {
      // Rule 1 -> rule 2: accumulator tiles become the A fragments of GEMM2.
      double af[N1 / 4];
#pragma unroll
      for (int j = 0; j < N1 / 8; ++j) f64_rearrange_tile(p, c[j][0], c[j][1], af[2 * j], af[2 * j + 1]);

      const double* Cb = C + static_cast<size_t>(b) * N1 * N2;
      double d[N2 / 8][2];
#pragma unroll
      for (int j = 0; j < N2 / 8; ++j) d[j][0] = d[j][1] = 0.0;
#pragma unroll
      for (int s = 0; s < N1 / 4; ++s) {
#pragma unroll
        for (int j = 0; j < N2 / 8; ++j)
          dmma_m8n8k4(d[j][0], d[j][1], af[s], __ldg(Cb + static_cast<size_t>(4 * s + t) * N2 + 8 * j + g));
      }
      if (valid) {
        double* Dr = D + (static_cast<size_t>(b) * p.M + row) * N2;
#pragma unroll
        for (int j = 0; j < N2 / 8; ++j)
          *reinterpret_cast<double2*>(Dr + 8 * j + 2 * t) = make_double2(d[j][0], d[j][1]);
      }
    }
  }
}

// Test support: run f64_rearrange_tile on `tiles` tiles of one warp.
__global__ void probe_f64_rearrange_kernel(const double* cfrag, double* afrag, int tiles,
                                           const F64Params p) {
  const int lane = threadIdx.x & 31;
  for (int j = 0; j < tiles; ++j) {
    const double c0 = cfrag[lane * tiles * 2 + 2 * j];
    const double c1 = cfrag[lane * tiles * 2 + 2 * j + 1];
    double a0, a1;
    f64_rearrange_tile(p, c0, c1, a0, a1);
    afrag[lane * tiles * 2 + 2 * j] = a0;
    afrag[lane * tiles * 2 + 2 * j + 1] = a1;
  }
}

}  // namespace b2b
