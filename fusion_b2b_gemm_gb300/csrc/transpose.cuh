// Batched 2-D transpose of 32-bit words: out[b][c][r] = in[b][r][c].
//
// The tf32 chain kernels read their weights either as stored ([K][N], an
// MN-major B operand; what plans do) or transposed ([N][K], K-major).  The
// allocation-free tf32 call takes the second form: this kernel turns the
// weights into [N][K] in the library's scratch array first.  Two matrices per
// launch (blockIdx.z = matrix * batch + b); 32x32 tiles through shared
// memory so that reads and writes are both coalesced.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace b2b {

struct TransposeJob {
  const uint32_t* in[2];
  uint32_t* out[2];
  int rows[2], cols[2];  // of the input matrix
  int batch;
  int count;             // matrices in this launch (1 or 2)
};

__global__ void __launch_bounds__(256) transpose32_kernel(const __grid_constant__ TransposeJob job) {
  __shared__ uint32_t tile[32][33];
  const int z = blockIdx.z;
  const int mat = z < job.count * job.batch ? z / job.batch : 0;
  const int b = z % job.batch;
  const int R = job.rows[mat], C = job.cols[mat];
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const bool active = z < job.count * job.batch && r0 < R && c0 < C;
  const uint32_t* in = job.in[mat] + static_cast<size_t>(b) * R * C;
  // Pull this tile's input rows into L2 before waiting for the earlier
  // kernels (the weights may be their output, but a prefetch touches L2
  // only, where their writes land too, and the loads below come after the
  // wait).
  if (active && threadIdx.x < 32 && r0 + static_cast<int>(threadIdx.x) < R)
    ptx::prefetch_l2(in + static_cast<size_t>(r0 + threadIdx.x) * C + c0);
  // Wait for the earlier kernels (the previous chain kernel may read the
  // array written below), then let the chain kernel start.
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();
  if (!active) return;
  uint32_t* out = job.out[mat] + static_cast<size_t>(b) * R * C;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    const int r = r0 + ty + i, c = c0 + tx;
    if (r < R && c < C) tile[ty + i][tx] = in[static_cast<size_t>(r) * C + c];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    const int c = c0 + ty + i, r = r0 + tx;
    if (r < R && c < C) out[static_cast<size_t>(c) * R + r] = tile[tx][ty + i];
  }
}

}  // namespace b2b
