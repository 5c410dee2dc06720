// C ABI of the fused cascaded GEMM library (include/b2b.h).
//
// b2b_plan_create is the operator-determination and relation-determination
// step (patent "数据处理方法、装置、设备及介质", Alibaba 2023, Detailed
// description para. 46-53, apparatus modules 51 and 52, para. 140-142): the
// caller names the chain, the data type fixes the accumulator layout (rule 1)
// and the operand layout (rule 2), and the plan picks the compiled
// rearrangement and tiling.  b2b_run is the rearrangement module 53
// (para. 143): one kernel launch that computes, rearranges and consumes every
// intermediate on chip.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "b2b.h"
#include "chain_f64.cuh"
#include "registry.h"
#include "transpose.cuh"

using namespace b2b;

static_assert(kMaxStages == B2B_MAX_STAGES, "stage limit of the C interface");

namespace {

constexpr uint64_t kDefaultBudgetNs = 2000000000ull;
constexpr uint64_t kMinBudgetNs = 1000000ull;  // 1 ms
constexpr int kSmemOptin = 232448;         // 227 KB per CTA on sm_100 / sm_103
constexpr int kSmemBudget = kSmemOptin - 1024;  // minus the 1024-byte alignment slack

enum PlanKind : int {
  kPlanChainTC = 0,
  kPlanGemmTC = 1,
  kPlanChainF64 = 2,
  kPlanGemmF64 = 3,
  kPlanEmpty = 4
};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int64_t pad64(int64_t n) { return (n + 63) / 64 * 64; }

// Width of a compiled panel set that holds n columns: 64, 128 or 256.
int64_t pad_width(int64_t n) { return n <= 64 ? 64 : (n <= 128 ? 128 : 256); }

uint32_t pow2_cols(uint32_t n) {
  uint32_t c = 32;
  while (c < n) c <<= 1;
  return c;
}

const ChainKernelEntry* find_chain_kernel(int in, int out, int S, int n1p, int n2p, int nf,
                                          bool res) {
  const ChainTable tables[] = {chain_table_f16(), chain_table_bf16(), chain_table_tf32()};
  for (const ChainTable& t : tables)
    for (int i = 0; i < t.count; ++i) {
      const ChainKernelEntry& e = t.entries[i];
      if (e.in == in && e.out == out && e.S == S && e.nf == nf && e.res == res &&
          (S < 2 || e.n1p == n1p) && (S < 3 || e.n2p == n2p))
        return &e;
    }
  return nullptr;
}

const ChainNEntry* find_chainn_kernel(int in, int out, int nf, bool tf0) {
  const ChainNTable tables[] = {chainn_table_f16(), chainn_table_bf16(), chainn_table_tf32()};
  for (const ChainNTable& t : tables)
    for (int i = 0; i < t.count; ++i) {
      const ChainNEntry& e = t.entries[i];
      if (e.in == in && e.out == out && e.nf == nf && e.tf0 == tf0) return &e;
    }
  return nullptr;
}

// Rearrangement relation of the fp64 path and its coordination matrix
// (patent para. 61-102).  Rule 1, the m8n8k4 fp64 accumulator: lane 4g+t
// holds row g, columns 2t and 2t+1.  Rule 2, the m8n8k4 A operand: lane
// 4g+t holds row g, column t.  One 8-column accumulator tile feeds two k4
// slices: receiver t of a group needs column 4h + t for its slot h, which
// sender (4h + t) / 2 holds as its value (4h + t) % 2.
struct F64Tables {
  uint32_t fsrc[2], qsend[2], hslot[2];
  bool ok;
};

F64Tables f64_tables() {
  static F64Tables tab{};
  static std::once_flag once;
  std::call_once(once, [] {
    int st[8], sr[8], P[8], Q[8], R[8];
    for (int t = 0; t < 4; ++t)
      for (int h = 0; h < 2; ++h) {
        const int col = 4 * h + t;
        st[t * 2 + h] = col / 2;
        sr[t * 2 + h] = col % 2;
      }
    tab.ok = b2b_coordination_matrix(4, 2, st, sr, P, Q, R) == B2B_OK;
    if (!tab.ok) return;
    for (int j = 0; j < 2; ++j) {
      tab.fsrc[j] = tab.qsend[j] = tab.hslot[j] = 0;
      for (int i = 0; i < 4; ++i) {
        const int p = P[i * 2 + j], q = Q[i * 2 + j], r = R[i * 2 + j];
        tab.fsrc[j] |= static_cast<uint32_t>(p) << (2 * i);
        tab.hslot[j] |= static_cast<uint32_t>(r) << (2 * i);
        tab.qsend[j] |= static_cast<uint32_t>(q) << (2 * p);  // sender p offers its value q
      }
    }
  });
  return tab;
}

b2b_status_t check_device(int* dev_out, int* sms_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_DEVICE;
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return B2B_ERR_DEVICE;
  if (dev_out) *dev_out = dev;
  if (sms_out) *sms_out = sms;
  return B2B_OK;
}

}  // namespace

struct b2b_plan_s {
  int kind;
  b2b_dtype_t dtype;
  int device;
  int sms;
  int stages;
  int64_t batch, M, K, N[kMaxStages];
  int in_kind, out_kind, esz, osz;
  bool tf0;  // mixed-type cascade: the first GEMM on tf32 operands (fp32 A, W0)
  int n1p, n2p, nf;
  bool res;
  ChainParams prm;
  // Cascades of 16-bit GEMMs with three or more stages (or an intermediate
  // wider than 256 columns) run chainn_kernel on clusters of two CTAs.
  bool sn;
  ChainNParams pn;
  int smem_bytes, grid, threads;
  const void* fn;
  F64Params f64;
  int* d_status;
  uint64_t budget_ns;
  uint32_t debug;
  // tf32 weights: read as stored (MN-major), or (w_kmajor, the
  // allocation-free call only) transposed to [N][K] into d_wt before every
  // run, which then launches two kernels
  bool w_kmajor;
  void* d_wt;
  size_t wt_bytes;
  // resident weights: the tile schedule (host copy, then device copy)
  std::vector<int> sched_host;
  int* d_sched;
  // Encoded tensor maps of recent runs, keyed by the pointer set (encoding
  // costs host time on every call otherwise).  Guarded by `mu`.
  struct MapSet {
    const void* key[kMaxStages + 2];
    ChainNMaps maps;
    uint64_t stamp;
  };
  std::mutex mu;
  MapSet cache[8];
  int cache_n;
  uint64_t clock;
};

namespace {

std::vector<int> res_schedule(int64_t batch, int64_t m_tiles, int G);

// Which intermediates of a pair-kernel cascade stay in tensor memory (bit s
// for intermediate s, of padded width wpad[s]): a 16-bit intermediate of at
// most 256 columns, unless the GEMM after next would overwrite its region
// while the next GEMM still reads it (a next intermediate wider than 256
// columns takes both regions; a second pass of the last GEMM takes the
// region of the last intermediate).  tf32 chains keep theirs in tensor
// memory in their own form.
int chainn_tmem_mask(bool pt, int nint, const int* wpad, int npass) {
  int mask = 0;
  for (int s = 0; s < nint; ++s) {
    const bool next_fits = (s + 1 < nint) ? wpad[s + 1] <= 256 : npass == 1;
    if (!pt && wpad[s] <= 256 && next_fits) mask |= 1 << s;
  }
  return mask;
}

// Cascades of 16-bit GEMMs on CTA pairs (chainn_kernel): 256-row tiles,
// intermediates padded to a multiple of 128 columns (at most 512), every GEMM
// in passes of at most 256 columns; shared memory holds the operand image of
// the widest intermediate that does not stay in tensor memory, two staging
// buffers per epilogue warp, and the ring of 16 KB slots in what is left.
b2b_status_t setup_chainn(b2b_plan_s* p) {
  const int S = p->stages;
  p->sn = true;
  p->res = false;
  ChainNParams& c = p->pn;
  std::memset(&c, 0, sizeof(c));
  c.batch = static_cast<int>(p->batch);
  c.M = static_cast<int>(p->M);
  c.K = static_cast<int>(p->K);
  c.S = S;
  c.m_tiles = static_cast<int>((p->M + 255) / 256);
  const int64_t tiles = p->batch * c.m_tiles;
  if (tiles > (1ll << 30)) return B2B_ERR_UNSUPPORTED;
  c.total_tiles = static_cast<int>(tiles);
  p->nf = p->N[S - 1] > 128 ? 256 : 128;
  // a two-GEMM tf32 chain: the intermediate (at most 256 columns) stays in
  // tensor memory and the second GEMM runs in one pass
  const bool pt = p->in_kind == kInTF32;
  if (pt && (S != 2 || p->N[0] > 256 || p->N[1] > 256)) return B2B_ERR_UNSUPPORTED;
  // 128-byte K panels: 64 16-bit or 32 tf32 elements
  const int ck = pt ? 32 : 64;
  c.kpan[0] = static_cast<int>(p->tf0 || pt ? (p->K + 31) / 32 : (p->K + 63) / 64);
  for (int s = 0; s < S - 1; ++s) {
    const int w = static_cast<int>((p->N[s] + 127) / 128 * 128);
    if (w > 512) return B2B_ERR_UNSUPPORTED;
    c.wpad[s] = w;
    // passes of 256 columns where they tile the width, else of 128
    c.pw[s] = (w % 256 == 0) ? 256 : 128;
    c.kpan[s + 1] = w / ck;
    // the first GEMM: an A slot and a weight slot per K panel; later GEMMs:
    // one weight slot per K panel, or per two 16-bit ones with 128-column
    // passes
    const int kps = (!pt && s > 0 && c.pw[s] == 128) ? 2 : 1;
    c.slots0 += (w / c.pw[s]) * (s == 0 ? 2 * c.kpan[s] : c.kpan[s] / kps);
  }
  c.pw[S - 1] = p->nf;
  c.npass = static_cast<int>((p->N[S - 1] + p->nf - 1) / p->nf);
  p->n1p = c.wpad[0];
  p->n2p = S >= 3 ? c.wpad[1] : 0;
  // intermediates packed in tensor memory where they were accumulated; the
  // operand image holds the others
  c.ptm = chainn_tmem_mask(pt, S - 1, c.wpad, c.npass);
  int wimg = 0;
  for (int s = 0; s < S - 1; ++s)
    if (!((c.ptm >> s) & 1)) wimg = std::max(wimg, c.wpad[s]);
  const uint32_t p_bytes = pt ? 0u : 256u * static_cast<uint32_t>(wimg);
  // the rest of shared memory: ring slots of 16 KB (an A panel or a weight
  // half panel each), at most sixteen, after one or two 4 KB staging buffers
  // per epilogue warp (two, unless one buffer buys a ring slot in a ring of
  // fewer than six)
  auto slots_with = [&](int nstg) -> int {
    const int64_t room = kSmemBudget - kBarBytes - int64_t(p_bytes) - int64_t(nstg) * kPanelBytes;
    return static_cast<int>(std::min<int64_t>(16, room / kPanelBytes));
  };
  c.nstg = (slots_with(2) < 6 && slots_with(1) > slots_with(2)) ? 1 : 2;
  c.nslot = slots_with(c.nstg);
  if (c.nslot < 4) return B2B_ERR_UNSUPPORTED;
  c.off_ring = 0;
  c.off_p = static_cast<uint32_t>(c.nslot) * kPanelBytes;
  c.off_stg = c.off_p + p_bytes;
  c.off_bar = c.off_stg + static_cast<uint32_t>(c.nstg) * kPanelBytes;
  p->smem_bytes = static_cast<int>(c.off_bar + kBarBytes + 1024);
  if (p->smem_bytes > kSmemOptin) return B2B_ERR_UNSUPPORTED;
  // a weight whose width is a multiple of its 128-byte block (64 16-bit or
  // 32 tf32 columns) is read in 4-D boxes (tf32 weights as stored only)
  c.w_kmajor = p->w_kmajor ? 1 : 0;
  c.w_merged = 0;
  for (int s = 0; s < S; ++s) {
    const bool t32 = pt || (p->tf0 && s == 0);
    if (t32 ? (!p->w_kmajor && p->N[s] % 32 == 0) : p->N[s] % 64 == 0) c.w_merged |= 1 << s;
  }
  const ChainNEntry* e = find_chainn_kernel(p->in_kind, p->out_kind, p->nf, p->tf0 || pt);
  if (!e) return B2B_ERR_UNSUPPORTED;
  p->fn = e->fn;
  p->threads = kChainNThreads;
  // the number of co-resident clusters is known once the kernel's shared
  // memory size is set (pair_grid)
  p->grid = static_cast<int>(std::min<int64_t>(2 * tiles, p->sms & ~1));
  return B2B_OK;
}

// A two-GEMM tf32 chain runs on CTA pairs when both widths fit one 256-column
// pass and there are at least two 128-row tiles: each SM then loads half of
// every weight panel (measured: 2 x 65536 rows 84.0 -> 60.6 us, 20480 rows
// 27.3 -> 21.7 us), and with at most one tile per SM the second GEMM, which
// waits on its weight panels in the one-CTA kernel, runs at the tensor
// pipe's rate (16384 rows: 13.5 -> 13.1 us).
bool tf32_pairs(const b2b_plan_s* p) {
  return p->in_kind == kInTF32 && p->stages == 2 && p->N[0] <= 256 && p->N[1] <= 256 &&
         p->batch * ((p->M + 127) / 128) >= 2;
}

// Tiling of a tcgen05 chain of one or two GEMMs (chain_tc_kernel): padded
// widths, final-pass width, tensor-memory regions, shared-memory carve-up,
// and whether the weights stay resident.  Longer cascades, intermediates
// wider than 256 columns and mixed types go to setup_chainn.
b2b_status_t setup_chain_tc(b2b_plan_s* p) {
  const int S = p->stages;
  if (p->tf0 || (p->in_kind != kInTF32 && (S >= 3 || (S == 2 && p->N[0] > 256))) || tf32_pairs(p))
    return setup_chainn(p);
  p->sn = false;
  const int CK = 128 / p->esz;
  const int64_t wmin = 64;
  p->n1p = S >= 2 ? static_cast<int>(pad_width(p->N[0])) : 64;
  p->n2p = S >= 3 ? static_cast<int>(pad_width(p->N[1])) : 64;
  const int64_t nlast = p->N[S - 1];
  const int nl = static_cast<int>(std::max<int64_t>(wmin, pad64(nlast)));
  const int base_z = (S >= 2 ? p->n1p : 0) + (S >= 3 ? p->n2p : 0);

  int nf = 0, nz = -1, lookahead = 0;
  const int cands[3] = {256, 128, 64};
  // Two-stage chains: prefer a double-buffered GEMM1 accumulator (GEMM1 of
  // the next tile then runs while the current tile is rearranged).
  if (S == 2 && p->in_kind != kInTF32) {
    const int base_la = 2 * p->n1p;
    for (int k = 2; k >= 1 && nz < 0; --k)
      for (int c : cands)
        if (c >= wmin && c <= nl && base_la + k * c <= 512) { nf = c; nz = k; lookahead = 1; break; }
  }
  // One tile per CTA: nothing to overlap across tiles, so one wide final
  // accumulator (fewer, larger MMAs) beats two narrower alternating ones.
  const bool one_tile = p->batch * ((p->M + 127) / 128) <= p->sms;
  if (nz < 0 && one_tile)
    for (int c : cands)
      if (c >= wmin && c <= nl && base_z + c <= 512 && c >= std::min(nl, 256)) { nf = c; nz = 1; break; }
  if (nz < 0)
    for (int c : cands)
      if (c >= wmin && c <= nl && base_z + 2 * c <= 512) { nf = c; nz = 2; break; }
  if (nz < 0)
    for (int c : cands)
      if (c >= wmin && c <= nl && base_z + c <= 512) { nf = c; nz = 1; break; }
  if (nz < 0) return B2B_ERR_UNSUPPORTED;
  if (nf == 0) return B2B_ERR_UNSUPPORTED;
  p->nf = nf;

  ChainParams& c = p->prm;
  std::memset(&c, 0, sizeof(c));
  c.batch = static_cast<int>(p->batch);
  c.M = static_cast<int>(p->M);
  c.K = static_cast<int>(p->K);
  c.m_tiles = static_cast<int>((p->M + 127) / 128);
  const int64_t tiles = p->batch * c.m_tiles;
  if (tiles > (1ll << 30)) return B2B_ERR_UNSUPPORTED;
  c.total_tiles = static_cast<int>(tiles);
  c.npass = static_cast<int>((nlast + nf - 1) / nf);
  c.kpan0 = static_cast<int>((p->K + CK - 1) / CK);
  c.nz = nz;
  c.lookahead = lookahead;
  const int zbase = lookahead ? 2 * p->n1p : base_z;
  c.region_col[0] = 0;
  c.region_col[1] = (S >= 3 || lookahead) ? p->n1p : 0;
  c.region_col[2] = zbase;
  c.region_col[3] = zbase + nf;
  if (nz == 0) {  // the final passes reuse X and Y in turn
    c.region_col[2] = c.region_col[0];
    c.region_col[3] = c.region_col[1];
  }
  const uint32_t cols_used =
      nz > 0 ? static_cast<uint32_t>(zbase + nz * nf) : static_cast<uint32_t>(base_z);
  c.tmem_cols = pow2_cols(cols_used);
  if (c.tmem_cols > 512) return B2B_ERR_UNSUPPORTED;

  const bool p_smem = (S >= 2) && p->in_kind != kInTF32;
  uint32_t p_bytes =
      p_smem ? static_cast<uint32_t>(std::max(p->n1p, S >= 3 ? p->n2p : 0)) * 128u * p->esz : 0u;
  const int maxw = std::max({S >= 2 ? p->n1p : 0, S >= 3 ? p->n2p : 0, nf});
  // Streamed weights: A panels get a ring of their own when CTAs run more
  // than one tile (the next tile's A then loads during this tile's later
  // GEMMs); with one tile per CTA A shares each GEMM1 stage with its weight
  // panel (one wait per stage instead of two).
  const bool split_a = c.total_tiles > p->sms;

  // Layouts in order of preference: weights resident for the whole batch
  // with two operand images for the intermediate, resident with one image,
  // or weights streamed per tile (a ring of weight panels and a separate
  // ring of A panels).
  struct Layout { bool res, dbl; uint32_t stage, wres0, wres1; int nst, nsta, nstg; };
  auto fit = [&](bool res, bool dbl) -> Layout {
    Layout L{res, dbl, 0, 0, 0, 0, 0, 0};
    // resident: a ring stage holds a whole A tile (all K panels); streamed:
    // one weight panel (behind its A panel when A has no ring of its own)
    L.stage = res ? static_cast<uint32_t>(c.kpan0) * kPanelBytes
                  : 128u * static_cast<uint32_t>(maxw) + (split_a ? 0u : kPanelBytes);
    if (res) {
      L.wres0 = static_cast<uint32_t>(c.kpan0) * 128u * p->n1p;
      L.wres1 = static_cast<uint32_t>(p->n1p / CK) * 128u * nf;
    }
    const int64_t fixed = int64_t(L.wres0) + L.wres1 + int64_t(p_bytes) * (dbl ? 2 : 1) + kBarBytes;
    for (int nstg = 2; nstg >= 1; --nstg) {
      const int64_t room = kSmemBudget - fixed - int64_t(nstg) * kPanelBytes;
      L.nstg = nstg;
      if (res) {
        L.nst = room > 0 ? static_cast<int>(std::min<int64_t>(8, room / L.stage)) : 0;
        L.nsta = 0;
        if (L.nst >= 3 || (dbl && L.nst >= 2)) break;
      } else if (split_a) {
        // up to four weight panels in flight; the rest of the room (up to
        // eight panels) for A
        const int64_t wroom = room - 2 * int64_t(kPanelBytes);
        L.nst = wroom > 0 ? static_cast<int>(std::min<int64_t>(4, wroom / L.stage)) : 0;
        const int64_t aroom = room - int64_t(L.nst) * L.stage;
        L.nsta = aroom > 0 ? static_cast<int>(std::min<int64_t>(8, aroom / kPanelBytes)) : 0;
        if (L.nst >= 3 && L.nsta >= 4) break;
      } else {
        L.nst = room > 0 ? static_cast<int>(std::min<int64_t>(8, room / L.stage)) : 0;
        L.nsta = 0;
        if (L.nst >= 3) break;
      }
    }
    return L;
  };
  Layout L = fit(false, false);
  const bool res_ok = S == 2 && c.npass == 1 && c.kpan0 <= 4 &&
                      find_chain_kernel(p->in_kind, p->out_kind, S, p->n1p, p->n2p, nf, true);
  bool p_tmem16 = false;
  if (res_ok) {
    // 16-bit, resident weights, lookahead: keep the intermediate in tensor
    // memory (packed in place in its GEMM1 region, one region per tile
    // parity), which frees shared memory for a deeper ring.
    if (p_smem && lookahead) {
      p_bytes = 0;
      p_tmem16 = true;
      L = fit(true, true);
    } else {
      const Layout R = fit(true, false);
      if (R.nst >= 3) L = R;
    }
  }
  if (L.nst < 2 || (!L.res && split_a && L.nsta < 2)) return B2B_ERR_UNSUPPORTED;
  p->res = L.res;
  c.dbl_p = L.dbl ? 1 : 0;
  c.p_tmem = p_tmem16 ? 1 : 0;
  c.w_kmajor = p->w_kmajor ? 1 : 0;
  c.w_merged = 0;
  // 4-D boxes for widths that are a multiple of the 128-byte block (64
  // 16-bit or 32 tf32 columns); transposed tf32 weights are plain 3-D
  if (!p->w_kmajor)
    for (int s = 0; s < S; ++s)
      if (p->N[s] % (128 / p->esz) == 0) c.w_merged |= 1 << s;
  c.p_bytes = p_bytes;
  c.nst = L.nst;
  c.nsta = L.nsta;
  c.nstg = L.nstg;
  c.stage_bytes = L.stage;
  c.off_ring = 0;
  c.off_aring = static_cast<uint32_t>(L.nst) * L.stage;
  c.off_wres0 = c.off_aring + static_cast<uint32_t>(L.nsta) * kPanelBytes;
  c.off_wres1 = c.off_wres0 + L.wres0;
  c.off_p = c.off_wres1 + L.wres1;
  c.off_stg = c.off_p + p_bytes * (L.dbl ? 2u : 1u);
  c.off_bar = c.off_stg + static_cast<uint32_t>(L.nstg) * kPanelBytes;
  p->smem_bytes = static_cast<int>(c.off_bar + kBarBytes + 1024);
  if (p->smem_bytes > kSmemOptin) return B2B_ERR_UNSUPPORTED;

  const ChainKernelEntry* e =
      find_chain_kernel(p->in_kind, p->out_kind, S, p->n1p, p->n2p, nf, p->res);
  if (!e) return B2B_ERR_UNSUPPORTED;
  p->fn = e->fn;
  p->threads = kChainThreads;
  p->grid = static_cast<int>(std::min<int64_t>(c.total_tiles, p->sms));
  c.sched = nullptr;
  p->sched_host.clear();
  if (p->res) p->sched_host = res_schedule(p->batch, c.m_tiles, p->grid);
  return B2B_OK;
}

// Tile schedule for resident weights.  A CTA's weights change only where its
// tiles cross into another batch, and a change drains the pipeline: the new
// weights may replace the old ones only after the old batch's last GEMM2, and
// their load then queues behind the A tiles in flight -- about kSwitchTiles
// tiles' time on a GB300 (batched_f16: 3.3 us per change against 1.1 us per
// tile, measured per CTA).  The default split (one contiguous range of
// ceil(T / G) tiles per CTA) makes about a third of the CTAs change batch once.
// Instead every batch is cut into pieces of L tiles, one CTA each, and the
// shorter leftovers of consecutive batches are packed into shared CTAs while
// their tiles plus kSwitchTiles per change stay within L; the smallest L that
// fits in G CTAs is taken if it beats the default split's largest cost.
// Returns the table (kSchedStride ints per CTA) or an empty vector.
constexpr int kSwitchTiles = 3;

std::vector<int> res_schedule(int64_t batch, int64_t m_tiles, int G) {
  std::vector<int> none;
  const int64_t T = batch * m_tiles;
  if (batch < 2 || G < 1 || T <= G) return none;
  int64_t c_contig = 0;
  for (int64_t i = 0; i < G; ++i) {
    const int64_t b0 = i * T / G, b1 = (i + 1) * T / G;
    if (b1 <= b0) continue;
    const int64_t changes = (b1 - 1) / m_tiles - b0 / m_tiles;
    c_contig = std::max(c_contig, (b1 - b0) + kSwitchTiles * changes);
  }
  for (int64_t L = (T + G - 1) / G; L < c_contig; ++L) {
    // pieces of L tiles per batch, then leftovers packed in batch order
    struct Seg { int64_t first, count; };
    std::vector<std::vector<Seg>> ctas;
    std::vector<Seg> pack;
    int64_t pack_cost = 0;
    auto flush = [&]() {
      if (!pack.empty()) ctas.push_back(pack);
      pack.clear();
      pack_cost = 0;
    };
    for (int64_t b = 0; b < batch && static_cast<int64_t>(ctas.size()) <= G; ++b) {
      const int64_t full = m_tiles / L, rest = m_tiles - full * L;
      for (int64_t j = 0; j < full; ++j) ctas.push_back({Seg{b * m_tiles + j * L, L}});
      if (rest == 0) continue;
      const Seg s{b * m_tiles + full * L, rest};
      const int64_t cost = pack.empty() ? rest : pack_cost + kSwitchTiles + rest;
      if (!pack.empty() && (cost > L || static_cast<int>(pack.size()) == kSchedSegs)) flush();
      pack_cost = pack.empty() ? rest : pack_cost + kSwitchTiles + rest;
      pack.push_back(s);
    }
    flush();
    if (static_cast<int64_t>(ctas.size()) > G) continue;
    std::vector<int> table(static_cast<size_t>(G) * kSchedStride, 0);
    for (size_t i = 0; i < ctas.size(); ++i) {
      int* row = table.data() + i * kSchedStride;
      row[0] = static_cast<int>(ctas[i].size());
      for (size_t k = 0; k < ctas[i].size(); ++k) {
        row[1 + 2 * k] = static_cast<int>(ctas[i][k].first);
        row[2 + 2 * k] = static_cast<int>(ctas[i][k].count);
      }
    }
    return table;
  }
  return none;
}

// A paired chain runs one persistent cluster of two CTAs per tile slot: as
// many clusters as can be resident at once (clusters must fit within a GPC,
// so this can be fewer than half the SMs), at most one per 256-row tile.
b2b_status_t pair_grid(b2b_plan_s* p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p->grid));
  cfg.blockDim = dim3(static_cast<unsigned>(p->threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(p->smem_bytes);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, p->fn, &cfg) != cudaSuccess || clusters < 1) {
    cudaGetLastError();
    return B2B_ERR_UNSUPPORTED;
  }
  // Leftover tiles (when the tiles do not divide evenly among the clusters)
  // are shared by two clusters each, one half of the last GEMM's passes
  // apiece, if that leaves no cluster idle and there are passes to share.
  ChainNParams& c = p->pn;
  const int64_t total = c.total_tiles;
  const int64_t ncl = std::min<int64_t>(clusters, c.npass >= 2 ? 2 * total : total);
  p->grid = 2 * static_cast<int>(ncl);
  const int64_t left = total % ncl;
  c.split = (c.npass >= 2 && left > 0 && 2 * left <= ncl) ? static_cast<int>(left) : 0;
  return B2B_OK;
}

b2b_status_t setup_f64(b2b_plan_s* p) {
  const F64Tables tab = f64_tables();
  if (!tab.ok) return B2B_ERR_UNSUPPORTED;
  F64Params& f = p->f64;
  std::memset(&f, 0, sizeof(f));
  f.batch = static_cast<int>(p->batch);
  f.M = static_cast<int>(p->M);
  f.K = static_cast<int>(p->K);
  f.m8_tiles = static_cast<int>((p->M + 7) / 8);
  f.total = p->batch * f.m8_tiles;
  for (int j = 0; j < 2; ++j) {
    f.fsrc[j] = tab.fsrc[j];
    f.qsend[j] = tab.qsend[j];
    f.hslot[j] = tab.hslot[j];
  }
  const int n1 = static_cast<int>(p->N[0]);
  const int n2 = p->stages >= 2 ? static_cast<int>(p->N[1]) : 0;
  const void* fn = nullptr;
#define B2B_F64_CASE(A, B)                                                              \
  if (p->stages == 2 && n1 == A && n2 == B)                                             \
    fn = reinterpret_cast<const void*>(&chain_f64_kernel<A, B, 2>);
  B2B_F64_CASE(16, 16) B2B_F64_CASE(16, 32) B2B_F64_CASE(16, 64)
  B2B_F64_CASE(32, 16) B2B_F64_CASE(32, 32) B2B_F64_CASE(32, 64)
  B2B_F64_CASE(64, 16) B2B_F64_CASE(64, 32) B2B_F64_CASE(64, 64)
#undef B2B_F64_CASE
  if (p->stages == 1) {
    if (n1 == 16) fn = reinterpret_cast<const void*>(&chain_f64_kernel<16, 8, 1>);
    if (n1 == 32) fn = reinterpret_cast<const void*>(&chain_f64_kernel<32, 8, 1>);
    if (n1 == 64) fn = reinterpret_cast<const void*>(&chain_f64_kernel<64, 8, 1>);
  }
  if (!fn) return B2B_ERR_UNSUPPORTED;
  p->fn = fn;
  p->threads = 128;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 128, 0) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    per_sm = 4;
  }
  const int64_t need = (f.total + 3) / 4;
  p->grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(need, int64_t(p->sms) * per_sm)));
  p->smem_bytes = 0;
  return B2B_OK;
}

b2b_status_t validate_sizes(b2b_dtype_t dt, int stages, int64_t batch, int64_t M, int64_t K,
                            const int64_t* N) {
  if (batch < 0 || M < 0 || K < 1 || stages < 1 || stages > kMaxStages) return B2B_ERR_INVALID_ARG;
  for (int s = 0; s < stages; ++s)
    if (N[s] < 1) return B2B_ERR_INVALID_ARG;
  if (batch > (1 << 24) || M > (1ll << 30) || K > (1 << 20)) return B2B_ERR_UNSUPPORTED;
  switch (dt) {
    case B2B_F16_F32OUT:
    case B2B_F16:
    case B2B_BF16:
    case B2B_BF16_F32OUT:
      if (K % 8) return B2B_ERR_UNSUPPORTED;
      for (int s = 0; s < stages; ++s) {
        if (N[s] % 8) return B2B_ERR_UNSUPPORTED;
        if (s < stages - 1 && N[s] > 512) return B2B_ERR_UNSUPPORTED;
        if (N[s] > 4096) return B2B_ERR_UNSUPPORTED;
      }
      return B2B_OK;
    case B2B_TF32_F16:
    case B2B_TF32_BF16:
      if (stages < 2 || batch > 32767) return B2B_ERR_UNSUPPORTED;
      if (K % 4) return B2B_ERR_UNSUPPORTED;
      for (int s = 0; s < stages; ++s) {
        if (N[s] % 8) return B2B_ERR_UNSUPPORTED;
        if (s < stages - 1 && N[s] > 512) return B2B_ERR_UNSUPPORTED;
        if (N[s] > 4096) return B2B_ERR_UNSUPPORTED;
      }
      return B2B_OK;
    case B2B_TF32:
      if (stages > 2 || batch > 32767) return B2B_ERR_UNSUPPORTED;
      if (K % 4) return B2B_ERR_UNSUPPORTED;
      for (int s = 0; s < stages; ++s) {
        if (N[s] % 4) return B2B_ERR_UNSUPPORTED;
        if (s < stages - 1 && N[s] > 256) return B2B_ERR_UNSUPPORTED;
        if (N[s] > 4096) return B2B_ERR_UNSUPPORTED;
      }
      return B2B_OK;
    case B2B_F64:
      if (stages > 2) return B2B_ERR_UNSUPPORTED;
      if (K % 4) return B2B_ERR_UNSUPPORTED;
      for (int s = 0; s < stages; ++s)
        if (N[s] != 16 && N[s] != 32 && N[s] != 64) return B2B_ERR_UNSUPPORTED;
      return B2B_OK;
    default:
      return B2B_ERR_INVALID_ARG;
  }
}

void type_info(b2b_dtype_t dt, int* in_kind, int* out_kind, int* esz, int* osz) {
  switch (dt) {
    case B2B_F16_F32OUT: *in_kind = kInF16; *out_kind = kOutF32; *esz = 2; *osz = 4; break;
    case B2B_F16: *in_kind = kInF16; *out_kind = kOutF16; *esz = 2; *osz = 2; break;
    case B2B_BF16: *in_kind = kInBF16; *out_kind = kOutBF16; *esz = 2; *osz = 2; break;
    case B2B_BF16_F32OUT: *in_kind = kInBF16; *out_kind = kOutF32; *esz = 2; *osz = 4; break;
    case B2B_TF32: *in_kind = kInTF32; *out_kind = kOutF32; *esz = 4; *osz = 4; break;
    // mixed: the type of the intermediates and of the later weights (the
    // first GEMM's fp32 operands are described by the plan's tf0 flag)
    case B2B_TF32_F16: *in_kind = kInF16; *out_kind = kOutF32; *esz = 2; *osz = 4; break;
    case B2B_TF32_BF16: *in_kind = kInBF16; *out_kind = kOutF32; *esz = 2; *osz = 4; break;
    default: *in_kind = -1; *out_kind = -1; *esz = 8; *osz = 8; break;
  }
}

b2b_status_t create_common(b2b_plan_t* out, b2b_dtype_t dt, int stages, bool single,
                           int64_t batch, int64_t M, int64_t K, const int64_t* N) {
  if (!out) return B2B_ERR_INVALID_ARG;
  *out = nullptr;
  if (dt < B2B_F16_F32OUT || dt > B2B_TF32_BF16) return B2B_ERR_INVALID_ARG;
  b2b_status_t st = validate_sizes(dt, stages, batch, M, K, N);
  if (st != B2B_OK) return st;
  int dev = 0, sms = 0;
  st = check_device(&dev, &sms);
  if (st != B2B_OK) return st;

  b2b_plan_s* p = new (std::nothrow) b2b_plan_s();
  if (!p) return B2B_ERR_CUDA;
  p->dtype = dt;
  p->device = dev;
  p->sms = sms;
  p->stages = stages;
  p->batch = batch;
  p->M = M;
  p->K = K;
  for (int s = 0; s < kMaxStages; ++s) p->N[s] = s < stages ? N[s] : 0;
  p->budget_ns = kDefaultBudgetNs;
  type_info(dt, &p->in_kind, &p->out_kind, &p->esz, &p->osz);
  p->tf0 = dt == B2B_TF32_F16 || dt == B2B_TF32_BF16;
  if (batch == 0 || M == 0) {
    // An empty chain: valid, and every run is a no-op.
    p->kind = kPlanEmpty;
    p->grid = 0;
    p->threads = 0;
  } else if (dt == B2B_F64) {
    p->kind = single ? kPlanGemmF64 : kPlanChainF64;
    st = setup_f64(p);
  } else {
    p->kind = single ? kPlanGemmTC : kPlanChainTC;
    st = setup_chain_tc(p);
    // (the limit is a property of the kernel, shared by every plan that runs
    // it: always the largest any plan asks for, so that a plan created later
    // never lowers it below an earlier plan's size)
    if (st == B2B_OK &&
        cudaFuncSetAttribute(p->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOptin) !=
            cudaSuccess) {
      cudaGetLastError();
      st = B2B_ERR_CUDA;
    }
    if (st == B2B_OK && p->sn) st = pair_grid(p);
  }
  if (st == B2B_OK) {
    p->d_status = nullptr;
    if (cudaMalloc(&p->d_status, sizeof(int)) != cudaSuccess ||
        cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      st = B2B_ERR_CUDA;
    }
  }
  if (st == B2B_OK && !p->sched_host.empty()) {
    const size_t bytes = p->sched_host.size() * sizeof(int);
    if (cudaMalloc(&p->d_sched, bytes) != cudaSuccess ||
        cudaMemcpy(p->d_sched, p->sched_host.data(), bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      st = B2B_ERR_CUDA;
    } else {
      p->prm.sched = p->d_sched;
    }
  }
  if (st != B2B_OK) {
    if (p->d_status) cudaFree(p->d_status);
    if (p->d_wt) cudaFree(p->d_wt);
    if (p->d_sched) cudaFree(p->d_sched);
    delete p;
    return st;
  }
  *out = p;
  return B2B_OK;
}

b2b_status_t encode_3d(CUtensorMap* map, CUtensorMapDataType dt, int esz, const void* ptr,
                       int64_t inner, int64_t rows, int64_t batch, uint32_t box_inner,
                       uint32_t box_rows, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return B2B_ERR_CUDA;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner * esz),
                                 static_cast<cuuint64_t>(inner * rows * esz)};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? B2B_OK : B2B_ERR_CUDA;
}

// Weight W[b][K][N] (N a multiple of the block width `blk`, whose row is
// 128 bytes: 64 16-bit or 32 fp32 columns) seen as a 4-D tensor (blk
// columns, K rows, N/blk column blocks, batch): one box of (blk, k_rows,
// blocks, 1) covers k_rows rows of `blocks` adjacent column blocks, and
// lands in shared memory as `blocks` consecutive 128-byte-wide swizzled
// blocks of k_rows rows each.
b2b_status_t encode_w4d(CUtensorMap* map, CUtensorMapDataType dt, int esz, const void* ptr,
                        int64_t n, int64_t k, int64_t batch, uint32_t k_rows, uint32_t blocks,
                        CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return B2B_ERR_CUDA;
  const int64_t blk = 128 / esz;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(blk), static_cast<cuuint64_t>(k),
                              static_cast<cuuint64_t>(n / blk), static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(n * esz), static_cast<cuuint64_t>(blk * esz),
                                 static_cast<cuuint64_t>(n * k * esz)};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(blk), k_rows, blocks, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, dt, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? B2B_OK : B2B_ERR_CUDA;
}

// A tf32 weight W[b][K][N] as stored, for an MN-major B operand: blocks of
// 32 columns (128 bytes) by k_rows rows, swizzled in 32-byte atoms (the
// form the tf32 MMA reads MN-major); one 4-D box of `blocks` blocks when
// `merged` (N a multiple of 32), else 3-D boxes of one block each.
b2b_status_t encode_w_mn32(CUtensorMap* map, const void* ptr, int64_t n, int64_t k, int64_t batch,
                           uint32_t k_rows, uint32_t blocks, bool merged) {
  if (merged)
    return encode_w4d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, n, k, batch, k_rows, blocks,
                      CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B);
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, n, k, batch, 32, k_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B);
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream is finishing; it waits (griddepcontrol)
// before its first global-memory access.
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, void** args, size_t smem,
                       cudaStream_t stream, int cluster = 1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

b2b_status_t encode_chain_maps(b2b_plan_s* p, const void* const* W, const void* A, void* D,
                               ChainNMaps* maps) {
  const int S = p->stages;
  const CUtensorMapDataType in_dt = p->in_kind == kInF16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                    : p->in_kind == kInBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const CUtensorMapDataType out_dt = p->out_kind == kOutF16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                     : p->out_kind == kOutBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const uint32_t CK = 128 / p->esz;
  std::memset(maps, 0, sizeof(*maps));
  // A in its own storage type: fp32 in panels of 32 elements for a mixed-type
  // cascade, else the chain's input type
  b2b_status_t st = p->tf0 ? encode_3d(&maps->a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, A, p->K, p->M, p->batch, 32, 128)
                           : encode_3d(&maps->a, in_dt, p->esz, A, p->K, p->M, p->batch, CK, 128);
  int64_t kin = p->K;
  if (p->in_kind == kInTF32 && p->w_kmajor) {
    // the weights as transposed into the workspace ([N][K] per batch)
    const uint32_t* dst = static_cast<const uint32_t*>(p->d_wt);
    for (int s = 0; s < S && st == B2B_OK; ++s) {
      // boxes of a pass's rows (CTA pairs: of this CTA's half of them)
      const uint32_t rows = p->sn            ? static_cast<uint32_t>(p->pn.pw[s] / 2)
                            : s < S - 1      ? static_cast<uint32_t>(s == 0 ? p->n1p : p->n2p)
                                             : static_cast<uint32_t>(p->nf);
      st = encode_3d(&maps->w[s], in_dt, p->esz, dst, kin, p->N[s], p->batch, CK, rows);
      dst += p->batch * kin * p->N[s];
      kin = p->N[s];
    }
  } else if (p->sn) {
    // CTA pairs: each CTA loads half of a pass's column blocks
    for (int s = 0; s < S && st == B2B_OK; ++s) {
      const bool merged = (p->pn.w_merged >> s) & 1;
      if (p->in_kind == kInTF32 || (p->tf0 && s == 0)) {
        // a tf32 weight as stored: 32 K rows of this CTA's half of a pass
        const uint32_t wcols = static_cast<uint32_t>(p->pn.pw[s] / 2);
        st = encode_w_mn32(&maps->w[s], W[s], p->N[s], kin, p->batch, 32, wcols / 32, merged);
      } else if (merged) {
        // a box of this CTA's column blocks of a pass, over one K panel, or
        // two for 128-column passes after the first GEMM
        const uint32_t kps = (s > 0 && p->pn.pw[s] == 128) ? 2u : 1u;
        st = encode_w4d(&maps->w[s], in_dt, p->esz, W[s], p->N[s], kin, p->batch, CK * kps,
                        static_cast<uint32_t>(p->pn.pw[s] / 128));
      } else {
        st = encode_3d(&maps->w[s], in_dt, p->esz, W[s], p->N[s], kin, p->batch, CK, CK);
      }
      kin = p->N[s];
    }
  } else {
    for (int s = 0; s < S && st == B2B_OK; ++s) {
      const bool merged = (p->prm.w_merged >> s) & 1;
      // a whole K panel of every 128-byte column block of the stage's width
      // in one box when merged, laid out in shared memory block after block
      const int64_t width = s < S - 1 ? (s == 0 ? p->n1p : p->n2p) : p->nf;
      if (p->in_kind == kInTF32) {
        st = encode_w_mn32(&maps->w[s], W[s], p->N[s], kin, p->batch, CK, static_cast<uint32_t>(width / 32),
                           merged);
      } else if (merged) {
        st = encode_w4d(&maps->w[s], in_dt, p->esz, W[s], p->N[s], kin, p->batch, CK,
                        static_cast<uint32_t>(width / 64));
      } else {
        st = encode_3d(&maps->w[s], in_dt, p->esz, W[s], p->N[s], kin, p->batch, CK, CK);
      }
      kin = p->N[s];
    }
  }
  for (int s = S; s < kMaxStages; ++s) maps->w[s] = maps->w[0];
  // (paired chains: every epilogue warp stores its own 32 rows)
  if (st == B2B_OK)
    st = encode_3d(&maps->out, out_dt, p->osz, D, p->N[S - 1], p->M, p->batch, 128 / p->osz, p->sn ? 32 : 128);
  return st;
}

b2b_status_t run_chain_tc(b2b_plan_s* p, const void* const* W, const void* A, void* D,
                          cudaStream_t stream) {
  const int S = p->stages;
  if (p->w_kmajor) {
    // K-major tf32 weights (the allocation-free call): transpose every
    // weight to [N][K] into the workspace first.
    TransposeJob job;
    std::memset(&job, 0, sizeof(job));
    job.batch = static_cast<int>(p->batch);
    job.count = S;
    uint32_t* dst = static_cast<uint32_t*>(p->d_wt);
    int64_t kin = p->K;
    int max_r = 0, max_c = 0;
    for (int s = 0; s < job.count; ++s) {
      job.in[s] = static_cast<const uint32_t*>(W[s]);
      job.out[s] = dst;
      job.rows[s] = static_cast<int>(kin);
      job.cols[s] = static_cast<int>(p->N[s]);
      max_r = std::max(max_r, job.rows[s]);
      max_c = std::max(max_c, job.cols[s]);
      dst += p->batch * kin * p->N[s];
      kin = p->N[s];
    }
    const dim3 grid((max_c + 31) / 32, (max_r + 31) / 32, static_cast<unsigned>(job.count * p->batch));
    void* targs[1] = {&job};
    if (launch_pdl(reinterpret_cast<const void*>(&transpose32_kernel), grid, dim3(256), targs, 0,
                   stream) != cudaSuccess) {
      cudaGetLastError();
      return B2B_ERR_CUDA;
    }
  }
  ChainNMaps maps;
  {
    const void* key[kMaxStages + 2];
    key[0] = A;
    key[1] = D;
    for (int s = 0; s < kMaxStages; ++s) key[2 + s] = s < S ? W[s] : nullptr;
    std::lock_guard<std::mutex> lock(p->mu);
    ++p->clock;
    int hit = -1, victim = 0;
    for (int i = 0; i < p->cache_n; ++i) {
      if (std::memcmp(p->cache[i].key, key, sizeof(key)) == 0) hit = i;
      if (p->cache[i].stamp < p->cache[victim].stamp) victim = i;
    }
    if (hit < 0) {
      ChainNMaps fresh;
      const b2b_status_t st = encode_chain_maps(p, W, A, D, &fresh);
      if (st != B2B_OK) return st;
      hit = p->cache_n < 8 ? p->cache_n++ : victim;
      std::memcpy(p->cache[hit].key, key, sizeof(key));
      std::memcpy(&p->cache[hit].maps, &fresh, sizeof(fresh));
    }
    p->cache[hit].stamp = p->clock;
    std::memcpy(&maps, &p->cache[hit].maps, sizeof(maps));
  }

  cudaError_t e;
  if (p->sn) {
    ChainNParams prm = p->pn;
    prm.status = p->d_status;
    prm.budget_ns = p->budget_ns;
    prm.debug = p->debug;
    void* args[2] = {&maps, &prm};
    e = launch_pdl(p->fn, dim3(p->grid), dim3(p->threads), args, static_cast<size_t>(p->smem_bytes),
                   stream, 2);
  } else {
    ChainParams prm = p->prm;
    prm.status = p->d_status;
    prm.budget_ns = p->budget_ns;
    prm.debug = p->debug;
    void* args[6] = {&maps.a, &maps.w[0], &maps.w[1], &maps.w[2], &maps.out, &prm};
    e = launch_pdl(p->fn, dim3(p->grid), dim3(p->threads), args, static_cast<size_t>(p->smem_bytes),
                   stream);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  return B2B_OK;
}

b2b_status_t run_f64(b2b_plan_s* p, const void* A, const void* B, const void* C, void* D,
                     cudaStream_t stream) {
  F64Params prm = p->f64;
  const double* a = static_cast<const double*>(A);
  const double* b = static_cast<const double*>(B);
  const double* c = static_cast<const double*>(C);
  double* d = static_cast<double*>(D);
  void* args[5] = {&a, &b, &c, &d, &prm};
  const cudaError_t e = launch_pdl(p->fn, dim3(p->grid), dim3(p->threads), args, 0, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  return B2B_OK;
}

// Argument checks shared by b2b_run and b2b_chain_run, then the launch.
b2b_status_t run_checked(b2b_plan_s* p, const void* A, const void* const* W, void* D,
                         b2b_stream_t stream) {
  if (p->kind == kPlanEmpty) return B2B_OK;
  const int S = p->stages;
  if (!A || !D) return B2B_ERR_INVALID_ARG;
  for (int s = 0; s < S; ++s)
    if (!W[s]) return B2B_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(A) & 15u) return B2B_ERR_ALIGNMENT;
  for (int s = 0; s < S; ++s)
    if (reinterpret_cast<uintptr_t>(W[s]) & 15u) return B2B_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(D) & 15u) return B2B_ERR_ALIGNMENT;
  // element sizes: A and W[0] are fp32 in a mixed-type cascade
  const size_t e = static_cast<size_t>(p->esz), e0 = p->tf0 ? 4u : e;
  const size_t dbytes = static_cast<size_t>(p->batch * p->M * p->N[S - 1]) * p->osz;
  if (overlaps(D, dbytes, A, static_cast<size_t>(p->batch * p->M * p->K) * e0)) return B2B_ERR_ALIAS;
  int64_t kin = p->K;
  for (int s = 0; s < S; ++s) {
    if (overlaps(D, dbytes, W[s], static_cast<size_t>(p->batch * kin * p->N[s]) * (s == 0 ? e0 : e)))
      return B2B_ERR_ALIAS;
    kin = p->N[s];
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  if (dev != p->device) return B2B_ERR_DEVICE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (p->kind == kPlanChainF64 || p->kind == kPlanGemmF64)
    return run_f64(p, A, W[0], S >= 2 ? W[1] : nullptr, D, st);
  return run_chain_tc(p, W, A, D, st);
}

}  // namespace

extern "C" {

b2b_status_t b2b_chain_plan_create(b2b_plan_t* out, b2b_dtype_t dtype, int64_t batch, int64_t M,
                                   int64_t K, int n_stages, const int64_t* N) {
  if (!out) return B2B_ERR_INVALID_ARG;
  *out = nullptr;
  if (!N || n_stages < 1 || n_stages > kMaxStages) return B2B_ERR_INVALID_ARG;
  return create_common(out, dtype, n_stages, n_stages == 1, batch, M, K, N);
}

b2b_status_t b2b_plan_create(b2b_plan_t* out, b2b_dtype_t dtype, int64_t batch, int64_t M,
                             int64_t K, int64_t N1, int64_t N2, int64_t N3) {
  if (N3 < 0) return B2B_ERR_INVALID_ARG;
  const int64_t N[3] = {N1, N2, N3};
  return create_common(out, dtype, N3 > 0 ? 3 : 2, false, batch, M, K, N);
}

b2b_status_t b2b_gemm_plan_create(b2b_plan_t* out, b2b_dtype_t dtype, int64_t batch, int64_t M,
                                  int64_t K, int64_t N) {
  const int64_t Ns[3] = {N, 0, 0};
  return create_common(out, dtype, 1, true, batch, M, K, Ns);
}

b2b_status_t b2b_run(b2b_plan_t p, const void* A, const void* B, const void* C, const void* F,
                     void* D, b2b_stream_t stream) {
  if (!p) return B2B_ERR_INVALID_ARG;
  if (p->kind == kPlanEmpty) return B2B_OK;
  const int S = p->stages;
  if (S > 3) return B2B_ERR_INVALID_ARG;
  if ((S >= 2) != (C != nullptr)) return B2B_ERR_INVALID_ARG;
  if ((S >= 3) != (F != nullptr)) return B2B_ERR_INVALID_ARG;
  const void* W[3] = {B, C, F};
  return run_checked(p, A, W, D, stream);
}

b2b_status_t b2b_chain_run(b2b_plan_t p, const void* A, const void* const* W, void* D,
                           b2b_stream_t stream) {
  if (!p || !W) return B2B_ERR_INVALID_ARG;
  for (int s = 0; s < p->stages; ++s)
    if (!W[s]) return B2B_ERR_INVALID_ARG;
  return run_checked(p, A, W, D, stream);
}

b2b_status_t b2b_plan_destroy(b2b_plan_t p) {
  if (!p) return B2B_OK;
  if (p->d_status) cudaFree(p->d_status);
  if (p->d_wt) cudaFree(p->d_wt);
  if (p->d_sched) cudaFree(p->d_sched);
  delete p;
  return B2B_OK;
}

b2b_status_t b2b_plan_device_status(b2b_plan_t p, b2b_stream_t stream) {
  if (!p) return B2B_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  int v = 0;
  if (cudaMemcpy(&v, p->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  return v == 0 ? B2B_OK : static_cast<b2b_status_t>(v);
}

b2b_status_t b2b_plan_set_wait_budget(b2b_plan_t p, uint64_t budget_ns) {
  if (!p) return B2B_ERR_INVALID_ARG;
  // After an abort the same budget bounds the waits for copies and MMAs
  // already in flight before tensor memory is freed: it must stay long
  // against any one of them (microseconds), hence the floor.
  p->budget_ns = budget_ns ? std::max<uint64_t>(budget_ns, kMinBudgetNs) : kDefaultBudgetNs;
  return B2B_OK;
}

b2b_status_t b2b_plan_set_debug(b2b_plan_t p, uint32_t flags) {
  if (!p) return B2B_ERR_INVALID_ARG;
  if (flags & ~B2B_DEBUG_DROP_FIRST_LOAD) return B2B_ERR_INVALID_ARG;
  p->debug = flags;
  return B2B_OK;
}

b2b_status_t b2b_plan_info(b2b_plan_t p, int* launches, int* grid, int* threads, int* smem,
                           int* tmem_cols, int* ring_stages, int* passes) {
  if (!p) return B2B_ERR_INVALID_ARG;
  const bool tc = p->kind == kPlanChainTC || p->kind == kPlanGemmTC;
  if (launches) *launches = p->kind == kPlanEmpty ? 0 : (p->w_kmajor ? 2 : 1);
  if (grid) *grid = p->grid;
  if (threads) *threads = p->threads;
  if (smem) *smem = p->smem_bytes;
  if (tmem_cols) *tmem_cols = !tc ? 0 : (p->sn ? 512 : static_cast<int>(p->prm.tmem_cols));
  if (ring_stages) *ring_stages = !tc ? 0 : (p->sn ? p->pn.nslot : p->prm.nst);
  if (passes) *passes = !tc ? 1 : (p->sn ? p->pn.npass : p->prm.npass);
  return B2B_OK;
}

const char* b2b_status_string(b2b_status_t s) {
  switch (s) {
    case B2B_OK: return "ok";
    case B2B_ERR_INVALID_ARG: return "invalid argument";
    case B2B_ERR_UNSUPPORTED: return "unsupported size or type";
    case B2B_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case B2B_ERR_ALIAS: return "output overlaps an input";
    case B2B_ERR_DEVICE: return "current device is not an sm_103 GPU";
    case B2B_ERR_CUDA: return "CUDA call failed";
    case B2B_ERR_TIMEOUT: return "a bounded wait inside a kernel timed out";
    default: return "unknown status";
  }
}

b2b_status_t b2b_probe_operand_image(b2b_dtype_t dtype, int width, const void* acc, void* image,
                                     b2b_stream_t stream) {
  if (!acc || !image) return B2B_ERR_INVALID_ARG;
  if (width != 64 && width != 128 && width != 256) return B2B_ERR_INVALID_ARG;
  int in_kind, out_kind, esz, osz;
  type_info(dtype, &in_kind, &out_kind, &esz, &osz);
  if (in_kind < 0) return B2B_ERR_UNSUPPORTED;
  b2b_status_t st = check_device(nullptr, nullptr);
  if (st != B2B_OK) return st;
  const void* fn = in_kind == kInF16    ? reinterpret_cast<const void*>(&probe_operand_kernel<kInF16>)
                   : in_kind == kInBF16 ? reinterpret_cast<const void*>(&probe_operand_kernel<kInBF16>)
                                        : reinterpret_cast<const void*>(&probe_operand_kernel<kInTF32>);
  const int smem = in_kind == kInTF32 ? 1024 : width * 256 + 1024;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  const uint32_t* a = static_cast<const uint32_t*>(acc);
  uint32_t* o = static_cast<uint32_t*>(image);
  uint32_t cols = pow2_cols(static_cast<uint32_t>(width));
  void* args[4] = {&a, &o, &width, &cols};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaLaunchKernel(fn, dim3(1), dim3(128), args, static_cast<size_t>(smem), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  return B2B_OK;
}

b2b_status_t b2b_probe_operand_layout(b2b_dtype_t dtype, int form, int width, int region, const void* acc,
                                      void* out, b2b_stream_t stream) {
  if (!acc || !out) return B2B_ERR_INVALID_ARG;
  int in_kind, out_kind, esz, osz;
  type_info(dtype, &in_kind, &out_kind, &esz, &osz);
  if (in_kind != kInF16 && in_kind != kInBF16) return B2B_ERR_UNSUPPORTED;
  if (form == B2B_PROBE_TMEM16) {
    if ((width != 64 && width != 128 && width != 256) || region != 0) return B2B_ERR_INVALID_ARG;
  } else if (form == B2B_PROBE_PAIR_CONVERTERS) {
    if (width < 128 || width > 512 || width % 128 || (region != 0 && region != 1)) return B2B_ERR_INVALID_ARG;
  } else {
    return B2B_ERR_INVALID_ARG;
  }
  b2b_status_t st = check_device(nullptr, nullptr);
  if (st != B2B_OK) return st;
  const bool f16 = in_kind == kInF16;
  const void* fn = form == B2B_PROBE_TMEM16
                       ? (f16 ? reinterpret_cast<const void*>(&probe_layout_kernel<kInF16, 1>)
                              : reinterpret_cast<const void*>(&probe_layout_kernel<kInBF16, 1>))
                       : (f16 ? reinterpret_cast<const void*>(&probe_layout_kernel<kInF16, 2>)
                              : reinterpret_cast<const void*>(&probe_layout_kernel<kInBF16, 2>));
  const int smem = form == B2B_PROBE_TMEM16 ? 1024 : width * 256 + 1024;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  const uint32_t* a = static_cast<const uint32_t*>(acc);
  uint32_t* o = static_cast<uint32_t*>(out);
  uint32_t r0 = static_cast<uint32_t>(region);
  uint32_t cols = form == B2B_PROBE_TMEM16 ? pow2_cols(static_cast<uint32_t>(width)) : 512u;
  void* args[5] = {&a, &o, &width, &r0, &cols};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaLaunchKernel(fn, dim3(1), dim3(256), args, static_cast<size_t>(smem), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  return B2B_OK;
}

b2b_status_t b2b_schedule_table(int table, const int64_t* args, int nargs, int64_t* out, int nout) {
  if (!args || !out || nout < 1) return B2B_ERR_INVALID_ARG;
  switch (table) {
    case B2B_TABLE_REGION_USE: {
      // args: S, npass, nz, lookahead, tiles; out: (region, use) of every
      // phase of every tile, tile-major
      if (nargs != 5) return B2B_ERR_INVALID_ARG;
      const int S = static_cast<int>(args[0]), tiles = static_cast<int>(args[4]);
      ChainParams c;
      std::memset(&c, 0, sizeof(c));
      c.npass = static_cast<int>(args[1]);
      c.nz = static_cast<int>(args[2]);
      c.lookahead = static_cast<int>(args[3]);
      if (S < 1 || S > 3 || c.npass < 1 || tiles < 0) return B2B_ERR_INVALID_ARG;
      const int nph = S - 1 + c.npass;
      if (static_cast<int64_t>(tiles) * nph * 2 > nout) return B2B_ERR_INVALID_ARG;
      for (int it = 0; it < tiles; ++it)
        for (int ph = 0; ph < nph; ++ph) {
          int r;
          uint32_t u;
          region_use(c, S, it, ph, r, u);
          out[2 * (it * nph + ph)] = r;
          out[2 * (it * nph + ph) + 1] = u;
        }
      return B2B_OK;
    }
    case B2B_TABLE_PAIR_UNITS: {
      // args: total_tiles, m_tiles, npass, split, ncl, cid; out[0] = the
      // cluster's unit count, then (batch, tile, p0, p1) per unit
      if (nargs != 6) return B2B_ERR_INVALID_ARG;
      ChainNParams c;
      std::memset(&c, 0, sizeof(c));
      c.total_tiles = static_cast<int>(args[0]);
      c.m_tiles = static_cast<int>(args[1]);
      c.npass = static_cast<int>(args[2]);
      c.split = static_cast<int>(args[3]);
      const int ncl = static_cast<int>(args[4]), cid = static_cast<int>(args[5]);
      if (c.m_tiles < 1 || ncl < 1 || cid < 0 || cid >= ncl) return B2B_ERR_INVALID_ARG;
      const int n = chainn_units(c, cid, ncl);
      if (1 + 4 * static_cast<int64_t>(n) > nout) return B2B_ERR_INVALID_ARG;
      out[0] = n;
      for (int i = 0; i < n; ++i) {
        const ChainNUnit u = chainn_unit(c, cid, ncl, i);
        out[1 + 4 * i] = u.b;
        out[2 + 4 * i] = u.mt;
        out[3 + 4 * i] = u.p0;
        out[4 + 4 * i] = u.p1;
      }
      return B2B_OK;
    }
    case B2B_TABLE_PAIR_TMEM_INTERMEDIATES: {
      // args: tf32 chain (0 / 1), last-GEMM passes, padded widths of the
      // intermediates; out[0] = the mask of those kept in tensor memory
      if (nargs < 3 || nargs - 2 > kMaxStages - 1) return B2B_ERR_INVALID_ARG;
      int wpad[kMaxStages];
      for (int s = 0; s < nargs - 2; ++s) wpad[s] = static_cast<int>(args[2 + s]);
      out[0] = chainn_tmem_mask(args[0] != 0, nargs - 2, wpad, static_cast<int>(args[1]));
      return B2B_OK;
    }
    case B2B_TABLE_PAIR_REGIONS: {
      // args: accumulator widths in the order they are taken; out: the
      // region each starts in (RegionCursor), then for each the tensor-memory
      // column of its columns 0, 128, 256, 384 (tmem_col)
      if (nargs < 1 || static_cast<int64_t>(nargs) * 5 > nout) return B2B_ERR_INVALID_ARG;
      RegionCursor rc;
      for (int i = 0; i < nargs; ++i) {
        const uint32_t r0 = rc.take(static_cast<int>(args[i]));
        out[5 * i] = r0;
        for (int q = 0; q < 4; ++q) out[5 * i + 1 + q] = tmem_col(r0, 128 * q);
      }
      return B2B_OK;
    }
    default:
      return B2B_ERR_INVALID_ARG;
  }
}

b2b_status_t b2b_probe_f64_rearrange(int tiles, const double* cfrag, double* afrag,
                                     b2b_stream_t stream) {
  if (!cfrag || !afrag || tiles < 1 || tiles > 8) return B2B_ERR_INVALID_ARG;
  b2b_status_t st = check_device(nullptr, nullptr);
  if (st != B2B_OK) return st;
  const F64Tables tab = f64_tables();
  if (!tab.ok) return B2B_ERR_UNSUPPORTED;
  F64Params prm;
  std::memset(&prm, 0, sizeof(prm));
  for (int j = 0; j < 2; ++j) {
    prm.fsrc[j] = tab.fsrc[j];
    prm.qsend[j] = tab.qsend[j];
    prm.hslot[j] = tab.hslot[j];
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  probe_f64_rearrange_kernel<<<1, 32, 0, s>>>(cfrag, afrag, tiles, prm);
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return B2B_ERR_CUDA;
  }
  return B2B_OK;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// tf32 chain without any allocation.
//
// Some callers cannot allocate device memory at all: code running where a
// cudaMalloc would stall or fail (inside a memory-pool-managed framework that
// forbids untracked allocations, or after the device memory has been handed
// out up front), or callers that must not create the plan objects that own
// device memory.  This entry point needs no plan: it runs the tf32 chain in
// the form that reads its weights transposed to [N][K] (a plan reads them as
// stored), and the scratch space of that form, the transposed weights, is a
// fixed array in device memory that belongs to the library itself.
//
// The array is `kNoAllocScratchWords` 32-bit words (4 MiB) on every GPU that
// loads the library, held until the process exits.  Its device address is
// looked up once per device (and again only if that device's context has
// been replaced, e.g. after a device reset), on the first call made while
// that device is current; make that first call before any stream capture.
// The same first call sets the kernel's shared-memory limit on that device.
// Every call shares the one array and leaves the last call's transposed
// weights in it; calls whose kernels overlap on the GPU (different streams,
// no ordering) race on it.  Nothing in it needs to start at zero: each call
// writes the part it reads before reading it.  A kernel that gives up a
// bounded wait still returns, but this entry point has no status word to
// report it.
namespace {

constexpr size_t kNoAllocScratchWords = size_t(1) << 20;
__device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;

// Per device: the context the entries below belong to, the scratch address
// in it, and the kernels whose shared-memory limit is already raised there.
struct NoAllocDevice {
  void* ctx;
  void* scratch;
  std::vector<const void*> configured;
};
NoAllocDevice g_noalloc_dev[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

// Set-up of the current device `dev` for the allocation-free call: the
// scratch array's device address (looked up with cudaGetSymbolAddress, not
// the host-side name of the array, which is no device address), and the
// dynamic shared-memory limit of kernel `fn`.  Both are cached per device
// and context, so later calls make no runtime call for them.
b2b_status_t noalloc_setup(int dev, const void* fn, void** scratch) {
  if (dev < 0 || dev >= kMaxDevices) return B2B_ERR_DEVICE;
  const CtxGetCurrentFn get = ctx_get_current_fn();
  if (!get) return B2B_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return B2B_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!ctx || d.ctx != static_cast<void*>(ctx) || !d.scratch) {
    // (the runtime makes the device's primary context current here if no
    // context was current yet)
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return B2B_ERR_CUDA;
    }
    if (!ctx && (get(&ctx) != CUDA_SUCCESS || !ctx)) return B2B_ERR_CUDA;
    d.ctx = ctx;
    d.scratch = ptr;
    d.configured.clear();
  }
  if (std::find(d.configured.begin(), d.configured.end(), fn) == d.configured.end()) {
    // the largest dynamic shared memory any plan of this kernel asks for
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOptin) != cudaSuccess) {
      cudaGetLastError();
      return B2B_ERR_CUDA;
    }
    d.configured.push_back(fn);
  }
  *scratch = d.scratch;
  return B2B_OK;
}

}  // namespace

extern "C" b2b_status_t b2b_run_tf32_noalloc(int64_t batch, int64_t M, int64_t K, int64_t N1,
                                             int64_t N2, const void* A, const void* B,
                                             const void* C, void* D, b2b_stream_t stream) {
  const int64_t N[2] = {N1, N2};
  b2b_status_t st = validate_sizes(B2B_TF32, 2, batch, M, K, N);
  if (st != B2B_OK) return st;
  if (batch == 0 || M == 0) return B2B_OK;
  const int64_t words = batch * (K * N1 + N1 * N2);
  if (words > static_cast<int64_t>(kNoAllocScratchWords)) return B2B_ERR_UNSUPPORTED;
  if (!A || !B || !C || !D) return B2B_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  st = check_device(&dev, &sms);
  if (st != B2B_OK) return st;
  // A plan on the stack: tiling only, no device memory of its own.
  b2b_plan_s pl;
  pl.kind = kPlanChainTC;
  pl.dtype = B2B_TF32;
  pl.device = dev;
  pl.sms = sms;
  pl.stages = 2;
  pl.batch = batch;
  pl.M = M;
  pl.K = K;
  for (int s = 0; s < kMaxStages; ++s) pl.N[s] = 0;
  pl.N[0] = N1;
  pl.N[1] = N2;
  pl.budget_ns = kDefaultBudgetNs;
  pl.debug = 0;
  pl.tf0 = false;
  pl.w_kmajor = true;  // weights transposed into the library's scratch array
  pl.d_status = nullptr;
  pl.d_wt = nullptr;
  pl.d_sched = nullptr;
  pl.wt_bytes = kNoAllocScratchWords * sizeof(uint32_t);
  pl.cache_n = 0;
  pl.clock = 0;
  type_info(B2B_TF32, &pl.in_kind, &pl.out_kind, &pl.esz, &pl.osz);
  st = setup_chain_tc(&pl);
  if (st != B2B_OK) return st;
  void* scratch = nullptr;
  st = noalloc_setup(dev, pl.fn, &scratch);
  if (st != B2B_OK) return st;
  pl.d_wt = scratch;
  if (pl.sn) {
    st = pair_grid(&pl);
    if (st != B2B_OK) return st;
  }
  const void* ins[3] = {A, B, C};
  for (const void* q : ins)
    if (reinterpret_cast<uintptr_t>(q) & 15u) return B2B_ERR_ALIGNMENT;
  if (reinterpret_cast<uintptr_t>(D) & 15u) return B2B_ERR_ALIGNMENT;
  const size_t in_bytes[3] = {static_cast<size_t>(batch * M * K) * 4, static_cast<size_t>(batch * K * N1) * 4,
                              static_cast<size_t>(batch * N1 * N2) * 4};
  const size_t dbytes = static_cast<size_t>(batch * M * N2) * 4;
  for (int i = 0; i < 3; ++i)
    if (overlaps(D, dbytes, ins[i], in_bytes[i])) return B2B_ERR_ALIAS;
  const void* W[3] = {B, C, nullptr};
  return run_chain_tc(&pl, W, A, D, reinterpret_cast<cudaStream_t>(stream));
}
