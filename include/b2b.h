/*
 * b2b.h -- fused cascaded (back-to-back) GEMM for GB300 (sm_103a).
 *
 *   D = (A.B).C              (two cascaded GEMMs)
 *   E = ((A.B).C).F          (three cascaded GEMMs)
 *   E = (..((A.W0).W1)..).W[S-1]   (S cascaded GEMMs, S <= B2B_MAX_STAGES)
 *
 * The method is the one of patent "数据处理方法、装置、设备及介质"
 * (Alibaba, 2023): two (or three) cascaded operators are fused so that the
 * result of operator 1 is never written to memory.  Operator 1's result,
 * held in the layout of the accumulator ("first data processing rule"), is
 * rearranged on chip into the operand layout operator 2 reads ("second data
 * processing rule") and handed straight to operator 2 (Detailed description
 * para. 35-37, steps 101-103; para. 54-60; more than two operators, each
 * one's output the next one's input: para. 41).
 * The apparatus splits this into an operator-determination module, a
 * relation-determination module and a rearrangement module (para. 140-143,
 * Fig. 5); here b2b_plan_create plays the first two (the caller names the
 * chain; the relation is fixed from the data types at plan time) and b2b_run
 * the third.
 *
 * Conventions for every entry point
 *   - Matrices are dense, row-major, batched: A[batch][M][K],
 *     B[batch][K][N1], C[batch][N1][N2], F[batch][N2][N3], and the output
 *     D[batch][M][N2] (two stages) or E[batch][M][N3] (three stages).  Each
 *     batch has its own weights; the batch stride is the matrix size.
 *   - Device pointers are CUDA device addresses on the device that was
 *     current when the plan was created.  The caller owns every buffer and
 *     stream and keeps them alive until the work on the stream has finished.
 *   - Status codes are returned; nothing is thrown across this interface.
 *   - Computation: inputs are read in their storage type, products are
 *     accumulated in fp32 (fp64 for B2B_F64), every intermediate is rounded
 *     to the operand type of the next GEMM (fp16 / bf16: round to nearest
 *     even; tf32: round to nearest, ties away from zero; fp64: kept), and the
 *     last product is rounded to the output type.
 */
#ifndef B2B_H_
#define B2B_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct b2b_plan_s* b2b_plan_t;
/* Most GEMMs one plan chains (b2b_chain_plan_create). */
#define B2B_MAX_STAGES 8
/* A cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st* b2b_stream_t;

typedef enum {
  B2B_OK = 0,
  B2B_ERR_INVALID_ARG = 1, /* null plan/pointer, bad size                   */
  B2B_ERR_UNSUPPORTED = 2, /* valid request the library has no kernel for  */
  B2B_ERR_ALIGNMENT = 3,   /* pointer not 16-byte aligned                   */
  B2B_ERR_ALIAS = 4,       /* output overlaps an input                      */
  B2B_ERR_DEVICE = 5,      /* current device is not sm_103 (GB300)          */
  B2B_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed             */
  B2B_ERR_TIMEOUT = 7      /* a bounded wait inside a kernel gave up        */
} b2b_status_t;

/* Storage and compute types of a chain (inputs / intermediate / output). */
typedef enum {
  B2B_F16_F32OUT = 0,  /* fp16 in, fp16 intermediates, fp32 out            */
  B2B_F16 = 1,         /* fp16 in, fp16 intermediates, fp16 out            */
  B2B_BF16 = 2,        /* bf16 in, bf16 intermediates, bf16 out            */
  B2B_TF32 = 3,        /* fp32 storage, tf32 operands and intermediate, fp32 out */
  B2B_F64 = 4,         /* fp64 throughout                                   */
  B2B_BF16_F32OUT = 5, /* bf16 in, bf16 intermediates, fp32 out           */
  /* Mixed-type cascades (two or more stages): A and W[0] in fp32 storage,
   * multiplied as tf32 operands; every intermediate and every later weight
   * fp16 (B2B_TF32_F16) or bf16 (B2B_TF32_BF16); fp32 out. */
  B2B_TF32_F16 = 6,
  B2B_TF32_BF16 = 7
} b2b_dtype_t;

/*
 * Create a plan for a fused chain (operator determination and relation
 * determination, patent para. 46-53, 140-142).
 *   out      receives the plan handle (set to NULL on failure).
 *   dtype    see b2b_dtype_t.
 *   batch, M >= 0 (any M: the last row tile is partial; batch == 0 or
 *            M == 0 gives an empty chain whose runs do nothing).
 *   K        contraction length of GEMM1, >= 1.
 *   N1, N2   output widths of GEMM1 and GEMM2.
 *   N3       output width of GEMM3, or 0 for a two-stage chain.
 * Sizes the library supports (otherwise B2B_ERR_UNSUPPORTED):
 *   16-bit types: K % 8 == 0; N1, N2 (and N3) % 8 == 0; intermediate
 *                 widths (N1, and N2 of a three-stage chain) <= 512; the
 *                 last width <= 4096 (the last GEMM runs in passes of up to
 *                 256 columns).
 *   B2B_TF32:     two stages; K % 4 == 0; N1 <= 256; N1, N2 % 4 == 0.
 *   B2B_TF32_F16, B2B_TF32_BF16: two or more stages; K % 4 == 0; every
 *                 width % 8 == 0; intermediate widths <= 512, the last
 *                 <= 4096.
 *   B2B_F64:      two stages; K % 4 == 0; N1, N2 in {16, 32, 64}.
 * Binds to the current CUDA device, which must be an sm_103 GPU
 * (B2B_ERR_DEVICE otherwise).  Allocates a 4-byte device status word; a
 * two-stage 16-bit plan whose weights stay resident over several batches
 * also a tile-schedule table (36 bytes per CTA, copied once).  Weights of
 * every type are read as stored.  No kernel is launched.
 */
b2b_status_t b2b_plan_create(b2b_plan_t* out, b2b_dtype_t dtype, int64_t batch, int64_t M,
                             int64_t K, int64_t N1, int64_t N2, int64_t N3);

/*
 * Create a plan for a cascade of n_stages GEMMs, 1 <= n_stages <= B2B_MAX_STAGES
 * (patent para. 41: the output of each operator is the input of the next):
 *   E = (..((A.W[0]).W[1])..).W[n_stages-1],
 * with A[batch][M][K], W[s][batch][N[s-1]][N[s]] (N[-1] = K) and the output
 * E[batch][M][N[n_stages-1]], rounded as described above between GEMMs.
 *   N        n_stages output widths (host array, read during the call).
 * Supported sizes are those of b2b_plan_create, for every intermediate
 * width N[0..n_stages-2] (16-bit types: any n_stages; B2B_TF32 and B2B_F64:
 * n_stages <= 2).  n_stages == 1 gives the single-GEMM plan of
 * b2b_gemm_plan_create; 2 or 3 give the plans of b2b_plan_create.  Run the
 * plan with b2b_chain_run (or, for at most three stages, b2b_run).
 * Returns B2B_ERR_INVALID_ARG for a null `out` or `N`, or n_stages out of range.
 */
b2b_status_t b2b_chain_plan_create(b2b_plan_t* out, b2b_dtype_t dtype, int64_t batch, int64_t M,
                                   int64_t K, int n_stages, const int64_t* N);

/*
 * A single GEMM D = A.B (one operator, no fusion), used to build the unfused
 * reference chain.  dtype gives the input and output types as above (the
 * output of B2B_F16 / B2B_BF16 is 16-bit, of B2B_TF32 fp32).  Run it with
 * b2b_run(plan, A, B, NULL, NULL, D, stream).
 */
b2b_status_t b2b_gemm_plan_create(b2b_plan_t* out, b2b_dtype_t dtype, int64_t batch, int64_t M,
                                  int64_t K, int64_t N);

/*
 * Run the fused chain asynchronously on `stream` (rearrangement and
 * execution, patent para. 54-60, 143).
 *   A, B, C  device inputs as described above; F is the third weight for a
 *            three-stage plan and must be NULL for a two-stage plan.
 *            For a single-GEMM plan C and F must be NULL.
 *   D        device output [batch][M][N_last]; must not overlap any input.
 * Every pointer must be 16-byte aligned (B2B_ERR_ALIGNMENT).
 * Returns B2B_ERR_CUDA if the launch fails.  A kernel that gives up a
 * bounded wait records B2B_ERR_TIMEOUT in the plan's status word, which
 * b2b_plan_device_status reports.  Runs on one plan from several streams
 * may overlap: the plan is not modified by b2b_run.  A plan of more than
 * three stages is rejected (B2B_ERR_INVALID_ARG): use b2b_chain_run.
 */
b2b_status_t b2b_run(b2b_plan_t plan, const void* A, const void* B, const void* C, const void* F,
                     void* D, b2b_stream_t stream);

/*
 * Run any plan asynchronously on `stream`: W is a host array of the plan's
 * n_stages device weight pointers (read during the call), `out` the device
 * output [batch][M][N_last].  Pointer rules, errors and the status word are
 * those of b2b_run; a null W or a null entry in it is B2B_ERR_INVALID_ARG.
 */
b2b_status_t b2b_chain_run(b2b_plan_t plan, const void* A, const void* const* W, void* out,
                           b2b_stream_t stream);

/* Destroy a plan (NULL is accepted).  No run on it may still be in flight. */
b2b_status_t b2b_plan_destroy(b2b_plan_t plan);

/*
 * Synchronise `stream`, then read and clear the plan's device status word:
 * B2B_OK, or B2B_ERR_TIMEOUT if a kernel gave up a bounded wait since the
 * last query.  Returns B2B_ERR_CUDA if the synchronisation itself fails.
 */
b2b_status_t b2b_plan_device_status(b2b_plan_t plan, b2b_stream_t stream);

/* Time budget of every bounded wait inside the kernels of this plan, in
 * nanoseconds (default 2e9).  0 restores the default; budgets below 1e6
 * (1 ms) are raised to 1 ms, because after a wait runs out the same budget
 * bounds the waits for the copies and MMAs still in flight, which must end
 * before the kernel frees its tensor memory. */
b2b_status_t b2b_plan_set_wait_budget(b2b_plan_t plan, uint64_t budget_ns);

/*
 * Test support for failure detection.  With B2B_DEBUG_DROP_FIRST_LOAD set,
 * the next runs of a tensor-core plan arm the first shared-memory stage of
 * every CTA but never copy data into it, so the MMA thread's wait on that
 * stage runs out after the plan's wait budget; every role then leaves its
 * loops, in-flight copies and MMAs are drained, tensor memory is freed, and
 * b2b_plan_device_status reports B2B_ERR_TIMEOUT.  The output is not written.
 * No fault, trap or unbounded wait is involved.  Other flag bits are
 * rejected (B2B_ERR_INVALID_ARG); 0 restores normal runs.  fp64 plans (which
 * have no waits) ignore the flag.
 */
#define B2B_DEBUG_DROP_FIRST_LOAD 1u
b2b_status_t b2b_plan_set_debug(b2b_plan_t plan, uint32_t flags);

/*
 * Describe a plan: kernel launches per b2b_run, grid size, threads per CTA,
 * dynamic shared memory per CTA, tensor-memory columns, ring depth and the
 * number of passes of the last GEMM.  Any pointer may be NULL.
 */
b2b_status_t b2b_plan_info(b2b_plan_t plan, int* launches_per_run, int* grid, int* threads,
                           int* smem_bytes, int* tmem_cols, int* ring_stages, int* passes);

/* Human-readable name of a status code (static storage). */
const char* b2b_status_string(b2b_status_t status);

/*
 * Coordination matrix of a register rearrangement (patent para. 75-102,
 * Fig. 4; host only, no GPU needed).
 * n threads each hold m values; receiver i's value r must come from thread
 * src_thread[i*m + r], register src_reg[i*m + r].  The result is an n x m
 * matrix H of triples (p, q, r) in P, Q, R (row-major, index i*m + j): in
 * exchange round j, thread i takes value q of thread p and keeps it as its
 * value r.  In every column the p's are distinct, so no thread is asked for
 * two values in one round (para. 90).  Receivers are scheduled in order and
 * each takes, round by round, its first remaining source that is still free
 * in that round; if that greedy order gets stuck a depth-first search
 * finishes the matrix.
 * Returns B2B_OK, B2B_ERR_INVALID_ARG (bad sizes, a source used twice, or a
 * thread asked for a number of values other than m), or B2B_ERR_UNSUPPORTED
 * (no conflict-free schedule exists).
 */
b2b_status_t b2b_coordination_matrix(int n, int m, const int* src_thread, const int* src_reg,
                                     int* P, int* Q, int* R);

/*
 * Layout probe of the accumulator -> operand rearrangement (test support).
 * Runs the converter device code of the tcgen05 kernels on one 128-row tile:
 * acc[128][width] (device, fp32 bit patterns) is written to tensor memory in
 * the accumulator layout, read back by the same converter routine the fused
 * kernel uses, rounded to the operand type of `dtype`, and the operand image
 * is copied to `image` (device):
 *   16-bit types: the K-major 128-byte-swizzled shared-memory image,
 *                 width*256 bytes;
 *   B2B_TF32:     the tensor-memory operand, 128 x width 32-bit words, row m
 *                 then column k.
 * width is 64, 128 or 256.  Synchronous.
 */
b2b_status_t b2b_probe_operand_image(b2b_dtype_t dtype, int width, const void* acc, void* image,
                                     b2b_stream_t stream);

/*
 * Layout probes of the other forms of the 16-bit rearrangement (test
 * support).  acc[128][width] (device, fp32 bit patterns) is put into tensor
 * memory in the accumulator layout and rearranged by the same device code
 * the fused kernels run; the result is copied to `out` (device):
 *   B2B_PROBE_TMEM16: the intermediate kept in tensor memory as the A
 *     operand of the next GEMM (two-stage 16-bit chains with resident
 *     weights): packed in place, two K elements per 32-bit column; out is
 *     [128][width / 2] 32-bit words, row (= TMEM lane) major.  width is 64,
 *     128 or 256; region must be 0.
 *   B2B_PROBE_PAIR_CONVERTERS: the converters of the CTA-pair kernel (eight
 *     warps, two per TMEM lane quadrant, each taking 64 of every 128
 *     columns), the accumulator starting in tensor-memory region `region`
 *     (0 or 1, of 256 columns each; a wider one continues in the other);
 *     out is the K-major 128-byte-swizzled shared-memory image,
 *     width * 256 bytes.  width is 128, 256, 384 or 512.
 * dtype is a 16-bit type (B2B_F16*, B2B_BF16*); other dtypes give
 * B2B_ERR_UNSUPPORTED, bad forms, widths or regions B2B_ERR_INVALID_ARG.
 * Synchronous.
 */
#define B2B_PROBE_TMEM16 1
#define B2B_PROBE_PAIR_CONVERTERS 2
b2b_status_t b2b_probe_operand_layout(b2b_dtype_t dtype, int form, int width, int region, const void* acc,
                                      void* out, b2b_stream_t stream);

/*
 * Scheduling tables of the kernels (test support, host only, no GPU
 * needed): the same host-and-device functions the kernels walk, evaluated
 * on the host, so that the CPU models of the kernels' barrier protocols can
 * be checked against them.  args / out are host arrays of nargs / nout
 * integers.
 *   B2B_TABLE_REGION_USE (one-CTA kernel): args S, npass, nz, lookahead,
 *     tiles; out receives (region, use count) for every phase of every
 *     tile, tile-major, 2 * tiles * (S - 1 + npass) integers.
 *   B2B_TABLE_PAIR_UNITS (CTA-pair kernel): args total_tiles, m_tiles,
 *     npass, split, clusters, cluster; out receives the cluster's unit count
 *     and (batch, 256-row tile, first pass, end pass) of each unit.
 *   B2B_TABLE_PAIR_REGIONS (CTA-pair kernel): args the widths of successive
 *     accumulators; out receives, per accumulator, the tensor-memory region
 *     it starts in and the tensor-memory column of its columns 0, 128, 256
 *     and 384 (5 integers each).
 *   B2B_TABLE_PAIR_TMEM_INTERMEDIATES (CTA-pair kernel): args 1 for a tf32
 *     chain else 0, the last GEMM's pass count, then the padded widths of
 *     the intermediates; out[0] receives the mask (bit s: intermediate s)
 *     of the intermediates a plan keeps packed in tensor memory rather than
 *     in the shared-memory operand image.
 * Returns B2B_ERR_INVALID_ARG for an unknown table, bad arguments or too
 * small an `out`.
 */
#define B2B_TABLE_REGION_USE 1
#define B2B_TABLE_PAIR_UNITS 2
#define B2B_TABLE_PAIR_REGIONS 3
#define B2B_TABLE_PAIR_TMEM_INTERMEDIATES 4
b2b_status_t b2b_schedule_table(int table, const int64_t* args, int nargs, int64_t* out, int nout);

/*
 * Register probe of the fp64 rearrangement (test support).  One warp loads
 * cfrag[lane][tiles*2] (device, the m8n8k4 accumulator fragments of `tiles`
 * 8-column tiles, lane-major) into registers, performs the shuffle rounds
 * the fp64 kernel derives from its coordination matrix, and writes the
 * operand fragments afrag[lane][tiles*2] (device, lane-major).  tiles is 1..8.
 * Synchronous.
 */
b2b_status_t b2b_probe_f64_rearrange(int tiles, const double* cfrag, double* afrag,
                                     b2b_stream_t stream);

/*
 * tf32 chain D = (A.B).C without any device allocation (no counterpart in the
 * patent; it exists for callers that cannot allocate device memory: code that
 * runs where cudaMalloc is forbidden or would fail, such as inside a framework
 * that hands out all device memory itself, and callers that must not create
 * plan objects, which own device memory).
 *   Sizes, layout and arguments as for a B2B_TF32 plan with N3 = 0; A, B, C
 *   and D are the caller's device buffers (fp32, row-major, 16-byte aligned).
 *   It runs the kernels of a B2B_TF32 plan in their form that reads the
 *   weights transposed ([N][K], K-major; a plan reads them as stored), and
 *   the weights are first transposed by a second kernel into a fixed scratch
 *   array owned by the library: 4 MiB (2^20 32-bit words) on every GPU that
 *   loads the library, kept until the process exits.  batch * (K*N1 + N1*N2)
 *   must not exceed 2^20, otherwise B2B_ERR_UNSUPPORTED.
 *   The first call on a device (and the first after that device's context
 *   has been replaced) looks up the array's device address and raises the
 *   kernel's shared-memory limit: make it before any stream capture.  Later
 *   calls make neither runtime call.  All calls share the array; calls whose
 *   kernels overlap on the GPU race on it.  Nothing in it must start at zero.
 *   No cudaMalloc or cudaFree is made.  Asynchronous on `stream`; a bounded
 *   wait that runs out inside the kernel is not reported (there is no status
 *   word).
 */
b2b_status_t b2b_run_tf32_noalloc(int64_t batch, int64_t M, int64_t K, int64_t N1, int64_t N2,
                                  const void* A, const void* B, const void* C, void* D,
                                  b2b_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* B2B_H_ */
