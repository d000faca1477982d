// prnn_internal.h -- shapes, plans and kernel launchers shared by the
// translation units of libprnn.so (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace prnn {

// ---- input projection: P[m][n] = bias[n] + sum_k x[m][k] * Wx[n][k] -------
// m < M = T*B, n < N = H, k < K = I.  Optionally also fills y (same shape as
// P) with the "not yet written" sentinel.
struct ProjArgs {
  int M, N, K;
  const float* x;      // [M][K] fp32
  const void* Wx;      // [N][K] fp32 or fp16
  const float* bias;   // [N]
  float* P;            // [M][N]
  float* y_fill;       // [M][N] or nullptr
};
cudaError_t launch_projection_simt(const ProjArgs& a, bool wx_fp16, cudaStream_t s);

// tcgen05 projection: x is converted to fp16 into x16 [M][Kp] (Kp = K rounded
// up to 64, zero padded), Wx16 is [N][Kp] fp16 zero padded.
struct ProjTcArgs {
  int M, N, K, Kp;
  const float* x;        // [M][K] fp32
  __half_raw* x16;       // [M][Kp] workspace
  const __half_raw* Wx16;// [N][Kp]
  const float* bias;     // [N]
  float* P;              // [M][N]
  float* y_fill;         // [M][N] or nullptr
};
bool projection_tc_supported();
cudaError_t launch_projection_tc(const ProjTcArgs& a, int* status, cudaStream_t s);
// C[M][N] (fp32, row-major) = sum_k A[m][k] * B[n][k] on the tensor cores;
// A [M][Kp] and B [N][Kp] fp16 or bf16, K-major, Kp a multiple of 64 (zero
// padded), 16-byte aligned.
struct GemmTcArgs {
  int M, N, Kp;
  const void* A;
  const void* B;
  bool bf16;
  float* C;
};
cudaError_t launch_gemm_tc(const GemmTcArgs& g, int* status, cudaStream_t s);

// ---- persistent recurrent kernels --------------------------------------
// Default pause (ns) before the first poll of a step's input (see
// spin_cycles), per kernel family, from sweeps on GB300: the dense kernels
// (every thread polls its own chunks straight into registers) gain from
// 50-100 ns and need it on boxes where the exchange otherwise settles into
// its slow state; the sparse kernels (h staged through shared memory) are
// fastest without it up to H ~ 2000 (H=1792: 1.58 / 1.63 us/step at 0 / 50
// ns) and gain 3-8 % from 100 ns at H = 5760.
constexpr int kDenseDelayNs = 100;
// The dense kernel's first pass of a step polls bw batch columns of h (bw*H*4
// bytes per CTA).  When that pass is the step's only one (its data was
// published at the end of the previous step) and it polls more than 16 KiB,
// the 100 ns pause does not keep the exchange in its fast state: with all 4
// columns of B = 4 in one pass (one CTA group), H=1792 runs 4.4-7.5 us/step at
// 100 ns and 2.4 at 200 ns, H=2048 6.0-7.0 and 2.4 (about 10 at 0 ns for H =
// 1536 .. 2048).  With several passes the first pass reads data published
// passes earlier, and 200 ns only costs 1-2 %.  A single-column pass (B = 1)
// is bimodal at 100 ns too (H=1152: 1.1 or 2.1 us/step from run to run,
// H=4096: 3.5-5.5) and steady at 200 (1.17, 3.7; H=2304 1.76 against a
// 1.68 median with a 2.1 tail).
__host__ __device__ constexpr int dense_delay_ns(int H, int bw, int passes) {
  return passes == 1 && (bw == 1 || (long long)bw * H * 4 > 16384) ? 200 : kDenseDelayNs;
}
__host__ __device__ constexpr int sparse_delay_ns(int H) { return H > 4096 ? 100 : 0; }
// Default first pause (ns) before re-polling stale step data (Waiter::pause):
// none for the single-layer kernels (it only slows them), 250 ns for the
// stacked kernel, whose slices otherwise fall into the slow exchange state
// (H=1152, L=2: 11.6 -> 3.6 us/step; H=256, L=4: 4.5 -> 1.4).
constexpr int kBackoffNs = 0;
constexpr int kStackBackoffNs = 250;
struct RecurCommon {
  int T, B, H;
  int n_cta, R;          // CTAs (G * cpg) and rows per CTA (last CTA of a group may own fewer)
  int G, cpg;            // CTA groups (each owns a contiguous slice of the batch) and CTAs per group
  int nthreads;
  size_t smem;           // dynamic shared memory bytes
  const float* P;        // [T][B][H] projection (bias included)
  const float* h0;       // [B][H] or nullptr
  float* y;              // [T][B][H], pre-filled with the sentinel
  // Reverse mode (the backward pass): steps run t = T-1 .. 0, h_prev is
  // y[t+1] (P = the masked dy, W = Wh^T, y = delta).  With p_masked the
  // output is P + sum, or 0 where P holds kMaskedMarker, instead of ReLU.
  int reverse;
  int p_masked;
  int* status;           // int[4]
  long long timeout_ns;
  int poll_delay;        // SM cycles between publishing a step and the first poll of the next
  int poll_backoff;      // SM cycles before re-polling stale data (doubling, up to 4x)
  int sync_mode;         // 0 flags in data, 1 grid barrier
  unsigned* bar;         // grid barrier counter (sync_mode 1)
  int drop_cta, drop_step;  // fault hook (-1 = off)
  // nullptr, or a second [T][B][H] destination of every output the kernel
  // publishes (plain stores): a page-locked host buffer the device can
  // address, so the result reaches the host while the recurrence runs
  float* y_mirror;
};

// Dense: thread i owns 4-column chunks i, i+nthreads, ...; weights packed as
// [chunk-slot j][row][thread] vectors of 4 (fp16: 8 bytes, fp32: 16 bytes).
struct DenseRecurArgs {
  RecurCommon c;
  const void* Wpk;       // packed per CTA: n_cta blocks of cpt*R*nthreads vec4
  int cpt;               // chunk slots per thread = ceil((H/4) / nthreads)
  int wfp16;
};
cudaError_t launch_recur_dense(const DenseRecurArgs& a, int bw, cudaStream_t s);

// Dense fp16 for wide batches (persistent_dense_wide.cu): CTAs of c.R rows
// (8 or 16), R / 4 x S threads, passes of 8 batch columns staged by bulk
// copies one or two passes ahead; one CTA group (c.G = 1).  Wpk per CTA: Wlo[R/4][H/4]
// then Whi[R/4][H/4] uint4; Wlo[q][c] holds rows 4q, 4q+1 and Whi[q][c] rows
// 4q+2, 4q+3 of columns 4c .. 4c+3 (fp16, row by row).
constexpr int kDenseWideMinB = 16;  // two passes of 8 columns or more
struct DenseWideArgs {
  RecurCommon c;
  const void* Wpk;
  const float* h0_rows;  // [B][H]: h0, or zeros
  int S;                 // threads per 4-row group: 96, 64 or 32, dividing H / 4
  int depth;             // passes a copy is issued ahead (1 or 2; depth + 1 h buffers)
};
cudaError_t launch_recur_dense_wide(const DenseWideArgs& a, cudaStream_t s);
// Whether the wide kernel serves H on this device; its rows per CTA, S,
// prefetch depth and shared memory.
bool recur_dense_wide_plan(int H, int sm_count, size_t smem_optin, int* R, int* S, int* depth,
                           size_t* smem);

// Dense fp16 for wide batches on the tensor cores with the product split over
// K inside clusters (persistent_dense_ksplit.cu): H / 128 clusters of cs CTAs
// (2 <= cs <= 8); CTA j of cluster c multiplies rows [128c, 128c + 128) of Wh
// by K slice j of h_{t-1} (ksplit_slice: the H / 16 K steps of 16 columns
// shared out as evenly as they go) and finalizes batch columns
// [j B / cs, (j + 1) B / cs) of those rows.  Wimg per CTA (cluster-major, then
// j): nat atoms of 128 rows x 128 bytes, fp16, K-major, 16-byte chunk q of
// row m at q ^ (m & 7) (the 128-byte swizzle), columns past the slice zero;
// nat = the widest slice's 64-column atoms.
constexpr int kKsplitMaxCluster = 8;
constexpr int kKsplitMaxSlice = 384;  // K columns per CTA at most (plans with wider slices are not made)
constexpr int kKsplitMaxSliceStream = 1024;  // the same for the streamed-A plan (B <= 16)
constexpr int kKsplitMaxB = 32;
// The default rule (PRNN_OPT_DENSE_KSPLIT = 1): where the kernel measured
// faster than the CUDA-core kernels on GB300.  Its step has a fixed cost of
// about 2.5 us (the L2 exchange, the MMA chain, the reduction through
// distributed shared memory), so it wins once their arithmetic per step is
// larger: H=2304 B=4 2.65 against 2.97 us, H=1536 B=8 2.54 / 4.30, H=640
// B=12 2.47 / 3.03; it loses at H=1152 B=8 (2.49 / 2.21).  Monotone in B.
__host__ __device__ constexpr bool ksplit_default(int H, int B) {
  return (H >= 2048 && B >= 4) || (H >= 1536 && B >= 8) || (H >= 640 && B >= 12);
}
// Sparse layers run their densified matrix on the K-split kernel by default
// (PRNN_OPT_SPARSE_KSPLIT = 1) where that measured faster than the sparse
// kernel, whose gathers are bound by shared memory at wide batch: from about
// 3600 entries per row x batch column at H >= 1536 (H=2304 10 % B=16 3.22
// against 3.54 us, 5 % B=32 4.14 / 4.27, H=1792 25 % B=8 2.62 / 2.78), and
// from 8192 at H >= 1152 (25 % B=32 3.06 / 3.25); the sparse kernel stays
// faster below (H=1792 10 % B=16 2.91 / 2.31, H=1152 25 % B=16 2.61 / 2.26).
// Where the weights are streamed (H >= 2560: the step costs about 7.3 us
// whatever the batch) it takes 6000: H=4096 10 % B=16 8.8 against 11.1 us,
// while 25 % B=4 stays on the sparse kernel (6.3 us).  Monotone in B.
__host__ __device__ constexpr size_t ksplit_sparse_threshold(int H) {
  return H >= 2560 ? 6000 : (H >= 1536 ? 3600 : (H >= 1152 ? 8192 : (size_t)1 << 40));
}
__host__ __device__ constexpr bool ksplit_sparse_default(int H, size_t nnz, int B) {
  return ksplit_default(H, B) && nnz * (size_t)B >= ksplit_sparse_threshold(H) * (size_t)H;
}
struct DenseSplitArgs {
  RecurCommon c;
  const void* Wimg;
  const float* h0_rows;  // [B][H]: h0, or zeros
  int cs, nat;
  uint32_t* trace;       // null, or [T][n_cta][kTraceWords] phase records (the
                         // first kKsplitTraceWords words of each, below)
  int stream;            // 1: Wh streamed from Wimg through rings (B <= 16), not resident
};
// Phase-trace record of the K-split kernel (one step, one CTA), words:
// 0 SM id, 1 CTA index, 2 cluster size, 3 K slice; SM-clock stamps (low 32
// bits) of thread 128 (the first epilogue thread) at 4 step start, 5 its own
// polls done, 6 the CTA barrier after the fill, 7 the MMAs seen complete,
// 8 partial sums staged, 9 copies issued, 10 the second CTA barrier, 11 the
// peers' partial sums received, 12 publish done; 13 thread 0's clock after it
// issued the MMAs; 14-15 globaltimer ns after the first barrier (low, high),
// 16-17 after the publish (low, high); 18 the most re-poll rounds of thread
// 128; 19 unused.
constexpr int kKsplitTraceWords = 20;
// K slice j of cs: first column k0 and width kl (multiples of 16)
__host__ __device__ constexpr int ksplit_k0(int H, int cs, int j) { return j * (H / 16) / cs * 16; }
__host__ __device__ constexpr int ksplit_kl(int H, int cs, int j) {
  return ksplit_k0(H, cs, j + 1) - ksplit_k0(H, cs, j);
}
__host__ __device__ constexpr int ksplit_nat(int H, int cs) {
  return ((H / 16 + cs - 1) / cs + 3) / 4;
}
// Dynamic shared memory of the kernel for a batch of B columns.
size_t recur_dense_ksplit_smem(int nat, int B, int cs, bool stream);
// The largest cluster size (8 .. 2) for which all H / 128 clusters of the
// kernel are resident at once (one CTA per SM) and its shared memory fits;
// 0 when none does or H % 128 != 0.  When Wh does not fit on chip beside the
// operand tiles, the plan streams it (*stream = true; batches of <= 16).
int recur_dense_ksplit_plan(int H, bool* stream);
cudaError_t launch_recur_dense_ksplit(const DenseSplitArgs& a, cudaStream_t s);

// Dense fp16 on the tensor cores (persistent_dense_tc.cu): per CTA an image of
// its rows of Wh, nslices = H/64 K slices of N rows x 128 bytes (fp16,
// 128-byte swizzle, rows past R zero), N = R rounded up to 16, N <= 32; the
// group's batch columns Bl <= 32.
struct DenseTcArgs {
  RecurCommon c;
  const void* Wimg;
  int N, nslices, nring;  // nring: A slots (2 .. 8)
};
cudaError_t launch_recur_dense_tc(const DenseTcArgs& a, cudaStream_t s);
size_t recur_dense_tc_smem(int H, int N, int nring);
int recur_dense_tc_ring(int H, int N, size_t smem_optin);  // 0: does not fit
int recur_dense_tc_threads();
size_t recur_dense_smem(int R, int cpt, int nthreads, bool fp16, int bw);
int recur_dense_rmax(int R);   // 0 if R unsupported
int recur_dense_bw(int batch_cols);          // batch columns per pass: 1, 2 or 4

// Register model of recur_dense_kernel<F16, RMAX, BW, CPT>: accumulators,
// the thread's h chunks, the weights of RB rows in flight, overhead.  The
// compiler hoists every weight load of the unrolled loop (best ILP); when
// that would not fit in registers the rows are processed in blocks of
// RB = 8.  The model sets the kernel's launch bound (512 threads when it fits
// 128 registers, else 256) and lets the planner avoid variants that spill.
__host__ __device__ constexpr int dense_regs_rows(bool f16, int rmax, int bw, int cpt, int rb) {
  return rmax * bw + cpt * bw * 4 + rb * cpt * (f16 ? 2 : 4) + 32;
}
__host__ __device__ constexpr int dense_row_block(bool f16, int rmax, int bw, int cpt) {
  return dense_regs_rows(f16, rmax, bw, cpt, rmax) <= 240 ? rmax : 8;
}
__host__ __device__ constexpr int dense_reg_estimate(bool f16, int rmax, int bw, int cpt) {
  return dense_regs_rows(f16, rmax, bw, cpt, dense_row_block(f16, rmax, bw, cpt));
}
__host__ __device__ constexpr int dense_launch_bound(bool f16, int rmax, int bw, int cpt) {
  return dense_reg_estimate(f16, rmax, bw, cpt) <= 120 ? 512 : 256;
}

// Stacked dense layers in one persistent launch (persistent_stack.cu).  Grid
// = L slices of c.n_cta CTAs; slice l computes layer l from the concatenated
// weights [Wx_l | Wh_l] (K = I_l + H columns), packed per CTA like the dense
// kernel's weights.  All layers share H, R, G, cpg, nthreads and cpt.
constexpr int kStackMaxLayers = 8;
struct StackLayerArgs {
  const void* Wpk;       // [cpg][cpt][R][nthreads] vec4 of [Wx_l | Wh_l]
  const float* bias;     // [H]
  const float* xin;      // [T][B][I]: x (layer 0) or y of layer l-1
  float* y;              // [T][B][H], pre-filled with the sentinel
  const float* h0;       // [B][H] or nullptr
  int I;                 // input width (multiple of 4)
  int poll_in;           // 1: xin is produced during this launch (poll it)
};
struct StackArgs {
  RecurCommon c;         // per-slice plan; c.P, c.y, c.h0 unused
  int L, cpt, wfp16;
  StackLayerArgs layer[kStackMaxLayers];
};
cudaError_t launch_recur_stack(const StackArgs& a, int bw, cudaStream_t s);
// Variants of the stack kernel that compile without spills (measured with
// -Xptxas -v): the dense register model plus the per-slot source offsets,
// and no 32-row variant with 8 or more (batch x chunk) vectors in flight.
__host__ __device__ constexpr bool stack_variant_ok(bool f16, int rmax, int bw, int cpt) {
  return dense_reg_estimate(f16, rmax, bw, cpt) + 4 * cpt + 8 <= 240 &&
         !(rmax == 32 && bw * cpt >= 8) && !(rmax == 32 && !f16 && cpt == 4);
}
size_t recur_stack_smem(int R, int cpt, int nthreads, bool fp16, int bw);

// Sparse row-balanced: per CTA, R rows x kp entries; thread (row, seg) with
// seg < tpr owns ept = kp/tpr entries, read as uint4 (4 packed entries).
// Packed entry = fp16 value bits | (column << 16).
struct SparseRecurArgs {
  RecurCommon c;
  const uint32_t* Wpk;   // [n_cta][R][ept/4][tpr] uint4
  int tpr, ept;
  int bgroup;            // batch columns staged per pass: 1, 2, 4, 8, 16 or 32
  int dbuf;              // 1: two h staging buffers (one CTA barrier per pass)
  int narrow;            // 1: stage h with 32-bit loads (ablation); 0: 128-bit
  const uint32_t* place; // [cpg][H/4] staging order of h (H % 128 == 0), or null:
                         // column c of group g = c/4 is staged at
                         // 128*(g/32) + 32*(c%4) + byte (c%4) of place[g]
  uint32_t* trace;       // null, or [T][n_cta][kTraceWords] phase records (column
                         // order and wide staging only)
  int regw;              // 1: the register-weight build (column order, nthreads <=
                         // 384, bgroup <= 4; see sparse_regw_fits)
  int umax;              // staging depth (float4 loads per thread per round): 0 for
                         // the default (12 for passes of <= 4 columns), or 2 or 6
                         // (bgroup <= 4; see sparse_staging_depth)
};
// The staging depth for a pass of bgroup columns of H over nthreads threads:
// the smallest of 2, 6 (else 0: the default 12) that covers each thread's
// share of the pass in one round.
inline int sparse_staging_depth(int H, int bgroup, int nthreads, bool placed) {
  (void)placed;
  if (bgroup > 4 || nthreads < 1) return 0;
  const int need = (bgroup * (H / 4) + nthreads - 1) / nthreads;
  return need <= 2 ? 2 : (need <= 6 ? 6 : 0);
}
// Whether the register-weight build of the sparse kernel serves a plan: at
// most 384 threads, batch passes of at most 4 columns, column-order staging,
// and at least 6 uint4 weight groups per thread (fewer would leave registers
// holding zero-valued padding groups that still cost gathers).
inline bool sparse_regw_fits(int nthreads, int bgroup, int ept, bool placed) {
  return nthreads <= 384 && bgroup <= 4 && ept / 4 >= 6 && !placed;
}
// Words of one phase-trace record (one step, one CTA): 17 slots of 16 words.
// Slot 0: SM id, CTA index, warps, then unused.  Slot 1 + w, warp w: SM-clock
// stamps (low 32 bits) of pass start, projection value requested, pause end,
// the warp's last staging poll fresh, barrier passed, gathers done, reduction
// done, publish issued; the most re-poll rounds of the warp's lanes;
// globaltimer ns after the barrier (low, high) and after the publish (low,
// high); the SM clock after the record's globaltimer reads; 2 unused.
constexpr int kTraceWords = 17 * 16;
cudaError_t launch_recur_sparse(const SparseRecurArgs& a, cudaStream_t s);
cudaError_t launch_recur_sparse_placed(const SparseRecurArgs& a, cudaStream_t s);
cudaError_t launch_recur_sparse_trace(const SparseRecurArgs& a, cudaStream_t s);
cudaError_t launch_recur_sparse_um(const SparseRecurArgs& a, cudaStream_t s);
cudaError_t launch_recur_sparse_regw(const SparseRecurArgs& a, cudaStream_t s);
cudaError_t launch_recur_sparse_trace_regw(const SparseRecurArgs& a, cudaStream_t s);
size_t recur_sparse_smem(int H, int R, int ept, int tpr, int bgroup, bool dbuf);

// The sparse kernel's exchange with no arithmetic; umax as in SparseRecurArgs
// (0 here: 8 float4 in flight per thread).
cudaError_t launch_sync_probe(const RecurCommon& c, int bgroup, int umax, cudaStream_t s);

// Host packing of row-balanced sparse rows into the kernel layout (pack.cu).
// vals/cols: [H][k]; writes out_packed[n_cta][R][ept/4][tpr][4]; returns ept.
struct PackStats {
  int ept = 0;               // entries per thread (multiple of 4)
  int cap = 0;               // max lanes per bank residue per slot that was needed
  long long conflicts = 0;   // lane-slots that share a bank with an earlier lane
};
// place_out (optional): per-CTA staging order of h, [n_cta][H/4] words, one
// per group of 4 columns, byte j = bank of column 4g+j within its class; the
// packed index field is then the staged position (see pack.cu).  Left empty
// when the layer keeps column order (not bank-aware, or H % 128 != 0).
int pack_sparse_rows(int H, int k, int R, int n_cta, int tpr, const uint16_t* vals,
                     const uint16_t* cols, std::vector<uint32_t>& out_packed, PackStats* stats,
                     int max_ept = 1 << 30, bool bank_aware = true,
                     std::vector<uint32_t>* place_out = nullptr);
bool staging_placement_supported(int H);
size_t sync_probe_smem(int H, int bgroup);

// ---- per-step path ------------------------------------------------------
struct StepArgs {
  int t, B, H;
  const float* P;        // [T][B][H]
  const float* hprev;    // [B][H] (h0, or y[t-1])
  float* y;              // [T][B][H]
  const void* W;         // dense: [H][H] (fp16 or fp32); sparse: [H][kp] packed
  int wfp16, sparse, kp;
};
cudaError_t launch_step(const StepArgs& a, cudaStream_t s);

cudaError_t launch_fill_sentinel(float* y, size_t n, cudaStream_t s);

// ---- backward: batched gradient products (grad.cu) ----------------------
// C[M][N] = sum_k A[k][m] * Brow(k)[n]; Brow(k) = B0 + k*ldb for k < K0
// (zeros if B0 is null), else B1 + (k-K0)*ldb.
struct GemmTnArgs {
  int M, N, K, K0;
  const float* A;
  int lda;
  const float* B0;
  const float* B1;
  int ldb;
  float* C;              // [M][N]
};
// C[M][N] = sum_k A[m][k] * W[k][n]; W fp32 or fp16.
struct GemmNnArgs {
  int M, N, K;
  const float* A;
  int lda;
  const void* W;
  int ldw, wf16;
  float* C;              // [M][N]
};
cudaError_t launch_gemm_tn(const GemmTnArgs& g, cudaStream_t s);
cudaError_t launch_gemm_nn(const GemmNnArgs& g, cudaStream_t s);
cudaError_t launch_colsum(const float* A, int K, int N, float* out, cudaStream_t s);
cudaError_t launch_transpose_rows(int K, int N, int K0, const float* B0, const float* B1, int ldb,
                                  float* out, cudaStream_t s);
cudaError_t launch_sddmm(int H, int kp, int K, const float* dT, const float* hT,
                         const uint16_t* cols, const int32_t* caller_pos, float* out,
                         cudaStream_t s);
cudaError_t launch_gather_pattern(int H, int kp, const float* dense, const uint16_t* cols,
                                  const int32_t* caller_pos, float* out, cudaStream_t s);
cudaError_t launch_fold_mask(const float* dy, const float* y, size_t n, float* out,
                             cudaStream_t s);
cudaError_t launch_transpose_bf16(int K, int Kp, int N, int K0, const float* B0, const float* B1,
                                  int ldb, void* out, cudaStream_t s);
cudaError_t launch_rows_bf16(int M, int K, int Kp, const float* src, void* out, cudaStream_t s);
cudaError_t launch_sparse_dh0(int B, int H, int kT, const uint16_t* valsT, const uint16_t* colsT,
                              const float* delta0, float* dh0, cudaStream_t s);

}  // namespace prnn
