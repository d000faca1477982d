/*
 * prnn.h -- C ABI of the persistent ReLU-RNN recurrence library (libprnn.so),
 * written for GB300 (sm_103a).
 *
 * The operation is the forward pass of one vanilla ("basic", non-LSTM) RNN
 * layer, the only layer kind of the persistent-rnn library page
 * (gitmyhub.com/pineking/persistent-rnn, "Important Constraints"):
 *
 *     h_t = ReLU(Wx x_t + Wh h_{t-1} + b),   t = 0 .. T-1,   y[t] = h_t
 *
 * computed in two stages: the input projection Wx x_t + b for every step at
 * once (the parallel work the "Optimizing Performance of Recurrent Neural
 * Networks on GPUs" abstract exposes), then the serial recurrence in one
 * persistent kernel that keeps Wh on chip for the whole sequence instead of
 * re-reading it every step (persistent-rnn page, "What This Project Does").
 * Wh is dense, or row-balanced sparse with the same number of non-zeros in
 * every row (load-balanced pruning, "Sparse Persistent RNNs: Squeezing Large
 * Recurrent Networks On-Chip", measured-effects table).  The call sequence
 * follows the cuDNN-like shape the persistent-rnn page describes ("Who Would
 * Use This"): create a handle for one layer shape, set weights, run forward.
 *
 * Conventions for every call:
 *  - Every function returns a prnn_status_t; nothing throws, nothing aborts.
 *  - Matrices are row-major, y = W x (W is [rows][columns]).
 *  - Sequences are time-major: x[T][B][I], y[T][B][H]; h0 is [B][H].
 *  - x, h0 and y are fp32.  Weights are fp32 or fp16 (IEEE binary16 bits
 *    passed as uint16_t); the bias is fp32; column indices are uint16_t.
 *  - A "stream" is a cudaStream_t passed as void*; NULL means the legacy
 *    default stream.
 *  - The library owns everything it allocates (packed weights, workspaces,
 *    the status word); the caller owns every pointer it passes in.
 *  - A handle's calls share its workspaces, so they must not overlap: call a
 *    handle from one host thread at a time, and keep its forward and backward
 *    passes ordered (one stream, or synchronize between streams).  Different
 *    handles are independent.
 */
#ifndef PRNN_H
#define PRNN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct prnn_handle* prnn_t;

typedef enum {
  PRNN_OK = 0,
  PRNN_ERR_INVALID_ARG = 1,  /* bad pointer, size, index set, alignment or aliasing */
  PRNN_ERR_UNSUPPORTED = 2,  /* layer does not fit on chip, or no usable GPU        */
  PRNN_ERR_NOT_READY = 3,    /* forward before weights were set                     */
  PRNN_ERR_CUDA = 4,         /* a CUDA runtime call failed                          */
  PRNN_ERR_OOM = 5,          /* device allocation failed                            */
  PRNN_ERR_TIMEOUT = 6       /* a step wait in the persistent kernel ran out (sticky) */
} prnn_status_t;

typedef enum { PRNN_F32 = 0, PRNN_F16 = 1 } prnn_dtype_t;

typedef enum {
  PRNN_ALGO_PERSISTENT = 0,  /* one persistent launch for all T steps, Wh on chip      */
  PRNN_ALGO_PER_STEP = 1     /* T launches (one CUDA graph), Wh re-read every step      */
} prnn_algo_t;

/* Tunables and test hooks for prnn_set_option(). */
typedef enum {
  PRNN_OPT_WAIT_TIMEOUT_US = 0,   /* limit of one step wait, microseconds (default 500000)    */
  PRNN_OPT_SYNC_MODE = 1,         /* 0: flags carried in the data (default); 1: grid barrier  */
  PRNN_OPT_DEBUG_DROP_CTA = 2,    /* fault hook: CTA that skips one publish (-1 = off)         */
  PRNN_OPT_DEBUG_DROP_STEP = 3,   /* fault hook: the step whose publish it skips               */
  PRNN_OPT_TIMING = 4,            /* 1: record CUDA events around each stage of forward        */
  PRNN_OPT_PROJECTION = 5,        /* 0: tensor cores when possible (default); 1: fp32 CUDA cores */
  PRNN_OPT_CTA_GROUPS = 6,        /* persistent: CTA groups splitting the batch (0 = automatic);
                                     takes effect at the next set_weights call                 */
  PRNN_OPT_WIDE_LOADS = 7,        /* sparse: 1 = stage h with 128-bit loads (default); 0 = 32-bit */
  PRNN_OPT_BANK_AWARE = 8,        /* sparse: 1 = bank-aware entry placement (default); 0 = plain,
                                     takes effect at the next set_weights call                 */
  PRNN_OPT_POLL_DELAY_NS = 9,     /* persistent: pause after publishing a step before the first
                                     poll of the next, ns, 0 .. 10000 (default: dense 100, or
                                     200 when a step is one batch pass of one column or polling
                                     more than 16 KiB of h per CTA; stacked 100; sparse 0, or
                                     100 for H > 4096)                                          */
  PRNN_OPT_POLL_BACKOFF_NS = 10,  /* persistent: pause before re-polling stale step data, ns,
                                     doubling per round up to 4x; 0 .. 10000 (default: 0, and
                                     250 for stacks)                                            */
  PRNN_OPT_RECURRENT_TC = 11,     /* dense fp16 persistent: 0 = tcgen05 recurrence when
                                     max_batch >= 16, 1 = never (default: at B <= 32 its chain
                                     of small dependent MMAs is slower than the CUDA-core
                                     kernel), 2 = whenever it fits; takes effect at the next
                                     set_weights call                                           */
  PRNN_OPT_STAGED_ORDER = 12,     /* sparse, bank-aware, H % 128 == 0: 1 = each CTA stages h in
                                     its own bank-balancing order (one lane per bank in every
                                     gather slot, at the cost of scattered staging stores);
                                     0 = column order; 2 = chosen per packing (default): with
                                     batch passes of >= 4 columns, the staged order when it
                                     packs rows tighter than column order, or when rows hold
                                     >= 256 entries and it packs at most 12 % looser (measured:
                                     it wins at wide batch and many entries, loses at B <= 4
                                     and at 1 % density).  Applies to Wh and to the backward's Wh^T
                                     alike; takes effect at the next set_weights call          */
  PRNN_OPT_SPARSE_REG_WEIGHTS = 13,/* sparse persistent: 1 = the register-weight build of the
                                     kernel (launch bound 384 threads, each thread's first 24
                                     entries in registers) wherever its plan fits: at most 384
                                     threads, batch passes of at most 4 columns, column order,
                                     at least 24 entries per thread (default); 0 = never       */
  PRNN_OPT_SPARSE_STAGING_DEPTH = 14,/* sparse persistent, passes of at most 4 columns (either
                                     staging order): 1 = stage h_{t-1} with the fewest float4 loads in
                                     flight per thread (2 or 6) that cover the thread's share of
                                     a pass in one round (default); 0 = always 12.  The sync
                                     floor probe follows the same choice                       */
  PRNN_OPT_DENSE_WIDE = 15,       /* dense fp16 persistent, flags in the data, H % 128 == 0 and
                                     H / 16 CTAs fit: the wide-batch kernel (CTAs of 8 or 16
                                     rows, passes of 8 batch columns staged by bulk copies a
                                     pass ahead) for forwards of B >= 16.  1 = where it
                                     measured faster than the B <= 4 kernel: B >= 17 with
                                     H >= 1024, or B >= 16 with H >= 2048 (default); 2 = for
                                     every B >= 16; 0 = never.  Takes effect at the next
                                     forward                                                    */
  PRNN_OPT_DENSE_KSPLIT = 16,     /* dense fp16 persistent, flags in the data, H % 128 == 0 and
                                     all H / 128 clusters of 2 .. 8 CTAs resident at once, one
                                     CTA per SM (on 152 SMs: clusters of 8 up to H = 1920, of
                                     6 up to 2304; from H = 2560 to 4096 clusters of 4 with
                                     Wh streamed from device memory each step, B <= 16): the
                                     tensor-core kernel that splits each step's product over
                                     K inside clusters (h split into fp16 hi + lo parts,
                                     about 22 bits; partial sums reduced through distributed
                                     shared memory) for forwards of B <= 32.
                                     1 = where it measured faster than the CUDA-core kernels
                                     (default): H >= 2048 and B >= 4, H >= 1536 and B >= 8,
                                     or H >= 640 and B >= 12; 2 = for every B <= 32; 0 =
                                     never.  Its weight image is built at set_weights when
                                     the default covers max_batch or the option is 2; it
                                     takes precedence over PRNN_OPT_DENSE_WIDE                  */
  PRNN_OPT_SPARSE_KSPLIT = 17     /* sparse persistent, flags in the data: run the layer's
                                     densified matrix (fp16, the same values) on the
                                     K-split kernel of PRNN_OPT_DENSE_KSPLIT for forwards
                                     of B <= 32.  1 = where it measured faster than the
                                     sparse kernel (default): the dense rule of
                                     PRNN_OPT_DENSE_KSPLIT, and (stored entries / H) x B
                                     >= 8192 at H >= 1152, >= 3600 at H >= 1536, >= 6000 at
                                     H >= 2560 (streamed weights); 2 = for every B <= 32
                                     (16 with streamed weights); 0 = never.
                                     Its image is built at set_weights when the default
                                     covers max_batch or the option is 2                     */
} prnn_option_t;

/* Plan and sizes chosen at create / set_weights time (read-only report). */
typedef struct {
  int hidden, input, max_batch;
  int wdtype, algo, sparse, weights_set;
  int k, k_padded;                 /* sparse: non-zeros per row, and per row after padding  */
  int sm_count, n_cta, rows_per_cta, threads_per_cta, threads_per_row;
  int projection_tensor_cores;     /* 1 if forward uses the tcgen05 projection               */
  int sparse_bank_cap;             /* sparse: max lanes of a warp sharing a bank per gather  */
  int cta_groups;                  /* CTA groups, each owning a slice of the batch columns   */
  size_t smem_bytes;               /* dynamic shared memory per CTA at max_batch             */
  size_t onchip_weight_bytes;      /* packed Wh bytes held on chip, all CTAs                 */
  size_t nnz;                      /* non-zeros of Wh (H*H when dense)                       */
  int recurrent_tensor_cores;      /* 1 if the dense recurrence runs on tcgen05 (wide batch) */
  int sparse_staged_order;         /* sparse: 1 if each CTA stages h_{t-1} in its own
                                      bank-balancing order (prnn_pack_sparse_host_placed)   */
  int sparse_reg_weights;          /* sparse: 1 if the forward at max_batch runs the
                                      register-weight build (PRNN_OPT_SPARSE_REG_WEIGHTS)   */
  int dense_wide_batch;            /* dense: 1 if the forward at max_batch runs the
                                      wide-batch kernel (PRNN_OPT_DENSE_WIDE); the plan
                                      fields above then describe that kernel's launch       */
  int dense_ksplit;                /* if the forward at max_batch runs the tensor-core
                                      K-split kernel (PRNN_OPT_DENSE_KSPLIT; a sparse
                                      layer's densified matrix: PRNN_OPT_SPARSE_KSPLIT),
                                      its cluster size (2 .. 8), else 0; the plan fields
                                      above then describe its launch (rows_per_cta: the
                                      128 rows of a cluster)                                */
} prnn_info_t;

/*
 * Create a handle for one layer shape on the current CUDA device.
 *   hidden    H >= 1, input I >= 1, 1 <= max_batch <= 32: upper bound of B in
 *             forward (the library targets the small-batch regime).
 *   wdtype    storage type of Wx and Wh.
 *   algo      PRNN_ALGO_PERSISTENT or PRNN_ALGO_PER_STEP.
 * Returns PRNN_ERR_UNSUPPORTED when the device is not sm_103 / lacks
 * cooperative launch, or when the dense layer cannot fit on chip (the
 * persistent-rnn page notes that on-chip weights cap the layer size,
 * "Important Constraints").  *out is NULL
 * on failure.
 */
prnn_status_t prnn_create(prnn_t* out, int hidden, int input, int max_batch,
                          prnn_dtype_t wdtype, prnn_algo_t algo);

/*
 * Set dense weights.  Wx [H][I] and Wh [H][H] in the handle's wdtype, bias [H]
 * fp32.  Pointers may be device, managed or host memory.  The library copies
 * and repacks them and synchronizes `stream` before returning, so the caller
 * may free its buffers on return.
 */
prnn_status_t prnn_set_weights_dense(prnn_t h, const void* Wx, const void* Wh,
                                     const float* bias, void* stream);

/*
 * Set row-balanced sparse recurrent weights: every row r holds exactly k
 * non-zeros, vals[r][j] (fp16 bits) at column cols[r][j].  Columns must lie in
 * [0, H) and be distinct within a row (any order); H <= 65535, 0 < k <= H,
 * handle wdtype PRNN_F16.  Wx [H][I] fp16 and bias [H] as for the dense call.
 * Invalid index sets give PRNN_ERR_INVALID_ARG and leave the handle unchanged.
 */
prnn_status_t prnn_set_weights_sparse(prnn_t h, const void* Wx, int k,
                                      const uint16_t* vals, const uint16_t* cols,
                                      const float* bias, void* stream);

/*
 * Set unbalanced sparse recurrent weights in compressed-row form: row r holds
 * the entries row_ptr[r] .. row_ptr[r+1]-1 of cols (uint16) and vals (fp16
 * bits); row_ptr has H+1 int32 entries from 0 to nnz; rows may differ in
 * length (or be empty) -- the matrix straightforward global magnitude pruning
 * leaves, the comparison point of the load-balanced pruning rows ("Sparse
 * Persistent RNNs: Squeezing Large Recurrent Networks On-Chip",
 * measured-effects table).  Columns in [0, H), distinct within a row.  The
 * library pads every row to the longest row's length with zero-valued
 * entries, so each row costs as much as the longest: prnn_get_info reports
 * that length as k.  Otherwise as prnn_set_weights_sparse.
 */
prnn_status_t prnn_set_weights_csr(prnn_t h, const void* Wx, int nnz, const int32_t* row_ptr,
                                   const uint16_t* cols, const uint16_t* vals,
                                   const float* bias, void* stream);

/*
 * Forward pass: y[t] = h_t for t < T.  x [T][B][I], h0 [B][H] (NULL = zeros),
 * y [T][B][H], all fp32 DEVICE pointers, 16-byte aligned; y must not overlap
 * x or h0.  1 <= B <= max_batch; T == 0 or B == 0 is a no-op.  Asynchronous
 * on `stream`.  y is fully overwritten.  If a step wait times out, y is
 * undefined and this and every later call on the handle return
 * PRNN_ERR_TIMEOUT (see prnn_get_status).
 */
prnn_status_t prnn_forward(prnn_t h, int T, int B, const float* x, const float* h0,
                           float* y, void* stream);

/*
 * The same forward pass on HOST buffers: x [T][B][I], h0 [B][H] (NULL =
 * zeros) and y [T][B][H] are fp32 in page-locked host memory that the device
 * can address (cudaHostAlloc / cudaMallocHost, or cudaHostRegister'ed), each
 * float-aligned.  Precondition, which the library cannot verify: each buffer
 * holds at least the elements its shape says within ONE allocation (the
 * recurrent kernel stores into y at every [t][b][r] offset).  As a best-effort
 * guard only, a buffer whose first or last element lies outside every
 * page-locked allocation is refused; a short buffer followed by another
 * page-locked allocation is not detected.  y must not overlap x or h0.  h0 is copied to a
 * device workspace owned by the handle (grown on demand, freed by
 * prnn_destroy).  With the tensor-core projection (prnn_info_t
 * projection_tensor_cores = 1) the projection's staging kernel reads x
 * straight from the host buffer, once; otherwise x is copied to a device
 * workspace first.  The persistent CUDA-core
 * recurrent kernels write every output into y itself, over the host link, as
 * they publish it, so the result needs no separate copy back; the per-step
 * path and the tcgen05 dense recurrence copy y back after the recurrence.
 * Asynchronous on `stream`: x, h0 and y belong to the library until the stream
 * is synchronized.  Results are bit-identical to prnn_forward on device copies
 * of the same inputs.  Errors: PRNN_ERR_INVALID_ARG for a pointer that CUDA
 * does not report as page-locked host memory (pageable or device memory),
 * otherwise as prnn_forward.
 */
prnn_status_t prnn_forward_host(prnn_t h, int T, int B, const float* x, const float* h0,
                                float* y, void* stream);

/* Release everything the handle owns.  NULL is accepted. */
prnn_status_t prnn_destroy(prnn_t h);

/*
 * Backward pass (backpropagation through time) of the layer for the loss L
 * whose gradient with respect to the outputs is dy = dL/dy:
 *
 *   delta_T = 0;  for t = T-1 .. 0:  delta_t = [y_t > 0] (dy_t + Wh^T delta_{t+1})
 *   db = sum_{t,b} delta_t,  dWh = sum_{t,b} delta_t h_{t-1}^T (h_{-1} = h0),
 *   dWx = sum_{t,b} delta_t x_t^T,  dx_t = Wx^T delta_t,  dh0 = Wh^T delta_0
 *
 * -- training is what the persistent kernels are for ("Optimizing
 * Performance of Recurrent Neural Networks on GPUs", Abstract).  The serial
 * reverse recurrence runs in the same persistent kernel as the forward with
 * Wh^T held on chip (a transposed copy packed at set_weights time); the five
 * gradients are batched products over all T*B rows.  The derivative of ReLU
 * at 0 is taken as 0 (y_t = 0 gives delta_t = 0); internally the mask is
 * folded into a copy of dy as one NaN bit pattern (0x7fc0beef), so a dy word
 * holding exactly that pattern reads as masked.
 *
 * Inputs (device, fp32, 16-byte aligned): x [T][B][I] and h0 [B][H] (NULL =
 * zeros) as given to prnn_forward, y [T][B][H] the output prnn_forward
 * produced for them with these weights, dy [T][B][H].  Outputs (device, fp32,
 * overwritten; NULL skips that gradient): delta [T][B][H] (dL/da_t, the
 * gradient at the pre-activations; the library's workspace is used when
 * NULL), dx [T][B][I], dh0 [B][H], dWx [H][I], db [H], and dWh: [H][H] for
 * dense weights; for sparse weights the gradient of every stored value, in
 * the order the values were passed to set_weights ([H][k] row-balanced, or
 * [nnz] compressed rows).  Outputs must not overlap the inputs or each other.
 * Asynchronous on `stream`; T == 0 or B == 0 writes zero gradients.
 * Persistent handles (PRNN_ERR_UNSUPPORTED for PRNN_ALGO_PER_STEP, or when
 * the transposed sparse matrix does not fit on chip).  After a timed
 * backward, prnn_get_timing reports (gradient products, reverse recurrence).
 */
prnn_status_t prnn_backward(prnn_t h, int T, int B, const float* x, const float* h0,
                            const float* y, const float* dy, float* delta, float* dx, float* dh0,
                            float* dWx, float* dWh, float* db, void* stream);

/* Synchronize `stream` and report the device-side status of past forwards
 * (PRNN_ERR_TIMEOUT once a step wait has run out; sticky). */
prnn_status_t prnn_get_status(prnn_t h, void* stream);

/* Human-readable name of a status code (static string). */
const char* prnn_status_string(prnn_status_t s);

prnn_status_t prnn_set_option(prnn_t h, prnn_option_t opt, long long value);
prnn_status_t prnn_get_info(prnn_t h, prnn_info_t* info);

/*
 * Stage times of the most recent forward, in milliseconds, measured with CUDA
 * events on the forward's stream (PRNN_OPT_TIMING must be 1).  Synchronizes.
 * ms_projection covers input staging + projection; ms_recurrence covers the
 * recurrent kernel (or the T per-step launches).  Either pointer may be NULL.
 */
prnn_status_t prnn_get_timing(prnn_t h, float* ms_projection, float* ms_recurrence);

/*
 * Phase trace of the sparse persistent kernel and of the dense K-split
 * kernel (a diagnostic; off unless a buffer is set).  While `buffer` (a
 * DEVICE pointer, 16-byte aligned, owned by the caller) is set, every
 * prnn_forward / prnn_forward_host of this handle runs the trace build of its
 * recurrent kernel.  The sparse kernel writes one record of
 * 17 x 16 uint32 words per step and CTA, [T][n_cta][17][16], for the step's
 * first batch pass.  Slot 0: SM id, CTA index, number of warps, then unused.
 * Slot 1 + w, warp w: SM clock (low 32 bits) at pass start, after its
 * projection value was requested, at the end of the pause before the first
 * poll, when the warp's last staging poll of h_{t-1} was fresh, after the CTA
 * barrier, after its gathers, its reduction and its publish; the most
 * re-poll rounds any of its lanes needed; globaltimer ns (a device-wide clock)
 * after the barrier (low word, high word) and after the publish (low, high);
 * the SM clock after those readings; 2 unused.  Slots of warps the CTA does
 * not have, and records of CTAs whose group has no batch column, are left as
 * they were.
 * The dense K-split kernel (PRNN_OPT_DENSE_KSPLIT) writes the first 20 words
 * of each record: SM id, CTA index, cluster size, K slice; SM-clock stamps of
 * its first epilogue thread at step start, its polls done, the CTA barrier
 * after the fill, the MMAs seen complete, partial sums staged, copies issued,
 * the second CTA barrier, the peers' partial sums received, publish done; the
 * MMA-issuing thread's clock after its last MMA; globaltimer ns after the
 * first barrier (low, high) and after the publish (low, high); the most
 * re-poll rounds of that thread; 1 unused.
 * The pages time the effect of each measure on whole steps (Sparse
 * Persistent RNNs, measured-effects table); this records where inside a step
 * the time goes.  Results are the same bits as without the trace.  Requires
 * `bytes` >= T * n_cta * 1088 at each forward (PRNN_ERR_INVALID_ARG otherwise)
 * and a sparse layer on the persistent path with column-order, wide staging,
 * or a forward that runs the K-split kernel (PRNN_ERR_UNSUPPORTED otherwise).
 * buffer = NULL turns the trace off.
 * Errors: INVALID_ARG for a misaligned, too small or non-device buffer.
 */
prnn_status_t prnn_set_trace_buffer(prnn_t h, void* buffer, size_t bytes);

/*
 * Step-synchronisation floor: runs the persistent grid of this handle for T
 * steps doing only the step-to-step exchange (every CTA waits for all of
 * h_{t-1}, then publishes its rows of h_t) with no arithmetic, so its time per
 * step is the latency floor of the recurrent kernel.  y [T][B][H] fp32 device
 * scratch.  Its time is reported by prnn_get_timing as ms_recurrence.
 */
prnn_status_t prnn_probe_sync_floor(prnn_t h, int T, int B, float* y, void* stream);

/*
 * Diagnostic (no handle): the step exchange of h inside thread-block clusters,
 * through distributed shared memory, with no arithmetic -- the alternative to
 * the L2 exchange of the persistent kernels (prnn_probe_sync_floor), measured
 * on the device.  `clusters` clusters of `cluster_size` CTAs (2, 4, 8 or 16)
 * each exchange a vector of `hidden` floats per step for `steps` steps
 * (hidden a multiple of 4 * cluster_size, at most 16384; steps >= 2): CTA r
 * owns rows [r*R, (r+1)*R), R = hidden / cluster_size, and pushes them into
 * the shared memory of every CTA of its cluster (its own included) with
 * st.async, 16 bytes at a time, completing on the receiver's mbarrier; a CTA
 * waits for the whole vector of a step before it sends its rows of the next
 * step.  Every received word is checked, one step late (off the exchange's
 * critical path).
 * Outputs: *ns_per_step, the mean over clusters of each cluster's exchange
 * time (globaltimer, its first CTA) divided by steps; *mismatches, the words
 * received with a wrong value (0 unless the exchange is broken).
 * Synchronous: runs on the current device's default stream and waits for it;
 * allocates and frees a few bytes of device memory.
 * Errors: INVALID_ARG for a size outside the above or a NULL output;
 * UNSUPPORTED when the device cannot launch clusters or cannot hold all the
 * clusters at once (cudaOccupancyMaxActiveClusters: on GB300, 9 sixteen-CTA
 * clusters of this probe); TIMEOUT when a wait ran out (1 s); CUDA, OOM.
 */
prnn_status_t prnn_probe_cluster_exchange(int hidden, int cluster_size, int clusters, int steps,
                                          double* ns_per_step, long long* mismatches);

/*
 * Host only (no GPU): the packing the persistent sparse kernel applies to
 * row-balanced weights, exposed so the layout can be checked bit for bit.
 * Rows are split over n_cta CTAs of rows_per_cta rows; each row over
 * threads_per_row (1, 2, 4, 8, 16 or 32) threads holding the same number of
 * entries each.  Output: packed[n_cta][rows_per_cta][ept/4][threads_per_row][4]
 * 32-bit words, word = fp16 value bits | column << 16, padding words have value
 * 0.  Within a row, entries are permuted among the row's threads so that in
 * every gather slot the 32 lanes of a warp use different shared-memory banks
 * (column mod 32) where possible (bank-aware layout, sparse persistent RNN
 * ablation table).  *ept receives the entries per thread (a multiple of 4),
 * *bank_cap the most lanes that had to share a bank.  capacity_words is the
 * size of `packed`; if it is too small the call returns PRNN_ERR_INVALID_ARG
 * with *ept set, so the caller can size the buffer and call again.
 */
prnn_status_t prnn_pack_sparse_host(int hidden, int k, int n_cta, int rows_per_cta,
                                    int threads_per_row, const uint16_t* vals,
                                    const uint16_t* cols, uint32_t* packed,
                                    size_t capacity_words, int* ept, int* bank_cap);

/*
 * Host only (no GPU): the packing the persistent sparse kernel actually uses
 * for bank-aware layers whose hidden size is a multiple of 128.  Each CTA
 * stages h_{t-1} in shared memory in an order of its own, chosen so that the
 * entries of every warp spread evenly over the 32 banks (so that the
 * bank-aware placement above can give each lane of a gather slot its own
 * bank); the index field of each packed word is then the staged position of
 * the column instead of the column itself.
 *   place [n_cta][hidden/4] receives one word per group of four columns g:
 *   byte j (0..3) is a bank b_j, and column 4g+j is staged at
 *       128*(g/32) + 32*j + b_j.
 *   Within each class (one block of 128 columns, one j) the 32 banks are a
 *   permutation of 0..31, so the staging stores of a warp are conflict-free.
 * *placed = 1 when the staged order is used; 0 for hidden not a multiple of
 * 128, where columns stay in order, packed equals prnn_pack_sparse_host's
 * output and place is not written.  place_capacity_words is the size of
 * place (n_cta*hidden/4 words needed when *placed = 1).  The other arguments,
 * the sizing protocol and the errors are those of prnn_pack_sparse_host;
 * placed must not be NULL.
 */
prnn_status_t prnn_pack_sparse_host_placed(int hidden, int k, int n_cta, int rows_per_cta,
                                           int threads_per_row, const uint16_t* vals,
                                           const uint16_t* cols, uint32_t* packed,
                                           size_t capacity_words, uint32_t* place,
                                           size_t place_capacity_words, int* ept,
                                           int* bank_cap, int* placed);

/*
 * Host only (no GPU): the weight image the tensor-core K-split kernel keeps
 * in shared memory (dense fp16 layers at wide batch), so that its index
 * handling can be checked without a device.  The layer's rows are split into
 * hidden/128 blocks of 128 rows; each block's K (the columns) into
 * cluster_size slices of whole 16-column steps, slice j starting at column
 * k0(j) = 16 * floor(j * (hidden/16) / cluster_size); each slice is stored as
 * nat = ceil(ceil((hidden/16) / cluster_size) / 4) atoms of 128 rows x 64
 * columns.  Element (row r, column c) of the block-row bk = r / 128, slice j
 * (k0(j) <= c < k0(j+1)), kc = c - k0(j), m = r mod 128 sits at
 *     ((bk * cluster_size + j) * nat + kc / 64) * 8192
 *       + m * 64 + (((kc mod 64) / 8) XOR (m mod 8)) * 8 + kc mod 8,
 * the 128-byte swizzle of the tensor cores' K-major shared-memory operand; every
 * other element is 0.
 *   wh16 [hidden][hidden]: fp16 bits of Wh, row-major (input, caller-owned).
 *   transpose != 0 builds the image of Wh^T (the reverse recurrence's).
 *   image [capacity_elems] uint16: output, caller-owned.
 *   *image_elems receives the elements needed.
 * hidden must be a multiple of 128 (at most 65536), 2 <= cluster_size <= 8
 * and hidden/16 >= cluster_size; otherwise, or when wh16 or image_elems is
 * NULL, PRNN_ERR_INVALID_ARG.  When image is NULL or too small the call sets
 * *image_elems and returns PRNN_ERR_INVALID_ARG, so the caller can size the
 * buffer and call again.
 */
prnn_status_t prnn_pack_dense_ksplit_host(int hidden, int cluster_size, const uint16_t* wh16,
                                          int transpose, uint16_t* image, size_t capacity_elems,
                                          size_t* image_elems);

/*
 * Forward pass that allocates no device memory.  The pages have no
 * counterpart to this call: it exists for callers that cannot call
 * cudaMalloc -- code in a latency-critical loop where cudaMalloc/cudaFree may
 * synchronize the whole device, or a process whose device memory is owned by
 * another allocator or capped by a fixed budget.
 *
 * Computes the same layer as prnn_forward with dense weights, straight from
 * the caller's buffers (no handle, no repacking): x [T][B][I] fp32, Wx [H][I]
 * and Wh [H][H] row-major in `wdtype`, bias [H] fp32, h0 [B][H] fp32 or NULL
 * (zeros), y [T][B][H] fp32 -- all DEVICE pointers; Wh, y and h0 16-byte
 * aligned.  It runs the per-step path: the fp32 CUDA-core projection, then T
 * step kernels reading Wh from memory each step.
 *
 * Scratch: the projection P [T][B][H] lives in a file-scope device array of
 * 4 Mi floats (16 MiB) that the library's CUDA module carries; every GPU on
 * which the library's kernels are loaded holds it until the process exits.
 * Limits: T*B*H <= 4194304 and 1 <= B <= 32, else PRNN_ERR_INVALID_ARG.
 * Every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress, a host-side query; nothing is cached, so a call after
 * cudaDeviceReset finds the array where the reloaded module put it).  The
 * first call on a device may load the library's module there: make it before
 * any stream capture.  Every call shares the one array and it keeps the last
 * call's contents (P is fully rewritten before use, nothing needs zeroing):
 * calls whose work overlaps on the GPU -- on different streams, or from
 * different threads -- race on it and must be serialized by the caller.
 * Asynchronous on `stream`; T == 0 or B == 0 is a no-op.
 */
prnn_status_t prnn_forward_dense_noalloc(int T, int B, int H, int I, prnn_dtype_t wdtype,
                                         const float* x, const void* Wx, const void* Wh,
                                         const float* bias, const float* h0, float* y,
                                         void* stream);

/* ---- stacked layers ---------------------------------------------------
 *
 * A stack of L dense ReLU RNN layers, each with `hidden` units: layer 0 reads
 * x, layer l > 0 reads layer l-1's output sequence:
 *
 *     h^l_t = ReLU(b_l + Wx_l h^{l-1}_t + Wh_l h^l_{t-1}),   h^{-1}_t = x_t,
 *
 * the multi-layer network that "Optimizing Performance of Recurrent Neural
 * Networks on GPUs" (Abstract) optimises as a whole, with the on-chip weights
 * of the persistent-rnn page ("What This Project Does").
 *
 * PRNN_STACK_WAVEFRONT runs the whole stack in ONE persistent cooperative
 * launch: the SMs are split into L slices, slice l keeps [Wx_l | Wh_l] on
 * chip and computes step t of layer l as soon as layer l-1 has published its
 * step t, so the stack takes about T + L - 1 step times instead of L * T.
 * All L layers' weights must fit on chip at once (about
 * L * hidden * (hidden + input) * weight-size bytes over the SMs' shared
 * memory), else PRNN_ERR_UNSUPPORTED from prnn_stack_create.
 * PRNN_STACK_LAYERWISE runs the layers one after another, each as
 * prnn_forward does (batched input projection, then its persistent
 * recurrence); it is the comparison point of the wavefront.
 */
typedef struct prnn_stack* prnn_stack_t;

typedef enum {
  PRNN_STACK_WAVEFRONT = 0,
  PRNN_STACK_LAYERWISE = 1
} prnn_stack_algo_t;

/*
 * Create a stack: 1 <= layers <= 8; hidden, input >= 1 and, for the
 * wavefront, multiples of 4; 1 <= max_batch <= 32; weights fp32 or fp16.
 * Plans the launch for the current device.  Errors: INVALID_ARG (sizes),
 * UNSUPPORTED (weights cannot all be on chip, or no usable GPU), OOM.
 */
prnn_status_t prnn_stack_create(prnn_stack_t* out, int layers, int hidden, int input,
                                int max_batch, prnn_dtype_t wdtype, prnn_stack_algo_t algo);

/*
 * Set layer `layer` (0 .. layers-1): Wx [hidden][I_l] with I_0 = input and
 * I_l = hidden for l > 0, Wh [hidden][hidden], both row-major in the stack's
 * dtype; bias [hidden] fp32.  Device or host pointers; the library copies and
 * repacks them, synchronizing `stream` first, so the caller may free them on
 * return.
 */
prnn_status_t prnn_stack_set_layer(prnn_stack_t s, int layer, const void* Wx, const void* Wh,
                                   const float* bias, void* stream);

/*
 * Forward the stack over T steps for B <= max_batch sequences: x [T][B][input]
 * fp32; h0 [layers][B][hidden] fp32 or NULL (zeros); y [layers][T][B][hidden]
 * fp32 receives every layer's output sequence (the top layer is
 * y + (layers-1)*T*B*hidden).  Device pointers, 16-byte aligned; y must not
 * overlap x or h0.  Asynchronous on `stream`; T == 0 or B == 0 is a no-op.
 * Errors: NOT_READY until every layer is set; INVALID_ARG; a wait that runs
 * out inside the launch makes the stack report PRNN_ERR_TIMEOUT from then on.
 */
prnn_status_t prnn_stack_forward(prnn_stack_t s, int T, int B, const float* x, const float* h0,
                                 float* y, void* stream);

/* Synchronize `stream`, then report the stack's device status (sticky TIMEOUT). */
prnn_status_t prnn_stack_get_status(prnn_stack_t s, void* stream);

/*
 * Options: PRNN_OPT_WAIT_TIMEOUT_US, PRNN_OPT_POLL_DELAY_NS, PRNN_OPT_POLL_BACKOFF_NS,
 * PRNN_OPT_TIMING (events around the last
 * forward, read with prnn_stack_get_timing), PRNN_OPT_DEBUG_DROP_CTA /
 * PRNN_OPT_DEBUG_DROP_STEP (the CTA index counts over all slices; wavefront
 * only), PRNN_OPT_CTA_GROUPS (wavefront: force the batch groups per slice;
 * re-plans and clears the layers, which must be set again).  Others:
 * INVALID_ARG.
 */
prnn_status_t prnn_stack_set_option(prnn_stack_t s, prnn_option_t opt, long long value);

/* Milliseconds of the last timed forward (PRNN_ERR_NOT_READY if none). */
prnn_status_t prnn_stack_get_timing(prnn_stack_t s, float* ms);

typedef struct {
  int layers, hidden, input, max_batch, wdtype, algo, layers_set;
  int n_cta_per_layer;     /* wavefront: CTAs of one layer slice                     */
  int rows_per_cta, threads_per_cta, cta_groups, batch_per_pass, chunks_per_thread;
  long long smem_bytes;    /* dynamic shared memory per CTA                          */
  long long onchip_weight_bytes;  /* all slices, all groups                          */
} prnn_stack_info_t;

prnn_status_t prnn_stack_get_info(prnn_stack_t s, prnn_stack_info_t* info);

/* Free everything the stack owns.  NULL is accepted. */
prnn_status_t prnn_stack_destroy(prnn_stack_t s);

#ifdef __cplusplus
}
#endif

#endif /* PRNN_H */
