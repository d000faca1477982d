// api.cu -- the C ABI of libprnn.so: handle, validation, planning, weight
// packing, forward orchestration, status and timing.  Declarations and the
// contract of every call are in include/prnn.h.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "host_util.h"
#include "prnn.h"
#include "prnn_internal.h"

using namespace prnn;

namespace {

constexpr int kMaxBatch = 32;
constexpr int kSparseMaxThreads = 512;

}  // namespace

struct prnn_handle {
  int H = 0, I = 0, maxB = 0;
  prnn_dtype_t wdtype = PRNN_F32;
  prnn_algo_t algo = PRNN_ALGO_PERSISTENT;
  int device = 0, sm_count = 0;
  size_t smem_optin = 0;
  bool weights_set = false, sparse = false;
  int k = 0;
  // persistent plan
  int n_cta = 0, R = 0, nthreads = 0, cpt = 0, tpr = 0, kp = 0, ept = 0, pack_cap = 0;
  int G = 1, cpg = 0, groups_opt = 0, dense_bw = 4;
  // dense fp16 for wide batches (CTA groups of >= 8 batch columns): its own
  // plan, packed weights and a zero h0 for forwards without one
  int wide_opt = 1;
  bool wide = false;
  int w_R = 0, w_S = 0, w_depth = 1;
  size_t w_smem = 0;
  void* Wpk_wide = nullptr;
  float* zeros = nullptr;
  // dense fp16 for wide batches on the tensor cores, K split in clusters:
  // its plan and weight image
  int ks_opt = 1;
  int sks_opt = 1;    // sparse layers on the K-split kernel (their densified matrix)
  size_t ks_nnz = 0;  // sparse: stored entries behind the K-split image
  bool ks = false;
  int ks_cs = 0, ks_nat = 0;
  bool ks_stream = false;  // Wh streamed through rings (it does not fit on chip), B <= 16
  void* Wimg_ks = nullptr;
  void* WimgT_ks = nullptr;  // the same for Wh^T (the backward's reverse recurrence)
  // tensor-core dense recurrence (wide batch): its own plan and weight image
  int rtc_opt = 1;  // the tensor-core recurrence is opt-in (slower than the CUDA cores so far)
  bool rtc = false;
  int t_n_cta = 0, t_R = 0, t_G = 1, t_cpg = 0, t_N = 0, t_ring = 0;
  void* Wimg = nullptr;
  int wide_loads = 1, bank_aware = 1, staged_order = 2;
  int regw_opt = 1;  // sparse: register-weight build of the kernel where its plan fits
  int depth_opt = 1; // sparse: staging depth matched to the plan (0: always 12)
  size_t onchip_bytes = 0, smem_at_max = 0;
  bool tc_proj = false;
  int Kp = 0;  // I rounded up to 64 (tcgen05 projection)
  // device buffers owned by the handle
  void* Wx = nullptr;        // [H][I] in wdtype
  __half_raw* Wx16 = nullptr;  // [H][Kp] fp16, zero padded (tcgen05 projection)
  float* bias = nullptr;
  void* Wpk = nullptr;       // persistent packed recurrent weights
  void* Wpk_T = nullptr;     // the same packing of Wh^T (backward pass, dense)
  uint32_t* place = nullptr;    // sparse: per-CTA staging order of h ([cpg][H/4]) or null
  uint32_t* place_T = nullptr;  // the same for the Wh^T plan of the backward pass
  void* Wh_nat = nullptr;    // Wh row-major [H][H] in wdtype (backward pass, dense)
  // sparse backward: plan of the persistent kernel for Wh^T (packed in
  // Wpk_T), the forward's padded column lists and each padded entry's index
  // in the caller's order, Wh^T padded to kT entries per row, and the
  // transposed-delta workspace
  bool bwd_ok = false;
  size_t n_caller = 0;            // entries the caller passed (H*k, or nnz)
  int b_n_cta = 0, b_R = 0, b_G = 1, b_cpg = 0, b_nthreads = 0, b_tpr = 0, b_ept = 0, kT = 0;
  uint16_t* cols_pad = nullptr;   // [H][k]
  int32_t* caller_pos = nullptr;  // [H][k], -1 for padding
  uint16_t* valsT = nullptr;      // [H][kT] fp16 bits
  uint16_t* colsT = nullptr;      // [H][kT]
  float* tws = nullptr;           // masked dy, then transposes or a dense dWh
  size_t tws_cap = 0;
  // tensor-core gradient products (fp16 handles): Wx^T in bf16 [I][Hp]
  // (Hp = H rounded up to 64), and bf16 staging of delta, h and x
  uint16_t* WxT16 = nullptr;
  uint16_t* gws16 = nullptr;
  size_t gws16_cap = 0;
  void* Wstep = nullptr;     // per-step layout of the recurrent weights
  float* P = nullptr;
  size_t P_cap = 0;
  // device copies of x, h0 and y for prnn_forward_host
  float* hx = nullptr;
  float* hh0 = nullptr;
  float* hy = nullptr;
  size_t hx_cap = 0, hh0_cap = 0, hy_cap = 0;
  __half_raw* x16 = nullptr;
  size_t x16_cap = 0;
  int* status = nullptr;     // device int[4]
  unsigned* bar = nullptr;   // grid-barrier counter
  // caller's device buffer for the sparse kernel's phase trace (or null)
  uint32_t* trace = nullptr;
  size_t trace_words = 0;
  // options
  long long timeout_us = 500000;
  int poll_delay_ns = -1, clock_khz = 0;  // -1: the kernel family's default
  int backoff_ns = kBackoffNs;
  int sync_mode = 0, drop_cta = -1, drop_step = -1, timing = 0, proj_mode = 0;
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  bool ev_valid = false;
  bool last_backward = false;  // which call the timing events belong to
  bool sticky_timeout = false;
  // per-step graph cache
  cudaStream_t cap_stream = nullptr;
  cudaGraphExec_t gexec = nullptr;
  int g_T = -1, g_B = -1;
  const void *g_h0 = nullptr, *g_y = nullptr, *g_P = nullptr, *g_W = nullptr;
};

namespace {



// ---- planning ----------------------------------------------------------
struct DensePlan {
  int G, cpg, R, n_cta, nthreads, cpt, bw;
  size_t smem;
  bool ok;
};

// Candidate CTA-group counts, largest first: G groups of SMs/G CTAs, each
// group owning ceil(B/G) batch columns and a full copy of Wh.
int max_groups(const prnn_handle* h) {
  if (h->groups_opt > 0) return std::min(h->groups_opt, h->maxB);
  return std::min(h->maxB, 8);
}

DensePlan plan_dense_g(const prnn_handle* h, int G) {
  DensePlan p{};
  const int H = h->H;
  const bool f16 = h->wdtype == PRNN_F16;
  p.G = G;
  p.cpg = h->sm_count / G;
  p.ok = false;
  if (p.cpg < 1 || H % 4 != 0) return p;
  p.R = (H + p.cpg - 1) / p.cpg;
  p.cpg = (H + p.R - 1) / p.R;
  p.n_cta = p.G * p.cpg;
  const int rmax = recur_dense_rmax(p.R);
  if (rmax == 0) return p;
  const int nchunks = H / 4;
  // widest batch pass first; within it the most threads; skip variants the
  // register model says would spill
  for (int bw = recur_dense_bw((h->maxB + G - 1) / G); bw >= 1; bw /= 2) {
    for (int cap : {512, 256}) {
      const int cpt = (nchunks + cap - 1) / cap;
      if (cpt > 4) continue;
      const int nt = std::max(32, round_up((nchunks + cpt - 1) / cpt, 32));
      if (nt > dense_launch_bound(f16, rmax, bw, cpt)) continue;
      if (dense_reg_estimate(f16, rmax, bw, cpt) > 240) continue;
      const size_t sm = recur_dense_smem(p.R, cpt, nt, f16, bw);
      if (sm > h->smem_optin) continue;
      p.bw = bw;
      p.cpt = cpt;
      p.nthreads = nt;
      p.smem = sm;
      p.ok = true;
      return p;
    }
  }
  return p;
}

// Tensor-core dense plan: G groups (batch columns Bl = ceil(maxB/G) <= 32),
// R = ceil(H/cpg) <= 32 rows per CTA (N = R rounded up to 16), weights image
// plus the A ring within shared memory; among the fits, the least estimated
// step time: exchange ~1.1 us + ~17 ns per KiB of h each CTA pulls + the
// MMAs (M = 128 rows of A, N, K = H at ~14.8 TFLOP/s per SM).
struct TcPlan {
  int G, cpg, R, N, n_cta, nring;
  size_t smem;
  bool ok;
};
TcPlan plan_dense_tc(const prnn_handle* h) {
  TcPlan best{};
  double best_ns = 1e30;
  if (h->wdtype != PRNN_F16 || h->H % 64 != 0) return best;
  for (int G = 1; G <= std::min(h->maxB, 8); G *= 2) {
    const int bl = (h->maxB + G - 1) / G;
    if (bl > 32) continue;
    int cpg = h->sm_count / G;
    if (cpg < 1) continue;
    const int R = (h->H + cpg - 1) / cpg;
    cpg = (h->H + R - 1) / R;
    const int N = round_up(R, 16);
    if (N > 32) continue;
    const int nring = recur_dense_tc_ring(h->H, N, h->smem_optin);
    if (nring < 2) continue;
    const size_t sm = recur_dense_tc_smem(h->H, N, nring);
    const double ns = 1100.0 + 17.0 * bl * h->H * 4 / 1024.0 + 2.0 * 128 * N * h->H / 14800.0;
    if (ns < best_ns) {
      best_ns = ns;
      best = TcPlan{G, cpg, R, N, G * cpg, nring, sm, true};
    }
  }
  return best;
}

DensePlan plan_dense(const prnn_handle* h) {
  for (int G = max_groups(h); G >= 1; --G) {
    if (h->groups_opt == 0 && G > 1 && (G & (G - 1)) != 0) continue;
    DensePlan p = plan_dense_g(h, G);
    if (h->groups_opt > 0) return p;
    // automatic: at most 16 rows per CTA (more rows lengthen every thread's
    // per-step chain more than the smaller exchange saves)
    if (p.ok && (p.R <= 16 || G == 1)) return p;
  }
  return DensePlan{};
}

struct SparsePlan {
  int G, cpg, R, n_cta, tpr, kp, ept, nthreads;
  bool ok;
};

SparsePlan plan_sparse_g(const prnn_handle* h, int k, int G) {
  SparsePlan p{};
  const int H = h->H;
  p.G = G;
  p.cpg = h->sm_count / G;
  if (p.cpg < 1 || H % 4 != 0) return p;
  p.R = (H + p.cpg - 1) / p.cpg;
  p.cpg = (H + p.R - 1) / p.R;
  p.n_cta = p.G * p.cpg;
  // threads per row: the widest split whose padding stays under ~15 % and
  // whose R * tpr threads fit one CTA; else the least padding that fits.
  int best = -1;
  double best_waste = 1e30;
  for (int t = 32; t >= 1; t >>= 1) {
    if (p.R * t > kSparseMaxThreads) continue;
    const int kp = round_up(k, 4 * t);
    const double waste = (double)kp / k;
    if (waste <= 1.15) {
      best = t;
      break;
    }
    if (waste < best_waste) {
      best_waste = waste;
      best = t;
    }
  }
  if (best <= 0) return p;
  p.tpr = best;
  p.ept = ((k + best - 1) / best + 3) / 4 * 4;
  p.kp = p.ept * best;
  // enough threads to keep one staging round of the group's columns in flight
  const int bl = std::min(4, (h->maxB + G - 1) / G);
  const int stage_threads = round_up((H * std::max(bl, 1) / 4 + 11) / 12, 32);
  p.nthreads = std::min(kSparseMaxThreads,
                        std::max({256, round_up(p.R * best, 32), stage_threads}));
  // at least a one-column batch pass must fit
  p.ok = recur_sparse_smem(H, p.R, p.ept, p.tpr, 1, false) <= h->smem_optin;
  return p;
}

// Estimated ns per step of a sparse plan (model fitted to GB300 measurements
// of this kernel): the step exchange costs ~1.0 us plus ~17 ns per KiB of
// h that each CTA pulls from L2; the gather-multiply costs ~1.9 shared-memory
// wavefronts per gather slot (bank-aware packing) plus the wavefronts of the
// weights kept in smem rather than registers, and each thread's chain of ept
// dependent updates.
double sparse_step_ns(const prnn_handle* h, const SparsePlan& p) {
  const int bl = (h->maxB + p.G - 1) / p.G;
  const double kib = (double)bl * h->H * 4.0 / 1024.0;
  const double warps = (double)((p.R * p.tpr + 31) / 32);
  const double gather = warps * p.ept * bl * 1.9;
  const double wsmem = warps * std::max(0, p.ept / 4 - 4) * 4.0;
  const double chain = p.ept * 4.0 * bl + 60.0;
  const double ghz = 1.9;
  return 1000.0 + 17.0 * kib + (gather + wsmem) / ghz + chain / ghz;
}

// Feasible plans, fastest (by the model) first; a forced group count gives
// exactly that plan.
std::vector<SparsePlan> plan_sparse(const prnn_handle* h, int k) {
  std::vector<std::pair<double, SparsePlan>> cand;
  for (int G = max_groups(h); G >= 1; --G) {
    if (h->groups_opt == 0 && G > 1 && (G & (G - 1)) != 0) continue;
    SparsePlan p = plan_sparse_g(h, k, G);
    if (h->groups_opt > 0) {
      if (p.ok) cand.push_back({0.0, p});
      break;
    }
    if (p.ok) cand.push_back({sparse_step_ns(h, p), p});
  }
  std::stable_sort(cand.begin(), cand.end(),
                   [](const std::pair<double, SparsePlan>& a, const std::pair<double, SparsePlan>& b) {
                     return a.first < b.first;
                   });
  std::vector<SparsePlan> out;
  for (auto& c : cand) out.push_back(c.second);
  return out;
}

// Batch group and staging buffers of the sparse kernel for a given B, for
// the plan (G, R, ept, tpr): the forward's by default.
bool sparse_batch_plan(const prnn_handle* h, int B, int* bgroup, bool* dbuf, size_t* smem,
                       bool transposed = false) {
  const int G = transposed ? h->b_G : h->G, R = transposed ? h->b_R : h->R;
  const int ept = transposed ? h->b_ept : h->ept, tpr = transposed ? h->b_tpr : h->tpr;
  const int bl = (B + G - 1) / G;  // batch columns of one CTA group
  int want = 1;
  while (want < bl && want < 32) want *= 2;
  for (int bg = want; bg >= 1; bg /= 2) {
    for (int db = 1; db >= 0; --db) {
      const size_t s = recur_sparse_smem(h->H, R, ept, tpr, bg, db == 1);
      if (s <= h->smem_optin) {
        *bgroup = bg;
        *dbuf = db == 1;
        *smem = s;
        return true;
      }
    }
  }
  return false;
}

void invalidate_graph(prnn_handle* h) {
  if (h->gexec) cudaGraphExecDestroy(h->gexec);
  h->gexec = nullptr;
  h->g_T = h->g_B = -1;
}

cudaError_t ensure_P(prnn_handle* h, size_t n) {
  if (n <= h->P_cap) return cudaSuccess;
  invalidate_graph(h);
  free_dev(h->P);
  cudaError_t e = cudaMalloc((void**)&h->P, n * sizeof(float));
  if (e != cudaSuccess) {
    h->P_cap = 0;
    return e;
  }
  h->P_cap = n;
  return cudaSuccess;
}

// Grow a float device buffer to at least n elements (contents not kept).
cudaError_t ensure_f32(float** p, size_t* cap, size_t n) {
  if (n <= *cap) return cudaSuccess;
  free_dev(*p);
  *cap = 0;
  cudaError_t e = cudaMalloc((void**)p, n * sizeof(float));
  if (e == cudaSuccess) *cap = n;
  return e;
}

// prnn_forward_host: the projection's staging kernel reads x from the host
// buffer itself (no copy) when the layer uses the tensor-core projection.
constexpr bool kHostXDirect = true;

// The device address of page-locked host memory, or nullptr for anything
// else (pageable or device memory, or a pointer CUDA does not know).
const void* mapped_host(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost) return nullptr;
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, const_cast<void*>(p), 0) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return d;
}

cudaError_t ensure_x16(prnn_handle* h, size_t n) {
  if (n <= h->x16_cap) return cudaSuccess;
  free_dev(h->x16);
  cudaError_t e = cudaMalloc((void**)&h->x16, n * sizeof(__half_raw));
  if (e != cudaSuccess) {
    h->x16_cap = 0;
    return e;
  }
  h->x16_cap = n;
  return cudaSuccess;
}

// IEEE binary16 bits -> float (exact), and float -> bfloat16 bits rounded to
// nearest even (finite inputs).
float half_bits_to_float(uint16_t h) {
  const uint32_t sign = (uint32_t)(h >> 15) << 31;
  const int exp = (h >> 10) & 0x1f;
  const uint32_t man = h & 0x3ff;
  float v;
  if (exp == 0) {
    v = (float)man * (1.0f / 16777216.0f);  // subnormal: man * 2^-24
  } else if (exp == 31) {
    v = man ? __builtin_nanf("") : __builtin_inff();
  } else {
    uint32_t bits = ((uint32_t)(exp - 15 + 127) << 23) | (man << 13);
    std::memcpy(&v, &bits, 4);
  }
  uint32_t b;
  std::memcpy(&b, &v, 4);
  b |= sign;
  std::memcpy(&v, &b, 4);
  return v;
}
uint16_t float_to_bf16_bits(float f) {
  uint32_t b;
  std::memcpy(&b, &f, 4);
  b += 0x7fffu + ((b >> 16) & 1u);
  return (uint16_t)(b >> 16);
}

// Wx in the handle's dtype ([H][I]) plus, for fp16, a [H][Kp] zero-padded
// copy for the tensor-core projection and Wx^T in bf16 [I][Hp] for the
// tensor-core input gradient.  Host vectors in, device buffers out.
prnn_status_t stage_wx_bias(prnn_handle* h, const void* Wx, const float* bias,
                            void** dWx, __half_raw** dWx16, float** dbias) {
  const size_t esz = h->wdtype == PRNN_F16 ? 2 : 4;
  std::vector<unsigned char> wx((size_t)h->H * h->I * esz);
  std::vector<float> b((size_t)h->H);
  PRNN_TRY(to_host(wx.data(), Wx, wx.size()));
  PRNN_TRY(to_host(b.data(), bias, b.size() * sizeof(float)));
  PRNN_TRY(upload(dWx, wx.data(), wx.size()));
  PRNN_TRY(upload(dbias, b.data(), b.size() * sizeof(float)));
  if (h->wdtype == PRNN_F16) {
    std::vector<uint16_t> w16((size_t)h->H * h->Kp, 0);
    const uint16_t* src = reinterpret_cast<const uint16_t*>(wx.data());
    for (int r = 0; r < h->H; ++r)
      std::memcpy(&w16[(size_t)r * h->Kp], src + (size_t)r * h->I, (size_t)h->I * 2);
    PRNN_TRY(upload(dWx16, w16.data(), w16.size() * 2));
    const int Hp = round_up(h->H, 64);
    std::vector<uint16_t> wt((size_t)h->I * Hp, 0);
    for (int r = 0; r < h->H; ++r)
      for (int c = 0; c < h->I; ++c)
        wt[(size_t)c * Hp + r] = float_to_bf16_bits(half_bits_to_float(src[(size_t)r * h->I + c]));
    PRNN_TRY(upload(&h->WxT16, wt.data(), wt.size() * 2));
  }
  return PRNN_OK;
}

void free_weights(prnn_handle* h) {
  invalidate_graph(h);
  free_dev(h->Wx);
  free_dev(h->Wx16);
  free_dev(h->bias);
  free_dev(h->Wpk);
  free_dev(h->Wpk_T);
  free_dev(h->place);
  free_dev(h->place_T);
  free_dev(h->Wh_nat);
  free_dev(h->Wimg);
  h->rtc = false;
  free_dev(h->Wpk_wide);
  free_dev(h->Wimg_ks);
  free_dev(h->WimgT_ks);
  h->ks = false;
  free_dev(h->zeros);
  h->wide = false;
  free_dev(h->cols_pad);
  free_dev(h->caller_pos);
  free_dev(h->valsT);
  free_dev(h->colsT);
  free_dev(h->WxT16);
  h->bwd_ok = false;
  free_dev(h->Wstep);
  h->weights_set = false;
}

RecurCommon common_args(const prnn_handle* h, int T, int B, const float* h0, float* y) {
  RecurCommon c{};
  c.T = T;
  c.B = B;
  c.H = h->H;
  c.n_cta = h->n_cta;
  c.R = h->R;
  c.G = h->G;
  c.cpg = h->cpg;
  c.nthreads = h->nthreads;
  c.P = h->P;
  c.h0 = h0;
  c.y = y;
  c.status = h->status;
  c.timeout_ns = h->timeout_us * 1000LL;
  const int delay_ns = h->poll_delay_ns >= 0 ? h->poll_delay_ns
                                            : (h->sparse ? sparse_delay_ns(h->H) : kDenseDelayNs);
  c.poll_delay = (int)((long long)delay_ns * h->clock_khz / 1000000LL);
  c.poll_backoff = (int)((long long)h->backoff_ns * h->clock_khz / 1000000LL);
  c.sync_mode = h->sync_mode;
  c.bar = h->bar;
  c.drop_cta = h->drop_cta;
  c.drop_step = h->drop_step;
  return c;
}

}  // namespace

// Plan and pack [H][k] row-padded sparse rows for the persistent kernel:
// the first plan (fastest by the model) whose packing fits shared memory.
// place: nullptr for column order, else it receives each CTA's staging order
// (left empty where the layer cannot use one).
static bool plan_and_pack_order(prnn_t h, int k, const std::vector<uint16_t>& hv,
                                const std::vector<uint16_t>& hc, SparsePlan* plan,
                                std::vector<uint32_t>* pk, PackStats* pst,
                                std::vector<uint32_t>* place) {
  const int H = h->H;
  for (const SparsePlan& cand : plan_sparse(h, k)) {
    // largest entries-per-thread whose weights plus one h column fit in smem
    const size_t hs1 = (size_t)H * sizeof(float);
    if (hs1 >= h->smem_optin) continue;
    const int max_ept = (int)(((h->smem_optin - hs1) / ((size_t)cand.R * cand.tpr * 4)) / 4 * 4);
    *plan = cand;
    plan->ept = pack_sparse_rows(H, k, plan->R, plan->cpg, plan->tpr, hv.data(), hc.data(), *pk,
                                 pst, max_ept, h->bank_aware != 0, place);
    if (plan->ept > 0) {
      plan->kp = plan->ept * plan->tpr;
      return true;
    }
  }
  return false;
}

// The staging order of a packing: PRNN_OPT_STAGED_ORDER 0 column order, 1 each
// CTA's bank-balancing order, 2 (default) the order this rule picks from
// both packings: with batch passes of at least 4 columns, the staged order
// when it needs fewer padded entries per row than column order, or when rows
// hold at least 256 entries and it needs at most 12 % more.  Fitted to
// measurements of both orders at every sparse point of the H x B x density
// sweep and the named layers: the staged order's scattered staging stores
// cost more than its conflict-free gathers save unless the gathers dominate
// the step (wide batch, many entries); with one or two columns a pass it
// loses even where it packs tighter (H=5760 5 %, B=4: 4.10 against 3.40 us
// per step).
static bool plan_and_pack(prnn_t h, int k, const std::vector<uint16_t>& hv,
                          const std::vector<uint16_t>& hc, SparsePlan* plan,
                          std::vector<uint32_t>* pk, PackStats* pst,
                          std::vector<uint32_t>* place) {
  place->clear();
  if (h->staged_order != 2)
    return plan_and_pack_order(h, k, hv, hc, plan, pk, pst, h->staged_order ? place : nullptr);
  const bool okc = plan_and_pack_order(h, k, hv, hc, plan, pk, pst, nullptr);
  if (!h->bank_aware || !staging_placement_supported(h->H)) return okc;
  SparsePlan ps{};
  std::vector<uint32_t> pks, pls;
  PackStats sts;
  if (!plan_and_pack_order(h, k, hv, hc, &ps, &pks, &sts, &pls) || pls.empty()) return okc;
  bool staged = !okc;
  if (okc) {
    const int cols = (h->maxB + plan->G - 1) / plan->G;  // batch columns of a group
    staged = cols >= 4 && (ps.kp < plan->kp || (plan->kp >= 256 && (long long)ps.kp * 100 <=
                                                                        (long long)plan->kp * 112));
  }
  if (staged) {
    *plan = ps;
    pk->swap(pks);
    *pst = sts;
    place->swap(pls);
  }
  return true;
}

// Plan, pack and upload row-padded sparse weights (hv/hc [H][k], each row
// sorted by column, padding entries valued 0), and build the packed Wh^T and
// the index maps the backward pass uses.  Shared by the row-balanced and the
// compressed-row entry points.
// caller_pos[r*k + j] is the index of padded entry (r, j) in the caller's
// value array, -1 for padding.
// The K-split kernel's weight images from Wh as fp16 [H][H] (row-major), if
// the device can hold the plan: for Wh and for Wh^T (the backward's reverse
// recurrence), per CTA (cluster-major, then K slice j) nat atoms of 128 rows x
// 64 columns, 16-byte chunk q of row m at q ^ (m & 7) (the 128-byte swizzle of
// the K-major MMA operand).  Sets h->ks.
// The A operand's image of the K-split kernel: for row block bk and K slice j
// of cs, nat atoms of 128 rows x 64 fp16 (K-major, 128 bytes a row), each
// row's 16-byte chunks in the 128-byte swizzle (chunk q of row m at
// q ^ (m mod 8)); zeros past the slice's width.  The transposed image (rows
// of Wh^T) serves the reverse recurrence.  img must hold
// (H / 128) * cs * nat * 8192 elements and be zero-filled.
static void build_ksplit_image(int H, int cs, int nat, const uint16_t* w16, bool transpose,
                               uint16_t* img) {
  const int nblk = H / 128;
  for (int bk = 0; bk < nblk; ++bk)
    for (int j = 0; j < cs; ++j) {
      const int k0 = ksplit_k0(H, cs, j), kl = ksplit_kl(H, cs, j);
      for (int at = 0; at < nat; ++at)
        for (int m = 0; m < 128; ++m)
          for (int q = 0; q < 8; ++q)
            for (int e = 0; e < 8; ++e) {
              const int kcol = at * 64 + q * 8 + e;  // column within the slice
              if (kcol >= kl) continue;
              const size_t atom = ((size_t)bk * cs + j) * nat + at;
              const size_t r = (size_t)(bk * 128 + m), cc = (size_t)(k0 + kcol);
              img[atom * 128 * 64 + (size_t)m * 64 + ((q ^ (m & 7)) * 8) + e] =
                  transpose ? w16[cc * H + r] : w16[r * H + cc];
            }
    }
}

static prnn_status_t install_ksplit(prnn_t h, const uint16_t* w16) {
  const int H = h->H;
  bool stream = false;
  const int kcs = recur_dense_ksplit_plan(H, &stream);
  if (kcs == 0) return PRNN_OK;
  const int nblk = H / 128, knat = ksplit_nat(H, kcs);
  std::vector<uint16_t> img((size_t)nblk * kcs * knat * 128 * 64);
  for (int tr = 0; tr < 2; ++tr) {  // Wh, then Wh^T
    std::fill(img.begin(), img.end(), (uint16_t)0);
    build_ksplit_image(H, kcs, knat, w16, tr != 0, img.data());
    PRNN_TRY(upload(tr ? &h->WimgT_ks : &h->Wimg_ks, img.data(), img.size() * 2));
  }
  if (!h->zeros) {
    std::vector<float> z((size_t)h->maxB * H, 0.f);
    PRNN_TRY(upload(&h->zeros, z.data(), z.size() * sizeof(float)));
  }
  h->ks = true;
  h->ks_cs = kcs;
  h->ks_nat = knat;
  h->ks_stream = stream;
  return PRNN_OK;
}

static prnn_status_t install_sparse(prnn_t h, const void* Wx, const float* bias,
                                    std::vector<uint16_t>& hv, std::vector<uint16_t>& hc, int k,
                                    const std::vector<int32_t>& caller_pos) {
  const int H = h->H;
  SparsePlan plan{};
  std::vector<uint32_t> pk, place;
  PackStats pst;
  if (h->algo == PRNN_ALGO_PERSISTENT && !plan_and_pack(h, k, hv, hc, &plan, &pk, &pst, &place))
    return PRNN_ERR_UNSUPPORTED;
  // Wh^T: row c lists the stored (r, value) of column c in ascending r,
  // padded to the longest such list with zero-valued absent columns
  std::vector<std::vector<std::pair<uint16_t, uint16_t>>> tr((size_t)H);
  for (int r = 0; r < H; ++r)
    for (int j = 0; j < k; ++j)
      if (caller_pos[(size_t)r * k + j] >= 0)
        tr[hc[(size_t)r * k + j]].push_back({(uint16_t)r, hv[(size_t)r * k + j]});
  int kT = 1;
  for (const auto& v : tr) kT = std::max(kT, (int)v.size());
  std::vector<uint16_t> hvT((size_t)H * kT, 0), hcT((size_t)H * kT, 0);
  {
    std::vector<int> in_row((size_t)H, -1);
    for (int c = 0; c < H; ++c) {
      auto& v = tr[c];
      for (const auto& e : v) in_row[e.first] = c;
      for (int r = 0; r < H && (int)v.size() < kT; ++r)
        if (in_row[r] != c) v.push_back({(uint16_t)r, 0});
      std::sort(v.begin(), v.end(),
                [](const std::pair<uint16_t, uint16_t>& a, const std::pair<uint16_t, uint16_t>& b) {
                  return a.first < b.first;
                });
      for (int j = 0; j < kT; ++j) {
        hcT[(size_t)c * kT + j] = v[j].first;
        hvT[(size_t)c * kT + j] = v[j].second;
      }
    }
  }
  SparsePlan tplan{};
  std::vector<uint32_t> pkT, placeT;
  PackStats pstT;
  const bool bwd = h->algo == PRNN_ALGO_PERSISTENT &&
                   plan_and_pack(h, kT, hvT, hcT, &tplan, &pkT, &pstT, &placeT);
  free_weights(h);
  prnn_status_t st = stage_wx_bias(h, Wx, bias, &h->Wx, &h->Wx16, &h->bias);
  if (st != PRNN_OK) return st;
  auto entry = [&](int r, int j) -> uint32_t {
    return (uint32_t)hv[(size_t)r * k + j] | ((uint32_t)hc[(size_t)r * k + j] << 16);
  };
  if (h->algo == PRNN_ALGO_PERSISTENT) {
    PRNN_TRY(upload(&h->Wpk, pk.data(), pk.size() * 4));
    if (!place.empty()) PRNN_TRY(upload(&h->place, place.data(), place.size() * 4));
    h->n_cta = plan.n_cta;
    h->R = plan.R;
    h->G = plan.G;
    h->cpg = plan.cpg;
    h->nthreads = plan.nthreads;
    h->tpr = plan.tpr;
    h->kp = plan.kp;
    h->ept = plan.ept;
    h->pack_cap = pst.cap;
    h->onchip_bytes = (size_t)plan.n_cta * plan.R * plan.kp * 4;  // all groups' copies
    int bg = 4;
    bool db = false;
    size_t sm = 0;
    sparse_batch_plan(h, h->maxB, &bg, &db, &sm);
    h->smem_at_max = sm;
    if (bwd) {
      PRNN_TRY(upload(&h->Wpk_T, pkT.data(), pkT.size() * 4));
      if (!placeT.empty()) PRNN_TRY(upload(&h->place_T, placeT.data(), placeT.size() * 4));
      PRNN_TRY(upload(&h->cols_pad, hc.data(), hc.size() * 2));
      PRNN_TRY(upload(&h->caller_pos, caller_pos.data(), caller_pos.size() * 4));
      PRNN_TRY(upload(&h->valsT, hvT.data(), hvT.size() * 2));
      PRNN_TRY(upload(&h->colsT, hcT.data(), hcT.size() * 2));
      h->b_n_cta = tplan.n_cta;
      h->b_R = tplan.R;
      h->b_G = tplan.G;
      h->b_cpg = tplan.cpg;
      h->b_nthreads = tplan.nthreads;
      h->b_tpr = tplan.tpr;
      h->b_ept = tplan.ept;
      h->kT = kT;
      h->bwd_ok = true;
      size_t n = 0;
      for (int32_t p : caller_pos) n += p >= 0 ? 1 : 0;
      h->n_caller = n;
    }
    // wide batches: the densified matrix on the K-split kernel, where that
    // measured faster than the sparse kernel (its gathers are bound by
    // shared memory at wide batch)
    size_t nnz = 0;
    for (int32_t p : caller_pos) nnz += p >= 0 ? 1 : 0;
    if (h->sks_opt == 2 || (h->sks_opt == 1 && ksplit_sparse_default(H, nnz, h->maxB))) {
      std::vector<uint16_t> dense((size_t)H * H, 0);
      for (int r = 0; r < H; ++r)
        for (int j = 0; j < k; ++j)
          if (caller_pos[(size_t)r * k + j] >= 0)
            dense[(size_t)r * H + hc[(size_t)r * k + j]] = hv[(size_t)r * k + j];
      const prnn_status_t kst = install_ksplit(h, dense.data());
      if (kst != PRNN_OK) return kst;
      h->ks_nnz = nnz;
    }
  } else {
    std::vector<uint32_t> ws((size_t)H * k);
    for (int r = 0; r < H; ++r)
      for (int j = 0; j < k; ++j) ws[(size_t)r * k + j] = entry(r, j);
    PRNN_TRY(upload(&h->Wstep, ws.data(), ws.size() * 4));
    h->onchip_bytes = 0;
    h->kp = k;
  }
  h->sparse = true;
  h->k = k;
  h->tc_proj = h->wdtype == PRNN_F16 && projection_tc_supported();
  h->weights_set = true;
  return PRNN_OK;
}


extern "C" {

const char* prnn_status_string(prnn_status_t s) {
  switch (s) {
    case PRNN_OK: return "PRNN_OK";
    case PRNN_ERR_INVALID_ARG: return "PRNN_ERR_INVALID_ARG";
    case PRNN_ERR_UNSUPPORTED: return "PRNN_ERR_UNSUPPORTED";
    case PRNN_ERR_NOT_READY: return "PRNN_ERR_NOT_READY";
    case PRNN_ERR_CUDA: return "PRNN_ERR_CUDA";
    case PRNN_ERR_OOM: return "PRNN_ERR_OOM";
    case PRNN_ERR_TIMEOUT: return "PRNN_ERR_TIMEOUT";
  }
  return "PRNN_ERR_UNKNOWN";
}

prnn_status_t prnn_create(prnn_t* out, int hidden, int input, int max_batch,
                          prnn_dtype_t wdtype, prnn_algo_t algo) {
  if (!out) return PRNN_ERR_INVALID_ARG;
  *out = nullptr;
  if (hidden < 1 || input < 1 || max_batch < 1 || max_batch > kMaxBatch)
    return PRNN_ERR_INVALID_ARG;
  if (wdtype != PRNN_F32 && wdtype != PRNN_F16) return PRNN_ERR_INVALID_ARG;
  if (algo != PRNN_ALGO_PERSISTENT && algo != PRNN_ALGO_PER_STEP) return PRNN_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PRNN_ERR_UNSUPPORTED;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return PRNN_ERR_UNSUPPORTED;
  if (prop.major != 10 || prop.minor != 3) return PRNN_ERR_UNSUPPORTED;  // built for sm_103a
  if (!prop.cooperativeLaunch) return PRNN_ERR_UNSUPPORTED;
  prnn_handle* h = new (std::nothrow) prnn_handle();
  if (!h) return PRNN_ERR_OOM;
  h->H = hidden;
  h->I = input;
  h->maxB = max_batch;
  h->wdtype = wdtype;
  h->algo = algo;
  h->device = dev;
  h->sm_count = prop.multiProcessorCount;
  h->smem_optin = prop.sharedMemPerBlockOptin;
  if (cudaDeviceGetAttribute(&h->clock_khz, cudaDevAttrClockRate, dev) != cudaSuccess)
    h->clock_khz = 2000000;
  h->Kp = round_up(input, 64);
  prnn_status_t st = PRNN_OK;
  if (cudaMalloc((void**)&h->status, 4 * sizeof(int)) != cudaSuccess ||
      cudaMalloc((void**)&h->bar, sizeof(unsigned)) != cudaSuccess ||
      cudaMemset(h->status, 0, 4 * sizeof(int)) != cudaSuccess ||
      cudaMemset(h->bar, 0, sizeof(unsigned)) != cudaSuccess)
    st = PRNN_ERR_OOM;
  for (int i = 0; i < 3 && st == PRNN_OK; ++i)
    if (cudaEventCreate(&h->ev[i]) != cudaSuccess) st = PRNN_ERR_CUDA;
  if (st == PRNN_OK &&
      cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking) != cudaSuccess)
    st = PRNN_ERR_CUDA;
  if (st != PRNN_OK) {
    prnn_destroy(h);
    return st;
  }
  *out = h;
  return PRNN_OK;
}

prnn_status_t prnn_destroy(prnn_t h) {
  if (!h) return PRNN_OK;
  cudaSetDevice(h->device);
  free_weights(h);
  free_dev(h->P);
  free_dev(h->x16);
  free_dev(h->hx);
  free_dev(h->hh0);
  free_dev(h->hy);
  free_dev(h->tws);
  free_dev(h->gws16);
  free_dev(h->status);
  free_dev(h->bar);
  for (auto& e : h->ev)
    if (e) cudaEventDestroy(e);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  delete h;
  return PRNN_OK;
}

prnn_status_t prnn_set_weights_dense(prnn_t h, const void* Wx, const void* Wh,
                                     const float* bias, void* stream) {
  if (!h || !Wx || !Wh || !bias) return PRNN_ERR_INVALID_ARG;
  if (h->sticky_timeout) return PRNN_ERR_TIMEOUT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PRNN_TRY(cudaStreamSynchronize(s));
  const int H = h->H;
  const size_t esz = h->wdtype == PRNN_F16 ? 2 : 4;
  DensePlan plan{};
  if (h->algo == PRNN_ALGO_PERSISTENT) {
    plan = plan_dense(h);
    if (!plan.ok) return PRNN_ERR_UNSUPPORTED;
  }
  std::vector<unsigned char> wh((size_t)H * H * esz);
  PRNN_TRY(to_host(wh.data(), Wh, wh.size()));

  free_weights(h);
  prnn_status_t st = stage_wx_bias(h, Wx, bias, &h->Wx, &h->Wx16, &h->bias);
  if (st != PRNN_OK) return st;
  if (h->algo == PRNN_ALGO_PERSISTENT) {
    // per CTA: [chunk slot j][row r][thread i] -> 4 weights of row cta*R+r,
    // columns 4*(i + j*nthreads) .. +3 (zero outside the matrix)
    const int NT = plan.nthreads, nchunks = H / 4;
    const size_t vec = 4 * esz;
    // one block per CTA of a group; every group reads the same blocks
    std::vector<unsigned char> pk((size_t)plan.cpg * plan.cpt * plan.R * NT * vec, 0);
    std::vector<unsigned char> pt(pk.size(), 0);  // the same layout of Wh^T (backward)
    for (int cta = 0; cta < plan.cpg; ++cta)
      for (int j = 0; j < plan.cpt; ++j)
        for (int r = 0; r < plan.R; ++r)
          for (int i = 0; i < NT; ++i) {
            const int row = cta * plan.R + r, ch = i + j * NT;
            if (row >= H || ch >= nchunks) continue;
            const size_t dst = ((((size_t)cta * plan.cpt + j) * plan.R + r) * NT + i) * vec;
            std::memcpy(&pk[dst], &wh[((size_t)row * H + (size_t)ch * 4) * esz], vec);
            for (int q = 0; q < 4; ++q)  // Wh^T[row][4ch + q] = Wh[4ch + q][row]
              std::memcpy(&pt[dst + q * esz], &wh[((size_t)(ch * 4 + q) * H + row) * esz], esz);
          }
    PRNN_TRY(upload(&h->Wpk, pk.data(), pk.size()));
    PRNN_TRY(upload(&h->Wpk_T, pt.data(), pt.size()));
    PRNN_TRY(upload(&h->Wh_nat, wh.data(), wh.size()));
    // tensor-core recurrence for wide batches: per CTA, K slice s of 64
    // columns holds N rows of 128 bytes, 16-byte chunk c of row n at
    // c ^ (n & 7) (the 128-byte swizzle of the K-major MMA operand)
    const TcPlan tp = plan_dense_tc(h);
    const bool want = h->rtc_opt == 2 || (h->rtc_opt == 0 && h->maxB >= 16);  // 1: off
    if (tp.ok && want) {
      const int nsl = H / 64;
      std::vector<uint16_t> img((size_t)tp.cpg * nsl * tp.N * 64, 0);
      const uint16_t* w16 = reinterpret_cast<const uint16_t*>(wh.data());
      for (int cta = 0; cta < tp.cpg; ++cta)
        for (int s = 0; s < nsl; ++s)
          for (int n = 0; n < tp.R; ++n) {
            const int row = cta * tp.R + n;
            if (row >= H) continue;
            for (int c = 0; c < 8; ++c)
              for (int e = 0; e < 8; ++e)
                img[(((size_t)cta * nsl + s) * tp.N + n) * 64 + ((c ^ (n & 7)) * 8) + e] =
                    w16[(size_t)row * H + s * 64 + c * 8 + e];
          }
      PRNN_TRY(upload(&h->Wimg, img.data(), img.size() * 2));
      h->rtc = true;
      h->t_n_cta = tp.n_cta;
      h->t_R = tp.R;
      h->t_G = tp.G;
      h->t_cpg = tp.cpg;
      h->t_N = tp.N;
      h->t_ring = tp.nring;
    }
    // wide batches: CTAs of 8 or 16 rows, one group over all batch columns
    int wR = 0, wS = 0, wD = 0;
    size_t wsm = 0;
    if (h->wdtype == PRNN_F16 && h->maxB >= kDenseWideMinB &&
        recur_dense_wide_plan(H, h->sm_count, h->smem_optin, &wR, &wS, &wD, &wsm)) {
      const int nch = H / 4, qg = wR / 4, ncta = H / wR;
      const uint16_t* w16 = reinterpret_cast<const uint16_t*>(wh.data());
      std::vector<uint16_t> img((size_t)ncta * 2 * qg * nch * 8);  // per CTA 2 x qg x nch uint4
      for (int cta = 0; cta < ncta; ++cta)
        for (int half = 0; half < 2; ++half)      // Wlo, Whi
          for (int q = 0; q < qg; ++q)
            for (int ch = 0; ch < nch; ++ch)
              for (int i = 0; i < 2; ++i) {       // two rows per uint4
                const int row = cta * wR + 4 * q + 2 * half + i;
                const size_t dst = ((((size_t)cta * 2 + half) * qg + q) * nch + ch) * 8 + i * 4;
                for (int e = 0; e < 4; ++e) img[dst + e] = w16[(size_t)row * H + ch * 4 + e];
              }
      PRNN_TRY(upload(&h->Wpk_wide, img.data(), img.size() * 2));
      std::vector<float> z((size_t)h->maxB * H, 0.f);
      PRNN_TRY(upload(&h->zeros, z.data(), z.size() * sizeof(float)));
      h->wide = true;
      h->w_R = wR;
      h->w_S = wS;
      h->w_depth = wD;
      h->w_smem = wsm;
    }
    // wide batches on the tensor cores (the K-split kernel)
    if (h->wdtype == PRNN_F16 && (ksplit_default(H, h->maxB) || h->ks_opt == 2)) {
      const prnn_status_t kst = install_ksplit(h, reinterpret_cast<const uint16_t*>(wh.data()));
      if (kst != PRNN_OK) return kst;
    }
    h->n_cta = plan.n_cta;
    h->R = plan.R;
    h->G = plan.G;
    h->cpg = plan.cpg;
    h->nthreads = plan.nthreads;
    h->cpt = plan.cpt;
    h->dense_bw = plan.bw;
    h->smem_at_max = plan.smem;
    h->onchip_bytes = pk.size() * plan.G;
  } else {
    PRNN_TRY(upload(&h->Wstep, wh.data(), wh.size()));
    h->onchip_bytes = 0;
  }
  h->sparse = false;
  h->k = H;
  h->tc_proj = h->wdtype == PRNN_F16 && projection_tc_supported();
  h->weights_set = true;
  return PRNN_OK;
}

prnn_status_t prnn_set_weights_sparse(prnn_t h, const void* Wx, int k, const uint16_t* vals,
                                      const uint16_t* cols, const float* bias, void* stream) {
  if (!h || !Wx || !vals || !cols || !bias) return PRNN_ERR_INVALID_ARG;
  if (h->sticky_timeout) return PRNN_ERR_TIMEOUT;
  if (h->wdtype != PRNN_F16) return PRNN_ERR_INVALID_ARG;
  const int H = h->H;
  if (H > 65535 || k < 1 || k > H) return PRNN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PRNN_TRY(cudaStreamSynchronize(s));
  std::vector<uint16_t> hv((size_t)H * k), hc((size_t)H * k);
  PRNN_TRY(to_host(hv.data(), vals, hv.size() * 2));
  PRNN_TRY(to_host(hc.data(), cols, hc.size() * 2));
  // validate: columns in range, distinct within each row; sort each row by column
  std::vector<int> seen((size_t)H, -1);
  std::vector<int32_t> pos((size_t)H * k);
  std::vector<std::pair<uint16_t, int>> row(k);  // (column, index in the caller's row)
  std::vector<uint16_t> rv(k);
  for (int r = 0; r < H; ++r) {
    for (int j = 0; j < k; ++j) {
      const int c = hc[(size_t)r * k + j];
      if (c >= H || seen[c] == r) return PRNN_ERR_INVALID_ARG;
      seen[c] = r;
      row[j] = {hc[(size_t)r * k + j], j};
      rv[j] = hv[(size_t)r * k + j];
    }
    std::sort(row.begin(), row.end(),
              [](const std::pair<uint16_t, int>& a, const std::pair<uint16_t, int>& b) {
                return a.first < b.first;
              });
    for (int j = 0; j < k; ++j) {
      hc[(size_t)r * k + j] = row[j].first;
      hv[(size_t)r * k + j] = rv[row[j].second];
      pos[(size_t)r * k + j] = r * k + row[j].second;
    }
  }
  return install_sparse(h, Wx, bias, hv, hc, k, pos);
}

prnn_status_t prnn_set_weights_csr(prnn_t h, const void* Wx, int nnz, const int32_t* row_ptr,
                                   const uint16_t* cols, const uint16_t* vals, const float* bias,
                                   void* stream) {
  if (!h || !Wx || !row_ptr || !bias || nnz < 0) return PRNN_ERR_INVALID_ARG;
  if (nnz > 0 && (!cols || !vals)) return PRNN_ERR_INVALID_ARG;
  if (h->sticky_timeout) return PRNN_ERR_TIMEOUT;
  if (h->wdtype != PRNN_F16) return PRNN_ERR_INVALID_ARG;
  const int H = h->H;
  if (H > 65535) return PRNN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PRNN_TRY(cudaStreamSynchronize(s));
  std::vector<int32_t> rp((size_t)H + 1);
  std::vector<uint16_t> cv((size_t)nnz), vv((size_t)nnz);
  PRNN_TRY(to_host(rp.data(), row_ptr, rp.size() * 4));
  if (nnz > 0) {
    PRNN_TRY(to_host(cv.data(), cols, cv.size() * 2));
    PRNN_TRY(to_host(vv.data(), vals, vv.size() * 2));
  }
  // validate: offsets monotone from 0 to nnz, columns in range and distinct per row
  if (rp[0] != 0 || rp[H] != nnz) return PRNN_ERR_INVALID_ARG;
  int kmax = 1;
  for (int r = 0; r < H; ++r) {
    if (rp[r + 1] < rp[r]) return PRNN_ERR_INVALID_ARG;
    kmax = std::max(kmax, rp[r + 1] - rp[r]);
  }
  std::vector<int> seen((size_t)H, -1);
  for (int r = 0; r < H; ++r)
    for (int j = rp[r]; j < rp[r + 1]; ++j) {
      const int c = cv[j];
      if (c >= H || seen[c] == r) return PRNN_ERR_INVALID_ARG;
      seen[c] = r;
    }
  // pad every row to the longest one with zero-valued entries: the kernels
  // then give every row kmax entries of work (the cost of imbalance).  The
  // padding takes the columns the row lacks, in ascending order, so padded
  // rows keep distinct columns spread over the shared-memory banks.
  std::vector<uint16_t> hv((size_t)H * kmax, 0), hc((size_t)H * kmax, 0);
  std::vector<int32_t> pos((size_t)H * kmax, -1);
  struct Ent {
    uint16_t col, val;
    int32_t src;  // index in the caller's arrays, -1 for padding
  };
  std::vector<Ent> row;
  std::vector<int> in_row((size_t)H, -1);
  for (int r = 0; r < H; ++r) {
    row.clear();
    for (int j = rp[r]; j < rp[r + 1]; ++j) {
      row.push_back({cv[j], vv[j], j});
      in_row[cv[j]] = r;
    }
    for (int c = 0; c < H && (int)row.size() < kmax; ++c)
      if (in_row[c] != r) row.push_back({(uint16_t)c, 0, -1});
    std::sort(row.begin(), row.end(), [](const Ent& a, const Ent& b) { return a.col < b.col; });
    for (int j = 0; j < kmax; ++j) {
      hc[(size_t)r * kmax + j] = row[j].col;
      hv[(size_t)r * kmax + j] = row[j].val;
      pos[(size_t)r * kmax + j] = row[j].src;
    }
  }
  return install_sparse(h, Wx, bias, hv, hc, kmax, pos);
}

// Whether a dense persistent forward of B columns runs the wide-batch kernel:
// planned at set_weights, enabled, flags in the data, and at least two
// passes of 8 columns per step (so a pass's copy is fetched during the
// previous pass).  By default only where it measured faster than the B <= 4
// kernel: three or more passes at H >= 1024, two at H >= 2048.
static bool dense_wide_for(const prnn_t h, int B) {
  if (h->algo != PRNN_ALGO_PERSISTENT || h->sparse || !h->wide || h->wide_opt == 0 ||
      h->sync_mode != 0 || h->rtc || B < kDenseWideMinB)
    return false;
  const int passes = (B + 7) / 8;
  return h->wide_opt == 2 || (passes >= 3 ? h->H >= 1024 : h->H >= 2048);
}

// Whether a persistent forward of B columns runs the tensor-core K-split
// kernel: planned at set_weights, enabled, flags in the data, B <= 32, and by
// default only where it measured faster (ksplit_default for dense layers,
// ksplit_sparse_default for sparse ones, which run their densified matrix).
static bool ksplit_for(const prnn_t h, int B) {
  if (h->algo != PRNN_ALGO_PERSISTENT || !h->ks || h->sync_mode != 0 || B < 1 || B > kKsplitMaxB)
    return false;
  if (h->ks_stream && B > 16) return false;  // the streamed plan serves up to 16 columns
  if (h->sparse) return h->sks_opt == 2 || (h->sks_opt == 1 && ksplit_sparse_default(h->H, h->ks_nnz, B));
  if (h->ks_opt == 0 || h->rtc) return false;
  return h->ks_opt == 2 || ksplit_default(h->H, B);
}

// Whether the recurrent kernel prnn_forward would launch can also write every
// output into a second buffer (the persistent CUDA-core kernels can).
static bool recurrence_mirrors(const prnn_t h) {
  return h->algo == PRNN_ALGO_PERSISTENT && (h->sparse || !(h->rtc && h->sync_mode == 0));
}

// The forward on device buffers; y_mirror (nullptr, or a device-addressable
// [T][B][H] buffer; only when recurrence_mirrors) receives a copy of every
// output as the recurrence publishes it.  Arguments are checked by the callers.
static prnn_status_t forward_impl(prnn_t h, int T, int B, const float* x, const float* h0,
                                  float* y, float* y_mirror, cudaStream_t s) {
  if (h->trace) {  // the phase trace: sparse persistent kernel (column order, wide
                   // staging) or the dense K-split kernel
    const bool ks = ksplit_for(h, B);
    if (!ks && (h->algo != PRNN_ALGO_PERSISTENT || !h->sparse || h->place || !h->wide_loads))
      return PRNN_ERR_UNSUPPORTED;
    const size_t n_cta = ks ? (size_t)(h->H / 128 * h->ks_cs) : (size_t)h->n_cta;
    if ((size_t)T * n_cta * kTraceWords > h->trace_words) return PRNN_ERR_INVALID_ARG;
  }
  const size_t ny = (size_t)T * B * h->H;
  PRNN_TRY(ensure_P(h, ny));
  const bool persistent = h->algo == PRNN_ALGO_PERSISTENT;
  if (h->timing) PRNN_TRY(cudaEventRecord(h->ev[0], s));
  h->last_backward = false;

  // 1. projection for all steps (+ sentinel fill of y on the persistent path)
  if (h->tc_proj && h->proj_mode == 0) {
    PRNN_TRY(ensure_x16(h, (size_t)T * B * h->Kp));
    ProjTcArgs ta{T * B, h->H, h->I, h->Kp, x, h->x16, h->Wx16, h->bias, h->P,
                  persistent ? y : nullptr};
    PRNN_TRY(launch_projection_tc(ta, h->status, s));
  } else {
    ProjArgs pa{T * B, h->H, h->I, x, h->Wx, h->bias, h->P, persistent ? y : nullptr};
    PRNN_TRY(launch_projection_simt(pa, h->wdtype == PRNN_F16, s));
  }
  if (h->timing) PRNN_TRY(cudaEventRecord(h->ev[1], s));

  // 2. recurrence
  if (persistent) {
    RecurCommon c = common_args(h, T, B, h0, y);
    c.y_mirror = y_mirror;
    if (h->sync_mode == 1) PRNN_TRY(cudaMemsetAsync(h->bar, 0, sizeof(unsigned), s));
    if (ksplit_for(h, B)) {  // dense, or a sparse layer's densified matrix
      c.n_cta = h->H / 128 * h->ks_cs;
      c.R = 128;
      c.cpg = c.n_cta;
      c.G = 1;
      c.nthreads = 512;
      c.smem = recur_dense_ksplit_smem(h->ks_nat, B, h->ks_cs, h->ks_stream);
      if (h->poll_delay_ns < 0) c.poll_delay = 0;  // measured: no pause is fastest here
      DenseSplitArgs a{c, h->Wimg_ks, h0 ? h0 : h->zeros, h->ks_cs, h->ks_nat, h->trace,
                       h->ks_stream ? 1 : 0};
      PRNN_TRY(launch_recur_dense_ksplit(a, s));
    } else if (h->sparse) {
      SparseRecurArgs a{};
      int bg = 4;
      bool db = false;
      size_t sm = 0;
      if (!sparse_batch_plan(h, B, &bg, &db, &sm)) return PRNN_ERR_UNSUPPORTED;
      c.smem = sm;
      a.c = c;
      a.Wpk = static_cast<const uint32_t*>(h->Wpk);
      a.tpr = h->tpr;
      a.ept = h->ept;
      a.bgroup = bg;
      a.dbuf = db ? 1 : 0;
      a.narrow = h->wide_loads ? 0 : 1;
      a.place = h->place;
      a.trace = h->trace;
      a.regw = h->regw_opt && sparse_regw_fits(c.nthreads, bg, h->ept, h->place != nullptr);
      a.umax = h->depth_opt ? sparse_staging_depth(h->H, bg, c.nthreads, h->place != nullptr) : 0;
      PRNN_TRY(launch_recur_sparse(a, s));
    } else if (h->rtc && h->sync_mode == 0) {
      DenseTcArgs a{};
      c.n_cta = h->t_n_cta;
      c.R = h->t_R;
      c.G = h->t_G;
      c.cpg = h->t_cpg;
      c.nthreads = recur_dense_tc_threads();
      c.smem = recur_dense_tc_smem(h->H, h->t_N, h->t_ring);
      a.c = c;
      a.Wimg = h->Wimg;
      a.N = h->t_N;
      a.nslices = h->H / 64;
      a.nring = h->t_ring;
      PRNN_TRY(launch_recur_dense_tc(a, s));
    } else if (dense_wide_for(h, B)) {
      c.R = h->w_R;
      c.cpg = (h->H + h->w_R - 1) / h->w_R;
      c.n_cta = c.cpg;
      c.G = 1;
      c.nthreads = h->w_R / 4 * h->w_S;
      c.smem = h->w_smem;
      DenseWideArgs a{c, h->Wpk_wide, h0 ? h0 : h->zeros, h->w_S, h->w_depth};
      PRNN_TRY(launch_recur_dense_wide(a, s));
    } else {
      DenseRecurArgs a{};
      const int bw = std::min(recur_dense_bw((B + h->G - 1) / h->G), h->dense_bw);
      c.smem = recur_dense_smem(h->R, h->cpt, h->nthreads, h->wdtype == PRNN_F16, bw);
      if (h->poll_delay_ns < 0) {
        const int passes = ((B + h->G - 1) / h->G + bw - 1) / bw;
        c.poll_delay =
            (int)((long long)dense_delay_ns(h->H, bw, passes) * h->clock_khz / 1000000LL);
      }
      a.c = c;
      a.Wpk = h->Wpk;
      a.cpt = h->cpt;
      a.wfp16 = h->wdtype == PRNN_F16;
      PRNN_TRY(launch_recur_dense(a, bw, s));
    }
  } else {
    const bool hit = h->gexec && h->g_T == T && h->g_B == B && h->g_h0 == h0 && h->g_y == y &&
                     h->g_P == h->P && h->g_W == h->Wstep;
    if (!hit) {
      invalidate_graph(h);
      PRNN_TRY(cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
      cudaError_t e = cudaSuccess;
      for (int t = 0; t < T && e == cudaSuccess; ++t) {
        StepArgs sa{};
        sa.t = t;
        sa.B = B;
        sa.H = h->H;
        sa.P = h->P;
        sa.hprev = t == 0 ? h0 : y + (size_t)(t - 1) * B * h->H;
        sa.y = y;
        sa.W = h->Wstep;
        sa.wfp16 = h->wdtype == PRNN_F16;
        sa.sparse = h->sparse;
        sa.kp = h->kp;
        e = launch_step(sa, h->cap_stream);
      }
      cudaGraph_t g = nullptr;
      cudaError_t e2 = cudaStreamEndCapture(h->cap_stream, &g);
      if (e == cudaSuccess) e = e2;
      if (e == cudaSuccess) e = cudaGraphInstantiate(&h->gexec, g, 0);
      if (g) cudaGraphDestroy(g);
      if (e != cudaSuccess) {
        h->gexec = nullptr;
        return cuda_status(e);
      }
      h->g_T = T;
      h->g_B = B;
      h->g_h0 = h0;
      h->g_y = y;
      h->g_P = h->P;
      h->g_W = h->Wstep;
    }
    PRNN_TRY(cudaGraphLaunch(h->gexec, s));
  }
  if (h->timing) {
    PRNN_TRY(cudaEventRecord(h->ev[2], s));
    h->ev_valid = true;
  }
  return PRNN_OK;
}

prnn_status_t prnn_forward(prnn_t h, int T, int B, const float* x, const float* h0, float* y,
                           void* stream) {
  if (!h) return PRNN_ERR_INVALID_ARG;
  if (h->sticky_timeout) return PRNN_ERR_TIMEOUT;
  if (!h->weights_set) return PRNN_ERR_NOT_READY;
  if (T < 0 || B < 0 || B > h->maxB) return PRNN_ERR_INVALID_ARG;
  if (T == 0 || B == 0) return PRNN_OK;
  if (!x || !y) return PRNN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || (h0 && !aligned16(h0))) return PRNN_ERR_INVALID_ARG;
  const size_t ny = (size_t)T * B * h->H;
  if (overlaps(y, ny * 4, x, (size_t)T * B * h->I * 4)) return PRNN_ERR_INVALID_ARG;
  if (h0 && overlaps(y, ny * 4, h0, (size_t)B * h->H * 4)) return PRNN_ERR_INVALID_ARG;
  return forward_impl(h, T, B, x, h0, y, nullptr, static_cast<cudaStream_t>(stream));
}

prnn_status_t prnn_forward_host(prnn_t h, int T, int B, const float* x, const float* h0,
                                float* y, void* stream) {
  if (!h) return PRNN_ERR_INVALID_ARG;
  if (h->sticky_timeout) return PRNN_ERR_TIMEOUT;
  if (!h->weights_set) return PRNN_ERR_NOT_READY;
  if (T < 0 || B < 0 || B > h->maxB) return PRNN_ERR_INVALID_ARG;
  if (T == 0 || B == 0) return PRNN_OK;
  if (!x || !y) return PRNN_ERR_INVALID_ARG;
  const size_t nx = (size_t)T * B * h->I, ny = (size_t)T * B * h->H, n0 = (size_t)B * h->H;
  if (((uintptr_t)x | (uintptr_t)y | (uintptr_t)h0) & 3u) return PRNN_ERR_INVALID_ARG;
  if (overlaps(y, ny * 4, x, nx * 4)) return PRNN_ERR_INVALID_ARG;
  if (h0 && overlaps(y, ny * 4, h0, n0 * 4)) return PRNN_ERR_INVALID_ARG;
  // all three must be page-locked host memory the device can address.  The
  // last element is checked too, as a best-effort guard only: a buffer
  // shorter than its shape is refused when its end falls outside every
  // page-locked allocation, not when another allocation follows it (the
  // element counts are the caller's precondition, include/prnn.h)
  float* ydev = static_cast<float*>(const_cast<void*>(mapped_host(y)));
  const float* xdev = static_cast<const float*>(mapped_host(x));
  if (!xdev || !mapped_host(x + nx - 1) || !ydev || !mapped_host(y + ny - 1) ||
      (h0 && (!mapped_host(h0) || !mapped_host(h0 + n0 - 1))))
    return PRNN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // With the tensor-core projection x is read once, by its fp16 staging
  // kernel, which then reads it straight from the host buffer over the host
  // link: no copy of x.  The CUDA-core projection reads each x tile many
  // times, so there x is copied to a device workspace first.
  const bool x_direct = h->tc_proj && h->proj_mode == 0 && kHostXDirect;
  const float* xin = xdev;
  if (!x_direct) {
    PRNN_TRY(ensure_f32(&h->hx, &h->hx_cap, nx));
    PRNN_TRY(cudaMemcpyAsync(h->hx, x, nx * 4, cudaMemcpyHostToDevice, s));
    xin = h->hx;
  }
  PRNN_TRY(ensure_f32(&h->hy, &h->hy_cap, ny));
  if (h0) PRNN_TRY(ensure_f32(&h->hh0, &h->hh0_cap, n0));
  if (h0) PRNN_TRY(cudaMemcpyAsync(h->hh0, h0, n0 * 4, cudaMemcpyHostToDevice, s));
  const bool mirror = recurrence_mirrors(h);
  const prnn_status_t st =
      forward_impl(h, T, B, xin, h0 ? h->hh0 : nullptr, h->hy, mirror ? ydev : nullptr, s);
  if (st != PRNN_OK) return st;
  if (!mirror) PRNN_TRY(cudaMemcpyAsync(y, h->hy, ny * 4, cudaMemcpyDeviceToHost, s));
  return PRNN_OK;
}

prnn_status_t prnn_backward(prnn_t h, int T, int B, const float* x, const float* h0,
                            const float* y, const float* dy, float* delta_out, float* dx,
                            float* dh0, float* dWx, float* dWh, float* db, void* stream) {
  if (!h) return PRNN_ERR_INVALID_ARG;
  if (h->sticky_timeout) return PRNN_ERR_TIMEOUT;
  if (!h->weights_set) return PRNN_ERR_NOT_READY;
  if (h->algo != PRNN_ALGO_PERSISTENT || (h->sparse && !h->bwd_ok)) return PRNN_ERR_UNSUPPORTED;
  if (T < 0 || B < 0 || B > h->maxB) return PRNN_ERR_INVALID_ARG;
  const int H = h->H, I = h->I;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0 || B == 0) {  // no steps: every gradient is zero
    if (dWx) PRNN_TRY(cudaMemsetAsync(dWx, 0, (size_t)H * I * 4, s));
    if (dWh) PRNN_TRY(cudaMemsetAsync(dWh, 0, (h->sparse ? h->n_caller : (size_t)H * H) * 4, s));
    if (db) PRNN_TRY(cudaMemsetAsync(db, 0, (size_t)H * 4, s));
    if (dh0 && B > 0) PRNN_TRY(cudaMemsetAsync(dh0, 0, (size_t)B * H * 4, s));
    return PRNN_OK;
  }
  if (!x || !y || !dy) return PRNN_ERR_INVALID_ARG;
  const void* ins[] = {x, h0, y, dy};
  const void* outs[] = {dx, dh0, dWx, dWh, db, delta_out};
  for (const void* p : ins)
    if (p && !aligned16(p)) return PRNN_ERR_INVALID_ARG;
  for (const void* p : outs)
    if (p && !aligned16(p)) return PRNN_ERR_INVALID_ARG;
  const size_t ny = (size_t)T * B * H;
  const size_t dwh_n = h->sparse ? h->n_caller : (size_t)H * H;
  const size_t out_bytes[] = {(size_t)T * B * I * 4, (size_t)B * H * 4, (size_t)H * I * 4,
                              dwh_n * 4, (size_t)H * 4, ny * 4};
  const size_t in_bytes[] = {(size_t)T * B * I * 4, (size_t)B * H * 4, ny * 4, ny * 4};
  for (int o = 0; o < 6; ++o) {
    if (!outs[o]) continue;
    for (int i = 0; i < 4; ++i)
      if (ins[i] && overlaps(outs[o], out_bytes[o], ins[i], in_bytes[i])) return PRNN_ERR_INVALID_ARG;
    for (int o2 = 0; o2 < o; ++o2)
      if (outs[o2] && overlaps(outs[o], out_bytes[o], outs[o2], out_bytes[o2]))
        return PRNN_ERR_INVALID_ARG;
  }
  float* delta = delta_out;
  if (!delta) {
    PRNN_TRY(ensure_P(h, ny));  // the projection workspace holds the deltas
    delta = h->P;
  }
  if (h->timing) PRNN_TRY(cudaEventRecord(h->ev[0], s));

  // 1. reverse recurrence: delta_t = [y_t > 0] (dy_t + Wh^T delta_{t+1}),
  // the mask folded into a copy of dy in the transposed-delta workspace
  // (sized once here for every later use: the masked dy, the transposed
  // delta and h of the fp32 value gradients, the dense product of the
  // tensor-core value gradients)
  const bool tc_vals = h->sparse && h->wdtype == PRNN_F16 && h->tc_proj && h->proj_mode == 0 &&
                       h->WxT16;
  const size_t need_tws = std::max({(size_t)2 * H * T * B, ny, tc_vals ? (size_t)H * H : 0});
  if (need_tws > h->tws_cap) {
    free_dev(h->tws);
    h->tws_cap = 0;
    PRNN_TRY(cudaMalloc((void**)&h->tws, need_tws * sizeof(float)));
    h->tws_cap = need_tws;
  }
  PRNN_TRY(launch_fold_mask(dy, y, ny, h->tws, s));
  PRNN_TRY(launch_fill_sentinel(delta, ny, s));
  RecurCommon c = common_args(h, T, B, nullptr, delta);
  c.P = h->tws;
  c.reverse = 1;
  c.p_masked = 1;
  c.sync_mode = 0;
  if (ksplit_for(h, B) && h->WimgT_ks) {  // wide batch: Wh^T on the K-split kernel
    c.n_cta = h->H / 128 * h->ks_cs;
    c.R = 128;
    c.cpg = c.n_cta;
    c.G = 1;
    c.nthreads = 512;
    c.smem = recur_dense_ksplit_smem(h->ks_nat, B, h->ks_cs, h->ks_stream);
    if (h->poll_delay_ns < 0) c.poll_delay = 0;
    DenseSplitArgs a{c, h->WimgT_ks, h->zeros, h->ks_cs, h->ks_nat, nullptr, h->ks_stream ? 1 : 0};
    PRNN_TRY(launch_recur_dense_ksplit(a, s));
  } else if (h->sparse) {  // Wh^T has its own plan (its rows are Wh's columns)
    c.n_cta = h->b_n_cta;
    c.R = h->b_R;
    c.G = h->b_G;
    c.cpg = h->b_cpg;
    c.nthreads = h->b_nthreads;
    c.poll_delay = h->poll_delay_ns >= 0
                       ? (int)((long long)h->poll_delay_ns * h->clock_khz / 1000000LL)
                       : (int)((long long)sparse_delay_ns(h->H) * h->clock_khz / 1000000LL);
    SparseRecurArgs a{};
    int bg = 4;
    bool dbuf = false;
    size_t sm = 0;
    if (!sparse_batch_plan(h, B, &bg, &dbuf, &sm, true)) return PRNN_ERR_UNSUPPORTED;
    c.smem = sm;
    a.c = c;
    a.Wpk = static_cast<const uint32_t*>(h->Wpk_T);
    a.tpr = h->b_tpr;
    a.ept = h->b_ept;
    a.bgroup = bg;
    a.dbuf = dbuf ? 1 : 0;
    a.narrow = 0;
    a.place = h->place_T;
    a.regw = h->regw_opt && sparse_regw_fits(c.nthreads, bg, h->b_ept, h->place_T != nullptr);
    a.umax = h->depth_opt ? sparse_staging_depth(h->H, bg, c.nthreads, h->place_T != nullptr) : 0;
    PRNN_TRY(launch_recur_sparse(a, s));
  } else {
    DenseRecurArgs a{};
    const int bw = std::min(recur_dense_bw((B + h->G - 1) / h->G), h->dense_bw);
    c.smem = recur_dense_smem(h->R, h->cpt, h->nthreads, h->wdtype == PRNN_F16, bw);
    if (h->poll_delay_ns < 0) {
      const int passes = ((B + h->G - 1) / h->G + bw - 1) / bw;
      c.poll_delay =
          (int)((long long)dense_delay_ns(h->H, bw, passes) * h->clock_khz / 1000000LL);
    }
    a.c = c;
    a.Wpk = h->Wpk_T;
    a.cpt = h->cpt;
    a.wfp16 = h->wdtype == PRNN_F16;
    PRNN_TRY(launch_recur_dense(a, bw, s));
  }
  if (h->timing) PRNN_TRY(cudaEventRecord(h->ev[1], s));

  // 2. batched gradients over all T*B rows of delta
  const int K = T * B;
  const bool f16 = h->wdtype == PRNN_F16;
  // fp16 weights: the three large products on the tensor cores in bf16
  // (fp32 accumulation); fp32 weights keep full fp32 CUDA-core products
  const bool tc = f16 && h->tc_proj && h->proj_mode == 0 && h->WxT16;
  if (db) PRNN_TRY(launch_colsum(delta, K, H, db, s));
  if (tc && (dWx || dx || dWh)) {
    const int Kp = round_up(K, 64), Hp = round_up(H, 64);
    const size_t n_dT = (size_t)H * Kp, n_hT = (size_t)H * Kp, n_xT = (size_t)I * Kp;
    const size_t n_d = (size_t)K * Hp;
    const size_t need = n_dT + n_hT + n_xT + n_d;
    if (need > h->gws16_cap) {
      free_dev(h->gws16);
      h->gws16_cap = 0;
      PRNN_TRY(cudaMalloc((void**)&h->gws16, need * 2));
      h->gws16_cap = need;
    }
    uint16_t* dT16 = h->gws16;
    uint16_t* hT16 = dT16 + n_dT;
    uint16_t* xT16 = hT16 + n_hT;
    uint16_t* d16 = xT16 + n_xT;
    if (dWx || dWh) PRNN_TRY(launch_transpose_bf16(K, Kp, H, 0, nullptr, delta, H, dT16, s));
    if (dWh) {
      PRNN_TRY(launch_transpose_bf16(K, Kp, H, B, h0, y, H, hT16, s));
      float* dense = dWh;
      if (h->sparse) dense = h->tws;  // the dense product, then the stored entries
      GemmTcArgs g{H, H, Kp, dT16, hT16, true, dense};
      PRNN_TRY(launch_gemm_tc(g, h->status, s));
      if (h->sparse)
        PRNN_TRY(launch_gather_pattern(H, h->k, dense, h->cols_pad, h->caller_pos, dWh, s));
    }
    if (dWx) {
      PRNN_TRY(launch_transpose_bf16(K, Kp, I, 0, nullptr, x, I, xT16, s));
      GemmTcArgs g{H, I, Kp, dT16, xT16, true, dWx};
      PRNN_TRY(launch_gemm_tc(g, h->status, s));
    }
    if (dx) {
      PRNN_TRY(launch_rows_bf16(K, H, Hp, delta, d16, s));
      GemmTcArgs g{K, I, Hp, d16, h->WxT16, true, dx};
      PRNN_TRY(launch_gemm_tc(g, h->status, s));
    }
    dWx = nullptr;  // done
    dx = nullptr;
    dWh = nullptr;
  }
  if (dWh && !h->sparse) {
    GemmTnArgs g{H, H, K, B, delta, H, h0, y, H, dWh};
    PRNN_TRY(launch_gemm_tn(g, s));
  }
  if (dWh && h->sparse) {  // only at the stored entries, in the caller's order
    float* dT = h->tws;  // the folded dy is no longer needed: 2*H*K floats
    float* hT = h->tws + (size_t)H * K;
    PRNN_TRY(launch_transpose_rows(K, H, 0, nullptr, delta, H, dT, s));
    PRNN_TRY(launch_transpose_rows(K, H, B, h0, y, H, hT, s));
    PRNN_TRY(launch_sddmm(H, h->k, K, dT, hT, h->cols_pad, h->caller_pos, dWh, s));
  }
  if (dWx) {
    GemmTnArgs g{H, I, K, 0, delta, H, nullptr, x, I, dWx};
    PRNN_TRY(launch_gemm_tn(g, s));
  }
  if (dx) {
    GemmNnArgs g{K, I, H, delta, H, h->Wx, I, f16 ? 1 : 0, dx};
    PRNN_TRY(launch_gemm_nn(g, s));
  }
  if (dh0 && !h->sparse) {
    GemmNnArgs g{B, H, H, delta, H, h->Wh_nat, H, f16 ? 1 : 0, dh0};
    PRNN_TRY(launch_gemm_nn(g, s));
  }
  if (dh0 && h->sparse) PRNN_TRY(launch_sparse_dh0(B, H, h->kT, h->valsT, h->colsT, delta, dh0, s));
  if (h->timing) {
    PRNN_TRY(cudaEventRecord(h->ev[2], s));
    h->ev_valid = true;
    h->last_backward = true;
  }
  return PRNN_OK;
}

prnn_status_t prnn_get_status(prnn_t h, void* stream) {
  if (!h) return PRNN_ERR_INVALID_ARG;
  PRNN_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  int st[4] = {0, 0, 0, 0};
  PRNN_TRY(cudaMemcpy(st, h->status, sizeof(st), cudaMemcpyDeviceToHost));
  if (st[0] != 0) h->sticky_timeout = true;
  return h->sticky_timeout ? PRNN_ERR_TIMEOUT : PRNN_OK;
}

prnn_status_t prnn_set_option(prnn_t h, prnn_option_t opt, long long value) {
  if (!h) return PRNN_ERR_INVALID_ARG;
  switch (opt) {
    case PRNN_OPT_WAIT_TIMEOUT_US:
      if (value < 1 || value > 60LL * 1000 * 1000) return PRNN_ERR_INVALID_ARG;
      h->timeout_us = value;
      return PRNN_OK;
    case PRNN_OPT_SYNC_MODE:
      if (value != 0 && value != 1) return PRNN_ERR_INVALID_ARG;
      h->sync_mode = (int)value;
      return PRNN_OK;
    case PRNN_OPT_DEBUG_DROP_CTA:
      if (value < -1 || value > 1 << 20) return PRNN_ERR_INVALID_ARG;
      h->drop_cta = (int)value;
      return PRNN_OK;
    case PRNN_OPT_DEBUG_DROP_STEP:
      if (value < -1 || value > 1 << 30) return PRNN_ERR_INVALID_ARG;
      h->drop_step = (int)value;
      return PRNN_OK;
    case PRNN_OPT_TIMING:
      if (value != 0 && value != 1) return PRNN_ERR_INVALID_ARG;
      h->timing = (int)value;
      h->ev_valid = false;
      return PRNN_OK;
    case PRNN_OPT_PROJECTION:
      if (value != 0 && value != 1) return PRNN_ERR_INVALID_ARG;
      h->proj_mode = (int)value;
      return PRNN_OK;
    case PRNN_OPT_CTA_GROUPS:
      if (value < 0 || value > 32) return PRNN_ERR_INVALID_ARG;
      h->groups_opt = (int)value;
      return PRNN_OK;
    case PRNN_OPT_WIDE_LOADS:
      if (value != 0 && value != 1) return PRNN_ERR_INVALID_ARG;
      h->wide_loads = (int)value;
      return PRNN_OK;
    case PRNN_OPT_BANK_AWARE:
      if (value != 0 && value != 1) return PRNN_ERR_INVALID_ARG;
      h->bank_aware = (int)value;
      return PRNN_OK;
    case PRNN_OPT_POLL_DELAY_NS:
      if (value < 0 || value > 10000) return PRNN_ERR_INVALID_ARG;
      h->poll_delay_ns = (int)value;
      return PRNN_OK;
    case PRNN_OPT_POLL_BACKOFF_NS:
      if (value < 0 || value > 10000) return PRNN_ERR_INVALID_ARG;
      h->backoff_ns = (int)value;
      return PRNN_OK;
    case PRNN_OPT_RECURRENT_TC:
      if (value < 0 || value > 2) return PRNN_ERR_INVALID_ARG;
      h->rtc_opt = (int)value;
      return PRNN_OK;
    case PRNN_OPT_STAGED_ORDER:
      if (value < 0 || value > 2) return PRNN_ERR_INVALID_ARG;
      h->staged_order = (int)value;
      return PRNN_OK;
    case PRNN_OPT_SPARSE_REG_WEIGHTS:
      if (value != 0 && value != 1) return PRNN_ERR_INVALID_ARG;
      h->regw_opt = (int)value;
      return PRNN_OK;
    case PRNN_OPT_SPARSE_STAGING_DEPTH:
      if (value != 0 && value != 1) return PRNN_ERR_INVALID_ARG;
      h->depth_opt = (int)value;
      return PRNN_OK;
    case PRNN_OPT_DENSE_WIDE:
      if (value < 0 || value > 2) return PRNN_ERR_INVALID_ARG;
      h->wide_opt = (int)value;
      return PRNN_OK;
    case PRNN_OPT_DENSE_KSPLIT:
      if (value < 0 || value > 2) return PRNN_ERR_INVALID_ARG;
      h->ks_opt = (int)value;
      return PRNN_OK;
    case PRNN_OPT_SPARSE_KSPLIT:
      if (value < 0 || value > 2) return PRNN_ERR_INVALID_ARG;
      h->sks_opt = (int)value;
      return PRNN_OK;
  }
  return PRNN_ERR_INVALID_ARG;
}

prnn_status_t prnn_get_info(prnn_t h, prnn_info_t* info) {
  if (!h || !info) return PRNN_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  info->hidden = h->H;
  info->input = h->I;
  info->max_batch = h->maxB;
  info->wdtype = h->wdtype;
  info->algo = h->algo;
  info->sparse = h->sparse;
  info->weights_set = h->weights_set;
  info->k = h->k;
  info->k_padded = h->sparse ? h->kp : h->H;
  info->sm_count = h->sm_count;
  info->n_cta = h->n_cta;
  info->rows_per_cta = h->R;
  info->threads_per_cta = h->nthreads;
  info->threads_per_row = h->tpr;
  info->projection_tensor_cores = h->tc_proj && h->proj_mode == 0;
  info->sparse_bank_cap = h->sparse ? h->pack_cap : 0;
  info->cta_groups = h->G;
  info->smem_bytes = h->smem_at_max;
  info->onchip_weight_bytes = h->onchip_bytes;
  info->nnz = h->sparse ? (size_t)h->H * h->k : (size_t)h->H * h->H;
  info->recurrent_tensor_cores = h->rtc ? 1 : 0;
  info->sparse_staged_order = h->sparse && h->place != nullptr ? 1 : 0;
  if (h->sparse && h->algo == PRNN_ALGO_PERSISTENT && h->weights_set) {
    int bg = 4;
    bool db = false;
    size_t sm = 0;
    info->sparse_reg_weights =
        h->regw_opt && sparse_batch_plan(h, h->maxB, &bg, &db, &sm) &&
                sparse_regw_fits(h->nthreads, bg, h->ept, h->place != nullptr)
            ? 1
            : 0;
  }
  if (h->weights_set && ksplit_for(h, h->maxB)) {
    info->dense_ksplit = h->ks_cs;
    info->n_cta = h->H / 128 * h->ks_cs;
    info->rows_per_cta = 128;
    info->threads_per_cta = 512;
    info->cta_groups = 1;
    info->smem_bytes = recur_dense_ksplit_smem(h->ks_nat, h->maxB, h->ks_cs, h->ks_stream);
  } else if (h->weights_set && dense_wide_for(h, h->maxB)) {
    info->dense_wide_batch = 1;
    info->n_cta = (h->H + h->w_R - 1) / h->w_R;
    info->rows_per_cta = h->w_R;
    info->threads_per_cta = h->w_R / 4 * h->w_S;
    info->cta_groups = 1;
    info->smem_bytes = h->w_smem;
  }
  if (h->rtc) {
    info->n_cta = h->t_n_cta;
    info->rows_per_cta = h->t_R;
    info->threads_per_cta = recur_dense_tc_threads();
    info->cta_groups = h->t_G;
    info->smem_bytes = recur_dense_tc_smem(h->H, h->t_N, h->t_ring);
  }
  return PRNN_OK;
}

prnn_status_t prnn_get_timing(prnn_t h, float* ms_projection, float* ms_recurrence) {
  if (!h) return PRNN_ERR_INVALID_ARG;
  if (!h->timing || !h->ev_valid) return PRNN_ERR_NOT_READY;
  PRNN_TRY(cudaEventSynchronize(h->ev[2]));
  float a = 0.f, b = 0.f;
  PRNN_TRY(cudaEventElapsedTime(&a, h->ev[0], h->ev[1]));
  PRNN_TRY(cudaEventElapsedTime(&b, h->ev[1], h->ev[2]));
  // forward: (projection, recurrence); backward: (gradient products, reverse recurrence)
  if (ms_projection) *ms_projection = h->last_backward ? b : a;
  if (ms_recurrence) *ms_recurrence = h->last_backward ? a : b;
  return PRNN_OK;
}

prnn_status_t prnn_set_trace_buffer(prnn_t h, void* buffer, size_t bytes) {
  if (!h) return PRNN_ERR_INVALID_ARG;
  if (buffer == nullptr) {
    h->trace = nullptr;
    h->trace_words = 0;
    return PRNN_OK;
  }
  if (!aligned16(buffer) || bytes < kTraceWords * sizeof(uint32_t)) return PRNN_ERR_INVALID_ARG;
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, buffer) != cudaSuccess) {
    cudaGetLastError();
    return PRNN_ERR_INVALID_ARG;
  }
  if (at.type != cudaMemoryTypeDevice) return PRNN_ERR_INVALID_ARG;
  h->trace = static_cast<uint32_t*>(buffer);
  h->trace_words = bytes / sizeof(uint32_t);
  return PRNN_OK;
}

prnn_status_t prnn_probe_sync_floor(prnn_t h, int T, int B, float* y, void* stream) {
  if (!h) return PRNN_ERR_INVALID_ARG;
  if (h->sticky_timeout) return PRNN_ERR_TIMEOUT;
  if (!h->weights_set || h->algo != PRNN_ALGO_PERSISTENT) return PRNN_ERR_NOT_READY;
  if (T < 0 || B < 0 || B > h->maxB) return PRNN_ERR_INVALID_ARG;
  if (T == 0 || B == 0) return PRNN_OK;
  if (!y || !aligned16(y)) return PRNN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int bl = (B + h->G - 1) / h->G;
  int bg = std::min(32, std::max(4, round_up(bl, 4)));
  int um = 0;
  if (h->sparse) {  // the sparse forward's batch passes and staging depth
    bool db = false;
    size_t sm = 0;
    if (!sparse_batch_plan(h, B, &bg, &db, &sm)) return PRNN_ERR_UNSUPPORTED;
    um = h->depth_opt ? sparse_staging_depth(h->H, bg, h->nthreads, h->place != nullptr) : 0;
  }
  RecurCommon c = common_args(h, T, B, nullptr, y);
  c.smem = sync_probe_smem(h->H, bg);
  if (c.smem > h->smem_optin) return PRNN_ERR_UNSUPPORTED;
  if (h->timing) PRNN_TRY(cudaEventRecord(h->ev[0], s));
  h->last_backward = false;
  PRNN_TRY(launch_fill_sentinel(y, (size_t)T * B * h->H, s));
  if (h->timing) PRNN_TRY(cudaEventRecord(h->ev[1], s));
  PRNN_TRY(launch_sync_probe(c, bg, um, s));
  if (h->timing) {
    PRNN_TRY(cudaEventRecord(h->ev[2], s));
    h->ev_valid = true;
  }
  return PRNN_OK;
}

prnn_status_t prnn_pack_sparse_host(int hidden, int k, int n_cta, int rows_per_cta,
                                    int threads_per_row, const uint16_t* vals,
                                    const uint16_t* cols, uint32_t* packed,
                                    size_t capacity_words, int* ept, int* bank_cap) {
  const int H = hidden, R = rows_per_cta, tpr = threads_per_row;
  if (H < 1 || H > 65535 || k < 1 || k > H || n_cta < 1 || R < 1 || (size_t)n_cta * R < (size_t)H)
    return PRNN_ERR_INVALID_ARG;
  if (tpr != 1 && tpr != 2 && tpr != 4 && tpr != 8 && tpr != 16 && tpr != 32)
    return PRNN_ERR_INVALID_ARG;
  if (!vals || !cols || !ept) return PRNN_ERR_INVALID_ARG;
  std::vector<int> seen((size_t)H, -1);
  for (int r = 0; r < H; ++r)
    for (int j = 0; j < k; ++j) {
      const int c = cols[(size_t)r * k + j];
      if (c >= H || seen[c] == r) return PRNN_ERR_INVALID_ARG;
      seen[c] = r;
    }
  std::vector<uint32_t> pk;
  PackStats st;
  *ept = pack_sparse_rows(H, k, R, n_cta, tpr, vals, cols, pk, &st);
  if (bank_cap) *bank_cap = st.cap;
  if (!packed || capacity_words < pk.size()) return PRNN_ERR_INVALID_ARG;
  std::memcpy(packed, pk.data(), pk.size() * sizeof(uint32_t));
  return PRNN_OK;
}

prnn_status_t prnn_pack_dense_ksplit_host(int hidden, int cluster_size, const uint16_t* wh16,
                                          int transpose, uint16_t* image, size_t capacity_elems,
                                          size_t* image_elems) {
  const int H = hidden, cs = cluster_size;
  if (H < 128 || H % 128 != 0 || H > 65536 || cs < 2 || cs > kKsplitMaxCluster || H / 16 < cs)
    return PRNN_ERR_INVALID_ARG;
  if (!wh16 || !image_elems) return PRNN_ERR_INVALID_ARG;
  const int nat = ksplit_nat(H, cs);
  const size_t need = (size_t)(H / 128) * cs * nat * 128 * 64;
  *image_elems = need;
  if (!image || capacity_elems < need) return PRNN_ERR_INVALID_ARG;
  std::fill(image, image + need, (uint16_t)0);
  build_ksplit_image(H, cs, nat, wh16, transpose != 0, image);
  return PRNN_OK;
}

prnn_status_t prnn_pack_sparse_host_placed(int hidden, int k, int n_cta, int rows_per_cta,
                                           int threads_per_row, const uint16_t* vals,
                                           const uint16_t* cols, uint32_t* packed,
                                           size_t capacity_words, uint32_t* place,
                                           size_t place_capacity_words, int* ept,
                                           int* bank_cap, int* placed) {
  const int H = hidden, R = rows_per_cta, tpr = threads_per_row;
  if (H < 1 || H > 65535 || k < 1 || k > H || n_cta < 1 || R < 1 || (size_t)n_cta * R < (size_t)H)
    return PRNN_ERR_INVALID_ARG;
  if (tpr != 1 && tpr != 2 && tpr != 4 && tpr != 8 && tpr != 16 && tpr != 32)
    return PRNN_ERR_INVALID_ARG;
  if (!vals || !cols || !ept || !placed) return PRNN_ERR_INVALID_ARG;
  std::vector<int> seen((size_t)H, -1);
  for (int r = 0; r < H; ++r)
    for (int j = 0; j < k; ++j) {
      const int c = cols[(size_t)r * k + j];
      if (c >= H || seen[c] == r) return PRNN_ERR_INVALID_ARG;
      seen[c] = r;
    }
  std::vector<uint32_t> pk, pl;
  PackStats st;
  *ept = pack_sparse_rows(H, k, R, n_cta, tpr, vals, cols, pk, &st, 1 << 30, true, &pl);
  *placed = pl.empty() ? 0 : 1;
  if (bank_cap) *bank_cap = st.cap;
  if (!packed || capacity_words < pk.size()) return PRNN_ERR_INVALID_ARG;
  if (!pl.empty() && (!place || place_capacity_words < pl.size())) return PRNN_ERR_INVALID_ARG;
  std::memcpy(packed, pk.data(), pk.size() * sizeof(uint32_t));
  if (!pl.empty()) std::memcpy(place, pl.data(), pl.size() * sizeof(uint32_t));
  return PRNN_OK;
}

}  // extern "C"
